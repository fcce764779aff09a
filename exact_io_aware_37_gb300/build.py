"""Build libfa_gb300.so in-tree with nvcc for sm_103a.

Each CUDA translation unit is compiled in parallel to an object file, then
linked into one shared library (CUDA runtime linked statically, the driver
entry point for tensor maps resolved at run time), so the library loads on a
machine without a GPU and exports only the C ABI of include/fa.h.
"""

import concurrent.futures as cf
import os
import re
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB_NAME = "libfa_gb300.so"
LIB_PATH = os.path.join(BUILD, LIB_NAME)

SOURCES = ["fa_api.cu", "fa_simt.cu", "fa_tc_fwd.cu", "fa_tc_bwd.cu", "fa_tc_bwd128.cu", "fa_static_ws.cu",
           "fa_decode.cu", "fa_tc_bwd_dq.cu", "fa_probe.cu", "fa_selftest.cu"]

# The tensor-core kernels move registers between warpgroups with setmaxnreg
# (384-thread kernels from 168 registers per thread at launch: the forward
# 200 + 200 + 104, the backward 184 + 184 + 136).  Each split is only safe
# when every thread starts with the launch count it was sized for; a kernel
# that ptxas compiled with fewer would wait forever in setmaxnreg.inc, so the
# build refuses it.
# kernel name -> registers per thread it must be compiled with (checked in order)
SPLIT_KERNELS = {"tc_bwd128_kernel": 168, "tc_fwd_kernel": 168, "tc_bwd_dq_kernel": 168}
SPLIT_SOURCES = ("fa_tc_fwd.cu", "fa_tc_bwd128.cu", "fa_tc_bwd_dq.cu")  # each must report its split kernels
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-Xptxas", "-v", "-I", INCLUDE, "-I", CSRC]


def nvcc_path():
    for cand in (os.environ.get("NVCC"),
                 os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc"),
                 shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or CUDA_HOME)")


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh", ".h"))]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return files


def up_to_date():
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(f) <= t for f in _inputs() + [os.path.abspath(__file__)])


def check_register_split(log_text, src):
    """Raise unless every split kernel in a ptxas -v log uses its expected
    register count; returns how many such kernels the log reports."""
    current = None
    seen = 0
    for line in log_text.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            current = m.group(1)
            continue
        m = re.search(r"Used (\d+) registers", line)
        name = next((k for k in SPLIT_KERNELS if current and k in current), None)
        if m and name:
            regs = int(m.group(1))
            if regs != SPLIT_KERNELS[name]:
                raise RuntimeError(f"{src}: {current} compiled with {regs} registers; the warpgroup register "
                                   f"split needs exactly {SPLIT_KERNELS[name]}")
            seen += 1
            current = None
    return seen


def build(force=False, verbose=False, jobs=None):
    """Compile and link; returns the library path.  Raises on failure."""
    if not force and up_to_date():
        return LIB_PATH
    os.makedirs(BUILD, exist_ok=True)
    nvcc = nvcc_path()

    def compile_one(src):
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        log = os.path.join(BUILD, src.replace(".cu", ".ptxas.txt"))
        cmd = [nvcc, *ARCH, *FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        with open(log, "w") as f:
            f.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr[-6000:]}")
        if check_register_split(r.stdout + r.stderr, src) == 0 and src in SPLIT_SOURCES:
            raise RuntimeError(f"{src}: no register report found for the split kernels")
        if verbose:
            sys.stderr.write(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=jobs or len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB_PATH + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr[-6000:]}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
