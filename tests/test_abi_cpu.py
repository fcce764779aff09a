"""The C ABI without a GPU: the library builds, loads, exports every function
include/fa.h declares, and rejects bad arguments on the host before touching
CUDA."""

import ctypes
import os
import re

import numpy as np

import pytest
import torch

from exact_io_aware_37_gb300 import build as fa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]

OK, INVALID, UNSUPPORTED, ALIGN, CUDA, TIMEOUT, WORKSPACE = 0, -1, -2, -3, -4, -5, -6


@pytest.fixture(scope="module")
def lib():
    fa_build.build()
    from exact_io_aware_37_gb300 import _lib
    return _lib.lib()


def declared_functions():
    names = []
    for h in HEADERS:
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        for m in re.finditer(r"\b([A-Za-z_][A-Za-z0-9_]*)\s*\(", src):
            name = m.group(1)
            if name.startswith("fa_") and name not in names:
                names.append(name)
    return names


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("fa_fwd", "fa_bwd", "fa_bwd_workspace_size", "fa_strerror", "fa_get_last_device_error"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    handle = ctypes.CDLL(fa_build.LIB_PATH)
    for name in declared_functions():
        assert hasattr(handle, name), f"{name} declared in include/ but not exported"


def _fwd(lib, q=0x1000, k=0x1000, v=0x1000, o=0x1000, lse=0x1000, B=1, H=1, N=128, D=128, scale=0.1,
         causal=0, cu=None, T=0, dt=0):
    return lib.fa_fwd(q, k, v, o, lse, B, H, N, D, scale, causal, cu, T, dt, None)


def test_forward_argument_validation(lib):
    assert _fwd(lib, D=96) == UNSUPPORTED
    assert _fwd(lib, D=48, dt=1) == UNSUPPORTED
    assert _fwd(lib, dt=7) == UNSUPPORTED
    assert _fwd(lib, D=32, dt=2) == UNSUPPORTED     # fp16 runs on the tensor cores only: D 64 or 128
    assert _fwd(lib, B=-1) == INVALID
    assert _fwd(lib, N=-5) == INVALID
    assert _fwd(lib, scale=float("nan")) == INVALID
    assert _fwd(lib, scale=float("inf")) == INVALID
    # the kernels take each row's maximum over unscaled scores: only a positive scale is accepted
    assert _fwd(lib, scale=0.0) == INVALID
    assert _fwd(lib, scale=-0.0) == INVALID
    assert _fwd(lib, scale=-0.125) == INVALID
    assert _fwd(lib, scale=-0.125, dt=1, D=64) == INVALID
    assert _fwd(lib, causal=2) == INVALID
    assert _fwd(lib, q=None) == INVALID
    assert _fwd(lib, lse=None) == INVALID
    assert _fwd(lib, v=0x1008) == ALIGN
    assert _fwd(lib, o=0x1001) == ALIGN
    assert _fwd(lib, cu=0x1000, T=-1) == INVALID
    # nothing to do: succeeds without launching anything (and without a GPU)
    assert _fwd(lib, B=0) == OK
    assert _fwd(lib, N=0) == OK
    assert _fwd(lib, cu=0x1000, T=0) == OK


def test_backward_argument_validation(lib):
    def bwd(ws=0x100000, ws_bytes=1 << 30, **kw):
        a = dict(q=0x1000, k=0x1000, v=0x1000, o=0x1000, lse=0x1000, do=0x1000, dq=0x1000, dk=0x1000,
                 dv=0x1000, B=1, H=1, N=128, D=128, scale=0.1, causal=1, cu=None, T=0, dt=0)
        a.update(kw)
        return lib.fa_bwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["do"], a["dq"], a["dk"], a["dv"], a["B"],
                          a["H"], a["N"], a["D"], a["scale"], a["causal"], a["cu"], a["T"], a["dt"], ws, ws_bytes,
                          None)
    assert bwd(D=80) == UNSUPPORTED
    assert bwd(dk=None) == INVALID
    assert bwd(dv=0x1004) == ALIGN
    assert bwd(ws=None) == WORKSPACE
    assert bwd(ws=0x100010) == WORKSPACE          # not 256-byte aligned
    assert bwd(ws_bytes=16) == WORKSPACE
    assert bwd(H=0) == OK
    assert bwd(scale=0.0) == INVALID
    assert bwd(scale=-1.0) == INVALID
    det = lib.fa_bwd_deterministic(0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 1, 1,
                                   128, 128, -0.1, 1, None, 0, 0, 0.0, 7, 0, 0x100000, 1 << 30, None)
    assert det == INVALID


def test_tile_selftest_argument_validation(lib):
    def tile(a=0x1000, b=0x1000, s=0x1000, o=0x1000, ac=0x1000, D=128, dt=0):
        return lib.fa_selftest_tile(a, b, s, o, ac, D, dt, None)
    assert tile(D=96) == UNSUPPORTED
    assert tile(D=32) == UNSUPPORTED
    assert tile(dt=1) == UNSUPPORTED     # float32 has no tensor-core tile
    assert tile(dt=7) == UNSUPPORTED
    assert tile(a=None) == INVALID
    assert tile(ac=None) == INVALID
    assert tile(s=0x1004) == ALIGN
    assert tile(o=0x1008) == ALIGN


def test_workspace_size(lib):
    f = lib.fa_bwd_workspace_size
    # D vector (4 B per row) + float32 dQ accumulator + a 256-byte block for the
    # backward's tile counter, for the tensor-core path
    assert f(2, 32, 4096, 128, None, 0, 0) == 2 * 32 * 4096 * 4 + 2 * 32 * 4096 * 128 * 4 + 256
    # packed: rows = H * T, rounded up to 256 bytes per part
    assert f(16, 32, 8192, 128, 0x1000, 1001, 0) == (32 * 1001 * 4 + 255) // 256 * 256 + 32 * 1001 * 128 * 4 + 256
    # fp16 uses the same tensor-core path and workspace as bf16
    assert f(2, 32, 4096, 128, None, 0, 2) == f(2, 32, 4096, 128, None, 0, 0)
    # float32 path needs only the D vector
    assert f(1, 1, 128, 64, None, 0, 1) == 512
    assert f(-1, 1, 1, 64, None, 0, 0) == 0


def test_strerror_and_path_names(lib):
    for code in (OK, INVALID, UNSUPPORTED, ALIGN, CUDA, TIMEOUT, WORKSPACE):
        assert lib.fa_strerror(code)
    assert lib.fa_path_name(1, 64) == b"simt_f32"
    assert lib.fa_path_name(0, 96) is None
    assert lib.fa_path_name(0, 128) is not None
    assert lib.fa_path_name(2, 64) == lib.fa_path_name(0, 64) == b"tcgen05"
    assert lib.fa_path_name(2, 32) is None


def test_dropout_validation(lib):
    def fwd(p, dt=0, **kw):
        a = dict(q=0x1000, k=0x1000, v=0x1000, o=0x1000, lse=0x1000, B=1, H=1, N=128, D=128, scale=0.1, causal=1,
                 cu=None, T=0)
        a.update(kw)
        return lib.fa_fwd_dropout(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"], a["D"],
                                  a["scale"], a["causal"], a["cu"], a["T"], dt, p, 7, 0, None)
    assert fwd(-0.1) == INVALID
    assert fwd(1.0) == INVALID
    assert fwd(float("nan")) == INVALID
    assert fwd(0.2, dt=1, D=64) == UNSUPPORTED   # no dropout on the float32 path
    assert fwd(0.2, B=0) == OK
    assert fwd(0.2, scale=-0.1) == INVALID
    bwd = lib.fa_bwd_dropout(0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 1, 1, 128, 128,
                             0.1, 1, None, 0, 0, 1.5, 7, 0, 0x100000, 1 << 30, None)
    assert bwd == INVALID


def test_decode_validation_and_workspace(lib):
    def dec(ws=0x100000, ws_bytes=1 << 30, **kw):
        a = dict(q=0x1000, k=0x1000, v=0x1000, o=0x1000, lse=0x1000, B=1, H=2, nq=1, nk=1000, D=128, scale=0.1,
                 causal=1, dt=0)
        a.update(kw)
        return lib.fa_decode(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["nq"], a["nk"], a["D"],
                             a["scale"], a["causal"], a["dt"], ws, ws_bytes, None)
    assert dec(D=96) == UNSUPPORTED
    assert dec(D=32) == UNSUPPORTED
    assert dec(dt=7) == UNSUPPORTED
    assert dec(nq=-1) == INVALID
    assert dec(nk=-1) == INVALID
    assert dec(causal=2) == INVALID
    assert dec(scale=float("nan")) == INVALID
    assert dec(scale=0.0) == INVALID
    assert dec(scale=-0.1) == INVALID
    assert dec(q=None) == INVALID
    assert dec(lse=None) == INVALID
    assert dec(k=0x1008) == ALIGN
    assert dec(ws=None) == WORKSPACE
    assert dec(ws=0x100010) == WORKSPACE
    assert dec(ws_bytes=16) == WORKSPACE
    assert dec(B=0) == OK and dec(nq=0) == OK
    assert dec(k=None) == INVALID
    size = lib.fa_decode_workspace_size
    # 1 x 2 heads, 1000 keys: four splits of 250 keys; per split and row D floats + (m, l)
    assert size(1, 2, 1, 1000, 128, 0) == 4 * 2 * 128 * 4 + 256
    # enough (b, h) pairs to fill the GPU: one split, no scratch
    assert size(16, 64, 1, 8192, 128, 0) == 0
    assert size(1, 1, 1, 100, 64, 0) == 0 and size(0, 1, 1, 100, 64, 0) == 0


# Calls that pass validation would launch kernels on fake pointers where a GPU
# is present, so they run only where there is none.
@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU error path")
def test_valid_call_without_gpu_reports_cuda_error(lib):
    assert _fwd(lib) == CUDA
    assert _fwd(lib, D=64, dt=1) == CUDA            # float32 with D = 64 is supported (SIMT path)
    # an empty cache needs no K / V pointers
    assert lib.fa_decode(0x1000, None, None, 0x1000, 0x1000, 1, 2, 1, 0, 128, 0.1, 1, 0, 0x100000, 1 << 30,
                         None) == CUDA


def test_no_kernel_spills_registers(lib):
    """ptxas's report of every translation unit the library is built from: no
    kernel stores registers to local memory (a spill in a role of a
    warp-specialised kernel puts local-memory round trips on its critical path)."""
    spills = []
    for src in fa_build.SOURCES:
        log = os.path.join(fa_build.BUILD, src.replace(".cu", ".ptxas.txt"))
        assert os.path.exists(log), f"no ptxas report for {src}"
        kernel = None
        for line in open(log):
            m = re.search(r"Compiling entry function '(\S+)'", line)
            if m:
                kernel = m.group(1)
            m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
            if m and (int(m.group(1)) or int(m.group(2))):
                spills.append((src, kernel, line.strip()))
    assert not spills, spills


def test_static_scratch_limit(lib):
    """fa_bwd_static_ws's fixed scratch holds the workspace of at most 32,513
    rows at D = 128, 64,526 at D = 64 and 4,194,304 in float32; one row more
    needs more than FA_BWD_STATIC_WS_BYTES (refused before any launch)."""
    limit = 16 << 20
    size = lib.fa_bwd_workspace_size
    for D, dt, rows in ((128, 0, 32513), (64, 0, 64526), (128, 2, 32513), (64, 1, 4194304)):
        assert size(1, 1, rows, D, None, 0, dt) <= limit < size(1, 1, rows + 1, D, None, 0, dt)
        # the packed layout counts H * total_tokens rows
        assert size(3, 1, rows, D, 0x1000, rows, dt) <= limit < size(3, 1, rows, D, 0x1000, rows + 1, dt)
    with open(os.path.join(ROOT, "include", "fa.h")) as f:
        assert "#define FA_BWD_STATIC_WS_BYTES ((size_t)16 << 20)" in f.read()


def test_python_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    from exact_io_aware_37_gb300 import _lib
    monkeypatch.setattr(_lib, "_LIB", None)
    monkeypatch.setattr(_lib, "library_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no fallback"):
        _lib.lib()


# Work lists of the persistent launches (host logic, no GPU).  Weights are the
# per-item step counts plus the per-item overheads the table builder charges:
# 1 step for a forward query-tile pair, 2 for a backward key tile.
def _preview(lib, kernel, B, H, N, causal, ctas, lengths=None, cap=1 << 17, D=128):
    cu = None
    if lengths is not None:
        cu = (ctypes.c_int32 * (len(lengths) + 1))(*([0] + list(np.cumsum(lengths))))
    off = (ctypes.c_int * (ctas + 1))()
    items = (ctypes.c_uint * cap)()
    form = ctypes.c_int(-1)
    n = lib.fa_schedule_preview(kernel, cu, B, H, N, D, causal, ctas, off, items, cap, ctypes.byref(form))
    return n, list(off), list(items[:max(n, 0)]), form.value


def _weights(kernel, H, B, N, causal, lengths=None):
    """code -> weight of every real item (codes as fa_schedule_preview writes them)."""
    lens = lengths if lengths is not None else [N] * B
    ranks = ((N + 127) // 128 + 1) // 2 if kernel == 0 else (N + 127) // 128
    out = {}
    for b, n in enumerate(lens):
        n_t = (n + 127) // 128
        for h in range(H):
            u = b * H + h
            if kernel == 0:
                for pr in range((n_t + 1) // 2):
                    out[u * ranks + pr] = (min(2 * pr + 2, n_t) if causal else n_t) + 1
            else:
                for kt in range(n_t):
                    out[u * ranks + kt] = (n_t - kt if causal else n_t) + 2
    return out


def _loads(n, off, items, weight, used):
    assert n == len(weight)
    assert sorted(items) == sorted(weight)          # every item exactly once
    assert off[0] == 0 and off[used] == n
    assert all(off[c] <= off[c + 1] for c in range(used))
    return [sum(weight[code] for code in items[off[c]:off[c + 1]]) for c in range(used)]


@pytest.mark.parametrize("kernel,B,H,N,causal,ctas", [
    (0, 2, 32, 4096, 1, 152), (0, 2, 32, 4096, 0, 152), (1, 2, 32, 4096, 1, 152), (1, 2, 32, 4096, 0, 152),
    (0, 4, 16, 1024, 1, 152), (1, 4, 16, 1024, 1, 152), (0, 1, 3, 300, 1, 152), (1, 1, 3, 300, 0, 7),
    (0, 1, 32, 32768, 1, 152), (1, 2, 5, 2000, 1, 64)])
def test_persistent_table_covers_and_balances(lib, kernel, B, H, N, causal, ctas):
    n, off, items, form = _preview(lib, kernel, B, H, N, causal, ctas)
    assert form == 0                                  # dense, at most 4096 items: the host table
    weight = _weights(kernel, H, B, N, causal)
    loads = _loads(n, off, items, weight, min(ctas, 160, n))
    # greedy assignment to the least-loaded CTA: no CTA ends more than one item heavier than another
    assert max(loads) - min(loads) <= max(weight.values())
    assert max(loads) <= sum(loads) / len(loads) + max(weight.values())


@pytest.mark.parametrize("kernel", [0, 1])
def test_table_groups_heads_only_beyond_l2(lib, kernel):
    """The host table groups heads only to keep the operands they re-read in L2.
    B4 H16 N1024 at D = 64 (K, V: 16 MB; Q, dO, dQ accumulator: 32 MB) is one
    group: CTA c < 64 starts on head c's heaviest item, and the load spread is
    below what grouping gave (forward max/avg 1.39, backward 1.23).  B2 H32
    N4096 at D = 128 (128 MB / 256 MB) keeps its groups of 16 / 4 heads."""
    ranks_of = lambda N: ((N + 127) // 128 + 1) // 2 if kernel == 0 else (N + 127) // 128
    heaviest = lambda N: ranks_of(N) - 1 if kernel == 0 else 0   # last pair / first key tile
    n, off, items, form = _preview(lib, kernel, 4, 16, 1024, 1, 152, D=64)
    assert form == 0
    r = ranks_of(1024)
    firsts = [items[off[c]] for c in range(64)]
    assert sorted(code // r for code in firsts) == list(range(64))
    assert all(code % r == heaviest(1024) for code in firsts)
    weight = _weights(kernel, 16, 4, 1024, 1)
    loads = _loads(n, off, items, weight, 152)
    assert max(loads) / (sum(loads) / len(loads)) < (1.2 if kernel == 0 else 1.1)
    n, off, items, form = _preview(lib, kernel, 2, 32, 4096, 1, 152, D=128)
    group = 16 if kernel == 0 else 4
    r = ranks_of(4096)
    firsts = [items[off[c]] for c in range(group + 1)]
    assert sorted(code // r for code in firsts[:group]) == list(range(group))
    assert firsts[group] % r != heaviest(4096)   # the group's next-heaviest items come before other heads


@pytest.mark.parametrize("kernel,N", [(0, 2048), (1, 1024)])
def test_table_depends_on_the_head_width(lib, kernel, N):
    """At B4 H16 the operands the items re-read fit in L2 together at D = 64
    but not at D = 128 (forward at N = 2048: K, V 32 MB / 64 MB; backward at
    N = 1024: Q, dO, dQ accumulator 32 MB / 64 MB), so the two head widths get
    different tables for the same B, H, N and mask: a table cached on the host
    has to be keyed by D as well."""
    a = _preview(lib, kernel, 4, 16, N, 1, 152, D=64)
    b = _preview(lib, kernel, 4, 16, N, 1, 152, D=128)
    assert a[3] == 0 and b[3] == 0
    assert sorted(a[2]) == sorted(b[2])          # the same items...
    assert (a[1], a[2]) != (b[1], b[2])          # ...handed out differently


@pytest.mark.parametrize("kernel,B,H,N,causal", [
    (0, 1, 64, 32768, 1),     # 8192 pairs
    (0, 3, 40, 12345, 1)])    # ragged length
def test_persistent_closed_form_dense(lib, kernel, B, H, N, causal):
    """Beyond 4096 items the forward's closed form: every item once, heaviest
    ranks first across all heads, a snake over the CTAs; for a list sorted by
    weight the snake keeps every CTA within one item of the average."""
    ctas = 152
    n, off, items, form = _preview(lib, kernel, B, H, N, causal, ctas)
    assert form == 1
    weight = _weights(kernel, H, B, N, causal)
    loads = _loads(n, off, items, weight, ctas)
    avg = sum(loads) / ctas
    assert max(loads) <= avg + max(weight.values())
    assert min(loads) >= avg - max(weight.values())
    # CTA 0 takes virtual items 0, 2P-1, 2P, 4P-1, ...: its first item is unit 0's heaviest
    ranks = ((N + 127) // 128 + 1) // 2 if kernel == 0 else (N + 127) // 128
    first = items[off[0]]
    assert first // ranks == 0 and weight[first] == max(weight.values())


@pytest.mark.parametrize("causal", [0, 1])
def test_persistent_closed_form_packed(lib, causal):
    """Packed sequences in the forward (the 16-sequence workload's seeded
    lengths): every (sequence, head) item once, none of a sequence of length
    0 or of a malformed sequence, and every CTA within 10 % of the ideal
    finish time."""
    from exact_io_aware_37_gb300 import synth
    kernel = 0
    lengths = synth.varlen_lengths(16, 128, 8192).tolist()
    H, N = 32, max(lengths)
    n, off, items, form = _preview(lib, kernel, len(lengths), H, N, causal, 152, lengths=lengths)
    assert form == 1
    weight = _weights(kernel, H, len(lengths), N, causal, lengths)
    loads = _loads(n, off, items, weight, 152)
    ideal = max(sum(loads) / 152, max(weight.values()))
    assert max(loads) <= 1.1 * ideal
    # empty sequences contribute nothing; small problems use fewer CTAs than SMs
    lens2 = [300, 0, 129, 1]
    n2, off2, items2, _ = _preview(lib, kernel, 4, 2, 300, causal, 152, lengths=lens2)
    weight2 = _weights(kernel, 2, 4, 300, causal, lens2)
    used = 4 * 2 * (((300 + 127) // 128 + 1) // 2 if kernel == 0 else (300 + 127) // 128)
    _loads(n2, off2, items2, weight2, used)


@pytest.mark.parametrize("B,H,N,causal,lengths", [
    (1, 32, 32768, 1, None),                 # 8192 key tiles: the long-window backward
    (4, 32, 8192, 0, None),                  # no mask
    (9, 7, 12345, 1, None),                  # ragged length, a short last group
    (6, 3, 5000, 1, [300, 0, 5000, 129, 1, 4000]),
    (16, 32, 8192, 1, "varlen16")])
def test_backward_queue_order(lib, B, H, N, causal, lengths):
    """Beyond the table (and for packed input) the backward's CTAs take key
    tiles from one queue: every real tile exactly once; (sequence, head) units
    in groups of about 4, each group's tiles contiguous and rank-major, so the
    heaviest tiles of a group come first."""
    if lengths == "varlen16":
        from exact_io_aware_37_gb300 import synth
        lengths = synth.varlen_lengths(16, 128, 8192).tolist()
        N = max(lengths)
    n, off, items, form = _preview(lib, 1, B, H, N, causal, 152, lengths=lengths)
    assert form == 2
    assert off[0] == 0 and all(o == n for o in off[1:])
    weight = _weights(1, H, B, N, causal, lengths)
    assert n == len(weight) and sorted(items) == sorted(weight)
    ranks = (N + 127) // 128
    units = [code // ranks for code in items]
    tiles = [code % ranks for code in items]
    n_units = B * H
    per = -(-n_units // -(-n_units // 4))      # about 4 units per group, spread evenly
    groups = [u // per for u in units]
    assert groups == sorted(groups)          # one group after the other
    for g in set(groups):
        t = [kt for kt, gg in zip(tiles, groups) if gg == g]
        assert t == sorted(t)                # rank-major: key tile 0 (the heaviest) of every unit first


def test_persistent_schedule_refusals(lib):
    assert _preview(lib, 2, 1, 1, 128, 1, 152)[0] == -1         # no such kernel
    assert _preview(lib, 0, 1, 1, 0, 1, 152)[0] == -1           # empty problem
    assert _preview(lib, 1, 2, 32, 4096, 1, 152, cap=4)[0] == -2
    assert _preview(lib, 1, 1, 32, 32768, 1, 152, cap=100)[0] == -2
    assert _preview(lib, 0, 1, 64, 32768, 1, 152, cap=100)[0] == -2


# Host calls that allocate device or pinned memory, or wait for the device.
_ALLOC_OR_SYNC = re.compile(r"\b(cudaMalloc\w*|cudaFree\w*|cudaHostAlloc|cudaMallocHost|cudaDeviceSynchronize|"
                            r"cudaStreamSynchronize|cudaEventSynchronize|cudaMemcpy|cudaMemset|cudaMemcpyToSymbol|"
                            r"cudaMemcpyFromSymbol)\s*\(")


def _strip_comments(src):
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return re.sub(r"//[^\n]*", "", src)


def test_compute_calls_neither_allocate_nor_wait():
    """The attention and decoding entry points only enqueue work on the
    caller's stream (which is what lets a caller capture them in a CUDA
    graph): no translation unit calls an allocator or a waiting or
    synchronous copy call, except the status read-back
    (fa_get_last_device_error, which the self-tests return) and the ex2 rate
    probe, both documented as synchronising."""
    csrc = os.path.join(ROOT, "exact_io_aware_37_gb300", "csrc")
    allowed = {"fa_api.cu": 3, "fa_probe.cu": 2}
    for name in sorted(os.listdir(csrc)):
        if not name.endswith((".cu", ".cuh")):
            continue
        hits = _ALLOC_OR_SYNC.findall(_strip_comments(open(os.path.join(csrc, name)).read()))
        assert len(hits) == allowed.get(name, 0), (name, hits)
    api = _strip_comments(open(os.path.join(csrc, "fa_api.cu")).read())
    body = api[api.index("fa_status fa_get_last_device_error("):]
    body = body[:body.index("\n}\n")]
    assert len(_ALLOC_OR_SYNC.findall(body)) == 3       # all three sit in the status read-back


C_CALLER = r"""
#include <stdio.h>
#include <string.h>
#include "fa.h"

int main(void) {
  /* argument checks return before any CUDA call, so this runs without a GPU */
  if (fa_fwd((void*)0, (void*)0, (void*)0, (void*)0, (float*)0, 1, 1, 128, 128, 0.125f, 1, NULL, 0, FA_BF16,
             NULL) != FA_ERR_INVALID) return 1;
  if (fa_fwd((void*)0x1000, (void*)0x1000, (void*)0x1000, (void*)0x1000, (float*)0x1000, 1, 1, 128, 96, 0.125f, 0,
             NULL, 0, FA_BF16, NULL) != FA_ERR_UNSUPPORTED) return 2;
  if (fa_bwd_workspace_size(2, 32, 4096, 128, NULL, 0, FA_BF16) !=
      (size_t)2 * 32 * 4096 * 4 + (size_t)2 * 32 * 4096 * 128 * 4 + 256) return 3;
  if (strcmp(fa_strerror(FA_ERR_ALIGN), "tensor pointer not 16-byte aligned") != 0) return 4;
  if (fa_path_name(FA_BF16, 128) == NULL || fa_path_name(FA_BF16, 96) != NULL) return 5;
  if (FA_BWD_STATIC_WS_BYTES != (size_t)16 << 20) return 6;
  printf("ok\n");
  return 0;
}
"""


def test_header_is_plain_c_and_the_library_links_from_c(lib, tmp_path):
    """A C99 caller that includes include/fa.h, links libfa_gb300.so and calls
    the host-side parts of the boundary: the header needs no C++ and the
    library no Python."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc") or shutil.which("cc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "caller.c"
    src.write_text(C_CALLER)
    exe = tmp_path / "caller"
    libdir = os.path.dirname(fa_build.LIB_PATH)
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                        "-L", libdir, "-lfa_gb300", f"-Wl,-rpath,{libdir}", "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout, r.stderr)
