"""Throughput of exact attention, forward + backward, on GB300.

One step = fa_fwd then fa_bwd over one batch of seeded synthetic bf16 input
of the causal B=2 H=32 N=4096 D=128 workload (the seq-4096, 32-head shape of
the pages' timing example), inputs resident in device memory.  Prints ONE
JSON line (rank 0).  ``value`` is fwd+bwd TFLOP/s with FLOPs counted as
4*B*H*N^2*D (halved when causal) for the forward pass and 2.5x that for the
backward pass; ``fwd_tflops`` is the forward pass alone.

The step is first run eagerly (one host launch per kernel), with CUDA events
between the passes and around the main backward kernel: that loop gives the
forward / backward split and the roofline of the dominant kernel, and goes
under ``eager``.  The same step is then captured once in a CUDA graph and
replayed ``steps`` times; the replays (the same kernels and work, without the
host launch path between them) give ``value`` and ``ms_per_step``.  If the
capture fails the eager loop gives them.  After the headline's timed regions
the default run on one GPU also measures the other configurations (mid, long
non-causal, packed, long window) for a few steps each and carries their figures under
``workloads`` (``--no-workloads`` leaves them out; ``--workload NAME`` gives
one configuration's full line).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs its own replica (the path has no exchange
step), the timed region is bracketed by barriers and the slowest rank's time
is reported.  ``--impl reference`` times the float64 CPU oracle on a bounded
sample of the same workload (rank 0 only).
"""

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "long_b2h32n4096d128"
CAUSAL = True
METRIC = "attention fwd & fwd+bwd TFLOP/s (bf16, causal) and % of GB300 BF16 tensor peak"
L2_BYTES = 129 * 2 ** 20
FALLBACK_PEAK_TFLOPS = 1900.0

# dram__bytes_read.sum + dram__bytes_write.sum per launch of the dominant
# kernel from one ncu capture, keyed by the SHA-256 of that kernel's source
# file at capture time (reported as null once the source has changed).
TRAFFIC_BY_SOURCE = {
    # tc_bwd128_kernel<128, bf16>, B2 H32 N4096 D128 causal: 405.0 MB read + 220.6 MB written
    "ce594b4f7f1d737c9d87a65e888f7f6a4c6bfdfd89f587f781844eb3c667351c": 625.6e6,
    # the same file with only its host code changed (the cached schedule's key
    # also holds the head width); the kernel's device code is as captured
    "4a6f022408ced7574c15298975ae7ebd1f8b8b42f797497503f9dd5c947c92e8": 625.6e6,
    # decode_split_kernel, B16 H32 nq1 nk8192 D128: 2147.7 MB read + 3.8 MB written
    "fee09d5aa4225f18dc40dd1517d297a22d708da1eb55e0890c30901cdf5a3bb5": 2151.5e6,
}


def flops_fwd(B, H, N, D, causal):
    f = 4.0 * B * H * N * N * D
    return f / 2 if causal else f


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p["hbm_gbs"]), "measured"
    return FALLBACK_PEAK_TFLOPS, 6800.0, "fallback"


def hbm_peak():
    _, gbs, kind = peaks()
    return gbs, f"HBM copy, {kind}"


class ClockSampler:
    """SM clock, power and clock-event reasons sampled while the timed region
    runs: read in-process through NVML (read-only queries, every ~0.2 ms, so a
    timed region of a few milliseconds still gets many samples); nvidia-smi
    at 50 ms where the NVML library cannot be loaded."""

    # NVML clock-event reason bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index, period_s=0.0002):
        self.index = index
        self.period_s = period_s
        self.samples = []  # (sm_mhz, max_mhz, power_w, reason_bits)
        self.lines = []
        self.source = None
        self.proc = None
        self.thread = None
        self._stop = threading.Event()

    def _nvml_handle(self):
        import ctypes
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        props = torch.cuda.get_device_properties(self.index)
        bus = None
        if all(hasattr(props, a) for a in ("pci_domain_id", "pci_bus_id", "pci_device_id")):
            bus = f"{props.pci_domain_id:08X}:{props.pci_bus_id:02X}:{props.pci_device_id:02X}.0".encode()
        if bus is None or nv.nvmlDeviceGetHandleByPciBusId_v2(bus, ctypes.byref(h)) != 0:
            if nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index), ctypes.byref(h)) != 0:
                raise OSError("no NVML handle")
        return nv, h

    def _poll_nvml(self, nv, h):
        import ctypes
        sm, mx, pw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        max_ok = nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0  # fixed: read once
        n = 0
        while not self._stop.is_set():
            ok = max_ok and nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(sm)) == 0      # NVML_CLOCK_SM
            ok = ok and reasons_fn(h, ctypes.byref(rs)) == 0
            power = n % 8 == 0 and nv.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw)) == 0
            if ok:
                self.samples.append((sm.value, mx.value, pw.value / 1e3 if power else None, rs.value))
            n += 1
            self._stop.wait(self.period_s)

    def __enter__(self):
        try:
            nv, h = self._nvml_handle()
            self.source = "nvml"
            self.thread = threading.Thread(target=self._poll_nvml, args=(nv, h), daemon=True)
            self.thread.start()
            return self
        except (OSError, AttributeError, RuntimeError):
            pass
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi"
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        self._stop.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self):
        sm, mx, pw, reasons = [], [], [], set()
        for s_mhz, m_mhz, p_w, bits in self.samples:
            sm.append(float(s_mhz))
            mx.append(float(m_mhz))
            if p_w is not None:
                pw.append(p_w)
            reasons.update(name for bit, name in self.REASONS.items() if bits & bit)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
                pw.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[3:7]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": self.source}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "sm_min_mhz": min(sm),
                "reasons": sorted(reasons), "samples": len(sm), "power_w_max": max(pw) if pw else None,
                "source": self.source}


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        return dist, rank, world, local
    return None, 0, 1, 0


def max_over_ranks(dist, x, device):
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


def graph_replay_measure(step, flops, steps, warmup, device, dist, world, local, unit="TFLOP/s"):
    """The step captured once in a CUDA graph and replayed: the library's calls
    enqueue no host synchronisation and no allocation, so the step's kernels
    (the same launches, the same work) replay without the host launch path
    between them.  `step(stream)` enqueues one step on `stream`.  Times `steps`
    replays with CUDA events on the replay stream, barrier and synchronize on
    both sides, max over ranks, clocks sampled meanwhile; returns a dict for
    the JSON line ("unavailable" and the reason if the capture fails)."""
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step(torch.cuda.current_stream(device))
        for _ in range(max(warmup, 3)):
            g.replay()
        torch.cuda.synchronize()
        stream = torch.cuda.current_stream(device)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(local) as clocks:
            barrier(dist)
            torch.cuda.synchronize()
            t0.record(stream)
            for _ in range(steps):
                g.replay()
            t1.record(stream)
            torch.cuda.synchronize()
            barrier(dist)
        ms = max_over_ranks(dist, t0.elapsed_time(t1), device) / steps
        del g
        per_s = 1e12 if unit == "TFLOP/s" else 1e9  # flops: FLOPs, or bytes for GB/s
        return {"value": world * flops / (ms * 1e-3) / per_s, "unit": unit, "ms_per_step": ms,
                "launch": "the step's kernels replayed from one CUDA graph", "clocks": clocks.summary()}
    except Exception as e:  # reported, not fatal: the eager measurement stands on its own
        return {"unavailable": f"{type(e).__name__}: {e}"[:200]}


def headline_from_graph(line, graph, launches, world, peak_tf):
    """Make the graph-replayed step the line's headline when it was measured:
    value, ms_per_step and clocks come from the replays, the eager loop's go
    under "eager"; the replays launch the same kernels per step as the eager
    loop, whose count the library took."""
    eager = {"value": line["value"], "ms_per_step": line["ms_per_step"], "clocks": line["clocks"],
             "launch": "one host launch per kernel"}
    if "value" not in graph:
        line["graph_replay"] = graph
        return
    line["value"], line["ms_per_step"], line["clocks"] = graph["value"], graph["ms_per_step"], graph["clocks"]
    line["config"]["launch"] = "CUDA graph replay of the whole step (its calls captured once)"
    line["gpu_launches"] = launches
    if peak_tf is not None:
        line["fwdbwd_frac_of_peak"] = graph["value"] / world / peak_tf
    line["eager"] = eager


def kernel_source_sha(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def cpu_oracle_sample(q, k, v, do, scale, causal, budget_s=12.0, max_heads=None):
    """Time the float64 oracle (forward + backward) head by head until
    ``budget_s`` has passed.  Returns (TFLOP/s, heads done, seconds)."""
    import oracle
    B, H, N, D = q.shape
    heads = [(b, h) for b in range(B) for h in range(H)][:max_heads]
    done, t0 = 0, time.perf_counter()
    for b, h in heads:
        qn, kn, vn, don = (x[b, h].double().numpy() for x in (q, k, v, do))
        oracle.forward_head(qn, kn, vn, scale, causal)
        oracle.backward_head(qn, kn, vn, don, scale, causal)
        done += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    flops = 3.5 * flops_fwd(1, done, N, D, causal)
    return flops / dt / 1e12, done, dt


def run_reference(args, rank):
    """The oracle as the reference arm, on the host cores: each step is the
    oracle's forward + backward on a bounded sample of the workload -- one
    (b, h) head (train and the other dense configurations), one (sequence,
    head) of the packed workload in turn, or, for the 32768-token window (whose
    n x n head would take 8.6 GB a matrix), 256 query rows of a head at the end
    of the sequence, forward and dQ rows, counted by the FLOPs they take."""
    if rank != 0:
        return
    from exact_io_aware_37_gb300 import synth
    import oracle
    wl = "train" if args.workload == "train" else args.workload
    if wl == "decode":
        print(json.dumps({"impl": "reference", "unavailable": "the reference arm times fwd+bwd workloads only"}))
        return
    name, causal = (WORKLOAD, CAUSAL) if wl == "train" else CONFIG_WORKLOADS[wl]
    cfg = synth.WORKLOADS[name]
    samples = []  # (q, k, v, do) of one sample as float64 arrays, and its FLOPs
    if "n_seqs" in cfg:
        q, k, v, do, cu, lengths = synth.make_varlen(cfg)
        D = q.shape[-1]
        for s, n in enumerate(lengths):
            if n > 0:
                a0, a1 = int(cu[s]), int(cu[s + 1])
                samples.append((tuple(x[s % q.shape[0], a0:a1].double().numpy() for x in (q, k, v, do)),
                                3.5 * flops_fwd(1, 1, int(n), D, causal)))
        shape = dict(H=q.shape[0], T=int(cu[-1]), D=D, n_seqs=len(lengths))
        sample = "one (sequence, head) of the packed workload per step, float64 numpy fwd+bwd"
        rows = None
    else:
        q, k, v, do = synth.make_dense(cfg)
        B, H, N, D = q.shape
        shape = dict(B=B, H=H, N=N, D=D)
        rows = np.arange(N - 256, N) if N > 8192 else None
        for b in range(B):
            for h in range(H):
                arrs = tuple(x[b, h].double().numpy() for x in (q, k, v, do))
                if rows is None:
                    samples.append((arrs, 3.5 * flops_fwd(1, 1, N, D, causal)))
                else:  # forward rows 4 D n_i + dQ rows 6 D n_i flops (scores recomputed)
                    keys = (rows + 1) if causal else np.full(len(rows), N)
                    samples.append((arrs, 10.0 * D * float(keys.sum())))
        sample = ("one (b,h) head per step, float64 numpy fwd+bwd" if rows is None else
                  "256 query rows at the end of one head per step: forward rows and dQ rows (float64 numpy), "
                  "counted by the FLOPs they take")
    scale = 1.0 / D ** 0.5

    def one(arrs):
        qn, kn, vn, don = arrs
        if rows is None:
            oracle.forward_head(qn, kn, vn, scale, causal)
            oracle.backward_head(qn, kn, vn, don, scale, causal)
        else:
            oracle.forward_rows(qn, kn, vn, rows, scale, causal)
            oracle.backward_dq_rows(qn, kn, vn, don, rows, scale, causal)

    for w in range(args.warmup):
        one(samples[w % len(samples)][0])
    times, flops = [], 0.0
    for s in range(args.steps):
        arrs, f = samples[s % len(samples)]
        t0 = time.perf_counter()
        one(arrs)
        times.append(time.perf_counter() - t0)
        flops += f
    total = sum(times)
    value = flops / total / 1e12
    cores = os.cpu_count()
    label = f"{name} {'causal' if causal else 'non-causal'}"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict({"workload": f"{label} (one sample per step)", "causal": causal}, **shape),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{sample}; {label}"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="train workload only: leave out the short measurements of the other configurations")
    ap.add_argument("--dtype", choices=["bf16", "f16"], default="bf16",
                    help="16-bit input type (the same synthetic draws, rounded to it)")
    ap.add_argument("--dropout", type=float, default=0.0,
                    help="attention dropout probability for the train workload (fa_fwd_dropout / fa_bwd_dropout)")
    ap.add_argument("--deterministic", action="store_true",
                    help="train workload with fa_bwd_deterministic (dQ without atomics)")
    ap.add_argument("--probe", choices=["ex2"], default=None,
                    help="ex2: measure the special-function units' ex2.approx rate and print, for the train "
                         "workload's kernels, the exponential-bound time beside the tensor-core-bound time")
    ap.add_argument("--workload", choices=["train", "decode"] + sorted(CONFIG_WORKLOADS), default="train",
                    help="train: causal fwd+bwd at B2 H32 N4096 D128 (the default, with the e2e and CPU legs); "
                         "decode: one cached decoding step, B16 H32, 1 query, 8192 keys, D128; "
                         "mid / long / long_nc / varlen / window: fwd+bwd of the other configurations "
                         "(device-resident inputs, kernel timings and roofline only)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    dist, rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank)
        barrier(dist)
        return

    import exact_io_aware_37_gb300 as fa
    from exact_io_aware_37_gb300 import synth

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if args.probe == "ex2":
        probe_ex2(fa, synth, local, device)
        return
    if args.workload == "decode":
        bench_decode(fa, synth, args, dist, rank, world, local, device)
        return
    if args.workload in CONFIG_WORKLOADS:
        bench_config(fa, synth, args, dist, rank, world, local, device)
        return
    cfg = dict(synth.WORKLOADS[WORKLOAD], dtype=args.dtype)
    q_h, k_h, v_h, do_h = synth.make_dense(cfg)
    B, H, N, D = q_h.shape
    scale = 1.0 / D ** 0.5
    q, k, v, do = (x.to(device) for x in (q_h, k_h, v_h, do_h))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.fa_bwd_workspace_size(q), dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    fwd_call, bwd_call = attention_calls(fa, args.dropout, deterministic=args.deterministic)

    def step():
        fwd_call(q, k, v, o, lse, scale, stream)
        bwd_call(q, k, v, o, lse, do, dq, dk, dv, scale, ws, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_error() == 0

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    for e in ev:  # create the events the library records around the main backward kernel
        e[3].record(stream)
        e[4].record(stream)
    torch.cuda.synchronize()
    launches0 = fa.fa_launch_count()
    with ClockSampler(local) as clocks:
        barrier(dist)
        torch.cuda.synchronize()
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for s in range(args.steps):
            ev[s][0].record(stream)
            fwd_call(q, k, v, o, lse, scale, stream)
            ev[s][1].record(stream)
            fa.fa_bwd_time_main_kernel(ev[s][3], ev[s][4])
            bwd_call(q, k, v, o, lse, do, dq, dk, dv, scale, ws, stream)
            ev[s][2].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
        barrier(dist)
    launches = fa.fa_launch_count() - launches0
    assert fa.fa_get_last_device_error() == 0
    total_ms = max_over_ranks(dist, t_start.elapsed_time(t_end), device)
    fwd_ms = [e[0].elapsed_time(e[1]) for e in ev]
    bwd_ms = [e[1].elapsed_time(e[2]) for e in ev]
    main_ms = [e[3].elapsed_time(e[4]) for e in ev]  # main backward kernel alone

    f_fwd = flops_fwd(B, H, N, D, CAUSAL)
    f_step = 3.5 * f_fwd
    ms_per_step = total_ms / args.steps
    value = world * f_step / (ms_per_step * 1e-3) / 1e12
    fwd_tflops = f_fwd / (statistics.mean(fwd_ms) * 1e-3) / 1e12
    bwd_tflops = 2.5 * f_fwd / (statistics.mean(bwd_ms) * 1e-3) / 1e12
    peak_tf, _, peak_kind = peaks()
    path = fa.fa_path_name(q.dtype, D)

    # dominant kernel: the main backward kernel (2.5x the forward FLOPs), timed
    # by events the library records right around it
    dom_ms = statistics.mean(main_ms)
    dom_name = "tc_bwd128_kernel<128>" if path == "tcgen05" else "simt backward kernels"
    if args.deterministic:
        dom_name = "tc_bwd128_kernel (dK, dV) + tc_bwd_dq_kernel (dQ)"
    src = os.path.join(ROOT, "exact_io_aware_37_gb300", "csrc",
                       "fa_tc_bwd128.cu" if path == "tcgen05" else "fa_simt.cu")
    # the ncu capture behind the table was of the bf16 run
    traffic = (TRAFFIC_BY_SOURCE.get(kernel_source_sha(src))
               if args.dtype == "bf16" and args.dropout == 0 and not args.deterministic else None)
    achieved = 2.5 * f_fwd / (dom_ms * 1e-3) / 1e12
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s",
                "frac": achieved / peak_tf, "traffic": traffic, "kernel": dom_name,
                "peak_kind": f"bf16 dense burst, {peak_kind}" + (
                    "" if args.dtype == "bf16" else "; fp16 has the same nominal dense rate")}

    line = {
        "metric": (METRIC if args.dtype == "bf16" else METRIC.replace("bf16", args.dtype))
                  + (f", attention dropout p={args.dropout:g}" if args.dropout > 0 else "")
                  + (", deterministic backward" if args.deterministic else ""), "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": args.dtype, "data": "synthetic",
        "config": {"workload": f"{WORKLOAD} causal", "B": B, "H": H, "N": N, "D": D, "causal": CAUSAL,
                   "kernel_path": path, "dropout": args.dropout, "deterministic_bwd": args.deterministic,
                   "l2": f"inputs {4 * q.numel() * 2 / 2**20:.0f} MiB > 129 MiB L2; no flush",
                   "parallelism": f"replicas x{world}"},
        "fwd_tflops": fwd_tflops, "bwd_tflops": bwd_tflops,
        "fwd_frac_of_peak": fwd_tflops / peak_tf, "fwdbwd_frac_of_peak": value / world / peak_tf,
        "ms_fwd": statistics.mean(fwd_ms), "ms_bwd": statistics.mean(bwd_ms), "ms_bwd_main_kernel": dom_ms,
        "roofline": roofline,
        "gpu_launches": launches,
        "clocks": clocks.summary(),
    }

    if not args.no_e2e:
        line["e2e"] = e2e_measure(fa, q_h, k_h, v_h, do_h, scale, device, stream, dist, world, args)
    graph = graph_replay_measure(
        lambda st: (fwd_call(q, k, v, o, lse, scale, st), bwd_call(q, k, v, o, lse, do, dq, dk, dv, scale, ws, st)),
        f_step, args.steps, args.warmup, device, dist, world, local)
    assert fa.fa_get_last_device_error() == 0
    headline_from_graph(line, graph, launches, world, peak_tf)

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tf, heads, secs = cpu_oracle_sample(q_h, k_h, v_h, do_h, scale, CAUSAL)
        line["cpu_baseline"] = {"value": tf, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                                "sample": f"{heads} of {B * H} (b,h) heads of {WORKLOAD} causal, float64 "
                                          f"numpy fwd+bwd, {secs:.1f} s"}
    if (not args.no_workloads and world == 1 and args.dtype == "bf16" and args.dropout == 0
            and not args.deterministic):
        # the other configurations, each fwd+bwd on device-resident inputs (a
        # short eager loop, then the step replayed from a CUDA graph), after
        # the headline's timed regions so their heat does not reach it
        wl_steps = max(10, min(args.steps, 30))
        summaries = {}
        for w in WORKLOADS_IN_DEFAULT_RUN:
            wl = config_line(fa, synth, args, w, wl_steps, dist, rank, world, local, device)
            if wl is not None:
                summaries[w] = workload_summary(wl)
        line["workloads"] = summaries
    if rank == 0:
        print(json.dumps(line), flush=True)
    barrier(dist)
    if dist is not None:
        dist.destroy_process_group()


def probe_ex2(fa, synth, local, device):
    """Measured ex2.approx rate (exponentials per clock per SM) and, for each
    tensor-core kernel of the train workload, the time its exponentials take
    at that rate beside the time its products take at the tensor core's
    nominal bf16 rate (8192 flop per clock per SM) and at the measured peak."""
    with ClockSampler(local) as clocks:
        rates = [fa.fa_probe_ex2_rate(iters=1 << 14) for _ in range(5)]
    rate = statistics.median(rates)
    cfg = synth.WORKLOADS[WORKLOAD]
    B, H, N, D = cfg["B"], cfg["H"], cfg["N"], cfg["D"]
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    mhz = 2070.0
    peak_tf, _, peak_kind = peaks()
    exps = B * H * N * N / (2 if CAUSAL else 1)   # one exponential per allowed score, each pass
    f_fwd = flops_fwd(B, H, N, D, CAUSAL)
    kernels = {}
    for name, flops in (("tc_fwd_kernel", f_fwd), ("tc_bwd128_kernel", 2.5 * f_fwd)):
        kernels[name] = {
            "exponentials": exps,
            "ex2_bound_us": 1e6 * exps / (rate * sms * mhz * 1e6),
            "tensor_bound_us_nominal": 1e6 * flops / (8192.0 * sms * mhz * 1e6),
            "tensor_bound_us_measured_peak": 1e6 * flops / (peak_tf * 1e12),
        }
    line = {"probe": "ex2.approx.f32 rate", "ex2_per_clk_per_sm": rate, "samples": rates, "sms": sms,
            "clock_mhz_for_times": mhz, "workload": f"{WORKLOAD} causal", "kernels": kernels,
            "peak_kind": f"bf16 dense burst, {peak_kind}", "clocks": clocks.summary()}
    print(json.dumps(line), flush=True)


# The other configurations: synth workload name and whether the mask is on.
# Carried by the default run's line under "workloads" (each a short measurement).
WORKLOADS_IN_DEFAULT_RUN = ("mid", "long_nc", "varlen", "window")
CONFIG_WORKLOADS = {
    "mid": ("mid_b4h16n1024d64", True),
    "long": ("long_b2h32n4096d128", True),
    "long_nc": ("long_b2h32n4096d128", False),
    "varlen": ("varlen16_h32d128", True),
    "window": ("window_b1h32n32768d128", True),
}


def bench_config(fa, synth, args, dist, rank, world, local, device):
    """Print the line of the configuration --workload names."""
    line = config_line(fa, synth, args, args.workload, args.steps, dist, rank, world, local, device)
    if line is not None:
        print(json.dumps(line), flush=True)


def workload_summary(line):
    """The figures of a configuration's line that the default run carries."""
    keep = ("value", "unit", "ms_per_step", "fwd_tflops", "bwd_tflops", "fwd_frac_of_peak", "fwdbwd_frac_of_peak",
            "ms_bwd_main_kernel", "steps")
    out = {k: line[k] for k in keep if k in line}
    out["workload"] = line["config"]["workload"]
    out["launch"] = line["config"].get("launch", "eager")
    out["eager_value"] = line.get("eager", {}).get("value", line["value"])
    out["roofline_frac"] = line["roofline"]["frac"]
    out["clocks"] = {k: line["clocks"].get(k) for k in ("sm_mhz", "sm_min_mhz", "reasons", "samples")}
    return out


def config_line(fa, synth, args, workload, steps, dist, rank, world, local, device):
    """fwd+bwd TFLOP/s of one configuration with inputs resident on the
    device: fa_fwd then fa_bwd per step, each timed with CUDA events on the
    launching stream, the main backward kernel timed alone by the events the
    library records around it, then the step replayed from a CUDA graph.
    Packed input counts sum_s 4 H n_s^2 D (half with the mask) forward FLOPs.
    Every rank measures; rank 0 gets the line, the others None."""
    name, causal = CONFIG_WORKLOADS[workload]
    cfg = dict(synth.WORKLOADS[name], dtype=args.dtype)
    cu = max_seqlen = None
    if "n_seqs" in cfg:
        q_h, k_h, v_h, do_h, cu_h, lengths = synth.make_varlen(cfg)
        H, T, D = q_h.shape
        f_fwd = sum(flops_fwd(1, H, int(n), D, causal) for n in lengths.tolist())
        cu, max_seqlen = cu_h.to(device), int(lengths.max())
        shape_cfg = {"H": H, "T": T, "D": D, "n_seqs": len(lengths), "max_seqlen": max_seqlen}
    else:
        q_h, k_h, v_h, do_h = synth.make_dense(cfg)
        B, H, N, D = q_h.shape
        f_fwd = flops_fwd(B, H, N, D, causal)
        shape_cfg = {"B": B, "H": H, "N": N, "D": D}
    scale = 1.0 / D ** 0.5
    q, k, v, do = (x.to(device) for x in (q_h, k_h, v_h, do_h))
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.fa_bwd_workspace_size(q, cu, max_seqlen), dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)

    def fwd_on(st):
        fa.fa_fwd(q, k, v, o, lse, causal, scale, cu, max_seqlen, stream=st)

    def bwd_on(st):
        fa.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, causal, scale, cu, max_seqlen, workspace=ws, stream=st)

    def fwd():
        fwd_on(stream)

    def bwd():
        bwd_on(stream)

    for _ in range(args.warmup):
        fwd()
        bwd()
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_error() == 0
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
    for e in ev:
        e[3].record(stream)
        e[4].record(stream)
    torch.cuda.synchronize()
    launches0 = fa.fa_launch_count()
    with ClockSampler(local) as clocks:
        barrier(dist)
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for st in range(steps):
            ev[st][0].record(stream)
            fwd()
            ev[st][1].record(stream)
            fa.fa_bwd_time_main_kernel(ev[st][3], ev[st][4])
            bwd()
            ev[st][2].record(stream)
        t1.record(stream)
        torch.cuda.synchronize()
        barrier(dist)
    launches = fa.fa_launch_count() - launches0
    assert fa.fa_get_last_device_error() == 0
    graph = graph_replay_measure(lambda st: (fwd_on(st), bwd_on(st)), 3.5 * f_fwd, steps,
                                 args.warmup, device, dist, world, local)
    assert fa.fa_get_last_device_error() == 0
    ms_step = max_over_ranks(dist, t0.elapsed_time(t1), device) / steps
    ms_fwd = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    ms_bwd = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    ms_main = statistics.mean(e[3].elapsed_time(e[4]) for e in ev)
    peak_tf, _, peak_kind = peaks()
    value = world * 3.5 * f_fwd / (ms_step * 1e-3) / 1e12
    bwd_main_tf = 2.5 * f_fwd / (ms_main * 1e-3) / 1e12
    kernel = f"tc_bwd128_kernel<{D}>"
    if rank != 0:
        return None
    line = {
        "metric": f"attention fwd & fwd+bwd TFLOP/s ({args.dtype}, {'causal' if causal else 'non-causal'}) "
                  "and % of GB300 BF16 tensor peak",
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": steps, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": args.dtype, "data": "synthetic",
        "config": dict({"workload": f"{name} {'causal' if causal else 'non-causal'}", "causal": causal,
                        "kernel_path": fa.fa_path_name(q.dtype, D),
                        "l2": f"inputs {4 * q.numel() * q.element_size() / 2**20:.0f} MiB; no flush",
                        "parallelism": f"replicas x{world}"}, **shape_cfg),
        "fwd_tflops": f_fwd / (ms_fwd * 1e-3) / 1e12, "bwd_tflops": 2.5 * f_fwd / (ms_bwd * 1e-3) / 1e12,
        "fwd_frac_of_peak": f_fwd / (ms_fwd * 1e-3) / 1e12 / peak_tf, "fwdbwd_frac_of_peak": value / world / peak_tf,
        "ms_fwd": ms_fwd, "ms_bwd": ms_bwd, "ms_bwd_main_kernel": ms_main,
        "roofline": {"bound": "tensor", "achieved": bwd_main_tf, "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": bwd_main_tf / peak_tf, "traffic": None, "kernel": kernel,
                     "peak_kind": f"bf16 dense burst, {peak_kind}"},
        "gpu_launches": launches, "clocks": clocks.summary(),
    }
    headline_from_graph(line, graph, launches, world, peak_tf)
    return line


DECODE_WORKLOAD = "decode_b16h32q1k8192d128"


def bench_decode(fa, synth, args, dist, rank, world, local, device):
    """One cached decoding step per timed iteration (fa_decode: split-KV pass +
    merge).  The cache (K, V: 2.1 GB, larger than L2) is resident; the metric
    is algorithmic HBM bytes (K, V, q, o, lse) per second, against the measured
    copy bandwidth."""
    cfg = dict(synth.WORKLOADS[DECODE_WORKLOAD], dtype=args.dtype)
    q_h, k_h, v_h = synth.make_decode(cfg)
    B, H, nq, D = q_h.shape
    nk = k_h.shape[2]
    scale = 1.0 / D ** 0.5
    q, k, v = (x.to(device) for x in (q_h, k_h, v_h))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, nq), dtype=torch.float32, device=device)
    ws_bytes = fa.fa_decode_workspace_size(q, k)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=device) if ws_bytes else None
    stream = torch.cuda.current_stream(device)
    for _ in range(args.warmup):
        fa.fa_decode(q, k, v, o, lse, True, scale, workspace=ws, stream=stream)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_error() == 0
    launches0 = fa.fa_launch_count()
    with ClockSampler(local) as clocks:
        barrier(dist)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.steps):
            fa.fa_decode(q, k, v, o, lse, True, scale, workspace=ws, stream=stream)
        b.record(stream)
        torch.cuda.synchronize()
        barrier(dist)
    launches = fa.fa_launch_count() - launches0
    assert fa.fa_get_last_device_error() == 0
    ms = max_over_ranks(dist, a.elapsed_time(b), device) / args.steps
    elem = q.element_size()
    step_bytes = (2 * B * H * nk * D + 2 * B * H * nq * D) * elem + B * H * nq * 4
    graph = graph_replay_measure(lambda st: fa.fa_decode(q, k, v, o, lse, True, scale, workspace=ws, stream=st),
                                 step_bytes, args.steps, args.warmup, device, dist, world, local, unit="GB/s")
    assert fa.fa_get_last_device_error() == 0
    gbs = world * step_bytes / (ms * 1e-3) / 1e9
    peak_gbs, peak_kind = hbm_peak()

    # end to end: the step's new query (and the new token's K / V rows, which a
    # caller appends to the cache) come from pinned host memory; o and lse go back
    hq = q_h.pin_memory()
    hkv = [x[:, :, -nq:].contiguous().pin_memory() for x in (k_h, v_h)]
    dkv = [torch.empty_like(x, device=device) for x in hkv]  # contiguous staging, then appended on the device
    ho, hl = torch.empty_like(q_h).pin_memory(), torch.empty((B, H, nq), dtype=torch.float32).pin_memory()
    steps = max(10, args.steps // 4)

    def e2e_step():
        q.copy_(hq, non_blocking=True)
        for hs, ds, cache in zip(hkv, dkv, (k, v)):
            ds.copy_(hs, non_blocking=True)
            cache[:, :, -nq:].copy_(ds)
        fa.fa_decode(q, k, v, o, lse, True, scale, workspace=ws, stream=stream)
        ho.copy_(o, non_blocking=True)
        hl.copy_(lse, non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    barrier(dist)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(steps):
        e2e_step()
    b.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(dist, a.elapsed_time(b), device) / steps
    h2d = (hq.numel() + hkv[0].numel() + hkv[1].numel()) * elem
    d2h = ho.numel() * elem + hl.numel() * 4
    if rank != 0:
        return
    line = {
        "metric": f"cached decoding step, algorithmic HBM GB/s ({args.dtype})", "value": gbs, "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": args.dtype,
        "data": "synthetic",
        "config": {"workload": DECODE_WORKLOAD, "B": B, "H": H, "nq": nq, "nk": nk, "D": D, "causal": True,
                   "kernel_path": "simt split-KV + merge" if ws_bytes else "simt split-KV (one split)",
                   "l2": f"K/V cache {2 * k.numel() * elem / 2**30:.1f} GiB > 129 MiB L2; no flush",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": gbs / world, "peak": peak_gbs, "unit": "GB/s",
                     "frac": gbs / world / peak_gbs, "kernel": "decode_split_kernel",
                     "traffic": TRAFFIC_BY_SOURCE.get(kernel_source_sha(
                         os.path.join(ROOT, "exact_io_aware_37_gb300", "csrc", "fa_decode.cu"))),
                     "peak_kind": peak_kind, "bytes_per_step": step_bytes},
        "gpu_launches": launches,
        "clocks": clocks.summary(),
        "e2e": {"value": world * step_bytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
    }
    headline_from_graph(line, graph, launches, world, None)
    print(json.dumps(line), flush=True)


def attention_calls(fa, p_drop, seed=20251203, deterministic=False):
    """(forward, backward) enqueue functions of the timed step; with dropout the
    same p, seed and offset in both."""
    if deterministic:
        fwd = (lambda q, k, v, o, lse, scale, st: fa.fa_fwd_dropout(q, k, v, o, lse, CAUSAL, p_drop, seed, 0, scale,
                                                                    stream=st))
        return (fwd, lambda q, k, v, o, lse, do, dq, dk, dv, scale, ws, st: fa.fa_bwd_deterministic(
            q, k, v, o, lse, do, dq, dk, dv, CAUSAL, scale, p_drop=p_drop, seed=seed, offset=0, workspace=ws,
            stream=st))
    if p_drop > 0:
        return (lambda q, k, v, o, lse, scale, st: fa.fa_fwd_dropout(q, k, v, o, lse, CAUSAL, p_drop, seed, 0, scale,
                                                                     stream=st),
                lambda q, k, v, o, lse, do, dq, dk, dv, scale, ws, st: fa.fa_bwd_dropout(
                    q, k, v, o, lse, do, dq, dk, dv, CAUSAL, p_drop, seed, 0, scale, workspace=ws, stream=st))
    return (lambda q, k, v, o, lse, scale, st: fa.fa_fwd(q, k, v, o, lse, CAUSAL, scale, stream=st),
            lambda q, k, v, o, lse, do, dq, dk, dv, scale, ws, st: fa.fa_bwd(
                q, k, v, o, lse, do, dq, dk, dv, CAUSAL, scale, workspace=ws, stream=st))


def e2e_measure(fa, q_h, k_h, v_h, do_h, scale, device, stream, dist, world, args):
    """Same metric through the public API with host buffers.  Every step copies
    its q, k, v, dO from pinned host memory, runs fa_fwd + fa_bwd and copies o,
    lse, dq, dk, dv back to pinned host memory, all inside the timed region.
    Steps are pipelined the way a host-fed caller would run them: two sets of
    device buffers, uploads on one stream, compute on another, downloads on a
    third, so step i+1's upload and step i-1's download overlap step i."""
    hin = [x.pin_memory() for x in (q_h, k_h, v_h, do_h)]
    B, H, N, D = q_h.shape
    nbuf = 2
    bufs = []
    for _ in range(nbuf):
        din = [torch.empty_like(x, device=device) for x in hin]
        o = torch.empty_like(din[0])
        lse = torch.empty((B, H, N), dtype=torch.float32, device=device)
        dq, dk, dv = (torch.empty_like(din[0]) for _ in range(3))
        ws = torch.empty(fa.fa_bwd_workspace_size(din[0]), dtype=torch.uint8, device=device)
        outs = [o, lse, dq, dk, dv]
        hout = [torch.empty_like(x, device="cpu").pin_memory() for x in outs]
        bufs.append((din, outs, ws, hout))
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev = lambda: torch.cuda.Event()
    in_ready = [ev() for _ in range(nbuf)]
    done = [ev() for _ in range(nbuf)]
    out_done = [ev() for _ in range(nbuf)]

    fwd_call, bwd_call = attention_calls(fa, args.dropout, deterministic=args.deterministic)

    def run(steps, start_ev=None, end_ev=None):
        if start_ev is not None:
            start_ev.record(s_in)
        for i in range(steps):
            b = i % nbuf
            din, outs, ws, hout = bufs[b]
            if i >= nbuf:
                s_in.wait_event(done[b])        # step i-2 has finished reading these inputs
            with torch.cuda.stream(s_in):
                for hsrc, ddst in zip(hin, din):
                    ddst.copy_(hsrc, non_blocking=True)
            in_ready[b].record(s_in)
            stream.wait_event(in_ready[b])
            if i >= nbuf:
                stream.wait_event(out_done[b])  # step i-2's results have been downloaded
            q, k, v, do = din
            o, lse, dq, dk, dv = outs
            fwd_call(q, k, v, o, lse, scale, stream)
            bwd_call(q, k, v, o, lse, do, dq, dk, dv, scale, ws, stream)
            done[b].record(stream)
            s_out.wait_event(done[b])
            with torch.cuda.stream(s_out):
                for dsrc, hdst in zip(outs, hout):
                    hdst.copy_(dsrc, non_blocking=True)
            out_done[b].record(s_out)
        if end_ev is not None:
            s_in.wait_stream(s_out)
            end_ev.record(s_in)

    run(4)
    torch.cuda.synchronize()
    steps = max(4, args.steps // 4)
    barrier(dist)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    run(steps, a, b)
    torch.cuda.synchronize()
    ms = max_over_ranks(dist, a.elapsed_time(b), device) / steps
    f_step = 3.5 * flops_fwd(B, H, N, D, CAUSAL)
    return {"value": world * f_step / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": sum(x.numel() * x.element_size() for x in hin),
            "d2h_bytes_per_step": sum(x.numel() * x.element_size() for x in bufs[0][3]),
            "ms_per_step": ms, "pipelined": "2 buffers; upload / compute / download streams"}


if __name__ == "__main__":
    main()
