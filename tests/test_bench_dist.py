"""bench.py on the CPU: the multi-process plumbing (gloo, world size 2) -- the
barrier and the max-over-ranks timing the replicas use, and the reference
arm doing its work on rank 0 only -- and how the graph-replayed step becomes
the headline, or, when it cannot be captured, leaves the eager one standing."""

import multiprocessing as mp
import os
import socket
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    dist, r, w, _ = bench.dist_setup(world)
    slowest = bench.max_over_ranks(dist, 10.0 * (rank + 1), torch.device("cpu"))
    bench.barrier(dist)

    class Args:
        steps, warmup, gpus = 1, 3, world
    if r != 0:
        bench.run_reference(Args, r)   # returns at once: only rank 0 times the oracle
    out.put((r, w, slowest))
    dist.destroy_process_group()


def test_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(rank, 2, port, out)) for rank in range(2)]
    for p in procs:
        p.start()
    results = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert results == [(0, 2, 20.0), (1, 2, 20.0)]


def test_reference_arm_prints_one_contract_line():
    """bench.py --impl reference times the oracle on the host and prints one JSON line
    carrying the metric, the oracle as its cpu_baseline and a copy-free e2e."""
    import json
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["warmup"] >= 3 and d["steps"] == 1 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_graph_replay_headline_and_fallback():
    """The graph-replayed step becomes the headline with the eager loop kept
    beside it; when the capture fails (here: no GPU) the eager line stands and
    says why."""
    sys.path.insert(0, ROOT)
    import bench
    eager_clocks = {"sm_mhz": 2070.0, "samples": 3}
    line = {"value": 100.0, "ms_per_step": 2.0, "clocks": eager_clocks, "config": {"workload": "w"},
            "gpu_launches": 8, "fwdbwd_frac_of_peak": 0.05}
    graph = {"value": 125.0, "unit": "TFLOP/s", "ms_per_step": 1.6, "launch": "graph",
             "clocks": {"sm_mhz": 2070.0, "samples": 9}}
    bench.headline_from_graph(line, graph, 8, 1, 2000.0)
    assert line["value"] == 125.0 and line["ms_per_step"] == 1.6 and line["clocks"]["samples"] == 9
    assert line["eager"]["value"] == 100.0 and line["eager"]["ms_per_step"] == 2.0
    assert line["eager"]["clocks"] is eager_clocks
    assert line["fwdbwd_frac_of_peak"] == 125.0 / 2000.0 and line["gpu_launches"] == 8
    assert "graph" in line["config"]["launch"].lower()

    failed = bench.graph_replay_measure(lambda st: None, 1e12, 2, 1, torch.device("cpu"), None, 1, 0)
    assert set(failed) == {"unavailable"}
    line2 = {"value": 100.0, "ms_per_step": 2.0, "clocks": eager_clocks, "config": {"workload": "w"}}
    bench.headline_from_graph(line2, failed, 8, 1, 2000.0)
    assert line2["value"] == 100.0 and "eager" not in line2 and line2["graph_replay"] == failed


def test_workload_summary_keeps_the_headline_figures():
    sys.path.insert(0, ROOT)
    import bench
    line = {"value": 385.0, "unit": "TFLOP/s", "ms_per_step": 0.078, "fwd_tflops": 320.0, "bwd_tflops": 318.0,
            "fwd_frac_of_peak": 0.17, "fwdbwd_frac_of_peak": 0.2, "ms_bwd_main_kernel": 0.05, "steps": 20,
            "config": {"workload": "mid_b4h16n1024d64 causal", "launch": "graph"},
            "eager": {"value": 315.0}, "roofline": {"frac": 0.22},
            "clocks": {"sm_mhz": 2070.0, "sm_min_mhz": 2002.0, "reasons": [], "samples": 4, "power_w_max": 1.0}}
    s = bench.workload_summary(line)
    assert s["value"] == 385.0 and s["eager_value"] == 315.0 and s["roofline_frac"] == 0.22
    assert s["workload"] == "mid_b4h16n1024d64 causal" and s["launch"] == "graph"
    assert s["clocks"] == {"sm_mhz": 2070.0, "sm_min_mhz": 2002.0, "reasons": [], "samples": 4}
    assert set(bench.WORKLOADS_IN_DEFAULT_RUN) <= set(bench.CONFIG_WORKLOADS)
