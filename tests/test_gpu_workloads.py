"""The four bf16 workloads at full size, through the same calls the bench
times.  The oracle checks sampled heads in full and sampled query rows of
every head; properties that hold at any size (gradient sums, finiteness,
guard bands) are checked on every head."""

import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_37_gb300 import synth
from parity import TOL, compare, default_scale, f64, rel_frob, run

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _sample(n, k, seed):
    g = np.random.default_rng(seed)
    return sorted(g.choice(n, size=min(k, n), replace=False).tolist())


def _invariants(got, do, causal_unused=None):
    """Per head: sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i (rows of P sum to
    one; rows of dS sum to zero).  Tokens are on axis -2."""
    dk = got["dk"].float()
    dv = got["dv"].float()
    dod = do.to(dk.device).float()
    sk = dk.sum(-2)
    scale_k = dk.abs().sum(-2).clamp_min(1e-6)
    assert (sk.abs() / scale_k).max().item() < 2e-2, "sum_j dK_j != 0"
    sv = dv.sum(-2) - dod.sum(-2)
    scale_v = dod.abs().sum(-2).clamp_min(1e-6)
    assert (sv.abs() / scale_v).max().item() < 2e-2, "sum_j dV_j != sum_i dO_i"


def _check_dense(name, full_heads, rows_per_head, causal):
    cfg = synth.WORKLOADS[name]
    q, k, v, do = synth.make_dense(cfg)
    B, H, N, D = q.shape
    scale = default_scale(D)
    got = run(q, k, v, do, causal, scale)
    for t in got.values():
        assert torch.isfinite(t).all()
    _invariants(got, do)
    # full oracle on sampled (b, h) heads
    heads = [(b, h) for b in range(B) for h in range(H)]
    for idx in _sample(len(heads), full_heads, 7):
        b, h = heads[idx]
        qn, kn, vn, don = (x[b, h].double().numpy() for x in (q, k, v, do))
        if N <= 4096:
            O, L = oracle.forward_head(qn, kn, vn, scale, causal)
            dQ, dK, dV, _ = oracle.backward_head(qn, kn, vn, don, scale, causal)
        else:
            O, L, dQ, dK, dV = oracle.backward_head_blocked(qn, kn, vn, don, scale, causal)
        compare(torch.bfloat16, {n: f64(t[b, h]) for n, t in got.items()},
                dict(o=O, lse=L, dq=dQ, dk=dK, dv=dV), f"{name} head {(b, h)}")
    # sampled rows of every head: O, L and dQ need only their own row
    tol = TOL[torch.bfloat16]
    for b in range(B):
        for h in range(H):
            rows = _sample(N, rows_per_head, 1000 + b * H + h)
            qn, kn, vn, don = (x[b, h].double().numpy() for x in (q, k, v, do))
            O, L = oracle.forward_rows(qn, kn, vn, rows, scale, causal)
            assert np.abs(f64(got["o"][b, h, rows]) - O).max() <= tol["o_max"]
            assert np.abs(f64(got["lse"][b, h, rows]) - L).max() <= tol["lse_max"]
            dQ = oracle.backward_dq_rows(qn, kn, vn, don, rows, scale, causal)
            assert rel_frob(f64(got["dq"][b, h, rows]), dQ) <= tol["grad_rel"]


def test_mid_b4h16n1024d64_causal():
    _check_dense("mid_b4h16n1024d64", full_heads=64, rows_per_head=8, causal=True)


@pytest.mark.parametrize("causal", [False, True])
def test_long_b2h32n4096d128(causal):
    _check_dense("long_b2h32n4096d128", full_heads=3, rows_per_head=16, causal=causal)


def test_window_b1h32n32768d128_causal():
    _check_dense("window_b1h32n32768d128", full_heads=1, rows_per_head=8, causal=True)


def test_window_memory_is_linear():
    """N = 32768: device memory in use during the call stays at the inputs,
    outputs and workspace (O(N D) per head); an N x N score buffer for one
    head alone would be 2 GiB in bf16."""
    import exact_io_aware_37_gb300 as fa
    cfg = synth.WORKLOADS["window_b1h32n32768d128"]
    dev = torch.device("cuda:0")
    q, k, v, do = (x.to(dev) for x in synth.make_dense(cfg))
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    base = torch.cuda.memory_allocated()
    o, lse = fa.forward(q, k, v, causal=True)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    peak = torch.cuda.max_memory_allocated() - base
    tensor = q.numel() * q.element_size()
    ws = fa.fa_bwd_workspace_size(q)
    expected = 4 * tensor + lse.numel() * 4 + ws      # o, dq, dk, dv + lse + workspace
    assert peak <= expected * 1.05 + (64 << 20), (peak, expected)
    assert peak < 32 * 32768 * 32768 * 2 / 8        # far below even 1/8 of the score matrices


def test_varlen16_h32d128_causal():
    cfg = synth.WORKLOADS["varlen16_h32d128"]
    q, k, v, do, cu, lengths = synth.make_varlen(cfg)
    H, T, D = q.shape
    scale = default_scale(D)
    got = run(q, k, v, do, True, scale, cu=cu, max_seqlen=int(lengths.max()))
    for t in got.values():
        assert torch.isfinite(t).all()
    # gradient sums per sequence and head
    for s in range(len(lengths)):
        a, b = int(cu[s]), int(cu[s + 1])
        _invariants({n: t[:, a:b] for n, t in got.items()}, do[:, a:b])
    heads = _sample(H, 2, 9)
    qn, kn, vn, don = (x[heads].double().numpy() for x in (q, k, v, do))
    O, L = oracle.forward_varlen(qn, kn, vn, cu, scale, True)
    dQ, dK, dV, _ = oracle.backward_varlen(qn, kn, vn, don, cu, scale, True)
    compare(torch.bfloat16, {n: f64(t[heads]) for n, t in got.items()},
            dict(o=O, lse=L, dq=dQ, dk=dK, dv=dV), "varlen sampled heads")


def test_beyond_32_bit_element_offsets():
    """B1 H72 N262144 D128 causal bf16: 2.4e9 elements (4.8 GB) per tensor and a
    9.7 GB float32 dQ accumulator, so element and byte offsets pass 2^31 and
    2^32; the forward walks its closed-form list (73,728 query-tile pairs) and
    the backward its queue (147,456 key tiles).  Every head: finite outputs and
    the gradient sums; sampled rows, among them the last rows of the last head
    (the largest offsets), against the oracle."""
    import exact_io_aware_37_gb300 as fa
    B, H, N, D = 1, 72, 262144, 128
    assert B * H * N * D > 2 ** 31
    dev = torch.device("cuda:0")
    q, k, v, do = (synth.normal_device((B, H, N, D), 500 + s, torch.bfloat16, dev, std=0.5) for s in range(4))
    scale = default_scale(D)
    o, lse = fa.forward(q, k, v, causal=True)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_error() == 0
    for h in range(H):
        got = dict(o=o[:, h], lse=lse[:, h], dq=dq[:, h], dk=dk[:, h], dv=dv[:, h])
        for t in got.values():
            assert torch.isfinite(t).all(), f"head {h}"
        _invariants(got, do[:, h])
    tol = TOL[torch.bfloat16]
    for h in (0, 35, H - 1):
        rows = sorted(set([0, 1, 127, 128, N // 2, N - 129, N - 2, N - 1] + _sample(N, 4, 2000 + h)))
        qn, kn, vn, don = (x[0, h].double().cpu().numpy() for x in (q, k, v, do))
        O, L = oracle.forward_rows(qn, kn, vn, rows, scale, True)
        assert np.abs(f64(o[0, h, rows]) - O).max() <= tol["o_max"], f"O head {h}"
        assert np.abs(f64(lse[0, h, rows]) - L).max() <= tol["lse_max"], f"L head {h}"
        dQ = oracle.backward_dq_rows(qn, kn, vn, don, rows, scale, True)
        assert rel_frob(f64(dq[0, h, rows]), dQ) <= tol["grad_rel"], f"dQ head {h}"
