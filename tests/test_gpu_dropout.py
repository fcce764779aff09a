"""Attention dropout on the GPU against the oracle: the regenerated keep mask
exactly (forward and backward orientation), and outputs / gradients within the
dtype's bounds."""

import numpy as np
import pytest
import torch

import exact_io_aware_37_gb300 as fa
import oracle
from exact_io_aware_37_gb300 import synth
from parity import Guarded, TOL, compare, default_scale, f64

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _p32(p):
    """The probability as the library sees it (a float)."""
    return float(np.float32(p))


def _fwd_bwd(q, k, v, do, causal, scale, p, seed, offset, cu=None, max_seqlen=None):
    qd, kd, vd, dod = (x.to(DEV) for x in (q, k, v, do))
    cud = None if cu is None else cu.to(DEV)
    o = Guarded(q.shape, q.dtype, DEV)
    lse = Guarded(q.shape[:-1], torch.float32, DEV)
    fa.fa_fwd_dropout(qd, kd, vd, o.t, lse.t, causal, p, seed, offset, scale, cud, max_seqlen)
    g = {n: Guarded(q.shape, q.dtype, DEV) for n in ("dq", "dk", "dv")}
    fa.fa_bwd_dropout(qd, kd, vd, o.t, lse.t, dod, g["dq"].t, g["dk"].t, g["dv"].t, causal, p, seed, offset, scale,
                      cud, max_seqlen)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_error() == 0
    for name, x in [("o", o), ("lse", lse)] + list(g.items()):
        assert x.guards_intact(), f"{name}: write outside the output tensor"
    return dict(o=f64(o.t), lse=f64(lse.t), **{n: f64(x.t) for n, x in g.items()})


@pytest.mark.parametrize("D", [64, 128])
def test_forward_mask_is_exact(D):
    """q = 0 makes every weight 1/N; with V one-hot on keys 256 .. 256+D-1 the
    output element (i, d) is nonzero exactly when weight (i, 256 + d) was kept."""
    B, H, N, p, seed, off = 2, 3, 512, 0.3, 0x1234_5678_9ABC, 11
    q = torch.zeros((B, H, N, D), dtype=torch.bfloat16)
    k = synth.normal((B, H, N, D), 1, torch.bfloat16)
    v = torch.zeros((B, H, N, D), dtype=torch.bfloat16)
    v[:, :, 256:256 + D] = torch.eye(D, dtype=torch.bfloat16)
    o = torch.empty((B, H, N, D), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=DEV)
    fa.fa_fwd_dropout(q.to(DEV), k.to(DEV), v.to(DEV), o, lse, False, p, seed, off)
    got = o.float().cpu().numpy() != 0
    for b in range(B):
        for h in range(H):
            keep = oracle.dropout_keep(N, N, b * H + h, _p32(p), seed, off)
            assert np.array_equal(got[b, h], keep[:, 256:256 + D]), (b, h)


@pytest.mark.parametrize("D", [64, 128])
def test_backward_mask_is_exact(D):
    """dV = (P o M)^T dO: with q = 0 and dO one-hot on rows 128 .. 128+D-1,
    dV element (j, d) is nonzero exactly when weight (128 + d, j) was kept --
    the backward regenerates the mask with keys on lanes."""
    B, H, N, p, seed, off = 1, 2, 384, 0.45, 987654321, 3
    q = torch.zeros((B, H, N, D), dtype=torch.bfloat16)
    k = synth.normal((B, H, N, D), 1, torch.bfloat16)
    v = synth.normal((B, H, N, D), 2, torch.bfloat16)
    do = torch.zeros((B, H, N, D), dtype=torch.bfloat16)
    do[:, :, 128:128 + D] = torch.eye(D, dtype=torch.bfloat16)
    got = _fwd_bwd(q, k, v, do, False, default_scale(D), p, seed, off)
    for h in range(H):
        keep = oracle.dropout_keep(N, N, h, _p32(p), seed, off)
        assert np.array_equal(got["dv"][0, h] != 0, keep[128:128 + D, :].T), h


CASES = [
    # (B, H, N, D, dtype, p)
    (2, 2, 300, 64, torch.bfloat16, 0.1),
    (1, 2, 384, 128, torch.bfloat16, 0.25),
    (2, 3, 129, 128, torch.float16, 0.5),
    (1, 1, 513, 128, torch.bfloat16, 0.7),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}N{}D{}-{}-p{}".format(
    *c[:4], str(c[4]).split(".")[-1], c[5]))
def test_dropout_matches_oracle(case, causal):
    B, H, N, D, dtype, p = case
    q, k, v, do = synth.qkv_do((B, H, N, D), dtype, seed_offset=90)
    scale, seed, off = default_scale(D), 20251203 + N, 5
    got = _fwd_bwd(q, k, v, do, causal, scale, p, seed, off)
    qn, kn, vn, don = (x.double().numpy() for x in (q, k, v, do))
    O, L = oracle.forward_dropout(qn, kn, vn, scale, causal, _p32(p), seed, off)
    dQ, dK, dV, _ = oracle.backward_dropout(qn, kn, vn, don, scale, causal, _p32(p), seed, off)
    # kept weights are magnified by 1 / (1 - p), and so are the absolute rounding
    # errors of P~ and O: the O bound scales with them
    compare(dtype, got, dict(o=O, lse=L, dq=dQ, dk=dK, dv=dV), f"dropout {case} causal={causal}",
            o_scale=1.0 / (1.0 - p))


def test_dropout_packed_sequences():
    """Packed sequences: positions count from each sequence's start and bh is
    (sequence index) * H + head."""
    lengths = [1, 200, 0, 129, 300]
    cu = synth.cu_seqlens(lengths)
    T, H, D, p, seed, off = int(cu[-1]), 2, 128, 0.2, 77, 9
    q, k, v, do = synth.qkv_do((H, T, D), torch.bfloat16, seed_offset=91)
    scale = default_scale(D)
    got = _fwd_bwd(q, k, v, do, True, scale, p, seed, off, cu=cu, max_seqlen=max(lengths))
    qn, kn, vn, don = (x.double().numpy() for x in (q, k, v, do))
    ref = {n: np.zeros((H, T, D)) for n in ("o", "dq", "dk", "dv")}
    ref["lse"] = np.zeros((H, T))
    for s, (a, b) in enumerate(zip(cu[:-1].tolist(), cu[1:].tolist())):
        if b == a:
            continue
        for h in range(H):
            keep = oracle.dropout_keep(b - a, b - a, s * H + h, _p32(p), seed, off)
            sl = (h, slice(a, b))
            ref["o"][sl], ref["lse"][sl] = oracle.forward_head_dropout(qn[sl], kn[sl], vn[sl], scale, True, _p32(p),
                                                                       keep)
            ref["dq"][sl], ref["dk"][sl], ref["dv"][sl], _ = oracle.backward_head_dropout(
                qn[sl], kn[sl], vn[sl], don[sl], scale, True, _p32(p), keep)
    compare(torch.bfloat16, got, ref, "dropout packed", o_scale=1.0 / (1.0 - p))


def test_zero_probability_is_plain_attention():
    q, k, v, do = synth.qkv_do((1, 2, 300, 128), torch.bfloat16, seed_offset=92)
    got = _fwd_bwd(q, k, v, do, True, 0.1, 0.0, 1, 0)
    qd, kd, vd, dod = (x.to(DEV) for x in (q, k, v, do))
    o, lse = fa.forward(qd, kd, vd, causal=True, scale=0.1)
    dq, dk, dv = fa.backward(qd, kd, vd, o, lse, dod, causal=True, scale=0.1)
    assert np.array_equal(got["o"], f64(o)) and np.array_equal(got["lse"], f64(lse))
    for n, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        assert np.abs(got[n] - f64(t)).max() <= 1e-2   # dQ's float32 accumulation order is not fixed


@pytest.mark.parametrize("D", [64, 128])
def test_dropout_beyond_the_table(D):
    """More items than the host-built table holds (the forward's closed-form list
    of 4608 query-tile pairs, the backward's queue of 9216 key tiles): every
    role derives a tile's head from the list, and the decisions regenerated from
    that head must still be the oracle's.  Sampled heads against the oracle."""
    B, H, N, p, seed, off = 8, 64, 2300, 0.1, 4242, 3
    q, k, v, do = synth.qkv_do((B, H, N, D), torch.bfloat16, seed_offset=310)
    scale = default_scale(D)
    qd, kd, vd, dod = (x.to(DEV) for x in (q, k, v, do))
    o, lse = torch.empty_like(qd), torch.empty((B, H, N), dtype=torch.float32, device=DEV)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(qd), torch.empty_like(qd)
    fa.fa_fwd_dropout(qd, kd, vd, o, lse, True, p, seed, off, scale)
    fa.fa_bwd_dropout(qd, kd, vd, o, lse, dod, dq, dk, dv, True, p, seed, off, scale)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_error() == 0
    got = dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv)
    g = np.random.default_rng(13)
    for idx in sorted(g.choice(B * H, size=3, replace=False).tolist()):
        b, h = divmod(idx, H)
        qn, kn, vn, don = (x[b, h].double().numpy() for x in (q, k, v, do))
        keep = oracle.dropout_keep(N, N, b * H + h, _p32(p), seed, off)
        O, L = oracle.forward_head_dropout(qn, kn, vn, scale, True, _p32(p), keep)
        dQ, dK, dV, _ = oracle.backward_head_dropout(qn, kn, vn, don, scale, True, _p32(p), keep)
        compare(torch.bfloat16, {n: f64(t[b, h]) for n, t in got.items()}, dict(o=O, lse=L, dq=dQ, dk=dK, dv=dV),
                f"dropout beyond the table D={D} head {(b, h)}", o_scale=1.0 / (1.0 - p))
