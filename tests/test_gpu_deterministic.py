"""The deterministic backward (fa_bwd_deterministic): the same gradients as the
oracle within the dtype's bounds, and bit-identical across repeated calls."""

import numpy as np
import pytest
import torch

import exact_io_aware_37_gb300 as fa
import oracle
from exact_io_aware_37_gb300 import synth
from parity import Guarded, compare, default_scale, f64

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _run(q, k, v, do, causal, scale, cu=None, max_seqlen=None, p=0.0, seed=0, offset=0):
    qd, kd, vd, dod = (x.to(DEV) for x in (q, k, v, do))
    cud = None if cu is None else cu.to(DEV)
    o = torch.empty_like(qd)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=DEV)
    if p > 0:
        fa.fa_fwd_dropout(qd, kd, vd, o, lse, causal, p, seed, offset, scale, cud, max_seqlen)
    else:
        fa.fa_fwd(qd, kd, vd, o, lse, causal, scale, cud, max_seqlen)
    g = {n: Guarded(q.shape, q.dtype, DEV) for n in ("dq", "dk", "dv")}
    fa.fa_bwd_deterministic(qd, kd, vd, o, lse, dod, g["dq"].t, g["dk"].t, g["dv"].t, causal, scale, cud, max_seqlen,
                            p_drop=p, seed=seed, offset=offset)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_error() == 0
    for n, x in g.items():
        assert x.guards_intact(), f"{n}: write outside the output tensor"
    return dict(o=f64(o), lse=f64(lse), **{n: f64(x.t) for n, x in g.items()})


CASES = [
    # (B, H, N, D, dtype)
    (2, 3, 17, 64, torch.bfloat16),
    (2, 2, 300, 64, torch.bfloat16),
    (1, 2, 384, 128, torch.bfloat16),
    (1, 1, 513, 128, torch.float16),
    (3, 6, 256, 128, torch.bfloat16),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}N{}D{}-{}".format(*c[:4], str(c[4]).split(".")[-1]))
def test_deterministic_matches_oracle(case, causal):
    B, H, N, D, dtype = case
    q, k, v, do = synth.qkv_do((B, H, N, D), dtype, seed_offset=100)
    scale = default_scale(D)
    got = _run(q, k, v, do, causal, scale)
    qn, kn, vn, don = (x.double().numpy() for x in (q, k, v, do))
    O, L = oracle.forward(qn, kn, vn, scale, causal)
    dQ, dK, dV, _ = oracle.backward(qn, kn, vn, don, scale, causal)
    compare(dtype, got, dict(o=O, lse=L, dq=dQ, dk=dK, dv=dV), f"deterministic {case} causal={causal}")


def test_deterministic_many_key_tiles():
    """Causal N = 1024 (eight query tiles, each visiting up to eight key tiles)."""
    q, k, v, do = synth.qkv_do((2, 4, 1024, 128), torch.bfloat16, seed_offset=101)
    got = _run(q, k, v, do, True, default_scale(128))
    qn, kn, vn, don = (x.double().numpy() for x in (q, k, v, do))
    O, L = oracle.forward(qn, kn, vn, default_scale(128), True)
    dQ, dK, dV, _ = oracle.backward(qn, kn, vn, don, default_scale(128), True)
    compare(torch.bfloat16, got, dict(o=O, lse=L, dq=dQ, dk=dK, dv=dV), "deterministic N=1024")


@pytest.mark.parametrize("causal", [False, True])
def test_deterministic_packed(causal):
    lengths = [1, 127, 128, 129, 300, 0, 5, 256]
    cu = synth.cu_seqlens(lengths)
    T = int(cu[-1])
    q, k, v, do = synth.qkv_do((2, T, 128), torch.bfloat16, seed_offset=102)
    scale = default_scale(128)
    got = _run(q, k, v, do, causal, scale, cu=cu, max_seqlen=max(lengths))
    qn, kn, vn, don = (x.double().numpy() for x in (q, k, v, do))
    O, L = oracle.forward_varlen(qn, kn, vn, cu, scale, causal)
    dQ, dK, dV, _ = oracle.backward_varlen(qn, kn, vn, don, cu, scale, causal)
    compare(torch.bfloat16, got, dict(o=O, lse=L, dq=dQ, dk=dK, dv=dV), f"deterministic packed causal={causal}")


@pytest.mark.parametrize("D", [64, 128])
def test_deterministic_with_dropout(D):
    q, k, v, do = synth.qkv_do((2, 2, 300, D), torch.bfloat16, seed_offset=103)
    p, seed, off = 0.3, 424242, 1
    scale = default_scale(D)
    got = _run(q, k, v, do, True, scale, p=p, seed=seed, offset=off)
    pf = float(np.float32(p))
    qn, kn, vn, don = (x.double().numpy() for x in (q, k, v, do))
    O, L = oracle.forward_dropout(qn, kn, vn, scale, True, pf, seed, off)
    dQ, dK, dV, _ = oracle.backward_dropout(qn, kn, vn, don, scale, True, pf, seed, off)
    compare(torch.bfloat16, got, dict(o=O, lse=L, dq=dQ, dk=dK, dv=dV), f"deterministic dropout D={D}",
            o_scale=1.0 / (1.0 - p))


def test_repeated_calls_are_bit_identical():
    q, k, v, do = synth.qkv_do((2, 8, 1024, 128), torch.bfloat16, seed_offset=104)
    a = _run(q, k, v, do, True, default_scale(128))
    for _ in range(3):
        b = _run(q, k, v, do, True, default_scale(128))
        for n in ("dq", "dk", "dv"):
            assert np.array_equal(a[n], b[n]), n


def test_deterministic_beyond_the_table():
    """Dense input with more key tiles (9216) than the host-built table holds:
    the dK / dV kernel takes them from the workspace queue.  Sampled heads
    against the oracle, and a second call bit-identical to the first."""
    B, H, N, D = 8, 64, 2300, 128
    q, k, v, do = synth.qkv_do((B, H, N, D), torch.bfloat16, seed_offset=320)
    scale = default_scale(D)
    qd, kd, vd, dod = (x.to(DEV) for x in (q, k, v, do))
    o, lse = torch.empty_like(qd), torch.empty((B, H, N), dtype=torch.float32, device=DEV)
    fa.fa_fwd(qd, kd, vd, o, lse, True, scale)
    runs = []
    for _ in range(2):
        dq, dk, dv = torch.empty_like(qd), torch.empty_like(qd), torch.empty_like(qd)
        fa.fa_bwd_deterministic(qd, kd, vd, o, lse, dod, dq, dk, dv, True, scale)
        torch.cuda.synchronize()
        assert fa.fa_get_last_device_error() == 0
        runs.append((dq, dk, dv))
    for a, b in zip(*runs):
        assert torch.equal(a, b), "repeated deterministic backward differs"
    dq, dk, dv = runs[0]
    got = dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv)
    g = np.random.default_rng(17)
    for idx in sorted(g.choice(B * H, size=3, replace=False).tolist()):
        b, h = divmod(idx, H)
        qn, kn, vn, don = (x[b, h].double().numpy() for x in (q, k, v, do))
        O, L = oracle.forward_head(qn, kn, vn, scale, True)
        dQ, dK, dV, _ = oracle.backward_head(qn, kn, vn, don, scale, True)
        compare(torch.bfloat16, {n: f64(t[b, h]) for n, t in got.items()}, dict(o=O, lse=L, dq=dQ, dk=dK, dv=dV),
                f"deterministic beyond the table head {(b, h)}")
