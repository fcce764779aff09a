"""Cached decoding (fa_decode) against the oracle: nq new queries against nk
cached keys, bottom-right causal alignment, split-KV merge."""

import numpy as np
import pytest
import torch

import exact_io_aware_37_gb300 as fa
import oracle
from exact_io_aware_37_gb300 import synth
from parity import TOL, f64

pytestmark = pytest.mark.gpu

CASES = [
    # (B, H, nq, nk, D, dtype, causal)
    (1, 2, 1, 1000, 128, torch.bfloat16, True),     # four key splits, merged
    (2, 3, 1, 1000, 128, torch.bfloat16, False),
    (1, 2, 3, 517, 64, torch.float16, True),
    (2, 2, 8, 300, 128, torch.bfloat16, True),      # one 8-row group
    (1, 3, 12, 777, 128, torch.bfloat16, True),     # two row groups, one of them ragged
    (1, 2, 5, 3, 64, torch.bfloat16, True),         # nq > nk: the first rows see no key
    (1, 2, 64, 64, 128, torch.bfloat16, True),      # square: the fa_fwd mask
    (1, 1, 4, 2049, 64, torch.float32, True),
    (1, 1, 2, 0, 128, torch.bfloat16, True),        # empty cache
]


def _run(q, k, v, causal, scale):
    dev = torch.device("cuda:0")
    qd, kd, vd = (x.to(dev) for x in (q, k, v))
    o = torch.full(q.shape, float("nan"), dtype=q.dtype, device=dev)
    lse = torch.full(q.shape[:-1], float("nan"), dtype=torch.float32, device=dev)
    fa.fa_decode(qd, kd, vd, o, lse, causal, scale)
    torch.cuda.synchronize()
    return f64(o), f64(lse)


def _inputs(B, H, nq, nk, D, dtype, seed):
    q = synth.normal((B, H, nq, D), synth.SEED_Q + seed, dtype)
    k = synth.normal((B, H, nk, D), synth.SEED_K + seed, dtype)
    v = synth.normal((B, H, nk, D), synth.SEED_V + seed, dtype)
    return q, k, v


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}q{}k{}D{}-{}-{}".format(
    *c[:5], str(c[5]).split(".")[-1], "causal" if c[6] else "full"))
def test_decode_matches_oracle(case):
    B, H, nq, nk, D, dtype, causal = case
    q, k, v = _inputs(B, H, nq, nk, D, dtype, 80)
    scale = D ** -0.5
    O, L = _run(q, k, v, causal, scale)
    Oref, Lref = oracle.forward_cached(*(x.double().numpy() for x in (q, k, v)), scale, causal)
    tol = TOL[dtype]
    assert np.isfinite(O).all()
    assert np.abs(O - Oref).max() <= tol["o_max"]
    finite = np.isfinite(Lref)
    assert np.array_equal(np.isfinite(L), finite)          # -inf exactly where no key is visible
    if finite.any():
        assert np.abs(L[finite] - Lref[finite]).max() <= tol["lse_max"]
    assert np.all(O[~finite] == 0.0)


def test_decode_square_case_equals_forward():
    """nq == nk: the bottom-right mask is fa_fwd's square causal mask."""
    q, k, v = _inputs(1, 2, 200, 200, 128, torch.bfloat16, 81)
    dev = torch.device("cuda:0")
    o1, l1 = fa.decode(*(x.to(dev) for x in (q, k, v)), causal=True)
    o2, l2 = fa.forward(*(x.to(dev) for x in (q, k, v)), causal=True)
    assert (o1.float() - o2.float()).abs().max().item() <= 2e-2
    assert (l1 - l2).abs().max().item() <= 1e-3


def test_decode_full_size_sampled_heads():
    """The decode bench shape (B16 H32, one new query, 8192 cached keys, D128):
    every row checked against the oracle on 6 sampled (b, h) heads."""
    B, H, nq, nk, D = 16, 32, 1, 8192, 128
    q, k, v = _inputs(B, H, nq, nk, D, torch.bfloat16, 82)
    O, L = _run(q, k, v, True, D ** -0.5)
    rng = np.random.default_rng(5)
    for b, h in zip(rng.integers(0, B, 6), rng.integers(0, H, 6)):
        Oref, Lref = oracle.forward_cached_head(*(x[b, h].double().numpy() for x in (q, k, v)), D ** -0.5, True)
        assert np.abs(O[b, h] - Oref).max() <= TOL[torch.bfloat16]["o_max"]
        assert np.abs(L[b, h] - Lref).max() <= TOL[torch.bfloat16]["lse_max"]
    assert np.isfinite(O).all() and np.isfinite(L).all()
