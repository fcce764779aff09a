"""The float64 oracle against what the pages and the mathematics fix (CPU only)."""

import math

import numpy as np
import pytest
import torch

import oracle
import oracle_pins
from exact_io_aware_37_gb300 import synth


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_pin(check):
    check(oracle)


def _sdpa(q, k, v, scale, causal):
    t = [torch.tensor(np.asarray(x, dtype=np.float64)) for x in (q, k, v)]
    return torch.nn.functional.scaled_dot_product_attention(*t, is_causal=causal, scale=scale).numpy()


@pytest.mark.parametrize("causal", [False, True])
def test_batched_layout_matches_library(causal):
    """[B, H, N, D] layout (tensortonic.com "FlashAttention" section 9) handled
    head by head: compared with torch SDPA over the 4-D tensors."""
    q, k, v, do = synth.qkv_do((2, 3, 17, 8), torch.float32)
    O, L = oracle.forward(q.numpy(), k.numpy(), v.numpy(), 0.25, causal)
    np.testing.assert_allclose(O, _sdpa(q, k, v, 0.25, causal), atol=1e-12)
    assert L.shape == (2, 3, 17)
    dQ, dK, dV, D = oracle.backward(q.numpy(), k.numpy(), v.numpy(), do.numpy(), 0.25, causal)
    t = [x.double().requires_grad_() for x in (q, k, v)]
    out = torch.nn.functional.scaled_dot_product_attention(*t, is_causal=causal, scale=0.25)
    out.backward(do.double())
    for mine, ref in ((dQ, t[0].grad), (dK, t[1].grad), (dV, t[2].grad)):
        np.testing.assert_allclose(mine, ref.numpy(), atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_is_per_sequence(causal):
    """Packed sequences attend only within themselves (nexusofnerds.com
    "FlashAttention": variable-length packing): each segment equals torch
    SDPA on that segment alone, and changing one sequence leaves the others
    untouched.  Includes a length-1 and a length-0 sequence."""
    lengths = [5, 1, 0, 9, 3]
    cu = synth.cu_seqlens(lengths)
    T = int(cu[-1])
    q, k, v, do = (x.numpy().astype(np.float64) for x in synth.qkv_do((2, T, 4), torch.float32))
    O, L = oracle.forward_varlen(q, k, v, cu, 0.5, causal)
    dQ, dK, dV, _ = oracle.backward_varlen(q, k, v, do, cu, 0.5, causal)
    for s in range(len(lengths)):
        a, b = int(cu[s]), int(cu[s + 1])
        if a == b:
            continue
        np.testing.assert_allclose(O[:, a:b], _sdpa(q[:, a:b], k[:, a:b], v[:, a:b], 0.5, causal), atol=1e-12)
    k2, v2 = k.copy(), v.copy()
    k2[:, int(cu[3]):int(cu[4])] += 5.0
    v2[:, int(cu[3]):int(cu[4])] -= 3.0
    O2, _ = oracle.forward_varlen(q, k2, v2, cu, 0.5, causal)
    keep = np.r_[0:int(cu[3]), int(cu[4]):T]
    np.testing.assert_allclose(O2[:, keep], O[:, keep], atol=0)
    # gradient sums per sequence (same invariants as the dense case)
    for s in range(len(lengths)):
        a, b = int(cu[s]), int(cu[s + 1])
        if a == b:
            continue
        np.testing.assert_allclose(dK[:, a:b].sum(1), 0.0, atol=1e-12)
        np.testing.assert_allclose(dV[:, a:b].sum(1), do[:, a:b].sum(1), atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_row_subset_and_blocked_forms(causal):
    r = np.random.default_rng(3)
    n, d = 300, 16
    q, k, v, do = r.standard_normal((4, n, d))
    O, L = oracle.forward_head(q, k, v, 0.25, causal)
    dQ, dK, dV, _ = oracle.backward_head(q, k, v, do, 0.25, causal)
    rows = [0, 1, 127, 128, 129, 299]
    Or, Lr = oracle.forward_rows(q, k, v, rows, 0.25, causal)
    np.testing.assert_allclose(Or, O[rows], atol=1e-13)
    np.testing.assert_allclose(Lr, L[rows], atol=1e-13)
    np.testing.assert_allclose(oracle.backward_dq_rows(q, k, v, do, rows, 0.25, causal), dQ[rows], atol=1e-13)
    Ob, Lb, dQb, dKb, dVb = oracle.backward_head_blocked(q, k, v, do, 0.25, causal, rows_per_block=64)
    for a, b in ((Ob, O), (Lb, L), (dQb, dQ), (dKb, dK), (dVb, dV)):
        np.testing.assert_allclose(a, b, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("br,bc", [(1, 1), (2, 3), (7, 5), (16, 16), (128, 128), (64, 32)])
def test_tiled_schedule_is_exact(causal, br, bc):
    """The query-first tiled schedule with running state and causal block
    skipping (tensortonic.com "FlashAttention" sections 5-6) reproduces the
    full-matrix definition (section 8: exact, up to rounding order)."""
    r = np.random.default_rng(4)
    n, d = 130, 8
    q, k, v = r.standard_normal((3, n, d)) * 2
    O, L = oracle.forward_head(q, k, v, 0.35, causal)
    Ot, Lt = oracle.tiled_forward_head(q, k, v, 0.35, causal, br, bc)
    np.testing.assert_allclose(Ot, O, atol=1e-12)
    np.testing.assert_allclose(Lt, L, atol=1e-12)


def test_memory_arithmetic_on_the_pages():
    """Sizes the pages print for the score matrix the method avoids:
    4096^2 fp32 entries = 64 MB per head, 2 GB for 32 heads
    (wiki.ai-engineering.at "Flash Attention", The Core Problem);
    fp16 entries: 32 MiB at 4096 tokens and 128 MiB at 8192
    (tensortonic.com "FlashAttention", section 2)."""
    assert 4096 * 4096 == 16_777_216
    assert 4096 * 4096 * 4 == 64 * 2 ** 20
    assert 32 * 4096 * 4096 * 4 == 2 * 2 ** 30
    assert 4096 * 4096 * 2 == 32 * 2 ** 20
    assert 8192 * 8192 * 2 == 128 * 2 ** 20
    assert math.isclose(2 ** 20, 1_048_576)
