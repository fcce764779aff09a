"""Unit checks of the tensor-core building blocks on one 128-row tile, against
CPU matrix products (no attention arithmetic involved).

``fa_selftest_tile`` runs, on one CTA, the pieces every attention kernel here
is assembled from: TMA boxes of 64 columns x 128 rows landing in shared memory
in the 128-byte swizzled layout, S = A B^T from two K-major shared-memory
operands into tensor memory (the forward's S = Q K^T, the backward's
S^T = K Q^T), S read back with tcgen05.ld, rounded and stored to tensor memory
as packed pairs, and O = round(S) B with the left operand in tensor memory and
B read MN-major (the forward's P V, the backward's dV += P^T dO).

Bounds: bf16 and fp16 products are exact in float32, so S and O differ from
the float64 products only by the float32 accumulation of D (or 128) terms:
|error| <= n u sum_i |a_i b_i| with u = 2^-24 for sums taken with rounding.
The tensor core's summation order and internal rounding are not documented,
so the tests allow four times that.  A transposed operand, a wrong swizzle
phase or a misplaced descriptor step gives errors of the size of the entries
themselves.  The copy of A read back from shared memory must equal A bit for
bit."""

import pytest
import torch

import exact_io_aware_37_gb300 as fa

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


def _run(D, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    a = torch.randn(128, D, generator=g).to(dtype)
    b = torch.randn(128, D, generator=g).to(dtype)
    dev = torch.device("cuda")
    ad, bd = a.to(dev), b.to(dev)
    s = torch.full((128, 128), float("nan"), device=dev)
    o = torch.full((128, D), float("nan"), device=dev)
    ac = torch.zeros(128, D, dtype=dtype, device=dev)
    st = fa.fa_selftest_tile(ad, bd, s, o, ac)
    assert st == 0, fa.lib().fa_strerror(st)
    return a, b, s.cpu(), o.cpu(), ac.cpu()


@pytest.mark.parametrize("seed", [0, 1])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "f16"])
@pytest.mark.parametrize("D", [64, 128])
def test_tile_products_and_swizzled_copy(D, dtype, seed):
    a, b, s, o, ac = _run(D, dtype, seed)

    # TMA box round trip through the swizzled shared-memory tile
    assert torch.equal(ac.view(torch.int16), a.view(torch.int16))

    # S = A B^T (both operands K-major)
    a64, b64 = a.double(), b.double()
    s_ref = a64 @ b64.T
    s_bound = 4 * D * U * (a64.abs() @ b64.abs().T)
    err_s = (s.double() - s_ref).abs()
    assert torch.isfinite(s).all()
    assert (err_s <= s_bound).all(), f"max |dS| {err_s.max():.3e}, worst ratio {(err_s / s_bound).max():.2f}"

    # O = round(S) B: the left operand is the kernel's own S rounded to the
    # 16-bit type (round to nearest even on both sides), B read MN-major
    p64 = s.to(dtype).double()
    o_ref = p64 @ b64
    o_bound = 4 * 128 * U * (p64.abs() @ b64.abs())
    err_o = (o.double() - o_ref).abs()
    assert torch.isfinite(o).all()
    assert (err_o <= o_bound).all(), f"max |dO| {err_o.max():.3e}, worst ratio {(err_o / o_bound).max():.2f}"


def test_tile_structured_operands():
    """Operands whose products are exact small integers: A = row index pattern,
    B a permutation matrix scaled by 2, so S and O are known exactly and any
    transposition, row or column shift in the path shows up as a wrong entry."""
    D = 128
    r = torch.arange(128)
    a = ((r[:, None] * 3 + r[None, :D] * 5) % 17 - 8).to(torch.bfloat16)   # small integers, exact in bf16
    perm = torch.randperm(128, generator=torch.Generator().manual_seed(7))
    b = torch.zeros(128, D)
    b[r, perm[:D]] = 2.0
    b = b.to(torch.bfloat16)
    dev = torch.device("cuda")
    s = torch.full((128, 128), float("nan"), device=dev)
    o = torch.full((128, D), float("nan"), device=dev)
    ac = torch.zeros(128, D, dtype=torch.bfloat16, device=dev)
    assert fa.fa_selftest_tile(a.to(dev), b.to(dev), s, o, ac) == 0
    s_ref = a.double() @ b.double().T
    assert torch.equal(s.cpu().double(), s_ref)
    o_ref = s_ref.to(torch.bfloat16).double() @ b.double()
    assert torch.equal(o.cpu().double(), o_ref)
    assert torch.equal(ac.cpu().view(torch.int16), a.view(torch.int16))
