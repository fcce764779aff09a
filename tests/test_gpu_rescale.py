"""The running-state merge on the GPU where the row maximum rises in a later
key tile (tensortonic.com "FlashAttention", section 4: a larger maximum can
turn up after earlier tiles were folded in; section 5: the running sums are
then rescaled by exp(m_old - m_new)).

The tensor-core forward rescales lazily (its accumulator in tensor memory is
multiplied only when a tile's maximum exceeds the row's reference by more
than 2^8), so these inputs (``rising_max``) force that branch: after the first
key tile, in query tile 0 and 1 of a pair, in the middle of the key range, in
the last (ragged) tile and on the causal diagonal, dense and packed, D = 64
and 128, bf16 and fp16, with dropout and with the deterministic backward.
Companion cases rise just below the threshold (weights up to ~2^7.3 formed
against the old reference and rounded to 16 bits).  Every output is compared
element by element with the float64 oracle at the stated bounds: O, L and dV
with the exact oracle; dQ and dK with the oracle evaluated with the
backward's own D_i = rowsum(dO o O) over the output as stored (the oracle's O
rounded to the dtype), because these inputs magnify that rounding in dQ and
dK far beyond what i.i.d. inputs do (for the split-tile example times 10 the
exact-D gradient differs from the stored-O one by 265 % in dQ).  The CPU test
test_rising_max_inputs shows that each case takes the branch it is meant to
take.

The split-tile example the page prints (one query, scores 1, 2 in one tile
and 3, 4 in the next) also runs on the GPU: through the tensor-core kernels
(128-key tiles), the float32 kernels and the cached-decoding split-KV merge,
against the closed forms of tests/golden/split_tile_softmax.txt, once as
printed and once with the scores times 10, where the maximum rises by 20
natural units between the tiles and the lazy rescale fires."""

import math

import numpy as np
import pytest
import torch

import exact_io_aware_37_gb300 as fa
import oracle
import rising_max as rm
from oracle_pins import load_split_tile_example
from parity import Guarded, TOL, compare, default_scale, f64, run

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
DTYPES = [torch.bfloat16, torch.float16]
DT_IDS = ["bf16", "f16"]


def _stored(O, dtype):
    """The oracle's output as the GPU stores it: rounded to nearest in dtype."""
    return torch.from_numpy(O).to(dtype).double().numpy()


def _dense_ref(q, k, v, do, scale, causal):
    """O, L, dV exact; dQ, dK with D from the stored output."""
    qn, kn, vn, don = (x.double().numpy() for x in (q, k, v, do))
    O, L = oracle.forward(qn, kn, vn, scale, causal)
    dQ, dK, dV, _ = oracle.backward(qn, kn, vn, don, scale, causal, o_stored=_stored(O, q.dtype))
    return dict(o=O, lse=L, dq=dQ, dk=dK, dv=dV)


@pytest.mark.parametrize("dtype", DTYPES, ids=DT_IDS)
@pytest.mark.parametrize("case", rm.DENSE_CASES, ids=rm.case_id)
def test_dense_rising_max(case, dtype):
    profile, step, rows, sigma_k, shape, causal, _ = case
    scale = default_scale(shape[-1])
    q, k, v, do = rm.dense(shape, dtype, scale, profile, step, rows, sigma_k, seed_offset=200)
    got = run(q, k, v, do, causal, scale)
    compare(dtype, {n: f64(t) for n, t in got.items()}, _dense_ref(q, k, v, do, scale, causal),
            f"rising max {rm.case_id(case)} {dtype}")


@pytest.mark.parametrize("dtype", DTYPES, ids=DT_IDS)
@pytest.mark.parametrize("case", rm.PACKED_CASES, ids=rm.case_id)
def test_packed_rising_max(case, dtype):
    profile, step, rows, sigma_k, H, D, causal, _ = case
    scale = default_scale(D)
    q, k, v, do, cu = rm.packed(rm.PACKED_LENGTHS, H, D, dtype, scale, profile, step, rows, sigma_k,
                                seed_offset=210)
    got = run(q, k, v, do, causal, scale, cu=cu, max_seqlen=max(rm.PACKED_LENGTHS))
    qn, kn, vn, don = (x.double().numpy() for x in (q, k, v, do))
    O, L = oracle.forward_varlen(qn, kn, vn, cu, scale, causal)
    dQ, dK, dV, _ = oracle.backward_varlen(qn, kn, vn, don, cu, scale, causal, o_stored=_stored(O, dtype))
    compare(dtype, {n: f64(t) for n, t in got.items()}, dict(o=O, lse=L, dq=dQ, dk=dK, dv=dV),
            f"packed rising max {rm.case_id(case)} {dtype}")


def _run_dropout(q, k, v, do, causal, scale, p, seed, offset, cu=None, max_seqlen=None):
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


DROPOUT_CASES = [
    # (profile, step, rows, sigma_k, shape, causal, dtype, p)
    ("ramp", rm.STEP_UP, "mixed", 1.0, (1, 2, 600, 128), True, torch.bfloat16, 0.2),
    ("jump", rm.STEP_UP, "even_tiles", 1.0, (1, 2, 600, 64), False, torch.float16, 0.3),
    ("jump", rm.NEAR_BELOW, "mixed", rm.QUIET_K, (1, 2, 600, 128), False, torch.bfloat16, 0.1),
]


@pytest.mark.parametrize("case", DROPOUT_CASES, ids=lambda c: rm.case_id(c[:-1]) + f"-p{c[-1]}")
def test_dropout_rising_max(case):
    profile, step, rows, sigma_k, shape, causal, dtype, p = case
    scale = default_scale(shape[-1])
    seed, offset = 0xC0FFEE, 5
    q, k, v, do = rm.dense(shape, dtype, scale, profile, step, rows, sigma_k, seed_offset=220)
    got = _run_dropout(q, k, v, do, causal, scale, p, seed, offset)
    pf = float(np.float32(p))
    qn, kn, vn, don = (x.double().numpy() for x in (q, k, v, do))
    O, L = oracle.forward_dropout(qn, kn, vn, scale, causal, pf, seed, offset)
    dQ, dK, dV, _ = oracle.backward_dropout(qn, kn, vn, don, scale, causal, pf, seed, offset,
                                            o_stored=_stored(O, dtype))
    compare(dtype, got, dict(o=O, lse=L, dq=dQ, dk=dK, dv=dV), f"dropout rising max {case}",
            o_scale=1.0 / (1.0 - pf))


def test_packed_dropout_rising_max():
    D, H, p, seed, offset = 128, 2, 0.15, 4242, 9
    scale = default_scale(D)
    q, k, v, do, cu = rm.packed(rm.PACKED_LENGTHS, H, D, torch.bfloat16, scale, "ramp", rm.STEP_UP,
                                seed_offset=230)
    got = _run_dropout(q, k, v, do, True, scale, p, seed, offset, cu=cu, max_seqlen=max(rm.PACKED_LENGTHS))
    pf = float(np.float32(p))
    qn, kn, vn, don = (x.double().numpy() for x in (q, k, v, do))
    T = qn.shape[1]
    ref = {n: np.zeros((H, T, D)) for n in ("o", "dq", "dk", "dv")}
    ref["lse"] = np.zeros((H, T))
    # positions count from each sequence's start and bh is (sequence index) * H + head
    for s_, (a, b) in enumerate(zip(cu[:-1].tolist(), cu[1:].tolist())):
        if b == a:
            continue
        for h in range(H):
            keep = oracle.dropout_keep(b - a, b - a, s_ * H + h, pf, seed, offset)
            sl = (h, slice(a, b))
            ref["o"][sl], ref["lse"][sl] = oracle.forward_head_dropout(qn[sl], kn[sl], vn[sl], scale, True, pf, keep)
            ref["dq"][sl], ref["dk"][sl], ref["dv"][sl], _ = oracle.backward_head_dropout(
                qn[sl], kn[sl], vn[sl], don[sl], scale, True, pf, keep, o_stored=_stored(ref["o"][sl], torch.bfloat16))
    compare(torch.bfloat16, got, ref, "packed dropout rising max", o_scale=1.0 / (1.0 - pf))


@pytest.mark.parametrize("case", [
    ("ramp", rm.STEP_UP, "mixed", 1.0, (1, 2, 600, 128), True, torch.bfloat16),
    ("ramp", rm.STEP_UP, "mixed", 1.0, (1, 2, 600, 64), False, torch.float16),
], ids=lambda c: rm.case_id(c[:-1]) + "-" + str(c[-1]).split(".")[-1])
def test_deterministic_backward_rising_max(case):
    profile, step, rows, sigma_k, shape, causal, dtype = case
    scale = default_scale(shape[-1])
    q, k, v, do = rm.dense(shape, dtype, scale, profile, step, rows, sigma_k, seed_offset=240)
    qd, kd, vd, dod = (x.to(DEV) for x in (q, k, v, do))
    o, lse = fa.forward(qd, kd, vd, causal=causal, scale=scale)
    g = [torch.full_like(qd, float("nan")) for _ in range(3)]
    fa.fa_bwd_deterministic(qd, kd, vd, o, lse, dod, *g, causal, scale)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_error() == 0
    got = dict(o=f64(o), lse=f64(lse), dq=f64(g[0]), dk=f64(g[1]), dv=f64(g[2]))
    compare(dtype, got, _dense_ref(q, k, v, do, scale, causal), f"deterministic rising max {case}")


@pytest.mark.parametrize("dtype", DTYPES, ids=DT_IDS)
@pytest.mark.parametrize("causal", [False, True])
def test_decode_rising_max(causal, dtype):
    """Cached decoding: the cache's levels rise every 128 keys; 4 new rows
    against 1000 keys run as four key splits whose states are merged."""
    B, H, nq, nk, D = 1, 2, 4, 1000, 128
    scale = default_scale(D)
    q, k, v = rm.cached(B, H, nq, nk, D, dtype, scale, "ramp", rm.STEP_UP, seed_offset=250)
    o = torch.full(q.shape, float("nan"), dtype=dtype, device=DEV)
    lse = torch.full(q.shape[:-1], float("nan"), dtype=torch.float32, device=DEV)
    fa.fa_decode(q.to(DEV), k.to(DEV), v.to(DEV), o, lse, causal, scale)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_error() == 0
    O, L = oracle.forward_cached(*(x.double().numpy() for x in (q, k, v)), scale, causal)
    tol = TOL[dtype]
    assert np.abs(f64(o) - O).max() <= tol["o_max"]
    assert np.abs(f64(lse) - L).max() <= tol["lse_max"]


# ------------------------------------------------------------------ split-tile example

def _split_tile_closed_form(mult):
    scores, tiles = load_split_tile_example()
    assert scores == [1.0, 2.0, 3.0, 4.0] and tiles == [(0, 2), (2, 4)]
    s = [mult * x for x in scores]
    top = max(s)
    e = [math.exp(x - top) for x in s]
    return [x / sum(e) for x in e], top + math.log(sum(e))


FILL = -1000.0  # score of every other key: exp(-1000 - max) is 0 in float32 and float64 alike


def _split_tile_inputs(mult, N, key_pos, D, dtype, seed=260):
    """One head whose every query has the dot products ``mult * [1, 2, 3, 4]``
    with the keys at ``key_pos`` and FILL with all others (scale 1); the value
    rows of those four keys are one-hot on columns 0..3."""
    q = torch.zeros((1, 1, N, D))
    q[..., 0] = 1.0
    k = torch.zeros((1, 1, N, D))
    k[..., 0] = FILL
    v = torch.randn((1, 1, N, D), generator=torch.Generator().manual_seed(seed))
    for c, j in enumerate(key_pos):
        k[0, 0, j, 0] = mult * (c + 1)
        v[0, 0, j] = 0.0
        v[0, 0, j, c] = 1.0
    do = torch.randn((1, 1, N, D), generator=torch.Generator().manual_seed(seed + 1))
    return tuple(x.to(dtype) for x in (q, k, v, do))


def _check_split_tile(o, lse, mult, o_rtol, what):
    """O against the closed-form weights (relative), L to float32 precision
    (32 units of 2^-24 relative to |L|: the scores, their maximum and the log
    of the sum are float32 values of that size)."""
    w, L = _split_tile_closed_form(mult)
    lse_atol = 32 * 2.0 ** -24 * abs(L)
    o, lse = f64(o).reshape(-1, o.shape[-1]), f64(lse).reshape(-1)
    for c in range(4):
        np.testing.assert_allclose(o[:, c], w[c], rtol=o_rtol, atol=0, err_msg=f"{what}: weight {c}")
    assert (o[:, 4:] == 0).all(), f"{what}: weight on a FILL key"
    np.testing.assert_allclose(lse, L, rtol=0, atol=lse_atol, err_msg=f"{what}: L")


@pytest.mark.parametrize("mult", [1.0, 10.0])
def test_split_tile_example_tensor_cores(mult):
    """Keys 0, 1 lie in the first 128-key tile and keys 128, 129 in the second
    (a ragged tile of 2 keys): the merge across tiles of the tensor-core
    forward.  mult = 10 makes the maximum rise by 20 > 5.5 natural units
    between the tiles, so the lazy rescale of the accumulator runs.  O carries
    two bf16 roundings (the weights before P V, the output), L none."""
    N, D = 130, 64
    q, k, v, do = _split_tile_inputs(mult, N, [0, 1, 128, 129], D, torch.bfloat16)
    got = run(q, k, v, do, False, 1.0)
    _check_split_tile(got["o"], got["lse"], mult, o_rtol=2.0 ** -7, what=f"tcgen05 x{mult}")
    compare(torch.bfloat16, {n: f64(t) for n, t in got.items()}, _dense_ref(q, k, v, do, 1.0, False),
            f"split tile x{mult}")


@pytest.mark.parametrize("mult", [1.0, 10.0])
def test_split_tile_example_float32(mult):
    """The same example through the float32 kernels (32-key tiles: the scores
    sit in tiles 0 and 4): to float32 precision."""
    N, D = 130, 64
    q, k, v, do = _split_tile_inputs(mult, N, [0, 1, 128, 129], D, torch.float32)
    got = run(q, k, v, do, False, 1.0, backward=False)
    _check_split_tile(got["o"], got["lse"], mult, o_rtol=1e-5, what=f"f32 x{mult}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("mult", [1.0, 10.0])
def test_split_tile_example_decode_merge(mult, dtype):
    """One new query against a 512-key cache runs as two key splits of 256
    (keys 0, 1 in the first, 256, 257 in the second); the merge kernel folds
    the two running states together by the rescaling rule.  The weights stay
    in float32, so O carries one rounding to its dtype."""
    nk, D = 512, 64
    q, k, v, _ = _split_tile_inputs(mult, nk, [0, 1, 256, 257], D, dtype)
    qn = q[:, :, -1:].contiguous()
    assert fa.fa_decode_workspace_size(qn, k) > 0  # two splits, merged
    o = torch.full(qn.shape, float("nan"), dtype=dtype, device=DEV)
    lse = torch.full(qn.shape[:-1], float("nan"), dtype=torch.float32, device=DEV)
    fa.fa_decode(qn.to(DEV), k.to(DEV), v.to(DEV), o, lse, False, 1.0)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_error() == 0
    rtol = 2.0 ** -8 if dtype == torch.bfloat16 else 1e-5
    _check_split_tile(o, lse, mult, o_rtol=rtol, what=f"decode {dtype} x{mult}")
