"""GPU path vs the float64 oracle, element by element, at sizes the oracle
finishes in seconds: several 128-row tiles, ragged tails, single rows,
packed sequences of awkward lengths, both masks."""

import numpy as np
import pytest
import torch

import exact_io_aware_37_gb300 as fa
import oracle
from exact_io_aware_37_gb300 import synth
from parity import compare, default_scale, f64, run

pytestmark = pytest.mark.gpu


def _dense_ref(q, k, v, do, scale, causal):
    qn, kn, vn, don = (x.double().numpy() for x in (q, k, v, do))
    O, L = oracle.forward(qn, kn, vn, scale, causal)
    dQ, dK, dV, _ = oracle.backward(qn, kn, vn, don, scale, causal)
    return dict(o=O, lse=L, dq=dQ, dk=dK, dv=dV)


DENSE_CASES = [
    # (B, H, N, D)
    (1, 1, 1, 64),
    (2, 3, 17, 64),
    (1, 2, 128, 64),
    (2, 2, 129, 128),
    (1, 2, 256, 128),
    (2, 2, 300, 64),
    (1, 1, 513, 128),
    (1, 2, 640, 64),
    # many (b, h) pairs: the causal block order cuts them into several head groups,
    # the last one short
    (3, 6, 384, 128),
    (5, 7, 300, 64),
    (6, 3, 520, 128),
    # many heads of one ragged tile each: 2048 and 256 tiny items in the host table
    (64, 32, 40, 64),
    (16, 16, 96, 128),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", DENSE_CASES, ids=lambda s: "x".join(map(str, s)))
def test_dense_bf16(shape, causal):
    q, k, v, do = synth.qkv_do(shape, torch.bfloat16, seed_offset=10)
    scale = default_scale(shape[-1])
    got = run(q, k, v, do, causal, scale)
    ref = _dense_ref(q, k, v, do, scale, causal)
    compare(torch.bfloat16, {n: f64(t) for n, t in got.items()}, ref, f"dense {shape} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_tiny_f32_workload(causal):
    """B=1 H=1 N=128 D=64 float32, scale 1/8: max|dO| <= 1e-4."""
    cfg = synth.WORKLOADS["tiny_f32"]
    q, k, v, do = synth.make_dense(cfg)
    got = run(q, k, v, do, causal, cfg["scale"])
    ref = _dense_ref(q, k, v, do, cfg["scale"], causal)
    compare(torch.float32, {n: f64(t) for n, t in got.items()}, ref, f"tiny f32 causal={causal}")


F16_CASES = [(2, 3, 17, 64), (2, 2, 300, 64), (1, 2, 256, 128), (1, 1, 513, 128), (3, 6, 384, 128)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", F16_CASES, ids=lambda s: "x".join(map(str, s)))
def test_dense_f16(shape, causal):
    q, k, v, do = synth.qkv_do(shape, torch.float16, seed_offset=10)
    scale = default_scale(shape[-1])
    got = run(q, k, v, do, causal, scale)
    ref = _dense_ref(q, k, v, do, scale, causal)
    compare(torch.float16, {n: f64(t) for n, t in got.items()}, ref, f"f16 dense {shape} causal={causal}")


@pytest.mark.parametrize("D", [32, 128])
def test_f32_other_widths(D):
    q, k, v, do = synth.qkv_do((1, 2, 200, D), torch.float32, seed_offset=20)
    scale = default_scale(D)
    got = run(q, k, v, do, True, scale)
    ref = _dense_ref(q, k, v, do, scale, True)
    compare(torch.float32, {n: f64(t) for n, t in got.items()}, ref, f"f32 D={D}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "f16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [64, 128])
def test_packed_16bit(D, causal, dtype):
    lengths = [1, 127, 128, 129, 300, 0, 5, 256]
    cu = synth.cu_seqlens(lengths)
    T = int(cu[-1])
    q, k, v, do = synth.qkv_do((2, T, D), dtype, seed_offset=30)
    scale = default_scale(D)
    got = run(q, k, v, do, causal, scale, cu=cu, max_seqlen=max(lengths))
    qn, kn, vn, don = (x.double().numpy() for x in (q, k, v, do))
    O, L = oracle.forward_varlen(qn, kn, vn, cu, scale, causal)
    dQ, dK, dV, _ = oracle.backward_varlen(qn, kn, vn, don, cu, scale, causal)
    compare(dtype, {n: f64(t) for n, t in got.items()}, dict(o=O, lse=L, dq=dQ, dk=dK, dv=dV),
            f"packed {dtype} D={D} causal={causal}")


@pytest.mark.parametrize("D", [64, 128])
def test_many_short_packed_sequences(D):
    """200 packed sequences of 0-150 tokens: hundreds of (sequence, head) units
    in the forward's closed-form list and the backward's queue, many of them
    empty or one ragged tile, ranks a sequence lacks skipped."""
    g = torch.Generator().manual_seed(4242 + D)
    lengths = torch.randint(0, 151, (200,), generator=g).tolist()
    lengths[:3] = [0, 1, 150]
    cu = synth.cu_seqlens(lengths)
    q, k, v, do = synth.qkv_do((4, int(cu[-1]), D), torch.bfloat16, seed_offset=40)
    scale = default_scale(D)
    got = run(q, k, v, do, True, scale, cu=cu, max_seqlen=max(lengths))
    qn, kn, vn, don = (x.double().numpy() for x in (q, k, v, do))
    O, L = oracle.forward_varlen(qn, kn, vn, cu, scale, True)
    dQ, dK, dV, _ = oracle.backward_varlen(qn, kn, vn, don, cu, scale, True)
    compare(torch.bfloat16, {n: f64(t) for n, t in got.items()}, dict(o=O, lse=L, dq=dQ, dk=dK, dv=dV),
            f"200 short packed sequences D={D}")


def test_causal_rows_ignore_future_keys():
    """Changing keys/values after row i leaves causal rows <= i unchanged
    (bit-identical: the kernel never reads them for those rows)."""
    q, k, v, do = synth.qkv_do((1, 2, 384, 128), torch.bfloat16, seed_offset=40)
    a = run(q, k, v, do, True, 0.1, backward=False)
    k2, v2 = k.clone(), v.clone()
    k2[:, :, 200:] = -k2[:, :, 200:] * 3
    v2[:, :, 200:] = v2[:, :, 200:] + 7
    b = run(q, k2, v2, do, True, 0.1, backward=False)
    assert torch.equal(a["o"][:, :, :200], b["o"][:, :, :200])
    assert torch.equal(a["lse"][:, :, :200], b["lse"][:, :, :200])
    assert not torch.equal(a["o"][:, :, 200:], b["o"][:, :, 200:])


def test_first_causal_row_is_v0():
    """Row 0 attends only to key 0: O_0 = V_0 and L_0 = scale * q_0 . k_0."""
    q, k, v, do = synth.qkv_do((2, 2, 130, 64), torch.bfloat16, seed_offset=50)
    got = run(q, k, v, do, True, 0.125, backward=False)
    np.testing.assert_allclose(f64(got["o"][:, :, 0]), v[:, :, 0].double().numpy(), atol=0)
    s00 = 0.125 * (q[:, :, 0].double() * k[:, :, 0].double()).sum(-1)
    np.testing.assert_allclose(f64(got["lse"][:, :, 0]), s00.numpy(), atol=1e-4)


def test_zero_query_closed_form():
    """Q = 0: causal O_i = mean(V[:i+1]) and L_i = log(i+1)."""
    _, k, v, do = synth.qkv_do((1, 1, 300, 128), torch.bfloat16, seed_offset=60)
    q = torch.zeros_like(k)
    got = run(q, k, v, do, True, 0.09, backward=False)
    vn = v[0, 0].double().numpy()
    mean = np.cumsum(vn, 0) / np.arange(1, 301)[:, None]
    assert np.abs(f64(got["o"][0, 0]) - mean).max() < 2e-2
    assert np.abs(f64(got["lse"][0, 0]) - np.log(np.arange(1, 301))).max() < 1e-4


def test_bad_seqlens_are_reported_not_faulted():
    """A sequence longer than max_seqlen is skipped on the device and latched
    as FA_ERR_INVALID; the well-formed sequences are still computed."""
    lengths = [100, 300, 50]
    cu = synth.cu_seqlens(lengths)
    q, k, v, do = synth.qkv_do((1, 450, 64), torch.bfloat16, seed_offset=70)
    dev = torch.device("cuda:0")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((1, 450), float("nan"), device=dev)
    fa.fa_fwd(qd, kd, vd, o, lse, True, 0.125, cu.to(dev), max_seqlen=200)   # 300 > 200
    assert fa.fa_get_last_device_error() == -1
    assert fa.fa_get_last_device_error() == 0        # cleared by the read
    O, L = oracle.forward_varlen(*(x.double().numpy() for x in (q, k, v)), cu, 0.125, True)
    for a, b in ((0, 100), (400, 450)):
        assert np.abs(f64(o[:, a:b]) - O[:, a:b]).max() < 2e-2
    assert torch.isnan(o[:, 100:400]).all()           # skipped, untouched


def test_bounded_wait_reports_timeout():
    """A kernel waiting on a barrier nothing signals gives up after the wait
    limit, latches FA_ERR_TIMEOUT and returns; the context stays usable."""
    fa.fa_set_wait_limit_ns(2_000_000)
    try:
        assert fa.fa_selftest_wait_timeout() == -5
    finally:
        fa.fa_set_wait_limit_ns(2_000_000_000)
    assert fa.fa_get_last_device_error() == 0
    q, k, v, do = synth.qkv_do((1, 1, 64, 64), torch.bfloat16)
    run(q, k, v, do, True, 0.125)


def test_empty_inputs():
    dev = torch.device("cuda:0")
    for shape in ((0, 2, 64, 64), (1, 0, 64, 128), (1, 2, 0, 64)):
        q = torch.zeros(shape, dtype=torch.bfloat16, device=dev)
        o, lse = fa.forward(q, q, q, causal=True)
        dq, dk, dv = fa.backward(q, q, q, o, lse, q, causal=True)
        assert o.numel() == 0 and dq.numel() == 0
    cu = torch.zeros(4, dtype=torch.int32, device=dev)
    q = torch.zeros((2, 0, 64), dtype=torch.bfloat16, device=dev)
    o, lse = fa.forward(q, q, q, causal=True, cu_seqlens=cu, max_seqlen=1)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_error() == 0


@pytest.mark.parametrize("D, causal, dtype", [(64, False, torch.bfloat16), (64, True, torch.bfloat16),
                                              (128, False, torch.bfloat16), (128, True, torch.bfloat16),
                                              (128, True, torch.float16)],
                         ids=lambda x: str(x).split(".")[-1])
def test_dense_beyond_the_table(D, causal, dtype):
    """Dense inputs with more than 4096 items: the forward walks its closed-form
    list (4608 query-tile pairs) and the backward takes key tiles from the
    workspace queue (9216 tiles), unlike the smaller cases above, which use the
    host-built table.  Sampled heads against the oracle, the gradient sums of
    every head (rows of P sum to one, rows of dS to zero)."""
    B, H, N = 8, 64, 2300
    q, k, v, do = synth.qkv_do((B, H, N, D), dtype, seed_offset=300)
    scale = default_scale(D)
    got = run(q, k, v, do, causal, scale)
    g = np.random.default_rng(11)
    for idx in sorted(g.choice(B * H, size=6, replace=False).tolist()):
        b, h = divmod(idx, H)
        qn, kn, vn, don = (x[b, h].double().numpy() for x in (q, k, v, do))
        O, L = oracle.forward_head(qn, kn, vn, scale, causal)
        dQ, dK, dV, _ = oracle.backward_head(qn, kn, vn, don, scale, causal)
        compare(dtype, {n: f64(t[b, h]) for n, t in got.items()}, dict(o=O, lse=L, dq=dQ, dk=dK, dv=dV),
                f"beyond the table D={D} causal={causal} {dtype} head {(b, h)}")
    dk, dv = got["dk"].float(), got["dv"].float()
    assert ((dk.sum(-2).abs() / dk.abs().sum(-2).clamp_min(1e-6)).max().item()) < 2e-2
    dod = do.to(dv.device).float()
    assert (((dv.sum(-2) - dod.sum(-2)).abs() / dod.abs().sum(-2).clamp_min(1e-6)).max().item()) < 2e-2
