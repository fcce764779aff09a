"""Every entry point at a caller-chosen scale, against the float64 oracle.

The other parity tests use the default 1/sqrt(D), so a kernel that applied
1/sqrt(D) itself -- in the exponent (scale * log2 e), in dK, or in the dQ
conversion -- instead of the scale it was given would still pass them.  Here
the scales range from a nearly flat softmax (0.02) to scores ten times the
default spread (1.0 at D = 128, where the running maximum also grows past the
lazy rescale threshold again and again).  As in the rescale tests, the
reference dQ and dK take D_i = rowsum(dO o O) over the oracle's own output
rounded to the input type, the quantity the one-pass backward forms: at
large scales the softmax is nearly one-hot, the true dQ and dK are small, and
the rounding of O would otherwise dominate their difference."""

import numpy as np
import pytest
import torch

import exact_io_aware_37_gb300 as fa
import oracle
from exact_io_aware_37_gb300 import synth
from parity import TOL, compare, f64, run
from test_gpu_deterministic import _run as _run_deterministic
from test_gpu_dropout import _fwd_bwd as _run_dropout, _p32
from test_gpu_rescale import _stored

pytestmark = pytest.mark.gpu

SCALES = [0.02, 0.3, 1.0]


def _dense_ref(q, k, v, do, scale, causal):
    qn, kn, vn, don = (x.double().numpy() for x in (q, k, v, do))
    O, L = oracle.forward(qn, kn, vn, scale, causal)
    dQ, dK, dV, _ = oracle.backward(qn, kn, vn, don, scale, causal, o_stored=_stored(O, q.dtype))
    return dict(o=O, lse=L, dq=dQ, dk=dK, dv=dV)


@pytest.mark.parametrize("scale", SCALES)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [64, 128])
def test_dense_bf16_scale(D, causal, scale):
    shape = (1, 2, 300, D)  # three query and key tiles, the last ragged
    q, k, v, do = synth.qkv_do(shape, torch.bfloat16, seed_offset=90)
    got = run(q, k, v, do, causal, scale)
    compare(torch.bfloat16, {n: f64(t) for n, t in got.items()}, _dense_ref(q, k, v, do, scale, causal),
            f"dense D={D} causal={causal} scale={scale}")


@pytest.mark.parametrize("scale", [0.05, 0.5])
def test_dense_f16_scale(scale):
    shape = (2, 2, 257, 64)
    q, k, v, do = synth.qkv_do(shape, torch.float16, seed_offset=91)
    got = run(q, k, v, do, True, scale)
    compare(torch.float16, {n: f64(t) for n, t in got.items()}, _dense_ref(q, k, v, do, scale, True),
            f"f16 scale={scale}")


@pytest.mark.parametrize("D", [64, 128])
def test_packed_scale(D):
    lengths = [130, 0, 255, 7]
    cu = synth.cu_seqlens(lengths)
    q, k, v, do = synth.qkv_do((2, int(cu[-1]), D), torch.bfloat16, seed_offset=92)
    scale = 0.3
    got = run(q, k, v, do, True, scale, cu=cu, max_seqlen=max(lengths))
    qn, kn, vn, don = (x.double().numpy() for x in (q, k, v, do))
    O, L = oracle.forward_varlen(qn, kn, vn, cu, scale, True)
    dQ, dK, dV, _ = oracle.backward_varlen(qn, kn, vn, don, cu, scale, True, o_stored=_stored(O, q.dtype))
    compare(torch.bfloat16, {n: f64(t) for n, t in got.items()}, dict(o=O, lse=L, dq=dQ, dk=dK, dv=dV),
            f"packed D={D} scale={scale}")


@pytest.mark.parametrize("D", [64, 128])
def test_dropout_scale(D):
    q, k, v, do = synth.qkv_do((1, 2, 300, D), torch.bfloat16, seed_offset=93)
    scale, p, seed, off = 0.3, 0.2, 777 + D, 3
    got = _run_dropout(q, k, v, do, True, scale, p, seed, off)
    qn, kn, vn, don = (x.double().numpy() for x in (q, k, v, do))
    O, L = oracle.forward_dropout(qn, kn, vn, scale, True, _p32(p), seed, off)
    dQ, dK, dV, _ = oracle.backward_dropout(qn, kn, vn, don, scale, True, _p32(p), seed, off,
                                            o_stored=_stored(O, q.dtype))
    compare(torch.bfloat16, got, dict(o=O, lse=L, dq=dQ, dk=dK, dv=dV), f"dropout D={D} scale={scale}",
            o_scale=1.0 / (1.0 - p))


@pytest.mark.parametrize("D", [64, 128])
def test_deterministic_scale(D):
    q, k, v, do = synth.qkv_do((1, 2, 300, D), torch.bfloat16, seed_offset=94)
    scale = 0.3
    got = _run_deterministic(q, k, v, do, True, scale)
    compare(torch.bfloat16, got, _dense_ref(q, k, v, do, scale, True), f"deterministic D={D} scale={scale}")


@pytest.mark.parametrize("scale", [0.02, 0.5])
def test_decode_scale(scale):
    B, H, nq, nk, D = 2, 3, 3, 700, 128
    q = synth.normal((B, H, nq, D), synth.SEED_Q + 95, torch.bfloat16)
    k = synth.normal((B, H, nk, D), synth.SEED_K + 95, torch.bfloat16)
    v = synth.normal((B, H, nk, D), synth.SEED_V + 95, torch.bfloat16)
    dev = torch.device("cuda:0")
    qd, kd, vd = (x.to(dev) for x in (q, k, v))
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, nq), dtype=torch.float32, device=dev)
    fa.fa_decode(qd, kd, vd, o, lse, True, scale)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_error() == 0
    Oref, Lref = oracle.forward_cached(*(x.double().numpy() for x in (q, k, v)), scale, True)
    tol = TOL[torch.bfloat16]
    assert np.abs(f64(o) - Oref).max() <= tol["o_max"]
    assert np.abs(f64(lse) - Lref).max() <= tol["lse_max"]
