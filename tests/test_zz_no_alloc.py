"""fa_bwd_static_ws: the backward pass for callers that cannot allocate device
memory (for example a plugin whose host application owns every device byte
through its own pool, or a loop that cannot afford cudaMalloc's latency).
It must give what fa_bwd gives with a caller workspace, on consecutive calls
that reuse the library's one fixed scratch array, and it must refuse problems
larger than that array without launching anything.

This file is named so that pytest collects it last."""

import numpy as np
import pytest
import torch

import exact_io_aware_37_gb300 as fa
from exact_io_aware_37_gb300 import build as fa_build
from exact_io_aware_37_gb300 import synth
from parity import TOL, rel_frob

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    fa_build.build()
    fa.lib()


def _both_ways(shape, dtype, causal, seed_offset):
    dev = torch.device("cuda:0")
    q, k, v, do = (x.to(dev) for x in synth.qkv_do(shape, dtype, seed_offset=seed_offset))
    scale = 1.0 / shape[-1] ** 0.5
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
    ref = fa.backward(q, k, v, o, lse, do, causal=causal, scale=scale)
    got = [torch.full_like(q, float("nan")) for _ in range(3)]
    fa.fa_bwd_static_ws(q, k, v, o, lse, do, *got, causal, scale)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_error() == 0
    return got, ref


def _check(got, ref, dtype):
    tol = TOL[dtype]
    for g, r, name in zip(got, ref, ("dq", "dk", "dv")):
        gn, rn = g.double().cpu().numpy(), r.double().cpu().numpy()
        assert np.isfinite(gn).all(), name
        assert rel_frob(gn, rn) <= tol["grad_rel"], name
        if "grad_max" in tol:
            assert np.abs(gn - rn).max() <= tol["grad_max"], name


def test_two_calls_in_a_row_match_fa_bwd():
    # first call: a larger problem (leaves the scratch full of its values)
    got, ref = _both_ways((1, 4, 1000, 128), torch.bfloat16, True, seed_offset=80)
    _check(got, ref, torch.bfloat16)
    # second call: new inputs, smaller problem, other head width and mask
    got, ref = _both_ways((2, 2, 300, 64), torch.bfloat16, False, seed_offset=81)
    _check(got, ref, torch.bfloat16)


def test_packed_sequences_match_the_oracle():
    """Packed sequences: their backward always takes key tiles from the queue,
    whose counter then lives in the fixed scratch too.  Checked against the
    oracle itself, not against fa_bwd."""
    import oracle
    dev = torch.device("cuda:0")
    lengths = [700, 1, 0, 383, 1290]
    cu = synth.cu_seqlens(lengths)
    H, T, D = 3, int(cu[-1]), 128
    q, k, v, do = synth.qkv_do((H, T, D), torch.bfloat16, seed_offset=83)
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, do))
    cud, scale = cu.to(dev), 1.0 / D ** 0.5
    o, lse = fa.forward(qd, kd, vd, causal=True, scale=scale, cu_seqlens=cud, max_seqlen=max(lengths))
    got = [torch.full_like(qd, float("nan")) for _ in range(3)]
    fa.fa_bwd_static_ws(qd, kd, vd, o, lse, dod, *got, True, scale, cud, max(lengths))
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_error() == 0
    qn, kn, vn, don = (x.double().numpy() for x in (q, k, v, do))
    dQ, dK, dV, _ = oracle.backward_varlen(qn, kn, vn, don, cu, scale, True)
    for g, r, name in zip(got, (dQ, dK, dV), ("dq", "dk", "dv")):
        gn = g.double().cpu().numpy()
        assert np.isfinite(gn).all(), name
        assert rel_frob(gn, r) <= TOL[torch.bfloat16]["grad_rel"], name


def test_float32_path_matches_fa_bwd():
    got, ref = _both_ways((1, 2, 200, 64), torch.float32, True, seed_offset=82)
    _check(got, ref, torch.float32)


def test_oversized_problem_is_refused_without_launch():
    dev = torch.device("cuda:0")
    B, H, N, D = 2, 8, 4096, 128                     # needs ~34 MB of scratch
    q = torch.zeros((B, H, N, D), dtype=torch.bfloat16, device=dev)
    lse = torch.zeros((B, H, N), dtype=torch.float32, device=dev)
    assert fa.fa_bwd_workspace_size(q) > fa.STATIC_WS_BYTES
    before = fa.fa_launch_count()
    with pytest.raises(fa.FAError) as e:
        fa.fa_bwd_static_ws(q, q, q, q, lse, q, q, q, q, True)
    assert e.value.status == -6
    assert "static buffer" in str(e.value)
    assert fa.fa_launch_count() == before
