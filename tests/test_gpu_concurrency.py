"""Two problems on two streams at once give what they give one after the other.

Each call's work list travels in its own kernel parameters and the backward's
tile counter in its own workspace, so persistent launches of different calls
may share the GPU.  Outputs that do not depend on timing -- O, L, dK, dV (each
written once by one CTA) -- must come out bit-identical; dQ, whose float32
partial sums the copy engine adds in whatever order they arrive, within one
rounding of the 16-bit result."""

import pytest
import torch

import exact_io_aware_37_gb300 as fa
from exact_io_aware_37_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _problem(shape, dtype, seed_offset):
    q, k, v, do = (x.to(DEV) for x in synth.qkv_do(shape, dtype, seed_offset=seed_offset))
    out = dict(o=torch.empty_like(q), lse=torch.empty(shape[:-1], dtype=torch.float32, device=DEV),
               dq=torch.empty_like(q), dk=torch.empty_like(q), dv=torch.empty_like(q))
    ws = torch.empty(max(fa.fa_bwd_workspace_size(q), 1), dtype=torch.uint8, device=DEV)
    return (q, k, v, do), out, ws


def _enqueue(inp, out, ws, causal, stream):
    q, k, v, do = inp
    fa.fa_fwd(q, k, v, out["o"], out["lse"], causal, stream=stream)
    fa.fa_bwd(q, k, v, out["o"], out["lse"], do, out["dq"], out["dk"], out["dv"], causal, workspace=ws, stream=stream)


def test_two_streams_match_one_after_the_other():
    cases = [((2, 4, 1024, 64), torch.bfloat16, True, 100), ((1, 8, 896, 128), torch.float16, False, 101)]
    probs = [_problem(shape, dt, so) for shape, dt, _, so in cases]
    # one after the other on the default stream
    for (inp, out, ws), (_, _, causal, _) in zip(probs, cases):
        _enqueue(inp, out, ws, causal, torch.cuda.current_stream())
    torch.cuda.synchronize()
    ref = [{n: t.clone() for n, t in out.items()} for _, out, _ in probs]
    for _, out, _ in probs:
        for t in out.values():
            t.fill_(float("nan"))
    torch.cuda.synchronize()  # the fills, on the default stream, before the other streams write
    # both at once, several rounds, each problem on a stream of its own
    streams = [torch.cuda.Stream(DEV), torch.cuda.Stream(DEV)]
    for _ in range(3):
        for (inp, out, ws), (_, _, causal, _), st in zip(probs, cases, streams):
            _enqueue(inp, out, ws, causal, st)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_error() == 0
    for (_, out, _), r in zip(probs, ref):
        for n in ("o", "lse", "dk", "dv"):
            assert torch.equal(out[n], r[n]), n
        a, b = out["dq"].float(), r["dq"].float()
        assert torch.isfinite(a).all()
        # the two orders of float32 additions differ by far less than one 16-bit rounding step
        assert ((a - b).abs() <= 2.0 ** -7 * b.abs() + 1e-6).all()
