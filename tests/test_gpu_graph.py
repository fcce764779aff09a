"""Calls captured in a CUDA graph and replayed give what eager calls give.

Every entry point enqueues its kernels on the caller's stream without a host
synchronisation or an allocation, and passes its work list by value in the
kernel parameters (the backward's tile counter lives in the caller's
workspace and is reset by the preprocess kernel of the same call), so a
training step's calls can be captured once and replayed on new input values.
Each case runs the calls eagerly first (one-time host look-ups happen there),
captures them, writes new values into the captured input buffers, replays the
graph twice and compares with eager calls on the same values: O, L, dK and dV
bit for bit, dQ of the one-pass backward within one rounding of the 16-bit
result (its float32 partial sums are added in arrival order), dQ of the
deterministic backward bit for bit."""

import pytest
import torch

import exact_io_aware_37_gb300 as fa
from exact_io_aware_37_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _capture(step):
    """Run `step(stream)` eagerly on a side stream, then capture it."""
    side = torch.cuda.Stream(DEV)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):
            step(side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(torch.cuda.current_stream())
    torch.cuda.synchronize()
    return g


def _close_dq(a, b):
    a, b = a.float(), b.float()
    return bool(torch.isfinite(a).all()) and bool(((a - b).abs() <= 2.0 ** -7 * b.abs() + 1e-6).all())


def _buffers(q):
    return dict(o=torch.empty_like(q), lse=torch.empty(q.shape[:-1], dtype=torch.float32, device=DEV),
                dq=torch.empty_like(q), dk=torch.empty_like(q), dv=torch.empty_like(q))


CASES = [
    # (shape: dense [B,H,N,D] or packed lengths + (H, D), dtype, causal, backward form)
    ((2, 4, 1024, 64), torch.bfloat16, True, "atomic"),        # host-built tables
    ((1, 36, 16384, 64), torch.bfloat16, True, "atomic"),      # 4608 key tiles: the backward's queue
    (([300, 1, 0, 2048, 777], 4, 128), torch.float16, True, "atomic"),  # packed: closed-form list and queue
    ((1, 8, 1000, 128), torch.bfloat16, False, "deterministic"),
    ((2, 4, 640, 128), torch.bfloat16, True, "dropout"),
]


def _case_id(c):
    shape, dt, causal, form = c
    s = "x".join(map(str, shape)) if isinstance(shape[0], int) else "packed" + "-".join(map(str, shape[0]))
    return f"{s}-{str(dt).split('.')[-1]}-{'causal' if causal else 'full'}-{form}"


@pytest.mark.parametrize("case", CASES, ids=_case_id)
def test_training_step_replays_from_a_graph(case):
    shape, dt, causal, form = case
    if isinstance(shape[0], int):
        full_shape = shape
        cu = max_seqlen = None
    else:
        lengths, H, D = shape
        T = sum(lengths)
        full_shape = (H, T, D)
        cu = synth.cu_seqlens(lengths).to(DEV)
        max_seqlen = max(lengths)
    inp = [x.to(DEV) for x in synth.qkv_do(full_shape, dt, seed_offset=40)]
    new = [x.to(DEV) for x in synth.qkv_do(full_shape, dt, seed_offset=41)]
    q, k, v, do = inp
    out = _buffers(q)
    ws = torch.empty(max(fa.fa_bwd_workspace_size(q, cu, max_seqlen), 1 << 16), dtype=torch.uint8, device=DEV)
    p_drop, seed = 0.2, 1234

    def step(stream, bufs=out, tensors=inp):
        q, k, v, do = tensors
        o, lse, dq, dk, dv = (bufs[n] for n in ("o", "lse", "dq", "dk", "dv"))
        if form == "dropout":
            fa.fa_fwd_dropout(q, k, v, o, lse, causal, p_drop, seed, cu_seqlens=cu, max_seqlen=max_seqlen,
                              stream=stream)
            fa.fa_bwd_dropout(q, k, v, o, lse, do, dq, dk, dv, causal, p_drop, seed, cu_seqlens=cu,
                              max_seqlen=max_seqlen, workspace=ws, stream=stream)
            return
        fa.fa_fwd(q, k, v, o, lse, causal, cu_seqlens=cu, max_seqlen=max_seqlen, stream=stream)
        if form == "deterministic":
            fa.fa_bwd_deterministic(q, k, v, o, lse, do, dq, dk, dv, causal, cu_seqlens=cu, max_seqlen=max_seqlen,
                                    workspace=ws, stream=stream)
        else:
            fa.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, causal, cu_seqlens=cu, max_seqlen=max_seqlen,
                      workspace=ws, stream=stream)

    g = _capture(step)
    for dst, src in zip(inp, new):
        dst.copy_(src)
    for t in out.values():
        t.fill_(float("nan"))
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_error() == 0

    ref = _buffers(q)
    step(torch.cuda.current_stream(), bufs=ref, tensors=new)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_error() == 0
    for n in ("o", "lse", "dk", "dv"):
        assert torch.equal(out[n], ref[n]), n
    if form == "deterministic":
        assert torch.equal(out["dq"], ref["dq"])
    else:
        assert _close_dq(out["dq"], ref["dq"])


def test_decoding_step_replays_from_a_graph():
    B, H, nq, nk, D = 2, 8, 3, 2500, 128
    q, k, v = (synth.normal_device(s, seed, torch.bfloat16, DEV)
               for s, seed in (((B, H, nq, D), 50), ((B, H, nk, D), 51), ((B, H, nk, D), 52)))
    o = torch.empty_like(q)
    lse = torch.empty(B, H, nq, dtype=torch.float32, device=DEV)
    ws = torch.empty(max(fa.fa_decode_workspace_size(q, k), 1), dtype=torch.uint8, device=DEV)

    def step(stream, o=o, lse=lse):
        fa.fa_decode(q, k, v, o, lse, True, workspace=ws, stream=stream)

    g = _capture(step)
    q.copy_(synth.normal_device((B, H, nq, D), 53, torch.bfloat16, DEV))
    k[:, :, -7:].copy_(synth.normal_device((B, H, 7, D), 54, torch.bfloat16, DEV))  # newest cache entries
    g.replay()
    torch.cuda.synchronize()
    o_ref, lse_ref = torch.empty_like(o), torch.empty_like(lse)
    step(torch.cuda.current_stream(), o_ref, lse_ref)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_error() == 0
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
