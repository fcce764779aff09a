"""Exact IO-aware tiled attention for GB300 (sm_103a).

Python binding of the C ABI in include/fa.h.  Functions with the C names
(``fa_fwd``, ``fa_bwd``, ``fa_bwd_workspace_size``, ``fa_get_last_device_error``,
``fa_strerror``, ...) marshal torch tensors to pointers and call the library;
``forward`` / ``backward`` also allocate the outputs.  Every step of the
computation runs in the library's CUDA kernels: torch only provides device
memory and the current stream.

Layouts: dense tensors are [B, H, N, D]; packed variable-length batches are
[H, T, D] with int32 ``cu_seqlens`` [B + 1] on the device and ``max_seqlen``.
"""

import math

import torch

from ._lib import FA_BF16, FA_F16, FA_F32, FAError, lib, library_path  # noqa: F401

__all__ = ["fa_fwd", "fa_bwd", "fa_bwd_workspace_size", "fa_get_last_device_error", "fa_strerror",
           "fa_set_wait_limit_ns", "fa_selftest_wait_timeout", "fa_selftest_tile", "fa_path_name", "fa_launch_count", "fa_bwd_static_ws", "fa_bwd_time_main_kernel", "forward", "backward",
           "fa_decode", "fa_decode_workspace_size", "decode", "fa_fwd_dropout", "fa_bwd_dropout",
           "fa_bwd_deterministic", "fa_probe_ex2_rate", "FAError"]

_DT = {torch.bfloat16: FA_BF16, torch.float32: FA_F32, torch.float16: FA_F16}


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dims(q, cu_seqlens, max_seqlen):
    """(B, H, N, D, T) from the tensor shapes."""
    if cu_seqlens is None:
        if q.dim() != 4:
            raise ValueError("dense tensors must be [B, H, N, D]")
        B, H, N, D = q.shape
        return B, H, N, D, 0
    if q.dim() != 3:
        raise ValueError("packed tensors must be [H, T, D]")
    if max_seqlen is None:
        raise ValueError("packed input needs max_seqlen")
    if cu_seqlens.dtype != torch.int32:
        raise ValueError("cu_seqlens must be int32")
    H, T, D = q.shape
    return cu_seqlens.numel() - 1, H, int(max_seqlen), D, T


def _check(*tensors):
    ref = tensors[0]
    for t in tensors:
        if t is None:
            continue
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
        if t.device != ref.device:
            raise ValueError("tensors must be on one device")


def fa_strerror(status):
    return lib().fa_strerror(int(status)).decode()


def fa_path_name(dtype, D):
    r = lib().fa_path_name(_DT[dtype] if isinstance(dtype, torch.dtype) else int(dtype), int(D))
    return None if r is None else r.decode()


def fa_launch_count():
    return int(lib().fa_launch_count())


def fa_bwd_time_main_kernel(start_event, stop_event):
    """Have the next fa_bwd on this thread record the two torch.cuda.Events
    (already recorded once, so they exist) around its main gradient kernel."""
    lib().fa_bwd_time_main_kernel(start_event.cuda_event, stop_event.cuda_event)


def fa_probe_ex2_rate(iters=4096, stream=None):
    """Measured ex2.approx throughput, exponentials per clock per SM (see
    fa_probe_ex2_rate in include/fa.h).  Synchronises the stream."""
    import ctypes
    out = ctypes.c_double(0.0)
    st = lib().fa_probe_ex2_rate(int(iters), ctypes.byref(out), _stream(stream))
    if st != 0:
        raise FAError(st, "fa_probe_ex2_rate")
    return out.value


def fa_set_wait_limit_ns(limit_ns):
    lib().fa_set_wait_limit_ns(int(limit_ns))


def fa_get_last_device_error(stream=None):
    return lib().fa_get_last_device_error(_stream(stream))


def fa_selftest_wait_timeout(stream=None):
    return lib().fa_selftest_wait_timeout(_stream(stream))


def fa_selftest_tile(a, b, s_out, o_out, a_copy, stream=None):
    """One-tile check of the tensor-core building blocks: s_out = a b^T,
    o_out = round(s_out) b (float32), a_copy = a read back from its swizzled
    shared-memory tile.  a, b, a_copy: [128, D] bf16 or fp16; returns the
    status code."""
    for t in (a, b, s_out, o_out, a_copy):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("fa_selftest_tile wants contiguous CUDA tensors")
    if s_out.dtype != torch.float32 or o_out.dtype != torch.float32 or a_copy.dtype != a.dtype:
        raise ValueError("s_out and o_out must be float32, a_copy of a's dtype")
    D = a.shape[-1]
    if (a.dim() != 2 or tuple(a.shape) != (128, D) or b.shape != a.shape or a_copy.shape != a.shape
            or b.dtype != a.dtype or tuple(s_out.shape) != (128, 128) or tuple(o_out.shape) != (128, D)):
        raise ValueError("fa_selftest_tile wants a, b, a_copy [128, D], s_out [128, 128], o_out [128, D]")
    dt = _DT.get(a.dtype, FA_F32)
    return lib().fa_selftest_tile(_ptr(a), _ptr(b), _ptr(s_out), _ptr(o_out), _ptr(a_copy), D, dt, _stream(stream))


def fa_fwd(q, k, v, o, lse, causal, scale=None, cu_seqlens=None, max_seqlen=None, stream=None):
    """Enqueue the forward kernel: writes o (dtype of q) and lse (float32)."""
    _check(q, k, v, o, lse, cu_seqlens)
    B, H, N, D, T = _dims(q, cu_seqlens, max_seqlen)
    if lse.dtype != torch.float32:
        raise ValueError("lse must be float32")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    st = lib().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, D, scale, int(bool(causal)),
                      _ptr(cu_seqlens), T, _DT[q.dtype], _stream(stream))
    if st != 0:
        raise FAError(st, "fa_fwd")


def fa_bwd_workspace_size(q, cu_seqlens=None, max_seqlen=None):
    B, H, N, D, T = _dims(q, cu_seqlens, max_seqlen)
    return int(lib().fa_bwd_workspace_size(B, H, N, D, _ptr(cu_seqlens), T, _DT[q.dtype]))


def fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, causal, scale=None, cu_seqlens=None, max_seqlen=None,
           workspace=None, stream=None):
    """Enqueue the backward kernels: writes dq, dk, dv (dtype of q)."""
    _check(q, k, v, o, lse, dout, dq, dk, dv, cu_seqlens)
    B, H, N, D, T = _dims(q, cu_seqlens, max_seqlen)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    if workspace is None:
        need = fa_bwd_workspace_size(q, cu_seqlens, max_seqlen)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    st = lib().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                      B, H, N, D, scale, int(bool(causal)), _ptr(cu_seqlens), T, _DT[q.dtype],
                      _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    if st != 0:
        raise FAError(st, "fa_bwd")


def fa_bwd_static_ws(q, k, v, o, lse, dout, dq, dk, dv, causal, scale=None, cu_seqlens=None, max_seqlen=None,
                     stream=None):
    """fa_bwd without a workspace argument: the library's own fixed device
    buffer (FA_BWD_STATIC_WS_BYTES, 16 MiB) serves as scratch, for callers
    that cannot allocate device memory.  Calls sharing a device must not
    overlap on the GPU; problems needing more scratch raise FAError
    (FA_ERR_WORKSPACE)."""
    _check(q, k, v, o, lse, dout, dq, dk, dv, cu_seqlens)
    B, H, N, D, T = _dims(q, cu_seqlens, max_seqlen)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    st = lib().fa_bwd_static_ws(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
                                _ptr(dv), B, H, N, D, scale, int(bool(causal)), _ptr(cu_seqlens), T, _DT[q.dtype],
                                _stream(stream))
    if st != 0:
        err = FAError(st, "fa_bwd_static_ws")
        detail = lib().fa_last_error_detail().decode()
        if detail and detail not in str(err):
            err = FAError(st, f"fa_bwd_static_ws [{detail}]")
        raise err


STATIC_WS_BYTES = 16 << 20


def fa_fwd_dropout(q, k, v, o, lse, causal, p_drop, seed, offset=0, scale=None, cu_seqlens=None, max_seqlen=None,
                   stream=None):
    """fa_fwd with attention dropout: weights dropped with probability p_drop
    (decisions regenerated from seed and offset), kept ones scaled by
    1 / (1 - p_drop); lse is that of the undropped softmax."""
    _check(q, k, v, o, lse, cu_seqlens)
    B, H, N, D, T = _dims(q, cu_seqlens, max_seqlen)
    if lse.dtype != torch.float32:
        raise ValueError("lse must be float32")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    st = lib().fa_fwd_dropout(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, D, scale, int(bool(causal)),
                              _ptr(cu_seqlens), T, _DT[q.dtype], float(p_drop), int(seed), int(offset),
                              _stream(stream))
    if st != 0:
        raise FAError(st, "fa_fwd_dropout")


def fa_bwd_dropout(q, k, v, o, lse, dout, dq, dk, dv, causal, p_drop, seed, offset=0, scale=None, cu_seqlens=None,
                   max_seqlen=None, workspace=None, stream=None):
    """fa_bwd for a forward run by fa_fwd_dropout with the same p_drop, seed, offset."""
    _check(q, k, v, o, lse, dout, dq, dk, dv, cu_seqlens)
    B, H, N, D, T = _dims(q, cu_seqlens, max_seqlen)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    if workspace is None:
        need = fa_bwd_workspace_size(q, cu_seqlens, max_seqlen)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    st = lib().fa_bwd_dropout(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                              B, H, N, D, scale, int(bool(causal)), _ptr(cu_seqlens), T, _DT[q.dtype], float(p_drop),
                              int(seed), int(offset), _ptr(workspace), workspace.numel() * workspace.element_size(),
                              _stream(stream))
    if st != 0:
        raise FAError(st, "fa_bwd_dropout")


def fa_bwd_deterministic(q, k, v, o, lse, dout, dq, dk, dv, causal, scale=None, cu_seqlens=None, max_seqlen=None,
                         p_drop=0.0, seed=0, offset=0, workspace=None, stream=None):
    """fa_bwd (or fa_bwd_dropout) with every sum in a fixed order: repeated
    calls give bit-identical gradients (dQ from a query-stationary kernel)."""
    _check(q, k, v, o, lse, dout, dq, dk, dv, cu_seqlens)
    B, H, N, D, T = _dims(q, cu_seqlens, max_seqlen)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    if workspace is None:
        rows = (H * T) if cu_seqlens is not None else (B * H * N)
        workspace = torch.empty((rows * 4 + 255) // 256 * 256 + 256, dtype=torch.uint8, device=q.device)
    st = lib().fa_bwd_deterministic(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
                                    _ptr(dv), B, H, N, D, scale, int(bool(causal)), _ptr(cu_seqlens), T,
                                    _DT[q.dtype], float(p_drop), int(seed), int(offset), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), _stream(stream))
    if st != 0:
        raise FAError(st, "fa_bwd_deterministic")


def fa_decode_workspace_size(q, k):
    """Bytes of scratch fa_decode needs for q [B, H, nq, D] against k [B, H, nk, D]."""
    B, H, nq, D = q.shape
    return int(lib().fa_decode_workspace_size(B, H, nq, k.shape[2], D, _DT[q.dtype]))


def fa_decode(q, k, v, o, lse, causal, scale=None, workspace=None, stream=None):
    """Enqueue a cached decoding step: q [B, H, nq, D] against the cache
    k, v [B, H, nk, D]; query i is at position nk - nq + i.  Writes o (dtype of
    q) and lse [B, H, nq] (float32)."""
    _check(q, k, v, o, lse)
    if q.dim() != 4 or k.dim() != 4 or k.shape != v.shape or k.shape[:2] != q.shape[:2] or k.shape[3] != q.shape[3]:
        raise ValueError("q must be [B, H, nq, D] and k, v [B, H, nk, D]")
    if lse.dtype != torch.float32:
        raise ValueError("lse must be float32")
    B, H, nq, D = q.shape
    nk = k.shape[2]
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    need = fa_decode_workspace_size(q, k)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().fa_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, nq, nk, D, scale, int(bool(causal)),
                         _DT[q.dtype], _ptr(workspace), nbytes, _stream(stream))
    if st != 0:
        raise FAError(st, "fa_decode")


def decode(q, k, v, causal=True, scale=None, stream=None):
    """Allocating convenience wrapper around fa_decode: returns (o, lse)."""
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    fa_decode(q, k, v, o, lse, causal, scale, stream=stream)
    return o, lse


def forward(q, k, v, causal=False, scale=None, cu_seqlens=None, max_seqlen=None, stream=None):
    """(o, lse) for dense [B,H,N,D] or packed [H,T,D] inputs."""
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    fa_fwd(q, k, v, o, lse, causal, scale, cu_seqlens, max_seqlen, stream)
    return o, lse


def backward(q, k, v, o, lse, dout, causal=False, scale=None, cu_seqlens=None, max_seqlen=None,
             workspace=None, stream=None):
    """(dq, dk, dv) given the forward outputs and the upstream gradient."""
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, causal, scale, cu_seqlens, max_seqlen, workspace, stream)
    return dq, dk, dv
