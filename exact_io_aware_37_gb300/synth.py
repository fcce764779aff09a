"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module holds no attention arithmetic: only random-number recipes and the
workload shapes.  Every tensor is drawn in fp32 on the CPU from its own
``torch.Generator`` seed and then rounded to the dtype the kernels read, so the
oracle (which upcasts the same rounded values to float64) and the GPU path see
identical inputs.  Tensors too large to draw on the host (the size-limit test)
are drawn by the same recipe on the device (``normal_device``); the oracle
then reads the rows it checks back from there.

Seeds: Q=0, K=1, V=2, dO=3, variable-length sequence lengths=4.
"""

import torch

SEED_Q, SEED_K, SEED_V, SEED_DO, SEED_LENS = 0, 1, 2, 3, 4

DTYPES = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}


def normal(shape, seed, dtype, std=1.0):
    """i.i.d. N(0, std^2) in fp32 from ``seed``, then rounded to ``dtype``."""
    g = torch.Generator().manual_seed(int(seed))
    x = torch.randn(tuple(shape), generator=g, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def normal_device(shape, seed, dtype, device, std=1.0):
    """i.i.d. N(0, std^2) in fp32 on ``device`` from ``seed``, rounded to
    ``dtype``; drawn one slice of the leading dimensions at a time (every slice
    in order from the same generator), so the fp32 temporary stays small."""
    g = torch.Generator(device=device).manual_seed(int(seed))
    out = torch.empty(tuple(shape), dtype=dtype, device=device)
    flat = out.view(-1, shape[-2], shape[-1])
    for i in range(flat.shape[0]):
        x = torch.randn((shape[-2], shape[-1]), generator=g, dtype=torch.float32, device=device)
        if std != 1.0:
            x.mul_(std)
        flat[i].copy_(x)
    return out


def qkv_do(shape, dtype, std=1.0, seed_offset=0):
    """(q, k, v, dO) CPU tensors of ``shape`` drawn with seeds 0..3 (+offset)."""
    return tuple(normal(shape, s + seed_offset, dtype, std)
                 for s in (SEED_Q, SEED_K, SEED_V, SEED_DO))


def varlen_lengths(n_seqs, lo, hi, seed=SEED_LENS):
    """Sequence lengths drawn uniformly from [lo, hi] (inclusive)."""
    g = torch.Generator().manual_seed(int(seed))
    return torch.randint(lo, hi + 1, (n_seqs,), generator=g, dtype=torch.int64)


def cu_seqlens(lengths):
    """int32 prefix offsets [0, l0, l0+l1, ...] of a packed batch."""
    lengths = torch.as_tensor(lengths, dtype=torch.int64)
    out = torch.zeros(lengths.numel() + 1, dtype=torch.int64)
    out[1:] = torch.cumsum(lengths, 0)
    return out.to(torch.int32)


# The five workloads.  Dense tensors are [B, H, N, D]; the packed batch is
# [H, T, D] with T = sum of the lengths.
WORKLOADS = {
    "tiny_f32": dict(B=1, H=1, N=128, D=64, dtype="f32", std=1.0,
                     causal=(False, True), scale=1.0 / 8.0),
    "mid_b4h16n1024d64": dict(B=4, H=16, N=1024, D=64, dtype="bf16", std=1.0,
                              causal=(True,)),
    "long_b2h32n4096d128": dict(B=2, H=32, N=4096, D=128, dtype="bf16", std=1.0,
                                causal=(False, True)),
    "varlen16_h32d128": dict(n_seqs=16, len_lo=128, len_hi=8192, H=32, D=128,
                             dtype="bf16", std=1.0, causal=(True,)),
    "window_b1h32n32768d128": dict(B=1, H=32, N=32768, D=128, dtype="bf16",
                                   std=0.5, causal=(True,)),
    # a cached decoding step: one new query per (b, h) against 8192 cached keys
    "decode_b16h32q1k8192d128": dict(B=16, H=32, nq=1, nk=8192, D=128, dtype="bf16",
                                     std=1.0, causal=(True,)),
}


def make_dense(name_or_cfg, seed_offset=0):
    """CPU (q, k, v, dO) for a dense workload."""
    cfg = WORKLOADS[name_or_cfg] if isinstance(name_or_cfg, str) else name_or_cfg
    shape = (cfg["B"], cfg["H"], cfg["N"], cfg["D"])
    return qkv_do(shape, DTYPES[cfg["dtype"]], cfg.get("std", 1.0), seed_offset)


def make_decode(name_or_cfg, seed_offset=0):
    """CPU (q [B,H,nq,D], k, v [B,H,nk,D]) for a cached decoding workload."""
    cfg = WORKLOADS[name_or_cfg] if isinstance(name_or_cfg, str) else name_or_cfg
    dt, std = DTYPES[cfg["dtype"]], cfg.get("std", 1.0)
    B, H, D = cfg["B"], cfg["H"], cfg["D"]
    return (normal((B, H, cfg["nq"], D), SEED_Q + seed_offset, dt, std),
            normal((B, H, cfg["nk"], D), SEED_K + seed_offset, dt, std),
            normal((B, H, cfg["nk"], D), SEED_V + seed_offset, dt, std))


def make_varlen(name_or_cfg, seed_offset=0):
    """CPU (q, k, v, dO, cu_seqlens, lengths) for a packed workload."""
    cfg = WORKLOADS[name_or_cfg] if isinstance(name_or_cfg, str) else name_or_cfg
    lengths = cfg.get("lengths")
    if lengths is None:
        lengths = varlen_lengths(cfg["n_seqs"], cfg["len_lo"], cfg["len_hi"])
    lengths = torch.as_tensor(lengths, dtype=torch.int64)
    cu = cu_seqlens(lengths)
    T = int(cu[-1])
    shape = (cfg["H"], T, cfg["D"])
    q, k, v, do = qkv_do(shape, DTYPES[cfg["dtype"]], cfg.get("std", 1.0), seed_offset)
    return q, k, v, do, cu, lengths
