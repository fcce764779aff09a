"""Helpers for the GPU parity tests: run the library through its Python
binding (which calls the C ABI), guard-band the outputs, and compare with the
float64 oracle under the stated tolerances."""

import math

import numpy as np
import torch

import exact_io_aware_37_gb300 as fa

# Acceptance bounds.  bf16: max|dO| <= 2e-2, |dL| <= 1e-3, relative Frobenius
# error of dQ/dK/dV <= 3e-2.  fp32: max|dO| <= 1e-4; the fp32 L and gradient
# bounds below follow from fp32 accumulation over n <= 128 terms of O(1)
# products (relative error ~1e-6) with a wide margin.
# fp16 (not among the stated bounds): the bf16 bounds scaled by the ratio of
# the two rounding units (2^-11 / 2^-8 = 1/8) and rounded up, except L, whose
# error comes from fp32 arithmetic on exact products and keeps the bf16 bound.
TOL = {
    torch.bfloat16: dict(o_max=2e-2, lse_max=1e-3, grad_rel=3e-2),
    torch.float16: dict(o_max=5e-3, lse_max=1e-3, grad_rel=5e-3),
    torch.float32: dict(o_max=1e-4, lse_max=1e-5, grad_rel=1e-5, grad_max=1e-4),
}

GUARD = 4096          # elements of sentinel before and after every output
SENTINEL = 12345.0


class Guarded:
    """An output tensor living inside a larger sentinel-filled buffer."""

    def __init__(self, shape, dtype, device, fill=float("nan")):
        n = int(np.prod(shape))
        self.buf = torch.full((n + 2 * GUARD,), SENTINEL, dtype=dtype, device=device)
        self.t = self.buf[GUARD:GUARD + n].view(shape)
        self.t.fill_(fill)

    def guards_intact(self):
        head = self.buf[:GUARD]
        tail = self.buf[-GUARD:]
        return bool((head == SENTINEL).all()) and bool((tail == SENTINEL).all())


def run(q, k, v, do, causal, scale, cu=None, max_seqlen=None, backward=True):
    """Forward (+ backward) on the GPU with guard-banded, NaN-filled outputs.
    Inputs are CPU tensors; returns a dict of GPU tensors."""
    dev = torch.device("cuda:0")
    qd, kd, vd = (x.to(dev) for x in (q, k, v))
    cud = None if cu is None else cu.to(dev)
    o = Guarded(q.shape, q.dtype, dev)
    lse = Guarded(q.shape[:-1], torch.float32, dev)
    fa.fa_fwd(qd, kd, vd, o.t, lse.t, causal, scale, cud, max_seqlen)
    out = dict(o=o, lse=lse)
    if backward:
        dod = do.to(dev)
        grads = {n: Guarded(q.shape, q.dtype, dev) for n in ("dq", "dk", "dv")}
        ws = fa.fa_bwd_workspace_size(qd, cud, max_seqlen)
        wbuf = torch.full((ws + 2 * 256,), 0x5A, dtype=torch.uint8, device=dev)
        fa.fa_bwd(qd, kd, vd, o.t, lse.t, dod, grads["dq"].t, grads["dk"].t, grads["dv"].t, causal, scale, cud,
                  max_seqlen, workspace=wbuf[256:256 + ws] if ws else wbuf)
        out.update(grads)
    torch.cuda.synchronize()
    st = fa.fa_get_last_device_error()
    assert st == 0, f"device status {st}"
    for name, g in out.items():
        assert g.guards_intact(), f"{name}: write outside the output tensor"
    return {n: g.t for n, g in out.items()}


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def rel_frob(a, b):
    den = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (den if den > 0 else 1.0)


def compare(dtype, got, ref, what, grads=True, o_scale=1.0):
    """got/ref: dicts with o, lse (and dq, dk, dv) as float64 arrays.  o_scale
    widens the O bound (dropout magnifies the weights by 1 / (1 - p))."""
    tol = dict(TOL[dtype])
    tol["o_max"] *= o_scale
    assert np.isfinite(got["o"]).all(), f"{what}: O has NaN/Inf (unwritten rows?)"
    e_o = np.abs(got["o"] - ref["o"]).max() if got["o"].size else 0.0
    assert e_o <= tol["o_max"], f"{what}: max|dO| = {e_o:.3e}"
    e_l = np.abs(got["lse"] - ref["lse"]).max() if got["lse"].size else 0.0
    assert e_l <= tol["lse_max"], f"{what}: max|dL| = {e_l:.3e}"
    errs = dict(o=e_o, lse=e_l)
    if grads:
        for n in ("dq", "dk", "dv"):
            assert np.isfinite(got[n]).all(), f"{what}: {n} has NaN/Inf"
            r = rel_frob(got[n], ref[n])
            assert r <= tol["grad_rel"], f"{what}: {n} relative Frobenius error {r:.3e}"
            errs[n] = r
            if "grad_max" in tol:
                m = np.abs(got[n] - ref[n]).max()
                assert m <= tol["grad_max"], f"{what}: {n} max error {m:.3e}"
    return errs


def default_scale(D):
    return 1.0 / math.sqrt(D)
