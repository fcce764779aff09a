"""Checks that pin the float64 oracle to facts outside itself.

Each check takes an implementation namespace ``impl`` exposing
``forward_head(q, k, v, scale, causal) -> (O, L)``,
``backward_head(q, k, v, dO, scale, causal) -> (dQ, dK, dV, D)`` and
``online_softmax_row``; the real oracle passes every check
(test_oracle_pins.py) and each deliberately broken copy of it fails at least
one (test_oracle_mutants.py).  None of the checks re-types the attention
formula: they use closed forms, a library routine (torch SDPA / autograd and
scipy logsumexp, both in float64 on the CPU), finite differences, or
invariants the mathematics fixes.
"""

import math
import os

import numpy as np
import torch
from scipy.special import logsumexp

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def load_split_tile_example():
    scores, tiles = None, []
    with open(os.path.join(GOLDEN, "split_tile_softmax.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "scores":
                scores = [float(x) for x in vals]
            elif key == "tile":
                tiles.append((int(vals[0]), int(vals[1])))
    return scores, tiles


# ---------------------------------------------------------------- worked example

def check_split_tile_example(impl):
    """tensortonic.com "FlashAttention" sections 4-5: scores [1,2,3,4] in tiles
    [1,2] and [3,4]; the merged running state must equal the full-row softmax."""
    scores, tiles = load_split_tile_example()
    assert scores == [1.0, 2.0, 3.0, 4.0] and tiles == [(0, 2), (2, 4)]
    e = [math.exp(s) for s in scores]
    weights = [x / sum(e) for x in e]
    lse = math.log(sum(e))
    # running state after each tile, in closed form
    m1, l1 = 2.0, math.exp(-1.0) + 1.0
    m2, l2 = 4.0, l1 * math.exp(2.0 - 4.0) + math.exp(-1.0) + 1.0
    out, L, states = impl.online_softmax_row(scores, np.eye(4), tiles)
    np.testing.assert_allclose(out, weights, rtol=0, atol=1e-15)
    assert abs(L - lse) < 1e-14
    assert abs(states[0][0] - m1) == 0 and abs(states[0][1] - l1) < 1e-15
    assert abs(states[1][0] - m2) == 0 and abs(states[1][1] - l2) < 1e-15
    # the same numbers through the full attention definition: one query whose
    # dot products with four keys are 1, 2, 3, 4 and one-hot values
    O, Lf = impl.forward_head(np.array([[1.0]]), np.array([[1.0], [2.0], [3.0], [4.0]]),
                              np.eye(4), 1.0, False)
    np.testing.assert_allclose(O[0], weights, rtol=0, atol=1e-15)
    assert abs(Lf[0] - lse) < 1e-14
    # the page's point: softmax per tile gives each tile a full unit of weight
    per_tile = sum(sum(math.exp(s) for s in scores[a:b]) / sum(math.exp(s) for s in scores[a:b])
                   for a, b in tiles)
    assert abs(per_tile - 2.0) < 1e-15


# ---------------------------------------------------------------- closed forms

def check_zero_query(impl):
    """Q = 0 makes every allowed score 0: uniform weights.  Non-causal
    O_i = mean(V), L_i = log n; causal O_i = mean(V[:i+1]), L_i = log(i+1)."""
    r = _rng(11)
    n, d = 9, 5
    q = np.zeros((n, d))
    k = r.standard_normal((n, d))
    v = r.standard_normal((n, d))
    O, L = impl.forward_head(q, k, v, 0.37, False)
    np.testing.assert_allclose(O, np.broadcast_to(v.mean(0), (n, d)), atol=1e-14)
    np.testing.assert_allclose(L, np.full(n, math.log(n)), atol=1e-14)
    O, L = impl.forward_head(q, k, v, 0.37, True)
    running_mean = np.cumsum(v, 0) / np.arange(1, n + 1)[:, None]
    np.testing.assert_allclose(O, running_mean, atol=1e-14)
    np.testing.assert_allclose(L, np.log(np.arange(1, n + 1)), atol=1e-14)


def check_one_hot(impl):
    """Orthogonal keys and q_i = c k_i with large c: weight ~1 on key i, so
    O = V (error ~ n exp(-c^2)) and L = c^2 up to the same error."""
    n = 6
    c = 8.0
    k = np.eye(n)
    q = c * np.eye(n)
    v = _rng(12).standard_normal((n, 3))
    O, L = impl.forward_head(q, c * k, v, 1.0, False)
    # off-diagonal weights are exp(-64) ~ 1.6e-28, far below float64 rounding
    np.testing.assert_allclose(O, v, rtol=0, atol=1e-15)
    np.testing.assert_allclose(L, np.full(n, c * c), rtol=0, atol=1e-13)


def check_rows_sum_to_one(impl):
    """tensortonic.com "FlashAttention" section 1: the weights of a row sum to
    one, so V = 1 gives O = 1 and V + c gives O + c."""
    r = _rng(13)
    n, d = 11, 4
    q, k, v = r.standard_normal((3, n, d))
    for causal in (False, True):
        O1, _ = impl.forward_head(q, k, np.ones((n, d)), 0.5, causal)
        np.testing.assert_allclose(O1, 1.0, atol=1e-14)
        O, _ = impl.forward_head(q, k, v, 0.5, causal)
        Oc, _ = impl.forward_head(q, k, v + 2.5, 0.5, causal)
        np.testing.assert_allclose(Oc, O + 2.5, atol=1e-13)


def check_causal_future_blind(impl):
    """tensortonic.com "FlashAttention" sections 1 and 6: a causal row never
    reads a later key; row 0 reads only key 0 (O_0 = V_0, L_0 = s_00)."""
    r = _rng(14)
    n, d = 10, 4
    q, k, v = r.standard_normal((3, n, d))
    O, L = impl.forward_head(q, k, v, 0.7, True)
    np.testing.assert_allclose(O[0], v[0], atol=1e-15)
    assert abs(L[0] - 0.7 * float(q[0] @ k[0])) < 1e-14
    for i in range(n - 1):
        k2, v2 = k.copy(), v.copy()
        k2[i + 1:] = r.standard_normal((n - i - 1, d)) * 3
        v2[i + 1:] = r.standard_normal((n - i - 1, d)) * 3
        O2, L2 = impl.forward_head(q, k2, v2, 0.7, True)
        np.testing.assert_allclose(O2[:i + 1], O[:i + 1], atol=1e-14)
        np.testing.assert_allclose(L2[:i + 1], L[:i + 1], atol=1e-14)
        assert np.abs(O2[i + 1:] - O[i + 1:]).max() > 1e-3   # later rows do see them


def check_logsumexp_library(impl):
    """L_i is the logarithm of the full row's exponential sum (tensortonic.com
    "FlashAttention" section 7) -- compared with scipy's logsumexp over the
    allowed entries of the row."""
    r = _rng(15)
    n, d = 13, 6
    q, k, v = r.standard_normal((3, n, d)) * 2.0
    for causal in (False, True):
        _, L = impl.forward_head(q, k, v, 0.3, causal)
        for i in range(n):
            lim = i + 1 if causal else n
            row = [0.3 * float(np.dot(q[i], k[j])) for j in range(lim)]
            assert abs(L[i] - logsumexp(row)) < 1e-12


def _torch_reference(q, k, v, do, scale, causal):
    """torch's scaled_dot_product_attention (float64 math path on the CPU)
    with autograd: a library routine independent of the oracle."""
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(
        tq[None, None], tk[None, None], tv[None, None], is_causal=causal, scale=scale)[0, 0]
    out.backward(torch.tensor(do, dtype=torch.float64))
    return (out.detach().numpy(), tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy())


def check_torch_sdpa(impl):
    """Forward and gradients against torch SDPA + autograd in float64."""
    r = _rng(16)
    for n, d, causal in ((7, 3, False), (7, 3, True), (33, 8, True), (20, 16, False)):
        q, k, v, do = r.standard_normal((4, n, d))
        scale = 1.0 / math.sqrt(d)
        O, _ = impl.forward_head(q, k, v, scale, causal)
        dQ, dK, dV, _ = impl.backward_head(q, k, v, do, scale, causal)
        tO, tdq, tdk, tdv = _torch_reference(q, k, v, do, scale, causal)
        np.testing.assert_allclose(O, tO, atol=1e-12)
        np.testing.assert_allclose(dQ, tdq, atol=1e-12)
        np.testing.assert_allclose(dK, tdk, atol=1e-12)
        np.testing.assert_allclose(dV, tdv, atol=1e-12)


def check_finite_differences(impl):
    """Central differences (h = 1e-6) of the scalar loss <dO, O> against the
    analytic gradients, n = 6, d = 4, causal and not."""
    r = _rng(17)
    n, d, h = 6, 4, 1e-6
    q, k, v, do = r.standard_normal((4, n, d))
    for causal in (False, True):
        dQ, dK, dV, _ = impl.backward_head(q, k, v, do, 0.45, causal)

        def loss(qq, kk, vv):
            return float((impl.forward_head(qq, kk, vv, 0.45, causal)[0] * do).sum())

        for which, grad in ((0, dQ), (1, dK), (2, dV)):
            fd = np.zeros((n, d))
            for i in range(n):
                for j in range(d):
                    args_p = [q.copy(), k.copy(), v.copy()]
                    args_m = [q.copy(), k.copy(), v.copy()]
                    args_p[which][i, j] += h
                    args_m[which][i, j] -= h
                    fd[i, j] = (loss(*args_p) - loss(*args_m)) / (2 * h)
            np.testing.assert_allclose(grad, fd, atol=2e-8, rtol=1e-6)


def check_gradient_invariants(impl):
    """Each row of dS sums to zero (softmax Jacobian), so sum_j dK_j = 0; each
    row of P sums to one, so sum_j dV_j = sum_i dO_i; and D_i = sum_j P_ij dP_ij
    equals rowsum(dO o O)."""
    r = _rng(18)
    n, d = 12, 5
    q, k, v, do = r.standard_normal((4, n, d))
    for causal in (False, True):
        dQ, dK, dV, D = impl.backward_head(q, k, v, do, 0.6, causal)
        np.testing.assert_allclose(dK.sum(0), 0.0, atol=1e-13)
        np.testing.assert_allclose(dV.sum(0), do.sum(0), atol=1e-13)
        O, _ = impl.forward_head(q, k, v, 0.6, causal)
        np.testing.assert_allclose(D, (do * O).sum(1), atol=1e-13)


def check_cached_decoding(impl):
    """Bottom-right aligned cached step: against torch SDPA with an explicit
    boolean mask (float64); the square case equals forward_head; every row
    equals an unmasked head over its visible key prefix; rows with no key
    give O = 0 and L = -inf; the batched wrapper matches the per-head one."""
    import torch
    r = _rng(19)
    for nq, nk, d in ((1, 9, 4), (3, 11, 5), (6, 6, 3), (5, 2, 4)):
        q = r.standard_normal((nq, d))
        k, v = r.standard_normal((2, nk, d))
        scale = 0.7
        O, L = impl.forward_cached_head(q, k, v, scale, True)
        allowed = np.arange(nk)[None, :] <= np.arange(nq)[:, None] + (nk - nq)
        for i in range(nq):
            vis = int(allowed[i].sum())
            if vis == 0:
                assert np.all(O[i] == 0.0) and L[i] == -np.inf
                continue
            Oi, Li = impl.forward_head(q[i:i + 1], k[:vis], v[:vis], scale, False)
            np.testing.assert_allclose(O[i], Oi[0], atol=1e-13)
            np.testing.assert_allclose(L[i], Li[0], atol=1e-13)
        rows = allowed.any(1)
        if rows.any():
            t = torch.nn.functional.scaled_dot_product_attention(
                torch.tensor(q[rows])[None], torch.tensor(k)[None], torch.tensor(v)[None],
                attn_mask=torch.tensor(allowed[rows])[None], scale=scale)[0].numpy()
            np.testing.assert_allclose(O[rows], t, atol=1e-12)
        if nq == nk:
            Of, Lf = impl.forward_head(q, k, v, scale, True)
            np.testing.assert_allclose(O, Of, atol=1e-13)
            np.testing.assert_allclose(L, Lf, atol=1e-13)
        On, _ = impl.forward_cached_head(q, k, v, scale, False)
        Ofull, _ = impl.forward_head(q, k, v, scale, False) if nq == nk else (None, None)
        if Ofull is not None:
            np.testing.assert_allclose(On, Ofull, atol=1e-13)
    qb = r.standard_normal((2, 3, 2, 4))
    kb, vb = r.standard_normal((2, 2, 3, 7, 4))
    Ob, Lb = impl.forward_cached(qb, kb, vb, 0.5, True)
    for b in range(2):
        for h in range(3):
            Oh, Lh = impl.forward_cached_head(qb[b, h], kb[b, h], vb[b, h], 0.5, True)
            np.testing.assert_allclose(Ob[b, h], Oh, atol=0)
            np.testing.assert_allclose(Lb[b, h], Lh, atol=0)


def check_philox_known_answers(impl):
    """Philox4x32-10 against the known-answer vectors published with the
    algorithm (counter, key) -> output."""
    vectors = [
        ((0, 0, 0, 0), (0, 0), (0x6627e8d5, 0xe169c58d, 0xbc57ac4c, 0x9b00dbd8)),
        ((0xffffffff,) * 4, (0xffffffff,) * 2, (0x408f276d, 0x41c83b0e, 0xa20bc7c6, 0x6d5451fd)),
        ((0x243f6a88, 0x85a308d3, 0x13198a2e, 0x03707344), (0xa4093822, 0x299f31d0),
         (0xd16cfe09, 0x94fdcceb, 0x5001e420, 0x24126ea1)),
    ]
    for ctr, key, want in vectors:
        got = impl.philox4x32_10(ctr, key)
        assert tuple(int(x) for x in got) == want


def check_dropout(impl):
    """Dropout: the keep fraction is binomial around 1 - p; p = 0 reduces to the
    plain functions; forward and gradients against torch autograd of the same
    masked computation (float64); finite differences; D_i = rowsum(dO o O)."""
    import torch
    keep = impl.dropout_keep(64, 256, 3, 0.3, 1234567, 5)
    frac = keep.mean()
    assert abs(frac - 0.7) < 4 * math.sqrt(0.7 * 0.3 / keep.size)
    assert not np.array_equal(keep, impl.dropout_keep(64, 256, 4, 0.3, 1234567, 5))   # depends on the head
    assert not np.array_equal(keep, impl.dropout_keep(64, 256, 3, 0.3, 1234568, 5))   # and on the seed
    np.testing.assert_array_equal(impl.dropout_keep(5, 9, 3, 0.3, 1234567, 5), keep[:5, :9])
    r = _rng(20)
    n, d = 9, 4
    q, k, v, do = r.standard_normal((4, n, d))
    for causal in (False, True):
        kp = impl.dropout_keep(n, n, 1, 0.0, 99, 0)
        O0, L0 = impl.forward_head_dropout(q, k, v, 0.5, causal, 0.0, kp)
        O1, L1 = impl.forward_head(q, k, v, 0.5, causal)
        np.testing.assert_allclose(O0, O1, atol=1e-14)
        g0 = impl.backward_head_dropout(q, k, v, do, 0.5, causal, 0.0, kp)
        g1 = impl.backward_head(q, k, v, do, 0.5, causal)
        for a, b in zip(g0, g1):
            np.testing.assert_allclose(a, b, atol=1e-13)
        p = 0.35
        kp = impl.dropout_keep(n, n, 2, p, 4242, 7)
        O, L = impl.forward_head_dropout(q, k, v, 0.5, causal, p, kp)
        dQ, dK, dV, D = impl.backward_head_dropout(q, k, v, do, 0.5, causal, p, kp)
        tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
        s = 0.5 * tq @ tk.T
        if causal:
            s = s.masked_fill(torch.triu(torch.ones(n, n, dtype=torch.bool), 1), float("-inf"))
        out = (torch.softmax(s, -1) * torch.tensor(kp / (1 - p))) @ tv
        out.backward(torch.tensor(do))
        np.testing.assert_allclose(O, out.detach().numpy(), atol=1e-12)
        np.testing.assert_allclose(dQ, tq.grad.numpy(), atol=1e-12)
        np.testing.assert_allclose(dK, tk.grad.numpy(), atol=1e-12)
        np.testing.assert_allclose(dV, tv.grad.numpy(), atol=1e-12)
        np.testing.assert_allclose(D, (do * O).sum(1), atol=1e-13)
        h = 1e-6
        for which, grad in ((0, dQ), (1, dK), (2, dV)):
            for (i, j) in ((0, 0), (4, 2), (8, 3)):
                a_p = [q.copy(), k.copy(), v.copy()]
                a_m = [q.copy(), k.copy(), v.copy()]
                a_p[which][i, j] += h
                a_m[which][i, j] -= h
                fp = (impl.forward_head_dropout(*a_p, 0.5, causal, p, kp)[0] * do).sum()
                fm = (impl.forward_head_dropout(*a_m, 0.5, causal, p, kp)[0] * do).sum()
                assert abs((fp - fm) / (2 * h) - grad[i, j]) < 1e-6


def check_stored_o(impl):
    """The o_stored form of the backward: D_i = rowsum(dO o O) over a given
    output.  With the exact O from forward_head it equals the default backward
    (the identity sum_j P_ij dP_ij = dO_i . O_i).  With O + E, dV is unchanged
    and, dS being linear in D, dQ and dK move by exactly
    -scale diag(delta) P K and -scale P^T diag(delta) Q, delta = rowsum(dO o E),
    with P read off forward_head with V = I.  The dense, packed and dropout
    forms pass the array through head by head."""
    r = _rng(31)
    for n, d, causal in ((9, 4, False), (12, 5, True)):
        q, k, v, do = r.standard_normal((4, n, d))
        scale = 0.4
        O, _ = impl.forward_head(q, k, v, scale, causal)
        ref = impl.backward_head(q, k, v, do, scale, causal)
        same = impl.backward_head(q, k, v, do, scale, causal, O)
        for a, b in zip(ref, same):
            np.testing.assert_allclose(b, a, atol=1e-12)
        E = 1e-3 * r.standard_normal((n, d))
        dQ, dK, dV, D = impl.backward_head(q, k, v, do, scale, causal, O + E)
        P, _ = impl.forward_head(q, k, np.eye(n), scale, causal)
        delta = (do * E).sum(1)
        np.testing.assert_allclose(D - ref[3], delta, atol=1e-13)
        assert np.array_equal(dV, ref[2])
        np.testing.assert_allclose(dQ - ref[0], -scale * delta[:, None] * (P @ k), atol=1e-12)
        np.testing.assert_allclose(dK - ref[1], -scale * P.T @ (delta[:, None] * q), atol=1e-12)
        # dropout form with every weight kept and p = 0: the plain form
        keep = np.ones((n, n), dtype=bool)
        got = impl.backward_head_dropout(q, k, v, do, scale, causal, 0.0, keep, O + E)
        for a, b in zip((dQ, dK, dV, D), got):
            np.testing.assert_allclose(b, a, atol=1e-12)
    # batched forms hand each head its own slice of o_stored
    B, H, n, d = 2, 3, 7, 4
    q, k, v, do = r.standard_normal((4, B, H, n, d))
    Ost = r.standard_normal((B, H, n, d))
    dQ, dK, dV, D = impl.backward(q, k, v, do, 0.3, True, Ost)
    for b in range(B):
        for h in range(H):
            one = impl.backward_head(q[b, h], k[b, h], v[b, h], do[b, h], 0.3, True, Ost[b, h])
            for a, x in zip(one, (dQ[b, h], dK[b, h], dV[b, h], D[b, h])):
                np.testing.assert_allclose(x, a, atol=1e-12)
    cu = np.array([0, 3, 3, 7])
    qp, kp, vp, dop, Op = (x.reshape(B * H, n, d)[:H] for x in (q, k, v, do, Ost))
    dQ, dK, dV, D = impl.backward_varlen(qp, kp, vp, dop, cu, 0.3, True, o_stored=Op)
    for h in range(H):
        for a0, a1 in ((0, 3), (3, 7)):
            one = impl.backward_head(qp[h, a0:a1], kp[h, a0:a1], vp[h, a0:a1], dop[h, a0:a1], 0.3, True,
                                     Op[h, a0:a1])
            for a, x in zip(one, (dQ[h, a0:a1], dK[h, a0:a1], dV[h, a0:a1], D[h, a0:a1])):
                np.testing.assert_allclose(x, a, atol=1e-12)
    keep = impl.dropout_keep(n, n, 4, 0.3, 99, 1)
    dQ, dK, dV, D = impl.backward_dropout(q, k, v, do, 0.3, False, 0.3, 99, 1, Ost)
    one = impl.backward_head_dropout(q[1, 1], k[1, 1], v[1, 1], do[1, 1], 0.3, False, 0.3, keep, Ost[1, 1])
    for a, x in zip(one, (dQ[1, 1], dK[1, 1], dV[1, 1], D[1, 1])):
        np.testing.assert_allclose(x, a, atol=1e-12)


ALL_CHECKS = [
    check_split_tile_example,
    check_zero_query,
    check_one_hot,
    check_rows_sum_to_one,
    check_causal_future_blind,
    check_logsumexp_library,
    check_torch_sdpa,
    check_finite_differences,
    check_gradient_invariants,
    check_cached_decoding,
    check_philox_known_answers,
    check_dropout,
    check_stored_o,
]
