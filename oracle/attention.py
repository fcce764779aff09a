"""Plain, slow, float64 definition of exact softmax attention and its gradients.

TEST INFRASTRUCTURE ONLY -- see the package docstring.  Nothing here is tiled,
fused or reordered beyond what the cited passage states; every array is
float64 numpy.  Inputs arrive already rounded to the dtype the GPU path reads
(bf16 or fp32) and are upcast here, so both sides see identical values.

Notation (tensortonic.com "FlashAttention"):
  q, k, v   : one head, shape [n, d]   (section 9: [batch, heads, tokens, head_width])
  S         : scaled, masked scores, S_ij = scale * q_i . k_j   (section 6)
  m_i, l_i  : row maximum and denominator of the stable softmax (sections 4, 5)
  L_i       : log-sum-exp, L_i = m_i + log(l_i)                  (section 7)
  P_ij      : exp(S_ij - L_i)                                    (section 7)
  O         : P V                                                (section 1)

Pins (what each function is checked against in tests/test_oracle_pins.py;
none of them re-types the formula below):
  score_matrix, forward_head     closed forms (Q = 0 gives uniform weights,
                                 one-hot scores give O = V), scipy logsumexp,
                                 torch SDPA (float64, CPU), rows of P sum to 1,
                                 causal rows blind to future keys, the printed
                                 [1, 2, 3, 4] example.
  backward_head                  central finite differences of <dO, O>,
                                 torch autograd (float64, CPU), sum_j dK_j = 0,
                                 sum_j dV_j = sum_i dO_i.
    (o_stored argument)          with the exact O it gives the default result;
                                 dV never changes; dQ and dK move by the
                                 closed-form first-order term of a shift of D
                                 (exact, dS being linear in D).
  forward / backward             reduce to the *_head functions per (b, h);
                                 pinned through them plus a layout test.
  forward_varlen/backward_varlen equal to running each packed sequence as its
                                 own dense head; no cross-sequence leakage.
  forward_rows, backward_dq_rows equal to the full-matrix functions on the
                                 sampled rows.
  backward_head_blocked          equal to backward_head.
  online_softmax_row             the printed [1, 2, 3, 4] split-tile example in
                                 closed form; equal to the full-row softmax.
  tiled_forward_head             equal to forward_head for several tile sizes.
  cached_score_matrix,           torch SDPA (float64) with the bottom-right
  forward_cached_head,           boolean mask; with nq == nk equal to
  forward_cached                 forward_head; row i equal to the unmasked
                                 forward_head over keys 0 .. nk - nq + i; rows
                                 with no allowed key give O = 0, L = -inf.
  philox4x32_10                  the published known-answer vectors of
                                 Philox4x32-10 (three counter/key pairs).
  dropout_keep                   keep fraction within binomial bounds;
                                 independent of the row/column orientation.
  forward_head_dropout,          p = 0 gives forward_head / backward_head;
  backward_head_dropout,         torch autograd (float64) of the same masked
  forward_dropout,               computation; central finite differences;
  backward_dropout               D_i = rowsum(dO o O) with the dropped O.
No function is "parity unpinned".
"""

import numpy as np


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def score_matrix(q, k, scale, causal):
    """S = scale * Q K^T with the causal mask applied before any softmax step.

    tensortonic.com "FlashAttention" section 6: the key/query dot products are
    scaled (by 1/sqrt(width) by default; the caller passes ``scale``) and "the
    causal mask is applied before those scores enter the softmax update".
    Causal means key j is allowed for query i iff j <= i, both counted from the
    start of their own sequence (square, top-left alignment -- the only layout
    the pages' example uses, section 9).  Masked entries are -inf.
    """
    q = _f64(q)
    k = _f64(k)
    s = scale * (q @ k.T)
    if causal:
        i = np.arange(s.shape[0])[:, None]
        j = np.arange(s.shape[1])[None, :]
        s = np.where(j <= i, s, -np.inf)
    return s


def _softmax_rows(s):
    """Stable row softmax of a masked score matrix.

    tensortonic.com "FlashAttention" section 4: subtract the row maximum before
    exponentiating; the weights are unchanged.  Section 7: L = m + log(l).
    A row with no allowed key (impossible for square causal or dense rows; the
    pages are silent) gets P = 0 and L = -inf.
    Returns (P, L, m, l).
    """
    m = s.max(axis=1) if s.shape[1] else np.full(s.shape[0], -np.inf)
    has_key = np.isfinite(m)
    m0 = np.where(has_key, m, 0.0)
    e = np.exp(s - m0[:, None])          # exp(-inf) = 0 for masked entries
    l = e.sum(axis=1)
    L = np.where(has_key, m0 + np.log(np.where(has_key, l, 1.0)), -np.inf)
    P = np.where(has_key[:, None], e / np.where(has_key, l, 1.0)[:, None], 0.0)
    return P, L, m, l


def forward_head(q, k, v, scale, causal):
    """Exact attention for one head: returns (O [n, d], L [n]).

    wiki.ai-engineering.at "Flash Attention", The Core Problem (the naive
    listing: scores, softmax, weights @ V) and tensortonic.com "FlashAttention"
    sections 1, 4, 7.  The full n x n matrix is formed: this is the definition
    the tiled method must reproduce exactly (up to rounding order, section 8).
    """
    s = score_matrix(q, k, scale, causal)
    P, L, _, _ = _softmax_rows(s)
    O = P @ _f64(v)
    return O, L


def backward_head(q, k, v, do, scale, causal, o_stored=None):
    """Analytic gradients of attention for one head given upstream dO.

    The pages state only that the backward pass rebuilds each weight as
    exp(s_ij - L_i) (tensortonic.com "FlashAttention" section 7); the gradient
    algebra below is the standard differentiation of O = softmax(S) V with
    S = scale * Q K^T:
        dV = P^T dO
        dP = dO V^T
        D_i = sum_j P_ij dP_ij
        dS = P o (dP - D)          (softmax Jacobian, row by row)
        dQ = scale * dS K
        dK = scale * dS^T Q
    ``o_stored``: a one-pass backward cannot form sum_j P_ij dP_ij before it
    needs dS, so it uses the identity sum_j P_ij (dO_i . v_j) = dO_i . O_i and
    takes D_i = rowsum(dO o O) over the forward output as stored (rounded to
    the output dtype).  Passing that array here evaluates the same formula;
    None (the default) keeps the exact D.  dV does not involve D.
    Returns (dQ, dK, dV, D).
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    s = score_matrix(q, k, scale, causal)
    P, L, _, _ = _softmax_rows(s)
    # P_ij = exp(s_ij - L_i): the same weights section 7 reconstructs.
    dV = P.T @ do
    dP = do @ v.T
    D = (P * dP).sum(axis=1) if o_stored is None else (do * _f64(o_stored)).sum(axis=1)
    dS = P * (dP - D[:, None])
    dQ = scale * (dS @ k)
    dK = scale * (dS.T @ q)
    return dQ, dK, dV, D


# --------------------------------------------------------------------------
# Batched layouts.  Dense tensors are [B, H, N, D] (tensortonic.com
# "FlashAttention" section 9: [batch, heads, tokens, head_width]).  Packed
# variable-length batches are [H, T, D] with sequence s occupying tokens
# cu_seqlens[s] : cu_seqlens[s+1] of every head and attending only within
# itself (nexusofnerds.com "FlashAttention": variable-length packing).
# --------------------------------------------------------------------------

def forward(q, k, v, scale, causal):
    """Dense [B, H, N, D] forward: (O [B,H,N,D], L [B,H,N])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, D = q.shape
    O = np.zeros((B, H, N, v.shape[-1]))
    L = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            O[b, h], L[b, h] = forward_head(q[b, h], k[b, h], v[b, h], scale, causal)
    return O, L


def backward(q, k, v, do, scale, causal, o_stored=None):
    """Dense [B, H, N, D] backward: (dQ, dK, dV, D).  ``o_stored`` as for
    backward_head ([B, H, N, D] or None)."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, H, N, _ = q.shape
    dQ = np.zeros_like(q)
    dK = np.zeros_like(k)
    dV = np.zeros_like(v)
    Dv = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            dQ[b, h], dK[b, h], dV[b, h], Dv[b, h] = backward_head(
                q[b, h], k[b, h], v[b, h], do[b, h], scale, causal,
                None if o_stored is None else o_stored[b, h])
    return dQ, dK, dV, Dv


# --------------------------------------------------------------------------
# Attention dropout (tensortonic.com "FlashAttention" section 7: with dropout
# the backward must reproduce the forward's dropout decisions from saved
# random-number-generator information rather than sample a new mask).
#
# The decisions come from the counter-based generator Philox4x32-10 (Salmon,
# Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011),
# so any element's decision can be regenerated from (seed, position) alone:
# element (i, j) of head bh (= b * H + h) takes 32-bit word j mod 4 of
# Philox4x32-10 with counter (floor(j / 4), i, bh, offset) and key
# (seed mod 2^32, seed div 2^32); it is kept iff word / 2^32 >= p.  Kept
# weights are scaled by 1 / (1 - p): O = (P o Z) V / (1 - p).  L is that of the
# undropped softmax.
# --------------------------------------------------------------------------

_PHILOX_M0, _PHILOX_M1 = 0xD2511F53, 0xCD9E8D57       # round multipliers
_PHILOX_W0, _PHILOX_W1 = 0x9E3779B9, 0xBB67AE85       # key increments (Weyl sequence)


def philox4x32_10(counter, key):
    """Philox4x32 with 10 rounds.  counter: four uint32 arrays (broadcastable),
    key: two uint32 values.  Each round multiplies words 0 and 2 by the round
    multipliers into 64-bit products, and the new words are
    (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0));
    the key is then advanced by the two increments.  Returns four uint32 arrays."""
    c = [np.asarray(x, dtype=np.uint64) & 0xFFFFFFFF for x in counter]
    k0, k1 = int(key[0]) & 0xFFFFFFFF, int(key[1]) & 0xFFFFFFFF
    mask = np.uint64(0xFFFFFFFF)
    for _ in range(10):
        p0 = np.uint64(_PHILOX_M0) * c[0]
        p1 = np.uint64(_PHILOX_M1) * c[2]
        c = [(p1 >> np.uint64(32)) ^ c[1] ^ np.uint64(k0), p1 & mask,
             (p0 >> np.uint64(32)) ^ c[3] ^ np.uint64(k1), p0 & mask]
        k0 = (k0 + _PHILOX_W0) & 0xFFFFFFFF
        k1 = (k1 + _PHILOX_W1) & 0xFFFFFFFF
    return [x.astype(np.uint32) for x in c]


def dropout_keep(nq, nk, bh, p, seed, offset):
    """Keep mask Z [nq, nk] (bool) of head bh for query rows 0..nq-1 and keys
    0..nk-1, as described above."""
    i = np.arange(nq, dtype=np.uint64)[:, None]
    j = np.arange(nk, dtype=np.uint64)[None, :]
    words = philox4x32_10((j >> np.uint64(2), i, np.uint64(bh), np.uint64(offset & 0xFFFFFFFF)),
                          (seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF))
    sel = (j & np.uint64(3)).astype(np.int64)
    w = np.choose(np.broadcast_to(sel, (nq, nk)), [np.broadcast_to(x, (nq, nk)) for x in words])
    return w.astype(np.float64) / 2.0**32 >= p


def forward_head_dropout(q, k, v, scale, causal, p, keep):
    """(O, L) with dropout on the attention weights: O = (P o Z) V / (1 - p)."""
    s = score_matrix(q, k, scale, causal)
    P, L, _, _ = _softmax_rows(s)
    return (P * keep / (1.0 - p)) @ _f64(v), L


def backward_head_dropout(q, k, v, do, scale, causal, p, keep, o_stored=None):
    """Gradients with dropout.  With M = Z / (1 - p) and P~ = P o M:
    dV = P~^T dO, dP = (dO V^T) o M, D_i = sum_j P_ij dP_ij (= dO_i . O_i),
    dS = P o (dP - D), dQ = scale dS K, dK = scale dS^T Q.  ``o_stored``
    (the dropped output as stored) replaces D as in backward_head."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    s = score_matrix(q, k, scale, causal)
    P, _, _, _ = _softmax_rows(s)
    M = keep / (1.0 - p)
    dV = (P * M).T @ do
    dP = (do @ v.T) * M
    D = (P * dP).sum(axis=1) if o_stored is None else (do * _f64(o_stored)).sum(axis=1)
    dS = P * (dP - D[:, None])
    return scale * (dS @ k), scale * (dS.T @ q), dV, D


def forward_dropout(q, k, v, scale, causal, p, seed, offset):
    """Dense [B, H, N, D] forward with dropout."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, _ = q.shape
    O = np.zeros((B, H, N, v.shape[-1]))
    L = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            keep = dropout_keep(N, N, b * H + h, p, seed, offset)
            O[b, h], L[b, h] = forward_head_dropout(q[b, h], k[b, h], v[b, h], scale, causal, p, keep)
    return O, L


def backward_dropout(q, k, v, do, scale, causal, p, seed, offset, o_stored=None):
    """Dense [B, H, N, D] backward with dropout: (dQ, dK, dV, D)."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, H, N, _ = q.shape
    dQ, dK, dV = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    Dv = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            keep = dropout_keep(N, N, b * H + h, p, seed, offset)
            dQ[b, h], dK[b, h], dV[b, h], Dv[b, h] = backward_head_dropout(
                q[b, h], k[b, h], v[b, h], do[b, h], scale, causal, p, keep,
                None if o_stored is None else o_stored[b, h])
    return dQ, dK, dV, Dv


# --------------------------------------------------------------------------
# Cached decoding: nq new queries against nk keys and values already in the
# cache (tensortonic.com "FlashAttention" section 8: a cached generation step
# may have a single new query and a long set of past keys and values; section
# 9: the newest query must be aligned with its actual position in the key
# cache, so the square causal mask does not apply when the lengths differ).
# --------------------------------------------------------------------------

def cached_score_matrix(q, k, scale, causal):
    """S = scale * Q K^T for nq queries that are the last nq positions of an
    nk-long sequence: query i sits at position nk - nq + i, so causal allows
    key j iff j <= i + (nk - nq) (the mask aligned at the bottom right).  For
    nq == nk this is score_matrix's square mask.  When nq > nk the first
    nq - nk rows have no allowed key.  Masked entries are -inf.
    """
    q = _f64(q)
    k = _f64(k)
    s = scale * (q @ k.T)
    if causal:
        nq, nk = s.shape
        i = np.arange(nq)[:, None]
        j = np.arange(nk)[None, :]
        s = np.where(j <= i + (nk - nq), s, -np.inf)
    return s


def forward_cached_head(q, k, v, scale, causal):
    """One head of a cached decoding step: (O [nq, d], L [nq]), by the same
    definition as forward_head (softmax of the masked scores, times V);
    rows without an allowed key get O = 0, L = -inf."""
    s = cached_score_matrix(q, k, scale, causal)
    P, L, _, _ = _softmax_rows(s)
    return P @ _f64(v), L


def forward_cached(q, k, v, scale, causal):
    """Dense cached step: q [B, H, nq, D], k and v [B, H, nk, D] ->
    (O [B, H, nq, D], L [B, H, nq])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, nq, _ = q.shape
    O = np.zeros((B, H, nq, v.shape[-1]))
    L = np.zeros((B, H, nq))
    for b in range(B):
        for h in range(H):
            O[b, h], L[b, h] = forward_cached_head(q[b, h], k[b, h], v[b, h], scale, causal)
    return O, L


def _segments(cu_seqlens):
    cu = [int(x) for x in np.asarray(cu_seqlens).reshape(-1)]
    return [(cu[s], cu[s + 1]) for s in range(len(cu) - 1)]


def forward_varlen(q, k, v, cu_seqlens, scale, causal, heads=None):
    """Packed [H, T, D] forward: (O [H,T,D], L [H,T]); each sequence alone.

    ``heads`` optionally restricts the work to a subset of heads (rows of the
    other heads are left as NaN)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    H, T, _ = q.shape
    O = np.full((H, T, v.shape[-1]), np.nan)
    L = np.full((H, T), np.nan)
    for h in (range(H) if heads is None else heads):
        for a, b in _segments(cu_seqlens):
            if b > a:
                O[h, a:b], L[h, a:b] = forward_head(q[h, a:b], k[h, a:b], v[h, a:b], scale, causal)
    return O, L


def backward_varlen(q, k, v, do, cu_seqlens, scale, causal, heads=None, o_stored=None):
    """Packed [H, T, D] backward: (dQ, dK, dV, D); each sequence alone.
    ``o_stored`` ([H, T, D] or None) as for backward_head."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    H, T, _ = q.shape
    dQ = np.full(q.shape, np.nan)
    dK = np.full(k.shape, np.nan)
    dV = np.full(v.shape, np.nan)
    Dv = np.full((H, T), np.nan)
    for h in (range(H) if heads is None else heads):
        for a, b in _segments(cu_seqlens):
            if b > a:
                dQ[h, a:b], dK[h, a:b], dV[h, a:b], Dv[h, a:b] = backward_head(
                    q[h, a:b], k[h, a:b], v[h, a:b], do[h, a:b], scale, causal,
                    None if o_stored is None else o_stored[h, a:b])
    return dQ, dK, dV, Dv


# --------------------------------------------------------------------------
# Row-subset forms for sequences too long for an n x n float64 matrix.  Each
# output row of attention depends on its own query row only, so a sampled row
# is computed exactly as in forward_head, one row at a time, in O(n d).
# --------------------------------------------------------------------------

def _row_scores(q, k, i, scale, causal):
    lim = i + 1 if causal else k.shape[0]
    return scale * (k[:lim] @ q[i]), lim


def forward_rows(q, k, v, rows, scale, causal):
    """(O [len(rows), d], L [len(rows)]) for the given query rows of one head."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    O = np.zeros((len(rows), v.shape[1]))
    L = np.zeros(len(rows))
    for r, i in enumerate(rows):
        s, lim = _row_scores(q, k, i, scale, causal)
        m = s.max()
        e = np.exp(s - m)
        l = e.sum()
        L[r] = m + np.log(l)
        O[r] = (e / l) @ v[:lim]
    return O, L


def backward_dq_rows(q, k, v, do, rows, scale, causal):
    """dQ rows of one head.  Row i of dQ needs only row i of P and dP and D_i
    (same algebra as backward_head, restricted to one row)."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    dQ = np.zeros((len(rows), q.shape[1]))
    for r, i in enumerate(rows):
        s, lim = _row_scores(q, k, i, scale, causal)
        m = s.max()
        e = np.exp(s - m)
        p = e / e.sum()
        dp = v[:lim] @ do[i]
        Di = (p * dp).sum()
        ds = p * (dp - Di)
        dQ[r] = scale * (ds @ k[:lim])
    return dQ


def backward_head_blocked(q, k, v, do, scale, causal, rows_per_block=512):
    """backward_head for long sequences without holding an n x n matrix.

    Rows of S, P, dP and dS are independent, and dK, dV are sums over rows, so
    the rows are visited in blocks; every quantity is the one backward_head
    defines.  Also returns O and L of the same head (forward_head, by rows).
    Returns (O, L, dQ, dK, dV).
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    n = q.shape[0]
    O = np.zeros_like(v[:n])
    L = np.zeros(n)
    dQ = np.zeros_like(q)
    dK = np.zeros_like(k)
    dV = np.zeros_like(v)
    for r0 in range(0, n, rows_per_block):
        r1 = min(n, r0 + rows_per_block)
        kmax = r1 if causal else k.shape[0]   # keys beyond r1 are masked for every row here
        s = scale * (q[r0:r1] @ k[:kmax].T)
        if causal:
            i = np.arange(r0, r1)[:, None]
            j = np.arange(kmax)[None, :]
            s = np.where(j <= i, s, -np.inf)
        P, Lb, _, _ = _softmax_rows(s)
        O[r0:r1] = P @ v[:kmax]
        L[r0:r1] = Lb
        dP = do[r0:r1] @ v[:kmax].T
        Db = (P * dP).sum(axis=1)
        dS = P * (dP - Db[:, None])
        dQ[r0:r1] = scale * (dS @ k[:kmax])
        dK[:kmax] += scale * (dS.T @ q[r0:r1])
        dV[:kmax] += P.T @ do[r0:r1]
    return O, L, dQ, dK, dV


# --------------------------------------------------------------------------
# The method's own algorithm, step by step, in the pages' order.  Used only to
# pin the printed worked example and to show the tiled schedule is exact; the
# GPU path is compared with the plain definitions above.
# --------------------------------------------------------------------------

def online_softmax_row(scores, values, tiles):
    """Running softmax over one query row, tile by tile.

    tensortonic.com "FlashAttention" section 5 (and the online-softmax block of
    wiki.ai-engineering.at "Flash Attention", Trick: Numerical Stability with
    Softmax, read per row with a vector accumulator): keep the largest score
    seen so far m, the sum of shifted exponentials l and the weighted value sum
    u.  When a tile raises the maximum, both sums are multiplied by
    exp(m_old - m_new); the tile's exponentials are then added on the new
    scale.  The output is u / l and L = m + log(l) (section 7).

    ``tiles`` is a list of (start, stop) index pairs covering the row.
    ``values`` is [n, d] (or [n] for scalar values).
    Returns (out, L, states) where states lists (m, l) after every tile.
    """
    scores = _f64(scores)
    values = _f64(values)
    m = -np.inf
    l = 0.0
    u = np.zeros(values.shape[1:])
    states = []
    for a, b in tiles:
        s = scores[a:b]
        m_new = max(m, s.max())
        rescale = np.exp(m - m_new) if np.isfinite(m) else 0.0
        e = np.exp(s - m_new)
        l = rescale * l + e.sum()
        u = rescale * u + e @ values[a:b]
        m = m_new
        states.append((m, l))
    return u / l, m + np.log(l), states


def tiled_forward_head(q, k, v, scale, causal, br, bc):
    """The query-first tiled forward schedule of tensortonic.com
    "FlashAttention" section 6, for one head.

    For each block of ``br`` query rows: start one running state per row;
    visit the key/value blocks of ``bc`` keys in turn, skipping blocks wholly
    in the future of every row of the block when causal (section 6, last
    paragraph); mask element by element on blocks that cross the diagonal;
    fold each block into the running state (section 5); finally divide by the
    denominator.  wiki.ai-engineering.at's printed tiling loop applies a
    softmax per tile and sums the results, which section 4 shows is wrong; it
    is not followed.
    Returns (O, L).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    n, nk = q.shape[0], k.shape[0]
    O = np.zeros((n, v.shape[1]))
    L = np.zeros(n)
    for r0 in range(0, n, br):
        r1 = min(n, r0 + br)
        rows = np.arange(r0, r1)
        m = np.full(r1 - r0, -np.inf)
        l = np.zeros(r1 - r0)
        u = np.zeros((r1 - r0, v.shape[1]))
        for c0 in range(0, nk, bc):
            c1 = min(nk, c0 + bc)
            if causal and c0 > r1 - 1:
                break                      # this and every later block is in the future
            s = scale * (q[r0:r1] @ k[c0:c1].T)
            if causal and c1 - 1 > r0:     # block crosses the diagonal: element mask
                cols = np.arange(c0, c1)
                s = np.where(cols[None, :] <= rows[:, None], s, -np.inf)
            m_new = np.maximum(m, s.max(axis=1))
            rescale = np.where(np.isfinite(m), np.exp(m - m_new), 0.0)
            e = np.exp(s - m_new[:, None])
            l = rescale * l + e.sum(axis=1)
            u = rescale[:, None] * u + e @ v[c0:c1]
            m = m_new
        O[r0:r1] = u / l[:, None]
        L[r0:r1] = m + np.log(l)
    return O, L
