"""Inputs whose running row maximum rises in later key tiles.

The method keeps, per query row, the largest score seen so far and rescales
its running sums by exp(m_old - m_new) whenever a later tile brings a larger
one (tensortonic.com "FlashAttention", sections 4 and 5).  The tensor-core
forward does this lazily: it keeps a reference maximum and multiplies the
accumulator in tensor memory only when a tile's maximum exceeds that
reference by more than 2^8 (8 in log2 units); otherwise the tile's weights
are formed against the old reference and may reach 2^8.  i.i.d. N(0, 1)
inputs put a row's first-tile maximum near 2.6 natural units and almost
never exceed it by 5.5 later, so they never take that branch.

These inputs do, on purpose and in a controlled way.  Channel 0 of Q holds a
per-row gain a_i, channel 0 of K a per-key level b_j that depends only on the
key's 128-key tile within its sequence; the other channels are the usual
seeded N(0, 1) draws (K's scaled by ``sigma_k``).  Score (i, j) is then
scale * (a_i b_j + noise), so a row with a_i > 0 sees its maximum step up by
``step_log2`` (log2 units) wherever the level steps up.

Level profiles (key tile t of n_t in the sequence):
  ramp  level t        -- a rise at every tile; causal rows peak on the diagonal
  jump  level [t >= n_t // 2]  -- one rise in the middle of the key range
  last  level [t == n_t - 1]   -- one rise in the last (possibly ragged) tile
  stairs level t // 8   -- a rise every 8 tiles (long sequences: the planted
                           values stay small, see below)
Row patterns (gain of row i, i counted within its sequence):
  mixed       GAIN, 0, -GAIN for i mod 3 = 0, 1, 2 (rising, flat and falling
              rows side by side in every warp)
  even_tiles  GAIN in even 128-row query tiles, 0 in odd ones
  odd_tiles   GAIN in odd query tiles, 0 in even ones

The planted channel makes the keys (queries) share a large common component,
which magnifies in dQ (dK) two roundings the 16-bit backward makes by design:
D_i = rowsum(dO o O) over the stored 16-bit O, and dS rounded to 16 bits
before the dQ / dK products.  The tests therefore take dQ and dK from the
oracle evaluated with the same D (its own O rounded to the dtype), and keep
the planted values moderate (a ramp over at most 5 tiles, stairs beyond).

Nothing here is attention arithmetic: the oracle computes the expected
outputs; ``lazy_rescale_events`` only replays the kernel's rescale decision on
the oracle's score matrix, so a test can show which branch its inputs take.
"""

import math

import numpy as np
import torch

from exact_io_aware_37_gb300 import synth

TILE = 128
GAIN = 4.0
THRESHOLD_LOG2 = 8.0


def _levels(n, profile):
    t = np.arange(n) // TILE
    n_t = max(1, (n + TILE - 1) // TILE)
    if profile == "ramp":
        return t.astype(np.float64)
    if profile == "jump":
        return (t >= n_t // 2).astype(np.float64)
    if profile == "last":
        return (t == n_t - 1).astype(np.float64)
    if profile == "stairs":
        return (t // 8).astype(np.float64)
    raise ValueError(profile)


def _gains(n, rows):
    i = np.arange(n)
    if rows == "mixed":
        return np.choose(i % 3, [GAIN, 0.0, -GAIN])
    tile_odd = (i // TILE) % 2 == 1
    if rows == "even_tiles":
        return np.where(tile_odd, 0.0, GAIN)
    if rows == "odd_tiles":
        return np.where(tile_odd, GAIN, 0.0)
    raise ValueError(rows)


def dense(shape, dtype, scale, profile, step_log2, rows="mixed", sigma_k=1.0, seed_offset=0):
    """CPU (q, k, v, dO) [B, H, N, D] with the planted channel 0."""
    B, H, N, D = shape
    q, k, v, do = synth.qkv_do(shape, torch.float32, seed_offset=seed_offset)
    k[..., 1:] *= sigma_k
    delta_b = step_log2 * math.log(2.0) / (scale * GAIN)   # key-level step for a rise of step_log2
    q[..., :, 0] = torch.as_tensor(_gains(N, rows), dtype=torch.float32)
    k[..., :, 0] = torch.as_tensor(_levels(N, profile) * delta_b, dtype=torch.float32)
    return tuple(x.to(dtype) for x in (q, k, v, do))


def packed(lengths, H, D, dtype, scale, profile, step_log2, rows="mixed", sigma_k=1.0, seed_offset=0):
    """CPU (q, k, v, dO) [H, T, D] and cu_seqlens; every sequence gets its own
    levels and gains, counted from its first token."""
    cu = synth.cu_seqlens(lengths)
    T = int(cu[-1])
    q, k, v, do = synth.qkv_do((H, T, D), torch.float32, seed_offset=seed_offset)
    k[..., 1:] *= sigma_k
    delta_b = step_log2 * math.log(2.0) / (scale * GAIN)
    for s in range(len(lengths)):
        a, b = int(cu[s]), int(cu[s + 1])
        if b == a:
            continue
        q[:, a:b, 0] = torch.as_tensor(_gains(b - a, rows), dtype=torch.float32)
        k[:, a:b, 0] = torch.as_tensor(_levels(b - a, profile) * delta_b, dtype=torch.float32)
    return tuple(x.to(dtype) for x in (q, k, v, do)) + (cu,)


def lazy_rescale_events(scores_nat):
    """Replay the lazy rule on one head's score matrix (natural units, masked
    entries -inf): for every row, walk the 128-key tiles in order, keep a
    reference maximum m_ref (log2 units) that moves only when a tile's maximum
    exceeds it by more than THRESHOLD_LOG2.  Returns (fired, peak): fired[i]
    counts the tiles after the first in which row i moved its reference (the
    accumulator rescale), peak[i] is the largest weight 2^(s - m_ref) the row
    formed in any tile (at most 2^8 by construction of the rule)."""
    s = np.asarray(scores_nat, dtype=np.float64) / math.log(2.0)
    n, nk = s.shape
    fired = np.zeros(n, dtype=np.int64)
    peak = np.zeros(n)
    for i in range(n):
        m_ref = -np.inf
        for j, c0 in enumerate(range(0, nk, TILE)):
            tile = s[i, c0:c0 + TILE]
            mt = tile.max()
            if mt == -np.inf:
                continue
            if mt > m_ref + THRESHOLD_LOG2:
                if j > 0 and m_ref != -np.inf:
                    fired[i] += 1
                m_ref = mt
            peak[i] = max(peak[i], 2.0 ** (mt - m_ref))
    return fired, peak


def cached(B, H, nq, nk, D, dtype, scale, profile, step_log2, rows="mixed", sigma_k=1.0, seed_offset=0):
    """CPU (q [B,H,nq,D], k, v [B,H,nk,D]) for a cached decoding step: the
    levels follow the cache's 128-key tiles, the gains the new query rows."""
    q = synth.normal((B, H, nq, D), synth.SEED_Q + seed_offset, torch.float32)
    k = synth.normal((B, H, nk, D), synth.SEED_K + seed_offset, torch.float32)
    v = synth.normal((B, H, nk, D), synth.SEED_V + seed_offset, torch.float32)
    k[..., 1:] *= sigma_k
    delta_b = step_log2 * math.log(2.0) / (scale * GAIN)
    q[..., :, 0] = torch.as_tensor(_gains(nq, rows), dtype=torch.float32)
    k[..., :, 0] = torch.as_tensor(_levels(nk, profile) * delta_b, dtype=torch.float32)
    return tuple(x.to(dtype) for x in (q, k, v))


# The cases the GPU tests run and the CPU test checks the premise of.
# expect "fires": some row moves its reference maximum after its first tile
#   (the accumulator rescale runs); "below": no row does, but weights formed
#   against the old reference reach above 2^7.
STEP_UP, NEAR_ABOVE, NEAR_BELOW = 12.0, 8.7, 7.3
QUIET_K = 0.05  # K noise scale that keeps the rises within ~0.2 of their step

# (profile, step_log2, rows, sigma_k, shape [B, H, N, D], causal, expect)
DENSE_CASES = [
    ("ramp", STEP_UP, "mixed", 1.0, (1, 2, 600, 128), False, "fires"),
    ("ramp", STEP_UP, "mixed", 1.0, (1, 2, 600, 128), True, "fires"),
    ("ramp", STEP_UP, "mixed", 1.0, (1, 2, 600, 64), False, "fires"),
    ("ramp", STEP_UP, "mixed", 1.0, (1, 2, 600, 64), True, "fires"),
    ("jump", STEP_UP, "even_tiles", 1.0, (1, 2, 600, 128), False, "fires"),
    ("jump", STEP_UP, "odd_tiles", 1.0, (1, 2, 600, 128), True, "fires"),
    ("last", STEP_UP, "odd_tiles", 1.0, (1, 2, 600, 64), False, "fires"),
    ("last", STEP_UP, "even_tiles", 1.0, (1, 2, 600, 64), True, "fires"),
    ("jump", NEAR_ABOVE, "mixed", QUIET_K, (1, 2, 600, 128), False, "fires"),
    ("ramp", NEAR_BELOW, "mixed", QUIET_K, (1, 2, 600, 128), True, "fires"),
    ("jump", NEAR_BELOW, "mixed", QUIET_K, (1, 2, 600, 128), False, "below"),
    ("jump", NEAR_BELOW, "mixed", QUIET_K, (1, 2, 600, 64), True, "below"),
    ("last", NEAR_BELOW, "mixed", QUIET_K, (1, 2, 600, 64), False, "below"),
    ("ramp", STEP_UP, "mixed", 1.0, (2, 3, 1000, 64), True, "fires"),
    ("stairs", STEP_UP, "mixed", 1.0, (1, 2, 4096, 128), True, "fires"),
]

PACKED_LENGTHS = [300, 700, 129, 1, 0, 520]
# (profile, step_log2, rows, sigma_k, H, D, causal, expect)
PACKED_CASES = [
    ("ramp", STEP_UP, "mixed", 1.0, 2, 64, False, "fires"),
    ("ramp", STEP_UP, "mixed", 1.0, 2, 64, True, "fires"),
    ("ramp", STEP_UP, "mixed", 1.0, 2, 128, False, "fires"),
    ("ramp", STEP_UP, "mixed", 1.0, 2, 128, True, "fires"),
    ("jump", NEAR_BELOW, "mixed", QUIET_K, 2, 128, True, "below"),
]


def case_id(case):
    return "-".join(str(x).replace(" ", "") for x in case[:-1]).replace("(", "").replace(")", "").replace(",", "x")
