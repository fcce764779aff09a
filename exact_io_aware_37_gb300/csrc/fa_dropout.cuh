// Attention dropout decisions, regenerated wherever they are needed
// (tensortonic.com "FlashAttention" section 7: the backward pass must
// reproduce the forward pass's dropout decisions from saved random-number-
// generator information instead of sampling a new mask).
//
// The generator is Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random
// numbers: as easy as 1, 2, 3", SC 2011), a counter-based generator: the
// decision for element (i, j) of head bh = b * H + h is word j mod 4 of
// Philox4x32-10 applied to counter (j / 4, i, bh, offset) under key
// (seed mod 2^32, seed / 2^32), and the element is kept iff that word is at
// least thr = ceil(p * 2^32) (i.e. word / 2^32 >= p).  Kept weights are
// multiplied by 1 / (1 - p).  i and j count from the start of the element's
// own sequence.
#pragma once

#include <stdint.h>

#include "fa_internal.cuh"

namespace fa {

struct DropParams {
  uint32_t thr;      // keep iff word >= thr
  float scale;       // 1 / (1 - p)
  uint32_t offset;
  // The key of round r: (seed mod 2^32, seed / 2^32) advanced r times by the
  // Weyl increments.  It is the same for every thread, so it is worked out
  // once on the host and read as a kernel-parameter operand.
  uint32_t rk0[10], rk1[10];
};

// Ten rounds; each multiplies words 0 and 2 by the round multipliers into
// 64-bit products and forms (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1,
// lo(M0 c0)) with the round's key (k0, k1).
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, const DropParams& d) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
    c = make_uint4(hi1 ^ c.y ^ d.rk0[r], lo1, hi0 ^ c.w ^ d.rk1[r], lo0);
  }
  return c;
}

// Keep bits (bit t for key j0 + t) of keys j0 .. j0 + 3 (j0 a multiple of 4)
// for query row i: one generator call.
__device__ __forceinline__ uint32_t keep4(const DropParams& d, uint32_t i, uint32_t j0, uint32_t bh) {
  const uint4 w = philox4x32_10(make_uint4(j0 >> 2, i, bh, d.offset), d);
  return (w.x >= d.thr ? 1u : 0u) | (w.y >= d.thr ? 2u : 0u) | (w.z >= d.thr ? 4u : 0u) | (w.w >= d.thr ? 8u : 0u);
}

// Keep bits (bit c for query q0 + c, c < 64) of this thread's key `key` when
// keys sit on the lanes of a warp and lanes 4m .. 4m+3 hold keys 4m' .. 4m'+3
// (key = 4 * (key / 4) + lane % 4).  The four lanes sharing key / 4 need the
// four words of the same generator call for each query, so each of them
// computes the calls for a quarter of the queries (q = q0 + 4g + lane % 4):
// call g's four decisions (bit k: key 4 * (key / 4) + k) form nibble g of a
// 64-bit word, and the quad exchanges whole words -- lane t takes bit t of
// every nibble of lane s's word, which is the decision for its key at query
// q0 + 4g + s.  Four pairs of shuffles and a few shifts per 64 decisions, no
// per-decision selects or variable shifts.  All 32 lanes must call this.
__device__ __forceinline__ uint64_t keep64_keys_on_lanes(const DropParams& d, uint32_t key, uint32_t q0,
                                                         uint32_t bh, int lane) {
  const uint32_t t = lane & 3;
  const int quad_base = lane & ~3;
  uint64_t nibs = 0;  // nibble g at bits 4g .. 4g + 3
#pragma unroll 4
  for (int g = 0; g < 16; ++g) {
    const uint4 w = philox4x32_10(make_uint4(key >> 2, q0 + 4 * g + t, bh, d.offset), d);
    const uint32_t nib = (w.x >= d.thr ? 1u : 0u) | (w.y >= d.thr ? 2u : 0u) | (w.z >= d.thr ? 4u : 0u) |
                         (w.w >= d.thr ? 8u : 0u);
    nibs |= (uint64_t)nib << (4 * g);
  }
  const uint32_t lo = (uint32_t)nibs, hi = (uint32_t)(nibs >> 32);
  uint64_t bits = 0;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const uint64_t word = (uint64_t)__shfl_sync(0xffffffffu, hi, quad_base | s) << 32 |
                          __shfl_sync(0xffffffffu, lo, quad_base | s);
    bits |= ((word >> t) & 0x1111111111111111ull) << s;
  }
  return bits;
}

inline DropParams drop_params_of(const Problem& p) {
  DropParams d;
  d.thr = p.drop_thr;
  d.scale = p.drop_scale;
  d.offset = p.drop_offset;
  uint32_t k0 = (uint32_t)(p.drop_seed & 0xffffffffu), k1 = (uint32_t)(p.drop_seed >> 32);
  for (int r = 0; r < 10; ++r, k0 += 0x9E3779B9u, k1 += 0xBB67AE85u) {
    d.rk0[r] = k0;
    d.rk1[r] = k1;
  }
  return d;
}

}  // namespace fa
