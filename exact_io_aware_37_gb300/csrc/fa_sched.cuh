// Work lists of the persistent tensor-core launches (host and device code).
//
// The pages hand every tile to its own thread block and let the blocks run in
// parallel (tensortonic.com "FlashAttention", section 6).  Here one CTA per
// SM works through a list of items instead, so its launch, tensor-memory
// allocation and pipeline fill are paid once and one item's epilogue
// overlaps the next item's loads.  An item is a pair of 128-row query tiles
// (forward) or one 128-key tile (backward) of one (sequence, head) unit.
//
// Two forms of list:
//   table        dense inputs whose items fit the kernel parameters (at most
//                4096): the host lists the items heaviest first inside
//                groups of heads and gives each to the CTA with the least work
//                so far (longest processing time first).
//   closed form  everything else (more items, or packed sequences whose
//                lengths live on the device): unit u = b * H + h; the units
//                are cut into groups of `per` (the last one may be smaller);
//                inside a group, rank r numbers a unit's items heaviest first
//                (causal) and the group's items run rank-major (all its units'
//                heaviest items first); virtual item f counts the groups' items
//                one group after the other.  CTA c takes f = k * n_ctas + c
//                (round robin) or, with `snake`, f = k * n_ctas + n_ctas - 1 - c
//                for odd k (which evens out the per-pass differences of a list
//                sorted by weight), skipping the ranks its unit's sequence does
//                not have.  The forward runs all units as one group with the
//                snake; the backward, whose units each stream Q, dO and a dQ
//                accumulator, groups a few units so the operands in use stay in
//                L2.  Every role of a CTA walks the same list from (CTA, k)
//                alone.
#pragma once

#include <stdint.h>

namespace fa {

constexpr int kSchedTile = 128;  // rows of a query tile and keys of a key tile

// A host table groups heads only so that the operands the items of the heads
// in flight re-read stay in L2; when those operands of all heads together take
// at most this many bytes (well inside the 129 MB L2), the table is one group:
// heaviest items first across all heads, which the least-loaded assignment
// balances best.
constexpr long long kSchedL2GroupBytes = 48ll << 20;

// 32-bit arithmetic throughout (a 64-bit division is a called routine on the
// GPU, which costs the register-starved roles a stack frame): the host only
// builds closed-form lists of at most kMaxVirtualItems virtual items.
constexpr uint32_t kMaxVirtualItems = 1u << 31;

struct ClosedSpec {
  uint32_t n_virtual;  // n_units * ranks
  uint32_t n_units;    // B * H
  uint32_t per;        // units per group (the last group may hold fewer)
  uint32_t ranks;      // items per unit of the longest sequence
  uint32_t n_ctas;
  uint32_t snake;      // 1: snake order over the CTAs, 0: round robin
};

// Virtual item of pass k of CTA `cta` (>= n_virtual: the CTA's list has ended;
// no overflow, since k * n_ctas <= n_virtual + n_ctas < 2^32).
__host__ __device__ __forceinline__ uint32_t closed_item(const ClosedSpec& s, uint32_t cta, uint32_t k) {
  return k * s.n_ctas + ((s.snake && (k & 1u)) ? (s.n_ctas - 1u - cta) : cta);
}

// Unit and rank of virtual item f.
__host__ __device__ __forceinline__ void closed_unit_rank(const ClosedSpec& s, uint32_t f, uint32_t& unit,
                                                          uint32_t& rank) {
  const uint32_t group_items = s.per * s.ranks;
  const uint32_t g = f / group_items;
  const uint32_t r = f - g * group_items;
  const uint32_t left = s.n_units - g * s.per;
  const uint32_t in_group = left < s.per ? left : s.per;
  rank = r / in_group;
  unit = g * s.per + (r - rank * in_group);
}

// Units per group for about `target` units per group (the group count is
// rounded up and the units spread evenly, so no group is left nearly empty).
inline uint32_t closed_group_size(uint32_t n_units, uint32_t target) {
  const uint32_t n_groups = (n_units + target - 1) / target;
  return (n_units + n_groups - 1) / n_groups;
}

// Forward: the pair (query tiles 2p, 2p + 1) of rank r in a sequence of `len`
// rows, or -1 when the sequence has fewer pairs.  With the mask, pairs of late
// query tiles see the most keys and come first.
__host__ __device__ __forceinline__ int fwd_pair_of_rank(int len, int r, int causal) {
  const int n_qt = (len + kSchedTile - 1) / kSchedTile, n_pairs = (n_qt + 1) / 2;
  if (r >= n_pairs) return -1;
  return causal ? n_pairs - 1 - r : r;
}

// Backward: the key tile of rank r in a sequence of `len` keys, or -1.  With
// the mask, early key tiles meet the most query tiles and come first.
__host__ __device__ __forceinline__ int bwd_tile_of_rank(int len, int r) {
  const int n_kt = (len + kSchedTile - 1) / kSchedTile;
  return r < n_kt ? r : -1;
}

// Ranks per unit for a maximum sequence length of N rows.
inline int fwd_ranks(int N) { return ((N + kSchedTile - 1) / kSchedTile + 1) / 2; }
inline int bwd_ranks(int N) { return (N + kSchedTile - 1) / kSchedTile; }

}  // namespace fa
