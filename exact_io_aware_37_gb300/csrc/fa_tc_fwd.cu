// Tensor-core forward kernel for sm_103a (bf16 in, fp32 accumulate).
//
// The method is the query-first tiled schedule of tensortonic.com
// "FlashAttention" section 6 with the running softmax of section 5: a CTA
// works on two 128-row query tiles of one (sequence, head) at a time (a
// pair), loads them once, and visits the allowed 128-key K/V tiles in turn;
// it is persistent and works through a list of pairs (see FwdSched).  The
// score tile and the output accumulator never leave the SM: S = Q K^T and u += P V are tcgen05
// MMAs whose accumulators live in tensor memory (TMEM), and only O = u / l and
// L = m + log(l) are written to device memory (section 7).
//
// Warp roles (12 warps; warps 10-11 only complete the third warpgroup):
//   warps 0-3  softmax for query tile 0, warps 4-7 for query tile 1: one
//              thread per query row (its TMEM lane), so row max and row sum
//              are thread-local; exp2 of scores pre-scaled by scale*log2(e);
//              P is rounded to bf16 and written back into the score columns.
//              The same threads rescale their accumulator row when the
//              running maximum grows by more than 2^8 (a lazy rescale: the
//              final u / l uses the same reference maximum, so it is exact),
//              and run the epilogue.
//   The softmax warpgroups raise their register limit to 200 and the third
//   warpgroup lowers its to 104 (setmaxnreg) so the 128 scores of a row stay
//   in registers.
//   warp 8     TMA producer: Q tiles once, then K_j / V_j into rings of
//              shared-memory stages.  A stage is handed back by the softmax
//              thread that sees the last query tile's S(j) complete (every
//              MMA issued before it is then complete too), so K runs a step
//              ahead of V and the MMA thread commits nothing for it.
//   warp 9     MMA issuer (one thread): S_t = Q_t K_j^T, then, once the
//              softmax of tile t has produced P_t, O_t += P_t V_j, then the
//              next S_t.  The two query tiles alternate so the tensor core
//              works on one tile while the other tile's softmax runs.
// Causal: key tiles wholly in the future of a query tile are never loaded;
// the diagonal tile (and the ragged last tile of a sequence) gets an
// element-wise mask (section 6).  Packed variable-length batches use the
// same kernel with per-sequence row ranges from cu_seqlens.
//
// TMEM columns (512 allocated): S_0 [0,128), S_1 [128,256), O_0 [256,256+D),
// O_1 [384,384+D); P_t (bf16 pairs) overwrites S_t columns [0,64).
#include <math.h>

#include <algorithm>
#include <mutex>
#include <queue>
#include <vector>

#include "fa_dropout.cuh"
#include "fa_internal.cuh"
#include "fa_sched.cuh"
#include "fa_tmap.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

using namespace ptx;

constexpr int kBM = 128;              // query rows per tile
constexpr int kBN = 128;              // keys per tile
constexpr int kThreads = 384;  // 2 softmax warpgroups + 1 support warpgroup
constexpr int kTmaWarp = 8;
constexpr int kMmaWarp = 9;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when the max grows by > 2^8
constexpr int kFwdHeadGroup = 16;  // heads per group of the causal block order (measured best of 8..64)

// Each CTA of the (always persistent) launch walks a list of query-tile pairs
// (fa_sched.cuh): the CTA launch, tensor-memory allocation and first loads are
// paid once per CTA and a pair's epilogue overlaps the next pair's loads.
// Dense inputs of at most kMaxSchedItems pairs get a host-built table (the
// causal heavy-first order inside groups of heads, each pair to the CTA with
// the least work so far); larger and packed inputs the closed-form list.
constexpr int kMaxSchedCtas = 160;
constexpr int kMaxSchedItems = 4096;
constexpr int kSchedTable = 0, kSchedClosed = 1;

struct FwdSched {
  int n_ctas;                       // CTAs of the launch
  int mode;                         // kSchedTable or kSchedClosed
  int n_pairs;                      // table: pairs per (b, h)
  uint32_t n_virtual;               // closed form: (B * H) * ranks
  uint32_t per, ranks, snake;       // closed form: units per group, pairs per unit, CTA order
  uint16_t off[kMaxSchedCtas + 1];  // table: CTA c works on item[off[c] .. off[c + 1])
  uint32_t item[kMaxSchedItems];    // table: (b * H + h) * n_pairs + pair
};

struct FwdParams {
  CUtensorMap tq, tk, tv;
  DropParams drop;  // used by the dropout instantiation only
  __nv_bfloat16* o;  // 16-bit storage: bf16 or fp16 per F16
  float* lse;
  const int32_t* cu;
  unsigned* status;
  unsigned long long limit_ns;
  int B, H, N, T;
  float c2;  // scale * log2(e)
  int causal;
  FwdSched sched;
};

template <int D>
struct FwdCfg {
  static constexpr int kStages = D == 64 ? 4 : 2;
  static constexpr int kTileBytes = kBM * D * 2;  // one Q, K or V tile
  static constexpr int kHalves = D / 64;          // 64-column (128-byte) swizzle blocks
  static constexpr int kHalfBytes = kBM * 128;    // 16 KB
  static constexpr int kQOff = 0;
  static constexpr int kKOff = 2 * kTileBytes;
  static constexpr int kVOff = kKOff + kStages * kTileBytes;
  static constexpr int kSmemBytes = kVOff + kStages * kTileBytes + 1024;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

template <int D, bool F16, bool kDrop>
__global__ void __launch_bounds__(kThreads, 1) tc_fwd_kernel(const __grid_constant__ FwdParams p) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  // bar_q: a pair's Q tiles (the first pair's also K_0); bar_kv[g % stages]: V_g and
  // K_{g+1} (the two loads one stage release allows, so the MMA thread waits once
  // per step for its operands; K_{g+1} may be the next pair's K_0).  Steps g are
  // counted over all of the CTA's pairs, so every ring and per-step barrier keeps
  // its phase from one pair to the next.
  __shared__ __align__(8) uint64_t bar_q, bar_qfree, bar_done;
  __shared__ __align__(8) uint64_t bar_kv[C::kStages], bar_kfree[C::kStages], bar_vfree[C::kStages];
  __shared__ __align__(8) uint64_t bar_s[2], bar_p[2], bar_epi[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- the query-tile pairs this CTA works on
  struct Pair {
    int b, h, len, row0, slab, qt0, nkv0, nkv1, nmax, t_last;
    long long out_base;
  };
  const bool table = p.sched.mode == kSchedTable;
  const int first_item = table ? p.sched.off[blockIdx.x] : 0;
  const int n_table = table ? p.sched.off[blockIdx.x + 1] - first_item : 0;
  const ClosedSpec closed{p.sched.n_virtual, (uint32_t)p.B * (uint32_t)p.H, p.sched.per, p.sched.ranks,
                          (uint32_t)p.sched.n_ctas, p.sched.snake};
  // steps of the two query tiles of pair `pair` of q's sequence
  auto set_geometry = [&](Pair& q, int pair) {
    const int n_qt = (q.len + kBM - 1) / kBM;
    const int n_kv = (q.len + kBN - 1) / kBN;
    q.qt0 = 2 * pair;
    q.nkv0 = p.causal ? min(q.qt0 + 1, n_kv) : n_kv;
    q.nkv1 = q.qt0 + 1 < n_qt ? (p.causal ? min(q.qt0 + 2, n_kv) : n_kv) : 0;
    q.nmax = max(q.nkv0, q.nkv1);
    q.t_last = q.nkv1 > 0 ? 1 : 0;  // its MMAs are issued last in every step; its count is nmax
  };
  // The CTA's next pair after list position k (k moves past it); false once
  // the list has ended.  Every role walks the same list.
  auto next_pair = [&](uint32_t& k, Pair& q) -> bool {
    if (table) {  // dense: every listed pair is in range
      if (k >= (uint32_t)n_table) return false;
      const uint32_t code = p.sched.item[first_item + (int)k++];
      const int bh = (int)(code / (uint32_t)p.sched.n_pairs);
      const int pair = (int)(code - (uint32_t)bh * (uint32_t)p.sched.n_pairs);
      q.b = bh / p.H;
      q.h = bh - q.b * p.H;
      q.len = p.N;
      q.row0 = 0;
      q.slab = bh;
      q.out_base = (long long)bh * p.N;
      set_geometry(q, pair);
      return true;
    }
    for (;;) {
      const uint32_t f = closed_item(closed, blockIdx.x, k);
      if (f >= closed.n_virtual) return false;
      ++k;
      uint32_t uu, rr;
      closed_unit_rank(closed, f, uu, rr);
      const int r = (int)rr, u = (int)uu;
      q.b = u / p.H;
      q.h = u - q.b * p.H;
      if (p.cu != nullptr) {
        const int s0 = p.cu[q.b], s1 = p.cu[q.b + 1];
        if (s0 < 0 || s1 < s0 || s1 > p.T || s1 - s0 > p.N) {  // skipped and reported
          if (threadIdx.x == 0) atomicOr(p.status, kDevBadSeqlens);
          continue;
        }
        q.len = s1 - s0;
        q.row0 = s0;
        q.slab = q.h;
        q.out_base = (long long)q.h * p.T + s0;
      } else {
        q.len = p.N;
        q.row0 = 0;
        q.slab = u;
        q.out_base = (long long)u * p.N;
      }
      const int pair = fwd_pair_of_rank(q.len, r, p.causal);
      if (pair < 0) continue;  // the sequence has fewer pairs
      set_geometry(q, pair);
      return true;
    }
  };
  {
    uint32_t k0 = 0;
    Pair first;
    if (!next_pair(k0, first)) return;  // nothing for this CTA
  }

  if (threadIdx.x == 0) {
    mbar_init(&bar_q, 1);
    mbar_init(&bar_qfree, 1);
    mbar_init(&bar_done, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bar_kv[s], 1);
      mbar_init(&bar_kfree[s], 1);
      mbar_init(&bar_vfree[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bar_s[t], 1);
      mbar_init(&bar_p[t], 4);    // one arrival per softmax warp
      mbar_init(&bar_epi[t], 4);  // the tile's softmax warps have seen its last P V complete
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&tmem_base_sh, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const WaitCtx w{&abort_flag, p.status, p.limit_ns};

  if (warp < 8) {
    // ------------------------------------------------------------ softmax / epilogue
    setmaxnreg_inc<kComputeRegs>();
    const int t = warp >> 2;
    const int quad = warp & 3;          // TMEM lanes 32*quad .. 32*quad+31
    const int r = quad * 32 + lane;     // row within the query tile
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t t_s = tmem + lane_off + t * 128;
    const uint32_t t_o = tmem + lane_off + 256 + t * 128;
    bool ok = true;
    int G = 0;   // steps of the earlier pairs
    int cs = 0;  // completions of bar_s[t] seen so far
    uint32_t cur = 0;
    Pair q;
    while (ok && next_pair(cur, q)) {
      const int n = t == 0 ? q.nkv0 : q.nkv1;
      const int len = q.len;
      if (n > 0) {
        const int qt = q.qt0 + t;
        const int i = qt * kBM + r;       // row within the sequence
        float m_ref = -INFINITY;          // reference maximum of the exponentials (log2 units)
        float l = 0.f;
        for (int j = 0; j < n; ++j) {
          const int g = G + j;
          // dropout: the tile's keep decisions (bit k of kw[x]: key j * kBN + 32 x + k)
          // depend on positions alone, so they are drawn before S is ready: 32
          // independent generator calls the warp interleaves while the MMA runs
          // (eight calls a pass; the passes rotate their words through kw, so no
          // index is dynamic)
          uint32_t kw[4] = {0u, 0u, 0u, 0u};
          if constexpr (kDrop) {
            const uint32_t bh = (uint32_t)(q.b * p.H + q.h);
#pragma unroll 1
            for (int x = 0; x < 4; ++x) {
              uint32_t word = 0;
#pragma unroll
              for (int gk = 0; gk < 8; ++gk)
                word |= keep4(p.drop, (uint32_t)i, (uint32_t)(j * kBN + 32 * x + 4 * gk), bh) << (4 * gk);
              kw[0] = kw[1];
              kw[1] = kw[2];
              kw[2] = kw[3];
              kw[3] = word;
            }
          }
          if (!warp_wait(&bar_s[t], cs & 1, w)) {
            ok = false;
            break;
          }
          ++cs;
          if (t == q.t_last && quad == 0 && lane == 0) {
            // S_t(j) of the last query tile is complete, and with it every MMA issued
            // before it: S_0(j) (K_g is consumed), both tiles' P V of the step before
            // (V_{g-1}, possibly the previous pair's last V) and, at the pair's last
            // step, every S of the pair (its Q tiles are free)
            mbar_arrive(&bar_kfree[g % C::kStages]);
            if (g > 0) mbar_arrive(&bar_vfree[(g - 1) % C::kStages]);
            if (j == n - 1) mbar_arrive(&bar_qfree);
          }
          tc_fence_after();
          uint32_t sr[4][32];
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32(t_s + c * 32, sr[c]);
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld_wait(sr[c]);
          const int k0 = j * kBN;
          if ((p.causal && j == qt) || (k0 + kBN > len)) {
            // diagonal or ragged tile: keys [k0, k0 + kmax) are allowed, the rest get -inf
            const int kmax = min(len, p.causal ? i + 1 : len) - k0;
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
              for (int e = 0; e < 32; ++e)
                if (c * 32 + e >= kmax) sr[c][e] = __float_as_uint(-INFINITY);
          }
          // row maximum of the raw scores (scale > 0 preserves the order), as eight
          // independent partial maxima so that the exponentials wait for a chain of
          // 11 dependent steps instead of 64 (the maximum is exact in any order)
          float mp[8];
#pragma unroll
          for (int r = 0; r < 8; ++r) mp[r] = -INFINITY;
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 32; e += 2)
              mp[(e >> 1) & 7] = fmax3(mp[(e >> 1) & 7], __uint_as_float(sr[c][e]), __uint_as_float(sr[c][e + 1]));
          const float mt = fmaxf(fmax3(mp[0], mp[1], mp[2]), fmax3(fmax3(mp[3], mp[4], mp[5]), mp[6], mp[7]));
          const float m_new = fmaxf(m_ref, mt * p.c2);
          float alpha = 1.f;
          const bool grow = m_new > m_ref + kRescaleThreshold;
          if (grow) {
            alpha = (m_ref == -INFINITY) ? 0.f : ex2_approx(m_ref - m_new);
            m_ref = m_new;
            l *= alpha;
          }
          const float nmu = (m_ref == -INFINITY) ? 0.f : -m_ref;
          // p = 2^(s * scale * log2(e) - m_ref), two columns per packed FMA
          float rs0 = 0.f, rs1 = 0.f;
          // P goes to tensor memory in parts of kPer packed columns (quarters with
          // dropout, whose keep words take registers the halves would need)
          constexpr int kParts = kDrop ? 4 : 2, kPer = kBN / 2 / kParts;
#pragma unroll
          for (int hf = 0; hf < kParts; ++hf) {
            uint32_t pk[kPer];
#pragma unroll
            for (int c = 0; c < kPer; ++c) {
              const int e0 = 2 * kPer * hf + 2 * c;
              float a0, a1;
              ffma2(a0, a1, __uint_as_float(sr[e0 >> 5][e0 & 31]), __uint_as_float(sr[(e0 + 1) >> 5][(e0 + 1) & 31]),
                    p.c2, nmu, nmu);
              const float p0 = ex2_approx(a0);
              const float p1 = ex2_approx(a1);
              fadd2(rs0, rs1, p0, p1);  // the normaliser is that of the undropped weights
              if constexpr (kDrop) {
                // dropped weights enter PV scaled by 1 / (1 - p)
                const uint32_t kb = kw[e0 >> 5] >> (e0 & 31);
                pk[c] = pack16x2<F16>(kb & 1u ? p0 * p.drop.scale : 0.f, kb & 2u ? p1 * p.drop.scale : 0.f);
              } else {
                pk[c] = pack16x2<F16>(p0, p1);
              }
            }
            if constexpr (kPer == 32)
              tmem_st32(t_s + 32 * hf, pk);
            else
              tmem_st16(t_s + 16 * hf, pk);
          }
          l += rs0 + rs1;
          if (j > 0 && __any_sync(0xffffffffu, grow)) {
            // accumulator rows rescaled in place: the previous PV is complete (the
            // wait on bar_s covers it) and this tile's PV waits for bar_p below
#pragma unroll 1
            for (int c = 0; c < D; c += 32) {
              uint32_t o[32];
              tmem_ld32(t_o + c, o);
              tmem_ld_wait(o);
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
              tmem_st32(t_o + c, o);
            }
          }
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar_p[t]);
        }
        if (ok && warp_wait(&bar_s[t], cs & 1, w)) {
          ++cs;
          // the tile's last P V is complete: the MMA thread may start the next
          // pair's S over this tile's score columns
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar_epi[t]);
          tc_fence_after();
          const bool row_ok = i < len;
          const float inv = l > 0.f ? 1.f / l : 0.f;
          if constexpr (kDrop || D == 64) {
            // row-per-lane stores: with dropout the exchange's registers would spill
            // next to the keep words (and the generator bounds that forward anyway);
            // at D = 64 the exchange's latency outweighs the store lines it saves
            // (measured)
            __nv_bfloat16* orow = p.o + (q.out_base + i) * D;
#pragma unroll 1
            for (int c = 0; c < D; c += 32) {
              uint32_t o[32];
              tmem_ld32(t_o + c, o);
              tmem_ld_wait(o);
              if (row_ok) {
                uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
                for (int v4 = 0; v4 < 4; ++v4) {
                  uint4 u;
                  u.x = pack16x2<F16>(__uint_as_float(o[8 * v4 + 0]) * inv, __uint_as_float(o[8 * v4 + 1]) * inv);
                  u.y = pack16x2<F16>(__uint_as_float(o[8 * v4 + 2]) * inv, __uint_as_float(o[8 * v4 + 3]) * inv);
                  u.z = pack16x2<F16>(__uint_as_float(o[8 * v4 + 4]) * inv, __uint_as_float(o[8 * v4 + 5]) * inv);
                  u.w = pack16x2<F16>(__uint_as_float(o[8 * v4 + 6]) * inv, __uint_as_float(o[8 * v4 + 7]) * inv);
                  dst[v4] = u;
                }
              }
            }
          } else {
            // 64 columns at a time: read out, normalised and packed by the row's own
            // thread, then an 8 x 8 exchange of 16-byte chunks inside groups of eight
            // lanes gives each store instruction four whole 128-byte row segments
            // (one line each, instead of one line per lane)
            const int grp = lane & ~7, sub = lane & 7;
#pragma unroll 1
            for (int c = 0; c < D; c += 64) {
              uint32_t pk[32];
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                uint32_t o[32];
                tmem_ld32(t_o + c + 32 * h, o);
                tmem_ld_wait(o);
#pragma unroll
                for (int e = 0; e < 16; ++e)
                  pk[16 * h + e] = pack16x2<F16>(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
              }
              exchange_chunks<8>(pk, lane);
              // slot s now holds chunk `sub` of row grp + s of this warp's 32
#pragma unroll
              for (int s8 = 0; s8 < 8; ++s8) {
                const int row = qt * kBM + quad * 32 + grp + s8;
                if (row < len)
                  *reinterpret_cast<uint4*>(p.o + (q.out_base + row) * D + c + sub * 8) =
                      make_uint4(pk[4 * s8], pk[4 * s8 + 1], pk[4 * s8 + 2], pk[4 * s8 + 3]);
              }
            }
          }
          if (row_ok) p.lse[q.out_base + i] = l > 0.f ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
        } else {
          ok = false;
        }
      }
      G += q.nmax;
    }
  } else {
    // warps 8-11: producer, MMA issuer and two idle warps completing the warpgroup
    setmaxnreg_dec<kSupportRegs>();
    if (warp == kTmaWarp && lane == 0) {
      // ---------------------------------------------------------- producer
      tma_prefetch_desc(&p.tq);
      tma_prefetch_desc(&p.tk);
      tma_prefetch_desc(&p.tv);
      auto load_q = [&](const Pair& q, int extra) {
        const int nq = q.nkv1 > 0 ? 2 : 1;
        mbar_arrive_expect_tx(&bar_q, (nq + extra) * C::kTileBytes);
        for (int t = 0; t < nq; ++t)
          for (int hf = 0; hf < C::kHalves; ++hf)
            tma_load_3d(smem + C::kQOff + t * C::kTileBytes + hf * C::kHalfBytes, &p.tq, &bar_q, hf * 64,
                        q.row0 + (q.qt0 + t) * kBM, q.slab);
      };
      auto load_k = [&](const Pair& q, int j, int g, uint64_t* bar) {
        for (int hf = 0; hf < C::kHalves; ++hf)
          tma_load_3d(smem + C::kKOff + (g % C::kStages) * C::kTileBytes + hf * C::kHalfBytes, &p.tk, bar, hf * 64,
                      q.row0 + j * kBN, q.slab);
      };
      // Stage release: the softmax thread that waits for the last query tile's
      // S(g) arrives on kfree[g % stages] (K_g consumed: S_0 precedes S_1) and on
      // vfree[(g-1) % stages] (both P V of step g - 1 precede S_1(g)).  V_g and
      // K_{g+1} both need the release of step g + 1 - stages, so they share one
      // barrier, and K runs a step ahead of V without costing the MMA thread a
      // commit.  A pair's Q tiles go out once the previous pair's every S is
      // complete (qfree).  Each wait below is unambiguous: the next completion of
      // the barrier it polls needs a load issued after the wait.
      int issued = 0, q_issued = 0, G = 0;
      bool good = true;
      uint32_t cur = 0;
      Pair q, nx;
      next_pair(cur, q);  // the CTA has at least one pair
      load_q(q, 1);
      load_k(q, 0, 0, &bar_q);
      q_issued = 1;
      bool have = true;
      for (int ii = 0; good && have; ++ii) {
        const bool has_next = next_pair(cur, nx);
        for (int j = 0; j < q.nmax; ++j) {
          const int g = G + j;
          const int s = g % C::kStages;
          // K_{g+1}: this pair's next K, or the next pair's K_0
          const bool k_next = j + 1 < q.nmax || has_next;
          if (g >= C::kStages && !mbar_wait(&bar_vfree[s], (g / C::kStages - 1) & 1, w)) {
            good = false;
            break;
          }
          if (k_next && g + 1 >= C::kStages &&
              !mbar_wait(&bar_kfree[(g + 1) % C::kStages], ((g + 1) / C::kStages - 1) & 1, w)) {
            good = false;
            break;
          }
          mbar_arrive_expect_tx(&bar_kv[s], (k_next ? 2 : 1) * C::kTileBytes);
          for (int hf = 0; hf < C::kHalves; ++hf)
            tma_load_3d(smem + C::kVOff + s * C::kTileBytes + hf * C::kHalfBytes, &p.tv, &bar_kv[s], hf * 64,
                        q.row0 + j * kBN, q.slab);
          if (k_next) {
            if (j + 1 < q.nmax)
              load_k(q, j + 1, g + 1, &bar_kv[s]);
            else
              load_k(nx, 0, g + 1, &bar_kv[s]);
          }
          issued = g + 1;
        }
        if (!good) break;
        G += q.nmax;
        if (has_next) {
          // the next pair's Q tiles over this pair's, once every S of this pair is complete
          if (!mbar_wait(&bar_qfree, ii & 1, w)) break;
          load_q(nx, 0);
          q_issued = ii + 2;
        }
        q = nx;
        have = has_next;
      }
      if (abort_flag) {
        // let copies already in flight land before the CTA's memory is released
        if (q_issued > 0) mbar_wait_drain(&bar_q, (q_issued - 1) & 1, p.limit_ns);
        for (int g = max(0, issued - C::kStages); g < issued; ++g)
          mbar_wait_drain(&bar_kv[g % C::kStages], (g / C::kStages) & 1, p.limit_ns);
      }
    } else if (warp == kMmaWarp && lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      const uint32_t id_s = idesc16<F16>(kBM, kBN, false, false);
      const uint32_t id_o = idesc16<F16>(kBM, D, false, true);
      // Descriptors are built once and advanced by adding (byte offset >> 4)
      // to their start-address field.
      const uint64_t dq0 = sdesc_sw128(smem_u32(smem + C::kQOff), 16, 1024);
      const uint64_t dk0 = sdesc_sw128(smem_u32(smem + C::kKOff), 16, 1024);
      const uint64_t dv0 = sdesc_sw128(smem_u32(smem + C::kVOff), C::kHalfBytes, 1024);
      // S_t = Q_t K^T (both K-major): D/16 MMAs of K = 16, issued back to back
      auto issue_s = [&](int t, int s) {
        const uint64_t a0 = dq0 + ((t * C::kTileBytes) >> 4);
        const uint64_t b0 = dk0 + ((s * C::kTileBytes) >> 4);
        if constexpr (D == 128) {
          uint64_t a[8], b[8];
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t off = ((ks >> 2) * C::kHalfBytes + (ks & 3) * 32) >> 4;
            a[ks] = a0 + off;
            b[ks] = b0 + off;
          }
          mma_ss_x8(tmem + t * 128, a, b, id_s, 0u);
        } else {
          uint64_t a[4], b[4];
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            a[ks] = a0 + ks * 2;
            b[ks] = b0 + ks * 2;
          }
          mma_ss_x4(tmem + t * 128, a, b, id_s, 0u);
        }
      };
      // O_t += P_t V (P from TMEM, V MN-major): 8 MMAs of K = 16 keys
      auto issue_pv = [&](int t, int s, bool acc) {
        const uint64_t b0 = dv0 + ((s * C::kTileBytes) >> 4);
        uint32_t a[8];
        uint64_t b[8];
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          a[ks] = tmem + t * 128 + ks * 8;
          b[ks] = b0 + ((ks * 2048) >> 4);
        }
        mma_ts_x8(tmem + 256 + t * 128, a, b, id_o, acc ? 1u : 0u);
      };
      bool ok = true;
      int G = 0;
      int cp[2] = {0, 0};    // completions of bar_p[t] waited for
      int used[2] = {0, 0};  // pairs that used query tile t so far
      uint32_t cur = 0;
      Pair q;
      for (int ii = 0; ok && next_pair(cur, q); ++ii) {
        // the pair's step counts (the rest of its geometry is not needed here)
        const int nk[2] = {q.nkv0, q.nkv1};
        const int nmax = max(nk[0], nk[1]);
        // Q tiles (and, for the first pair, K_0; later pairs' K_0 came with the
        // previous pair's last V, whose barrier was waited for); each tile's S goes
        // over score columns its softmax warps must have finished with
        ok = mbar_wait(&bar_q, ii & 1, w);
        if (!ok) break;
        tc_fence_after();
        for (int t = 0; t < 2; ++t) {
          if (nk[t] == 0) continue;
          if (used[t] > 0 && !mbar_wait(&bar_epi[t], (used[t] - 1) & 1, w)) {
            ok = false;
            break;
          }
          ++used[t];
          tc_fence_after();
          issue_s(t, G % C::kStages);
          mma_commit(&bar_s[t]);
        }
        for (int j = 0; ok && j < nmax; ++j) {
          const int g = G + j;
          const int s = g % C::kStages, s1 = (g + 1) % C::kStages;
          // V_g and K_{g+1}
          if (!mbar_wait(&bar_kv[s], (g / C::kStages) & 1, w)) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int t = 0; t < 2; ++t) {
            if (j >= nk[t]) continue;
            if (!mbar_wait(&bar_p[t], cp[t] & 1, w)) {
              ok = false;
              break;
            }
            ++cp[t];
            tc_fence_after();
            issue_pv(t, s, j > 0);
            if (j + 1 < nk[t]) issue_s(t, s1);
            mma_commit(&bar_s[t]);
          }
        }
        G += nmax;
      }
      // every MMA issued must be complete before tensor memory is released
      mma_commit(&bar_done);
      mbar_wait_drain(&bar_done, 0, p.limit_ns);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
}

// Per-pair cost, in steps, of what a persistent CTA does besides the pair's
// steps (waiting for its Q tiles, the epilogue); it only steers the balance.
constexpr int kPairOverheadSteps = 1;

// The work list for at most `ctas_max` CTAs: the table for dense inputs with
// at most kMaxSchedItems pairs, the closed-form list otherwise; false when
// there is nothing to do.
bool fill_fwd_sched(const Problem& p, int ctas_max, FwdSched& sc) {
  sc.n_ctas = 0;
  const int n_qt = (p.N + kBM - 1) / kBM, n_kv = (p.N + kBN - 1) / kBN;
  const int n_pairs = (n_qt + 1) / 2;
  const long long n_bh = (long long)p.B * p.H;
  const long long n = n_bh * n_pairs;
  if (n <= 0 || ctas_max <= 0) return false;
  sc.n_pairs = n_pairs;
  if (p.cu != nullptr || n > kMaxSchedItems) {
    sc.mode = kSchedClosed;
    const long long v = n_bh * fwd_ranks(p.N);
    if (v > (long long)kMaxVirtualItems) return false;
    sc.n_virtual = (uint32_t)v;
    sc.per = (uint32_t)n_bh;  // one group: every unit's heaviest pairs first
    sc.ranks = (uint32_t)fwd_ranks(p.N);
    sc.snake = 1;
    sc.n_ctas = (int)std::min<long long>(v, ctas_max);
    return true;
  }
  sc.mode = kSchedTable;
  sc.n_virtual = (uint32_t)n;
  const int ctas = (int)std::min<long long>(n, std::min(ctas_max, kMaxSchedCtas));
  // Pairs in the order the grid used: with the mask, heaviest first inside
  // balanced groups of kFwdHeadGroup heads (the order of grouped_heavy_first),
  // or of all heads when their K and V fit in L2 together.
  std::vector<uint32_t> order((size_t)n);
  std::vector<int> weight((size_t)n);
  const long long head_bytes = 4ll * p.N * p.D;  // K and V (16-bit)
  const long long group_heads = n_bh * head_bytes <= kSchedL2GroupBytes ? n_bh : (long long)kFwdHeadGroup;
  const long long n_groups = (n_bh + group_heads - 1) / group_heads;
  const long long per = (n_bh + n_groups - 1) / n_groups;
  for (long long f = 0; f < n; ++f) {
    long long bh, pair;
    if (p.causal) {
      const long long group = f / (per * n_pairs), r = f - group * per * n_pairs;
      const long long heads = std::min(per, n_bh - group * per);
      bh = group * per + r % heads;
      pair = n_pairs - 1 - r / heads;
    } else {
      bh = f / n_pairs;
      pair = f % n_pairs;
    }
    order[(size_t)f] = (uint32_t)(bh * n_pairs + pair);
    const int steps = p.causal ? std::min((int)(2 * pair + 2), n_kv) : n_kv;
    weight[(size_t)f] = steps + kPairOverheadSteps;
  }
  // Each pair to the CTA with the least work so far (lowest index on ties).
  using Slot = std::pair<long long, int>;
  std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap;
  for (int c = 0; c < ctas; ++c) heap.push({0, c});
  std::vector<std::vector<uint32_t>> lists((size_t)ctas);
  for (long long f = 0; f < n; ++f) {
    Slot t = heap.top();
    heap.pop();
    lists[(size_t)t.second].push_back(order[(size_t)f]);
    t.first += weight[(size_t)f];
    heap.push(t);
  }
  int at = 0;
  for (int c = 0; c < ctas; ++c) {
    sc.off[c] = (uint16_t)at;
    for (uint32_t code : lists[(size_t)c]) sc.item[at++] = code;
  }
  sc.off[ctas] = (uint16_t)at;
  sc.n_ctas = ctas;
  return true;
}

// The schedule of a launch on the current device (one CTA per SM), cached for
// the last problem shape.
bool build_fwd_sched(const Problem& p, FwdSched& sc) {
  const int ctas = sm_count();
  static std::mutex mu;
  static long long key[6] = {-1, -1, -1, -1, -1, -1};
  static FwdSched cached;
  const long long want[6] = {p.B, p.H, p.N, p.D, p.causal, ctas};  // the table's head groups depend on D
  if (p.cu != nullptr) return fill_fwd_sched(p, ctas, sc);  // closed form: nothing to cache
  std::lock_guard<std::mutex> lock(mu);
  if (std::equal(want, want + 6, key)) {
    sc = cached;
    return true;
  }
  if (!fill_fwd_sched(p, ctas, sc)) return false;
  cached = sc;
  std::copy(want, want + 6, key);
  return true;
}

template <int D, bool F16, bool kDrop>
cudaError_t launch_fwd_d(const Problem& p, cudaStream_t s) {
  using C = FwdCfg<D>;
  static FwdParams fp;  // large (the schedule); filled in full below on every call
  static std::mutex launch_mu;
  std::lock_guard<std::mutex> launch_lock(launch_mu);
  if (!make_map16(&fp.tq, p.q, p, kBM) || !make_map16(&fp.tk, p.k, p, kBN) ||
      !make_map16(&fp.tv, p.v, p, kBN))
    return note_error("forward tensor map encode", cudaErrorInvalidValue);
  fp.o = static_cast<__nv_bfloat16*>(p.o);
  fp.lse = p.lse;
  fp.cu = p.cu;
  fp.status = p.status;
  fp.limit_ns = p.wait_limit_ns;
  fp.B = p.B;
  fp.H = p.H;
  fp.N = p.N;
  fp.T = p.T;
  fp.c2 = p.scale * kLog2e;
  fp.causal = p.causal;
  fp.drop = drop_params_of(p);
  cudaError_t e = cudaFuncSetAttribute(tc_fwd_kernel<D, F16, kDrop>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return note_error("forward smem attribute", e);
  if (!build_fwd_sched(p, fp.sched)) return note_error("forward schedule (no multiprocessor count, or more than 2^31 work items)", cudaErrorInvalidValue);
  tc_fwd_kernel<D, F16, kDrop><<<fp.sched.n_ctas, kThreads, C::kSmemBytes, s>>>(fp);
  note_launches(1);
  return note_error("forward launch", cudaGetLastError());
}

}  // namespace

int preview_fwd_schedule(const Problem& p, const int32_t* cu_host, int ctas, int* off, uint32_t* items, int cap,
                         int* form) {
  static FwdSched sc;  // large; previews are a host-side test aid
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (!fill_fwd_sched(p, ctas, sc)) return -1;
  *form = sc.mode;
  if (sc.mode == kSchedTable) {
    const int n = sc.off[sc.n_ctas];
    if (n > cap) return -2;
    for (int c = 0; c <= sc.n_ctas; ++c) off[c] = sc.off[c];
    std::copy(sc.item, sc.item + n, items);
    return n;
  }
  // the closed form, walked exactly as the kernel's roles walk it
  const ClosedSpec closed{sc.n_virtual, (uint32_t)p.B * (uint32_t)p.H, sc.per, sc.ranks, (uint32_t)sc.n_ctas,
                          sc.snake};
  const int ranks = fwd_ranks(p.N);
  int n = 0;
  for (int c = 0; c < sc.n_ctas; ++c) {
    off[c] = n;
    for (uint32_t k = 0;; ++k) {
      const uint32_t f = closed_item(closed, (uint32_t)c, k);
      if (f >= closed.n_virtual) break;
      uint32_t uu, rr;
      closed_unit_rank(closed, f, uu, rr);
      const int r = (int)rr, u = (int)uu;
      int len = p.N;
      if (cu_host != nullptr) {
        const int b = u / p.H, s0 = cu_host[b], s1 = cu_host[b + 1];
        if (s0 < 0 || s1 < s0 || s1 > p.T || s1 - s0 > p.N) continue;
        len = s1 - s0;
      }
      const int pair = fwd_pair_of_rank(len, r, p.causal);
      if (pair < 0) continue;
      if (n >= cap) return -2;
      items[n++] = (uint32_t)((long long)u * ranks + pair);
    }
  }
  off[sc.n_ctas] = n;
  return n;
}

cudaError_t launch_tc_fwd(const Problem& p, cudaStream_t s) {
  if (p.dropout) {
    if (p.D == 64) return p.f16 ? launch_fwd_d<64, true, true>(p, s) : launch_fwd_d<64, false, true>(p, s);
    if (p.D == 128) return p.f16 ? launch_fwd_d<128, true, true>(p, s) : launch_fwd_d<128, false, true>(p, s);
  } else {
    if (p.D == 64) return p.f16 ? launch_fwd_d<64, true, false>(p, s) : launch_fwd_d<64, false, false>(p, s);
    if (p.D == 128) return p.f16 ? launch_fwd_d<128, true, false>(p, s) : launch_fwd_d<128, false, false>(p, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace fa
