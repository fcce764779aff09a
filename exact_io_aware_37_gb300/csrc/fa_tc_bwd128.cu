// Tensor-core backward kernel for head width 128 (sm_103a, bf16 in, fp32
// accumulate).
//
// Same method as the D = 64 kernel (tensortonic.com "FlashAttention",
// section 7: every weight is rebuilt as P_ij = exp(s_ij - L_i) from the
// saved log-sum-exp; dV = P^T dO, dS = P o (dO V^T - D), dK = scale dS^T Q,
// dQ = scale dS K): a CTA holds one 128-key tile of K and V in shared memory
// at a time and visits the 128-query tiles that can see it; every launch is
// persistent: one CTA per SM takes key tiles one after another (see BwdSched)
// and hands each to its roles through a ring in shared memory.  All five
// products are
// tcgen05 MMAs with M = N = 128, placed in tensor memory as
//     [0,128)   S^T = K Q^T, then P^T (bf16) over its columns [0,32) and [64,96)
//     [128,256) dP^T = V dO^T, then dS^T (bf16) over [128,160) and [192,224),
//               then dQ^T = K^T dS^T (head width on lanes)
//     [256,384) dV += P^T dO        (A = P^T from tensor memory)
//     [384,512) dK += dS^T Q        (A = dS^T from tensor memory)
// dQ^T also needs dS^T as an MN-major shared-memory operand, so the compute
// warps write it to both places.  The MMA order per step k is
//     dP^T_k [after dQ^T_{k-1} is out], dV_k, S^T_{k+1}, dK_k, dQ^T_k
// and the compute warps work through
//     P^T_k, read out dQ^T_{k-1}, dS^T_k
// so dP^T_k is formed while they copy dQ^T_{k-1} to shared memory, and the
// next step's S^T while they build dS^T_k.
//
// Warp roles (12 warps): 0-3 and 4-7 compute P^T and dS^T for query columns
// [0,64) and [64,128), and copy dQ^T for the same query columns out of
// tensor memory into shared memory (half 0 into the dS^T buffer, which is
// free between dQ^T_k and dS^T_{k+1}; half 1 into a buffer of its own);
// 8 = TMA / L / D producer; 9 = MMA issuer; 10 = dQ reducer: it has the copy
// engine add both halves into the float32 accumulator
// (cp.reduce.async.bulk) and hands the buffers back once they have been
// read; 11 idle.  A CTA can push only about 24 bytes per clock of
// reductions out to L2, so the 64 KB of dQ per step are the backward's
// other bound besides the tensor core; the compute warps therefore never
// wait for a reduction except to reuse the dS^T buffer, and they form dS^T
// in registers before that wait.
// Registers: 168 per thread at launch, then 184 for the two compute
// warpgroups and 136 for the producer / MMA warpgroup (setmaxnreg).
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

constexpr int kTile = 128;  // keys per CTA and queries per step
constexpr int kBwdHeadGroup = 4;  // heads per group of the causal block order: Q, dO and the dQ
                                   // accumulator of a head take 4 MB at N = 4096 (measured best of 2..32)
constexpr int kThreads = 384;
constexpr int kTmaWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kReduceWarp = 10;
// D = 128: half 0 of a step's dQ is staged and reduced as two 16 KB pieces
// (query rows 0-31 and 32-63), each of which overlays one query half of the
// dS^T buffer, so the copy engine starts on the first piece while the second is
// still being written, and each half of the next dS^T waits only for its own
// piece to be read.
constexpr bool kH0Pieces = true;
// setmaxnreg split of the kLaunchRegs budget: the MMA issuer keeps five groups of
// eight descriptors in flight and needs more than the forward's support share
constexpr int kBwdComputeRegs = 184;
constexpr int kBwdSupportRegs = 136;
static_assert(2 * 128 * kBwdComputeRegs + 128 * kBwdSupportRegs <= kThreads * kLaunchRegs,
              "register split exceeds the launch budget");

// Each CTA of the (always persistent) launch works through key tiles
// (b, h, kt) one after another, so a CTA launch, tensor-memory allocation and
// pipeline fill are paid once and the next tile's loads and first products
// overlap the previous tile's last reductions and its dK / dV stores.  The
// producer warp takes the tiles and hands each to the other roles through a
// ring of kItemRing records in shared memory (bar_item / bar_itemfree), then
// an end record.  Where it takes them from:
//   table    dense inputs of at most kMaxSchedItems tiles: a list per CTA
//            worked out on the host -- items in the causal heavy-first order
//            inside groups of heads, each to the CTA with the least work so
//            far (longest processing time first);
//   queue    larger and packed inputs: a counter in the caller's workspace
//            (zeroed by the preprocess kernel) over the same order, written
//            in closed form over virtual items (fa_sched.cuh: groups of about
//            kBwdHeadGroup (sequence, head) units, rank-major inside a group,
//            ranks a sequence does not have skipped by the producer).  CTAs
//            take the next tile when they need one, as the block scheduler
//            would, so the tiles in flight stay a contiguous stretch of the
//            order (their operands stay in L2) and no CTA runs out of work
//            early.
constexpr int kMaxSchedCtas = 160;
constexpr int kMaxSchedItems = 4096;
constexpr int kSchedTable = 0, kSchedQueue = 2;
constexpr int kItemRing = 4;

struct BwdSched {
  int n_ctas;                         // CTAs of the launch
  int mode;                           // kSchedTable or kSchedQueue
  int n_kt;                           // table: key tiles per (b, h)
  uint32_t n_virtual;                 // queue: (B * H) * ranks
  uint32_t per, ranks;                // queue: units per group, key tiles per unit
  uint16_t off[kMaxSchedCtas + 1];    // table: CTA c works on item[off[c] .. off[c + 1])
  uint32_t item[kMaxSchedItems];      // table: (b * H + h) * n_kt + kt
};

// One key tile as the roles see it: its (b, h) rows and the query tiles that
// see it.  n_steps < 0 marks the end of the CTA's tiles.
struct ItemRec {
  int b, h, kt, len, row0, slab, q_first, n_steps;
  long long out_base;
};

struct Bwd128Params {
  CUtensorMap tq, tk, tv, tdo;
  CUtensorMap tdq;  // D = 64: the float32 dQ accumulator, for tensor reduce-adds
  DropParams drop;  // used by the dropout instantiation only
  const float* lse;
  const float* dvec;
  float* dq_acc;
  __nv_bfloat16* dk;  // 16-bit storage: bf16 or fp16 per F16
  __nv_bfloat16* dv;
  const int32_t* cu;
  unsigned* status;
  unsigned* queue;  // the tile counter of the queue form (workspace, zero at launch)
  unsigned long long limit_ns;
  int B, H, N, T;
  float c2;  // scale * log2(e)
  float scale;
  int causal;
  BwdSched sched;
};

// Shared memory, dynamic only (1024-byte aligned base, checked), for head
// width D (64 or 128).  A Q, K, V or dO tile is 128 rows of D elements in
// D / 64 blocks of 64 columns (128 bytes, one 128-byte swizzle row).  The dQ
// of a step leaves in two halves, each staged as one float32 box: at D = 128
// dQ^T (head width on TMEM lanes) gives [64 queries][128] per query half; at
// D = 64, dQ (queries on lanes) gives [128 queries][32] per head-width half.
// Half 0 is staged in the dS^T buffer, free between dQ_k and dS^T_{k+1}.
constexpr int kHalfBytes = kTile * 128;  // 16 KB: 64 columns of 128 rows

// (the two barriers of half 0's second piece exist at D = 128 only)
template <int D>
constexpr int num_bars() { return 20 + 2 * kItemRing + (D == 128 && kH0Pieces ? 2 : 0); }
template <int D>
struct BwdLayout {
  static constexpr int kTileBytes = kTile * D * 2;  // 32 KB or 16 KB; also one dQ half in float32
  static constexpr int kHalves = D / 64;
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kTileBytes;
  static constexpr int kQOff = 2 * kTileBytes;       // 2 stages
  static constexpr int kDOOff = 4 * kTileBytes;      // 1 stage
  static constexpr int kDSOff = 5 * kTileBytes;      // dS^T [128 keys][128 queries] bf16 (32 KB); dQ half 0
  static constexpr int kStageOff = kDSOff + 32768;   // dQ half 1
  static constexpr int kLOff = kStageOff + kTileBytes;  // 2 x 128 floats: L * log2(e)
  static constexpr int kDvOff = kLOff + 1024;           // 2 x 128 floats: D
  static constexpr int kBarOff = kDvOff + 1024;
  static constexpr int kNumBars = num_bars<D>();
  static constexpr int kRingOff = kBarOff + kNumBars * 8;  // kItemRing ItemRec
  static constexpr int kMiscOff = kRingOff + kItemRing * (int)sizeof(ItemRec);
  static constexpr int kSmemBytes = kMiscOff + 16;
  static_assert(kSmemBytes <= 232448, "shared-memory budget");
  static_assert(kDSOff % 1024 == 0 && kStageOff % 1024 == 0, "swizzled buffers need 1024-byte alignment");
};

// kDq = false: dK and dV only, for the deterministic backward (whose dQ comes
// from the query-stationary kernel): no dS^T copy in shared memory, no dQ^T
// product, read-out or reduction, and dP^T_k waits for nothing but dO_k.
template <int D, bool F16, bool kDrop, bool kDq>
__global__ void __launch_bounds__(kThreads, 1) tc_bwd128_kernel(const __grid_constant__ Bwd128Params p) {
  using C = BwdLayout<D>;
  constexpr int kTileBytes = C::kTileBytes, kKOff = C::kKOff, kVOff = C::kVOff, kQOff = C::kQOff,
                kDOOff = C::kDOOff, kDSOff = C::kDSOff, kStageOff = C::kStageOff, kLOff = C::kLOff,
                kDvOff = C::kDvOff, kBarOff = C::kBarOff, kRingOff = C::kRingOff, kMiscOff = C::kMiscOff;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (smem_u32(smem) & 1023u) {  // the swizzled tile layout needs a 1024-byte aligned base
    if (threadIdx.x == 0) atomicOr(p.status, kDevInternal);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* bar_kv = bars + 0;      // K, V loaded
  uint64_t* bar_qf = bars + 1;      // [2] Q tile + L / D of a stage loaded (2 arrivals + bytes)
  uint64_t* bar_qe = bars + 3;      // [2] Q / L / D stage free (dK done)
  uint64_t* bar_of = bars + 5;      // dO tile loaded
  uint64_t* bar_oe = bars + 6;      // dO buffer free (dV done)
  uint64_t* bar_s = bars + 7;       // S^T ready
  uint64_t* bar_dp = bars + 8;      // dP^T ready
  uint64_t* bar_p = bars + 9;       // P^T written (8 compute warps)
  uint64_t* bar_ds = bars + 10;     // dS^T written (8 compute warps)
  uint64_t* bar_dq = bars + 11;     // dQ^T ready
  uint64_t* bar_dqfree = bars + 12; // dQ^T read out of TMEM (8 compute warps)
  uint64_t* bar_dsfree = bars + 13; // dS^T buffer no longer read by the copy engine (reducer)
  uint64_t* bar_done = bars + 14;   // every MMA complete
  uint64_t* bar_staged = bars + 15; // [2] dQ half staged in shared memory (4 warps each)
  uint64_t* bar_stfree = bars + 17; // half 1's staging buffer read by the copy engine (reducer)
  uint64_t* bar_itemdone = bars + 18; // every product of a key tile complete (its dK / dV final, K / V free)
  uint64_t* bar_accfree = bars + 19;  // dK / dV of a key tile read out of TMEM (8 compute warps)
  uint64_t* bar_item = bars + 20;     // [kItemRing] a tile's record written (producer)
  uint64_t* bar_itemfree = bars + 20 + kItemRing;  // [kItemRing] record read (every consumer role)
  // D = 128 with kH0Pieces: bar_staged[0] / bar_dsfree cover half 0's first piece
  // (and the first query half of the dS^T buffer), these two its second piece
  constexpr bool kPieces = D == 128 && kH0Pieces;
  uint64_t* bar_staged0b = kPieces ? bars + 20 + 2 * kItemRing : nullptr;  // half 0's second piece staged (4 warps)
  uint64_t* bar_dsfree1 = kPieces ? bars + 21 + 2 * kItemRing : nullptr;   // second query half of the dS^T buffer read
  ItemRec* ring = reinterpret_cast<ItemRec*>(smem + kRingOff);
  uint32_t* tmem_base_sh = reinterpret_cast<uint32_t*>(smem + kMiscOff);
  int* abort_flag = reinterpret_cast<int*>(smem + kMiscOff + 4);
  float* s_l = reinterpret_cast<float*>(smem + kLOff);
  float* s_d = reinterpret_cast<float*>(smem + kDvOff);

  // ---- where the producer takes this CTA's key tiles from (see BwdSched)
  const bool table = p.sched.mode == kSchedTable;
  const int first_item = table ? p.sched.off[blockIdx.x] : 0;
  const int n_table = table ? p.sched.off[blockIdx.x + 1] - first_item : 0;
  const ClosedSpec order{p.sched.n_virtual, (uint32_t)p.B * (uint32_t)p.H, p.sched.per, p.sched.ranks, 1u, 0u};
  auto set_steps = [&](ItemRec& it) {
    const int n_t = (it.len + kTile - 1) / kTile;
    it.q_first = p.causal ? it.kt : 0;  // earlier query tiles never see these keys
    it.n_steps = n_t - it.q_first;
  };
  // the tile of virtual item f of the queue, or false for a rank its sequence lacks
  auto tile_of_virtual = [&](uint32_t f, ItemRec& it) -> bool {
    uint32_t uu, rr;
    closed_unit_rank(order, f, uu, rr);
    const int u = (int)uu;
    it.b = u / p.H;
    it.h = u - it.b * p.H;
    if (p.cu != nullptr) {
      const int s0 = p.cu[it.b], s1 = p.cu[it.b + 1];
      if (s0 < 0 || s1 < s0 || s1 > p.T || s1 - s0 > p.N) {  // skipped and reported
        atomicOr(p.status, kDevBadSeqlens);
        return false;
      }
      it.len = s1 - s0;
      it.row0 = s0;
      it.slab = it.h;
      it.out_base = (long long)it.h * p.T + s0;
    } else {
      it.len = p.N;
      it.row0 = 0;
      it.slab = u;
      it.out_base = (long long)u * p.N;
    }
    it.kt = bwd_tile_of_rank(it.len, (int)rr);
    if (it.kt < 0) return false;
    set_steps(it);
    return true;
  };
  if (table && n_table <= 0) return;  // (a table gives every CTA of the launch work)

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kNumBars; ++i) {
      uint64_t* bar = bars + i;
      const bool by8 = bar == bar_p || bar == bar_ds || bar == bar_dqfree || bar == bar_accfree;
      const bool by4 = bar == bar_staged || bar == bar_staged + 1 || bar == bar_staged0b;
      const bool by2 = bar == bar_qf || bar == bar_qf + 1;  // Q bytes + L / D written
      // a record is read by the 8 compute warps, the MMA issuer and the reducer
      const bool readers = bar >= bar_itemfree && bar < bar_itemfree + kItemRing;
      mbar_init(bar, readers ? (kDq ? 10 : 9) : by8 ? 8 : by4 ? 4 : by2 ? 2 : 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_base_sh, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_sh;
  const WaitCtx w{abort_flag, p.status, p.limit_ns};
  // Steps are counted over all of the CTA's key tiles (g = steps of the earlier
  // tiles + k): every per-step barrier keeps its phase across tiles.

  if (warp < 8) {
    // ------------------------------------------------------------ P^T, dS^T, dQ^T read-out, epilogue
    setmaxnreg_inc<kBwdComputeRegs>();
    const int ch = warp >> 2;        // query-column half
    const int quad = warp & 3;       // TMEM lanes 32*quad ..
    const int j = quad * 32 + lane;  // key row of S^T / dP^T; head-width column of dQ^T
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t t_s = tmem + lane_off + ch * 64;
    const uint32_t t_dp = tmem + lane_off + 128 + ch * 64;  // dP^T, dS^T, then (D = 128) dQ^T of this half
    uint8_t* ds_row = smem + kDSOff + ch * kHalfBytes + (j >> 3) * 1024 + (j & 7) * 128;
    float* stage = reinterpret_cast<float*>(smem + (ch == 0 ? kDSOff : kStageOff));
    bool ok = true;  // once a wait fails the rest are skipped (the abort flag is set)

    // dQ of global step gg leaves tensor memory.  D = 128: this warp holds
    // head-width column j of dQ^T for its half's 64 queries and writes them as
    // rows [64 queries][D] fp32.  D = 64: it holds query j's head-width
    // columns [32 ch, 32 ch + 32) of dQ and writes them as row j of a
    // [128 queries][32] fp32 box in the 128-byte swizzled layout the tensor
    // reduce reads (16-byte chunk c of row j at chunk c ^ (j % 8): no two lanes
    // of a quarter-warp write the same bank).
    auto drain_dq = [&](int gg) {
      ok = ok && warp_wait(bar_dq, gg & 1, w);
      tc_fence_after();
      uint32_t v[2][32];
      if constexpr (D == 128) {
        tmem_ld32(t_dp, v[0]);
        tmem_ld32(t_dp + 32, v[1]);
        tmem_ld_wait(v[0]);
        tmem_ld_wait(v[1]);
      } else {
        tmem_ld32(tmem + lane_off + 128 + ch * 32, v[0]);
        tmem_ld_wait(v[0]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_dqfree);
      // half 1's buffer must have been read by the previous reduction (half 0's
      // buffer is the dS^T buffer, already released before dS^T_gg was written)
      if (ch == 1) {
        // half 0 goes to the copy engine first and its buffer gates the next dS^T:
        // let its warps have the shared-memory write bandwidth to themselves
        ok = ok && warp_wait(kPieces ? bar_staged0b : bar_staged, gg & 1, w);
        if (gg > 0) ok = ok && warp_wait(bar_stfree, (gg - 1) & 1, w);
      }
      if constexpr (kPieces) {
        if (ch == 0) {
          // rows 0-31, published, then rows 32-63: two pieces for the copy engine
#pragma unroll
          for (int e = 0; e < 32; ++e) stage[e * D + j] = __uint_as_float(v[0][e]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_staged);
#pragma unroll
          for (int e = 32; e < 64; ++e) stage[e * D + j] = __uint_as_float(v[1][e - 32]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_staged0b);
          return;
        }
      }
      if constexpr (D == 128) {
#pragma unroll
        for (int e = 0; e < 64; ++e) stage[e * D + j] = __uint_as_float(v[e >> 5][e & 31]);
      } else {
        uint8_t* row = reinterpret_cast<uint8_t*>(stage) + j * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(row + ((c ^ (j & 7)) << 4)) =
              make_uint4(v[0][4 * c], v[0][4 * c + 1], v[0][4 * c + 2], v[0][4 * c + 3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_staged + ch);
    };

    int G = 0;
    for (int ii = 0; ok; ++ii) {
      // the tile's record (every lane waits: each acquires what the producer released)
      const int slot = ii % kItemRing;
      if (!warp_wait(bar_item + slot, (ii / kItemRing) & 1, w)) {
        ok = false;
        break;
      }
      const ItemRec it = ring[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_itemfree + slot);
      if (it.n_steps < 0) break;  // no tiles left
      const int b = it.b, h = it.h, len = it.len;
      const int key = it.kt * kTile + j;
      for (int k = 0; ok && k < it.n_steps; ++k) {
        const int g = G + k;
        const int qi = it.q_first + k;
        const int st = g & 1;
        const float4* sl4 = reinterpret_cast<const float4*>(s_l + st * 128 + ch * 64);
        const float4* sd4 = reinterpret_cast<const float4*>(s_d + st * 128 + ch * 64);
        // dropout decisions of (this half's 64 queries, this key), regenerated
        uint64_t keepm = ~0ull;
        if constexpr (kDrop) {
          keepm = keep64_keys_on_lanes(p.drop, (uint32_t)key, (uint32_t)(qi * kTile + ch * 64), (uint32_t)(b * p.H + h),
                                       lane);
          // formed here, before the waits, where the previous step's values are dead
          asm volatile("" : "+l"(keepm));
        }
        ok = ok && warp_wait(bar_qf + st, (g >> 1) & 1, w) && warp_wait(bar_s, g & 1, w);
        tc_fence_after();
        uint32_t sv[2][32];
        tmem_ld32(t_s, sv[0]);
        tmem_ld32(t_s + 32, sv[1]);
        tmem_ld_wait(sv[0]);
        tmem_ld_wait(sv[1]);
        const int q0 = qi * kTile + ch * 64;  // first query (within the sequence) of this half
        float pr[64];
#pragma unroll
        for (int c4 = 0; c4 < 16; ++c4) {
          const float4 l4 = sl4[c4];
          const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
          for (int e = 0; e < 4; e += 2) {
            const int c = 4 * c4 + e;
            float a0, a1;  // s * scale * log2(e) - L * log2(e), two columns per packed FMA
            ffma2(a0, a1, __uint_as_float(sv[c >> 5][c & 31]), __uint_as_float(sv[(c + 1) >> 5][(c + 1) & 31]), p.c2,
                  -lv[e], -lv[e + 1]);
            pr[c] = ex2_approx(a0);
            pr[c + 1] = ex2_approx(a1);
          }
        }
        if ((p.causal && qi == it.kt) || (it.kt * kTile + kTile > len) || (qi * kTile + kTile > len)) {
          // diagonal or ragged tile: weights of future keys, padding keys and padding queries are zero
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const int q = q0 + c;
            if (q >= len || key >= len || (p.causal && key > q)) pr[c] = 0.f;
          }
        }
        {
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            if constexpr (kDrop)  // dV takes the dropped weights, scaled by 1 / (1 - p)
              pk[c] = pack16x2<F16>((keepm >> (2 * c)) & 1 ? pr[2 * c] * p.drop.scale : 0.f,
                                    (keepm >> (2 * c + 1)) & 1 ? pr[2 * c + 1] * p.drop.scale : 0.f);
            else
              pk[c] = pack16x2<F16>(pr[2 * c], pr[2 * c + 1]);
          }
          tmem_st32(t_s, pk);
          tmem_st_wait();
        }
        if constexpr (kDrop) {
          // the keep decisions ride in the sign bits of the weights from here on
          // (every weight is >= 0; a dropped one becomes -P, a masked 0 -0), so the
          // mask's registers are free before the dQ read-out below
#pragma unroll
          for (int c = 0; c < 64; ++c)
            pr[c] = __uint_as_float(__float_as_uint(pr[c]) | ((~(uint32_t)(keepm >> c) & 1u) << 31));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_p);

        if constexpr (kDq)
          if (k > 0) drain_dq(g - 1);

        ok = ok && warp_wait(bar_dp, g & 1, w);
        tc_fence_after();
        if constexpr (!kDrop) {
          tmem_ld32(t_dp, sv[0]);
          tmem_ld32(t_dp + 32, sv[1]);
          tmem_ld_wait(sv[0]);
          tmem_ld_wait(sv[1]);
        }
        uint32_t dsp[32];
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
          if constexpr (kDrop) {
            // one 32-column half of dP^T at a time (the generator's work leaves no
            // registers for both at once)
            if (c8 % 4 == 0) {
              tmem_ld32(t_dp + 32 * (c8 / 4), sv[c8 / 4]);
              tmem_ld_wait(sv[c8 / 4]);
            }
          }
          const float4 da = sd4[2 * c8], db = sd4[2 * c8 + 1];
          const float dv[8] = {da.x, da.y, da.z, da.w, db.x, db.y, db.z, db.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c = c8 * 8 + 2 * e;
            float t0, t1, d0, d1;  // dS = P o (dP - D), two columns per packed op
            const float dp0 = __uint_as_float(sv[c >> 5][c & 31]), dp1 = __uint_as_float(sv[(c + 1) >> 5][(c + 1) & 31]);
            if constexpr (kDrop) {
              // dP of the dropped weights is masked and scaled like them: with w = +-P
              // (sign = dropped), dS = max(w, 0) * scale * dP - |w| * D
              d0 = fmaf(fmaxf(pr[c], 0.f) * p.drop.scale, dp0, -fabsf(pr[c]) * dv[2 * e]);
              d1 = fmaf(fmaxf(pr[c + 1], 0.f) * p.drop.scale, dp1, -fabsf(pr[c + 1]) * dv[2 * e + 1]);
            } else {
              fsub2(t0, t1, dp0, dp1, dv[2 * e], dv[2 * e + 1]);
              fmul2(d0, d1, pr[c], pr[c + 1], t0, t1);
            }
            dsp[4 * c8 + e] = pack16x2<F16>(d0, d1);
          }
        }
        tmem_st32(t_dp, dsp);  // dS^T as bf16 pairs over this half's first 32 dP^T columns (already read)
        if constexpr (kDq) {
          // the dS^T buffer held half 0 of the previous dQ until the copy engine read it
          // (with the two pieces, each query half waits for its own piece)
          if (g > 0)
            ok = ok && warp_wait((kPieces && ch == 1) ? bar_dsfree1 : bar_dsfree, (g - 1) & 1, w);
#pragma unroll
          for (int c8 = 0; c8 < 8; ++c8)  // 128-byte swizzle: 16-byte chunk c8 of row j sits at chunk c8 ^ (j % 8)
            *reinterpret_cast<uint4*>(ds_row + ((c8 ^ (j & 7)) << 4)) =
                make_uint4(dsp[4 * c8], dsp[4 * c8 + 1], dsp[4 * c8 + 2], dsp[4 * c8 + 3]);
          fence_proxy_async_smem();
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_ds);
      }
      if constexpr (kDq) drain_dq(G + it.n_steps - 1);
      // epilogue: dV and dK rows of this tile's keys, once its last products are complete.
      // Both are read out of tensor memory and packed first, so the accumulators are
      // handed back before any store; each thread then holds E 16-byte chunks of its
      // own key row, which an E x E exchange within groups of E lanes turns into whole
      // rows per store instruction (32 / E rows of a full 128-byte line each, instead
      // of one line per lane).
      if (ok && warp_wait(bar_itemdone, ii & 1, w)) {
        tc_fence_after();
        constexpr int E = D / 16;  // 16-byte chunks in this half's D / 2 columns
        uint32_t pk[2][4 * E];     // dV, dK of key row j, columns ch * D / 2 .., as 16-bit pairs
#pragma unroll
        for (int which = 0; which < 2; ++which) {
          const float mul = which == 0 ? 1.f : p.scale;
          const uint32_t t_acc = tmem + lane_off + (which == 0 ? 256 : 384) + ch * (D / 2);
#pragma unroll
          for (int c = 0; c < D / 2; c += 32) {
            uint32_t v[32];
            tmem_ld32(t_acc + c, v);
            tmem_ld_wait(v);
#pragma unroll
            for (int e = 0; e < 16; ++e)
              pk[which][c / 2 + e] = pack16x2<F16>(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
          }
        }
        // the accumulators are read: the next tile's dV / dK may start over them
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_accfree);
        const int grp = lane & ~(E - 1), sub = lane & (E - 1);
#pragma unroll
        for (int which = 0; which < 2; ++which) {
          exchange_chunks<E>(pk[which], lane);
          // chunk slot i now holds chunk `sub` of key row grp + i of this warp's 32
          __nv_bfloat16* out = (which == 0 ? p.dv : p.dk) + ch * (D / 2) + sub * 8;
#pragma unroll
          for (int i = 0; i < E; ++i) {
            const int r = it.kt * kTile + quad * 32 + grp + i;
            if (r < len)
              *reinterpret_cast<uint4*>(out + (it.out_base + r) * D) =
                  make_uint4(pk[which][4 * i], pk[which][4 * i + 1], pk[which][4 * i + 2], pk[which][4 * i + 3]);
          }
        }
      }
      G += it.n_steps;
    }
  } else {
    setmaxnreg_dec<kBwdSupportRegs>();
    if (warp == kTmaWarp) {
      // ---------------------------------------------------------- producer
      if (lane == 0) {
        tma_prefetch_desc(&p.tq);
        tma_prefetch_desc(&p.tk);
        tma_prefetch_desc(&p.tv);
        tma_prefetch_desc(&p.tdo);
      }
      int q_issued = 0, o_issued = 0, kv_issued = 0, G = 0;
      bool good_all = true;
      // K, V of a tile, once every product of the previous tile (their last
      // readers) is complete; lane 0 waits, the answer is broadcast
      auto load_kv = [&](const ItemRec& it, int ii) {
        int good = 1;
        if (lane == 0) {
          if (ii > 0) good = mbar_wait(bar_itemdone, (ii - 1) & 1, w);
          if (good) {
            mbar_arrive_expect_tx(bar_kv, 2 * kTileBytes);
            for (int hf = 0; hf < C::kHalves; ++hf) {
              tma_load_3d(smem + kKOff + hf * kHalfBytes, &p.tk, bar_kv, hf * 64, it.row0 + it.kt * kTile, it.slab);
              tma_load_3d(smem + kVOff + hf * kHalfBytes, &p.tv, bar_kv, hf * 64, it.row0 + it.kt * kTile, it.slab);
            }
          }
        }
        good = __shfl_sync(0xffffffffu, good, 0);
        if (good) kv_issued = ii + 1;
        return good != 0;
      };
      // ---- taking tiles (lane 0) and handing them to the roles
      uint32_t k_tab = 0;
      uint32_t reserved = 0;  // queue: the next virtual item, taken one tile ahead
      if (!table && lane == 0) reserved = atomicAdd(p.queue, 1u);
      auto take = [&](ItemRec& it) -> bool {
        if (table) {  // dense: every listed tile is in range
          if (k_tab >= (uint32_t)n_table) return false;
          const uint32_t code = p.sched.item[first_item + (int)k_tab++];
          const int bh = (int)(code / (uint32_t)p.sched.n_kt);
          it.kt = (int)(code - (uint32_t)bh * (uint32_t)p.sched.n_kt);
          it.b = bh / p.H;
          it.h = bh - it.b * p.H;
          it.len = p.N;
          it.row0 = 0;
          it.slab = bh;
          it.out_base = (long long)bh * p.N;
          set_steps(it);
          return true;
        }
        for (;;) {
          const uint32_t f = reserved;
          if (f >= p.sched.n_virtual) return false;
          reserved = atomicAdd(p.queue, 1u);  // in flight while this tile is worked on
          if (tile_of_virtual(f, it)) return true;
        }
      };
      // Tile ii (or the end) into ring slot ii % kItemRing, once every role has
      // read the record kItemRing tiles back; lane 0 writes, every lane reads the
      // record back.  Returns 1 for a tile, 0 at the end, -1 if a wait failed.
      auto next_tile = [&](int ii, ItemRec& it) -> int {
        const int slot = ii % kItemRing;
        int state = 1;
        if (lane == 0) {
          ItemRec t{};
          const bool have = take(t);
          if (ii >= kItemRing && !mbar_wait(bar_itemfree + slot, (ii / kItemRing - 1) & 1, w)) {
            state = -1;
          } else {
            if (!have) t.n_steps = -1;
            ring[slot] = t;
            mbar_arrive(bar_item + slot);  // releases the record to the roles' waits
            if (have && ii > 0)
              // its K and V wait for the previous tile's last products: have them in L2 by then
              for (int hf = 0; hf < C::kHalves; ++hf) {
                tma_prefetch_l2_3d(&p.tk, hf * 64, t.row0 + t.kt * kTile, t.slab);
                tma_prefetch_l2_3d(&p.tv, hf * 64, t.row0 + t.kt * kTile, t.slab);
              }
            state = have ? 1 : 0;
          }
        }
        state = __shfl_sync(0xffffffffu, state, 0);
        __syncwarp();
        if (state > 0) it = ring[slot];
        return state;
      };
      // L and D rows of a step (rows past the sequence's end read its last row and
      // are stored as zero).  A tile's first step fetches its own; every later
      // step's are fetched a step ahead, so the loads are in flight while the
      // producer waits for buffers instead of holding up the next Q copy.
      float lv[4], dv[4];
      auto fetch_ld = [&](const ItemRec& t, int q) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const long long row = t.out_base + min(q * kTile + lane * 4 + e, t.len - 1);
          lv[e] = p.lse[row];
          dv[e] = p.dvec[row];
        }
      };
      ItemRec it;
      int state = next_tile(0, it);
      if (state < 0) good_all = false;
      for (int ii = 0; good_all && state > 0; ++ii) {
        // The first tile's K and V go first; a later tile's wait until its first
        // Q, L / D and dO are on their way, which need no more than their buffers.
        if (ii == 0 && !load_kv(it, ii)) break;
        int good = 1;
        for (int k = 0; k < it.n_steps; ++k) {
          const int g = G + k;
          const int qi = it.q_first + k;
          const int st = g & 1;
          // Q / L / D stage st was last used by step g - 2 (free once its dK has
          // completed); the single dO buffer by step g - 1 (free once its dV has).
          // Lane 0 waits and the answer is broadcast, so the warp never splits.
          // The stage's barrier takes a second arrival once L and D are in shared
          // memory.
          if (k == 0) fetch_ld(it, qi);
          if (lane == 0 && g >= 2) good = mbar_wait(bar_qe + st, ((g >> 1) - 1) & 1, w);
          if (!__shfl_sync(0xffffffffu, good, 0)) {
            good_all = false;
            break;
          }
          if (lane == 0) {
            mbar_arrive_expect_tx(bar_qf + st, kTileBytes);
            for (int hf = 0; hf < C::kHalves; ++hf)
              tma_load_3d(smem + kQOff + st * kTileBytes + hf * kHalfBytes, &p.tq, bar_qf + st, hf * 64,
                          it.row0 + qi * kTile, it.slab);
          }
          q_issued = g + 1;
          {  // L and D into the stage, then its barrier's second arrival
            float l4[4], d4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const bool in = qi * kTile + lane * 4 + e < it.len;
              l4[e] = in ? lv[e] * kLog2e : 0.f;
              d4[e] = in ? dv[e] : 0.f;
            }
            *reinterpret_cast<float4*>(s_l + st * 128 + lane * 4) = make_float4(l4[0], l4[1], l4[2], l4[3]);
            *reinterpret_cast<float4*>(s_d + st * 128 + lane * 4) = make_float4(d4[0], d4[1], d4[2], d4[3]);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_qf + st);
          if (lane == 0 && g >= 1) good = mbar_wait(bar_oe, (g - 1) & 1, w);
          if (!__shfl_sync(0xffffffffu, good, 0)) {
            good_all = false;
            break;
          }
          if (lane == 0) {
            mbar_arrive_expect_tx(bar_of, kTileBytes);
            for (int hf = 0; hf < C::kHalves; ++hf)
              tma_load_3d(smem + kDOOff + hf * kHalfBytes, &p.tdo, bar_of, hf * 64, it.row0 + qi * kTile, it.slab);
          }
          o_issued = g + 1;
          if (k + 1 < it.n_steps) fetch_ld(it, qi + 1);
          if (k == 0 && ii > 0 && !load_kv(it, ii)) {
            good_all = false;
            break;
          }
        }
        if (!good_all) break;
        G += it.n_steps;
        state = next_tile(ii + 1, it);
        if (state < 0) good_all = false;
      }
      if (lane == 0 && *abort_flag) {
        // let copies already in flight land before the CTA's memory is released
        if (kv_issued > 0) mbar_wait_drain(bar_kv, (kv_issued - 1) & 1, p.limit_ns);
        if (o_issued > 0) mbar_wait_drain(bar_of, (o_issued - 1) & 1, p.limit_ns);
        for (int g = max(0, q_issued - 2); g < q_issued; ++g)
          mbar_wait_drain(bar_qf + (g & 1), (g >> 1) & 1, p.limit_ns);
      }
    } else if (kDq && warp == kReduceWarp && lane == 0) {
      // ---------------------------------------------------------- dQ reducer
      // Both halves go out back to back; half 0's buffer (the dS^T buffer) is
      // handed back as soon as it has been read, half 1's after that.
      int G = 0;
      bool good = true;
      for (int ii = 0; good; ++ii) {
        const int slot = ii % kItemRing;
        if (!mbar_wait(bar_item + slot, (ii / kItemRing) & 1, w)) break;
        const ItemRec it = ring[slot];
        mbar_arrive(bar_itemfree + slot);
        if (it.n_steps < 0) break;  // no tiles left
        for (int kk = 0; good && kk < it.n_steps; ++kk) {
          const int gg = G + kk;
          const int q0 = (it.q_first + kk) * kTile;
          if constexpr (kPieces) {
            // half 0 as two 32-row pieces from the dS^T buffer, then half 1
            for (int pc = 0; pc < 3; ++pc) {
              uint64_t* bar = pc == 0 ? bar_staged : pc == 1 ? bar_staged0b : bar_staged + 1;
              if (!mbar_wait(bar, gg & 1, w)) {
                good = false;
                break;
              }
              const int r0 = pc == 2 ? 64 : pc * 32;  // first query row of the piece: 0, 32, 64
              const int nq = min(pc == 2 ? 64 : 32, it.len - (q0 + r0));
              if (nq > 0)
                bulk_reduce_add_f32(p.dq_acc + (it.out_base + q0 + r0) * D,
                                    smem + (pc == 2 ? kStageOff : kDSOff + pc * 16384), (uint32_t)nq * D * 4);
              bulk_commit();
            }
            if (!good || *abort_flag) {
              good = false;
              break;
            }
            bulk_wait_read<2>();  // rows 0-31 read: the first query half of the dS^T buffer
            mbar_arrive(bar_dsfree);
            bulk_wait_read<1>();  // rows 32-63 read: the second
            mbar_arrive(bar_dsfree1);
            bulk_wait_read<0>();  // half 1 read
            mbar_arrive(bar_stfree);
            continue;
          }
          for (int hf = 0; hf < 2; ++hf) {
            if (!mbar_wait(bar_staged + hf, gg & 1, w)) {
              good = false;
              break;
            }
            if constexpr (D == 128) {
              // query half hf: rows of this sequence only
              const int nq = min(64, it.len - (q0 + hf * 64));
              if (nq > 0)
                bulk_reduce_add_f32(p.dq_acc + (it.out_base + q0 + hf * 64) * D,
                                    smem + (hf == 0 ? kDSOff : kStageOff), (uint32_t)nq * D * 4);
            } else {
              // head-width half hf of all 128 query rows: rows past the sequence
              // hold zeros (their weights are zero) and rows past the tensor are
              // clipped by the copy engine
              tma_reduce_add_2d(&p.tdq, smem + (hf == 0 ? kDSOff : kStageOff), hf * 32, (int)(it.out_base + q0));
            }
            bulk_commit();
          }
          if (!good || *abort_flag) {
            good = false;
            break;
          }
          bulk_wait_read<1>();  // half 0 read
          mbar_arrive(bar_dsfree);
          bulk_wait_read<0>();  // half 1 read
          mbar_arrive(bar_stfree);
        }
        G += it.n_steps;
      }
      bulk_wait_all();
    } else if (warp == kMmaWarp && lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      const uint32_t id_nn = idesc16<F16>(128, 128, false, false);  // S^T, dP^T: both K-major
      const uint32_t id_acc = idesc16<F16>(128, D, false, true);    // dV, dK: B MN-major
      // dQ^T = K^T dS^T (D = 128, M = head width) or dQ = dS K (D = 64, M = queries): both MN-major
      const uint32_t id_dq = idesc16<F16>(128, D == 128 ? 128 : D, true, true);
      // Descriptors, advanced by adding (byte offset >> 4) to the start field.
      // k* = K-major view, m* = MN-major view of the same tile.
      const uint64_t kK = sdesc_sw128(smem_u32(smem + kKOff), 16, 1024);
      const uint64_t kV = sdesc_sw128(smem_u32(smem + kVOff), 16, 1024);
      const uint64_t mK = sdesc_sw128(smem_u32(smem + kKOff), kHalfBytes, 1024);
      const uint64_t kQ = sdesc_sw128(smem_u32(smem + kQOff), 16, 1024);
      const uint64_t mQ = sdesc_sw128(smem_u32(smem + kQOff), kHalfBytes, 1024);
      const uint64_t kDO = sdesc_sw128(smem_u32(smem + kDOOff), 16, 1024);
      const uint64_t mDO = sdesc_sw128(smem_u32(smem + kDOOff), kHalfBytes, 1024);
      const uint64_t mDS = sdesc_sw128(smem_u32(smem + kDSOff), kHalfBytes, 1024);
      constexpr uint32_t kStageDesc = kTileBytes >> 4;
      auto koff = [](int ks) { return (uint32_t)(((ks >> 2) * kHalfBytes + (ks & 3) * 32) >> 4); };
      auto moff = [](int ks) { return (uint32_t)((ks * 2048) >> 4); };
      // Each group of 8 MMAs is issued back to back from one asm block.
      uint64_t a[8], b[8];
      uint32_t at[8];
      // D / 16 MMAs of K = 16 over the head width, back to back
      auto issue_nn = [&](uint32_t d_tmem, uint64_t adesc, uint64_t bdesc) {
        if constexpr (D == 128) {
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            a[ks] = adesc + koff(ks);
            b[ks] = bdesc + koff(ks);
          }
          mma_ss_x8(d_tmem, a, b, id_nn, 0u);
        } else {
          uint64_t a4[4], b4[4];
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            a4[ks] = adesc + koff(ks);
            b4[ks] = bdesc + koff(ks);
          }
          mma_ss_x4(d_tmem, a4, b4, id_nn, 0u);
        }
      };
      auto issue_s = [&](int g) {  // S^T of global step g = K Q_g^T -> [0,128)
        issue_nn(tmem + 0, kK, kQ + (g & 1) * kStageDesc);
        mma_commit(bar_s);
      };
      auto issue_dp = [&]() {  // dP^T = V dO^T -> [128,256)
        issue_nn(tmem + 128, kV, kDO);
        mma_commit(bar_dp);
      };
      bool ok = true;
      int G = 0;
      for (int ii = 0; ok; ++ii) {
        // the tile's step count from its record (the issuer has no registers
        // to spare for the rest of the tile's geometry)
        const int slot = ii % kItemRing;
        if (!mbar_wait(bar_item + slot, (ii / kItemRing) & 1, w)) {
          ok = false;
          break;
        }
        const int n_steps = ring[slot].n_steps;
        mbar_arrive(bar_itemfree + slot);
        if (n_steps < 0) break;  // no tiles left
        // K, V of this tile; S^T and dP^T of its first step.  dP^T goes over the
        // previous tile's last dQ^T, so it waits until that has been read out.
        ok = mbar_wait(bar_kv, ii & 1, w) && mbar_wait(bar_qf + (G & 1), (G >> 1) & 1, w);
        if (!ok) break;
        tc_fence_after();
        issue_s(G);
        ok = (!kDq || G == 0 || mbar_wait(bar_dqfree, (G - 1) & 1, w)) && mbar_wait(bar_of, G & 1, w);
        if (!ok) break;
        tc_fence_after();
        issue_dp();
        for (int k = 0; ok && k < n_steps; ++k) {
          const int g = G + k;
          const int st = g & 1;
          const uint32_t acc0 = k > 0 ? 1u : 0u;
          const bool more = k + 1 < n_steps;
          // dP^T over [128,256) once the previous dQ^T has left it
          if (k > 0) {
            if ((kDq && !mbar_wait(bar_dqfree, (g - 1) & 1, w)) || !mbar_wait(bar_of, g & 1, w)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_dp();
          }
          // dV += P^T dO: P^T (bf16) in TMEM columns [0,32) (queries 0-63) and [64,96);
          // the tile's first dV / dK start over accumulators the previous tile's
          // epilogue must have read
          if (!mbar_wait(bar_p, g & 1, w) || (k == 0 && ii > 0 && !mbar_wait(bar_accfree, (ii - 1) & 1, w))) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            at[ks] = tmem + (ks >> 2) * 64 + (ks & 3) * 8;
            b[ks] = mDO + moff(ks);
          }
          mma_ts_x8(tmem + 256, at, b, id_acc, acc0);
          mma_commit(bar_oe);  // dP^T and dV were the dO tile's last readers
          // S^T of the next step over the score columns (P^T is consumed in order by dV)
          if (more) {
            if (!mbar_wait(bar_qf + (st ^ 1), ((g + 1) >> 1) & 1, w)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_s(g + 1);
          }
          // dK += dS^T Q (dS^T bf16 in TMEM columns [128,160) and [192,224)), then
          // dQ^T = K^T dS^T over [128,256) (dS^T MN-major from shared memory)
          if (!mbar_wait(bar_ds, g & 1, w)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            at[ks] = tmem + 128 + (ks >> 2) * 64 + (ks & 3) * 8;
            b[ks] = mQ + st * kStageDesc + moff(ks);
          }
          mma_ts_x8(tmem + 384, at, b, id_acc, acc0);
          mma_commit(bar_qe + st);
          if constexpr (kDq) {
            // D = 128: dQ^T = K^T dS^T; D = 64: dQ = dS K (the same two MN-major
            // views, as A and B the other way round) -> [128, 128 + D or 128)
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              a[ks] = (D == 128 ? mK : mDS) + moff(ks);
              b[ks] = (D == 128 ? mDS : mK) + moff(ks);
            }
            mma_ss_x8(tmem + 128, a, b, id_dq, 0u);
            mma_commit(bar_dq);
          }
        }
        if (!ok) break;
        // the tile's dK / dV are final, and K / V have no later reader, once
        // every product issued so far is complete
        mma_commit(bar_itemdone);
        G += n_steps;
      }
      // every MMA issued must be complete before tensor memory is released
      mma_commit(bar_done);
      mbar_wait_drain(bar_done, 0, p.limit_ns);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
}

}  // namespace

// Multiprocessor count of the current device.
int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev] = n;
  }
  return cached[dev];
}

// Per-tile cost, in steps, of what a persistent CTA does for a key tile besides
// its steps (the K / V load it waits for, the epilogue); it only steers the
// balance of the schedule.
constexpr int kItemOverheadSteps = 2;

// The schedule for at most `ctas_max` CTAs: the table for dense inputs with
// at most kMaxSchedItems key tiles, the queue otherwise; false when there is
// nothing to do.
bool fill_bwd_sched(const Problem& p, int ctas_max, BwdSched& sc) {
  sc.n_ctas = 0;
  const int n_kt = (p.N + kTile - 1) / kTile;
  const long long n_bh = (long long)p.B * p.H;
  const long long n = n_bh * n_kt;
  if (n <= 0 || ctas_max <= 0) return false;
  sc.n_kt = n_kt;
  if (p.cu != nullptr || n > kMaxSchedItems) {
    sc.mode = kSchedQueue;
    const long long v = n_bh * bwd_ranks(p.N);
    if (v > (long long)kMaxVirtualItems) return false;
    sc.n_virtual = (uint32_t)v;
    sc.per = closed_group_size((uint32_t)n_bh, kBwdHeadGroup);  // a few units at a time stay in L2
    sc.ranks = (uint32_t)bwd_ranks(p.N);
    sc.n_ctas = (int)std::min<long long>(v, ctas_max);
    return true;
  }
  sc.mode = kSchedTable;
  sc.n_virtual = (uint32_t)n;
  const int ctas = (int)std::min<long long>(n, std::min(ctas_max, kMaxSchedCtas));
  // Items in the order the grid used: with the mask, heavy-first inside
  // balanced groups of kBwdHeadGroup heads (the order of grouped_heavy_first),
  // or of all heads when their Q, dO and dQ accumulators fit in L2 together.
  std::vector<uint32_t> order((size_t)n);
  std::vector<int> weight((size_t)n);
  const long long head_bytes = 8ll * p.N * p.D;  // Q, dO (16-bit) and the float32 dQ accumulator
  const long long group_heads = n_bh * head_bytes <= kSchedL2GroupBytes ? n_bh : (long long)kBwdHeadGroup;
  const long long n_groups = (n_bh + group_heads - 1) / group_heads;
  const long long per = (n_bh + n_groups - 1) / n_groups;
  for (long long f = 0; f < n; ++f) {
    long long bh, kt;
    if (p.causal) {
      const long long group = f / (per * n_kt), r = f - group * per * n_kt;
      const long long heads = std::min(per, n_bh - group * per);
      bh = group * per + r % heads;
      kt = r / heads;
    } else {
      bh = f / n_kt;
      kt = f % n_kt;
    }
    order[(size_t)f] = (uint32_t)(bh * n_kt + kt);
    weight[(size_t)f] = (p.causal ? (int)(n_kt - kt) : n_kt) + kItemOverheadSteps;
  }
  // Each item to the CTA with the least work so far (lowest index on ties).
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
bool build_sched(const Problem& p, BwdSched& sc) {
  const int ctas = sm_count();
  static std::mutex mu;
  static long long key[6] = {-1, -1, -1, -1, -1, -1};
  static BwdSched cached;
  const long long want[6] = {p.B, p.H, p.N, p.D, p.causal, ctas};  // the table's head groups depend on D
  if (p.cu != nullptr) return fill_bwd_sched(p, ctas, sc);  // closed form: nothing to cache
  std::lock_guard<std::mutex> lock(mu);
  if (std::equal(want, want + 6, key)) {
    sc = cached;
    return true;
  }
  if (!fill_bwd_sched(p, ctas, sc)) return false;
  cached = sc;
  std::copy(want, want + 6, key);
  return true;
}

int preview_bwd_schedule(const Problem& p, const int32_t* cu_host, int ctas, int* off, uint32_t* items, int cap,
                         int* form) {
  static BwdSched sc;  // large; previews are a host-side test aid
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (!fill_bwd_sched(p, ctas, sc)) return -1;
  *form = sc.mode;
  if (sc.mode == kSchedTable) {
    const int n = sc.off[sc.n_ctas];
    if (n > cap) return -2;
    for (int c = 0; c <= sc.n_ctas; ++c) off[c] = sc.off[c];
    std::copy(sc.item, sc.item + n, items);
    return n;
  }
  // the queue: one list, in the order the CTAs take the tiles (the kernel's
  // producer skips the ranks a sequence does not have)
  const ClosedSpec order{sc.n_virtual, (uint32_t)p.B * (uint32_t)p.H, sc.per, sc.ranks, 1u, 0u};
  const int ranks = bwd_ranks(p.N);
  int n = 0;
  for (uint32_t f = 0; f < sc.n_virtual; ++f) {
    uint32_t uu, rr;
    closed_unit_rank(order, f, uu, rr);
    const int u = (int)uu;
    int len = p.N;
    if (cu_host != nullptr) {
      const int b = u / p.H, s0 = cu_host[b], s1 = cu_host[b + 1];
      if (s0 < 0 || s1 < s0 || s1 > p.T || s1 - s0 > p.N) continue;
      len = s1 - s0;
    }
    const int kt = bwd_tile_of_rank(len, (int)rr);
    if (kt < 0) continue;
    if (n >= cap) return -2;
    items[n++] = (uint32_t)((long long)u * ranks + kt);
  }
  off[0] = 0;
  for (int c = 1; c <= sc.n_ctas; ++c) off[c] = n;
  return n;
}

template <int D, bool F16, bool kDrop, bool kDq>
cudaError_t launch_bwd128_t(const Problem& p, cudaStream_t s) {
  using C = BwdLayout<D>;
  static Bwd128Params bp;  // large (the schedule); filled in full below on every call
  static std::mutex launch_mu;
  std::lock_guard<std::mutex> launch_lock(launch_mu);
  if (!make_map16(&bp.tq, p.q, p, kTile) || !make_map16(&bp.tk, p.k, p, kTile) ||
      !make_map16(&bp.tv, p.v, p, kTile) || !make_map16(&bp.tdo, p.dout, p, kTile))
    return note_error("backward tensor map encode", cudaErrorInvalidValue);
  if constexpr (D == 64 && kDq) {
    // the tensor reduce addresses accumulator rows with 32-bit coordinates
    if (p.rows() > 0x7fffffffll) return note_error("backward: more than 2^31 rows at D = 64", cudaErrorInvalidValue);
    if (!make_map_acc32(&bp.tdq, p.dq_acc, (uint64_t)p.rows(), D))
      return note_error("backward dQ accumulator tensor map encode", cudaErrorInvalidValue);
  }
  bp.lse = p.lse;
  bp.dvec = p.dvec;
  bp.dq_acc = p.dq_acc;
  bp.dk = static_cast<__nv_bfloat16*>(p.dk);
  bp.dv = static_cast<__nv_bfloat16*>(p.dv);
  bp.cu = p.cu;
  bp.status = p.status;
  bp.queue = p.queue;
  bp.limit_ns = p.wait_limit_ns;
  bp.B = p.B;
  bp.H = p.H;
  bp.N = p.N;
  bp.T = p.T;
  bp.c2 = p.scale * kLog2e;
  bp.scale = p.scale;
  bp.causal = p.causal;
  bp.drop = drop_params_of(p);
  cudaError_t e = cudaFuncSetAttribute(tc_bwd128_kernel<D, F16, kDrop, kDq>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return note_error("backward smem attribute", e);
  if (!build_sched(p, bp.sched))
    return note_error("backward schedule (no multiprocessor count, or more than 2^31 work items)",
                      cudaErrorInvalidValue);
  tc_bwd128_kernel<D, F16, kDrop, kDq><<<bp.sched.n_ctas, kThreads, C::kSmemBytes, s>>>(bp);
  note_launches(1);
  return note_error("backward launch", cudaGetLastError());
}

template <int D, bool kDq>
cudaError_t launch_bwd_dispatch(const Problem& p, cudaStream_t s) {
  if (p.dropout) return p.f16 ? launch_bwd128_t<D, true, true, kDq>(p, s) : launch_bwd128_t<D, false, true, kDq>(p, s);
  return p.f16 ? launch_bwd128_t<D, true, false, kDq>(p, s) : launch_bwd128_t<D, false, false, kDq>(p, s);
}

cudaError_t launch_tc_bwd128(const Problem& p, cudaStream_t s) {
  if (p.D == 64) return launch_bwd_dispatch<64, true>(p, s);
  if (p.D == 128) return launch_bwd_dispatch<128, true>(p, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_tc_bwd128_dkdv(const Problem& p, cudaStream_t s) {
  if (p.D == 64) return launch_bwd_dispatch<64, false>(p, s);
  if (p.D == 128) return launch_bwd_dispatch<128, false>(p, s);
  return cudaErrorInvalidValue;
}

}  // namespace fa
