// Tensor-core backward kernels for sm_103a (bf16 in, fp32 accumulate).
//
// tensortonic.com "FlashAttention" section 7: the backward pass reloads
// blocks of queries and keys, recomputes each score tile and rebuilds its
// weights from the saved log-sum-exp, P_ij = exp(s_ij - L_i), so the n x n
// weight matrix is never stored.  With D_i = rowsum(dO o O) (computed by the
// preprocess kernel) the gradients are
//     dV = P^T dO,  dP = dO V^T,  dS = P o (dP - D),
//     dK = scale * dS^T Q,  dQ = scale * dS K.
//
// Main kernel: a CTA owns one 128-key tile of K and V (kept in shared
// memory) and visits the 128-query tiles that can see it (causal: from the
// diagonal tile on).  All five products are tcgen05 MMAs:
//     S^T  = K Q^T      -> TMEM [0,128)       (keys on lanes, queries on columns)
//     dP^T = V dO^T     -> TMEM [128,256)
//     dV  += P^T dO     (P^T read from TMEM)  -> TMEM [256,256+D)
//     dK  += dS^T Q     (dS^T from shared)    -> TMEM [384,384+D)
//     dQ_i^T = K^T dS^T (dS^T and K read MN-major) -> TMEM [0,128)   (D = 128)
//     dQ_i   = dS K                                 -> TMEM [0,D)     (D = 64)
// The dQ tile is added into a float32 accumulator in device memory with
// atomics (at D = 128 one warp's reductions cover one contiguous 128-byte
// line); a small kernel then scales and rounds it to bf16.  Q and dO tiles
// (with their L and D values) stream through a two-stage ring so the next
// step's loads overlap the current step.
//
// Warp roles (12 warps): warps 0-3 and 4-7 each own half of the 128 query
// columns of S^T / dP^T for all 128 key rows (one key row per thread, its
// TMEM lane): they form P^T, write it to TMEM as bf16, form dS^T and write
// it to shared memory in the 128-byte-swizzled layout the MMA reads, drain
// dQ, and finally write dK and dV.  Warp 8 loads tiles (TMA) and the L / D
// vectors; warp 9 issues the MMAs; warps 10-11 only complete the third
// warpgroup, whose register limit is lowered so the first two can raise
// theirs (setmaxnreg).
#include <math.h>

#include "fa_dropout.cuh"
#include "fa_internal.cuh"
#include "fa_tmap.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

using namespace ptx;

constexpr int kBM = 128;  // queries per tile
constexpr int kBN = 128;  // keys per tile (one per CTA)
constexpr int kThreads = 384;
constexpr int kTmaWarp = 8;
constexpr int kMmaWarp = 9;

struct BwdParams {
  CUtensorMap tq, tk, tv, tdo;
  DropParams drop;  // used by the dropout instantiation only
  const float* lse;
  const float* dvec;
  float* dq_acc;
  __nv_bfloat16* dk;  // 16-bit storage: bf16 or fp16 per F16
  __nv_bfloat16* dv;
  const int32_t* cu;
  unsigned* status;
  unsigned long long limit_ns;
  int B, H, N, T;
  float c2;  // scale * log2(e)
  float scale;
  int causal;
};

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

template <int D>
struct BwdCfg {
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kHalfBytes = 16384;  // 128 rows x 128 bytes
  static constexpr int kHalves = D / 64;
  // dQ^T = K^T dS^T (head width on TMEM lanes: coalesced reductions) needs
  // M = D = 128; at D = 64 the kernel forms dQ = dS K (queries on lanes).
  static constexpr bool kDqTransposed = D == 128;
  // Dynamic shared memory only (the tiles need a 1024-byte aligned base, which
  // the kernel checks): K, V, a 2-stage ring of Q and dO, dS^T, then the L / D
  // vectors of both stages and the barriers.
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kTileBytes;
  static constexpr int kQOff = 2 * kTileBytes;         // + stage * kTileBytes
  static constexpr int kDOOff = 4 * kTileBytes;        // + stage * kTileBytes
  static constexpr int kDSOff = 6 * kTileBytes;        // [128 keys][128 queries] bf16
  static constexpr int kLOff = kDSOff + 2 * kHalfBytes;  // 2 x 128 floats: L_i * log2(e)
  static constexpr int kDvOff = kLOff + 1024;            // 2 x 128 floats: D_i
  static constexpr int kBarOff = kDvOff + 1024;          // 16 mbarriers
  static constexpr int kMiscOff = kBarOff + 16 * 8;      // TMEM base, abort flag
  static constexpr int kSmemBytes = kMiscOff + 16;
  static_assert(kSmemBytes <= 232448, "backward tiles exceed the shared-memory limit");
};

// kDq = false: dK and dV only (the deterministic backward takes dQ from the
// query-stationary kernel in fa_tc_bwd_dq.cu).
template <int D, bool F16, bool kDrop, bool kDq>
__global__ void __launch_bounds__(kThreads, 1) tc_bwd_kernel(const __grid_constant__ BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (smem_u32(smem) & 1023u) {  // the swizzled tile layout needs a 1024-byte aligned base
    if (threadIdx.x == 0) atomicOr(p.status, kDevInternal);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* bar_kv = bars + 0;
  uint64_t* bar_qf = bars + 1;  // [2] Q tile + L / D of a stage loaded
  uint64_t* bar_qe = bars + 3;  // [2] stage's Q / L / D free (dK done)
  uint64_t* bar_of = bars + 5;  // [2] dO tile loaded
  uint64_t* bar_oe = bars + 7;  // [2] dO stage free (dV done)
  uint64_t* bar_s = bars + 9;
  uint64_t* bar_dp = bars + 10;
  uint64_t* bar_p = bars + 11;
  uint64_t* bar_ds = bars + 12;
  uint64_t* bar_dq = bars + 13;
  uint64_t* bar_dqfree = bars + 14;
  uint64_t* bar_done = bars + 15;
  uint32_t* tmem_base_sh = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
  int* abort_flag = reinterpret_cast<int*>(smem + C::kMiscOff + 4);

  const int b = blockIdx.z, h = blockIdx.y, kt = blockIdx.x;
  int len, row0, slab;
  long long out_base;
  if (p.cu != nullptr) {
    const int s0 = p.cu[b], s1 = p.cu[b + 1];
    if (s0 < 0 || s1 < s0 || s1 > p.T || s1 - s0 > p.N) {
      if (threadIdx.x == 0) atomicOr(p.status, kDevBadSeqlens);
      return;
    }
    len = s1 - s0;
    row0 = s0;
    slab = h;
    out_base = (long long)h * p.T + s0;
  } else {
    len = p.N;
    row0 = 0;
    slab = b * p.H + h;
    out_base = (long long)slab * p.N;
  }
  const int n_t = (len + kBM - 1) / kBM;  // query tiles = key tiles
  if (kt >= n_t) return;
  const int q_first = p.causal ? kt : 0;  // earlier query tiles never see these keys
  const int n_steps = n_t - q_first;

  if (threadIdx.x == 0) {
    mbar_init(bar_kv, 1);
    for (int st = 0; st < 2; ++st) {
      mbar_init(bar_qf + st, 1);
      mbar_init(bar_qe + st, 1);
      mbar_init(bar_of + st, 1);
      mbar_init(bar_oe + st, 1);
    }
    mbar_init(bar_s, 1);
    mbar_init(bar_dp, 1);
    mbar_init(bar_p, 8);
    mbar_init(bar_ds, 8);
    mbar_init(bar_dq, 1);
    mbar_init(bar_dqfree, 8);
    mbar_init(bar_done, 1);
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
  float* s_l = reinterpret_cast<float*>(smem + C::kLOff);
  float* s_d = reinterpret_cast<float*>(smem + C::kDvOff);

  if (warp < 8) {
    // ------------------------------------------------------------ P, dS, dQ drain, epilogue
    setmaxnreg_inc<kComputeRegs>();
    const int ch = warp >> 2;        // query-column half
    const int quad = warp & 3;       // TMEM lanes 32*quad ..
    const int j = quad * 32 + lane;  // this thread's TMEM lane: key row (and d or query row for dQ)
    const int key = kt * kBN + j;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t t_s = tmem + lane_off + ch * 64;
    const uint32_t t_dp = tmem + lane_off + 128 + ch * 64;
    uint8_t* ds_row = smem + C::kDSOff + ch * C::kHalfBytes + (j >> 3) * 1024 + (j & 7) * 128;
    bool ok = true;
    for (int k = 0; k < n_steps; ++k) {
      const int qi = q_first + k;
      const int st = k & 1;
      const float* sl = s_l + st * 128 + ch * 64;
      const float* sd = s_d + st * 128 + ch * 64;
      // dropout decisions of (this half's 64 queries, this key), regenerated
      uint64_t keepm = ~0ull;
      if constexpr (kDrop)
        keepm = keep64_keys_on_lanes(p.drop, (uint32_t)key, (uint32_t)(qi * kBM + ch * 64), (uint32_t)(b * p.H + h),
                                     lane);
      // L / D of this query tile are visible once bar_qf completes; S^T once bar_s does
      if (!warp_wait(bar_qf + st, (k >> 1) & 1, w) || !warp_wait(bar_s, k & 1, w)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sv[2][32];
      tmem_ld32(t_s, sv[0]);
      tmem_ld32(t_s + 32, sv[1]);
      tmem_ld_wait(sv[0]);
      tmem_ld_wait(sv[1]);
      const bool mask = (p.causal && qi == kt) || (kt * kBN + kBN > len) || (qi * kBM + kBM > len);
      const int q0 = qi * kBM + ch * 64;  // first query (within the sequence) of this half
      float pr[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const float x = fmaf(__uint_as_float(sv[c >> 5][c & 31]), p.c2, -sl[c]);
        float pv = ex2_approx(x);
        if (mask) {
          const int q = q0 + c;
          if (q >= len || key >= len || (p.causal && key > q)) pv = 0.f;
        }
        pr[c] = pv;
      }
      {
        // P^T as bf16 pairs into this half's first 32 score columns (already read)
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
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_p);

      if (!warp_wait(bar_dp, k & 1, w)) {
        ok = false;
        break;
      }
      tc_fence_after();
      tmem_ld32(t_dp, sv[0]);
      tmem_ld32(t_dp + 32, sv[1]);
      tmem_ld_wait(sv[0]);
      tmem_ld_wait(sv[1]);
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8) {
        uint32_t u[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int c = c8 * 8 + 2 * e;
          float dp0 = __uint_as_float(sv[c >> 5][c & 31]), dp1 = __uint_as_float(sv[(c + 1) >> 5][(c + 1) & 31]);
          if constexpr (kDrop) {  // dP of the dropped weights: masked and scaled like them
            dp0 = (keepm >> c) & 1 ? dp0 * p.drop.scale : 0.f;
            dp1 = (keepm >> (c + 1)) & 1 ? dp1 * p.drop.scale : 0.f;
          }
          const float d0 = pr[c] * (dp0 - sd[c]);
          const float d1 = pr[c + 1] * (dp1 - sd[c + 1]);
          u[e] = pack16x2<F16>(d0, d1);
        }
        // 128-byte swizzle: 16-byte chunk c8 of row j sits at chunk c8 ^ (j % 8)
        *reinterpret_cast<uint4*>(ds_row + ((c8 ^ (j & 7)) << 4)) = make_uint4(u[0], u[1], u[2], u[3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_ds);

      if constexpr (!kDq) continue;
      // dQ of this query tile into the float32 accumulator
      if (!warp_wait(bar_dq, k & 1, w)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if constexpr (C::kDqTransposed) {
        // dQ^T: lane j holds head-width column j for this half's 64 queries, so
        // a warp's 32 reductions for one query cover 128 contiguous bytes.
        tmem_ld32(tmem + lane_off + ch * 64, sv[0]);
        tmem_ld32(tmem + lane_off + ch * 64 + 32, sv[1]);
        tmem_ld_wait(sv[0]);
        tmem_ld_wait(sv[1]);
        float* dst = p.dq_acc + (out_base + q0) * D + j;
        const int nq = min(64, len - q0);
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c < nq) atomicAdd(dst + c * D, __uint_as_float(sv[c >> 5][c & 31]));
      } else {
        // dQ: lane j holds query row qi*128 + j, this half's D/2 columns
        const int q = qi * kBM + j;
        float* dst = p.dq_acc + (out_base + q) * D + ch * (D / 2);
        const uint32_t t_dq = tmem + lane_off + ch * (D / 2);
#pragma unroll 1
        for (int c = 0; c < D / 2; c += 32) {
          uint32_t v[32];
          tmem_ld32(t_dq + c, v);
          tmem_ld_wait(v);
          if (q < len) {
#pragma unroll
            for (int e = 0; e < 32; e += 4)
              red_add_v4(dst + c + e, __uint_as_float(v[e]), __uint_as_float(v[e + 1]), __uint_as_float(v[e + 2]),
                         __uint_as_float(v[e + 3]));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_dqfree);
    }
    // epilogue: dV and dK rows of this CTA's keys
    if (ok && warp_wait(bar_done, 0, w)) {
      tc_fence_after();
      const bool row_ok = key < len;
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        __nv_bfloat16* out = (which == 0 ? p.dv : p.dk) + (out_base + key) * D + ch * (D / 2);
        const float mul = which == 0 ? 1.f : p.scale;
        const uint32_t t_acc = tmem + lane_off + (which == 0 ? 256 : 384) + ch * (D / 2);
#pragma unroll 1
        for (int c = 0; c < D / 2; c += 32) {
          uint32_t v[32];
          tmem_ld32(t_acc + c, v);
          tmem_ld_wait(v);
          if (row_ok) {
            uint4* dst = reinterpret_cast<uint4*>(out + c);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) {
              uint4 u;
              u.x = pack16x2<F16>(__uint_as_float(v[8 * v4 + 0]) * mul, __uint_as_float(v[8 * v4 + 1]) * mul);
              u.y = pack16x2<F16>(__uint_as_float(v[8 * v4 + 2]) * mul, __uint_as_float(v[8 * v4 + 3]) * mul);
              u.z = pack16x2<F16>(__uint_as_float(v[8 * v4 + 4]) * mul, __uint_as_float(v[8 * v4 + 5]) * mul);
              u.w = pack16x2<F16>(__uint_as_float(v[8 * v4 + 6]) * mul, __uint_as_float(v[8 * v4 + 7]) * mul);
              dst[v4] = u;
            }
          }
        }
      }
    }
  } else {
    // warps 8-11: producer, MMA issuer and two idle warps completing the warpgroup
    setmaxnreg_dec<kSupportRegs>();
    if (warp == kTmaWarp) {
      // ---------------------------------------------------------- producer
      if (lane == 0) {
        tma_prefetch_desc(&p.tq);
        tma_prefetch_desc(&p.tk);
        tma_prefetch_desc(&p.tv);
        tma_prefetch_desc(&p.tdo);
        mbar_arrive_expect_tx(bar_kv, 2 * C::kTileBytes);
        for (int hf = 0; hf < C::kHalves; ++hf) {
          tma_load_3d(smem + C::kKOff + hf * C::kHalfBytes, &p.tk, bar_kv, hf * 64, row0 + kt * kBN, slab);
          tma_load_3d(smem + C::kVOff + hf * C::kHalfBytes, &p.tv, bar_kv, hf * 64, row0 + kt * kBN, slab);
        }
      }
      int q_issued = 0, o_issued = 0;
      for (int k = 0; k < n_steps; ++k) {
        const int qi = q_first + k;
        const int st = k & 1;
        // Stage st was last used by step k - 2; its Q / L / D are free once that
        // step's dK (their last reader) has completed, its dO once that step's
        // dV has.  Lane 0 waits and the answer is broadcast, so the warp never
        // splits.
        int good = 1;
        if (lane == 0 && k >= 2) good = mbar_wait(bar_qe + st, ((k >> 1) - 1) & 1, w);
        if (!__shfl_sync(0xffffffffu, good, 0)) break;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int r = lane * 4 + e;
          const int qrow = qi * kBM + r;
          const bool in = qrow < len;
          s_l[st * 128 + r] = in ? p.lse[out_base + qrow] * kLog2e : 0.f;
          s_d[st * 128 + r] = in ? p.dvec[out_base + qrow] : 0.f;
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_expect_tx(bar_qf + st, C::kTileBytes);
          for (int hf = 0; hf < C::kHalves; ++hf)
            tma_load_3d(smem + C::kQOff + st * C::kTileBytes + hf * C::kHalfBytes, &p.tq, bar_qf + st, hf * 64,
                        row0 + qi * kBM, slab);
        }
        q_issued = k + 1;
        if (lane == 0 && k >= 2) good = mbar_wait(bar_oe + st, ((k >> 1) - 1) & 1, w);
        if (!__shfl_sync(0xffffffffu, good, 0)) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(bar_of + st, C::kTileBytes);
          for (int hf = 0; hf < C::kHalves; ++hf)
            tma_load_3d(smem + C::kDOOff + st * C::kTileBytes + hf * C::kHalfBytes, &p.tdo, bar_of + st,
                        hf * 64, row0 + qi * kBM, slab);
        }
        o_issued = k + 1;
      }
      if (lane == 0 && *abort_flag) {
        // let copies already in flight land before the CTA's memory is released
        mbar_wait_drain(bar_kv, 0, p.limit_ns);
        for (int k = max(0, q_issued - 2); k < q_issued; ++k) mbar_wait_drain(bar_qf + (k & 1), (k >> 1) & 1, p.limit_ns);
        for (int k = max(0, o_issued - 2); k < o_issued; ++k) mbar_wait_drain(bar_of + (k & 1), (k >> 1) & 1, p.limit_ns);
      }
    } else if (warp == kMmaWarp && lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      const uint32_t id_nn = idesc16<F16>(128, 128, false, false);  // S^T, dP^T
      const uint32_t id_acc = idesc16<F16>(128, D, false, true);    // dV, dK: A K-major, B MN-major
      // dQ^T = K^T dS^T (M = D) or dQ = dS K (N = D): A and B both MN-major
      const uint32_t id_dq = C::kDqTransposed ? idesc16<F16>(128, 128, true, true) : idesc16<F16>(128, D, true, true);
      const uint32_t sk = smem_u32(smem + C::kKOff), sv = smem_u32(smem + C::kVOff);
      const uint32_t sq = smem_u32(smem + C::kQOff), sdo = smem_u32(smem + C::kDOOff);
      const uint32_t sds = smem_u32(smem + C::kDSOff);
      // Descriptors are built once and advanced by adding (byte offset >> 4)
      // to their start-address field.  k* = K-major view, m* = MN-major view.
      const uint64_t kK = sdesc_sw128(sk, 16, 1024), kV = sdesc_sw128(sv, 16, 1024);
      const uint64_t kQ = sdesc_sw128(sq, 16, 1024), kDO = sdesc_sw128(sdo, 16, 1024);
      const uint64_t kDS = sdesc_sw128(sds, 16, 1024);
      const uint64_t mQ = sdesc_sw128(sq, C::kHalfBytes, 1024), mDO = sdesc_sw128(sdo, C::kHalfBytes, 1024);
      const uint64_t mK = sdesc_sw128(sk, C::kHalfBytes, 1024), mDS = sdesc_sw128(sds, C::kHalfBytes, 1024);
      constexpr uint32_t kStageDesc = C::kTileBytes >> 4;
      // X^T = A B^T over the head width: A, B both [128 rows][D] K-major,
      // D/16 MMAs issued back to back
      auto issue_nn = [&](uint32_t d_col, uint64_t a0, uint64_t b0) {
        if constexpr (D == 128) {
          uint64_t a[8], b[8];
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t off = ((ks >> 2) * C::kHalfBytes + (ks & 3) * 32) >> 4;
            a[ks] = a0 + off;
            b[ks] = b0 + off;
          }
          mma_ss_x8(tmem + d_col, a, b, id_nn, 0u);
        } else {
          uint64_t a[4], b[4];
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            a[ks] = a0 + ks * 2;
            b[ks] = b0 + ks * 2;
          }
          mma_ss_x4(tmem + d_col, a, b, id_nn, 0u);
        }
      };
      bool ok = mbar_wait(bar_kv, 0, w);
      for (int k = 0; ok && k < n_steps; ++k) {
        const int st = k & 1;
        const uint32_t acc0 = k > 0 ? 1u : 0u;
        if (!mbar_wait(bar_qf + st, (k >> 1) & 1, w) || !mbar_wait(bar_of + st, (k >> 1) & 1, w)) break;
        tc_fence_after();
        // dP^T = V dO^T: its columns were consumed before the previous dS was published
        issue_nn(128, kV, kDO + st * kStageDesc);
        mma_commit(bar_dp);
        // S^T = K Q^T into the columns the previous dQ used, once it is drained
        if (kDq && k > 0) {
          if (!mbar_wait(bar_dqfree, (k - 1) & 1, w)) break;
          tc_fence_after();
        }
        issue_nn(0, kK, kQ + st * kStageDesc);
        mma_commit(bar_s);
        // dV += P^T dO: P^T (bf16) in TMEM, columns [0,32) for queries 0-63 and
        // [64,96) for queries 64-127; dO MN-major
        if (!mbar_wait(bar_p, k & 1, w)) break;
        tc_fence_after();
        {
          uint32_t at[8];
          uint64_t b[8];
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            at[ks] = tmem + (ks >> 2) * 64 + (ks & 3) * 8;
            b[ks] = mDO + st * kStageDesc + ((ks * 2048) >> 4);
          }
          mma_ts_x8(tmem + 256, at, b, id_acc, acc0);
        }
        mma_commit(bar_oe + st);
        // dK += dS^T Q: dS^T K-major from shared memory, Q MN-major
        if (!mbar_wait(bar_ds, k & 1, w)) break;
        tc_fence_after();
        {
          uint64_t a[8], b[8];
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            a[ks] = kDS + (((ks >> 2) * C::kHalfBytes + (ks & 3) * 32) >> 4);
            b[ks] = mQ + st * kStageDesc + ((ks * 2048) >> 4);
          }
          mma_ss_x8(tmem + 384, a, b, id_acc, acc0);
        }
        mma_commit(bar_qe + st);
        // dQ over the 128 keys (K = 16 keys per MMA): the dS buffer read MN-major
        // (queries contiguous) and K read MN-major (head width contiguous)
        if constexpr (kDq) {
          uint64_t a[8], b[8];
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            a[ks] = (C::kDqTransposed ? mK : mDS) + ((ks * 2048) >> 4);
            b[ks] = (C::kDqTransposed ? mDS : mK) + ((ks * 2048) >> 4);
          }
          mma_ss_x8(tmem + 0, a, b, id_dq, 0u);
          mma_commit(bar_dq);
        }
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

// dQ = scale * dQ_acc rounded to the 16-bit input type, four elements per thread.
template <bool F16>
__global__ void __launch_bounds__(256) dq_convert_kernel(const float4* __restrict__ acc, uint2* __restrict__ dq,
                                                         long long n4, float scale) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (long long)gridDim.x * blockDim.x) {
    const float4 a = acc[i];
    dq[i] = make_uint2(pack16x2<F16>(a.x * scale, a.y * scale), pack16x2<F16>(a.z * scale, a.w * scale));
  }
}

template <int D, bool F16, bool kDrop, bool kDq>
cudaError_t launch_bwd_d(const Problem& p, cudaStream_t s) {
  using C = BwdCfg<D>;
  BwdParams bp;
  if (!make_map16(&bp.tq, p.q, p, kBM) || !make_map16(&bp.tk, p.k, p, kBN) ||
      !make_map16(&bp.tv, p.v, p, kBN) || !make_map16(&bp.tdo, p.dout, p, kBM))
    return note_error("backward tensor map encode", cudaErrorInvalidValue);
  bp.lse = p.lse;
  bp.dvec = p.dvec;
  bp.dq_acc = p.dq_acc;
  bp.dk = static_cast<__nv_bfloat16*>(p.dk);
  bp.dv = static_cast<__nv_bfloat16*>(p.dv);
  bp.cu = p.cu;
  bp.status = p.status;
  bp.limit_ns = p.wait_limit_ns;
  bp.B = p.B;
  bp.H = p.H;
  bp.N = p.N;
  bp.T = p.T;
  bp.c2 = p.scale * kLog2e;
  bp.scale = p.scale;
  bp.causal = p.causal;
  bp.drop = drop_params_of(p);
  cudaError_t e = cudaFuncSetAttribute(tc_bwd_kernel<D, F16, kDrop, kDq>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return note_error("backward smem attribute", e);
  dim3 grid((p.N + kBN - 1) / kBN, p.H, p.B);
  tc_bwd_kernel<D, F16, kDrop, kDq><<<grid, kThreads, C::kSmemBytes, s>>>(bp);
  note_launches(1);
  return note_error("backward launch", cudaGetLastError());
}

}  // namespace

cudaError_t launch_dq_convert(const Problem& p, cudaStream_t s) {
  const int D = p.D;
  const long long n4 = p.rows() * D / 4;
  const long long want = (n4 + 255) / 256;
  const int blocks = (int)(want < 152 * 16 ? want : 152 * 16);
  const float4* acc = reinterpret_cast<const float4*>(p.dq_acc);
  uint2* dq = static_cast<uint2*>(p.dq);
  if (p.f16)
    dq_convert_kernel<true><<<blocks, 256, 0, s>>>(acc, dq, n4, p.scale);
  else
    dq_convert_kernel<false><<<blocks, 256, 0, s>>>(acc, dq, n4, p.scale);
  note_launches(1);
  return note_error("dq convert launch", cudaGetLastError());
}


cudaError_t launch_tc_bwd(const Problem& p, cudaStream_t s) {
  if (p.D == 64) {
    if (p.dropout) return p.f16 ? launch_bwd_d<64, true, true, true>(p, s) : launch_bwd_d<64, false, true, true>(p, s);
    return p.f16 ? launch_bwd_d<64, true, false, true>(p, s) : launch_bwd_d<64, false, false, true>(p, s);
  }
  if (p.D == 128) return launch_tc_bwd128(p, s);
  return cudaErrorInvalidValue;
}

// dK and dV without the dQ product (deterministic backward); D = 128 uses the
// dedicated kernel of fa_tc_bwd128.cu.
template <int D>
cudaError_t launch_dkdv_d(const Problem& p, cudaStream_t s) {
  if (p.dropout) return p.f16 ? launch_bwd_d<D, true, true, false>(p, s) : launch_bwd_d<D, false, true, false>(p, s);
  return p.f16 ? launch_bwd_d<D, true, false, false>(p, s) : launch_bwd_d<D, false, false, false>(p, s);
}

cudaError_t launch_tc_bwd_dkdv(const Problem& p, cudaStream_t s) {
  if (p.D == 64) return launch_dkdv_d<64>(p, s);
  if (p.D == 128) return launch_tc_bwd128_dkdv(p, s);
  return cudaErrorInvalidValue;
}

}  // namespace fa
