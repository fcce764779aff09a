// dQ without atomics: the query-stationary half of a deterministic backward
// pass (tensortonic.com "FlashAttention" section 7 rebuilds the weights tile
// by tile from the saved log-sum-exp; the same products, scheduled per query
// tile instead of per key tile, let dQ accumulate in tensor memory and be
// written once).  A CTA owns one 128-query tile (Q, dO and the rows' L and D
// stay put) and streams the K / V tiles it can see:
//     S_j  = Q K_j^T      -> TMEM [0,128) or [128,256) (alternating)
//     dP_j = dO V_j^T     -> TMEM [256,384), then dS_j (bf16) over its columns
//     dQ  += dS_j K_j     (A = dS from tensor memory, K_j MN-major)
//                         -> TMEM [384,384+D)
// with P_ij = exp(s_ij - L_i) and dS = P o (dP - D_i).  The order per step is
// S_{j+1}, [dS_j ready] dQ_j, dP_{j+1}, so the next scores are formed while
// the compute warps build dS_j.  The key-stationary kernel (fa_tc_bwd.cu,
// without its dQ product) supplies dK and dV; together they give a backward
// whose every sum is taken in a fixed order.
//
// Warp roles (12 warps): 0-3 and 4-7 build P and dS for key columns [0,64)
// and [64,128) of the tile (one query row per thread, its TMEM lane); 8 =
// TMA producer; 9 = MMA issuer; 10-11 idle.  Registers: 168 at launch, 200 for
// the compute warpgroups and 104 for the rest (setmaxnreg).
#include <math.h>

#include "fa_dropout.cuh"
#include "fa_internal.cuh"
#include "fa_tmap.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

using namespace ptx;

constexpr int kBM = 128;  // queries per CTA
constexpr int kBN = 128;  // keys per step
constexpr int kThreads = 384;
constexpr int kTmaWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kDqHeadGroup = 16;  // heads per group of the causal block order

struct DqParams {
  CUtensorMap tq, tk, tv, tdo;
  DropParams drop;
  const float* lse;
  const float* dvec;
  __nv_bfloat16* dq;  // 16-bit storage: bf16 or fp16 per F16
  const int32_t* cu;
  unsigned* status;
  unsigned long long limit_ns;
  int B, H, N, T;
  float c2;  // scale * log2(e)
  float scale;
  int causal;
};

template <int D>
struct DqCfg {
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kHalfBytes = 16384;
  static constexpr int kHalves = D / 64;
  static constexpr int kQOff = 0;
  static constexpr int kDOOff = kTileBytes;
  static constexpr int kKStages = 3;  // K_j is read until dQ_j, a step after V_j's last reader
  static constexpr int kVStages = 2;
  static constexpr int kKOff = 2 * kTileBytes;                  // + stage * kTileBytes
  static constexpr int kVOff = (2 + kKStages) * kTileBytes;     // + stage * kTileBytes
  static constexpr int kSmemBytes = (2 + kKStages + kVStages) * kTileBytes + 1024;  // + alignment slack
  static_assert(kSmemBytes + 256 <= 232448, "shared-memory budget");
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

template <int D, bool F16, bool kDrop>
__global__ void __launch_bounds__(kThreads, 1) tc_bwd_dq_kernel(const __grid_constant__ DqParams p) {
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  __shared__ __align__(8) uint64_t bar_qdo, bar_s, bar_dp, bar_ds, bar_done;
  __shared__ __align__(8) uint64_t bar_kfull[C::kKStages], bar_kfree[C::kKStages];
  __shared__ __align__(8) uint64_t bar_vfull[C::kVStages], bar_vfree[C::kVStages];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const GridItem item = p.causal ? grouped_heavy_first(kDqHeadGroup)
                                 : GridItem{(int)blockIdx.x, (int)blockIdx.z, (int)blockIdx.y};
  const int b = item.b, h = item.h;
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
  const int n_t = (len + kBM - 1) / kBM;
  // causal: late query tiles see the most keys and are handed out first
  const int qt = p.causal ? (int)gridDim.x - 1 - item.rank : item.rank;
  if (qt >= n_t) return;
  const int n_steps = p.causal ? qt + 1 : n_t;

  if (threadIdx.x == 0) {
    mbar_init(&bar_qdo, 1);
    for (int s = 0; s < C::kKStages; ++s) {
      mbar_init(&bar_kfull[s], 1);
      mbar_init(&bar_kfree[s], 1);
    }
    for (int s = 0; s < C::kVStages; ++s) {
      mbar_init(&bar_vfull[s], 1);
      mbar_init(&bar_vfree[s], 1);
    }
    mbar_init(&bar_s, 1);
    mbar_init(&bar_dp, 1);
    mbar_init(&bar_ds, 8);
    mbar_init(&bar_done, 1);
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
    // ------------------------------------------------------------ P, dS, epilogue
    setmaxnreg_inc<kComputeRegs>();
    const int ch = warp >> 2;         // key-column half
    const int quad = warp & 3;        // TMEM lanes 32*quad ..
    const int r = quad * 32 + lane;   // query row within the tile
    const int i = qt * kBM + r;       // query row within the sequence
    const bool row_ok = i < len;
    const float l2 = row_ok ? p.lse[out_base + i] * kLog2e : 0.f;  // L_i in log2 units
    const float di = row_ok ? p.dvec[out_base + i] : 0.f;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t t_dp = tmem + lane_off + 256 + ch * 64;
    bool ok = true;
    for (int j = 0; j < n_steps; ++j) {
      const int k0 = j * kBN + ch * 64;  // first key (within the sequence) of this half
      ok = ok && warp_wait(&bar_s, j & 1, w);
      tc_fence_after();
      uint32_t sv[2][32];
      const uint32_t t_s = tmem + lane_off + (j & 1) * 128 + ch * 64;
      tmem_ld32(t_s, sv[0]);
      tmem_ld32(t_s + 32, sv[1]);
      tmem_ld_wait(sv[0]);
      tmem_ld_wait(sv[1]);
      float pr[64];
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        float a0, a1;  // s * scale * log2(e) - L * log2(e)
        ffma2(a0, a1, __uint_as_float(sv[c >> 5][c & 31]), __uint_as_float(sv[(c + 1) >> 5][(c + 1) & 31]), p.c2,
              -l2, -l2);
        pr[c] = ex2_approx(a0);
        pr[c + 1] = ex2_approx(a1);
      }
      if ((p.causal && j == qt) || (k0 + 64 > len) || !row_ok) {
        // diagonal or ragged tile: future keys, padding keys and padding rows weigh zero
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const int key = k0 + c;
          if (!row_ok || key >= len || (p.causal && key > i)) pr[c] = 0.f;
        }
      }
      ok = ok && warp_wait(&bar_dp, j & 1, w);
      if (warp == 0 && lane == 0 && ok) {
        // dP_j is complete, and with it every MMA issued before it: dQ_{j-1}, the
        // last reader of K_{j-1}; dP_j itself was V_j's last reader
        if (j > 0) mbar_arrive(&bar_kfree[(j - 1) % C::kKStages]);
        mbar_arrive(&bar_vfree[j % C::kVStages]);
      }
      tc_fence_after();
      tmem_ld32(t_dp, sv[0]);
      tmem_ld32(t_dp + 32, sv[1]);
      tmem_ld_wait(sv[0]);
      tmem_ld_wait(sv[1]);
      uint32_t dsp[32];
      uint32_t kbits = 0xffffffffu;
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        float dp0 = __uint_as_float(sv[c >> 5][c & 31]), dp1 = __uint_as_float(sv[(c + 1) >> 5][(c + 1) & 31]);
        if constexpr (kDrop) {  // dP of the dropped weights: masked and scaled like them
          if ((c & 3) == 0) kbits = keep4(p.drop, (uint32_t)i, (uint32_t)(k0 + c), (uint32_t)(b * p.H + h));
          dp0 = (kbits >> (c & 3)) & 1u ? dp0 * p.drop.scale : 0.f;
          dp1 = (kbits >> ((c & 3) + 1)) & 1u ? dp1 * p.drop.scale : 0.f;
        }
        float t0, t1, d0, d1;  // dS = P o (dP - D)
        fsub2(t0, t1, dp0, dp1, di, di);
        fmul2(d0, d1, pr[c], pr[c + 1], t0, t1);
        dsp[c >> 1] = pack16x2<F16>(d0, d1);
      }
      tmem_st32(t_dp, dsp);  // dS as bf16 pairs over this half's first 32 dP columns (already read)
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_ds);
    }
    // epilogue: dQ row i = scale * accumulator, this half's D/2 columns
    if (ok && warp_wait(&bar_done, 0, w)) {
      tc_fence_after();
      const uint32_t t_acc = tmem + lane_off + 384 + ch * (D / 2);
      uint16_t* out = reinterpret_cast<uint16_t*>(p.dq) + (out_base + i) * D + ch * (D / 2);
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
            u.x = pack16x2<F16>(__uint_as_float(v[8 * v4 + 0]) * p.scale, __uint_as_float(v[8 * v4 + 1]) * p.scale);
            u.y = pack16x2<F16>(__uint_as_float(v[8 * v4 + 2]) * p.scale, __uint_as_float(v[8 * v4 + 3]) * p.scale);
            u.z = pack16x2<F16>(__uint_as_float(v[8 * v4 + 4]) * p.scale, __uint_as_float(v[8 * v4 + 5]) * p.scale);
            u.w = pack16x2<F16>(__uint_as_float(v[8 * v4 + 6]) * p.scale, __uint_as_float(v[8 * v4 + 7]) * p.scale);
            dst[v4] = u;
          }
        }
      }
    }
  } else {
    setmaxnreg_dec<kSupportRegs>();
    if (warp == kTmaWarp && lane == 0) {
      // ---------------------------------------------------------- producer
      tma_prefetch_desc(&p.tq);
      tma_prefetch_desc(&p.tdo);
      tma_prefetch_desc(&p.tk);
      tma_prefetch_desc(&p.tv);
      mbar_arrive_expect_tx(&bar_qdo, 2 * C::kTileBytes);
      for (int hf = 0; hf < C::kHalves; ++hf) {
        tma_load_3d(smem + C::kQOff + hf * C::kHalfBytes, &p.tq, &bar_qdo, hf * 64, row0 + qt * kBM, slab);
        tma_load_3d(smem + C::kDOOff + hf * C::kHalfBytes, &p.tdo, &bar_qdo, hf * 64, row0 + qt * kBM, slab);
      }
      // K_j and V_j both become free when a compute thread sees dP_{j+2} or
      // dP_j complete (K_j's last reader is dQ_j, V_j's is dP_j), i.e. two
      // steps before the ring needs the stage again.  Each wait polls a
      // barrier whose next completion needs the load issued after it.
      int k_issued = 0, v_issued = 0;
      for (int j = 0; j < n_steps; ++j) {
        const int sk = j % C::kKStages, sv = j % C::kVStages;
        if (j >= C::kKStages && !mbar_wait(&bar_kfree[sk], (j / C::kKStages - 1) & 1, w)) break;
        mbar_arrive_expect_tx(&bar_kfull[sk], C::kTileBytes);
        for (int hf = 0; hf < C::kHalves; ++hf)
          tma_load_3d(smem + C::kKOff + sk * C::kTileBytes + hf * C::kHalfBytes, &p.tk, &bar_kfull[sk], hf * 64,
                      row0 + j * kBN, slab);
        k_issued = j + 1;
        if (j >= C::kVStages && !mbar_wait(&bar_vfree[sv], (j / C::kVStages - 1) & 1, w)) break;
        mbar_arrive_expect_tx(&bar_vfull[sv], C::kTileBytes);
        for (int hf = 0; hf < C::kHalves; ++hf)
          tma_load_3d(smem + C::kVOff + sv * C::kTileBytes + hf * C::kHalfBytes, &p.tv, &bar_vfull[sv], hf * 64,
                      row0 + j * kBN, slab);
        v_issued = j + 1;
      }
      if (abort_flag) {
        // let copies already in flight land before the CTA's memory is released
        mbar_wait_drain(&bar_qdo, 0, p.limit_ns);
        for (int j = max(0, k_issued - C::kKStages); j < k_issued; ++j)
          mbar_wait_drain(&bar_kfull[j % C::kKStages], (j / C::kKStages) & 1, p.limit_ns);
        for (int j = max(0, v_issued - C::kVStages); j < v_issued; ++j)
          mbar_wait_drain(&bar_vfull[j % C::kVStages], (j / C::kVStages) & 1, p.limit_ns);
      }
    } else if (warp == kMmaWarp && lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      const uint32_t id_nn = idesc16<F16>(kBM, kBN, false, false);  // S, dP: both K-major
      const uint32_t id_dq = idesc16<F16>(kBM, D, false, true);     // dQ: A (dS) from TMEM, K MN-major
      const uint64_t kQ = sdesc_sw128(smem_u32(smem + C::kQOff), 16, 1024);
      const uint64_t kDO = sdesc_sw128(smem_u32(smem + C::kDOOff), 16, 1024);
      const uint64_t kK = sdesc_sw128(smem_u32(smem + C::kKOff), 16, 1024);
      const uint64_t kV = sdesc_sw128(smem_u32(smem + C::kVOff), 16, 1024);
      const uint64_t mK = sdesc_sw128(smem_u32(smem + C::kKOff), C::kHalfBytes, 1024);
      constexpr uint32_t kStageDesc = C::kTileBytes >> 4;
      // X = A B^T over the head width, A and B both [128 rows][D] K-major
      auto issue_nn = [&](uint32_t d_col, uint64_t a0, uint64_t b0) {
        if constexpr (D == 128) {
          uint64_t a[8], bb[8];
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t off = ((ks >> 2) * C::kHalfBytes + (ks & 3) * 32) >> 4;
            a[ks] = a0 + off;
            bb[ks] = b0 + off;
          }
          mma_ss_x8(tmem + d_col, a, bb, id_nn, 0u);
        } else {
          uint64_t a[4], bb[4];
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            a[ks] = a0 + ks * 2;
            bb[ks] = b0 + ks * 2;
          }
          mma_ss_x4(tmem + d_col, a, bb, id_nn, 0u);
        }
      };
      bool ok = mbar_wait(&bar_qdo, 0, w) && mbar_wait(&bar_kfull[0], 0, w);
      if (ok) {
        tc_fence_after();
        issue_nn(0, kQ, kK);
        mma_commit(&bar_s);
        ok = mbar_wait(&bar_vfull[0], 0, w);
        tc_fence_after();
        if (ok) {
          issue_nn(256, kDO, kV);
          mma_commit(&bar_dp);
        }
      }
      for (int j = 0; ok && j < n_steps; ++j) {
        const int sk = j % C::kKStages, sk1 = (j + 1) % C::kKStages, sv1 = (j + 1) % C::kVStages;
        const bool more = j + 1 < n_steps;
        // S_{j+1} into the other score region (its previous reader, step j - 1,
        // finished with it before publishing dS_{j-1})
        if (more) {
          if (!mbar_wait(&bar_kfull[sk1], ((j + 1) / C::kKStages) & 1, w)) break;
          tc_fence_after();
          issue_nn(((j + 1) & 1) * 128, kQ, kK + sk1 * kStageDesc);
          mma_commit(&bar_s);
        }
        // dQ += dS_j K_j: dS (bf16 pairs) in TMEM columns [256,288) (keys 0-63) and
        // [320,352) (keys 64-127); K_j MN-major (head width contiguous)
        if (!mbar_wait(&bar_ds, j & 1, w)) break;
        tc_fence_after();
        {
          uint32_t at[8];
          uint64_t bb[8];
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            at[ks] = tmem + 256 + (ks >> 2) * 64 + (ks & 3) * 8;
            bb[ks] = mK + sk * kStageDesc + ((ks * 2048) >> 4);
          }
          mma_ts_x8(tmem + 384, at, bb, id_dq, j > 0 ? 1u : 0u);
        }
        // dP_{j+1} over dS_j's columns (dQ_j, issued before, has read them)
        if (more) {
          if (!mbar_wait(&bar_vfull[sv1], ((j + 1) / C::kVStages) & 1, w)) break;
          tc_fence_after();
          issue_nn(256, kDO, kV + sv1 * kStageDesc);
          mma_commit(&bar_dp);
        }
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

template <int D, bool F16, bool kDrop>
cudaError_t launch_dq_t(const Problem& p, cudaStream_t s) {
  using C = DqCfg<D>;
  DqParams dp;
  if (!make_map16(&dp.tq, p.q, p, kBM) || !make_map16(&dp.tk, p.k, p, kBN) || !make_map16(&dp.tv, p.v, p, kBN) ||
      !make_map16(&dp.tdo, p.dout, p, kBM))
    return note_error("dQ tensor map encode", cudaErrorInvalidValue);
  dp.drop = drop_params_of(p);
  dp.lse = p.lse;
  dp.dvec = p.dvec;
  dp.dq = static_cast<__nv_bfloat16*>(p.dq);
  dp.cu = p.cu;
  dp.status = p.status;
  dp.limit_ns = p.wait_limit_ns;
  dp.B = p.B;
  dp.H = p.H;
  dp.N = p.N;
  dp.T = p.T;
  dp.c2 = p.scale * kLog2e;
  dp.scale = p.scale;
  dp.causal = p.causal;
  cudaError_t e = cudaFuncSetAttribute(tc_bwd_dq_kernel<D, F16, kDrop>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmemBytes);
  if (e != cudaSuccess) return note_error("dQ smem attribute", e);
  dim3 grid((p.N + kBM - 1) / kBM, p.H, p.B);
  tc_bwd_dq_kernel<D, F16, kDrop><<<grid, kThreads, C::kSmemBytes, s>>>(dp);
  note_launches(1);
  return note_error("dQ launch", cudaGetLastError());
}

template <int D>
cudaError_t launch_dq_d(const Problem& p, cudaStream_t s) {
  if (p.dropout) return p.f16 ? launch_dq_t<D, true, true>(p, s) : launch_dq_t<D, false, true>(p, s);
  return p.f16 ? launch_dq_t<D, true, false>(p, s) : launch_dq_t<D, false, false>(p, s);
}

}  // namespace

cudaError_t launch_tc_bwd_dq(const Problem& p, cudaStream_t s) {
  if (p.D == 64) return launch_dq_d<64>(p, s);
  if (p.D == 128) return launch_dq_d<128>(p, s);
  return cudaErrorInvalidValue;
}

}  // namespace fa
