// Tensor-core forward kernel for sm_103a (bf16 in, fp32 accumulate).
//
// The method is the query-first tiled schedule of tensortonic.com
// "FlashAttention" section 6 with the running softmax of section 5: a CTA
// owns two 128-row query tiles of one (sequence, head), loads them once, and
// visits the allowed 128-key K/V tiles in turn.  The score tile and the
// output accumulator never leave the SM: S = Q K^T and u += P V are tcgen05
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

#include "fa_dropout.cuh"
#include "fa_internal.cuh"
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
  __shared__ __align__(8) uint64_t bar_q, bar_done;
  // bar_q: both Q tiles and K_0; bar_kv[j % stages]: V_j and K_{j+1} (the two loads one
  // stage release allows, so the MMA thread waits once per step for its operands)
  __shared__ __align__(8) uint64_t bar_kv[C::kStages], bar_kfree[C::kStages], bar_vfree[C::kStages];
  __shared__ __align__(8) uint64_t bar_s[2], bar_p[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // causal: pairs of late query tiles see the most keys and are handed out first
  const GridItem item = p.causal ? grouped_heavy_first(kFwdHeadGroup) : GridItem{(int)blockIdx.x, (int)blockIdx.z, (int)blockIdx.y};
  const int b = item.b, h = item.h;

  // ---- the (sequence, head) this CTA works on
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
  const int n_qt = (len + kBM - 1) / kBM;
  const int n_pairs = (n_qt + 1) / 2;
  const int pair = p.causal ? (int)gridDim.x - 1 - item.rank : item.rank;
  if (pair >= n_pairs) return;
  const int qt0 = 2 * pair;
  const int n_kv = (len + kBN - 1) / kBN;
  int nkv[2];
  nkv[0] = p.causal ? min(qt0 + 1, n_kv) : n_kv;
  nkv[1] = (qt0 + 1 < n_qt) ? (p.causal ? min(qt0 + 2, n_kv) : n_kv) : 0;
  const int nmax = max(nkv[0], nkv[1]);
  const int t_last = nkv[1] > 0 ? 1 : 0;  // its MMAs are issued last in every step; nkv[t_last] == nmax

  if (threadIdx.x == 0) {
    mbar_init(&bar_q, 1);
    mbar_init(&bar_done, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bar_kv[s], 1);
      mbar_init(&bar_kfree[s], 1);
      mbar_init(&bar_vfree[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bar_s[t], 1);
      mbar_init(&bar_p[t], 4);  // one arrival per softmax warp
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
    const int qt = qt0 + t;
    const int n = nkv[t];
    if (n > 0) {
      const int i = qt * kBM + r;       // row within the sequence
      const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
      const uint32_t t_s = tmem + lane_off + t * 128;
      const uint32_t t_o = tmem + lane_off + 256 + t * 128;
      float m_ref = -INFINITY;          // reference maximum of the exponentials (log2 units)
      float l = 0.f;
      bool ok = true;
      for (int j = 0; j < n; ++j) {
        if (!warp_wait(&bar_s[t], j & 1, w)) {
          ok = false;
          break;
        }
        if (t == t_last && quad == 0 && lane == 0) {
          // S_t(j) of the last query tile is complete, and with it every MMA issued
          // before it: S_0(j) (K_j is consumed) and both tiles' P V_{j-1}
          mbar_arrive(&bar_kfree[j % C::kStages]);
          if (j > 0) mbar_arrive(&bar_vfree[(j - 1) % C::kStages]);
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
        // row maximum of the raw scores (scale > 0 preserves the order)
        float mt = -INFINITY;
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; e += 2) mt = fmax3(mt, __uint_as_float(sr[c][e]), __uint_as_float(sr[c][e + 1]));
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
        uint32_t kbits = 0;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int e0 = 64 * hf + 2 * c;
            float a0, a1;
            ffma2(a0, a1, __uint_as_float(sr[e0 >> 5][e0 & 31]), __uint_as_float(sr[(e0 + 1) >> 5][(e0 + 1) & 31]),
                  p.c2, nmu, nmu);
            const float p0 = ex2_approx(a0);
            const float p1 = ex2_approx(a1);
            fadd2(rs0, rs1, p0, p1);  // the normaliser is that of the undropped weights
            if constexpr (kDrop) {
              // dropped weights enter PV scaled by 1 / (1 - p); one generator call per 4 keys
              if ((c & 1) == 0) kbits = keep4(p.drop, (uint32_t)i, (uint32_t)(k0 + e0), (uint32_t)(b * p.H + h));
              const uint32_t sh = (c & 1) * 2;
              pk[c] = pack16x2<F16>((kbits >> sh) & 1u ? p0 * p.drop.scale : 0.f,
                                    (kbits >> (sh + 1)) & 1u ? p1 * p.drop.scale : 0.f);
            } else {
              pk[c] = pack16x2<F16>(p0, p1);
            }
          }
          tmem_st32(t_s + 32 * hf, pk);
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
      if (ok && warp_wait(&bar_s[t], n & 1, w)) {
        tc_fence_after();
        const bool row_ok = i < len;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        __nv_bfloat16* orow = p.o + (out_base + i) * D;
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
        if (row_ok) p.lse[out_base + i] = l > 0.f ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
      }
    }
  } else {
    // warps 8-11: producer, MMA issuer and two idle warps completing the warpgroup
    setmaxnreg_dec<kSupportRegs>();
    if (warp == kTmaWarp && lane == 0) {
      // ---------------------------------------------------------- producer
      tma_prefetch_desc(&p.tq);
      tma_prefetch_desc(&p.tk);
      tma_prefetch_desc(&p.tv);
      const int nq = nkv[1] > 0 ? 2 : 1;
      auto load_k = [&](int j, uint64_t* bar) {
        for (int hf = 0; hf < C::kHalves; ++hf)
          tma_load_3d(smem + C::kKOff + (j % C::kStages) * C::kTileBytes + hf * C::kHalfBytes, &p.tk, bar, hf * 64,
                      row0 + j * kBN, slab);
      };
      mbar_arrive_expect_tx(&bar_q, (nq + 1) * C::kTileBytes);
      for (int t = 0; t < nq; ++t)
        for (int hf = 0; hf < C::kHalves; ++hf)
          tma_load_3d(smem + C::kQOff + t * C::kTileBytes + hf * C::kHalfBytes, &p.tq, &bar_q, hf * 64,
                      row0 + (qt0 + t) * kBM, slab);
      load_k(0, &bar_q);
      // Stage release: the softmax thread that waits for the last query tile's
      // S(j) arrives on kfree[j % stages] (K_j consumed: S_0(j) precedes S_1(j))
      // and on vfree[(j-1) % stages] (both P V_{j-1} precede S_1(j)).  V_j and
      // K_{j+1} both need the release of softmax step j + 1 - stages, so they
      // share one barrier, and K runs a step ahead of V without costing the MMA
      // thread a commit.  Each wait below is unambiguous: the next completion of
      // the barrier it polls needs a load issued after the wait.
      int issued = 0;
      for (int j = 0; j < nmax; ++j) {
        const int s = j % C::kStages;
        const bool k_next = j + 1 < nmax;
        if (j >= C::kStages && !mbar_wait(&bar_vfree[s], (j / C::kStages - 1) & 1, w)) break;
        if (k_next && j + 1 >= C::kStages &&
            !mbar_wait(&bar_kfree[(j + 1) % C::kStages], ((j + 1) / C::kStages - 1) & 1, w))
          break;
        mbar_arrive_expect_tx(&bar_kv[s], (k_next ? 2 : 1) * C::kTileBytes);
        for (int hf = 0; hf < C::kHalves; ++hf)
          tma_load_3d(smem + C::kVOff + s * C::kTileBytes + hf * C::kHalfBytes, &p.tv, &bar_kv[s], hf * 64,
                      row0 + j * kBN, slab);
        if (k_next) load_k(j + 1, &bar_kv[s]);
        issued = j + 1;
      }
      if (abort_flag) {
        // let copies already in flight land before the CTA's memory is released
        mbar_wait_drain(&bar_q, 0, p.limit_ns);
        for (int j = max(0, issued - C::kStages); j < issued; ++j)
          mbar_wait_drain(&bar_kv[j % C::kStages], (j / C::kStages) & 1, p.limit_ns);
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
      bool ok = mbar_wait(&bar_q, 0, w);
      if (ok) {
        tc_fence_after();
        for (int t = 0; t < 2; ++t)
          if (nkv[t] > 0) {
            issue_s(t, 0);
            mma_commit(&bar_s[t]);
          }
      }
      for (int j = 0; ok && j < nmax; ++j) {
        const int s = j % C::kStages, s1 = (j + 1) % C::kStages;
        // V_j and K_{j+1}
        if (!mbar_wait(&bar_kv[s], (j / C::kStages) & 1, w)) break;
        tc_fence_after();
        for (int t = 0; t < 2; ++t) {
          if (j >= nkv[t]) continue;
          if (!mbar_wait(&bar_p[t], j & 1, w)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_pv(t, s, j > 0);
          if (j + 1 < nkv[t]) issue_s(t, s1);
          mma_commit(&bar_s[t]);
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
cudaError_t launch_fwd_d(const Problem& p, cudaStream_t s) {
  using C = FwdCfg<D>;
  FwdParams fp;
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
  const int n_qt = (p.N + kBM - 1) / kBM;
  dim3 grid((n_qt + 1) / 2, p.H, p.B);
  tc_fwd_kernel<D, F16, kDrop><<<grid, kThreads, C::kSmemBytes, s>>>(fp);
  note_launches(1);
  return note_error("forward launch", cudaGetLastError());
}

}  // namespace

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
