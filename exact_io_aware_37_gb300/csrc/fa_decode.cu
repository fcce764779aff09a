// Cached decoding step (tensortonic.com "FlashAttention" section 8: a
// generation step has a few new queries and a long set of cached keys and
// values, a different shape from training; section 9: the newest query is
// aligned with its position in the key cache).  q [B, H, nq, D] against
// k, v [B, H, nk, D]; query row i sits at position nk - nq + i, so causal
// allows key j iff j <= i + (nk - nq).
//
// The work is a stream over K and V with a handful of query rows, bound by
// HBM bandwidth, not by the tensor cores (a 128-row MMA tile would be almost
// all padding).  The key range of every (b, h) is split across CTAs
// (split-KV); each CTA keeps the running state of section 5 (maximum m, sum
// of shifted exponentials l, weighted value sum u) for every query row over
// its keys, and a second kernel combines the splits with the same rescaling
// rule: m = max_s m_s, l = sum_s l_s 2^(m_s - m), u = sum_s u_s 2^(m_s - m),
// O = u / l, L = (m + log2 l) ln 2 (section 7).  With one split the first
// kernel writes O and L itself.
//
// A CTA serves up to 8 query rows of one (b, h) over one key split; more rows
// are spread over further CTAs (row groups).  Layout inside a CTA (256
// threads): warp w takes keys k0 + 4w .. k0 + 4w + 3, then 32 keys further,
// and so on; lane l holds elements [l E, l E + E) (E = D / 32) of
// the key and value rows, so each row is one coalesced 2E-byte-per-lane load,
// and every query row's dot product is a 5-step butterfly over the warp.  The
// eight warps' states are merged through shared memory at the end.
#include <math.h>

#include "fa_internal.cuh"

namespace fa {
namespace {

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kKeysPerIter = 4;
constexpr int kDecodeMaxG = 8;  // query rows per CTA (static shared memory: 8 warps x 8 rows x 128 floats)

template <typename T, int E>
struct RowLoad;  // E (even) consecutive elements of a row, as float, in the widest aligned loads
template <int E>
struct RowLoad<float, E> {
  static __device__ __forceinline__ void load(const float* p, float (&x)[E]) {
    if constexpr (E % 4 == 0) {  // 16-byte loads (a lane's E elements start E * 4 bytes into a 16-byte aligned row)
#pragma unroll
      for (int e = 0; e < E; e += 4) {
        const float4 t = *reinterpret_cast<const float4*>(p + e);
        x[e] = t.x;
        x[e + 1] = t.y;
        x[e + 2] = t.z;
        x[e + 3] = t.w;
      }
    } else {
#pragma unroll
      for (int e = 0; e < E; e += 2) {
        const float2 t = *reinterpret_cast<const float2*>(p + e);
        x[e] = t.x;
        x[e + 1] = t.y;
      }
    }
  }
};
// 16-bit types: four elements per 8-byte load where E allows it
template <typename T2, typename T, int E>
__device__ __forceinline__ void load16(const T* p, float (&x)[E]) {
  if constexpr (E % 4 == 0) {
#pragma unroll
    for (int e = 0; e < E; e += 4) {
      const uint2 u = *reinterpret_cast<const uint2*>(p + e);
      const T2 a = *reinterpret_cast<const T2*>(&u.x), b = *reinterpret_cast<const T2*>(&u.y);
      x[e] = __low2float(a);
      x[e + 1] = __high2float(a);
      x[e + 2] = __low2float(b);
      x[e + 3] = __high2float(b);
    }
  } else {
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      const T2 t = *reinterpret_cast<const T2*>(p + e);
      x[e] = __low2float(t);
      x[e + 1] = __high2float(t);
    }
  }
}
template <int E>
struct RowLoad<__nv_bfloat16, E> {
  static __device__ __forceinline__ void load(const __nv_bfloat16* p, float (&x)[E]) {
    load16<__nv_bfloat162>(p, x);
  }
};
template <int E>
struct RowLoad<__half, E> {
  static __device__ __forceinline__ void load(const __half* p, float (&x)[E]) { load16<__half2>(p, x); }
};

struct DecodeArgs {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  float* part_u;  // [splits, B*H, nq, D] unnormalised value sums (splits > 1)
  float* part_ml; // [splits, B*H, nq, 2] (m in log2 units, l)
  int B, H, nq, nk, splits, keys_per_split, row_groups;
  float c2;       // scale * log2(e)
  int causal;
};

// Rows g0 .. g0 + G - 1 of the queries (those >= nq are skipped).
// Blocks per SM the register budget must allow: the one-row kernel is a pure
// stream and wants as many loads in flight as it can get; eight rows of state
// need the registers of one 256-thread block per SM.
template <int G, int D>
constexpr int dec_min_blocks() { return G == 1 ? (D == 64 ? 6 : 4) : G == 4 ? 2 : 1; }

template <typename T, int D, int G>
__global__ void __launch_bounds__(kDecThreads, dec_min_blocks<G, D>()) decode_split_kernel(const DecodeArgs a) {
  constexpr int E = D / 32;
  __shared__ float s_m[kDecWarps][G], s_l[kDecWarps][G];
  __shared__ float s_u[kDecWarps][G][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x % a.splits, g0 = (blockIdx.x / a.splits) * G;
  const int h = blockIdx.y, b = blockIdx.z;
  const int nrow = min(G, a.nq - g0);  // rows of this CTA
  const long long bh = (long long)b * a.H + h;
  const T* q = static_cast<const T*>(a.q) + (bh * a.nq + g0) * D;
  const T* kp = static_cast<const T*>(a.k) + bh * (long long)a.nk * D;
  const T* vp = static_cast<const T*>(a.v) + bh * (long long)a.nk * D;
  const int k0 = split * a.keys_per_split;
  const int k1 = min(a.nk, k0 + a.keys_per_split);
  const int shift = a.nk - a.nq + g0;  // local row g sees keys j <= g + shift when causal

  float qv[G][E];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    if (g < nrow) {
      RowLoad<T, E>::load(q + (long long)g * D + lane * E, qv[g]);
#pragma unroll
      for (int e = 0; e < E; ++e) qv[g][e] *= a.c2;  // scores come out in log2 units
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) qv[g][e] = 0.f;
    }
  }
  float m[G], l[G], u[G][E];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) u[g][e] = 0.f;
  }

  for (int j0 = k0 + warp * kKeysPerIter; j0 < k1; j0 += kDecWarps * kKeysPerIter) {
    float kr[kKeysPerIter][E], vr[kKeysPerIter][E];
#pragma unroll
    for (int t = 0; t < kKeysPerIter; ++t) {
      const int j = min(j0 + t, k1 - 1);  // clamped; masked below
      RowLoad<T, E>::load(kp + (long long)j * D + lane * E, kr[t]);
      RowLoad<T, E>::load(vp + (long long)j * D + lane * E, vr[t]);
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      if (g >= nrow) continue;
      float s[kKeysPerIter];
#pragma unroll
      for (int t = 0; t < kKeysPerIter; ++t) {
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) acc = fmaf(qv[g][e], kr[t][e], acc);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        const int j = j0 + t;
        s[t] = (j < k1 && (!a.causal || j <= g + shift)) ? acc : -INFINITY;
      }
      const float mt = fmaxf(fmaxf(s[0], s[1]), fmaxf(s[2], s[3]));
      const float m_new = fmaxf(m[g], mt);
      if (m_new == -INFINITY) continue;  // nothing visible to this row yet
      const float alpha = exp2f(m[g] - m_new);  // 0 when m[g] was -inf
      l[g] *= alpha;
#pragma unroll
      for (int e = 0; e < E; ++e) u[g][e] *= alpha;
#pragma unroll
      for (int t = 0; t < kKeysPerIter; ++t) {
        const float p = exp2f(s[t] - m_new);
        l[g] += p;
#pragma unroll
        for (int e = 0; e < E; ++e) u[g][e] = fmaf(p, vr[t][e], u[g][e]);
      }
      m[g] = m_new;
    }
  }

  // merge the warps' states for every row
#pragma unroll
  for (int g = 0; g < G; ++g) {
    if (lane == 0) {
      s_m[warp][g] = m[g];
      s_l[warp][g] = l[g];
    }
#pragma unroll
    for (int e = 0; e < E; ++e) s_u[warp][g][lane * E + e] = u[g][e];
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < nrow * D; idx += kDecThreads) {
    const int g = idx / D, d = idx % D;
    float mm = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) mm = fmaxf(mm, s_m[w][g]);
    float ll = 0.f, uu = 0.f;
    if (mm != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) {
        const float f = exp2f(s_m[w][g] - mm);
        ll += s_l[w][g] * f;
        uu += s_u[w][g][d] * f;
      }
    }
    const long long row = bh * a.nq + g0 + g;
    if (a.splits == 1) {
      st_elem(static_cast<T*>(a.o), row * D + d, ll > 0.f ? uu / ll : 0.f);
      if (d == 0) a.lse[row] = ll > 0.f ? (mm + log2f(ll)) * kLn2 : -INFINITY;
    } else {
      const long long prow = (long long)split * a.B * a.H * a.nq + row;
      a.part_u[prow * D + d] = uu;
      if (d == 0) {
        a.part_ml[prow * 2] = mm;
        a.part_ml[prow * 2 + 1] = ll;
      }
    }
  }
}

// Combine the splits of every (b, h, row): one CTA per row, one thread per
// element of the head width.
template <typename T>
__global__ void decode_merge_kernel(const DecodeArgs a, int D) {
  const long long row = blockIdx.x;  // over B * H * nq
  const long long rows = (long long)a.B * a.H * a.nq;
  float mm = -INFINITY;
  for (int s = 0; s < a.splits; ++s) mm = fmaxf(mm, a.part_ml[(s * rows + row) * 2]);
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float ll = 0.f, uu = 0.f;
    if (mm != -INFINITY) {
      for (int s = 0; s < a.splits; ++s) {
        const long long prow = s * rows + row;
        const float f = exp2f(a.part_ml[prow * 2] - mm);
        ll += a.part_ml[prow * 2 + 1] * f;
        uu += a.part_u[prow * D + d] * f;
      }
    }
    st_elem(static_cast<T*>(a.o), row * D + d, ll > 0.f ? uu / ll : 0.f);
    if (d == 0) a.lse[row] = ll > 0.f ? (mm + log2f(ll)) * kLn2 : -INFINITY;
  }
}

template <typename T, int D>
cudaError_t launch_decode_td(const DecodeArgs& a, cudaStream_t s) {
  dim3 grid((unsigned)(a.splits * a.row_groups), a.H, a.B);
  if (a.nq <= 1)
    decode_split_kernel<T, D, 1><<<grid, kDecThreads, 0, s>>>(a);
  else if (a.nq <= 4)
    decode_split_kernel<T, D, 4><<<grid, kDecThreads, 0, s>>>(a);
  else
    decode_split_kernel<T, D, kDecodeMaxG><<<grid, kDecThreads, 0, s>>>(a);
  note_launches(1);
  cudaError_t e = note_error("decode launch", cudaGetLastError());
  if (e != cudaSuccess || a.splits == 1) return e;
  decode_merge_kernel<T><<<(unsigned)((long long)a.B * a.H * a.nq), D, 0, s>>>(a, D);
  note_launches(1);
  return note_error("decode merge launch", cudaGetLastError());
}

template <typename T>
cudaError_t launch_decode_t(const DecodeArgs& a, int D, cudaStream_t s) {
  if (D == 64) return launch_decode_td<T, 64>(a, s);
  if (D == 128) return launch_decode_td<T, 128>(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace

DecodeSplit decode_split(int B, int H, int nq, int nk) {
  // About 1024 CTAs over the whole problem (several per SM on a 152-SM part),
  // but no split shorter than 256 keys.
  DecodeSplit sp{1, nk};
  const long long bh = (long long)B * H;
  if (bh <= 0 || nk <= 0) return sp;
  long long want = (1024 + bh - 1) / bh;
  const long long most = (nk + 255) / 256;
  if (want > most) want = most;
  if (want < 1) want = 1;
  sp.keys_per_split = (int)((nk + want - 1) / want);
  sp.splits = (nk + sp.keys_per_split - 1) / sp.keys_per_split;
  (void)nq;
  return sp;
}

size_t decode_workspace_bytes(int B, int H, int nq, int nk, int D) {
  const DecodeSplit sp = decode_split(B, H, nq, nk);
  if (sp.splits <= 1) return 0;
  const size_t rows = (size_t)sp.splits * B * H * nq;
  return (rows * D * sizeof(float) + 255) / 256 * 256 + (rows * 2 * sizeof(float) + 255) / 256 * 256;
}

cudaError_t launch_decode(const Problem& p, int nq, int nk, fa_dtype dt, void* workspace, cudaStream_t s) {
  DecodeArgs a;
  a.q = p.q;
  a.k = p.k;
  a.v = p.v;
  a.o = p.o;
  a.lse = p.lse;
  a.B = p.B;
  a.H = p.H;
  a.nq = nq;
  a.nk = nk;
  const DecodeSplit sp = decode_split(p.B, p.H, nq, nk);
  a.splits = sp.splits;
  a.keys_per_split = sp.keys_per_split;
  a.row_groups = nq <= 4 ? 1 : (nq + kDecodeMaxG - 1) / kDecodeMaxG;
  a.c2 = p.scale * kLog2e;
  a.causal = p.causal;
  const size_t rows = (size_t)sp.splits * p.B * p.H * nq;
  a.part_u = static_cast<float*>(workspace);
  a.part_ml = sp.splits > 1 ? reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                                      (rows * p.D * sizeof(float) + 255) / 256 * 256)
                            : nullptr;
  if (dt == FA_F32) return launch_decode_t<float>(a, p.D, s);
  if (dt == FA_F16) return launch_decode_t<__half>(a, p.D, s);
  return launch_decode_t<__nv_bfloat16>(a, p.D, s);
}

}  // namespace fa
