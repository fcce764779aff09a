// fp32-FMA (CUDA core) attention kernels.
//
// Used for float32 inputs, where the required accuracy (max |dO| <= 1e-4)
// rules out TF32 tensor cores.  Same method as the tensor-core path, at small
// tiles: a block of 32 query rows keeps one running softmax state per row
// (tensortonic.com "FlashAttention", section 5) while 32-key tiles of K and V
// pass through shared memory (section 3); causal blocks wholly in the future
// are never visited (section 6).  Four threads share a query row, each owning
// every fourth column, and combine their partial dot products with two warp
// shuffles.  The backward pass rebuilds P_ij = exp(s_ij - L_i) (section 7)
// in two kernels -- one per query row for dQ and one per key row for dK and
// dV -- so no atomics are needed.
#include <math.h>

#include "fa_internal.cuh"

namespace fa {
namespace {

constexpr int kBR = 32;        // query rows per CTA
constexpr int kBC = 32;        // keys per shared-memory tile
constexpr int kThreads = 128;  // 32 rows x 4 threads

__device__ __forceinline__ float quad_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  x += __shfl_xor_sync(0xffffffffu, x, 2);
  return x;
}

template <typename T, int D>
__device__ __forceinline__ void load_tile(float (*dst)[D], const T* src, long long base, int r0, int len, int tid) {
  for (int e = tid; e < kBC * D; e += kThreads) {
    const int rr = e / D, col = e % D;
    const int r = r0 + rr;
    dst[rr][col] = r < len ? ld_elem(src, (base + r) * D + col) : 0.f;
  }
}

// ---------------------------------------------------------------- forward
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) simt_fwd_kernel(Problem p) {
  constexpr int DC = D / 4;
  __shared__ float Ks[kBC][D];
  __shared__ float Vs[kBC][D];
  const int tid = threadIdx.x, r = tid >> 2, part = tid & 3;
  long long base;
  int len;
  if (!seq_range(p, blockIdx.y, blockIdx.z, base, len)) return;
  const int q0 = blockIdx.x * kBR;
  if (q0 >= len) return;
  const int i = q0 + r;
  const bool row_ok = i < len;
  const float c2 = p.scale * kLog2e;  // scores in the exp2 domain

  const T* Q = static_cast<const T*>(p.q);
  float qv[DC], acc[DC];
#pragma unroll
  for (int c = 0; c < DC; ++c) {
    qv[c] = row_ok ? ld_elem(Q, (base + i) * D + c * 4 + part) * c2 : 0.f;
    acc[c] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  const int kend = p.causal ? min(len, q0 + kBR) : len;
  for (int j0 = 0; j0 < kend; j0 += kBC) {
    __syncthreads();
    load_tile<T, D>(Ks, static_cast<const T*>(p.k), base, j0, len, tid);
    load_tile<T, D>(Vs, static_cast<const T*>(p.v), base, j0, len, tid);
    __syncthreads();
    float s[kBC];
    float mt = -INFINITY;
#pragma unroll
    for (int jj = 0; jj < kBC; ++jj) {
      float part_sum = 0.f;
#pragma unroll
      for (int c = 0; c < DC; ++c) part_sum = fmaf(qv[c], Ks[jj][c * 4 + part], part_sum);
      part_sum = quad_sum(part_sum);
      const int j = j0 + jj;
      const bool ok = j < len && (!p.causal || j <= i);
      s[jj] = ok ? part_sum : -INFINITY;
      mt = fmaxf(mt, s[jj]);
    }
    const float mn = fmaxf(m, mt);
    if (mn == -INFINITY) continue;  // nothing allowed yet in this row
    const float alpha = (m == -INFINITY) ? 0.f : exp2f(m - mn);
    l *= alpha;
#pragma unroll
    for (int c = 0; c < DC; ++c) acc[c] *= alpha;
#pragma unroll
    for (int jj = 0; jj < kBC; ++jj) {
      const float pj = (s[jj] == -INFINITY) ? 0.f : exp2f(s[jj] - mn);
      l += pj;
#pragma unroll
      for (int c = 0; c < DC; ++c) acc[c] = fmaf(pj, Vs[jj][c * 4 + part], acc[c]);
    }
    m = mn;
  }
  if (row_ok) {
    T* O = static_cast<T*>(p.o);
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int c = 0; c < DC; ++c) st_elem(O, (base + i) * D + c * 4 + part, acc[c] * inv);
    if (part == 0) p.lse[base + i] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
  }
}

// ---------------------------------------------------------------- backward: dQ
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) simt_bwd_dq_kernel(Problem p) {
  constexpr int DC = D / 4;
  __shared__ float Ks[kBC][D];
  __shared__ float Vs[kBC][D];
  const int tid = threadIdx.x, r = tid >> 2, part = tid & 3;
  long long base;
  int len;
  if (!seq_range(p, blockIdx.y, blockIdx.z, base, len)) return;
  const int q0 = blockIdx.x * kBR;
  if (q0 >= len) return;
  const int i = q0 + r;
  const bool row_ok = i < len;
  const float c2 = p.scale * kLog2e;
  const T* Q = static_cast<const T*>(p.q);
  const T* dO = static_cast<const T*>(p.dout);
  float qv[DC], dov[DC], dqa[DC];
#pragma unroll
  for (int c = 0; c < DC; ++c) {
    const long long e = (base + i) * D + c * 4 + part;
    qv[c] = row_ok ? ld_elem(Q, e) * c2 : 0.f;
    dov[c] = row_ok ? ld_elem(dO, e) : 0.f;
    dqa[c] = 0.f;
  }
  const float Lr = row_ok ? p.lse[base + i] * kLog2e : 0.f;
  const float Dr = row_ok ? p.dvec[base + i] : 0.f;
  const int kend = p.causal ? min(len, q0 + kBR) : len;
  for (int j0 = 0; j0 < kend; j0 += kBC) {
    __syncthreads();
    load_tile<T, D>(Ks, static_cast<const T*>(p.k), base, j0, len, tid);
    load_tile<T, D>(Vs, static_cast<const T*>(p.v), base, j0, len, tid);
    __syncthreads();
#pragma unroll 4
    for (int jj = 0; jj < kBC; ++jj) {
      float sk = 0.f, sv = 0.f;
#pragma unroll
      for (int c = 0; c < DC; ++c) {
        sk = fmaf(qv[c], Ks[jj][c * 4 + part], sk);
        sv = fmaf(dov[c], Vs[jj][c * 4 + part], sv);
      }
      sk = quad_sum(sk);
      sv = quad_sum(sv);
      const int j = j0 + jj;
      const bool ok = row_ok && j < len && (!p.causal || j <= i);
      const float pj = ok ? exp2f(sk - Lr) : 0.f;
      const float ds = pj * (sv - Dr);
#pragma unroll
      for (int c = 0; c < DC; ++c) dqa[c] = fmaf(ds, Ks[jj][c * 4 + part], dqa[c]);
    }
  }
  if (row_ok) {
    T* dQ = static_cast<T*>(p.dq);
#pragma unroll
    for (int c = 0; c < DC; ++c) st_elem(dQ, (base + i) * D + c * 4 + part, dqa[c] * p.scale);
  }
}

// ---------------------------------------------------------------- backward: dK, dV
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) simt_bwd_dkdv_kernel(Problem p) {
  constexpr int DC = D / 4;
  __shared__ float Qs[kBC][D];
  __shared__ float dOs[kBC][D];
  __shared__ float Ls[kBC];
  __shared__ float Dsh[kBC];
  const int tid = threadIdx.x, r = tid >> 2, part = tid & 3;
  long long base;
  int len;
  if (!seq_range(p, blockIdx.y, blockIdx.z, base, len)) return;
  const int k0 = blockIdx.x * kBR;
  if (k0 >= len) return;
  const int j = k0 + r;
  const bool row_ok = j < len;
  const float c2 = p.scale * kLog2e;
  const T* K = static_cast<const T*>(p.k);
  const T* V = static_cast<const T*>(p.v);
  float kv[DC], vv[DC], dka[DC], dva[DC];
#pragma unroll
  for (int c = 0; c < DC; ++c) {
    const long long e = (base + j) * D + c * 4 + part;
    kv[c] = row_ok ? ld_elem(K, e) * c2 : 0.f;
    vv[c] = row_ok ? ld_elem(V, e) : 0.f;
    dka[c] = 0.f;
    dva[c] = 0.f;
  }
  const int qstart = p.causal ? k0 : 0;  // earlier queries never see these keys
  for (int i0 = qstart; i0 < len; i0 += kBC) {
    __syncthreads();
    load_tile<T, D>(Qs, static_cast<const T*>(p.q), base, i0, len, tid);
    load_tile<T, D>(dOs, static_cast<const T*>(p.dout), base, i0, len, tid);
    if (tid < kBC) {
      const int i = i0 + tid;
      Ls[tid] = i < len ? p.lse[base + i] * kLog2e : 0.f;
      Dsh[tid] = i < len ? p.dvec[base + i] : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int ii = 0; ii < kBC; ++ii) {
      float s = 0.f, dp = 0.f;
#pragma unroll
      for (int c = 0; c < DC; ++c) {
        s = fmaf(kv[c], Qs[ii][c * 4 + part], s);
        dp = fmaf(vv[c], dOs[ii][c * 4 + part], dp);
      }
      s = quad_sum(s);
      dp = quad_sum(dp);
      const int i = i0 + ii;
      const bool ok = row_ok && i < len && (!p.causal || j <= i);
      const float pij = ok ? exp2f(s - Ls[ii]) : 0.f;
      const float ds = pij * (dp - Dsh[ii]);
#pragma unroll
      for (int c = 0; c < DC; ++c) {
        dva[c] = fmaf(pij, dOs[ii][c * 4 + part], dva[c]);
        dka[c] = fmaf(ds, Qs[ii][c * 4 + part], dka[c]);
      }
    }
  }
  if (row_ok) {
    T* dK = static_cast<T*>(p.dk);
    T* dV = static_cast<T*>(p.dv);
#pragma unroll
    for (int c = 0; c < DC; ++c) {
      const long long e = (base + j) * D + c * 4 + part;
      st_elem(dK, e, dka[c] * p.scale);
      st_elem(dV, e, dva[c]);
    }
  }
}

// ---------------------------------------------------------------- preprocess
// D_i = sum_d dO_id * O_id in fp32; optionally zeroes the float32 dQ
// accumulator row.  Each lane reads 16 bytes of O and of dO at a time, so a
// row of D elements takes L = D * sizeof(T) / 16 lanes and a warp covers
// 32 / L rows; the row sum is a butterfly over those L lanes.  The kernel is
// a stream over O and dO (and the accumulator it zeroes): HBM-bound.
template <typename T, int D>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(Problem p, long long rows, int zero_acc) {
  constexpr int E = 16 / (int)sizeof(T);  // elements per 16-byte load
  constexpr int L = D / E;                // lanes per row
  static_assert(L >= 1 && L <= 32 && 32 % L == 0, "row split");
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long row = tid / L;
  const int part = (int)(tid % L);
  if (tid == 0 && p.queue != nullptr) *p.queue = 0u;  // the tensor-core backward's tile counter
  const bool in = row < rows;
  float acc = 0.f;
  if (in) {
    const uint4 a = reinterpret_cast<const uint4*>(static_cast<const T*>(p.o) + row * D)[part];
    const uint4 b = reinterpret_cast<const uint4*>(static_cast<const T*>(p.dout) + row * D)[part];
    const T* ea = reinterpret_cast<const T*>(&a);
    const T* eb = reinterpret_cast<const T*>(&b);
#pragma unroll
    for (int e = 0; e < E; ++e) acc = fmaf(ld_elem(ea, e), ld_elem(eb, e), acc);
  }
#pragma unroll
  for (int o = L / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (!in) return;
  if (part == 0) p.dvec[row] = acc;
  if (zero_acc) {
    float4* r = reinterpret_cast<float4*>(p.dq_acc + row * D);
#pragma unroll
    for (int c = part; c < D / 4; c += L) r[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

template <typename T>
cudaError_t launch_preprocess_t(const Problem& p, long long rows, bool zero, cudaStream_t s) {
  auto go = [&](auto kernel, int lanes_per_row) {
    const long long threads = rows * lanes_per_row;
    kernel<<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(p, rows, zero ? 1 : 0);
    return cudaGetLastError();
  };
  constexpr int E = 16 / (int)sizeof(T);
  switch (p.D) {
    case 32: return go(bwd_preprocess_kernel<T, 32>, 32 / E);
    case 64: return go(bwd_preprocess_kernel<T, 64>, 64 / E);
    case 128: return go(bwd_preprocess_kernel<T, 128>, 128 / E);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T, int D>
cudaError_t launch_fwd_t(const Problem& p, cudaStream_t s) {
  dim3 grid((p.N + kBR - 1) / kBR, p.B, p.H);
  simt_fwd_kernel<T, D><<<grid, kThreads, 0, s>>>(p);
  note_launches(1);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_bwd_t(const Problem& p, cudaStream_t s) {
  dim3 grid((p.N + kBR - 1) / kBR, p.B, p.H);
  simt_bwd_dq_kernel<T, D><<<grid, kThreads, 0, s>>>(p);
  note_launches(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  simt_bwd_dkdv_kernel<T, D><<<grid, kThreads, 0, s>>>(p);
  note_launches(1);
  return cudaGetLastError();
}

template <typename T>
cudaError_t dispatch_fwd(const Problem& p, cudaStream_t s) {
  switch (p.D) {
    case 32: return launch_fwd_t<T, 32>(p, s);
    case 64: return launch_fwd_t<T, 64>(p, s);
    case 128: return launch_fwd_t<T, 128>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T>
cudaError_t dispatch_bwd(const Problem& p, cudaStream_t s) {
  switch (p.D) {
    case 32: return launch_bwd_t<T, 32>(p, s);
    case 64: return launch_bwd_t<T, 64>(p, s);
    case 128: return launch_bwd_t<T, 128>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_simt_fwd(const Problem& p, fa_dtype dt, cudaStream_t s) {
  return dt == FA_F32 ? dispatch_fwd<float>(p, s)
                       : dt == FA_F16 ? dispatch_fwd<__half>(p, s) : dispatch_fwd<__nv_bfloat16>(p, s);
}

cudaError_t launch_simt_bwd(const Problem& p, fa_dtype dt, cudaStream_t s) {
  return dt == FA_F32 ? dispatch_bwd<float>(p, s)
                       : dt == FA_F16 ? dispatch_bwd<__half>(p, s) : dispatch_bwd<__nv_bfloat16>(p, s);
}

cudaError_t launch_bwd_preprocess(const Problem& p, fa_dtype dt, bool zero_dq_acc, cudaStream_t s) {
  const long long rows = p.rows();
  if (rows == 0) return cudaSuccess;
  cudaError_t e;
  if (dt == FA_F32)
    e = launch_preprocess_t<float>(p, rows, zero_dq_acc, s);
  else if (dt == FA_F16)
    e = launch_preprocess_t<__half>(p, rows, zero_dq_acc, s);
  else
    e = launch_preprocess_t<__nv_bfloat16>(p, rows, zero_dq_acc, s);
  note_launches(1);
  return e;
}

}  // namespace fa
