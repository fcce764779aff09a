// Instrumentation: throughput of the special-function units for ex2.approx.
//
// Both tensor-core kernels form every attention weight with one ex2.approx
// (exp2 of a score pre-scaled by scale * log2(e)), so besides the tensor
// core their second bound is the multi-function unit: N^2 exponentials per
// (sequence, head) in the forward pass (half when causal) and as many again
// in the backward pass.  This probe measures the unit's rate on the GPU it
// runs on, so that bound is a measured number rather than a datasheet one.
//
// One CTA per SM; every thread runs kChains independent recurrences
// x <- 2^(-x) (which stay in (0, 1]) for `iters` rounds between two reads of
// the SM clock; the rate is (threads * kChains * iters) / cycles per CTA.
#include "fa_internal.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kProbeThreads = 512;
constexpr int kChains = 8;
constexpr int kMaxProbeCtas = 1024;

// Per-CTA start and end SM clocks and a sink for the results, so the
// recurrences cannot be optimised away.
__device__ unsigned long long g_probe_clocks[2 * kMaxProbeCtas];
__device__ float g_probe_sink[kMaxProbeCtas];

__global__ void __launch_bounds__(kProbeThreads, 1) ex2_rate_kernel(int iters) {
  float x[kChains];
#pragma unroll
  for (int c = 0; c < kChains; ++c) x[c] = 0.25f + 0.0625f * c + 1e-6f * threadIdx.x;
  __syncthreads();
  const unsigned long long t0 = clock64();
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int c = 0; c < kChains; ++c) x[c] = ptx::ex2_approx(-x[c]);
  }
  __syncthreads();
  const unsigned long long t1 = clock64();
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < kChains; ++c) s += x[c];
  if (threadIdx.x == 0) {
    g_probe_clocks[2 * blockIdx.x] = t0;
    g_probe_clocks[2 * blockIdx.x + 1] = t1;
  }
  if (s == 12345.f) g_probe_sink[blockIdx.x] = s;  // never true; keeps the chains live
}

SymbolAddress g_probe_clock_addr(g_probe_clocks);

}  // namespace
}  // namespace fa

extern "C" fa_status fa_probe_ex2_rate(int iters, double* ex2_per_clk_per_sm, void* stream) {
  using namespace fa;
  if (ex2_per_clk_per_sm == nullptr || iters < 1 || iters > (1 << 20)) return FA_ERR_INVALID;
  const int ctas = sm_count();
  if (ctas <= 0 || ctas > kMaxProbeCtas) return FA_ERR_CUDA;
  void* clocks = nullptr;
  if (note_error("probe clock address", g_probe_clock_addr.get(&clocks)) != cudaSuccess) return FA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ex2_rate_kernel<<<ctas, kProbeThreads, 0, s>>>(iters);
  note_launches(1);
  if (note_error("probe launch", cudaGetLastError()) != cudaSuccess) return FA_ERR_CUDA;
  if (note_error("probe sync", cudaStreamSynchronize(s)) != cudaSuccess) return FA_ERR_CUDA;
  unsigned long long host[2 * kMaxProbeCtas];
  if (note_error("probe read-back",
                 cudaMemcpy(host, clocks, sizeof(unsigned long long) * 2 * ctas, cudaMemcpyDeviceToHost)) !=
      cudaSuccess)
    return FA_ERR_CUDA;
  double sum = 0.0;
  for (int c = 0; c < ctas; ++c) {
    const double cycles = (double)(host[2 * c + 1] - host[2 * c]);
    if (cycles <= 0.0) return FA_ERR_CUDA;
    sum += (double)kProbeThreads * kChains * iters / cycles;
  }
  *ex2_per_clk_per_sm = sum / ctas;
  return FA_OK;
}
