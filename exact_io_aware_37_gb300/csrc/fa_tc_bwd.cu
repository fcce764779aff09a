// Backward pass, last step: the float32 dQ accumulator the main backward kernel
// (fa_tc_bwd128.cu, D = 64 and 128) reduces into is scaled and rounded to the
// 16-bit input type (tensortonic.com "FlashAttention" section 7:
// dQ = scale * dS K).  Also the entry points that select the main kernel.
#include "fa_internal.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

using namespace ptx;

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

cudaError_t launch_tc_bwd(const Problem& p, cudaStream_t s) { return launch_tc_bwd128(p, s); }

cudaError_t launch_tc_bwd_dkdv(const Problem& p, cudaStream_t s) { return launch_tc_bwd128_dkdv(p, s); }

}  // namespace fa
