// fa_bwd_static_ws: the backward pass with its scratch in a fixed array that
// lives in the library's own device memory, for callers that cannot allocate
// device memory themselves.
//
// The backward needs scratch (a float32 D_i per row and, on the tensor-core
// path, a float32 dQ accumulator the shape of Q).  fa_bwd takes that scratch
// from the caller.  Some callers have no way to obtain it: a plugin whose host
// application owns every device byte through its own pool and forbids direct
// cudaMalloc, or a latency-critical loop that must not pay for a cudaMalloc
// (which can synchronise the device).  This entry point serves them with a
// statically sized array that every GPU loading the library holds until the
// process exits.  It allocates nothing and only forwards to fa_bwd.
#include "fa_internal.cuh"

namespace fa {
namespace {

constexpr size_t kStaticScratchBytes = FA_BWD_STATIC_WS_BYTES;

// The scratch itself.  In host code this name is only a stand-in for the
// device array; its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_static_bwd_scratch[kStaticScratchBytes];

// Its device address on the current device and context, looked up with
// cudaGetSymbolAddress on the first call there (and again after a device
// reset) and cached.
SymbolAddress g_scratch_addr(g_static_bwd_scratch);

}  // namespace
}  // namespace fa

extern "C" fa_status fa_bwd_static_ws(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                      const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int D,
                                      float scale, int causal, const int32_t* cu_seqlens, int total_tokens,
                                      fa_dtype dtype, void* stream) {
  const size_t need = fa_bwd_workspace_size(B, H, N, D, cu_seqlens, total_tokens, dtype);
  if (need > fa::kStaticScratchBytes) {
    fa::note_detail("fa_bwd_static_ws: this problem needs more scratch than the static buffer "
                    "(FA_BWD_STATIC_WS_BYTES) holds; use fa_bwd with a caller-provided workspace");
    return FA_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  if (fa::note_error("fa_bwd_static_ws: scratch address lookup", fa::g_scratch_addr.get(&scratch)) != cudaSuccess)
    return FA_ERR_CUDA;
  // fa_bwd rewrites D_i and zeroes its dQ accumulator before reading either,
  // so whatever the previous call left in the array does not matter.
  return fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, D, scale, causal, cu_seqlens, total_tokens, dtype,
                scratch, fa::kStaticScratchBytes, stream);
}
