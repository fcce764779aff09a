// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fa.h"

namespace fa {

// Bits latched in the per-device status word by kernels.
enum : unsigned {
  kDevTimeout = 1u,     // a bounded wait ran out
  kDevBadSeqlens = 2u,  // cu_seqlens violated its contract
  kDevInternal = 4u,    // a kernel found its launch environment unusable (e.g. misaligned shared memory)
};

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// One attention problem as the kernels see it.  Dense tensors are
// [B, H, N, D]; packed ones are [H, T, D] split by cu_seqlens.  Either way a
// (sequence b, head h) pair owns `len` consecutive rows starting at row
// `base` of a row-major [rows, D] matrix, and lse/D vectors are indexed by
// the same row number.
struct Problem {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  const void* dout;
  void* dq;
  void* dk;
  void* dv;
  float* dvec;      // D_i workspace (backward)
  float* dq_acc;    // float32 dQ accumulator (backward, tensor-core path)
  unsigned* queue;  // tile counter of the backward's queue (workspace; zeroed by the preprocess kernel)
  int B, H, N, D;
  int T;            // packed token count (0 when dense)
  int f16;          // 16-bit tensors: 1 = fp16, 0 = bf16
  int dropout;      // attention dropout on (the tensor-core kernels only)
  uint32_t drop_thr;    // keep iff generator word >= drop_thr
  float drop_scale;     // 1 / (1 - p)
  uint64_t drop_seed;
  uint32_t drop_offset;
  float scale;
  int causal;
  const int32_t* cu;  // device pointer or nullptr
  unsigned* status;   // device status word
  unsigned long long wait_limit_ns;
  long long rows() const { return cu ? (long long)H * T : (long long)B * H * N; }
};

// Row range owned by (b, h); false (and a latched error) on bad cu_seqlens.
__device__ __forceinline__ bool seq_range(const Problem& p, int b, int h, long long& base, int& len) {
  if (p.cu == nullptr) {
    base = ((long long)b * p.H + h) * p.N;
    len = p.N;
    return true;
  }
  const int s0 = p.cu[b], s1 = p.cu[b + 1];
  if (s0 < 0 || s1 < s0 || s1 > p.T || s1 - s0 > p.N) {
    atomicOr(p.status, kDevBadSeqlens);
    return false;
  }
  base = (long long)h * p.T + s0;
  len = s1 - s0;
  return true;
}

// Block order for causal grids shaped (items, H, B), where items differ in cost. The
// flat block index is re-mapped so that the (b, h) pairs are cut into groups of about
// `target_heads` (the group count is rounded up and the pairs spread evenly, so no group
// is left nearly empty) and, inside a group, every head's rank-0 (heaviest) item is
// handed out before any rank-1 item, and so on. The light items of one group then fill
// in while the next group's heavy ones run, the grid ends on light items, and the
// operands in use at any time belong to only a couple of groups of heads, which keeps
// them in L2.
struct GridItem {
  int rank;  // 0 = heaviest
  int b, h;
};
__device__ __forceinline__ GridItem grouped_heavy_first(int target_heads) {
  const long long n_items = gridDim.x, n_bh = (long long)gridDim.y * gridDim.z;
  const long long n_groups = (n_bh + target_heads - 1) / target_heads;
  const long long per = (n_bh + n_groups - 1) / n_groups;  // heads in every group but the last
  const long long flat = blockIdx.x + n_items * (blockIdx.y + (long long)gridDim.y * blockIdx.z);
  const long long group = flat / (per * n_items);
  const long long r = flat - group * per * n_items;
  const long long heads = min(per, n_bh - group * per);
  const long long bh = group * per + r % heads;
  GridItem g;
  g.rank = (int)(r / heads);
  g.b = (int)(bh / gridDim.y);
  g.h = (int)(bh % gridDim.y);
  return g;
}

__device__ __forceinline__ float ld_elem(const float* p, long long i) { return p[i]; }
__device__ __forceinline__ float ld_elem(const __nv_bfloat16* p, long long i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ float ld_elem(const __half* p, long long i) { return __half2float(p[i]); }
__device__ __forceinline__ void st_elem(float* p, long long i, float x) { p[i] = x; }
__device__ __forceinline__ void st_elem(__nv_bfloat16* p, long long i, float x) { p[i] = __float2bfloat16_rn(x); }
__device__ __forceinline__ void st_elem(__half* p, long long i, float x) { p[i] = __float2half_rn(x); }

// Multiprocessor count of the current device (0 if it cannot be read); cached.
int sm_count();

// Device address of a __device__ variable in the calling thread's current
// context.  The lookup (cudaGetSymbolAddress) runs once per device and
// context and is cached: a device reset destroys the context together with the
// module holding the variable, and the next context may place it elsewhere, so
// a cached address is reused only while the context it was taken in is
// current.  Thread-safe.
class SymbolAddress {
 public:
  explicit SymbolAddress(const void* host_symbol) : symbol_(host_symbol) {}
  cudaError_t get(void** out);

 private:
  static constexpr int kMaxDevices = 64;
  const void* symbol_;  // the host-side stand-in the runtime maps to the device variable
  void* addr_[kMaxDevices] = {};
  unsigned long long ctx_[kMaxDevices] = {};
};

// Work lists of the persistent forward / backward launches for `ctas` CTAs
// (host only; see fa_schedule_preview).  cu_host: packed sequence offsets on
// the host, or nullptr for dense input.  *form: 0 = table, 1 = closed form
// (forward), 2 = queue (backward).
int preview_fwd_schedule(const Problem& p, const int32_t* cu_host, int ctas, int* off, uint32_t* items, int cap,
                         int* form);
int preview_bwd_schedule(const Problem& p, const int32_t* cu_host, int ctas, int* off, uint32_t* items, int cap,
                         int* form);

// Counts kernel launches (read by fa_launch_count); every launcher bumps it.
void note_launches(unsigned n);

// Records why a host-side CUDA step failed (read by fa_last_error_detail) and
// passes the error through.
cudaError_t note_error(const char* step, cudaError_t e);
// Records a plain message as the detail of the failure being returned.
void note_detail(const char* msg);

// ---- launchers (defined in the kernel translation units) -------------------
cudaError_t launch_simt_fwd(const Problem& p, fa_dtype dt, cudaStream_t s);
cudaError_t launch_simt_bwd(const Problem& p, fa_dtype dt, cudaStream_t s);
cudaError_t launch_bwd_preprocess(const Problem& p, fa_dtype dt, bool zero_dq_acc, cudaStream_t s);
cudaError_t launch_wait_selftest(unsigned* status, unsigned long long limit_ns, cudaStream_t s);
// One-tile check of the tensor-core building blocks (fa_selftest.cu); D in {64, 128}.
cudaError_t launch_tile_selftest(const void* a, const void* b, int D, bool f16, float* s_out, float* o_out,
                                 void* a_copy, unsigned* status, unsigned long long limit_ns, cudaStream_t s);

// tensor-core path (bf16, D in {64, 128})
cudaError_t launch_tc_fwd(const Problem& p, cudaStream_t s);
cudaError_t launch_tc_bwd(const Problem& p, cudaStream_t s);  // main kernel only
cudaError_t launch_tc_bwd128(const Problem& p, cudaStream_t s);  // main kernel only, D = 128
cudaError_t launch_tc_bwd128_dkdv(const Problem& p, cudaStream_t s);  // D = 128, dK / dV only
cudaError_t launch_dq_convert(const Problem& p, cudaStream_t s);  // dQ = bf16(scale * dQ_acc)
// Deterministic backward: dK / dV (key-stationary, no dQ product) and dQ
// (query-stationary, accumulated in tensor memory, no atomics).
cudaError_t launch_tc_bwd_dkdv(const Problem& p, cudaStream_t s);
cudaError_t launch_tc_bwd_dq(const Problem& p, cudaStream_t s);

// Cached decoding (fa_decode.cu).  Problem fields q, k, v, o, lse, B, H, D,
// scale, causal are used; nq / nk are the query and cached-key counts.
struct DecodeSplit {
  int splits;          // key splits per (b, h)
  int keys_per_split;
};
DecodeSplit decode_split(int B, int H, int nq, int nk);
size_t decode_workspace_bytes(int B, int H, int nq, int nk, int D);
cudaError_t launch_decode(const Problem& p, int nq, int nk, fa_dtype dt, void* workspace, cudaStream_t s);

}  // namespace fa
