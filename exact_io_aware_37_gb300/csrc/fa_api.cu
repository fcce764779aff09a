// Host side of the C ABI declared in include/fa.h: argument validation, the
// per-device status word, workspace carving and kernel dispatch.
#include <math.h>

#include <stdio.h>

#include <atomic>
#include <mutex>

#include <cuda.h>

#include "fa_internal.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

// Kernels latch failures here; read and cleared by fa_get_last_device_error.
__device__ unsigned g_status_word;

std::atomic<unsigned long long> g_wait_limit_ns{2000000000ull};
std::atomic<unsigned long long> g_launches{0};

SymbolAddress g_status_addr(&g_status_word);

// Device address of the current device's status word.
cudaError_t status_word(unsigned** out) {
  void* p = nullptr;
  const cudaError_t e = g_status_addr.get(&p);
  *out = static_cast<unsigned*>(p);
  return e;
}

// Identity of the calling thread's current context, or 0 when there is none
// or it cannot be read (the driver calls are resolved through the runtime, so
// the library needs no link-time dependency on libcuda).
unsigned long long current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(f);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(f);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

std::mutex g_symbol_mu;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// The tensor-core kernels cover bf16 and fp16 with D in {64, 128}.
constexpr bool kHaveTcFwd = true;
constexpr bool kHaveTcBwd = true;
bool use_tensor_cores(fa_dtype dt, int D) { return (dt == FA_BF16 || dt == FA_F16) && (D == 64 || D == 128); }

// The score scale must be finite and positive.  The kernels take each row's
// running maximum over the raw scores q.k and only then multiply by the
// scale, which picks the maximum of the scaled scores only when the scale is
// positive; masked scores are -inf, and -inf times zero or a negative scale
// is not -inf.  (The pages' scale is 1/sqrt(head width).)
bool scale_ok(float scale) { return isfinite(scale) && scale > 0.f; }

fa_status validate(int B, int H, int N, int D, float scale, int causal, const int32_t* cu, int T, fa_dtype dt) {
  if (B < 0 || H < 0 || N < 0 || D <= 0) return FA_ERR_INVALID;
  if (B > 65535 || H > 65535) return FA_ERR_UNSUPPORTED;  // grid y / z limits
  if (!scale_ok(scale)) return FA_ERR_INVALID;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID;
  if (dt != FA_BF16 && dt != FA_F32 && dt != FA_F16) return FA_ERR_UNSUPPORTED;
  if (fa_path_name(dt, D) == nullptr) return FA_ERR_UNSUPPORTED;
  if (cu != nullptr && T < 0) return FA_ERR_INVALID;
  return FA_OK;
}

long long row_count(int B, int H, int N, const int32_t* cu, int T) {
  return cu ? (long long)H * T : (long long)B * H * N;
}

bool no_work(int B, int H, int N, const int32_t* cu, int T) {
  return B == 0 || H == 0 || N == 0 || (cu != nullptr && T == 0);
}

fa_status check_tensor(const void* p) {
  if (p == nullptr) return FA_ERR_INVALID;
  if (!aligned(p, 16)) return FA_ERR_ALIGN;
  return FA_OK;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// The tensor-core backward's tile counter (see fa_tc_bwd128.cu), at the end of
// the workspace; one 256-byte block keeps the workspace's parts aligned.
constexpr size_t kQueueBytes = 256;

// Attention dropout arguments (nullptr: none).
struct DropArgs {
  float p;
  uint64_t seed;
  uint32_t offset;
};

// Keep iff the generator word w satisfies w / 2^32 >= p, i.e. w >= ceil(p 2^32)
// (exact in double: p is a float and 2^32 a power of two).
fa_status set_dropout(Problem& pr, fa_dtype dt, int D, const DropArgs* d) {
  pr.dropout = 0;
  if (d == nullptr) return FA_OK;
  if (!(d->p >= 0.f && d->p < 1.f)) return FA_ERR_INVALID;
  if (d->p == 0.f) return FA_OK;
  if (!use_tensor_cores(dt, D)) return FA_ERR_UNSUPPORTED;  // the fp32 kernels have no dropout
  pr.dropout = 1;
  pr.drop_thr = (uint32_t)ceil((double)d->p * 4294967296.0);
  pr.drop_scale = 1.0f / (1.0f - d->p);
  pr.drop_seed = d->seed;
  pr.drop_offset = d->offset;
  return FA_OK;
}

}  // namespace

cudaError_t SymbolAddress::get(void** out) {
  *out = nullptr;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_symbol_mu);
  const unsigned long long ctx = current_context_id();
  if (addr_[dev] == nullptr || ctx == 0 || ctx != ctx_[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, symbol_);  // makes the device's primary context current if needed
    if (e != cudaSuccess) return e;
    addr_[dev] = p;
    ctx_[dev] = current_context_id();
  }
  *out = addr_[dev];
  return cudaSuccess;
}

void note_launches(unsigned n) { g_launches.fetch_add(n); }

thread_local char g_detail[256];
thread_local cudaEvent_t g_main_start = nullptr, g_main_stop = nullptr;

cudaError_t note_error(const char* step, cudaError_t e) {
  if (e != cudaSuccess) snprintf(g_detail, sizeof(g_detail), "%s: %s", step, cudaGetErrorString(e));
  return e;
}

void note_detail(const char* msg) { snprintf(g_detail, sizeof(g_detail), "%s", msg); }

// Failure-detection self-test kernel: waits on a barrier nobody signals.
__global__ void wait_selftest_kernel(unsigned* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  ptx::WaitCtx w{&abort_flag, status, limit_ns};
  ptx::mbar_wait(&bar, 0, w);  // returns false once the limit passes
  __syncthreads();
}

cudaError_t launch_wait_selftest(unsigned* status, unsigned long long limit_ns, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace fa

using namespace fa;

extern "C" {

const char* fa_strerror(fa_status s) {
  switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported dtype or head width";
    case FA_ERR_ALIGN: return "tensor pointer not 16-byte aligned";
    case FA_ERR_CUDA: return "CUDA call failed";
    case FA_ERR_TIMEOUT: return "a bounded wait inside a kernel expired";
    case FA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
  }
  return "unknown status";
}

const char* fa_path_name(fa_dtype dt, int D) {
  if ((dt == FA_BF16 || dt == FA_F16) && (D == 64 || D == 128))
    return kHaveTcFwd ? (kHaveTcBwd ? "tcgen05" : "tcgen05_fwd+simt_bwd") : "simt_16bit";
  if (dt == FA_F32 && (D == 32 || D == 64 || D == 128)) return "simt_f32";
  return nullptr;
}

unsigned long long fa_launch_count(void) { return g_launches.load(); }

int fa_schedule_preview(int kernel, const int32_t* cu_seqlens, int B, int H, int N, int D, int causal, int n_ctas,
                        int* off, unsigned int* items, int cap, int* form) {
  if ((kernel != 0 && kernel != 1) || B <= 0 || H <= 0 || N <= 0 || (D != 64 && D != 128) ||
      (causal != 0 && causal != 1) || n_ctas <= 0 || off == nullptr || form == nullptr || cap < 0 ||
      (items == nullptr && cap > 0))
    return -1;
  fa::Problem p{};
  p.B = B;
  p.H = H;
  p.N = N;
  p.D = D;
  p.causal = causal;
  p.cu = cu_seqlens;  // only its presence matters to the schedule; the host copy is read below
  p.T = cu_seqlens ? cu_seqlens[B] : 0;
  return kernel == 0 ? fa::preview_fwd_schedule(p, cu_seqlens, n_ctas, off, items, cap, form)
                     : fa::preview_bwd_schedule(p, cu_seqlens, n_ctas, off, items, cap, form);
}

const char* fa_last_error_detail(void) { return g_detail; }

void fa_bwd_time_main_kernel(void* start_event, void* stop_event) {
  g_main_start = static_cast<cudaEvent_t>(start_event);
  g_main_stop = static_cast<cudaEvent_t>(stop_event);
}

void fa_set_wait_limit_ns(unsigned long long limit_ns) {
  g_wait_limit_ns.store(limit_ns < 1000ull ? 1000ull : limit_ns);
}

fa_status fa_get_last_device_error(void* stream) {
  unsigned* word = nullptr;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  if (status_word(&word) != cudaSuccess) return FA_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpy(&v, word, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
  const unsigned zero = 0;
  if (v != 0 && cudaMemcpy(word, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return FA_ERR_CUDA;
  if (v & kDevTimeout) return FA_ERR_TIMEOUT;
  if (v & kDevBadSeqlens) return FA_ERR_INVALID;
  if (v & kDevInternal) return FA_ERR_CUDA;
  return FA_OK;
}

fa_status fa_selftest_wait_timeout(void* stream) {
  unsigned* word = nullptr;
  if (status_word(&word) != cudaSuccess) return FA_ERR_CUDA;
  if (launch_wait_selftest(word, g_wait_limit_ns.load(), static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FA_ERR_CUDA;
  return fa_get_last_device_error(stream);
}

fa_status fa_selftest_tile(const void* a, const void* b, float* s_out, float* o_out, void* a_copy, int D,
                           fa_dtype dtype, void* stream) {
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  if (dtype != FA_BF16 && dtype != FA_F16) return FA_ERR_UNSUPPORTED;
  fa_status st;
  for (const void* p : {a, b, (const void*)s_out, (const void*)o_out, (const void*)a_copy})
    if ((st = check_tensor(p)) != FA_OK) return st;
  unsigned* word = nullptr;
  g_detail[0] = 0;
  if (note_error("status word", status_word(&word)) != cudaSuccess) return FA_ERR_CUDA;
  if (launch_tile_selftest(a, b, D, dtype == FA_F16, s_out, o_out, a_copy, word, g_wait_limit_ns.load(),
                           static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FA_ERR_CUDA;
  return fa_get_last_device_error(stream);
}

size_t fa_bwd_workspace_size(int B, int H, int N, int D, const int32_t* cu, int T, fa_dtype dt) {
  if (B < 0 || H < 0 || N < 0 || D <= 0 || (cu && T < 0)) return 0;
  const long long rows = row_count(B, H, N, cu, T);
  size_t bytes = round_up((size_t)rows * sizeof(float), 256);
  if (use_tensor_cores(dt, D)) bytes += round_up((size_t)rows * D * sizeof(float), 256) + kQueueBytes;
  return bytes;
}

static fa_status fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                          int D, float scale, int causal, const int32_t* cu, int T, fa_dtype dt, const DropArgs* drop,
                          void* stream) {
  fa_status st = validate(B, H, N, D, scale, causal, cu, T, dt);
  if (st != FA_OK) return st;
  if (no_work(B, H, N, cu, T)) return FA_OK;
  for (const void* p : {q, k, v, (const void*)o})
    if ((st = check_tensor(p)) != FA_OK) return st;
  if (lse == nullptr) return FA_ERR_INVALID;
  if (!aligned(lse, 4)) return FA_ERR_ALIGN;
  if (cu != nullptr && !aligned(cu, 4)) return FA_ERR_ALIGN;

  Problem p{};
  p.q = q; p.k = k; p.v = v; p.o = o; p.lse = lse;
  p.B = B; p.H = H; p.N = N; p.D = D; p.T = cu ? T : 0;
  p.f16 = dt == FA_F16;
  p.scale = scale; p.causal = causal; p.cu = cu;
  if ((st = set_dropout(p, dt, D, drop)) != FA_OK) return st;
  p.wait_limit_ns = g_wait_limit_ns.load();
  g_detail[0] = 0;
  if (note_error("status word", status_word(&p.status)) != cudaSuccess) return FA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = (kHaveTcFwd && use_tensor_cores(dt, D)) ? launch_tc_fwd(p, s) : launch_simt_fwd(p, dt, s);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

static fa_status bwd_impl(const void* q, const void* k, const void* v, const void* o, const float* lse,
                          const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int D, float scale,
                          int causal, const int32_t* cu, int T, fa_dtype dt, const DropArgs* drop, void* workspace,
                          size_t workspace_bytes, void* stream, bool deterministic = false) {
  fa_status st = validate(B, H, N, D, scale, causal, cu, T, dt);
  if (st != FA_OK) return st;
  if (no_work(B, H, N, cu, T)) return FA_OK;
  for (const void* p : {q, k, v, o, dout, (const void*)dq, (const void*)dk, (const void*)dv})
    if ((st = check_tensor(p)) != FA_OK) return st;
  if (lse == nullptr) return FA_ERR_INVALID;
  if (!aligned(lse, 4)) return FA_ERR_ALIGN;
  if (cu != nullptr && !aligned(cu, 4)) return FA_ERR_ALIGN;
  // the deterministic path keeps no float32 dQ accumulator: only D_i
  const size_t need = deterministic ? round_up((size_t)row_count(B, H, N, cu, T) * sizeof(float), 256) +
                                          (use_tensor_cores(dt, D) ? kQueueBytes : 0)
                                    : fa_bwd_workspace_size(B, H, N, D, cu, T, dt);
  if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < need) return FA_ERR_WORKSPACE;

  Problem p{};
  p.q = q; p.k = k; p.v = v; p.o = const_cast<void*>(o); p.lse = const_cast<float*>(lse);
  p.dout = dout; p.dq = dq; p.dk = dk; p.dv = dv;
  p.B = B; p.H = H; p.N = N; p.D = D; p.T = cu ? T : 0;
  p.f16 = dt == FA_F16;
  p.scale = scale; p.causal = causal; p.cu = cu;
  if ((st = set_dropout(p, dt, D, drop)) != FA_OK) return st;
  p.wait_limit_ns = g_wait_limit_ns.load();
  const long long rows = p.rows();
  p.dvec = static_cast<float*>(workspace);
  p.dq_acc = use_tensor_cores(dt, D) && !deterministic
                 ? reinterpret_cast<float*>(static_cast<char*>(workspace) + round_up((size_t)rows * 4, 256))
                 : nullptr;
  // the tensor-core backward's tile counter: the last kQueueBytes of the workspace it needs
  p.queue = use_tensor_cores(dt, D) ? reinterpret_cast<unsigned*>(static_cast<char*>(workspace) + need - kQueueBytes)
                                    : nullptr;
  g_detail[0] = 0;
  cudaEvent_t ev_start = g_main_start, ev_stop = g_main_stop;
  g_main_start = g_main_stop = nullptr;
  if (note_error("status word", status_word(&p.status)) != cudaSuccess) return FA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool tc = kHaveTcBwd && use_tensor_cores(dt, D);
  cudaError_t e = launch_bwd_preprocess(p, dt, p.dq_acc != nullptr, s);
  if (e == cudaSuccess && ev_start) e = note_error("timing event", cudaEventRecord(ev_start, s));
  if (e == cudaSuccess && tc && deterministic) {
    // dK, dV key-stationary and dQ query-stationary: no atomics anywhere
    e = launch_tc_bwd_dkdv(p, s);
    if (e == cudaSuccess) e = launch_tc_bwd_dq(p, s);
    if (e == cudaSuccess && ev_stop) e = note_error("timing event", cudaEventRecord(ev_stop, s));
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
  }
  if (e == cudaSuccess) e = tc ? launch_tc_bwd(p, s) : launch_simt_bwd(p, dt, s);
  if (e == cudaSuccess && ev_stop) e = note_error("timing event", cudaEventRecord(ev_stop, s));
  if (e == cudaSuccess && tc) e = launch_dq_convert(p, s);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int D,
                 float scale, int causal, const int32_t* cu, int T, fa_dtype dt, void* stream) {
  return fwd_impl(q, k, v, o, lse, B, H, N, D, scale, causal, cu, T, dt, nullptr, stream);
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                 void* dq, void* dk, void* dv, int B, int H, int N, int D, float scale, int causal,
                 const int32_t* cu, int T, fa_dtype dt, void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, D, scale, causal, cu, T, dt, nullptr, workspace,
                  workspace_bytes, stream);
}

fa_status fa_fwd_dropout(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                         int D, float scale, int causal, const int32_t* cu, int T, fa_dtype dt, float p_drop,
                         uint64_t seed, uint32_t offset, void* stream) {
  const DropArgs d{p_drop, seed, offset};
  return fwd_impl(q, k, v, o, lse, B, H, N, D, scale, causal, cu, T, dt, &d, stream);
}

fa_status fa_bwd_dropout(const void* q, const void* k, const void* v, const void* o, const float* lse,
                         const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int D, float scale,
                         int causal, const int32_t* cu, int T, fa_dtype dt, float p_drop, uint64_t seed,
                         uint32_t offset, void* workspace, size_t workspace_bytes, void* stream) {
  const DropArgs d{p_drop, seed, offset};
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, D, scale, causal, cu, T, dt, &d, workspace,
                  workspace_bytes, stream);
}

fa_status fa_bwd_deterministic(const void* q, const void* k, const void* v, const void* o, const float* lse,
                               const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int D,
                               float scale, int causal, const int32_t* cu, int T, fa_dtype dt, float p_drop,
                               uint64_t seed, uint32_t offset, void* workspace, size_t workspace_bytes,
                               void* stream) {
  const DropArgs d{p_drop, seed, offset};
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, D, scale, causal, cu, T, dt, &d, workspace,
                  workspace_bytes, stream, true);
}

size_t fa_decode_workspace_size(int B, int H, int nq, int nk, int D, fa_dtype dt) {
  (void)dt;
  if (B <= 0 || H <= 0 || nq <= 0 || nk < 0 || D <= 0) return 0;
  return decode_workspace_bytes(B, H, nq, nk, D);
}

fa_status fa_decode(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int nq, int nk,
                    int D, float scale, int causal, fa_dtype dt, void* workspace, size_t workspace_bytes,
                    void* stream) {
  if (B < 0 || H < 0 || nq < 0 || nk < 0) return FA_ERR_INVALID;
  if (B > 65535 || H > 65535) return FA_ERR_UNSUPPORTED;
  if (!scale_ok(scale)) return FA_ERR_INVALID;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID;
  if (dt != FA_BF16 && dt != FA_F32 && dt != FA_F16) return FA_ERR_UNSUPPORTED;
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  if ((long long)nq * B * H > (1ll << 31) - 1) return FA_ERR_UNSUPPORTED;  // merge grid
  if (B == 0 || H == 0 || nq == 0) return FA_OK;
  fa_status st;
  for (const void* p : {q, (const void*)o})
    if ((st = check_tensor(p)) != FA_OK) return st;
  if (nk > 0)  // an empty cache has no K or V to point at
    for (const void* p : {k, v})
      if ((st = check_tensor(p)) != FA_OK) return st;
  if (lse == nullptr) return FA_ERR_INVALID;
  if (!aligned(lse, 4)) return FA_ERR_ALIGN;
  const size_t need = fa_decode_workspace_size(B, H, nq, nk, D, dt);
  if (need > 0 && (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < need)) return FA_ERR_WORKSPACE;

  Problem p{};
  p.q = q; p.k = k; p.v = v; p.o = o; p.lse = lse;
  p.B = B; p.H = H; p.N = nq; p.D = D;
  p.scale = scale; p.causal = causal;
  p.wait_limit_ns = g_wait_limit_ns.load();
  g_detail[0] = 0;
  if (note_error("status word", status_word(&p.status)) != cudaSuccess) return FA_ERR_CUDA;
  cudaError_t e = launch_decode(p, nq, nk, dt, workspace, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // extern "C"
