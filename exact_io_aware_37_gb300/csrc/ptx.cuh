// Inline-PTX wrappers for the sm_103a features the tensor-core kernels use:
// mbarrier (with bounded waits), TMA tiled loads, tcgen05 tensor-memory
// allocation / load / store, tcgen05.mma (kind::f16, bf16 x bf16 -> fp32) and
// its commit, and the shared-memory / instruction descriptors.  Written from
// the public PTX ISA description of these instructions.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace fa {
namespace ptx {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t elect_one_sync() {
  uint32_t pred = 0;
  asm volatile(
      "{\n .reg .b32 r;\n .reg .pred p;\n elect.sync r|p, 0xffffffff;\n selp.b32 %0, 1, 0, p;\n}\n"
      : "=r"(pred));
  return pred;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Every wait in the tensor-core kernels is bounded: it gives up once
// `limit_ns` of wall time has passed (or another thread of the CTA already
// gave up), latches the timeout bit in the device status word and returns
// false so the caller can wind down without hanging the GPU.
struct WaitCtx {
  volatile int* abort;  // shared-memory flag, set by the first thread that gives up
  unsigned* status;     // device status word
  unsigned long long limit_ns;
};

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const WaitCtx& w) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*w.abort) return false;
      if (globaltimer_ns() - t0 > w.limit_ns) {
        *w.abort = 1;
        atomicOr(w.status, 1u);
        return false;
      }
    }
  }
}

// Warp-uniform form for warps whose lanes all wait (the softmax / gradient
// warps): every lane gets the same answer, so a warp never splits in front of
// a .sync.aligned tensor-memory instruction when a wait gives up.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtx& w) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, w)) != 0;
}

// Wait that ignores the abort flag (used only while winding down, to let
// copies already in flight land before the CTA exits).
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, unsigned long long limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// ------------------------------------------------------------------ register split
// Warpgroup-wide (all 128 threads) change of the per-thread register limit.
// The tensor-core kernels launch 384 threads at kLaunchRegs registers each;
// the two compute warpgroups raise theirs to kComputeRegs and the producer /
// MMA warpgroup lowers its to kSupportRegs.  The split must not exceed the
// launch budget or the raise would wait forever: the static_assert checks the
// arithmetic and build.py checks that ptxas gave the kernels kLaunchRegs.
constexpr int kLaunchRegs = 168;
constexpr int kComputeRegs = 200;
constexpr int kSupportRegs = 104;
static_assert(2 * 128 * kComputeRegs + 128 * kSupportRegs <= 384 * kLaunchRegs,
              "register split exceeds the launch budget");

template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled prefetch of one box into L2 (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* map, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}

// 3-D tiled load of one box into shared memory; completion is signalled on
// `bar` as transaction bytes.  c0 is the innermost (contiguous) coordinate.
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                            int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], "
      "[%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d_hint(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int c0,
                                                 int c1, int c2, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, "
      "{%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Bulk (non-tensor) reduce-add of `bytes` (multiple of 16, both addresses
// 16-byte aligned) of float32 from shared to global memory, done by the copy
// engine; tracked in the issuing thread's bulk groups.
__device__ __forceinline__ void bulk_reduce_add_f32(float* gdst, const void* ssrc, uint32_t bytes) {
  asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(gdst),
               "r"(smem_u32(ssrc)), "r"(bytes)
               : "memory");
}
// 2-D tiled reduce-add of one box from shared memory into global memory
// (float32 add by the copy engine, tracked in the issuing thread's bulk groups
// like bulk_reduce_add_f32).  c0 is the innermost coordinate (its byte offset
// must be a multiple of 16); rows past the tensor's end are not written.
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, const void* smem_src, int c0, int c1) {
  asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(smem_src)), "r"(c0), "r"(c1)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's committed bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Named barrier among `count` threads returning the AND of their predicates:
// every participant gets the same answer.
__device__ __forceinline__ bool named_bar_and(int id, int count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n barrier.red.and.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

// Named barrier among `count` threads (a multiple of 32); id 0 is __syncthreads.
__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ------------------------------------------------------------------ tcgen05: TMEM
// Allocation is warp-wide; the allocated base column address is written to
// shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Tensor-memory address: lane in bits 31..16, column in bits 15..0.
__device__ __forceinline__ uint32_t tmem_addr(uint32_t base, uint32_t lane, uint32_t col) {
  return base + (lane << 16) + col;
}

#define FA_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), "=r"(r[i + 5]), \
                 "=r"(r[i + 6]), "=r"(r[i + 7])
#define FA_W8(i) "+r"(r[i]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]), "+r"(r[i + 4]), "+r"(r[i + 5]), \
                 "+r"(r[i + 6]), "+r"(r[i + 7])
#define FA_I8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), "r"(r[i + 4]), "r"(r[i + 5]), \
                 "r"(r[i + 6]), "r"(r[i + 7])

// Each thread of a warp reads 32 consecutive 32-bit columns of its own lane
// (warp w of a warpgroup owns lanes 32*(w%4) .. 32*(w%4)+31).  The registers
// are not valid until tmem_ld_wait() has bound them.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : FA_R8(0), FA_R8(8), FA_R8(16), FA_R8(24)
      : "r"(taddr));
}
// Wait for this thread's outstanding tensor-memory loads; the "+r" operands
// keep the compiler from using the loaded registers before the wait.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : FA_W8(0), FA_W8(8), FA_W8(16), FA_W8(24)::"memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      FA_I8(0), FA_I8(8), FA_I8(16), FA_I8(24)
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      FA_I8(0), FA_I8(8)
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

#undef FA_R8
#undef FA_W8
#undef FA_I8

// ------------------------------------------------------------------ tcgen05: MMA
// D[tmem] (+)= A * B^T with A (M x K) and B (N x K) described by shared-memory
// descriptors (K = 16 for bf16).  `accumulate` = 0 overwrites D.
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Same with A read from tensor memory (M lanes x K/2 packed bf16 pairs).
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(
          d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Back-to-back groups of MMAs issued from one asm block, so no other
// instruction of the issuing thread sits between them (each tcgen05.mma
// occupies the issuer until the previous one has nearly finished, so any
// instruction in between adds directly to the per-MMA time).  The first MMA
// accumulates iff `acc` != 0; the others always accumulate.
__device__ __forceinline__ void mma_ss_x4(uint32_t d, const uint64_t (&a)[4], const uint64_t (&b)[4], uint32_t idesc,
                                          uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.b32 p, %9, 0;\n setp.eq.b32 q, %9, %9;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %5, %10, p;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %2, %6, %10, q;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %7, %10, q;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %4, %8, %10, q;\n}\n" ::"r"(d),
      "l"(a[0]), "l"(a[1]), "l"(a[2]), "l"(a[3]), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "r"(acc), "r"(idesc)
      : "memory");
}
__device__ __forceinline__ void mma_ss_x8(uint32_t d, const uint64_t (&a)[8], const uint64_t (&b)[8], uint32_t idesc,
                                          uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.b32 p, %17, 0;\n setp.eq.b32 q, %17, %17;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %9, %18, p;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %2, %10, %18, q;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %11, %18, q;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %4, %12, %18, q;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %13, %18, q;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %6, %14, %18, q;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %7, %15, %18, q;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %8, %16, %18, q;\n}\n" ::"r"(d),
      "l"(a[0]), "l"(a[1]), "l"(a[2]), "l"(a[3]), "l"(a[4]), "l"(a[5]), "l"(a[6]), "l"(a[7]), "l"(b[0]), "l"(b[1]),
      "l"(b[2]), "l"(b[3]), "l"(b[4]), "l"(b[5]), "l"(b[6]), "l"(b[7]), "r"(acc), "r"(idesc)
      : "memory");
}
// Same with A read from tensor memory at column addresses a[i].
__device__ __forceinline__ void mma_ts_x8(uint32_t d, const uint32_t (&a)[8], const uint64_t (&b)[8], uint32_t idesc,
                                          uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.b32 p, %17, 0;\n setp.eq.b32 q, %17, %17;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %9, %18, p;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%2], %10, %18, q;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], %11, %18, q;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%4], %12, %18, q;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%5], %13, %18, q;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%6], %14, %18, q;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%7], %15, %18, q;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%8], %16, %18, q;\n}\n" ::"r"(d),
      "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(a[4]), "r"(a[5]), "r"(a[6]), "r"(a[7]), "l"(b[0]), "l"(b[1]),
      "l"(b[2]), "l"(b[3]), "l"(b[4]), "l"(b[5]), "l"(b[6]), "l"(b[7]), "r"(acc), "r"(idesc)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle (the layout TMA writes
// with CU_TENSOR_MAP_SWIZZLE_128B into a 1024-byte aligned buffer: rows of
// 128 bytes, 16-byte chunks XOR-permuted by row % 8).
//   bits  0-13 start address >> 4
//   bits 16-29 leading-dimension byte offset >> 4
//   bits 32-45 stride-dimension byte offset >> 4
//   bits 46-47 descriptor version (1)
//   bits 61-63 layout: 2 = 128-byte swizzle
// K-major operand: SBO = 1024 (next group of 8 rows); LBO unused (1).
// MN-major operand: LBO = byte distance between 64-element MN blocks,
// SBO = 1024 (next group of 8 rows along K).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor, kind::f16 with bf16 A/B and fp32 D.
//   bits 4-5 D format (1 = f32); 7-9 A format (1 = bf16); 10-12 B format;
//   bit 15 A major (0 = K, 1 = MN); bit 16 B major; 17-22 N >> 3; 24-28 M >> 4.
// A and B have one type (F16: both fp16, else both bf16), D is fp32.
template <bool F16>
__host__ __device__ constexpr uint32_t idesc16(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | ((F16 ? 0u : 1u) << 7) | ((F16 ? 0u : 1u) << 10) | ((a_mn_major ? 1u : 0u) << 15) |
         ((b_mn_major ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major) {
  return idesc16<false>(M, N, a_mn_major, b_mn_major);
}

// Pack two fp32 into a bf16x2 word (round to nearest even); `lo` lands in
// bits 15..0.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// The same for fp16x2.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
template <bool F16>
__device__ __forceinline__ uint32_t pack16x2(float lo, float hi) {
  if constexpr (F16)
    return pack_f16x2(lo, hi);
  else
    return pack_bf16x2(lo, hi);
}

// Packed fp32 pair arithmetic (one instruction for two lanes of work).
// (d0, d1) = (a0, a1) * (b, b) + (c0, c1)
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a0, float a1, float b, float c0, float c1) {
  asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %4};\n mov.b64 rc, {%5, %6};\n"
      " fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}\n"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b), "f"(c0), "f"(c1));
}
// (s0, s1) += (a0, a1)
__device__ __forceinline__ void fadd2(float& s0, float& s1, float a0, float a1) {
  asm("{\n .reg .b64 ra, rs;\n mov.b64 ra, {%2, %3};\n mov.b64 rs, {%0, %1};\n add.rn.f32x2 rs, rs, ra;\n"
      " mov.b64 {%0, %1}, rs;\n}\n"
      : "+f"(s0), "+f"(s1)
      : "f"(a0), "f"(a1));
}
// (d0, d1) = (a0, a1) - (b0, b1)
__device__ __forceinline__ void fsub2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n sub.rn.f32x2 rd, ra, rb;\n"
      " mov.b64 {%0, %1}, rd;\n}\n"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
// (d0, d1) = (a0, a1) * (b0, b1)
__device__ __forceinline__ void fmul2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n mul.rn.f32x2 rd, ra, rb;\n"
      " mov.b64 {%0, %1}, rd;\n}\n"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// Transpose of 16-byte chunks within each group of E consecutive lanes (E a
// power of two): on entry chunk slot s of lane g + b (g the group's first lane)
// holds chunk s of row b; on return slot s holds chunk b of row s.  One xor
// step per bit swaps that bit between the lane and the slot index.
template <int E>
__device__ __forceinline__ void exchange_chunks(uint32_t (&u)[4 * E], int lane) {
#pragma unroll
  for (int m = E / 2; m >= 1; m >>= 1) {
    const bool hi = (lane & m) != 0;
#pragma unroll
    for (int s0 = 0; s0 < E; ++s0) {
      if (s0 & m) continue;
      const int s1 = s0 | m;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        // the lower lane keeps slot s0 and passes slot s1 up; the upper the reverse
        const uint32_t send = hi ? u[4 * s0 + q] : u[4 * s1 + q];
        const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, m);
        u[4 * s0 + q] = hi ? recv : u[4 * s0 + q];
        u[4 * s1 + q] = hi ? u[4 * s1 + q] : recv;
      }
    }
  }
}

// max(a, b, c)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace ptx
}  // namespace fa
