// Unit check of the tensor-core building blocks the attention kernels are
// assembled from, on one 128-row tile.
//
// One CTA of four warps:
//   1. loads A and B (each 128 x D, 16-bit, row-major) with the 3-D tiled TMA
//      boxes the kernels use (64 columns = one 128-byte swizzle row x 128
//      rows), completing on a transaction-count mbarrier;
//   2. forms S = A B^T in tensor memory with K-major shared-memory MMAs -- the
//      forward's S = Q K^T and the backward's S^T = K Q^T;
//   3. reads S back with tcgen05.ld (warp w owns lanes 32w .. 32w+31), writes
//      it out, rounds it to the 16-bit type and stores it to tensor memory as
//      packed pairs (key 2c in the low half of column c) -- the forward's P;
//   4. forms O = round16(S) B with tensor-memory-A MMAs and B read MN-major --
//      the forward's P V and the backward's dV += P^T dO;
//   5. writes O, and A as read back from the swizzled shared-memory tile
//      (16-byte chunk j of row r at chunk position j ^ (r % 8)), the layout
//      the shared-memory descriptors assume.
// Every wait is bounded and reports through the device status word.
#include "fa_internal.cuh"
#include "fa_tmap.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

using namespace ptx;

constexpr int kRows = 128;
constexpr int kBoxBytes = kRows * 128;  // one 64-column box of 128 rows
constexpr int kTmemCols = 256;          // S (and P) in columns 0..127, O from column 128

__device__ __forceinline__ uint8_t* align1024_ptr(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}

template <int D, bool F16>
__global__ void __launch_bounds__(128, 1)
    tile_selftest_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb,
                         float* __restrict__ s_out, float* __restrict__ o_out, uint4* __restrict__ a_copy,
                         unsigned* status, unsigned long long limit_ns) {
  constexpr int kBoxes = D / 64;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_tma;
  __shared__ __align__(8) uint64_t bar_mma;
  __shared__ uint32_t tmem_sh;
  __shared__ int abort_flag;
  uint8_t* sa = align1024_ptr(smem_raw);
  uint8_t* sb = sa + kBoxes * kBoxBytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = warp * 32 + lane;  // tile row = TMEM lane of this thread

  if (threadIdx.x == 0) {
    mbar_init(&bar_tma, 1);
    mbar_init(&bar_mma, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_sh, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_sh;
  const uint32_t tl = tmem_addr(tmem, warp * 32, 0);  // this warp's lanes
  const WaitCtx w{&abort_flag, status, limit_ns};

  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&bar_tma, 2 * kBoxes * kBoxBytes);
    for (int bx = 0; bx < kBoxes; ++bx) {
      tma_load_3d(sa + bx * kBoxBytes, &ta, &bar_tma, bx * 64, 0, 0);
      tma_load_3d(sb + bx * kBoxBytes, &tb, &bar_tma, bx * 64, 0, 0);
    }
  }
  bool ok = __syncthreads_and(warp_wait(&bar_tma, 0, w)) != 0;
  if (!ok) {
    // let the copies land before the CTA's shared memory is released
    if (threadIdx.x == 0) mbar_wait_drain(&bar_tma, 0, limit_ns);
  } else {
    // ---------------------------------------------------------------- S = A B^T
    if (threadIdx.x == 0) {
      tc_fence_after();
      const uint32_t id_s = idesc16<F16>(kRows, kRows, false, false);
      const uint64_t da = sdesc_sw128(smem_u32(sa), 16, 1024);
      const uint64_t db = sdesc_sw128(smem_u32(sb), 16, 1024);
      if constexpr (D == 128) {
        uint64_t a[8], b[8];
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {  // 16 columns (32 bytes) per MMA; boxes 16 KB apart
          const uint32_t off = ((ks >> 2) * kBoxBytes + (ks & 3) * 32) >> 4;
          a[ks] = da + off;
          b[ks] = db + off;
        }
        mma_ss_x8(tmem, a, b, id_s, 0u);
      } else {
        uint64_t a[4], b[4];
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          a[ks] = da + ks * 2;
          b[ks] = db + ks * 2;
        }
        mma_ss_x4(tmem, a, b, id_s, 0u);
      }
      mma_commit(&bar_mma);
    }
    ok = __syncthreads_and(warp_wait(&bar_mma, 0, w)) != 0;
    if (!ok) {
      if (threadIdx.x == 0) mbar_wait_drain(&bar_mma, 0, limit_ns);
    } else {
      tc_fence_after();
      // -------------------------------------------------------------- S out, P in
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tl + c * 32, sr[c]);
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_wait(sr[c]);
      float4* srow = reinterpret_cast<float4*>(s_out + (size_t)r * kRows);
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          srow[(c * 32 + e) >> 2] = make_float4(__uint_as_float(sr[c][e]), __uint_as_float(sr[c][e + 1]),
                                                __uint_as_float(sr[c][e + 2]), __uint_as_float(sr[c][e + 3]));
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int e0 = 64 * hf + 2 * c;
          pk[c] = pack16x2<F16>(__uint_as_float(sr[e0 >> 5][e0 & 31]), __uint_as_float(sr[(e0 + 1) >> 5][(e0 + 1) & 31]));
        }
        tmem_st32(tl + 32 * hf, pk);
      }
      tmem_st_wait();
      // ------------------------------------------------- A read back from the swizzled tile
#pragma unroll
      for (int bx = 0; bx < kBoxes; ++bx)
#pragma unroll
        for (int j = 0; j < 8; ++j)
          a_copy[(size_t)r * (D / 8) + bx * 8 + j] =
              *reinterpret_cast<const uint4*>(sa + bx * kBoxBytes + r * 128 + ((j ^ (r & 7)) << 4));
      tc_fence_before();
      __syncthreads();
      // -------------------------------------------------------------- O = P B
      if (threadIdx.x == 0) {
        tc_fence_after();
        const uint32_t id_o = idesc16<F16>(kRows, D, false, true);
        const uint64_t dbv = sdesc_sw128(smem_u32(sb), kBoxBytes, 1024);
        uint32_t a[8];
        uint64_t b[8];
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {  // 16 keys per MMA: 8 packed columns of P, 16 rows (2 KB) of B
          a[ks] = tmem + ks * 8;
          b[ks] = dbv + ((ks * 2048) >> 4);
        }
        mma_ts_x8(tmem + 128, a, b, id_o, 0u);
        mma_commit(&bar_mma);
      }
      ok = __syncthreads_and(warp_wait(&bar_mma, 1, w)) != 0;
      if (!ok) {
        if (threadIdx.x == 0) mbar_wait_drain(&bar_mma, 1, limit_ns);
      } else {
        tc_fence_after();
        float4* orow = reinterpret_cast<float4*>(o_out + (size_t)r * D);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tl + 128 + c * 32, o);
          tmem_ld_wait(o);
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            orow[(c * 32 + e) >> 2] = make_float4(__uint_as_float(o[e]), __uint_as_float(o[e + 1]),
                                                  __uint_as_float(o[e + 2]), __uint_as_float(o[e + 3]));
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool F16>
cudaError_t launch_tile_selftest_d(const CUtensorMap& ta, const CUtensorMap& tb, float* s_out, float* o_out,
                                   void* a_copy, unsigned* status, unsigned long long limit_ns, cudaStream_t s) {
  constexpr int kSmem = 2 * (D / 64) * kBoxBytes + 1024;
  cudaError_t e = cudaFuncSetAttribute(tile_selftest_kernel<D, F16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return note_error("tile self-test smem attribute", e);
  tile_selftest_kernel<D, F16><<<1, 128, kSmem, s>>>(ta, tb, s_out, o_out, static_cast<uint4*>(a_copy), status,
                                                      limit_ns);
  note_launches(1);
  return note_error("tile self-test launch", cudaGetLastError());
}

}  // namespace

cudaError_t launch_tile_selftest(const void* a, const void* b, int D, bool f16, float* s_out, float* o_out,
                                 void* a_copy, unsigned* status, unsigned long long limit_ns, cudaStream_t s) {
  Problem p{};
  p.B = 1;
  p.H = 1;
  p.N = kRows;
  p.D = D;
  p.f16 = f16 ? 1 : 0;
  CUtensorMap ta, tb;
  if (!make_map16(&ta, a, p, kRows) || !make_map16(&tb, b, p, kRows))
    return note_error("tile self-test tensor map encode", cudaErrorInvalidValue);
  if (D == 128)
    return f16 ? launch_tile_selftest_d<128, true>(ta, tb, s_out, o_out, a_copy, status, limit_ns, s)
               : launch_tile_selftest_d<128, false>(ta, tb, s_out, o_out, a_copy, status, limit_ns, s);
  return f16 ? launch_tile_selftest_d<64, true>(ta, tb, s_out, o_out, a_copy, status, limit_ns, s)
             : launch_tile_selftest_d<64, false>(ta, tb, s_out, o_out, a_copy, status, limit_ns, s);
}

}  // namespace fa
