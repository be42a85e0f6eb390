// rx_selftest_pair_mma: one cluster of two CTAs runs the tensor-core steps of the paired extend
// kernel once, on operands loaded from global memory, and writes the results back:
//   S = Q K^T     (M = 256 query rows, N = 128 keys, K = 128), A and B from shared memory;
//   O = P V       (M = 256, N = 128 columns of V, K = 128 keys), A = P from tensor memory.
// CTA r holds query rows [128 r, 128 r + 128), keys [64 r, 64 r + 64) of K (its half of S's N) and
// columns [64 r, 64 r + 64) of V (its half of O's N), in the layouts the kernel uses.  A test
// compares S and O with a plain matrix product, so the operand split, the descriptors and the
// pair's commits and barriers are checked on a small case before the kernel relies on them.
// Every wait is bounded; on a timeout the status word holds RX_ERR_TIMEOUT and the outputs are
// left unwritten.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "pair.cuh"
#include "rx_internal.h"
#include "tc.cuh"

namespace {

constexpr int kQHalf = 128 * 128;         // 64 columns of 128 rows (bf16): 16 KiB
constexpr int kKHalf = 64 * 128;          // 64 columns of 64 keys: 8 KiB
constexpr int kOffQ = 0, kOffK = 2 * kQHalf, kOffV = kOffK + 2 * kKHalf;  // V: 128 keys x 128 B
constexpr int kOffBar = kOffV + 128 * 128;
constexpr int kOffTmem = kOffBar + 8;
constexpr int kOffAbort = kOffTmem + 8;
constexpr size_t kSmem = 1024 + kOffAbort + 16;
constexpr uint32_t kCols = 256;           // S [0, 128) with P over [64, 128); O [128, 256)

// Byte offset of element (row, col) of a 128-byte-swizzled tile whose rows are 128 bytes (64
// bf16) wide: the 16-byte chunk index is XOR-ed with the row's low three bits.
__device__ __forceinline__ uint32_t sw128(int row, int col) {
  return (uint32_t)(row * 128 + ((((col >> 3) & 7) ^ (row & 7)) << 4) + (col & 7) * 2);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(256, 1)
    pair_mma_kernel(const __nv_bfloat16* q, const __nv_bfloat16* k, const __nv_bfloat16* v,
                    const __nv_bfloat16* p, float* s_out, float* o_out, int32_t* info) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = rx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023) & ~1023u;
  uint8_t* sp = smem_raw + (base - raw);
  const uint32_t rank = rx::pair::cta_rank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort = reinterpret_cast<volatile int*>(sp + kOffAbort);
  const uint32_t bar = base + kOffBar;
  if (threadIdx.x == 0) {
    rx::tc::mbar_init(bar, 1);
    *abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) rx::pair::alloc(base + kOffTmem, kCols);
  // operands of this CTA, in the kernel's layouts
  for (int i = threadIdx.x; i < 128 * 128; i += blockDim.x) {  // Q rows, K-major, two halves
    const int r = i >> 7, c = i & 127;
    *reinterpret_cast<__nv_bfloat16*>(sp + kOffQ + (c >> 6) * kQHalf + sw128(r, c)) =
        q[(int64_t)(128 * rank + r) * 128 + c];
  }
  for (int i = threadIdx.x; i < 64 * 128; i += blockDim.x) {  // keys 64 r .., K-major
    const int r = i >> 7, c = i & 127;
    *reinterpret_cast<__nv_bfloat16*>(sp + kOffK + (c >> 6) * kKHalf + sw128(r, c)) =
        k[(int64_t)(64 * rank + r) * 128 + c];
  }
  for (int i = threadIdx.x; i < 128 * 64; i += blockDim.x) {  // V columns 64 r .., MN-major
    const int key = i >> 6, c = i & 63;
    *reinterpret_cast<__nv_bfloat16*>(sp + kOffV + sw128(key, c)) =
        v[(int64_t)key * 128 + 64 * rank + c];
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  rx::tc::fence_before();
  __syncthreads();
  rx::pair::cluster_sync();  // both CTAs' operands and barriers are ready
  rx::tc::fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sp + kOffTmem);
  if (threadIdx.x == 0) info[1 + rank] = (int32_t)tmem;
  int32_t* status = info;

  constexpr uint32_t idS = rx::tc::idesc_bf16(256, 128, false, false);
  constexpr uint32_t idO = rx::tc::idesc_bf16(256, 128, false, true);
  if (rank == 0 && threadIdx.x == 0) {
    const uint64_t qd = rx::tc::desc_sw128(base + kOffQ, 16, 1024);
    const uint64_t kd = rx::tc::desc_sw128(base + kOffK, 16, 1024);
#pragma unroll
    for (int s = 0; s < 8; ++s)
      rx::pair::mma_ss(tmem, qd + (((s >> 2) * kQHalf + (s & 3) * 32) >> 4),
                       kd + (((s >> 2) * kKHalf + (s & 3) * 32) >> 4), idS, s > 0 ? 1u : 0u);
    rx::pair::commit_mc(bar, 0x3);
  }
  const uint32_t lane_t = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
  const int row = 128 * (int)rank + 32 * (warp & 3) + lane;
  bool ok = rx::pair::wait(bar, 0, abort, status, 2000000000ull);
  if (warp < 4) {
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      rx::tc::fence_after();
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        rx::tc::ld32(lane_t + 32 * c, r);
        rx::tc::wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) s_out[(int64_t)row * 128 + 32 * c + j] = __uint_as_float(r[j]);
      }
      // P over the upper half of S: 128 keys, two bf16 per column
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t w[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const __nv_bfloat16* src = p + (int64_t)row * 128 + 64 * c + 2 * j;
          w[j] = (uint32_t)__bfloat16_as_ushort(src[0]) |
                 ((uint32_t)__bfloat16_as_ushort(src[1]) << 16);
        }
        rx::tc::st32(lane_t + 64 + 32 * c, w);
      }
      rx::tc::wait_st();
    }
  }
  rx::tc::fence_before();
  __syncthreads();
  rx::pair::cluster_sync();  // both CTAs' P rows are in tensor memory
  rx::tc::fence_after();
  if (rank == 0 && threadIdx.x == 0 && !*abort) {
    const uint64_t vd = rx::tc::desc_sw128(base + kOffV, 128 * 128, 1024);
#pragma unroll
    for (int s = 0; s < 8; ++s)
      rx::pair::mma_ts(tmem + 128, tmem + 64 + 8 * s, vd + ((s * 2048) >> 4), idO,
                       s > 0 ? 1u : 0u);
    rx::pair::commit_mc(bar, 0x3);
  }
  ok = !*abort && rx::pair::wait(bar, 1, abort, status, 2000000000ull);
  if (warp < 4) {
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      rx::tc::fence_after();
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        rx::tc::ld32(lane_t + 128 + 32 * c, r);
        rx::tc::wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) o_out[(int64_t)row * 128 + 32 * c + j] = __uint_as_float(r[j]);
      }
    }
  }
  rx::tc::fence_before();
  __syncthreads();
  rx::pair::cluster_sync();  // no MMA of the pair is pending before the columns are released
  if (warp == 1) {
    rx::tc::fence_after();
    rx::pair::dealloc(tmem, kCols);
  }
}

}  // namespace

extern "C" rx_status rx_selftest_pair_mma(const void* q, const void* k, const void* v,
                                          const void* p, float* s_out, float* o_out,
                                          int32_t* info, rx_stream_t stream) {
  if (!q || !k || !v || !p || !s_out || !o_out || !info)
    return rx::set_error(RX_ERR_INVALID, "rx_selftest_pair_mma: NULL argument");
  cudaError_t e = cudaFuncSetAttribute(pair_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmem);
  if (e != cudaSuccess) return rx::set_error(RX_ERR_CUDA, cudaGetErrorString(e));
  pair_mma_kernel<<<2, 256, kSmem, (cudaStream_t)stream>>>(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
      static_cast<const __nv_bfloat16*>(v), static_cast<const __nv_bfloat16*>(p), s_out, o_out,
      info);
  e = cudaGetLastError();
  return e == cudaSuccess ? RX_OK : rx::set_error(RX_ERR_CUDA, cudaGetErrorString(e));
}
