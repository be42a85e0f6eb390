// rx_store_kv: scatter new tokens' K and V rows into their page-1 pool slots.
//
// The cache keeps each token's KV in a page of its own (SGLang explainer, RadixAttention: pages of
// one token), so storing a token is a copy of its [num_kv_heads, 128] bf16 K row and V row into
// the slot the allocator gave it.  Per token the source and the destination are contiguous runs of
// num_kv_heads * 256 bytes; the kernel moves them in 16-byte vectors, all loads of a thread issued
// before its stores.  Pure data movement: bytes = 2 (K, V) * 2 (read + write) * T * Hkv * 256.
#include <cuda_runtime.h>

#include "rx_internal.h"

namespace rx {
namespace {

constexpr int kVecPerThread = 4;

__global__ void __launch_bounds__(256) store_kv_kernel(uint4* __restrict__ k_pool,
                                                       uint4* __restrict__ v_pool,
                                                       const uint4* __restrict__ k_new,
                                                       const uint4* __restrict__ v_new,
                                                       const int32_t* __restrict__ slots,
                                                       int64_t n_vec, int vec_per_token,
                                                       int64_t pool_size) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t base = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; base < n_vec;
       base += stride * kVecPerThread) {
    uint4 kv[kVecPerThread], vv[kVecPerThread];
    int64_t dst[kVecPerThread];
#pragma unroll
    for (int u = 0; u < kVecPerThread; ++u) {
      const int64_t i = base + u * stride;
      dst[u] = -1;
      if (i < n_vec) {
        const int64_t t = i / vec_per_token;
        const int64_t w = i - t * vec_per_token;
        const int64_t s = __ldg(slots + t);
        if (s >= 0 && s < pool_size) {
          dst[u] = s * vec_per_token + w;
          kv[u] = __ldcs(k_new + i);
          vv[u] = __ldcs(v_new + i);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kVecPerThread; ++u) {
      if (dst[u] >= 0) {
        k_pool[dst[u]] = kv[u];
        v_pool[dst[u]] = vv[u];
      }
    }
  }
}

}  // namespace

int launch_store_kv(const rx_kv_desc* d, void* k_pool, void* v_pool, const void* k_new,
                    const void* v_new, const int32_t* slots, int64_t n, void* stream) {
  if (n == 0) return 0;
  const int vec_per_token = d->num_kv_heads * kHeadDim * 2 / 16;
  const int64_t n_vec = n * vec_per_token;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t blocks = (n_vec + 256LL * kVecPerThread - 1) / (256LL * kVecPerThread);
  const int64_t cap = (int64_t)sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  store_kv_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(
      (uint4*)k_pool, (uint4*)v_pool, (const uint4*)k_new, (const uint4*)v_new, slots, n_vec,
      vec_per_token, d->pool_size);
  return (int)cudaGetLastError();
}

}  // namespace rx
