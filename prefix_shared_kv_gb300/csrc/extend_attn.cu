// rx_extend_attn: attention of new tokens over their cached prefix plus causal self-attention.
//
// Only the unmatched tokens of a request are computed (SGLang explainer, prefix matching); their
// queries attend to the cached prefix KV and, causally, to the new tokens' KV (already stored in
// the pool).  When several requests share a cached prefix, their new rows are packed into one
// 128-row tile, so the prefix KV is read and multiplied once per tile for all of them -- the
// prefill-side counterpart of the shared-prefix reading in BatchLLM's horizontal fusion.  A tile
// walks a list of key segments: the shared prefix (visible to every row), then each member's own
// keys (visible to that member's rows only, causal on its new tokens).  One online softmax runs
// across all segments, so no partial results leave the CTA.
//
// This file holds the mma.m16n8k16 version of the tile loop: 8 warps x 16 rows, 64 keys per
// stage, 3-stage cp.async ring of swizzled K/V rows gathered by slot.
#include <cuda_runtime.h>
#include <math_constants.h>

#include "ptx.cuh"
#include "rx_internal.h"

namespace rx {
namespace {

struct ExtParams {
  const __nv_bfloat16* k_pool;
  const __nv_bfloat16* v_pool;
  const __nv_bfloat16* q;
  __nv_bfloat16* o;
  float* lse;
  const int32_t* req_to_token;
  int64_t stride;
  int hq, hkv, gq;
  float scale_log2;
  const ExtItem* items;
  const ExtRow* rows;
  const ExtSeg* segs;
  int64_t pool_size;
  int32_t* status;
};

constexpr int kThreads = 256;
constexpr int kNK = 64;
constexpr int kStages = 3;
constexpr int kHalf = kNK * kHeadDim * 2;       // 16 KiB: K (or V) rows of one stage
constexpr int kStage = 2 * kHalf;               // 32 KiB
constexpr int kMaxSegs = 1 + 128;
constexpr size_t kSmem = (size_t)kStages * kStage + kMaxSegs * sizeof(ExtSeg);

struct Cursor {
  int seg, k0;
};

__device__ __forceinline__ void advance(Cursor& c, const ExtSeg* segs, int n_seg) {
  c.k0 += kNK;
  if (c.k0 >= segs[c.seg].k_end) {
    ++c.seg;
    if (c.seg < n_seg) c.k0 = segs[c.seg].k_begin;
  }
}

__device__ __forceinline__ void load_tile(const ExtParams& p, const ExtSeg& sg, int k0, int kv_head,
                                          uint32_t kb) {
  const int32_t* r2t = p.req_to_token + (int64_t)sg.kv_row * p.stride;
#pragma unroll
  for (int u = 0; u < kNK * 16 / kThreads; ++u) {
    const int i = threadIdx.x + u * kThreads;
    const int key = i / 16, c = i % 16;
    const int kpos = k0 + key;
    int slot = kpos < sg.k_end ? __ldg(r2t + kpos) : -1;
    if (kpos < sg.k_end && (slot < 0 || slot >= p.pool_size)) {  // outside the pool: flag, skip
      atomicCAS(p.status, 0, (int)RX_ERR_RANGE);
      slot = -1;
    }
    const bool ok = slot >= 0;
    const int64_t off = ok ? ((int64_t)slot * p.hkv + kv_head) * kHeadDim + c * 8 : 0;
    const uint32_t so = swz256(key, c);
    cp_async16(kb + so, p.k_pool + off, ok);
    cp_async16(kb + kHalf + so, p.v_pool + off, ok);
  }
}

__global__ void __launch_bounds__(kThreads, 1) extend_mma_kernel(ExtParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const ExtItem it = p.items[blockIdx.x];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t sbase = smem_u32(smem);
  ExtSeg* s_segs = reinterpret_cast<ExtSeg*>(smem + kStages * kStage);
  for (int i = threadIdx.x; i < it.n_seg; i += kThreads) s_segs[i] = p.segs[it.seg_begin + i];

  // Query rows (token t = r / gq, query head kv_head*gq + r % gq) -> stage 2.
  const uint32_t qb = sbase + 2 * kStage;
  const int n_rows = it.n_tok * p.gq;
  for (int i = threadIdx.x; i < 128 * 16; i += kThreads) {
    const int r = i / 16, c = i % 16;
    const bool ok = r < n_rows;
    const __nv_bfloat16* src =
        ok ? p.q + ((int64_t)p.rows[it.row_begin + r / p.gq].q_row * p.hq + it.kv_head * p.gq +
                    r % p.gq) * kHeadDim + c * 8
           : p.q;
    cp_async16(qb + swz256(r, c), src, ok);
  }
  cp_async_commit();
  __syncthreads();  // segments visible

  // Row metadata of this thread's two rows.
  const int r0 = warp * 16 + lane / 4, r1 = r0 + 8;
  int own0 = -2, own1 = -2, kmx0 = 0, kmx1 = 0, qrow0 = 0, qrow1 = 0;
  if (r0 < n_rows) {
    const ExtRow e = p.rows[it.row_begin + r0 / p.gq];
    own0 = e.owner; kmx0 = e.kmax; qrow0 = e.q_row;
  }
  if (r1 < n_rows) {
    const ExtRow e = p.rows[it.row_begin + r1 / p.gq];
    own1 = e.owner; kmx1 = e.kmax; qrow1 = e.q_row;
  }
  const int w_lo = __reduce_min_sync(0xffffffffu, min(r0 < n_rows ? own0 : INT_MAX,
                                                      r1 < n_rows ? own1 : INT_MAX));
  const int w_hi = __reduce_max_sync(0xffffffffu, max(r0 < n_rows ? own0 : -1,
                                                      r1 < n_rows ? own1 : -1));
  const int w_kmax = __reduce_max_sync(0xffffffffu, max(kmx0, kmx1));

  int ntiles = 0;
  for (int s = 0; s < it.n_seg; ++s) ntiles += (s_segs[s].k_end - s_segs[s].k_begin + kNK - 1) / kNK;

  Cursor ld{0, it.n_seg > 0 ? s_segs[0].k_begin : 0};
  for (int pre = 0; pre < 2; ++pre) {
    if (pre < ntiles) {
      load_tile(p, s_segs[ld.seg], ld.k0, it.kv_head, sbase + pre * kStage);
      advance(ld, s_segs, it.n_seg);
    }
    cp_async_commit();
  }
  cp_async_wait<2>();
  __syncthreads();
  uint32_t qf[8][4];
  {
    const int r = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      ldsm_x4(qb + swz256(r, 2 * kk + (lane >> 4)), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
  }
  __syncthreads();

  float o[16][4];
#pragma unroll
  for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.f, l1 = 0.f;
  Cursor cc{0, it.n_seg > 0 ? s_segs[0].k_begin : 0};

  for (int t = 0; t < ntiles; ++t) {
    if (t + 2 < ntiles) {
      load_tile(p, s_segs[ld.seg], ld.k0, it.kv_head, sbase + ((t + 2) % kStages) * kStage);
      advance(ld, s_segs, it.n_seg);
    }
    cp_async_commit();
    cp_async_wait<2>();
    __syncthreads();

    const ExtSeg sg = s_segs[cc.seg];
    const int k0 = cc.k0;
    const bool active = (sg.owner < 0 || (sg.owner >= w_lo && sg.owner <= w_hi)) && k0 < w_kmax;
    if (active) {
      const uint32_t kb = sbase + (t % kStages) * kStage;
      const uint32_t vb = kb + kHalf;
      float s[8][4];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
        for (int k2 = 0; k2 < 4; ++k2) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kb + swz256(8 * j + (lane & 7), 4 * k2 + (lane >> 3)), b0, b1, b2, b3);
          mma_16816(s[j], qf[2 * k2], b0, b1);
          mma_16816(s[j], qf[2 * k2 + 1], b2, b3);
        }
      }
      const bool vis0 = sg.owner < 0 || sg.owner == own0;
      const bool vis1 = sg.owner < 0 || sg.owner == own1;
      const int lim0 = vis0 ? min(kmx0, sg.k_end) : INT_MIN;
      const int lim1 = vis1 ? min(kmx1, sg.k_end) : INT_MIN;
      float mx0 = -CUDART_INF_F, mx1 = -CUDART_INF_F;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int kp = k0 + 8 * j + 2 * (lane & 3);
        s[j][0] = (kp < lim0) ? s[j][0] * p.scale_log2 : -CUDART_INF_F;
        s[j][1] = (kp + 1 < lim0) ? s[j][1] * p.scale_log2 : -CUDART_INF_F;
        s[j][2] = (kp < lim1) ? s[j][2] * p.scale_log2 : -CUDART_INF_F;
        s[j][3] = (kp + 1 < lim1) ? s[j][3] * p.scale_log2 : -CUDART_INF_F;
        mx0 = fmaxf(mx0, fmaxf(s[j][0], s[j][1]));
        mx1 = fmaxf(mx1, fmaxf(s[j][2], s[j][3]));
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
      const float b0s = (n0 == -CUDART_INF_F) ? 0.f : n0;
      const float b1s = (n1 == -CUDART_INF_F) ? 0.f : n1;
      const float a0 = fast_exp2(m0 - b0s), a1 = fast_exp2(m1 - b1s);
      m0 = n0;
      m1 = n1;
      float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        s[j][0] = fast_exp2(s[j][0] - b0s);
        s[j][1] = fast_exp2(s[j][1] - b0s);
        s[j][2] = fast_exp2(s[j][2] - b1s);
        s[j][3] = fast_exp2(s[j][3] - b1s);
        ps0 += s[j][0] + s[j][1];
        ps1 += s[j][2] + s[j][3];
      }
      l0 = l0 * a0 + ps0;
      l1 = l1 * a1 + ps1;
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        o[n][0] *= a0;
        o[n][1] *= a0;
        o[n][2] *= a1;
        o[n][3] *= a1;
      }
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint32_t a[4] = {pack_bf16(s[2 * kk][0], s[2 * kk][1]),
                               pack_bf16(s[2 * kk][2], s[2 * kk][3]),
                               pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]),
                               pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3])};
        const int vr = 16 * kk + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
        for (int n2 = 0; n2 < 8; ++n2) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vb + swz256(vr, 2 * n2 + (lane >> 4)), b0, b1, b2, b3);
          mma_16816(o[2 * n2], a, b0, b1);
          mma_16816(o[2 * n2 + 1], a, b2, b3);
        }
      }
    }
    advance(cc, s_segs, it.n_seg);
    __syncthreads();
  }

  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
  if (r0 < n_rows) {
    const int qh = it.kv_head * p.gq + r0 % p.gq;
    __nv_bfloat16* dst = p.o + ((int64_t)qrow0 * p.hq + qh) * kHeadDim + 2 * (lane & 3);
#pragma unroll
    for (int n = 0; n < 16; ++n)
      *reinterpret_cast<uint32_t*>(dst + 8 * n) = pack_bf16(o[n][0] * inv0, o[n][1] * inv0);
    if ((lane & 3) == 0)
      p.lse[(int64_t)qrow0 * p.hq + qh] =
          l0 > 0.f ? (m0 + __log2f(l0)) * 0.69314718055994530942f : -CUDART_INF_F;
  }
  if (r1 < n_rows) {
    const int qh = it.kv_head * p.gq + r1 % p.gq;
    __nv_bfloat16* dst = p.o + ((int64_t)qrow1 * p.hq + qh) * kHeadDim + 2 * (lane & 3);
#pragma unroll
    for (int n = 0; n < 16; ++n)
      *reinterpret_cast<uint32_t*>(dst + 8 * n) = pack_bf16(o[n][2] * inv1, o[n][3] * inv1);
    if ((lane & 3) == 0)
      p.lse[(int64_t)qrow1 * p.hq + qh] =
          l1 > 0.f ? (m1 + __log2f(l1)) * 0.69314718055994530942f : -CUDART_INF_F;
  }
}

}  // namespace

int launch_extend(const rx_kv_desc* d, const PlanHeader* h, const void* k_pool,
                  const void* v_pool, const void* q, void* o, float* lse, void* ws,
                  void* stream) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(extend_mma_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    if (e != cudaSuccess) return (int)e;
    attr_set = true;
  }
  uint8_t* base = static_cast<uint8_t*>(ws);
  ExtParams p;
  p.k_pool = static_cast<const __nv_bfloat16*>(k_pool);
  p.v_pool = static_cast<const __nv_bfloat16*>(v_pool);
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.req_to_token = d->req_to_token;
  p.stride = d->req_to_token_stride;
  p.hq = d->num_q_heads;
  p.hkv = d->num_kv_heads;
  p.gq = d->num_q_heads / d->num_kv_heads;
  p.scale_log2 = d->softmax_scale * 1.4426950408889634f;
  p.items = reinterpret_cast<const ExtItem*>(base + h->off_items);
  p.rows = reinterpret_cast<const ExtRow*>(base + h->off_rows);
  p.segs = reinterpret_cast<const ExtSeg*>(base + h->off_segs);
  p.pool_size = d->pool_size;
  p.status = reinterpret_cast<int32_t*>(base + offsetof(PlanHeader, status));
  if (h->n_items > 0)
    extend_mma_kernel<<<h->n_items, kThreads, kSmem, (cudaStream_t)stream>>>(p);
  return (int)cudaGetLastError();
}

}  // namespace rx
