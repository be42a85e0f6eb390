// rx_decode_attn: split-KV decode over gathered page-1 slots with group-shared prefixes.
//
// Horizontal fusion (BatchLLM explainer, section Horizontal Fusion): the attention of a group's
// requests over their shared-prefix KV and over each request's own KV runs in ONE launch, with
// different thread blocks taking the two parts and a tiling chosen per part.  Here a CTA runs one
// work item (see DecItem):
//   * shared-prefix items stack the queries of every member (x gq query heads per KV head) into
//     16/32/64-row tiles, so each prefix KV row is read from HBM once per group and scored on the
//     tensor cores against all members at once;
//   * own-key items carry one request (gq rows padded to a 16-row tile).
// Both gather K/V rows by slot with 16-byte cp.async into a 3-stage XOR-swizzled shared-memory
// ring (the head block of a token is a contiguous run of HB*256 bytes), score with
// mma.m16n8k16 (bf16 in, fp32 accumulate), keep an online softmax in registers (quad shuffles)
// and leave a normalised partial output + base-2 log-sum-exp per (KV head, row).  A second pass
// (one warp per request and query head) merges a request's partials:
// lse = log2 sum 2^lse_i, o = sum 2^(lse_i - lse) o_i.
#include <cuda_runtime.h>
#include <math_constants.h>

#include <atomic>

#include "ptx.cuh"
#include "rx_internal.h"

namespace rx {
namespace {

struct DecParams {
  const __nv_bfloat16* k_pool;
  const __nv_bfloat16* v_pool;
  const __nv_bfloat16* q;
  const int32_t* req_to_token;
  int64_t stride;
  int hq, hkv, gq;
  float scale_log2;
  const DecItem* items;
  const int32_t* rows;
  float* part_o;
  float* part_lse;
  int64_t pool_size;
  int32_t* status;
};

constexpr int kThreads = 256;
constexpr int kStageHalf = kDecRows * kHeadDim * 2;  // one of K / V per stage: 32 KiB
static_assert(kDecRows == 128 && 2 * kStageHalf == kDecStageBytes,
              "the tilings below stage 128 (head, key) rows of K and of V");

template <int MT, int HB>
__device__ __forceinline__ void load_stage(const DecParams& p, const DecItem& it,
                                           const int32_t* s_slots, int nkeys, uint32_t kb,
                                           int tile) {
  constexpr int NK = 128 / HB;
  const int k0 = tile * NK;
#pragma unroll
  for (int u = 0; u < 128 * 16 / kThreads; ++u) {
    const int i = threadIdx.x + u * kThreads;
    const int key = i / (HB * 16);
    const int h = (i / 16) % HB;
    const int c = i % 16;
    const int hkv = it.head_block * HB + h;
    const int kk = k0 + key;
    const int slot = kk < nkeys ? s_slots[kk] : -1;
    const bool ok = (slot >= 0) && (hkv < p.hkv);
    const int64_t off = ok ? ((int64_t)slot * p.hkv + hkv) * kHeadDim + c * 8 : 0;
    const uint32_t so = swz256(h * NK + key, c);
    cp_async16(kb + so, p.k_pool + off, ok);
    cp_async16(kb + kStageHalf + so, p.v_pool + off, ok);
  }
}

template <int MT, int HB>
__device__ void run_item(const DecParams& p, const DecItem& it, uint8_t* smem) {
  constexpr int NK = 128 / HB;
  constexpr int ROWS = 16 * MT;
  constexpr int NT = NK / 8;  // 8-key n-tiles per stage
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int hl = warp / MT, mt = warp % MT;
  const int hkv = it.head_block * HB + hl;
  const int nkeys = it.k_end - it.k_begin;
  const int ntiles = (nkeys + NK - 1) / NK;
  const uint32_t sbase = smem_u32(smem);
  int32_t* s_slots = reinterpret_cast<int32_t*>(smem + kDecStages * kDecStageBytes);

  {
    const int32_t* r2t = p.req_to_token + (int64_t)it.kv_row * p.stride + it.k_begin;
    for (int i = threadIdx.x; i < nkeys; i += kThreads) {
      int slot = __ldg(r2t + i);
      if (slot < 0 || slot >= p.pool_size) {  // a table entry outside the pool: flag, never read
        atomicCAS(p.status, 0, (int)RX_ERR_RANGE);
        slot = -1;
      }
      s_slots[i] = slot;
    }
  }
  __syncthreads();

  // Query tile -> the K half of stage 2 (free until the pipeline reaches it).
  const uint32_t qb = sbase + 2 * kDecStageBytes;
  for (int i = threadIdx.x; i < 128 * 16; i += kThreads) {
    const int row = i / 16, c = i % 16;
    const int h = row / ROWS, r = row % ROWS;
    const int hk = it.head_block * HB + h;
    const int t = r / p.gq, g = r % p.gq;
    const bool ok = (hk < p.hkv) && (t < it.n_tok);
    const __nv_bfloat16* src =
        ok ? p.q + ((int64_t)__ldg(p.rows + it.row_begin + t) * p.hq + hk * p.gq + g) * kHeadDim +
                 c * 8
           : p.q;
    cp_async16(qb + swz256(row, c), src, ok);
  }
  cp_async_commit();
  load_stage<MT, HB>(p, it, s_slots, nkeys, sbase, 0);
  cp_async_commit();
  if (ntiles > 1) load_stage<MT, HB>(p, it, s_slots, nkeys, sbase + kDecStageBytes, 1);
  cp_async_commit();
  cp_async_wait<2>();
  __syncthreads();

  uint32_t qf[8][4];
  {
    const int r = hl * ROWS + mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      ldsm_x4(qb + swz256(r, 2 * kk + (lane >> 4)), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
  }
  __syncthreads();

  float o[16][4];
#pragma unroll
  for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.f, l1 = 0.f;

  for (int t = 0; t < ntiles; ++t) {
    if (t + 2 < ntiles)
      load_stage<MT, HB>(p, it, s_slots, nkeys, sbase + ((t + 2) % kDecStages) * kDecStageBytes,
                         t + 2);
    cp_async_commit();
    cp_async_wait<2>();
    __syncthreads();

    const uint32_t kb = sbase + (t % kDecStages) * kDecStageBytes;
    const uint32_t vb = kb + kStageHalf;
    float s[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
      for (int k2 = 0; k2 < 4; ++k2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kb + swz256(hl * NK + 8 * j + (lane & 7), 4 * k2 + (lane >> 3)), b0, b1, b2, b3);
        mma_16816(s[j], qf[2 * k2], b0, b1);
        mma_16816(s[j], qf[2 * k2 + 1], b2, b3);
      }
    }
    // scale to base 2, mask keys past the item, online softmax (rows lane/4 and lane/4 + 8)
    const int kbase = t * NK + 2 * (lane & 3);
    float mx0 = -CUDART_INF_F, mx1 = -CUDART_INF_F;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const bool ok = kbase + 8 * j + (e & 1) < nkeys;
        s[j][e] = ok ? s[j][e] * p.scale_log2 : -CUDART_INF_F;
      }
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
    for (int j = 0; j < NT; ++j) {
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
    for (int kk = 0; kk < NK / 16; ++kk) {
      const uint32_t a[4] = {pack_bf16(s[2 * kk][0], s[2 * kk][1]),
                             pack_bf16(s[2 * kk][2], s[2 * kk][3]),
                             pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]),
                             pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3])};
      const int vr = hl * NK + 16 * kk + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
      for (int n2 = 0; n2 < 8; ++n2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vb + swz256(vr, 2 * n2 + (lane >> 4)), b0, b1, b2, b3);
        mma_16816(o[2 * n2], a, b0, b1);
        mma_16816(o[2 * n2 + 1], a, b2, b3);
      }
    }
    __syncthreads();
  }

  // epilogue: partial rows of this warp
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  if (hkv >= p.hkv) return;
  const int rows_real = it.n_tok * p.gq;
  const int r0 = mt * 16 + lane / 4, r1 = r0 + 8;
  const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
  const int64_t base = (int64_t)it.part + (int64_t)hkv * rows_real;
  if (r0 < rows_real) {
    float* dst = p.part_o + (base + r0) * kHeadDim + 2 * (lane & 3);
#pragma unroll
    for (int n = 0; n < 16; ++n)
      *reinterpret_cast<float2*>(dst + 8 * n) = make_float2(o[n][0] * inv0, o[n][1] * inv0);
    if ((lane & 3) == 0) p.part_lse[base + r0] = l0 > 0.f ? m0 + __log2f(l0) : -CUDART_INF_F;
  }
  if (r1 < rows_real) {
    float* dst = p.part_o + (base + r1) * kHeadDim + 2 * (lane & 3);
#pragma unroll
    for (int n = 0; n < 16; ++n)
      *reinterpret_cast<float2*>(dst + 8 * n) = make_float2(o[n][2] * inv1, o[n][3] * inv1);
    if ((lane & 3) == 0) p.part_lse[base + r1] = l1 > 0.f ? m1 + __log2f(l1) : -CUDART_INF_F;
  }
}

__global__ void __launch_bounds__(kThreads, 1) decode_partial_kernel(DecParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const DecItem it = p.items[blockIdx.x];
  switch (it.kind) {
    case 0: run_item<1, 8>(p, it, smem); break;
    case 1: run_item<2, 4>(p, it, smem); break;
    default: run_item<4, 2>(p, it, smem); break;
  }
}

// One warp per (request, query head), eight to a CTA; lane owns 4 of the 128 columns.  One pass
// over the request's partials with a running maximum: acc and tot are rescaled when it grows.
constexpr int kMergeWarps = 8;
__global__ void __launch_bounds__(32 * kMergeWarps) decode_merge_kernel(
    const float* __restrict__ part_o, const float* __restrict__ part_lse,
    const int32_t* __restrict__ merge_idx, const DecMergeRef* __restrict__ refs, int batch, int hq,
    int gq, __nv_bfloat16* __restrict__ o, float* __restrict__ lse) {
  const int64_t task = (int64_t)blockIdx.x * kMergeWarps + threadIdx.x / 32;
  if (task >= (int64_t)batch * hq) return;
  const int lane = threadIdx.x % 32;
  const int b = (int)(task / hq), h = (int)(task % hq);
  const int hk = h / gq, g = h % gq;
  const int r_begin = merge_idx[b], r_end = merge_idx[b + 1];
  // Two passes per chunk of up to 32 partitions: the lanes fetch one partition's reference and
  // LSE each and agree on their maximum, so every weight is known before any row is read; the
  // row reads are then independent of one another (no load waits for the one before).
  float mx = -CUDART_INF_F, tot = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c0 = r_begin; c0 < r_end; c0 += 32) {
    const int i = c0 + lane;
    int64_t idx = 0;
    float li = -CUDART_INF_F;
    if (i < r_end) {
      const DecMergeRef rf = refs[i];
      idx = (int64_t)rf.part + (int64_t)hk * rf.rows_real + rf.row + g;
      li = part_lse[idx];
    }
    float cm = li;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, off));
    const float m_new = fmaxf(mx, cm);
    if (m_new == -CUDART_INF_F) continue;  // only empty partitions so far
    const float a = fast_exp2(mx - m_new);  // exp2(-inf) = 0
    const float w = li == -CUDART_INF_F ? 0.f : fast_exp2(li - m_new);  // empty: contributes 0
    float ws = w;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, off);
    tot = tot * a + ws;
    acc.x *= a;
    acc.y *= a;
    acc.z *= a;
    acc.w *= a;
    mx = m_new;
    const int cnt = min(32, r_end - c0);
#pragma unroll 4
    for (int j = 0; j < cnt; ++j) {
      const float wj = __shfl_sync(0xffffffffu, w, j);
      const int64_t ij = __shfl_sync(0xffffffffu, idx, j);
      if (wj == 0.f) continue;  // the same for the whole warp
      const float4 v = *reinterpret_cast<const float4*>(part_o + ij * kHeadDim + lane * 4);
      acc.x += wj * v.x;
      acc.y += wj * v.y;
      acc.z += wj * v.z;
      acc.w += wj * v.w;
    }
  }
  const float inv = tot > 0.f ? 1.f / tot : 0.f;
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
  uint2 packed;
  packed.x = *reinterpret_cast<uint32_t*>(&lo);
  packed.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(o + ((int64_t)b * hq + h) * kHeadDim + lane * 4) = packed;
  if (lane == 0)
    lse[(int64_t)b * hq + h] =
        tot > 0.f ? (mx + __log2f(tot)) * 0.69314718055994530942f : -CUDART_INF_F;
}

}  // namespace

int launch_decode(const rx_kv_desc* d, const PlanHeader* h, const void* k_pool,
                  const void* v_pool, const void* q, void* o, float* lse, void* ws,
                  void* stream, const AuxStream* aux) {
  // kernel attributes belong to the current device: set once per device (bit d of the mask)
  static std::atomic<uint64_t> attr_set{0};
  int cur = 0;
  cudaError_t de = cudaGetDevice(&cur);
  if (de != cudaSuccess) return (int)de;
  if (cur < 0 || cur >= 64) return (int)cudaErrorInvalidDevice;
  if (!((attr_set.load() >> cur) & 1)) {
    cudaError_t e = cudaFuncSetAttribute(decode_partial_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kDecSmemBytes);
    if (e != cudaSuccess) return (int)e;
    attr_set.fetch_or(1ull << cur);
  }
  uint8_t* base = static_cast<uint8_t*>(ws);
  DecParams p;
  p.k_pool = static_cast<const __nv_bfloat16*>(k_pool);
  p.v_pool = static_cast<const __nv_bfloat16*>(v_pool);
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.req_to_token = d->req_to_token;
  p.stride = d->req_to_token_stride;
  p.hq = d->num_q_heads;
  p.hkv = d->num_kv_heads;
  p.gq = d->num_q_heads / d->num_kv_heads;
  p.scale_log2 = d->softmax_scale * 1.4426950408889634f;
  p.items = reinterpret_cast<const DecItem*>(base + h->off_items);
  p.rows = reinterpret_cast<const int32_t*>(base + h->off_rows);
  p.part_o = reinterpret_cast<float*>(base + h->off_part_o);
  p.part_lse = reinterpret_cast<float*>(base + h->off_part_lse);
  p.pool_size = d->pool_size;
  p.status = reinterpret_cast<int32_t*>(base + offsetof(PlanHeader, status));
  cudaStream_t s = (cudaStream_t)stream;
  auto run_x = [&](cudaStream_t st) {  // shared-prefix units with many query rows: tcgen05 kernel
    return launch_attn_items(
        d, reinterpret_cast<const ExtItem*>(base + h->off_xitems),
        reinterpret_cast<const ExtRow*>(base + h->off_xrows),
        reinterpret_cast<const ExtSeg*>(base + h->off_xsegs), h->n_xitems, nullptr, 0, k_pool,
        v_pool, q, nullptr, nullptr, p.part_o, p.part_lse, p.status, st);
  };
  cudaStream_t merge_stream = s;
  if (h->n_xitems > 0 && h->n_items > 0) {
    // The tensor-core kernel takes whole SMs (one CTA fills an SM's shared memory), so it goes
    // first, on the caller's stream with nothing to wait for; the mma.sync units follow on the
    // plan's second stream (fork and join through events, so the pair also works under stream
    // capture) and fill the other SMs.  Each kernel's last wave would otherwise leave SMs idle.
    // The mma.sync units end last, so the merge is queued right behind them on the second stream
    // (after a wait for the tensor-core kernel, long done by then) and the caller's stream joins
    // after the merge: the merge starts as the units end instead of after a join and a launch.
    if (!aux || !aux->stream || !aux->fork || !aux->join) return (int)cudaErrorInvalidValue;
    cudaStream_t a = (cudaStream_t)aux->stream;
    cudaError_t ce = cudaEventRecord((cudaEvent_t)aux->fork, s);
    if (ce != cudaSuccess) return (int)ce;
    const int e = run_x(s);
    if (e) return e;
    ce = cudaStreamWaitEvent(a, (cudaEvent_t)aux->fork, 0);
    if (ce != cudaSuccess) return (int)ce;
    decode_partial_kernel<<<h->n_items, kThreads, kDecSmemBytes, a>>>(p);
    ce = cudaGetLastError();
    // the fork event again, now behind the tensor-core kernel (a wait takes the record before it)
    if (ce == cudaSuccess) ce = cudaEventRecord((cudaEvent_t)aux->fork, s);
    if (ce == cudaSuccess) ce = cudaStreamWaitEvent(a, (cudaEvent_t)aux->fork, 0);
    if (ce != cudaSuccess) return (int)ce;
    merge_stream = a;
  } else if (h->n_xitems > 0) {
    const int e = run_x(s);
    if (e) return e;
  } else if (h->n_items > 0) {
    decode_partial_kernel<<<h->n_items, kThreads, kDecSmemBytes, s>>>(p);
  }
  if (h->batch > 0) {
    const int64_t tasks = (int64_t)h->batch * p.hq;
    decode_merge_kernel<<<(unsigned)((tasks + kMergeWarps - 1) / kMergeWarps), 32 * kMergeWarps, 0,
                          merge_stream>>>(
        p.part_o, p.part_lse, reinterpret_cast<const int32_t*>(base + h->off_merge_idx),
        reinterpret_cast<const DecMergeRef*>(base + h->off_merge), h->batch, p.hq, p.gq,
        static_cast<__nv_bfloat16*>(o), lse);
  }
  cudaError_t ce = cudaGetLastError();
  if (ce == cudaSuccess && merge_stream != s) {
    ce = cudaEventRecord((cudaEvent_t)aux->join, merge_stream);
    if (ce == cudaSuccess) ce = cudaStreamWaitEvent(s, (cudaEvent_t)aux->join, 0);
  }
  return (int)ce;
}

}  // namespace rx
