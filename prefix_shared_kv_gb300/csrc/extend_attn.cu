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
// Blackwell tile loop (one CTA per work item, 256 threads, warp-specialised):
//   warps 5-7  producers: gather the next 128 keys' K and V rows by slot with 16-byte cp.async
//              into a 2-stage ring laid out as 128-byte-swizzled UMMA tiles; completion is
//              signalled per stage with cp.async.mbarrier.arrive;
//   warp 4     MMA issuer (one thread): S = Q K^T with tcgen05.mma (both operands K-major in
//              shared memory, fp32 accumulator in TMEM, double-buffered), then O += P V with P
//              read from TMEM and V as an MN-major shared-memory operand;
//   warps 0-3  softmax: thread r owns query row r (TMEM lane r): tcgen05.ld of its S row, masks,
//              online max / sum in base 2 (the running max is only moved -- and O in TMEM rescaled
//              -- when it grows by more than 2^8), P = exp2(.) packed to bf16 and written to its own
//              TMEM columns with tcgen05.st for the PV MMA; finally O / l and the LSE.
// Every mbarrier wait is bounded (globaltimer); a timeout records RX_ERR_TIMEOUT in the
// workspace status word and every role leaves its loop.
#include <cuda_runtime.h>
#include <math_constants.h>

#include "ptx.cuh"
#include "rx_internal.h"
#include "tc.cuh"

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
constexpr int kProducers = 96;          // warps 5..7
constexpr int kN = 128;                 // keys per tile
constexpr int kStages = 2;
constexpr int kMaxSegs = 1 + 128;
constexpr int kHalfBlock = 128 * 128;   // one 64-column half of a 128-row tile: 16 KiB
constexpr int kTile = 2 * kHalfBlock;   // 128 rows x 128 bf16: 32 KiB
constexpr int kOffQ = 0;
constexpr int kOffStage = kTile;                        // stage s: K at +s*2*kTile, V after it
constexpr int kOffSlots = kOffStage + kStages * 2 * kTile;
constexpr int kOffSegs = kOffSlots + kStages * kN * 4;
constexpr int kOffBar = kOffSegs + kMaxSegs * 16;
enum { B_KV_FULL = 0, B_KV_EMPTY = 2, B_Q_FULL = 4, B_S_FULL = 5, B_P_FULL = 7, B_PV_DONE = 9,
       B_FINAL = 10, B_COUNT = 11 };
constexpr int kOffTmem = kOffBar + B_COUNT * 8;
constexpr int kOffAbort = kOffTmem + 8;
constexpr size_t kSmem = 1024 + kOffAbort + 16;
constexpr uint32_t kTmemCols = 512;     // S0 [0,128), S1 [128,256), O [256,384), P0, P1 64 each
constexpr uint32_t kColO = 256;
constexpr uint32_t kColP = 384;
constexpr uint64_t kWaitNs = 2000000000ull;

static_assert(kSmem <= 227 * 1024, "shared memory budget");

struct TileIter {
  int seg, k0;
};
__device__ __forceinline__ void tile_next(TileIter& c, const ExtSeg* segs, int n_seg) {
  c.k0 += kN;
  if (c.k0 >= segs[c.seg].k_end) {
    ++c.seg;
    if (c.seg < n_seg) c.k0 = segs[c.seg].k_begin;
  }
}

// byte offset of 16-byte chunk c (0..15) of row r in a K-major 128-row tile (two SW128 halves)
__device__ __forceinline__ uint32_t tile_off(int r, int c) {
  return (uint32_t)((c >> 3) * kHalfBlock + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// Named barrier over `n` threads that also ORs a predicate across them.
__device__ __forceinline__ bool bar_any(int id, int n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n.reg .pred p, q;\nsetp.ne.u32 p, %1, 0;\nbar.red.or.pred q, %2, %3, p;\n"
      "selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void cp_async_mbar_arrive(uint32_t mbar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(mbar) : "memory");
}

__device__ __forceinline__ void producer(const ExtParams& p, const ExtItem& it,
                                         const ExtSeg* segs, int ntiles, uint32_t base,
                                         uint8_t* sp, volatile int* abort) {
  const int ptid = threadIdx.x - 160;
  const int n_rows = it.n_tok * p.gq;
  // query tile
  for (int i = ptid; i < 128 * 16; i += kProducers) {
    const int r = i >> 4, c = i & 15;
    const bool ok = r < n_rows;
    const __nv_bfloat16* src =
        ok ? p.q + ((int64_t)p.rows[it.row_begin + r / p.gq].q_row * p.hq + it.kv_head * p.gq +
                    r % p.gq) * kHeadDim + c * 8
           : p.q;
    cp_async16(base + kOffQ + tile_off(r, c), src, ok);
  }
  cp_async_mbar_arrive(base + kOffBar + 8 * B_Q_FULL);
  TileIter cur{0, segs[0].k_begin};
  for (int t = 0; t < ntiles; ++t) {
    const int st = t & 1;
    const bool waited = t < kStages ||
        tc::mbar_wait(base + kOffBar + 8 * (B_KV_EMPTY + st), ((t >> 1) - 1) & 1, abort,
                      p.status, kWaitNs);
    const ExtSeg sg = segs[cur.seg];
    int32_t* slots = reinterpret_cast<int32_t*>(sp + kOffSlots) + st * kN;
    const int32_t* r2t = p.req_to_token + (int64_t)sg.kv_row * p.stride;
    for (int k = ptid; waited && k < kN; k += kProducers) {
      const int kpos = cur.k0 + k;
      int s = kpos < sg.k_end ? __ldg(r2t + kpos) : -1;
      if (kpos < sg.k_end && (s < 0 || s >= p.pool_size)) {  // outside the pool: flag, skip
        atomicCAS(p.status, 0, (int)RX_ERR_RANGE);
        s = -1;
      }
      slots[k] = s;
    }
    // slots visible to all producers; leave together if any of them gave up waiting
    if (bar_any(1, kProducers, !waited || *abort)) break;
    const uint32_t kb = base + kOffStage + st * 2 * kTile;
    for (int i = ptid; i < kN * 16; i += kProducers) {
      const int key = i >> 4, c = i & 15;
      const int s = slots[key];
      const int64_t off = s >= 0 ? ((int64_t)s * p.hkv + it.kv_head) * kHeadDim + c * 8 : 0;
      const uint32_t so = tile_off(key, c);
      cp_async16(kb + so, p.k_pool + off, s >= 0);
      cp_async16(kb + kTile + so, p.v_pool + off, s >= 0);
    }
    cp_async_mbar_arrive(base + kOffBar + 8 * (B_KV_FULL + st));
    tile_next(cur, segs, it.n_seg);
  }
  cp_async_wait<0>();
}

__device__ __forceinline__ void mma_issuer(const ExtParams& p, int ntiles, uint32_t base,
                                           uint32_t tmem, volatile int* abort) {
  constexpr uint32_t idS = tc::idesc_bf16(128, kN, false, false);
  constexpr uint32_t idO = tc::idesc_bf16(128, 128, false, true);
  const uint32_t bar = base + kOffBar;
  auto pv = [&](int u) -> bool {
    if (!tc::mbar_wait(bar + 8 * (B_P_FULL + (u & 1)), (u >> 1) & 1, abort, p.status, kWaitNs))
      return false;
    tc::fence_after();
    const uint32_t vb = base + kOffStage + (u & 1) * 2 * kTile + kTile;
    const uint32_t pcol = tmem + kColP + (u & 1) * 64;
#pragma unroll
    for (int s = 0; s < kN / 16; ++s)
      tc::mma_ts(tmem + kColO, pcol + 8 * s, tc::desc_sw128(vb + s * 2048, kHalfBlock, 1024), idO,
                 (u > 0 || s > 0) ? 1u : 0u);
    tc::commit(bar + 8 * (B_KV_EMPTY + (u & 1)));
    tc::commit(bar + 8 * B_PV_DONE);
    return true;
  };
  bool ok = tc::mbar_wait(bar + 8 * B_Q_FULL, 0, abort, p.status, kWaitNs);
  for (int t = 0; ok && t < ntiles; ++t) {
    if (!tc::mbar_wait(bar + 8 * (B_KV_FULL + (t & 1)), (t >> 1) & 1, abort, p.status, kWaitNs)) {
      ok = false;
      break;
    }
    tc::fence_proxy_async();
    tc::fence_after();
    const uint32_t qb = base + kOffQ;
    const uint32_t kb = base + kOffStage + (t & 1) * 2 * kTile;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const uint32_t koff = (s >> 2) * kHalfBlock + (s & 3) * 32;
      tc::mma_ss(tmem + (t & 1) * 128, tc::desc_sw128(qb + koff, 16, 1024),
                 tc::desc_sw128(kb + koff, 16, 1024), idS, s > 0 ? 1u : 0u);
    }
    tc::commit(bar + 8 * (B_S_FULL + (t & 1)));
    if (t >= 1 && !pv(t - 1)) ok = false;
  }
  if (ok && ntiles > 0) pv(ntiles - 1);
  // drain: every MMA issued above completes before TMEM is released
  tc::commit(bar + 8 * B_FINAL);
  tc::mbar_wait(bar + 8 * B_FINAL, 0, abort, p.status, kWaitNs);
}

__device__ __forceinline__ void softmax_rows(const ExtParams& p, const ExtItem& it,
                                             const ExtSeg* segs, int ntiles, uint32_t base,
                                             uint32_t tmem, volatile int* abort) {
  const int r = threadIdx.x;  // query row == TMEM lane
  const int warp = r >> 5;
  const uint32_t lane_t = tmem + ((uint32_t)(32 * warp) << 16);
  const uint32_t bar = base + kOffBar;
  const int n_rows = it.n_tok * p.gq;
  const bool valid = r < n_rows;
  int owner = -2, kmax = 0, q_row = 0;
  if (valid) {
    const ExtRow e = p.rows[it.row_begin + r / p.gq];
    owner = e.owner;
    kmax = e.kmax;
    q_row = e.q_row;
  }
  const float sl2 = p.scale_log2;
  float m_used = -CUDART_INF_F, l = 0.f;
  TileIter cur{0, segs[0].k_begin};
  bool ok = true;
  for (int t = 0; t < ntiles; ++t) {
    const int b = t & 1;
    const bool w_ok = tc::mbar_wait(bar + 8 * (B_S_FULL + b), (t >> 1) & 1, abort, p.status,
                                    kWaitNs);
    if (__any_sync(0xffffffffu, !w_ok)) {  // the warp leaves together
      ok = false;
      break;
    }
    tc::fence_after();
    const ExtSeg sg = segs[cur.seg];
    const bool vis = valid && (sg.owner < 0 || sg.owner == owner);
    const int lim = vis ? min(kmax, sg.k_end) : 0;  // keys at positions >= lim are masked
    const int n_ok = max(0, min(kN, lim - cur.k0));
    uint32_t sr[4][32];
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) tc::ld32(lane_t + b * 128 + 32 * q4, sr[q4]);
    tc::wait_ld();
    float mx = -CUDART_INF_F;
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (32 * q4 + j < n_ok) mx = fmaxf(mx, __uint_as_float(sr[q4][j]));
    const float m_new = n_ok > 0 ? fmaxf(m_used, mx * sl2) : m_used;
    const bool need = m_new > m_used + 8.f;
    if (__any_sync(0xffffffffu, need)) {
      const float alpha = need ? fast_exp2(m_used - m_new) : 1.f;  // exp2(-inf) = 0
      if (t > 0) {
        const bool w_ok = tc::mbar_wait(bar + 8 * B_PV_DONE, (t - 1) & 1, abort, p.status,
                                        kWaitNs);
        if (__any_sync(0xffffffffu, !w_ok)) {
          ok = false;
          break;
        }
        tc::fence_after();
#pragma unroll 1
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t ov[32];
          tc::ld32(lane_t + kColO + 32 * q4, ov);
          tc::wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * alpha);
          tc::st32(lane_t + kColO + 32 * q4, ov);
        }
        tc::wait_st();
      }
      l *= alpha;
      if (need) m_used = m_new;
    }
    float ps = 0.f;
    uint32_t pk[2][32];
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        const int c = 32 * q4 + j;
        const float p0 = c < n_ok ? fast_exp2(fmaf(__uint_as_float(sr[q4][j]), sl2, -m_used)) : 0.f;
        const float p1 =
            c + 1 < n_ok ? fast_exp2(fmaf(__uint_as_float(sr[q4][j + 1]), sl2, -m_used)) : 0.f;
        ps += p0 + p1;
        pk[q4 >> 1][(c & 63) >> 1] = pack_bf16(p0, p1);
      }
    l += ps;
    tc::st32(lane_t + kColP + b * 64, pk[0]);
    tc::st32(lane_t + kColP + b * 64 + 32, pk[1]);
    tc::wait_st();
    tc::fence_before();
    tc::mbar_arrive(bar + 8 * (B_P_FULL + b));
    tile_next(cur, segs, it.n_seg);
  }
  if (!ok || ntiles == 0) return;
  const bool w_ok = tc::mbar_wait(bar + 8 * B_PV_DONE, (ntiles - 1) & 1, abort, p.status, kWaitNs);
  if (__any_sync(0xffffffffu, !w_ok)) return;
  tc::fence_after();
  const float inv = l > 0.f ? 1.f / l : 0.f;
  const int qh = it.kv_head * p.gq + (r % p.gq);
  __nv_bfloat16* dst = p.o + ((int64_t)q_row * p.hq + qh) * kHeadDim;
#pragma unroll 1
  for (int q4 = 0; q4 < 4; ++q4) {
    uint32_t ov[32];
    tc::ld32(lane_t + kColO + 32 * q4, ov);
    tc::wait_ld();
    if (valid) {
      uint32_t w[16];
#pragma unroll
      for (int j = 0; j < 16; ++j)
        w[j] = pack_bf16(__uint_as_float(ov[2 * j]) * inv, __uint_as_float(ov[2 * j + 1]) * inv);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        *reinterpret_cast<uint4*>(dst + 32 * q4 + 8 * j) =
            make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
    }
  }
  if (valid)
    p.lse[(int64_t)q_row * p.hq + qh] =
        l > 0.f ? (m_used + __log2f(l)) * 0.69314718055994530942f : -CUDART_INF_F;
}

__global__ void __launch_bounds__(kThreads, 1) extend_tc_kernel(ExtParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023) & ~1023u;
  uint8_t* sp = smem_raw + (base - raw);
  const ExtItem it = p.items[blockIdx.x];
  const int warp = threadIdx.x >> 5;
  ExtSeg* segs = reinterpret_cast<ExtSeg*>(sp + kOffSegs);
  volatile int* abort = reinterpret_cast<volatile int*>(sp + kOffAbort);
  for (int i = threadIdx.x; i < it.n_seg; i += kThreads) segs[i] = p.segs[it.seg_begin + i];
  if (threadIdx.x == 0) {
    const uint32_t bar = base + kOffBar;
    tc::mbar_init(bar + 8 * (B_KV_FULL + 0), kProducers);
    tc::mbar_init(bar + 8 * (B_KV_FULL + 1), kProducers);
    tc::mbar_init(bar + 8 * (B_KV_EMPTY + 0), 1);
    tc::mbar_init(bar + 8 * (B_KV_EMPTY + 1), 1);
    tc::mbar_init(bar + 8 * B_Q_FULL, kProducers);
    tc::mbar_init(bar + 8 * (B_S_FULL + 0), 1);
    tc::mbar_init(bar + 8 * (B_S_FULL + 1), 1);
    tc::mbar_init(bar + 8 * (B_P_FULL + 0), 128);
    tc::mbar_init(bar + 8 * (B_P_FULL + 1), 128);
    tc::mbar_init(bar + 8 * B_PV_DONE, 1);
    tc::mbar_init(bar + 8 * B_FINAL, 1);
    *abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 4) tc::alloc(base + kOffTmem, kTmemCols);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sp + kOffTmem);
  int ntiles = 0;
  for (int s = 0; s < it.n_seg; ++s) ntiles += (segs[s].k_end - segs[s].k_begin + kN - 1) / kN;

  if (warp < 4) {
    softmax_rows(p, it, segs, ntiles, base, tmem, abort);
  } else if (warp == 4) {
    if ((threadIdx.x & 31) == 0) mma_issuer(p, ntiles, base, tmem, abort);
    __syncwarp();
  } else {
    producer(p, it, segs, ntiles, base, sp, abort);
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 4) {
    tc::fence_after();
    tc::dealloc(tmem, kTmemCols);
  }
}

}  // namespace

int launch_extend(const rx_kv_desc* d, const PlanHeader* h, const void* k_pool,
                  const void* v_pool, const void* q, void* o, float* lse, void* ws,
                  void* stream) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(extend_tc_kernel,
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
    extend_tc_kernel<<<h->n_items, kThreads, kSmem, (cudaStream_t)stream>>>(p);
  return (int)cudaGetLastError();
}

}  // namespace rx
