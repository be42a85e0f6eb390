// rx_extend_attn on a pair of SMs: attention of new tokens over their cached prefix plus causal
// self-attention, the tensor-core work of each item shared by two CTAs (a cluster of two,
// tcgen05 .cta_group::2).
//
// Only the unmatched tokens of a request are computed (SGLang explainer, prefix matching); their
// queries attend to the cached prefix KV and, causally, to the new tokens' KV (already stored in
// the pool).  When several requests share a cached prefix, their new rows are packed into the same
// tiles, so the prefix KV is read and multiplied once per tile pair for all of them -- the
// prefill-side counterpart of the shared-prefix reading in BatchLLM's horizontal fusion.  A work
// item is two 128-row tiles of one KV head that walk one list of key segments: the shared prefix
// (visible to every row), then each member's own keys (visible to that member's rows only, causal
// on its new tokens).  One online softmax per row runs across all segments.
//
// The pair: tile A lives on the even CTA (rank 0), tile B on the odd one.  Every MMA has M = 256
// (both tiles) and N = 128, issued by one thread of the even CTA; each CTA keeps its own 128 query
// rows in its shared memory and supplies half of each B operand, so per SM the operand traffic
// and the gathered bytes per multiply are half those of one CTA running both tiles:
//   S = Q K^T over a step of 128 keys: each CTA gathers 64 of the keys (its half of N);
//   O += P V: each CTA gathers the step's 128 V rows restricted to its 64 columns of d (its half
//   of N; a 128-byte half row is the unit of the TMA gather), and P comes from tensor memory.
// Each CTA receives its 128 rows of S and O in its own tensor memory.
//
// Roles per CTA (512 threads):
//   warps 0-7    softmax, two warpgroups that take the steps in turn (warpgroup t % 2 takes
//                step t), a full row per thread (row r, tensor-memory lane r): the exponential
//                unit, 16 results per clock per SM, needs as long for a step as the tensor core,
//                and with the steps alternating one warpgroup's loads, maxima and stores run
//                while the other's exponentials do.  Per step: load the row's 128 scores, mask,
//                take the running max of the previous step from the other warpgroup (shared
//                memory), move it only when the row's max exceeds it by more than 2^8 (then O is
//                rescaled), hand it on, write P = 2^(s - m) as bf16 over the upper half of the S
//                buffer.  Each warpgroup keeps its own sum; at the end they merge (O, LSE).
//                exp2_poly2 can take part of the exponentials onto the FMA pipe (kPolyPairs).
//   warps 8-10   K producers (steps t = 0, 1, 2 mod 3), warps 11-13 V producers: gather rows by
//                slot with TMA tile::gather4 (four pool rows of 64 columns per instruction, 128-
//                byte swizzle by the copy engine) into 5-stage rings; a stage lands on the CTA's
//                own barrier (bytes counted).  The V warp that takes an item's first ring step
//                first copies the item's query rows in (cp.async), once the previous item's
//                copy is done and its last S MMA has read the old rows.
//   warp 14      even CTA: the MMA issuer (one thread); odd CTA: the relay, which forwards each
//                of its landed stages to the even CTA's barrier for the peer half.
//   warp 15      tensor-memory allocation for the pair (one warp in each CTA); in the even CTA
//                also the issuer's gate: it takes every barrier wait of the issuer, in order, and
//                publishes its progress in shared memory, since a barrier operation after a
//                commit holds the issuing thread until the tensor pipe has taken the MMAs before
//                it (measured: 40-75 ns per wait, most of a step's slack).
// With three S buffers the issuer keeps S up to three steps ahead of PV: per step t it issues
// O += P(t) V(t), then S(t+3) into the buffer P(t) sat in (one thread's MMAs execute in order).  Its commits arrive on the barriers of
// both CTAs at once (multicast).  Steps, S steps, P steps and items are running counts across
// the CTA's items, so the pipelines never drain between items.
// Every mbarrier wait is bounded (globaltimer); a timeout records RX_ERR_TIMEOUT in the workspace
// status word and every role leaves its loop; before the pair exits, the issuer waits for its
// MMAs and every producer for its copies still in flight.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include <atomic>

#include "pair.cuh"
#include "ptx.cuh"
#include "rx_internal.h"
#include "tc.cuh"

namespace rx {
namespace {

struct PairParams {
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
  int32_t oob_row;  // a row index past the end of the pool's [pool_size * Hkv, 128] view
  int n_items;
  bool o32;         // o is 32-byte aligned: rows go out in 32-byte stores, else 16-byte ones
};

constexpr int kN = kPairKeys;          // keys per step (128): the MMAs' N for S and K for PV
constexpr int kPW = 3;                 // producer warps per operand
constexpr int kWarpK = 8, kWarpV = kWarpK + kPW, kWarpMma = kWarpV + kPW, kWarpAlloc = kWarpMma + 1;
constexpr int kThreads = 512;
static_assert(kWarpAlloc == 15, "sixteen warps: two softmax warpgroups, two others");
constexpr int kRegsLaunch = 65536 / kThreads;  // 128
constexpr int kRegsSoftmax = 200, kRegsOther = 56;
static_assert(kRegsSoftmax * 256 + kRegsOther * 256 <= kRegsLaunch * kThreads, "register split");
constexpr int kStages = 4;  // (with two Q buffers, five stages would not fit in shared memory)
static_assert(kStages >= kPW, "a producer could run two phases ahead");
constexpr int kQHalf = 128 * 128;      // 64 columns of the 128 query rows: 16 KiB
constexpr int kQTile = 2 * kQHalf;
constexpr int kKHalf = 64 * 128;       // 64 columns of the CTA's 64 keys of a step: 8 KiB
constexpr int kKTile = 2 * kKHalf;     // 16 KiB
constexpr int kVTile = kN * 128;       // the CTA's 64 columns of the step's 128 V rows: 16 KiB
constexpr int kOffQ = 0;               // two Q buffers: item i uses buffer i % 2
constexpr int kOffK = 2 * kQTile;
constexpr int kOffV = kOffK + kStages * kKTile;
constexpr int kOffBar = kOffV + kStages * kVTile;
// Barriers, at the same offsets in both CTAs (each waiter is at most one phase behind):
//   KL[s] / VL[s]  this CTA's gathers for ring stage s landed (its producer's expect_tx + bytes)
//   KP[s] / VP[s]  even CTA only: the odd CTA's half of stage s landed (the relay's arrival)
//   KF[s] / VF[s]  stage s free: the MMAs that read it completed (multicast commit)
//   SF[b]          S(t) in S buffer b = t % 3 complete (phase t / 3; multicast commit issued after
//                  PV(t-3) and S(t), so the phase of step t+2 also tells that PV(t-1) is complete)
//   PF[b]          even CTA only: P(t) of both CTAs in buffer b = t % 3 (one arrival per warp of
//                  step t's softmax warpgroup, either CTA; one barrier per buffer, since the
//                  softmax may run up to two steps ahead of the issuer)
//   QF[q]          the CTA's query rows of an item are in Q buffer q (the Q loader; phase = the
//                  buffer's uses)
//   QP[q]          even CTA only: the odd CTA's query rows in buffer q landed (the relay)
//   QE[q]          every S MMA of the item in buffer q complete: the buffer may take the rows of
//                  the item after next (multicast commit after the item's last S).  One barrier
//                  per buffer, so that a loader that runs late never tests a phase two ahead
//   OD             every MMA of the item complete: O is final (multicast commit)
//   DR             even CTA only: every MMA complete, at the end (tensor memory may be released)
//   ML[i]          the CTA's two softmax warpgroups have stored their (max, sum) of the row for
//                  the item's merge (all 256 softmax threads; i = item parity)
//   MR[b]          the running max of a step of parity b is in shared memory (the 128 threads of
//                  the warpgroup that took the step)
enum {
  B_KL = 0,
  B_VL = B_KL + kStages,
  B_KP = B_VL + kStages,
  B_VP = B_KP + kStages,
  B_KF = B_VP + kStages,
  B_VF = B_KF + kStages,
  B_SF = B_VF + kStages,  // + b
  B_PF = B_SF + 3,        // + b
  B_QF = B_PF + 3,        // + Q buffer
  B_QP = B_QF + 2,        // + Q buffer
  B_QE = B_QP + 2,        // + Q buffer
  B_OD = B_QE + 2,
  B_DR = B_OD + 1,
  B_ML = B_DR + 1,        // + item parity
  B_MR = B_ML + 2,        // + step parity
  B_COUNT = B_MR + 2
};
constexpr int kOffFilled = kOffBar + B_COUNT * 8;  // int32 [2][kStages] + 1: fills issued per
                                                    // stage, then the Q loads issued
constexpr int kOffML = kOffFilled + (2 * kStages + 2) * 4;  // float2 [2 items][2 wgs][128 rows]
constexpr int kOffM = kOffML + 2 * 2 * 128 * 8;     // float [2 step parities][128 rows]
constexpr int kOffGate = kOffM + 2 * 128 * 4;       // uint32: the issuer's wait points passed
constexpr int kOffTmem = kOffGate + 8;
constexpr int kOffAbort = kOffTmem + 8;
constexpr size_t kSmem = 1024 + kOffAbort + 16;
static_assert(kSmem <= 227 * 1024, "shared memory budget");
// Tensor memory per CTA: three S buffers [0, 128), [128, 256), [256, 384) (P(t), 128 bf16 a row,
// two a column, over the upper half of S buffer t % 3), O [384, 512).  Three buffers let S run
// two steps ahead of the softmax: a step's hand-offs across the pair (commit, softmax, P arrival,
// gate, issue) take longer than one step of MMAs, and each buffer is a chain that overlaps the
// others.
constexpr int kSBuf = 3;  // (the P-full arrival in softmax_steps selects among three)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 384;
constexpr uint32_t kPOff = 64;
constexpr uint64_t kWaitNs = 2000000000ull;
__host__ __device__ constexpr uint32_t col_s_of(int b) { return (uint32_t)b * kN; }
constexpr uint16_t kBoth = 0x3;

// 2^x on the FMA pipe for a pair of values x <= 8 (-inf and anything below -127 give 0): with
// n = round(x) and f = x - n in [-1/2, 1/2], 2^x = p(f) * 2^n, p the minimax cubic for 2^f in
// relative error (Remez; coefficients from fit_exp2.py, relative error <= 7.5e-5) and 2^n built
// from its exponent bits (n = -127 gives the bits of 0.0).
constexpr float kExpC0 = 0.9999280571937561f;
constexpr float kExpC1 = 0.6932609677314758f;
constexpr float kExpC2 = 0.2426111251115799f;
constexpr float kExpC3 = 0.0551716685295105f;
__device__ __forceinline__ uint64_t exp2_poly2(float x0, float x1) {
  constexpr float kRound = 12582912.0f;  // 1.5 * 2^23: x + kRound holds round(x) in its low bits
  x0 = fmaxf(x0, -127.f);
  x1 = fmaxf(x1, -127.f);
  const uint64_t x = f2_pack(x0, x1);
  const uint64_t t = f2_add(x, f2_pack(kRound, kRound));
  const uint64_t nf = f2_add(t, f2_pack(-kRound, -kRound));
  const uint64_t f = f2_fma(nf, f2_pack(-1.f, -1.f), x);
  uint64_t p = f2_fma(f, f2_pack(kExpC3, kExpC3), f2_pack(kExpC2, kExpC2));
  p = f2_fma(p, f, f2_pack(kExpC1, kExpC1));
  p = f2_fma(p, f, f2_pack(kExpC0, kExpC0));
  float t0, t1;
  f2_unpack(t, t0, t1);
  // exponent bits of 2^n: (n + 127) << 23, n = bits(t) - bits(kRound)
  const uint32_t e0 = (__float_as_uint(t0) - 0x4B400000u + 127u) << 23;
  const uint32_t e1 = (__float_as_uint(t1) - 0x4B400000u + 127u) << 23;
  return f2_mul(p, f2_pack(__uint_as_float(e0), __uint_as_float(e1)));
}

struct TileIter {
  int seg, k0;
};
__device__ __forceinline__ void tile_next(TileIter& c, const ExtSeg* segs, int n_seg) {
  if (c.seg >= n_seg) return;
  c.k0 += kN;
  if (c.k0 >= segs[c.seg].k_end) {
    ++c.seg;
    if (c.seg < n_seg) c.k0 = segs[c.seg].k_begin;
  }
}

// The cluster's r-th item: the plan's list is dealt to the clusters in snake order (round r holds
// items r C .. r C + C - 1; cluster k takes the k-th of an even round and the (C - 1 - k)-th of an
// odd one).  Both CTAs of a cluster see the same sequence.  -1 past the end.
__device__ __forceinline__ int item_at(int r, int n_items) {
  const int C = gridDim.x >> 1, k = blockIdx.x >> 1;
  const int64_t i = (int64_t)r * C + ((r & 1) ? C - 1 - k : k);
  return i < n_items ? (int)i : -1;
}

// Byte offset of 16-byte chunk c (0..15) of row r in a K-major tile stored as two 128-byte-
// swizzled halves (d 0..63, d 64..127) of `half` bytes each.
__device__ __forceinline__ uint32_t tile_off(int r, int c, int half) {
  return (uint32_t)((c >> 3) * half + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ int fetch_slot(const PairParams& p, const ExtSeg& sg, int k0, int key) {
  const int kpos = k0 + key;
  return kpos < sg.k_end ? __ldg(p.req_to_token + (int64_t)sg.kv_row * p.stride + kpos) : -1;
}

__device__ __forceinline__ int check_slot(const PairParams& p, int s) {
  if (s >= p.pool_size || s < -1) {
    atomicCAS(p.status, 0, (int)RX_ERR_RANGE);
    return -1;
  }
  return s;
}

__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, int col, int r0,
                                            int r1, int r2, int r3, uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(map), "r"(col), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(mbar)
      : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t mbar, uint32_t bytes) {
  asm volatile("{\n.reg .b64 st;\nmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}\n" ::"r"(
                   mbar),
               "r"(bytes)
               : "memory");
}

struct Slot4 {
  int v[4];
};

// The CTA's query rows of item `it` (the nq-th with steps), copied by one warp into Q buffer
// nq % 2 (tile_off layout: two 64-column halves, 128-byte swizzle; rows past the tile's as zeros)
// with cp.async once every S MMA of item nq - 2, the buffer's previous user, has completed
// (QE[nq % 2]), so the rows land while item nq - 1 still runs; then the warp makes its writes
// visible to the tensor core (proxy fence) and lane 0 arrives on QF[nq % 2].  Lane l copies tile rows
// l, l + 32, l + 64, l + 96.  (A TMA copy would queue behind the ring's prefetched gathers:
// measured 5 us from the item's last S to its rows landing.)  Returns false when a wait gave up.
__device__ __forceinline__ bool load_q_rows(const PairParams& p, const ExtItem& it, uint32_t rank,
                                            uint32_t base, uint32_t nq, volatile int* filled_q,
                                            volatile int* abort) {
  const int lane = threadIdx.x & 31;
  const uint32_t q = nq & 1;
  const uint32_t bar = base + kOffBar, qb = base + kOffQ + q * kQTile;
  // Another V warp copies the previous item's rows and may still be waiting for its own turn:
  // this warp runs up to a ring ahead of the issuer, and testing QE[q]'s parity before the copy
  // of item nq - 2 has passed its previous phase would pass on that earlier phase.
  bool ok = true;
  if (nq > 0) {
    const uint64_t t0 = pair::globaltimer();
    while (*filled_q < (int)nq) {
      if (*abort) { ok = false; break; }
      if (pair::globaltimer() - t0 > kWaitNs) {
        *abort = 1;
        atomicCAS(p.status, 0, 5 /* RX_ERR_TIMEOUT */);
        ok = false;
        break;
      }
      __nanosleep(64);
    }
    if (nq > 1)
      ok = ok && pair::wait(bar + 8 * (B_QE + q), ((nq - 2) >> 1) & 1, abort, p.status, kWaitNs);
  }
  if (__any_sync(0xffffffffu, !ok)) return false;
  const int n_tok = rank ? it.n_tok[1] : it.n_tok[0];
  const int row_begin = rank ? it.row_begin[1] : it.row_begin[0];
#pragma unroll 1
  for (int tr = lane; tr < 128; tr += 32) {
    const bool valid = tr < n_tok * p.gq;
    const __nv_bfloat16* src =
        valid ? p.q + ((int64_t)__ldg(&p.rows[row_begin + tr / p.gq].q_row) * p.hq +
                       it.kv_head * p.gq + tr % p.gq) * kHeadDim
              : p.q;
#pragma unroll
    for (int c = 0; c < 16; ++c)
      cp_async16(qb + tile_off(tr, c, kQHalf), src + (valid ? c * 8 : 0), valid);
  }
  cp_async_commit();
  cp_async_wait<0>();
  tc::fence_proxy_async();
  __syncwarp();
  if (lane == 0) {
    tc::mbar_arrive(bar + 8 * (B_QF + q));
    *filled_q = (int)nq + 1;
  }
  return true;
}

// Producer warp w of one operand: ring steps w, w + kPW, ... counted over all the cluster's items.
// K: lane j gathers keys 64 rank + 4 (j % 16) .. + 3 of the step, column half j / 16 (both halves
// of the CTA's 64 keys: 16 KiB).  V: lane j gathers keys 4 j .. 4 j + 3 of the step, the CTA's
// column half (16 KiB).  Table entries are fetched one step of the warp's own ahead; keys past the
// segment (or flagged entries) read a row past the end of the map, which the TMA fills with
// zeros.  Each fill of stage s is recorded in filled[s] so that the CTA can wait for its last
// copies before it exits.  The V producer warp that takes an item's first ring step first copies
// the item's query rows in (load_q_rows).
__device__ __forceinline__ void producer(const PairParams& p, int w, bool is_k, uint32_t rank,
                                         uint32_t base, const CUtensorMap* map,
                                         volatile int* filled, volatile int* abort) {
  const int lane = threadIdx.x & 31;
  const int key0 = is_k ? 64 * (int)rank + 4 * (lane & 15) : 4 * lane;
  const int col = is_k ? 64 * (lane >> 4) : 64 * (int)rank;
  const uint32_t ring = base + (is_k ? kOffK : kOffV);
  const uint32_t dst_lane = is_k ? (uint32_t)((lane >> 4) * kKHalf + (lane & 15) * 512)
                                 : (uint32_t)(lane * 512);
  const uint32_t tile_bytes = is_k ? kKTile : kVTile;
  const uint32_t bar = base + kOffBar;
  const int b_l = is_k ? B_KL : B_VL, b_f = is_k ? B_KF : B_VF;
  uint32_t gs = 0, nq = 0;
  for (int ri = 0;; ++ri) {
    const int idx = item_at(ri, p.n_items);
    if (idx < 0) return;
    const ExtItem it = p.items[idx];
    const ExtSeg* segs = p.segs + it.seg_begin;
    const int ntiles = it.n_steps;
    TileIter at{0, ntiles > 0 ? segs[0].k_begin : 0};
    int at_step = 0;
    auto fetch = [&](Slot4& sl, int t) {
      for (; at_step < t; ++at_step) tile_next(at, segs, it.n_seg);
      const ExtSeg& sg = segs[at.seg];
#pragma unroll
      for (int i = 0; i < 4; ++i) sl.v[i] = fetch_slot(p, sg, at.k0, key0 + i);
    };
    const int t0 = (int)((w + kPW - gs % kPW) % kPW);
    if (!is_k && ntiles > 0 && t0 == 0 &&
        !load_q_rows(p, it, rank, base, nq, filled + kStages, abort))
      return;
    if (ntiles > 0) ++nq;
    Slot4 nxt{{-1, -1, -1, -1}};
    if (t0 < ntiles) fetch(nxt, t0);
    for (int t = t0; t < ntiles; t += kPW) {
      const Slot4 cur = nxt;
      if (t + kPW < ntiles) fetch(nxt, t + kPW);
      const uint32_t gt = gs + t;
      const int st = gt % kStages;
      const bool waited = gt < kStages || pair::wait(bar + 8 * (b_f + st), (gt / kStages - 1) & 1,
                                                     abort, p.status, kWaitNs);
      if (__any_sync(0xffffffffu, !waited)) return;
      int r[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int v = check_slot(p, cur.v[i]);
        r[i] = v >= 0 ? v * p.hkv + it.kv_head : p.oob_row;
      }
      if (lane == 0) {
        mbar_expect_tx(bar + 8 * (b_l + st), tile_bytes);
        filled[st] = (int)(gt / kStages) + 1;
      }
      __syncwarp();
      tma_gather4(ring + st * tile_bytes + dst_lane, map, col, r[0], r[1], r[2], r[3],
                  bar + 8 * (b_l + st));
    }
    gs += ntiles;
  }
}

// Even CTA, one thread: the issuer's wait points, in its order -- per item: both CTAs' query rows
// (QF); K of steps 0, 1 and 2 landed in both CTAs; then per step t: K(t+3) (when there is such a
// step) and V(t) landed and both CTAs' P(t) in tensor memory.  Each point passed is published in
// the gate counter, so the issuer itself never tests a barrier between its commits.
__device__ __forceinline__ void gate_role(const PairParams& p, uint32_t base,
                                          volatile int* abort) {
  const uint32_t bar = base + kOffBar, gate = base + kOffGate;
  bool ok = true;
  auto wait = [&](int b, uint32_t parity) {
    ok = ok && pair::wait(bar + 8 * b, parity, abort, p.status, kWaitNs);
    return ok;
  };
  auto landed = [&](int b_l, int b_p, uint32_t gt) {  // both CTAs' halves of ring step gt
    const int st = gt % kStages;
    const uint32_t ph = (gt / kStages) & 1;
    return wait(b_l + st, ph) && wait(b_p + st, ph);
  };
  uint32_t passed = 0, gs = 0, pb = 0, nq = 0;
  for (int ri = 0; ok; ++ri) {
    const int idx = item_at(ri, p.n_items);
    if (idx < 0) return;
    const int ntiles = p.items[idx].n_steps;
    if (ntiles == 0) continue;
    // both CTAs' query rows, in Q buffer nq % 2
    if (!wait(B_QF + (nq & 1), (nq >> 1) & 1) || !wait(B_QP + (nq & 1), (nq >> 1) & 1)) return;
    pair::st_release(gate, ++passed);
    for (int t = 0; t < kSBuf && t < ntiles; ++t) {
      if (!landed(B_KL, B_KP, gs + t)) return;
      pair::st_release(gate, ++passed);
    }
    for (int t = 0; t < ntiles; ++t) {
      const uint32_t gt = gs + t;
      if ((t + kSBuf < ntiles && !landed(B_KL, B_KP, gt + kSBuf)) || !landed(B_VL, B_VP, gt) ||
          !wait(B_PF + (pb + t) % kSBuf, ((pb + t) / kSBuf) & 1))
        return;
      pair::st_release(gate, ++passed);
    }
    gs += ntiles;
    pb += ntiles;
    ++nq;
  }
}

// Even CTA, one thread: per item S(0), S(1) and S(2); then per step t, once both CTAs' P(t) are
// in tensor memory, O += P(t) V(t) and S(t+3) right behind it (into the buffer P(t) sat in).  A ring
// stage is used once this CTA's gathers and the odd CTA's (forwarded by its relay) have landed.
// The MMAs of a step are issued back to back and their commits follow them.  The waits are the
// gate thread's: the issuer only reads its counter (bounded, like every wait).
__device__ __forceinline__ void mma_issuer(const PairParams& p, uint32_t base, uint32_t tmem,
                                           volatile int* abort) {
  constexpr uint32_t idS = tc::idesc_bf16(256, kN, false, false);
  constexpr uint32_t idO = tc::idesc_bf16(256, 128, false, true);
  const uint32_t bar = base + kOffBar, gate = base + kOffGate;
  const uint64_t qdesc0 = tc::desc_sw128(base + kOffQ, 16, 1024);
  const uint64_t kdesc0 = tc::desc_sw128(base + kOffK, 16, 1024);
  const uint64_t vdesc0 = tc::desc_sw128(base + kOffV, kVTile, 1024);
  const uint32_t d_o = tmem + kColO;
  bool ok = true;
  uint32_t gi = 0;
  auto pass = [&]() {  // the gate thread has passed the issuer's next wait point
    ++gi;
    if (pair::ld_acquire(gate) >= gi) return ok;
    const uint64_t t0 = pair::globaltimer();
    while (pair::ld_acquire(gate) < gi) {
      if (*abort) return ok = false;
      if (pair::globaltimer() - t0 > kWaitNs) {
        *abort = 1;
        atomicCAS(p.status, 0, (int)RX_ERR_TIMEOUT);
        return ok = false;
      }
    }
    return ok;
  };
  uint32_t gs = 0, sv = 0, pb = 0, nq = 0;
  for (int ri = 0; ok; ++ri) {
    const int idx = item_at(ri, p.n_items);
    if (idx < 0) break;
    const int ntiles = p.items[idx].n_steps;
    if (ntiles == 0) continue;  // (plans hold none; every role skips them alike)
    const uint64_t qdesc = qdesc0 + (((nq & 1) * kQTile) >> 4);  // the item's Q buffer
    auto qk = [&](int t) {  // S(t) = Q K(t)^T into buffer (sv + t) % 3
      const uint64_t kd = kdesc0 + ((((gs + t) % kStages) * kKTile) >> 4);
      const uint32_t d_s = tmem + col_s_of((sv + t) % kSBuf);
#pragma unroll
      for (int s = 0; s < 8; ++s)
        pair::mma_ss(d_s, qdesc + (((s >> 2) * kQHalf + (s & 3) * 32) >> 4),
                     kd + (((s >> 2) * kKHalf + (s & 3) * 32) >> 4), idS, s > 0 ? 1u : 0u);
    };
    auto pv = [&](int t) {  // O += P(t) V(t)
      const uint64_t vd = vdesc0 + ((((gs + t) % kStages) * kVTile) >> 4);
      const uint32_t a_p = tmem + col_s_of((sv + t) % kSBuf) + kPOff;
#pragma unroll
      for (int s = 0; s < kN / 16; ++s)
        pair::mma_ts(d_o, a_p + 8 * s, vd + ((s * 2048) >> 4), idO, (t > 0 || s > 0) ? 1u : 0u);
    };
    if (!pass()) break;
    for (int t = 0; t < kSBuf; ++t) {
      if (t < ntiles) {
        if (!pass()) break;
        tc::fence_after();
        qk(t);
        pair::commit_mc(bar + 8 * (B_SF + (sv + t) % kSBuf), kBoth);
        pair::commit_mc(bar + 8 * (B_KF + (gs + t) % kStages), kBoth);
        if (t == ntiles - 1) pair::commit_mc(bar + 8 * (B_QE + (nq & 1)), kBoth);  // last S
      } else {
        pair::commit_mc(bar + 8 * (B_SF + (sv + t) % kSBuf), kBoth);  // step without an MMA
      }
    }
    for (int t = 0; ok && t < ntiles; ++t) {
      const uint32_t gt = gs + t, gt3 = gt + kSBuf;
      const bool more = t + kSBuf < ntiles;
      if (!pass()) break;
      tc::fence_after();
      pv(t);
      if (more) qk(t + kSBuf);
      pair::commit_mc(bar + 8 * (B_VF + gt % kStages), kBoth);
      pair::commit_mc(bar + 8 * (B_SF + (sv + t) % kSBuf), kBoth);  // also after the last steps
      if (more) pair::commit_mc(bar + 8 * (B_KF + gt3 % kStages), kBoth);
      if (more && t + kSBuf == ntiles - 1) pair::commit_mc(bar + 8 * (B_QE + (nq & 1)), kBoth);
    }
    if (!ok) break;
    pair::commit_mc(bar + 8 * B_OD, kBoth);
    gs += ntiles;
    sv += ntiles + kSBuf;
    pb += ntiles;
    ++nq;
  }
  // every MMA issued above completes before tensor memory is released, after an abort too
  pair::commit_mc(bar + 8 * B_DR, 0x1);
  int no_abort = 0;
  pair::wait(bar + 8 * B_DR, 0, &no_abort, p.status, kWaitNs);
}

// Odd CTA, one thread: forwards each landed stage of this CTA to the even CTA's peer barriers, in
// the order the issuer uses them (per item: Q, K(0), K(1), K(2), then per step K(t + 3), V(t)).
__device__ __forceinline__ void relay(const PairParams& p, uint32_t base, volatile int* abort) {
  const uint32_t bar = base + kOffBar;
  uint32_t gs = 0, nq = 0;
  bool ok = true;
  auto fwd = [&](int b_l, int b_p, uint32_t gt) {
    const int st = gt % kStages;
    ok = ok && pair::wait(bar + 8 * (b_l + st), (gt / kStages) & 1, abort, p.status, kWaitNs);
    if (ok) pair::arrive_remote(pair::map_to(bar + 8 * (b_p + st), 0));
    return ok;
  };
  for (int ri = 0; ok; ++ri) {
    const int idx = item_at(ri, p.n_items);
    if (idx < 0) return;
    const int ntiles = p.items[idx].n_steps;
    if (ntiles == 0) continue;
    // the item's query rows first: the issuer waits for them before its first S
    ok = ok && pair::wait(bar + 8 * (B_QF + (nq & 1)), (nq >> 1) & 1, abort, p.status, kWaitNs);
    if (!ok) return;
    pair::arrive_remote(pair::map_to(bar + 8 * (B_QP + (nq & 1)), 0));
    ++nq;
    for (int t = 0; t < kSBuf && t < ntiles; ++t)
      if (!fwd(B_KL, B_KP, gs + t)) return;
    for (int t = 0; t < ntiles; ++t) {
      if (t + kSBuf < ntiles && !fwd(B_KL, B_KP, gs + t + kSBuf)) return;
      if (!fwd(B_VL, B_VP, gs + t)) return;
    }
    gs += ntiles;
  }
}

// Maximum of a row's 128 raw scores (three-input maxima, eight independent chains).
__device__ __forceinline__ float row_max(const uint32_t (&sr)[4][32]) {
  float m[8];
#pragma unroll
  for (int a = 0; a < 8; ++a) m[a] = __uint_as_float(sr[0][a]);
#pragma unroll
  for (int q = 0; q < 4; ++q)
#pragma unroll
    for (int j = 0; j < 32; j += 2)
      if (q > 0 || j >= 8)
        m[(j >> 1) & 7] =
            fmax3(m[(j >> 1) & 7], __uint_as_float(sr[q][j]), __uint_as_float(sr[q][j + 1]));
#pragma unroll
  for (int a = 0; a < 2; ++a) m[a] = fmax3(m[a], m[a + 2], m[a + 4]);
  return fmax3(m[0], m[1], fmaxf(m[6], m[7]));
}

// Of every 8 pairs of a row's scores, the first kPolyPairs take the FMA-pipe exponential and the
// rest the exponential unit, which alone would be as busy as the tensor core.
constexpr int kPolyPairs = 0;

// Chunk q (32 scores) of the row: s -> p = 2^(s scale_log2 - m) (a masked key's -inf gives 0),
// packed to bf16 pairs in pk[16 q ..], added into acc (packed partial sums).
__device__ __forceinline__ void row_chunk(const uint32_t (&c)[32], uint32_t* pk, float sl2,
                                          float m, uint64_t& acc) {
  const uint64_t k2 = f2_pack(sl2, sl2), nm2 = f2_pack(-m, -m);
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    const uint64_t x = f2_fma(f2_pack(__uint_as_float(c[j]), __uint_as_float(c[j + 1])), k2, nm2);
    float x0, x1, p0, p1;
    f2_unpack(x, x0, x1);
    if (((j >> 1) & 7) < kPolyPairs) {
      f2_unpack(exp2_poly2(x0, x1), p0, p1);
    } else {
      p0 = fast_exp2(x0);
      p1 = fast_exp2(x1);
    }
    acc = f2_add(acc, f2_pack(p0, p1));
    pk[j >> 1] = pack_bf16(p0, p1);
  }
}

__device__ __forceinline__ void st_global_v8(void* dst, const uint32_t* w) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(w[0]),
               "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

struct RowQ {
  int owner, kmax, q_row, qh;
  bool valid;
};

__device__ __forceinline__ RowQ row_of(const PairParams& p, const ExtItem& it, int x, int r) {
  RowQ q{-2, 0, 0, it.kv_head * p.gq + (r % p.gq), false};
  if (r < (x ? it.n_tok[1] : it.n_tok[0]) * p.gq) {
    const ExtRow e = p.rows[(x ? it.row_begin[1] : it.row_begin[0]) + r / p.gq];
    q.owner = e.owner;
    q.kmax = e.kmax;
    q.q_row = e.q_row;
    q.valid = true;
  }
  return q;
}

// Running counts over the CTA's earlier items: S steps (ntiles + kSBuf per item), P steps (= ring
// steps), items, and the phases of MR[0] / MR[1] (one per step of that parity).
struct SmCounts {
  uint32_t sv, pb, nq;
  uint32_t mr[2];
};

// Warpgroup w of the softmax over one item: the steps t = w (mod 2), a full row per thread.  The
// running max is one chain across both warpgroups: step t takes m(t-1) from the other warpgroup
// through shared memory (MR[(t-1) % 2]), sets m(t) (moved only when the row's scaled maximum
// exceeds it by more than 2^8) and hands it on before its exponentials.  O is one accumulator:
// when m moves at step t, the warpgroup of step t rescales O (after PV(t-1), before PV(t)).  Each
// warpgroup keeps its own sum l_w relative to the max of its last step.  ahead() looks up the
// next item's row.  Returns false when a wait gave up.
template <class Ahead>
__device__ __forceinline__ bool softmax_steps(const PairParams& p, const ExtItem& it,
                                              const ExtSeg* segs, int ntiles, const RowQ& row,
                                              int w, int r, SmCounts& c, uint32_t bar,
                                              const uint32_t (&pf_c)[kSBuf], uint32_t lane_t,
                                              float* m_buf, volatile int* abort, float& m_w,
                                              float& l_w, Ahead&& ahead) {
  const float sl2 = p.scale_log2;
  const bool any_valid = __any_sync(0xffffffffu, row.valid);
  int seg = 0, k0 = segs[0].k_begin, k_end = segs[0].k_end, s_owner = segs[0].owner;
  ExtSeg nsg = segs[it.n_seg > 1 ? 1 : 0];
  ahead();
  for (int t = 0; t < ntiles; ++t) {
    const int b = t & 1;
    if (b == w) {
      const uint32_t vs = c.sv + t;
      const uint32_t col_s = col_s_of(vs % kSBuf);
      const bool w_ok = pair::wait(bar + 8 * (B_SF + vs % kSBuf), (vs / kSBuf) & 1, abort,
                                   p.status, kWaitNs);
      if (__any_sync(0xffffffffu, !w_ok)) return false;
      tc::fence_after();
      // the max of step t-1 (always waited for, so that the hand-off's phases stay in step)
      float m_prev = -CUDART_INF_F;
      if (t > 0) {
        const bool w2 = tc::mbar_wait(bar + 8 * (B_MR + (1 - b)), (c.mr[1 - b] - 1) & 1, abort,
                                      p.status, kWaitNs);
        if (__any_sync(0xffffffffu, !w2)) return false;
        m_prev = m_buf[(1 - b) * 128 + r];
      }
      uint32_t pk[64];
      float m_t = m_prev;
      if (any_valid) {
        const bool vis = row.valid && (s_owner < 0 || s_owner == row.owner);
        const int lim = vis ? min(row.kmax, k_end) : 0;  // keys at positions >= lim are masked
        const int n_ok = max(0, min(kN, lim - k0));
        uint32_t sr[4][32];
#pragma unroll
        for (int q = 0; q < 4; ++q) tc::ld32(lane_t + col_s + 32 * q, sr[q]);
        tc::wait_ld();
        if (n_ok < kN) {  // keys at n_ok and beyond are masked: -inf
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (32 * q + j >= n_ok) sr[q][j] = 0xff800000u;
        }
        const float cand = n_ok > 0 ? row_max(sr) * sl2 : -CUDART_INF_F;
        if (cand > m_prev + 8.f) m_t = cand;
        m_buf[b * 128 + r] = m_t;  // hand m(t) on before the exponentials
        tc::mbar_arrive(bar + 8 * (B_MR + b));
        const bool bump = m_t > m_prev && m_prev != -CUDART_INF_F;  // O holds something to scale
        const bool rescale = __any_sync(0xffffffffu, bump) && t > 0;
        // a row that has seen no visible key yet has m = -inf and only masked keys: any finite
        // reference gives p = 0 for them
        const float mref = m_t == -CUDART_INF_F ? 0.f : m_t;
        uint64_t acc = 0ull;
#pragma unroll
        for (int q = 0; q < 4; ++q) row_chunk(sr[q], pk + 16 * q, sl2, mref, acc);
        {
          float a0, a1;
          f2_unpack(acc, a0, a1);
          const float lw_scale = (m_w == -CUDART_INF_F) ? 0.f : fast_exp2(m_w - mref);
          l_w = l_w * lw_scale + (a0 + a1);
          if (m_t != -CUDART_INF_F) m_w = m_t;
        }
        if (rescale) {
          // O must hold PV(t-1): the phase of S step t+2 covers it, and PV(t) waits for this P
          const uint32_t vn = vs + kSBuf - 1;
          const bool w3 = pair::wait(bar + 8 * (B_SF + vn % kSBuf), (vn / kSBuf) & 1, abort,
                                     p.status, kWaitNs);
          if (__any_sync(0xffffffffu, !w3)) return false;
          tc::fence_after();
          const float alpha = bump ? fast_exp2(m_prev - m_t) : 1.f;
#pragma unroll 1
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t ov[32];
            tc::ld32(lane_t + kColO + 32 * q4, ov);
            tc::wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * alpha);
            tc::st32(lane_t + kColO + 32 * q4, ov);
          }
        }
      } else {  // the CTA's tile has no rows in this item: P = 0 (its keys still feed the other's)
        m_buf[b * 128 + r] = m_t;
        tc::mbar_arrive(bar + 8 * (B_MR + b));
#pragma unroll
        for (int j = 0; j < 64; ++j) pk[j] = 0u;
      }
      ++c.mr[b];
      tc::st32(lane_t + col_s + kPOff, *reinterpret_cast<const uint32_t(*)[32]>(pk));
      tc::st32(lane_t + col_s + kPOff + 32, *reinterpret_cast<const uint32_t(*)[32]>(pk + 32));
      tc::wait_st();
      tc::fence_before();
      __syncwarp();
      if ((threadIdx.x & 31) == 0) {
        const uint32_t bb = (c.pb + t) % kSBuf;  // (selects: an indexed array sits on the stack)
        pair::arrive_remote(bb == 0 ? pf_c[0] : (bb == 1 ? pf_c[1] : pf_c[2]));
      }
    } else {
      ++c.mr[b];  // the other warpgroup's step: one phase of MR[b]
    }
    k0 += kN;
    if (k0 >= k_end && ++seg < it.n_seg) {
      k0 = nsg.k_begin;
      k_end = nsg.k_end;
      s_owner = nsg.owner;
      if (seg + 1 < it.n_seg) nsg = segs[seg + 1];
    }
  }
  return true;
}

// The row written out: O (one accumulator, relative to the item's last max m) / L with
// L = l_0 2^(m_0 - m) + l_1 2^(m_1 - m) over the two warpgroups' sums; warpgroup w writes columns
// 64 w .. 64 w + 63 of the bf16 row, warpgroup 0 the natural-log LSE.  The warpgroups swap
// (max, sum) through shared memory behind the item's ML barrier.
__device__ __forceinline__ bool write_rows(const PairParams& p, const RowQ& row, int w, int r,
                                           uint32_t lane_t, float m_w, float l_w, uint32_t nq,
                                           uint8_t* sp, uint32_t bar, volatile int* abort) {
  float2* ml = reinterpret_cast<float2*>(sp + kOffML) + (nq & 1) * 256;
  ml[w * 128 + r] = make_float2(m_w, l_w);
  tc::mbar_arrive(bar + 8 * (B_ML + (nq & 1)));
  const bool w_ok = tc::mbar_wait(bar + 8 * (B_ML + (nq & 1)), (nq >> 1) & 1, abort, p.status,
                                  kWaitNs);
  if (__any_sync(0xffffffffu, !w_ok)) return false;
  const float2 other = ml[(1 - w) * 128 + r];
  const float m = fmaxf(m_w, other.x);
  const float mr = m == -CUDART_INF_F ? 0.f : m;
  const float L = l_w * fast_exp2(m_w - mr) + other.y * fast_exp2(other.x - mr);  // 2^-inf = 0
  const bool none = !(L > 0.f);  // no key was visible: the row is zeros
  const float inv = none ? 0.f : 1.f / L;
  __nv_bfloat16* dst = p.o + ((int64_t)row.q_row * p.hq + row.qh) * kHeadDim + 64 * w;
#pragma unroll 1
  for (int q2 = 0; q2 < 2; ++q2) {
    uint32_t ov[32];
    tc::ld32(lane_t + kColO + 64 * w + 32 * q2, ov);
    tc::wait_ld();
    if (row.valid) {
      uint32_t wd[16];
#pragma unroll
      for (int j = 0; j < 16; ++j)
        wd[j] = pack_bf16(__uint_as_float(ov[2 * j]) * inv, __uint_as_float(ov[2 * j + 1]) * inv);
      if (p.o32) {
#pragma unroll
        for (int j = 0; j < 2; ++j) st_global_v8(dst + 32 * q2 + 16 * j, &wd[8 * j]);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          *reinterpret_cast<uint4*>(dst + 32 * q2 + 8 * j) =
              make_uint4(wd[4 * j], wd[4 * j + 1], wd[4 * j + 2], wd[4 * j + 3]);
      }
    }
  }
  if (row.valid && w == 0)
    p.lse[(int64_t)row.q_row * p.hq + row.qh] =
        (none ? -CUDART_INF_F : m + __log2f(L)) * 0.69314718055994530942f;
  return true;
}

// Softmax thread of the CTA's tile (tile A on the even CTA, tile B on the odd one): row r, in
// warpgroup w (the steps t = w mod 2 of every item), over the cluster's items.
__device__ __forceinline__ void softmax_role(const PairParams& p, uint32_t rank, uint32_t base,
                                             uint8_t* sp, uint32_t tmem, volatile int* abort) {
  const int r = threadIdx.x & 127;
  const int w = threadIdx.x >> 7;
  const int wq = (threadIdx.x >> 5) & 3;    // lane quarter of tensor memory
  const uint32_t lane_t = tmem + ((uint32_t)(32 * wq) << 16);
  const uint32_t bar = base + kOffBar;
  float* m_buf = reinterpret_cast<float*>(sp + kOffM);
  uint32_t pf_c[kSBuf];
#pragma unroll
  for (int b = 0; b < kSBuf; ++b) pf_c[b] = pair::map_to(bar + 8 * (B_PF + b), 0);
  int ri = 0;
  int idx = item_at(ri, p.n_items);
  while (idx >= 0 && p.items[idx].n_steps == 0) idx = item_at(++ri, p.n_items);
  if (idx < 0) return;
  ExtItem it = p.items[idx];
  RowQ row = row_of(p, it, (int)rank, r);
  SmCounts c{0u, 0u, 0u, {0u, 0u}};
  for (;;) {
    const ExtSeg* segs = p.segs + it.seg_begin;
    const int ntiles = it.n_steps;
    int nri = ri + 1;
    int nidx = item_at(nri, p.n_items);
    while (nidx >= 0 && p.items[nidx].n_steps == 0) nidx = item_at(++nri, p.n_items);
    ExtItem nit = it;
    RowQ nrow = row;
    auto ahead = [&]() {
      if (nidx >= 0) {
        nit = p.items[nidx];
        nrow = row_of(p, nit, (int)rank, r);
      }
    };
    float m_w = -CUDART_INF_F, l_w = 0.f;
    if (!softmax_steps(p, it, segs, ntiles, row, w, r, c, bar, pf_c, lane_t, m_buf, abort, m_w,
                       l_w, ahead))
      return;
    const bool w_ok = pair::wait(bar + 8 * B_OD, c.nq & 1, abort, p.status, kWaitNs);
    if (__any_sync(0xffffffffu, !w_ok)) return;
    tc::fence_after();
    if (!write_rows(p, row, w, r, lane_t, m_w, l_w, c.nq, sp, bar, abort)) return;
    c.sv += ntiles + kSBuf;
    c.pb += ntiles;
    ++c.nq;
    if (nidx < 0) return;
    ri = nri;
    idx = nidx;
    it = nit;
    row = nrow;
  }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    extend_pair_kernel(PairParams p, const __grid_constant__ CUtensorMap k_map,
                       const __grid_constant__ CUtensorMap v_map) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023) & ~1023u;
  uint8_t* sp = smem_raw + (base - raw);
  const int warp = threadIdx.x >> 5;
  const uint32_t rank = pair::cta_rank();
  volatile int* abort = reinterpret_cast<volatile int*>(sp + kOffAbort);
  volatile int* filled = reinterpret_cast<volatile int*>(sp + kOffFilled);
  const uint32_t bar = base + kOffBar;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      tc::mbar_init(bar + 8 * (B_KL + i), 1);
      tc::mbar_init(bar + 8 * (B_VL + i), 1);
      tc::mbar_init(bar + 8 * (B_KP + i), 1);
      tc::mbar_init(bar + 8 * (B_VP + i), 1);
      tc::mbar_init(bar + 8 * (B_KF + i), 1);
      tc::mbar_init(bar + 8 * (B_VF + i), 1);
    }
    for (int b = 0; b < kSBuf; ++b) {
      tc::mbar_init(bar + 8 * (B_SF + b), 1);
      tc::mbar_init(bar + 8 * (B_PF + b), 8);  // the four warps of a step's warpgroup, both CTAs
    }
    for (int q = 0; q < 2; ++q) {
      tc::mbar_init(bar + 8 * (B_QF + q), 1);
      tc::mbar_init(bar + 8 * (B_QP + q), 1);
      tc::mbar_init(bar + 8 * (B_QE + q), 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(bar + 8 * (B_ML + b), 256);
      tc::mbar_init(bar + 8 * (B_MR + b), 128);
    }
    tc::mbar_init(bar + 8 * B_OD, 1);
    tc::mbar_init(bar + 8 * B_DR, 1);
    for (int i = 0; i < 2 * kStages + 1; ++i) filled[i] = 0;
    *reinterpret_cast<volatile uint32_t*>(sp + kOffGate) = 0;
    *abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kWarpAlloc) pair::alloc(base + kOffTmem, kTmemCols);
  tc::fence_before();
  __syncthreads();
  pair::cluster_sync();  // both CTAs' barriers exist before any arrival crosses the pair
  tc::fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sp + kOffTmem);

  if (warp < kWarpK) {
    tc::regs_inc<kRegsSoftmax>();
    softmax_role(p, rank, base, sp, tmem, abort);
  } else {
    tc::regs_dec<kRegsOther>();
    if (warp < kWarpMma) {
      const bool k = warp < kWarpV;
      producer(p, warp - (k ? kWarpK : kWarpV), k, rank, base, k ? &k_map : &v_map,
               filled + (k ? 0 : kStages), abort);
    } else if (warp == kWarpMma) {
      if ((threadIdx.x & 31) == 0) {
        if (rank == 0)
          mma_issuer(p, base, tmem, abort);
        else
          relay(p, base, abort);
      }
      __syncwarp();
    } else if (rank == 0) {  // warp 15 of the even CTA: the issuer's gate
      if ((threadIdx.x & 31) == 0) gate_role(p, base, abort);
      __syncwarp();
    }
  }
  // Before the pair exits: this CTA's copies still in flight land (only the last fill of each
  // stage, and the last Q load, can be pending; the MMAs waited for every earlier one).
  __syncthreads();
  if (threadIdx.x < 2 * kStages + 1) {
    const int f = filled[threadIdx.x];
    const bool is_q = threadIdx.x == 2 * kStages;  // f = Q loads: the last went to buffer (f-1) % 2
    const int b = threadIdx.x < kStages       ? B_KL + threadIdx.x
                  : threadIdx.x < 2 * kStages ? B_VL + (threadIdx.x - kStages)
                                              : B_QF + ((f - 1) & 1);
    const uint32_t parity = is_q ? (uint32_t)((f - 1) >> 1) & 1 : (uint32_t)(f - 1) & 1;
    int no_abort = 0;
    if (f > 0) pair::wait(bar + 8 * b, parity, &no_abort, p.status, kWaitNs);
  }
  tc::fence_before();
  __syncthreads();
  pair::cluster_sync();  // no MMA of the pair and no arrival from the other CTA is pending
  if (warp == kWarpAlloc) {
    tc::fence_after();
    pair::dealloc(tmem, kTmemCols);
  }
}

// Clusters of two that can be resident at once on the current device, and the launch attributes
// checked, once per device.
struct PairDevice {
  int clusters = 0;
};
PairDevice g_pair_dev[64];
std::atomic<uint64_t> g_pair_ready{0};

int pair_device_setup(int dev) {
  if ((g_pair_ready.load() >> dev) & 1) return 0;
  // The softmax warpgroup raises its register budget with what the other warpgroups give up;
  // that only balances when every thread starts with exactly kRegsLaunch registers, so any other
  // build is refused.
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, extend_pair_kernel);
  if (e != cudaSuccess) return (int)e;
  if (fa.numRegs != kRegsLaunch) return (int)cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(extend_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kSmem);
  if (e != cudaSuccess) return (int)e;
  // the kernel's cluster shape is compiled in (two CTAs), so the query passes no attribute
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmem;
  cfg.numAttrs = 0;
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, extend_pair_kernel, &cfg);
  if (e != cudaSuccess || n < 1) {
    // without the query: one cluster per two SMs (clusters beyond what fits simply wait for a
    // pair to free up, since no cluster waits on another)
    (void)cudaGetLastError();
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return (int)e;
    n = sms / 2 > 0 ? sms / 2 : 1;
  }
  g_pair_dev[dev].clusters = n;
  g_pair_ready.fetch_or(1ull << dev);
  return 0;
}

}  // namespace

int launch_extend_pair(const rx_kv_desc* d, const ExtItem* items, const ExtRow* rows,
                       const ExtSeg* segs, int32_t n_items, const void* k_pool, const void* v_pool, const void* q, void* o,
                       float* lse, int32_t* status, void* stream) {
  int dev = 0;
  cudaError_t de = cudaGetDevice(&dev);
  if (de != cudaSuccess) return (int)de;
  if (dev < 0 || dev >= 64) return (int)cudaErrorInvalidDevice;
  int e = pair_device_setup(dev);
  if (e) return e;
  if (n_items == 0) return 0;
  PairParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.req_to_token = d->req_to_token;
  p.stride = d->req_to_token_stride;
  p.hq = d->num_q_heads;
  p.hkv = d->num_kv_heads;
  p.gq = d->num_q_heads / d->num_kv_heads;
  p.scale_log2 = d->softmax_scale * 1.4426950408889634f;
  p.items = items;
  p.rows = rows;
  p.segs = segs;
  p.pool_size = d->pool_size;
  p.status = status;
  p.oob_row = (int32_t)(d->pool_size * d->num_kv_heads);
  p.n_items = n_items;
  p.o32 = (reinterpret_cast<uintptr_t>(o) & 31u) == 0;
  CUtensorMap k_map, v_map;
  e = make_pool_map(&k_map, k_pool, d);
  if (!e) e = make_pool_map(&v_map, v_pool, d);
  if (e) return e;
  // persistent: one cluster per SM pair that can hold one, at most one per item
  const int clusters = n_items < g_pair_dev[dev].clusters ? n_items : g_pair_dev[dev].clusters;
  extend_pair_kernel<<<2 * clusters, kThreads, kSmem, (cudaStream_t)stream>>>(p, k_map, v_map);
  return (int)cudaGetLastError();
}

}  // namespace rx
