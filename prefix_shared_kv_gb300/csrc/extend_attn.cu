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
// Blackwell tile loop (a persistent CTA per SM walks its share of the work items; an item is two
// 128-row tiles A and B of one KV head; 512 threads, warp-specialised, 64 keys per step; every K/V
// step feeds both tiles, i.e. 256 rows):
//   warps 8-10  K producers (steps t = 0, 1, 2 mod 3), warps 11-13 V producers: gather the keys'
//              256-byte rows by slot with TMA (cp.async.bulk.tensor tile::gather4: four pool rows
//              per instruction, 128-byte swizzle applied by the copy engine) into 5-stage rings
//              laid out as UMMA tiles; slot indices are fetched one step of their own ahead; a
//              stage completes on its mbarrier's transaction count.
//   warps 14-15  MMA issuers (one thread each, one per tile X): S_X = Q_X K^T with tcgen05.mma
//              (K-major operands in shared memory, fp32 accumulator in TMEM) into one of two S
//              buffers, and O_X += P_X V with P_X read from TMEM and V as an MN-major shared-
//              memory operand.  P_X(t) is written over the upper half of the S buffer it came
//              from, and the issuer's order per step is PV_X(t), S_X(t+2) into that buffer: the
//              tensor pipe executes one thread's MMAs in order, so S_X(t+2) overwrites P_X(t) only
//              after PV_X(t) has read it, and S_X(t+1) is always computed a step ahead.
//   warps 0-3 (tile A), 4-7 (tile B)  softmax: thread r of a group owns row r of its tile (TMEM
//              lane r) and copies it into the tile's Q buffer first; per step: tcgen05.ld of its
//              64 scores, masks, online max / sum in base 2 (the running max is only moved -- and
//              O in TMEM rescaled -- when it grows by more than 2^8), P = exp2(.) packed to bf16
//              and written to TMEM with tcgen05.st for the PV MMA; finally O / l and the LSE.  The
//              two tiles take turns for the exponentials, so each has the SM's exp units to
//              itself while the tensor core works on the other tile; everything before the
//              exponentials (loads, masks, maximum, scale-and-shift) runs outside the turn.
// Items follow one another without a break in the pipelines: the rings, S buffers and barrier
// phases run on across items, the query rows of the next item are copied in as soon as the last
// S of the current one is computed, and the first two S of the next item are computed while the
// softmax warps write out the current one.
// Every mbarrier wait is bounded (globaltimer); a timeout records RX_ERR_TIMEOUT in the
// workspace status word and every role leaves its loop.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include <atomic>

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
  int32_t oob_row;  // a row index past the end of the pool's [pool_size * Hkv, 128] view
  float* part_o;    // non-null: write fp32 partial rows (decode shared-prefix units)
  float* part_lse;
  int n_items;
  const int32_t* cta_begin;  // per-CTA item lists ([gridDim.x + 1] starts), or null: snake deal
  bool o32;         // o is 32-byte aligned: rows go out in 32-byte stores, else 16-byte ones
};

constexpr int kN = kAttnKeys;          // keys per step (64)
constexpr int kPW = 3;                 // producer warps per operand (one gather in issue each)
constexpr int kWarpK = 8, kWarpV = kWarpK + kPW, kWarpMma = kWarpV + kPW;
constexpr int kThreads = 32 * (kWarpMma + 2);  // softmax A, B | K producers | V producers | MMA A, B
static_assert(kThreads == 512, "four warpgroups: the register split below assumes them");
constexpr int kRegsLaunch = 65536 / kThreads;  // 128: what each thread is launched with
constexpr int kRegsSoftmax = 160, kRegsOther = 96;
static_assert(2 * kRegsSoftmax + 2 * kRegsOther == 4 * kRegsLaunch, "register split");
constexpr int kStages = 5;             // K ring and V ring depth (64-key stages)
// A producer warp fills every kPW-th stage of its ring and first waits for that stage to be
// released.  That wait tests a phase parity, so it must never be two phases early: the warp's own
// previous wait covered every step up to kPW + kStages before the current one, which rules that
// out when the ring has at least kPW stages.
static_assert(kStages >= kPW, "a producer could run two phases ahead");
constexpr int kQHalf = 128 * 128;      // one 64-column half of a 128-row query tile: 16 KiB
constexpr int kQTile = 2 * kQHalf;     // 32 KiB
constexpr int kKVHalf = kN * 128;      // one 64-column half of a 64-key K or V tile: 8 KiB
constexpr int kKVTile = 2 * kKVHalf;   // 16 KiB
constexpr int kOffQ = 0;               // tile A, then tile B
constexpr int kOffK = 2 * kQTile;
constexpr int kOffV = kOffK + kStages * kKVTile;
constexpr int kOffBar = kOffV + kStages * kKVTile;
// Barriers (each waiter is at most one phase behind the barrier it tests):
//   K_FULL[k] / V_FULL[k]   step landed in ring stage k (expect_tx by the producer + TMA bytes)
//   K_FREE[k]  S_A and S_B of the step complete, K stage free  (two arrivals: a commit each)
//   V_FREE[k]  PV_A and PV_B of the step complete, V stage free
//   S_FULL[x][b]  S_x(t) complete in buffer b = t % 2 (phase t / 2).  The issuer commits it once
//              per step after PV_x(t) and S_x(t+2) (S_x(t+2) only when there is such a step), so
//              the phase of step t+1 also tells that PV_x(t-1) is complete: O_x may be rescaled.
//   P_FULL[x][b]  P_x(t) in S buffer b = t % 2 (phase t / 2; tile x's 128 softmax threads).  One
//              barrier per buffer: with S_x(t+1) already computed, the softmax can finish step
//              t+1 before the issuer has taken step t, so a single barrier could run two phases
//              ahead of the issuer; P_x(t+2) waits for S_x(t+2), which waits for P_x(t).
//   O_DONE[x]  every MMA of tile x's item complete: O_x final for the epilogue
//   Q_FULL[x]  tile x's query rows in shared memory (tile x's 128 softmax threads)
//   TURN[x]    tile x's softmax may run its exponentials for the next step (128 arrivals of the
//              other tile's softmax): A(0), B(0), A(1), B(1), ...
//   DRAIN[x]   every MMA of issuer x complete, at the end: TMEM may be released
// Phases count on across items.  Per item of tile x the issuer commits S_FULL[x] for steps
// 0 .. ntiles + 1 (the last two without an MMA), so the S steps of successive items are
// contiguous.  In an item with tile A only, issuer B releases each ring stage with a plain
// arrival once the stage has landed.
enum {
  B_K_FULL = 0,
  B_K_FREE = B_K_FULL + kStages,
  B_V_FULL = B_K_FREE + kStages,
  B_V_FREE = B_V_FULL + kStages,
  B_S_FULL = B_V_FREE + kStages,  // [x][b] at B_S_FULL + 2 * x + b
  B_P_FULL = B_S_FULL + 4,  // [x][b] at B_P_FULL + 2 * x + b
  B_O_DONE = B_P_FULL + 4,
  B_Q_FULL = B_O_DONE + 2,
  B_TURN = B_Q_FULL + 2,
  B_DRAIN = B_TURN + 2,
  B_COUNT = B_DRAIN + 2
};
constexpr int kOffTmem = kOffBar + B_COUNT * 8;
constexpr int kOffAbort = kOffTmem + 8;
constexpr size_t kSmem = 1024 + kOffAbort + 16;
// TMEM columns: S buffers S_A0, S_A1, S_B0, S_B1 of 64 columns from 0 (P_x(t), 64 bf16 a row, two
// a column, over the upper half of S_x's buffer t % 2), O_A [256,384), O_B [384,512)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;
constexpr uint32_t kPOff = 32;
constexpr uint64_t kWaitNs = 2000000000ull;
__host__ __device__ constexpr uint32_t col_s_of(int x, int b) { return (uint32_t)(2 * x + b) * kN; }

static_assert(kSmem <= 227 * 1024, "shared memory budget");

struct TileIter {
  int seg, k0;
};
__device__ __forceinline__ void tile_next(TileIter& c, const ExtSeg* segs, int n_seg) {
  if (c.seg >= n_seg) return;  // already past the last segment: never read beyond the item
  c.k0 += kN;
  if (c.k0 >= segs[c.seg].k_end) {
    ++c.seg;
    if (c.seg < n_seg) c.k0 = segs[c.seg].k_begin;
  }
}

// The CTA's r-th item, -1 past the end.  With per-CTA lists (extend plans) CTA k runs items
// cta_begin[k] .. cta_begin[k + 1] - 1 in order.  Without (decode shared-prefix units) the list is
// dealt to the grid in snake order (round r holds items r G .. r G + G - 1; CTA k takes the k-th
// of an even round and the (G - 1 - k)-th of an odd one), so that a list sorted by falling cost
// gives every CTA a similar total.
__device__ __forceinline__ int item_at(const ExtParams& p, int r) {
  const int k = blockIdx.x;
  if (p.cta_begin) {
    const int i = __ldg(&p.cta_begin[k]) + r;
    return i < __ldg(&p.cta_begin[k + 1]) ? i : -1;
  }
  const int G = gridDim.x;
  const int64_t i = (int64_t)r * G + ((r & 1) ? G - 1 - k : k);
  return i < p.n_items ? (int)i : -1;
}

// Byte offset of 16-byte chunk c (0..15) of row r in a K-major tile stored as two 128-byte-
// swizzled halves (d 0..63, d 64..127) of `half` bytes each.
__device__ __forceinline__ uint32_t tile_off(int r, int c, int half) {
  return (uint32_t)((c >> 3) * half + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// Raw table entry for key position k0 + key of segment sg (-1 past the segment).  No test on the
// loaded value here, so the load stays in flight until the slot is used; check_slot validates it.
__device__ __forceinline__ int fetch_slot(const ExtParams& p, const ExtSeg& sg, int k0, int key) {
  const int kpos = k0 + key;
  return kpos < sg.k_end ? __ldg(p.req_to_token + (int64_t)sg.kv_row * p.stride + kpos) : -1;
}

// -1 stays -1 (nothing to load); an entry outside the pool flags RX_ERR_RANGE and is not read.
__device__ __forceinline__ int check_slot(const ExtParams& p, int s) {
  if (s >= p.pool_size || s < -1) {
    atomicCAS(p.status, 0, (int)RX_ERR_RANGE);
    return -1;
  }
  return s;
}

// TMA gather of four pool rows (one 64-column half each) into consecutive 128-byte rows of a
// 128-byte-swizzled tile; completion is counted in bytes on `mbar`.
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


// Producer warp of one operand (K or V): steps t = w, w + kPW, ...  A warp has one
// tile::gather4 in issue at a time (about a hundred cycles each), so the rate at which the rings
// fill grows with the number of producer warps.  The pool is viewed by the tensor map as rows of
// 128 bf16 (row = slot * Hkv + head).  Per step lane j gathers keys 4 (j % 16) .. 4 (j % 16) + 3,
// half j / 16 of their 256-byte rows, with one tile::gather4 (32 gathers = the 64 keys' K or V);
// it fetches those keys' table entries one step of its own ahead.  Keys past the segment (or
// flagged entries) read a row past the end of the map, which the TMA fills with zeros.
struct Slot4 {
  int v[4];
};

__device__ __forceinline__ void producer(const ExtParams& p, int w, uint32_t base,
                                         const CUtensorMap* map, uint32_t ring, int b_full,
                                         int b_free, volatile int* abort) {
  const int lane = threadIdx.x & 31;
  const int g = lane & 15, h = lane >> 4;
  const uint32_t bar = base + kOffBar;
  uint32_t gs = 0;  // ring steps of the CTA's earlier items
  for (int ri = 0;; ++ri) {
    const int idx = item_at(p, ri);
    if (idx < 0) return;
    const ExtItem it = p.items[idx];
    const ExtSeg* segs = p.segs + it.seg_begin;
    const int ntiles = it.n_steps;
    TileIter at{0, ntiles > 0 ? segs[0].k_begin : 0};
    int at_step = 0;
    auto fetch = [&](Slot4& sl, int t) {  // entries of step t (t only grows)
      for (; at_step < t; ++at_step) tile_next(at, segs, it.n_seg);
      const ExtSeg& sg = segs[at.seg];
#pragma unroll
      for (int i = 0; i < 4; ++i) sl.v[i] = fetch_slot(p, sg, at.k0, 4 * g + i);
    };
    // this warp's steps are the ring steps w, w + kPW, ... counted over all the CTA's items
    const int t0 = (int)((w + kPW - gs % kPW) % kPW);
    Slot4 nxt{{-1, -1, -1, -1}};
    if (t0 < ntiles) fetch(nxt, t0);
    // per step: take the prefetched entries, prefetch t + kPW, wait for the stage, gather t
    for (int t = t0; t < ntiles; t += kPW) {
      const Slot4 cur = nxt;
      if (t + kPW < ntiles) fetch(nxt, t + kPW);
      const uint32_t gt = gs + t;
      const int st = gt % kStages;
      const bool waited = gt < kStages || tc::mbar_wait(bar + 8 * (b_free + st),
                                                        (gt / kStages - 1) & 1, abort, p.status,
                                                        kWaitNs);
      if (__any_sync(0xffffffffu, !waited)) return;  // the warp leaves together
      int r[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int v = check_slot(p, cur.v[i]);
        r[i] = v >= 0 ? v * p.hkv + it.kv_head : p.oob_row;
      }
      if (lane == 0) mbar_expect_tx(bar + 8 * (b_full + st), kN * kHeadDim * 2);
      __syncwarp();
      tma_gather4(ring + st * kKVTile + h * kKVHalf + g * 512, map, 64 * h, r[0], r[1], r[2],
                  r[3], bar + 8 * (b_full + st));
    }
    gs += ntiles;
  }
}

// MMA issuer of tile x (one thread), per item: S_x(0) and S_x(1); then per step t, once P_x(t) is
// in TMEM, PV_x(t) and S_x(t+2) right behind it (into the buffer P_x(t) sat in).  The two tiles
// have an issuer each (the last two warps, on different SM sub-partitions); both commit to the
// ring stages' free barriers, which therefore take two arrivals.  The MMAs of a step are issued
// back to back and their commits follow them: a commit holds up the issuing thread's next
// barrier operation until the tensor pipe has taken the MMAs before it, so every wait comes first.
// The S_x(0), S_x(1) of the next item go in right after PV_x of the current one's last step: the
// tensor pipe keeps one thread's MMAs in order, so they overwrite S buffers whose P has been used.
__device__ __forceinline__ void mma_issuer(const ExtParams& p, int x, uint32_t base,
                                           uint32_t tmem, volatile int* abort) {
  constexpr uint32_t idS = tc::idesc_bf16(128, kN, false, false);
  constexpr uint32_t idO = tc::idesc_bf16(128, 128, false, true);
  const uint32_t bar = base + kOffBar;
  // descriptors of the tile bases; an operand at byte offset o adds o >> 4 (no carry: shared
  // memory addresses stay below 256 KiB)
  const uint64_t qdesc = tc::desc_sw128(base + kOffQ + x * kQTile, 16, 1024);
  const uint64_t kdesc0 = tc::desc_sw128(base + kOffK, 16, 1024);
  const uint64_t vdesc0 = tc::desc_sw128(base + kOffV, kKVHalf, 1024);
  const uint32_t d_o = tmem + kColO + x * 128;
  bool ok = true;
  auto wait = [&](int b, uint32_t parity) {
    ok = ok && tc::mbar_wait(bar + 8 * b, parity, abort, p.status, kWaitNs);
    return ok;
  };
  // running counts over the CTA's earlier items: ring steps, S steps of tile x (ntiles + 2 per
  // item), P steps of tile x, items of tile x
  uint32_t gs = 0, sv = 0, pb = 0, nq = 0;
  for (int ri = 0; ok; ++ri) {
    const int idx = item_at(p, ri);
    if (idx < 0) break;
    const ExtItem it = p.items[idx];
    const int ntiles = it.n_steps;
    const bool two = it.n_tok[1] > 0;
    if (ntiles == 0) continue;  // (plans hold none; every role skips them alike)
    if (x == 1 && !two) {
      // no tile B: release the item's ring stages beside issuer A, one step after another (so
      // this thread never tests a ring barrier two phases away from the one it waits for)
      for (int t = 0; t < ntiles; ++t) {
        const uint32_t gt = gs + t;
        if (!wait(B_K_FULL + gt % kStages, (gt / kStages) & 1)) break;
        tc::mbar_arrive(bar + 8 * (B_K_FREE + gt % kStages));
        if (!wait(B_V_FULL + gt % kStages, (gt / kStages) & 1)) break;
        tc::mbar_arrive(bar + 8 * (B_V_FREE + gt % kStages));
      }
      gs += ntiles;
      continue;
    }
    auto release = [&](int b, uint32_t gt) { tc::commit(bar + 8 * (b + (int)(gt % kStages))); };
    auto qk = [&](int t) {  // S_x(t) = Q_x K(t)^T into buffer (sv + t) % 2
      const uint64_t kd = kdesc0 + ((((gs + t) % kStages) * kKVTile) >> 4);
      const uint32_t d_s = tmem + col_s_of(x, (sv + t) & 1);
#pragma unroll
      for (int s = 0; s < 8; ++s)
        tc::mma_ss(d_s, qdesc + (((s >> 2) * kQHalf + (s & 3) * 32) >> 4),
                   kd + (((s >> 2) * kKVHalf + (s & 3) * 32) >> 4), idS, s > 0 ? 1u : 0u);
    };
    auto pv = [&](int t) {  // O_x += P_x(t) V(t)
      const uint64_t vd = vdesc0 + ((((gs + t) % kStages) * kKVTile) >> 4);
      const uint32_t a_p = tmem + col_s_of(x, (sv + t) & 1) + kPOff;
#pragma unroll
      for (int s = 0; s < kN / 16; ++s)
        tc::mma_ts(d_o, a_p + 8 * s, vd + ((s * 2048) >> 4), idO, (t > 0 || s > 0) ? 1u : 0u);
    };
    if (!wait(B_Q_FULL + x, nq & 1)) break;
    for (int t = 0; t < 2; ++t) {
      if (t < ntiles) {
        if (!wait(B_K_FULL + (gs + t) % kStages, ((gs + t) / kStages) & 1)) break;
        tc::fence_after();
        qk(t);
        tc::commit(bar + 8 * (B_S_FULL + 2 * x + ((sv + t) & 1)));
        release(B_K_FREE, gs + t);
      } else {
        tc::commit(bar + 8 * (B_S_FULL + 2 * x + ((sv + t) & 1)));  // step without an MMA
      }
    }
    for (int t = 0; ok && t < ntiles; ++t) {
      const uint32_t gt = gs + t, gt2 = gt + 2;
      const bool more = t + 2 < ntiles;
      // the ring stages normally land long before the softmax hands P over: test them first, so
      // only the P wait stands between P and the MMAs
      if ((more && !wait(B_K_FULL + gt2 % kStages, (gt2 / kStages) & 1)) ||
          !wait(B_V_FULL + gt % kStages, (gt / kStages) & 1) ||
          !wait(B_P_FULL + 2 * x + ((pb + t) & 1), ((pb + t) >> 1) & 1))
        break;
      tc::fence_after();
      pv(t);
      if (more) qk(t + 2);
      release(B_V_FREE, gt);
      tc::commit(bar + 8 * (B_S_FULL + 2 * x + ((sv + t) & 1)));  // also after the last steps
      if (more) release(B_K_FREE, gt2);
    }
    if (!ok) break;
    tc::commit(bar + 8 * (B_O_DONE + x));
    gs += ntiles;
    sv += ntiles + 2;
    pb += ntiles;
    ++nq;
  }
  // every MMA issued above completes before TMEM is released, after an abort too
  tc::commit(bar + 8 * (B_DRAIN + x));
  int no_abort = 0;
  tc::mbar_wait(bar + 8 * (B_DRAIN + x), 0, &no_abort, p.status, kWaitNs);
}

// Row maximum of the 64 raw scores (three-input maxima, eight independent chains).  Masked keys
// hold -inf, so one code path serves every step (a smaller kernel keeps the instruction cache
// warm for all the roles that share an SM sub-partition).
__device__ __forceinline__ float row_max(const uint32_t (&sr)[2][32]) {
  float m[8];
#pragma unroll
  for (int a = 0; a < 8; ++a) m[a] = __uint_as_float(sr[0][a]);
#pragma unroll
  for (int q = 0; q < 2; ++q)
#pragma unroll
    for (int j = 0; j < 32; j += 2)
      if (q > 0 || j >= 8)
        m[(j >> 1) & 7] =
            fmax3(m[(j >> 1) & 7], __uint_as_float(sr[q][j]), __uint_as_float(sr[q][j + 1]));
#pragma unroll
  for (int a = 0; a < 2; ++a) m[a] = fmax3(m[a], m[a + 2], m[a + 4]);
  return fmax3(m[0], m[1], fmaxf(m[6], m[7]));
}

// In place, on packed fp32 pairs: s_j -> s_j * scale_log2 - m (a masked key's -inf stays -inf; m
// is finite).
__device__ __forceinline__ void row_shift(uint32_t (&sr)[2][32], float sl2, float m) {
  const uint64_t k2 = f2_pack(sl2, sl2), nm2 = f2_pack(-m, -m);
#pragma unroll
  for (int q = 0; q < 2; ++q)
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
      float x0, x1;
      f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[q][j]), __uint_as_float(sr[q][j + 1])), k2,
                       nm2),
                x0, x1);
      sr[q][j] = __float_as_uint(x0);
      sr[q][j + 1] = __float_as_uint(x1);
    }
}

// p_e = 2^x_e for the row's 64 elements (-inf gives 0), packed to bf16 pairs in pk and added into
// two chains of packed (even, odd) partial sums.
__device__ __forceinline__ void row_exp(const uint32_t (&sr)[2][32], uint32_t (&pk)[32],
                                        uint64_t (&acc)[2]) {
#pragma unroll
  for (int e = 0; e < kN; e += 2) {
    const int q = e >> 5, j = e & 31;
    const float p0 = fast_exp2(__uint_as_float(sr[q][j]));
    const float p1 = fast_exp2(__uint_as_float(sr[q][j + 1]));
    acc[(j >> 1) & 1] = f2_add(acc[(j >> 1) & 1], f2_pack(p0, p1));
    pk[e >> 1] = pack_bf16(p0, p1);
  }
}

// 32 bytes to global memory (the address 32-byte aligned).
__device__ __forceinline__ void st_global_v8(void* dst, const uint32_t* w) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(w[0]),
               "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// A softmax thread's query row in an item: row r of tile x.
struct RowQ {
  int owner, kmax, q_row, qh;
  bool valid;
};

__device__ __forceinline__ RowQ row_of(const ExtParams& p, const ExtItem& it, int x, int r) {
  // (selects rather than it.n_tok[x]: indexing the item with a runtime x would put it on the stack)
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

// Starts the copy of the thread's query row into row r of the tile's Q buffer (16 chunks of 16
// bytes; zeros for a row past the tile's rows).
__device__ __forceinline__ void load_q(const ExtParams& p, const RowQ& q, uint32_t qb, int r) {
  const __nv_bfloat16* src = p.q + ((int64_t)q.q_row * p.hq + q.qh) * kHeadDim;
#pragma unroll
  for (int c = 0; c < 16; ++c)
    cp_async16(qb + tile_off(r, c, kQHalf), q.valid ? src + c * 8 : p.q, q.valid);
  cp_async_commit();
}

// Whether tile x's softmax and issuer take part in an item (items without steps: none).
__device__ __forceinline__ bool has_tile(const ExtItem& it, int x) {
  return it.n_steps > 0 && (x == 0 || it.n_tok[1] > 0);
}

// The CTA's first item from round *ri on that has tile x (-1: none); *ri is left at its round.
__device__ __forceinline__ int first_item(const ExtParams& p, int x, int* ri) {
  for (;; ++*ri) {
    const int idx = item_at(p, *ri);
    if (idx < 0 || has_tile(p.items[idx], x)) return idx;
  }
}

// Running counts over the CTA's earlier items of tile x: S steps (ntiles + 2 per item), P steps,
// exponential turns (steps of items with both tiles), items.
struct SmCounts {
  uint32_t sv, pb, tb, nq;
};

// The steps of one item for a softmax thread (TWO: tile B present, the tiles take turns for the
// exponentials -- a compile-time choice: a runtime test inside the step loop costs a few percent).
// At the first step ahead() looks up the next item's row; at the last step, once S_x of it is in
// TMEM (every S_x of the item computed, the Q buffer no longer read), prefetch() starts the copy
// of the next item's query row.  Returns false when a wait gave up (the warp then leaves
// together).
template <bool TWO, class Ahead, class Prefetch>
__device__ __forceinline__ bool softmax_steps(const ExtParams& p, const ExtItem& it,
                                              const ExtSeg* segs, int ntiles, const RowQ& row,
                                              const SmCounts& c, uint32_t bar, uint32_t lane_t,
                                              volatile int* abort, float& m_used, float& l,
                                              Ahead&& ahead, Prefetch&& prefetch) {
  constexpr bool two = TWO;
  const int x = threadIdx.x >> 7;  // tile: 0 = A, 1 = B
  const uint32_t col_o = kColO + x * 128;
  const float sl2 = p.scale_log2;
  // the current key segment lives in registers; the next one's record is loaded when a segment
  // starts, so no step waits for a table read
  int seg = 0, k0 = segs[0].k_begin, k_end = segs[0].k_end, s_owner = segs[0].owner;
  ExtSeg nsg = segs[it.n_seg > 1 ? 1 : 0];
  if (two && x == 1) tc::mbar_arrive(bar + 8 * B_TURN);  // tile A goes first
  // (a lone tile A takes no turns)
  for (int t = 0; t < ntiles; ++t) {
    const uint32_t vs = c.sv + t;  // S step
    const uint32_t col_s = col_s_of(x, vs & 1);
    const bool w_ok = tc::mbar_wait(bar + 8 * (B_S_FULL + 2 * x + (vs & 1)), (vs >> 1) & 1, abort,
                                    p.status, kWaitNs);
    if (__any_sync(0xffffffffu, !w_ok)) return false;
    tc::fence_after();
    if (t == 0) ahead();
    if (t == ntiles - 1) prefetch();
    const bool vis = row.valid && (s_owner < 0 || s_owner == row.owner);
    const int lim = vis ? min(row.kmax, k_end) : 0;  // keys at positions >= lim are masked
    const int n_ok = max(0, min(kN, lim - k0));
    uint32_t sr[2][32];
    tc::ld32(lane_t + col_s, sr[0]);
    tc::ld32(lane_t + col_s + 32, sr[1]);
    tc::wait_ld();
    if (n_ok < kN) {  // keys at n_ok and beyond are masked: -inf
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (32 * q + j >= n_ok) sr[q][j] = 0xff800000u;
    }
    const float mx = row_max(sr);
    const float m_new = n_ok > 0 ? fmaxf(m_used, mx * sl2) : m_used;
    const bool need = m_new > m_used + 8.f;
    const bool rescale = __any_sync(0xffffffffu, need);
    const float alpha = need ? fast_exp2(m_used - m_new) : 1.f;  // exp2(-inf) = 0
    if (need) m_used = m_new;
    // a row that has seen no visible key yet has m_used = -inf and only masked keys: any finite
    // reference gives p = 0 for them
    row_shift(sr, sl2, m_used == -CUDART_INF_F ? 0.f : m_used);
    // only the exponentials wait for the turn: masking, the maximum and the scale-and-shift run
    // while the other tile has the exp units
    const bool turn = !two || tc::mbar_wait(bar + 8 * (B_TURN + x), (c.tb + t) & 1, abort,
                                            p.status, kWaitNs);
    if (__any_sync(0xffffffffu, !turn)) return false;
    uint32_t pk[32];
    uint64_t acc[2] = {0ull, 0ull};
    row_exp(sr, pk, acc);
    if (two && (x == 0 || t + 1 < ntiles)) tc::mbar_arrive(bar + 8 * (B_TURN + 1 - x));  // other's turn
    {
      float a0, a1, b0, b1;
      f2_unpack(acc[0], a0, a1);
      f2_unpack(acc[1], b0, b1);
      l = l * alpha + ((a0 + a1) + (b0 + b1));
    }
    if (rescale && t > 0) {
      // O_x must hold PV_x(t-1): the phase of S step t+1 covers it, and PV_x(t) waits for this
      // step's P
      const uint32_t vn = vs + 1;
      const bool w2 = tc::mbar_wait(bar + 8 * (B_S_FULL + 2 * x + (vn & 1)), (vn >> 1) & 1, abort,
                                    p.status, kWaitNs);
      if (__any_sync(0xffffffffu, !w2)) return false;
      tc::fence_after();
#pragma unroll 1
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t ov[32];
        tc::ld32(lane_t + col_o + 32 * q4, ov);
        tc::wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * alpha);
        tc::st32(lane_t + col_o + 32 * q4, ov);
      }
    }
    tc::st32(lane_t + col_s + kPOff, pk);
    tc::wait_st();
    tc::fence_before();
    tc::mbar_arrive(bar + 8 * (B_P_FULL + 2 * x + ((c.pb + t) & 1)));
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

// O_x / l out of TMEM: bf16 O and natural-log LSE; for decode shared-prefix units fp32 partial
// rows and base-2 LSE for the merge (row part[x] + r of the item).
__device__ __forceinline__ void write_rows(const ExtParams& p, int idx, const RowQ& row,
                                           uint32_t lane_t, float m_used, float l) {
  const int x = threadIdx.x >> 7, r = threadIdx.x & 127;
  const uint32_t col_o = kColO + x * 128;
  // l = 0: no key was visible: the row is zeros, whatever O_x holds
  const bool none = !(l > 0.f);
  const float inv = none ? 0.f : 1.f / l;
  const bool partial = p.part_o != nullptr;
  int64_t prow = 0;
  if (partial) {
    const ExtItem& itg = p.items[idx];
    prow = (int64_t)__ldg(x ? &itg.part[1] : &itg.part[0]) + r;
  }
  __nv_bfloat16* dst = p.o + ((int64_t)row.q_row * p.hq + row.qh) * kHeadDim;
  float* pdst = p.part_o + prow * kHeadDim;
#pragma unroll 1
  for (int q4 = 0; q4 < 4; ++q4) {
    uint32_t ov[32];
    tc::ld32(lane_t + col_o + 32 * q4, ov);
    tc::wait_ld();
    if (none) {
#pragma unroll
      for (int j = 0; j < 32; ++j) ov[j] = 0u;
    }
    // 32-byte stores where alignment allows: each thread writes a row of its own, so a store
    // instruction touches 32 rows; wider stores mean fewer of them (partial rows sit in the
    // 256-byte aligned workspace)
    if (row.valid && partial) {
#pragma unroll
      for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * inv);
#pragma unroll
      for (int j = 0; j < 4; ++j) st_global_v8(pdst + 32 * q4 + 8 * j, &ov[8 * j]);
    } else if (row.valid) {
      uint32_t w[16];
#pragma unroll
      for (int j = 0; j < 16; ++j)
        w[j] = pack_bf16(__uint_as_float(ov[2 * j]) * inv, __uint_as_float(ov[2 * j + 1]) * inv);
      if (p.o32) {
#pragma unroll
        for (int j = 0; j < 2; ++j) st_global_v8(dst + 32 * q4 + 16 * j, &w[8 * j]);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          *reinterpret_cast<uint4*>(dst + 32 * q4 + 8 * j) =
              make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
      }
    }
  }
  if (!row.valid) return;
  const float lse2 = l > 0.f ? m_used + __log2f(l) : -CUDART_INF_F;
  if (partial)
    p.part_lse[prow] = lse2;
  else
    p.lse[(int64_t)row.q_row * p.hq + row.qh] = lse2 * 0.69314718055994530942f;
}

// Softmax thread r of tile x (TMEM lane r) over the CTA's items of tile x.  The next item's
// record is loaded when an item starts and its row at the item's first step, so neither load
// waits at the item boundary.
__device__ __forceinline__ void softmax_role(const ExtParams& p, uint32_t base, uint32_t tmem,
                                             volatile int* abort) {
  const int x = threadIdx.x >> 7;
  const int r = threadIdx.x & 127;
  const int wq = (threadIdx.x >> 5) & 3;
  const uint32_t lane_t = tmem + ((uint32_t)(32 * wq) << 16);
  const uint32_t bar = base + kOffBar;
  const uint32_t qb = base + kOffQ + x * kQTile;
  int ri = 0;
  int idx = first_item(p, x, &ri);
  if (idx < 0) return;
  ExtItem it = p.items[idx];
  RowQ row = row_of(p, it, x, r);
  load_q(p, row, qb, r);
  cp_async_wait<0>();
  tc::fence_proxy_async();
  tc::mbar_arrive(bar + 8 * (B_Q_FULL + x));
  SmCounts c{0u, 0u, 0u, 0u};
  for (;;) {
    const ExtSeg* segs = p.segs + it.seg_begin;
    const int ntiles = it.n_steps;
    const bool two = it.n_tok[1] > 0;
    const int nidx = item_at(p, ri + 1);
    ExtItem nit = it;
    if (nidx >= 0) nit = p.items[nidx];
    RowQ nrow = row;
    bool pre = false;  // the next item has tile x: its query row is copied in during this one
    auto ahead = [&]() {
      if (nidx >= 0 && has_tile(nit, x)) {
        nrow = row_of(p, nit, x, r);
        pre = true;
      }
    };
    auto prefetch = [&]() {
      if (pre) load_q(p, nrow, qb, r);
    };
    float m_used = -CUDART_INF_F, l = 0.f;
    const bool ok = two ? softmax_steps<true>(p, it, segs, ntiles, row, c, bar, lane_t, abort,
                                              m_used, l, ahead, prefetch)
                        : softmax_steps<false>(p, it, segs, ntiles, row, c, bar, lane_t, abort,
                                               m_used, l, ahead, prefetch);
    if (!ok) return;
    if (pre) {  // the next item's query rows: its S_x(0), S_x(1) run during the write-out
      cp_async_wait<0>();
      tc::fence_proxy_async();
      tc::mbar_arrive(bar + 8 * (B_Q_FULL + x));
    }
    const bool w_ok = tc::mbar_wait(bar + 8 * (B_O_DONE + x), c.nq & 1, abort, p.status, kWaitNs);
    if (__any_sync(0xffffffffu, !w_ok)) return;
    tc::fence_after();
    write_rows(p, idx, row, lane_t, m_used, l);
    c.sv += ntiles + 2;
    c.pb += ntiles;
    if (two) c.tb += ntiles;
    ++c.nq;
    ++ri;
    if (nidx < 0) return;
    if (pre) {
      idx = nidx;
      it = nit;
      row = nrow;
      continue;
    }
    // the next item is not one of tile x's (tile B, and an item with tile A only): find the next
    // one that is and copy its query rows in now
    idx = first_item(p, x, &ri);
    if (idx < 0) return;
    it = p.items[idx];
    row = row_of(p, it, x, r);
    load_q(p, row, qb, r);
    cp_async_wait<0>();
    tc::fence_proxy_async();
    tc::mbar_arrive(bar + 8 * (B_Q_FULL + x));
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    extend_tc_kernel(ExtParams p, const __grid_constant__ CUtensorMap k_map,
                     const __grid_constant__ CUtensorMap v_map) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023) & ~1023u;
  uint8_t* sp = smem_raw + (base - raw);
  const int warp = threadIdx.x >> 5;
  volatile int* abort = reinterpret_cast<volatile int*>(sp + kOffAbort);
  if (threadIdx.x == 0) {
    const uint32_t bar = base + kOffBar;
    for (int i = 0; i < kStages; ++i) {
      tc::mbar_init(bar + 8 * (B_K_FULL + i), 1);
      tc::mbar_init(bar + 8 * (B_K_FREE + i), 2);
      tc::mbar_init(bar + 8 * (B_V_FULL + i), 1);
      tc::mbar_init(bar + 8 * (B_V_FREE + i), 2);
    }
    for (int i = 0; i < 4; ++i) {
      tc::mbar_init(bar + 8 * (B_S_FULL + i), 1);
      tc::mbar_init(bar + 8 * (B_P_FULL + i), 128);
    }
    for (int x = 0; x < 2; ++x) {
      tc::mbar_init(bar + 8 * (B_O_DONE + x), 1);
      tc::mbar_init(bar + 8 * (B_Q_FULL + x), 128);
      tc::mbar_init(bar + 8 * (B_TURN + x), 128);
      tc::mbar_init(bar + 8 * (B_DRAIN + x), 1);
    }
    *abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kWarpMma) tc::alloc(base + kOffTmem, kTmemCols);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sp + kOffTmem);

  if (warp < kWarpK) {
    tc::regs_inc<kRegsSoftmax>();
    softmax_role(p, base, tmem, abort);
  } else {
    tc::regs_dec<kRegsOther>();
    if (warp < kWarpMma) {
      const bool k = warp < kWarpV;
      producer(p, warp - (k ? kWarpK : kWarpV), base, k ? &k_map : &v_map,
               base + (k ? kOffK : kOffV), k ? B_K_FULL : B_V_FULL, k ? B_K_FREE : B_V_FREE, abort);
    } else {
      if ((threadIdx.x & 31) == 0) mma_issuer(p, warp - kWarpMma, base, tmem, abort);
      __syncwarp();
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc::fence_after();
    tc::dealloc(tmem, kTmemCols);
  }
}

}  // namespace

int make_pool_map(CUtensorMap* map, const void* pool, const rx_kv_desc* d) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess) return (int)e;
    if (!fn || q != cudaDriverEntryPointSuccess) return (int)cudaErrorNotSupported;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  const cuuint64_t dims[2] = {(cuuint64_t)kHeadDim,
                              (cuuint64_t)d->pool_size * (cuuint64_t)d->num_kv_heads};
  const cuuint64_t strides[1] = {(cuuint64_t)kHeadDim * 2};
  const cuuint32_t box[2] = {64, 1};
  const cuuint32_t es[2] = {1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(pool), dims,
                            strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : (int)cudaErrorInvalidValue;
}

int launch_attn_items(const rx_kv_desc* d, const ExtItem* items, const ExtRow* rows,
                      const ExtSeg* segs, int32_t n_items, const int32_t* cta_begin,
                      int32_t n_ctas, const void* k_pool, const void* v_pool, const void* q,
                      void* o, float* lse, float* part_o, float* part_lse, int32_t* status,
                      void* stream) {
  // kernel attributes belong to the current device: set once per device (bit d of the mask)
  static std::atomic<uint64_t> attr_set{0};
  int dev = 0;
  cudaError_t de = cudaGetDevice(&dev);
  if (de != cudaSuccess) return (int)de;
  if (dev < 0 || dev >= 64) return (int)cudaErrorInvalidDevice;
  if (!((attr_set.load() >> dev) & 1)) {
    // The softmax warpgroups raise their register budget with what the other warpgroups give up;
    // that only balances when every thread starts with exactly kRegsLaunch registers (with fewer,
    // the raise would wait for registers that never come), so any other build is refused.
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, extend_tc_kernel);
    if (e != cudaSuccess) return (int)e;
    if (fa.numRegs != kRegsLaunch) return (int)cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(extend_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmem);
    if (e != cudaSuccess) return (int)e;
    attr_set.fetch_or(1ull << dev);
  }
  if (n_items == 0) return 0;
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
  p.items = items;
  p.rows = rows;
  p.segs = segs;
  p.pool_size = d->pool_size;
  p.status = status;
  p.part_o = part_o;
  p.part_lse = part_lse;
  CUtensorMap k_map, v_map;
  int e = make_pool_map(&k_map, k_pool, d);
  if (!e) e = make_pool_map(&v_map, v_pool, d);
  if (e) return e;
  p.oob_row = (int32_t)(d->pool_size * d->num_kv_heads);
  p.n_items = n_items;
  p.cta_begin = cta_begin;
  p.o32 = (reinterpret_cast<uintptr_t>(o) & 31u) == 0;
  // one persistent CTA per SM (a CTA fills an SM's shared memory), at most one per item; with
  // per-CTA lists, one CTA per list (a plan made for a GPU with more SMs still runs: its extra
  // CTAs start as others finish)
  int grid = n_ctas;
  if (!cta_begin) {
    int n_sm = 0;
    const cudaError_t ce = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
    if (ce != cudaSuccess) return (int)ce;
    grid = n_items < n_sm ? n_items : n_sm;
  }
  if (grid <= 0) return 0;
  extend_tc_kernel<<<grid, kThreads, kSmem, (cudaStream_t)stream>>>(p, k_map, v_map);
  return (int)cudaGetLastError();
}

int launch_extend(const rx_kv_desc* d, const PlanHeader* h, const void* k_pool,
                  const void* v_pool, const void* q, void* o, float* lse, void* ws,
                  void* stream) {
  uint8_t* base = static_cast<uint8_t*>(ws);
  const ExtItem* items = reinterpret_cast<const ExtItem*>(base + h->off_items);
  const ExtRow* rows = reinterpret_cast<const ExtRow*>(base + h->off_rows);
  const ExtSeg* segs = reinterpret_cast<const ExtSeg*>(base + h->off_segs);
  int32_t* status = reinterpret_cast<int32_t*>(base + offsetof(PlanHeader, status));
  if (h->ext_kernel == RX_EXTEND_PAIR)
    return launch_extend_pair(d, items, rows, segs, h->n_items, k_pool, v_pool, q, o, lse, status,
                              stream);
  return launch_attn_items(d, items, rows, segs, h->n_items,
                           reinterpret_cast<const int32_t*>(base + h->off_cta), h->n_ctas, k_pool,
                           v_pool, q, o, lse, nullptr, nullptr, status, stream);
}

}  // namespace rx
