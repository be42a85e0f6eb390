// Internal tables shared by the host planner (rx_api.cpp) and the kernels (*.cu).
#pragma once
#include <cuda.h>
#include <stddef.h>
#include <stdint.h>

#include "rx.h"

namespace rx {

constexpr int kHeadDim = 128;
constexpr uint32_t kPlanMagic = 0x52585031u;  // "RXP1"

// ---------------------------------------------------------------------------------------------
// Decode.  A work item reads keys [k_begin, k_end) of one table row, for a block of KV heads, and
// scores them against up to 64 query rows (n_tok requests x gq query heads per KV head).  Items of
// a group's shared prefix carry all members (or a tile of them); items of a request's own keys
// carry that request alone.  Each item leaves normalised partial outputs + base-2 LSE per (KV head,
// row); the merge pass combines a request's partials.
// Tilings ("kinds"): warps of a 256-thread CTA map to (KV head in block, 16-row m-tile).
//   kind 0: 1 m-tile  x 8 heads, 16 keys per stage
//   kind 1: 2 m-tiles x 4 heads, 32 keys per stage
//   kind 2: 4 m-tiles x 2 heads, 64 keys per stage
// Every kind stages 128 (head, key) rows of K and of V per pipeline stage (64 KiB).
// ---------------------------------------------------------------------------------------------
struct DecItem {
  int32_t kind;
  int32_t head_block;   // KV heads [head_block*HB, head_block*HB + HB)
  int32_t kv_row;       // req_to_token row giving the slots
  int32_t k_begin;
  int32_t k_end;
  int32_t row_begin;    // first entry in dec_rows (batch indices of the item's requests)
  int32_t n_tok;        // requests in the item
  int32_t part;         // partial-row base of the item's work unit (all KV heads)
};

struct DecMergeRef {    // one partial of a request
  int32_t part;         // work unit base
  int32_t rows_real;    // n_tok * gq of that unit
  int32_t row;          // the request's first row in the unit (token index * gq)
  int32_t pad;
};

constexpr int kDecMaxKeysPerItem = 2048;
constexpr int kDecStages = 3;
constexpr int kDecRows = 128;                              // (head, key) rows per stage
constexpr int kDecStageBytes = 2 * kDecRows * kHeadDim * 2;   // K + V, 128 rows each
constexpr size_t kDecSmemBytes = (size_t)kDecStages * kDecStageBytes + kDecMaxKeysPerItem * 4;

// ---------------------------------------------------------------------------------------------
// Extend.  A row tile holds up to 128 query rows (new tokens x gq query heads of one KV head); a
// work item pairs two row tiles with one list of key segments.  Segment owner -1 is visible to
// every row (a shared prefix); owner r is visible only to rows of request r, and only keys at
// positions < the row's limit.
// ---------------------------------------------------------------------------------------------
struct ExtRow {         // one new token
  int32_t q_row;        // row in q / o / lse
  int32_t kmax;         // keys at positions >= kmax are masked (prefix_len + i + 1)
  int32_t owner;        // batch index of the request
  int32_t pad;
};

struct ExtSeg {
  int32_t kv_row;
  int32_t k_begin;
  int32_t k_end;
  int32_t owner;        // -1 = all rows of the item
};

// Keys per step of the tensor-core attention kernel of decode shared-prefix units (one CTA), and
// of the extend kernel that runs on a pair of SMs.
constexpr int kAttnKeys = 64;
constexpr int kPairKeys = 128;

// Two row tiles (A, B) of the same KV head that walk the same key segments: every K/V step feeds
// 256 query rows.  Tile B may be empty (n_tok[1] == 0: the CTA runs tile A alone).  The same
// kernel serves a decode plan's shared-prefix units with many query rows: its rows are then
// decode requests, and each tile writes fp32 partial rows part[x] + r (row r = token * gq + g)
// for the decode merge instead of final outputs.
struct ExtItem {
  int32_t row_begin[2];  // into ext_rows
  int32_t n_tok[2];      // tokens per tile (rows = n_tok * gq <= 128)
  int32_t seg_begin;     // into ext_segs: the union of both tiles' segments
  int32_t n_seg;
  int32_t kv_head;
  int32_t n_steps;       // 64-key steps over the segments (each segment's keys rounded up)
  int32_t part[2];       // decode plans: first partial row of each tile; unused for extend
};

// Workspace layout written by rx_plan_upload: a 256-byte header, then the tables, then (decode)
// the partial outputs.  Offsets are in bytes from the workspace base and 256-byte aligned.
struct PlanHeader {
  uint32_t magic;
  int32_t kind;          // 1 = extend, 2 = decode
  int32_t status;        // device-side error word (rx_status), 0 = OK
  int32_t n_items;
  int32_t num_q_heads, num_kv_heads;
  int32_t batch;
  int32_t n_rows;        // decode: entries of dec_rows; extend: ext_rows
  int64_t off_items, off_rows, off_segs, off_merge_idx, off_merge, off_part_o, off_part_lse;
  int64_t n_part_rows;
  int64_t total_bytes;
  // decode plans: shared-prefix units run by the tensor-core attention kernel (ExtItem / ExtRow /
  // ExtSeg tables writing partial rows); n_xitems = 0 when there are none
  int64_t off_xitems, off_xrows, off_xsegs;
  int32_t n_xitems;
  int32_t ext_kernel;    // extend plans: RX_EXTEND_TILES or RX_EXTEND_PAIR
  // extend plans on the one-SM kernel: per-CTA item lists, int32 [n_ctas + 1] starts into the
  // item table (which is stored CTA by CTA); n_ctas = 0 when the items are dealt in snake order
  int64_t off_cta;
  int32_t n_ctas, pad32;
  int64_t pad[13];
};
static_assert(sizeof(PlanHeader) == 256, "header is 256 bytes");

// A second stream (and its fork / join events) on which a decode call runs its mma.sync units
// beside the tensor-core units; owned by the plan, created on the device of its first use.
// All NULL when the plan's calls need no second stream.
struct AuxStream {
  void* stream;
  void* fork;
  void* join;
};

// Launchers (defined in the .cu files).  Return cudaError_t as int.
int launch_store_kv(const rx_kv_desc* d, void* k_pool, void* v_pool, const void* k_new,
                    const void* v_new, const int32_t* slots, int64_t n, void* stream);
int launch_decode(const rx_kv_desc* d, const PlanHeader* h, const void* k_pool,
                  const void* v_pool, const void* q, void* o, float* lse, void* ws,
                  void* stream, const AuxStream* aux);
// The extend kernel on SM pairs over `n_items` items (one tile per CTA of a pair, kPairKeys-key
// steps).
int launch_extend(const rx_kv_desc* d, const PlanHeader* h, const void* k_pool,
                  const void* v_pool, const void* q, void* o, float* lse, void* ws,
                  void* stream);
int launch_extend_pair(const rx_kv_desc* d, const ExtItem* items, const ExtRow* rows,
                       const ExtSeg* segs, int32_t n_items, const void* k_pool,
                       const void* v_pool, const void* q, void* o, float* lse, int32_t* status,
                       void* stream);
// Tensor map viewing a pool as [pool_size * num_kv_heads rows, 128 bf16 columns] (row stride
// 256 bytes), boxes of 64 columns x 1 row, 128-byte swizzle: the unit of tile::gather4.
int make_pool_map(CUtensorMap* map, const void* pool, const rx_kv_desc* d);
// The tensor-core attention kernel over `n_items` items of tables in device memory; with
// part_o != nullptr every tile writes fp32 partial rows (normalised O, base-2 LSE) instead of o /
// lse.  `status` is the plan's device status word.  With `cta_begin` (device, [n_ctas + 1]) the
// grid is n_ctas CTAs and CTA k runs items cta_begin[k] .. cta_begin[k + 1] - 1; with null the
// items are dealt to one CTA per SM in snake order.
int launch_attn_items(const rx_kv_desc* d, const ExtItem* items, const ExtRow* rows,
                      const ExtSeg* segs, int32_t n_items, const int32_t* cta_begin,
                      int32_t n_ctas, const void* k_pool, const void* v_pool, const void* q,
                      void* o, float* lse, float* part_o, float* part_lse, int32_t* status,
                      void* stream);

// The plan's second stream for a decode call on the current device (created on first use); all
// NULL when the plan's calls launch a single kernel.
rx_status plan_aux_stream(const rx_plan* plan, AuxStream* out);
// Records `msg` as the calling thread's last error and returns `st`.
rx_status set_error(rx_status st, const char* msg);
// Checks a decode plan and the call's tensors for rx_decode_attn_noalloc, with the library's own
// scratch (`scratch`, `scratch_bytes`) in place of a caller workspace; on success returns the
// plan header.
rx_status plan_for_noalloc(const rx_plan* plan, const rx_kv_desc* desc, const void* k,
                           const void* v, const void* q, const void* o, const void* lse,
                           const void* scratch, size_t scratch_bytes, PlanHeader* hdr);

}  // namespace rx
