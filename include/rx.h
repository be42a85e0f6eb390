/*
 * rx.h -- prefix-shared KV attention on a page-size-1 KV pool, for sm_103a (GB300).
 *
 * The operations follow the pages' statement of the problem:
 *   - the KV cache is held on the GPU in pages of ONE token, and each cached token sequence refers
 *     to the pages of its tokens (SGLang explainer "論文解説: SGLang - RadixAttention...",
 *     section RadixAttention; LMSYS blog translation, RadixAttention backend);
 *   - a new request reuses the KV of its longest cached prefix and computes only the unmatched
 *     tokens (same explainer, "主要な操作: プレフィックスマッチング");
 *   - requests that share a prefix attend to the shared-prefix KV and to their own KV in one
 *     kernel, different thread blocks taking the two parts (BatchLLM explainer
 *     "論文解説: BatchLLM - ...", section Horizontal Fusion).
 *
 * Conventions for every call
 * --------------------------
 *  Memory   All tensors are caller-owned.  Pointers marked (device) are CUDA device memory,
 *           (host) are ordinary host memory.  The library allocates no device memory: scratch
 *           ("workspace") is sized by the library and passed in by the caller (the no-allocation
 *           decode below uses a static array inside the library instead).  A plan owns a pinned
 *           host buffer through which it is uploaded.
 *  Layout   bf16 tensors, row-major, 16-byte aligned:
 *             K pool, V pool   [pool_size, num_kv_heads, head_dim]   slot-major (page = 1 token)
 *             q, o             [rows, num_q_heads, head_dim]
 *             lse              [rows, num_q_heads] float32, natural log of sum_j exp(s_j)
 *             req_to_token     [rows_of_table, stride] int32: entry (r, j) is the pool slot of
 *                              key position j of the request stored in table row r.
 *  Heads    query head h reads KV head h / (num_q_heads / num_kv_heads).
 *  Shapes   head_dim must be 128; num_q_heads / num_kv_heads in {1, 2, 4, 8}.
 *  Streams  Device work is enqueued on `stream` (a cudaStream_t, NULL = legacy default stream)
 *           and is asynchronous; calls return RX_OK once it is enqueued.
 *  Errors   Argument checks run on the host before anything is enqueued; a failed check returns
 *           its code and enqueues nothing.  rx_last_error() gives a message for the calling
 *           thread's last failure.  Kernels never trap and never wait without a bound: a device
 *           wait that runs out records RX_ERR_TIMEOUT in the workspace status word, read back with
 *           rx_read_status().
 */
#ifndef RX_H_
#define RX_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  RX_OK = 0,
  RX_ERR_INVALID = 1,      /* bad pointer, alignment, negative length, inconsistent plan */
  RX_ERR_RANGE = 2,        /* a length or index exceeds the table, pool or plan limits */
  RX_ERR_UNSUPPORTED = 3,  /* head_dim != 128, head ratio outside {1,2,4,8} */
  RX_ERR_CUDA = 4,         /* a CUDA runtime call failed (see rx_last_error) */
  RX_ERR_TIMEOUT = 5,      /* a bounded device wait ran out (reported by rx_read_status) */
  RX_ERR_WORKSPACE = 6     /* workspace missing or smaller than the plan needs */
} rx_status;

typedef void* rx_stream_t; /* a cudaStream_t */

const char* rx_status_string(int status);
const char* rx_last_error(void);

/* Shape of the KV pool and of the request -> slot table. */
typedef struct {
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;             /* must be 128 */
  float softmax_scale;          /* scores are softmax_scale * q.k */
  int64_t pool_size;            /* slots in each of the K and V pools */
  const int32_t* req_to_token;  /* (device) [req_to_token_rows, req_to_token_stride] */
  int64_t req_to_token_rows;
  int64_t req_to_token_stride;  /* elements per table row; every length is <= this */
} rx_kv_desc;

/* ---------------------------------------------------------------------------------------------
 * rx_store_kv -- write the KV of new tokens into their pool pages.
 *
 * The cache keeps each token's KV in a page of its own (SGLang explainer, RadixAttention: one
 * token per page); storing a newly computed token is a scatter into its slot:
 *   k_pool[slots[t]] = k_new[t],  v_pool[slots[t]] = v_new[t]   for t < num_tokens.
 *   k_new, v_new (device) [num_tokens, num_kv_heads, head_dim] bf16; slots (device) int32.
 * Bit-exact copy.  Slots must be distinct and in [0, pool_size); a slot outside that range is
 * skipped by the kernel (nothing is written for that token).  Duplicate slots leave one of the
 * writers' rows (unspecified which).  num_tokens == 0 is a no-op.
 * ------------------------------------------------------------------------------------------- */
rx_status rx_store_kv(const rx_kv_desc* desc, void* k_pool, void* v_pool, const void* k_new,
                      const void* v_new, const int32_t* slots, int64_t num_tokens,
                      rx_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * Plans.  Attention work is split into work items on the host from host copies of the lengths
 * (the radix-tree match that produces them runs on the CPU as well: SGLang explainer, RadixAttention
 * -- the tree is kept on the CPU).  A plan is built once per batch, uploaded into the caller's
 * device workspace once, and can then drive any number of attention calls (e.g. every layer)
 * with the same lengths.
 * ------------------------------------------------------------------------------------------- */
typedef struct rx_plan rx_plan;

rx_status rx_plan_create(rx_plan** out);
void rx_plan_destroy(rx_plan* plan);
/* Which tensor-core kernel the extend plans built on `plan` after this call run on (host; the
 * plan's existing tables are not changed).  Both compute the same attention (within the
 * extend tolerance); they differ in speed only.
 *   RX_EXTEND_TILES (default)  one SM per item: two 128-row query tiles, 64-key steps, the two
 *                              tiles' softmax and MMAs interleaved.
 *   RX_EXTEND_PAIR             two SMs per item (a cluster of two, tcgen05 cta_group::2): one
 *                              128-row tile per SM, 128-key steps, M = 256 MMAs.
 * Any other value returns RX_ERR_INVALID. */
#define RX_EXTEND_TILES 0
#define RX_EXTEND_PAIR 1
rx_status rx_plan_set_extend_kernel(rx_plan* plan, int32_t kernel);
/* Number of kernels one attention call with the built plan launches (0 for a plan without work;
 * a decode plan launches up to three: tensor-core shared-prefix units, mma.sync units, merge).
 * For a caller's and a benchmark's bookkeeping; (host). */
rx_status rx_plan_launches(const rx_plan* plan, int32_t* launches);
/* Rows of q / o / lse an attention call with the built plan reads and writes: the sum of
 * extend_len for an extend plan, the batch for a decode plan.  The calls take raw pointers and
 * cannot see the buffers' sizes: a caller checks its tensors against this (the Python binding
 * does, before every call).  (host) */
rx_status rx_plan_rows(const rx_plan* plan, int64_t* rows);
/* Bytes of device workspace the built plan needs (tables + partial results). */
rx_status rx_plan_workspace_size(const rx_plan* plan, size_t* bytes);
/* Copy the plan's tables into `workspace` (device, >= rx_plan_workspace_size bytes, 256-byte
 * aligned) with cudaMemcpyAsync on `stream`.  The tables are first copied into a pinned host
 * buffer the plan owns, so the call returns without waiting for `stream`; a later upload of the
 * same plan waits (on the host) for this copy to finish before reusing that buffer.  The plan
 * object may be rebuilt or destroyed as soon as this returns (destroying it waits for its last
 * copy). */
rx_status rx_plan_upload(const rx_plan* plan, void* workspace, size_t workspace_bytes,
                         rx_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * rx_extend_plan / rx_extend_attn -- attention of new tokens over their cached prefix plus causal
 * attention among themselves (prefill with a radix-cache hit: only the unmatched part is computed;
 * SGLang explainer, prefix matching; SGLang paper notes App. A.1).
 *
 * Request r (r < batch) owns table row req_idx[r]; its key positions 0..prefix_len[r]-1 are
 * cached and positions prefix_len[r]..prefix_len[r]+extend_len[r]-1 are its new tokens, whose KV
 * must already be stored (rx_store_kv).  Its new rows sit in q/o/lse at rows
 * cu[r]..cu[r]+extend_len[r]-1, cu = exclusive prefix sum of extend_len (requests packed in batch
 * order).  New row i attends to key positions 0..prefix_len[r]+i:
 *   o = softmax_j(scale * q.k_j) v_j,   lse = log sum_j exp(scale * q.k_j).
 * Shared prefixes: group_of_req[r] = g >= 0 declares that the first group_prefix_len[g] entries of
 * row req_idx[r] equal those of every other member of g (g < num_groups, group_prefix_len[g] <=
 * prefix_len[r]); the kernel then reads that prefix KV once for all new rows of the group.  -1 (or
 * group_of_req == NULL) declares no sharing.  The result does not depend on the grouping.
 * All arrays of rx_extend_plan are (host).  extend_len[r] == 0 is allowed; sum of extend_len must
 * be < 2^31.  batch == 0 builds a plan with no work: the attention call then enqueues nothing and
 * may be given NULL tensors.  o needs 16-byte alignment; at 32-byte alignment rows are written in
 * 32-byte pieces.
 * On the default kernel (rx_plan_set_extend_kernel) the plan deals its work items into one list
 * per SM of the calling thread's current GPU (152 where no GPU is visible); the attention call
 * launches one CTA per list, so the plan runs on any GPU, at its best on one with as many SMs.
 * ------------------------------------------------------------------------------------------- */
rx_status rx_extend_plan(rx_plan* plan, const rx_kv_desc* desc, int32_t batch,
                         const int32_t* req_idx, const int32_t* prefix_len,
                         const int32_t* extend_len, const int32_t* group_of_req,
                         int32_t num_groups, const int32_t* group_prefix_len);
rx_status rx_extend_attn(const rx_plan* plan, const rx_kv_desc* desc, const void* k_pool,
                         const void* v_pool, const void* q, void* o, float* lse,
                         void* workspace, size_t workspace_bytes, rx_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * Prefix trees (SGLang explainer, "RadixAttention: Radix Tree KV cache management"; SGLang paper
 * notes, Figure 9: tree-structured sharing).  Groups may form a forest: group_parent[g] is the
 * group whose prefix g's prefix extends, or -1 for a root (group_parent == NULL: every group is a
 * root).  Requirements: group_parent[g] < g (parents listed first), and
 * group_prefix_len[parent] <= group_prefix_len[g].  A request of group g shares the first
 * group_prefix_len[a] entries of its table row with every request of a's subtree, for each group a
 * on the path from g to its root.  Node a's own keys are positions
 * group_prefix_len[parent(a)] .. group_prefix_len[a]-1 (from 0 for a root).
 *
 * rx_extend_plan_tree: as rx_extend_plan; new rows are packed by the deepest group on a request's
 * path that holds at least two requests with new tokens, so rows that share the most keys share
 * tiles.  The result does not depend on the tree.
 * rx_decode_plan_tree: as rx_decode_plan, with each node's own keys read from HBM once for all
 * requests beneath it (one work unit per node, KV head and key chunk), each request's keys past
 * its deepest group's prefix read once for it, and all of a request's partial softmax states
 * combined by one log-sum-exp merge (cascade across the levels of the tree).
 * Arrays are (host).  Errors: RX_ERR_RANGE for a parent that is not listed first or a prefix
 * shorter than its parent's; otherwise as the one-level planners.
 * ------------------------------------------------------------------------------------------- */
rx_status rx_extend_plan_tree(rx_plan* plan, const rx_kv_desc* desc, int32_t batch,
                              const int32_t* req_idx, const int32_t* prefix_len,
                              const int32_t* extend_len, const int32_t* group_of_req,
                              int32_t num_groups, const int32_t* group_prefix_len,
                              const int32_t* group_parent);
rx_status rx_decode_plan_tree(rx_plan* plan, const rx_kv_desc* desc, int32_t batch,
                              const int32_t* req_idx, const int32_t* seq_len,
                              const int32_t* group_of_req, int32_t num_groups,
                              const int32_t* group_prefix_len, const int32_t* group_parent);

/* Number of (key, KV head) rows of the pool the built plan's kernels read, each counted once per
 * read (a shared prefix read for 16 members counts once; a prefix re-read for a second member
 * tile counts twice).  With rx_kv_desc's head size this gives the plan's K+V bytes:
 * rows * 2 * head_dim * 2.  For a tests' and a benchmark's bookkeeping; (host). */
rx_status rx_plan_key_reads(const rx_plan* plan, int64_t* rows);

/* ---------------------------------------------------------------------------------------------
 * rx_decode_plan / rx_decode_attn -- one query token per request over all of its keys, the current
 * token included (the caller stores it first).  Request b owns table row req_idx[b] and attends to
 * key positions 0..seq_len[b]-1; q/o rows are b, lse row b.
 * Horizontal fusion (BatchLLM explainer, Horizontal Fusion): for a group g (group_of_req[b] = g),
 * the first group_prefix_len[g] keys -- equal in every member's row -- are read from HBM once and
 * scored against all members' queries; each member's remaining keys are read by other thread
 * blocks of the same launch, and the partial softmax states are combined by a log-sum-exp merge.
 * seq_len[b] >= 1 and >= group_prefix_len[group_of_req[b]].  Arrays of rx_decode_plan are (host).
 * rx_decode_attn: when a plan has work for both partial kernels (tensor-core shared-prefix units
 * and mma.sync units), the call runs the mma.sync units on a second stream that the plan owns,
 * forked from and joined back to `stream` with events, so that neither kernel's last wave idles
 * the GPU.  Calls that share one plan share that stream: give callers on different streams (or
 * host threads) plans of their own, and they never wait on one another.
 * ------------------------------------------------------------------------------------------- */
rx_status rx_decode_plan(rx_plan* plan, const rx_kv_desc* desc, int32_t batch,
                         const int32_t* req_idx, const int32_t* seq_len,
                         const int32_t* group_of_req, int32_t num_groups,
                         const int32_t* group_prefix_len);
rx_status rx_decode_attn(const rx_plan* plan, const rx_kv_desc* desc, const void* k_pool,
                         const void* v_pool, const void* q, void* o, float* lse,
                         void* workspace, size_t workspace_bytes, rx_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * rx_decode_attn_noalloc -- rx_decode_attn for callers that cannot allocate device memory.
 * The pages have no counterpart: this is a convenience of the library, not a step of the method.
 *
 * Some callers have no way to allocate device memory when attention runs: a host framework that
 * hands a custom operator only its input and output buffers, or a serving runtime that owns all
 * device memory under a fixed budget and does not allow allocation while requests are in flight.
 * This call needs no workspace: the plan's tables and the partial results live in a scratch array
 * inside the library itself (RX_NOALLOC_SCRATCH_BYTES of device memory that every GPU loading the
 * library holds until the process exits).  It allocates nothing.
 *   plan      a decode plan (rx_decode_plan); it is copied into the scratch on every call, so no
 *             rx_plan_upload is needed.  A plan needing more than RX_NOALLOC_SCRATCH_BYTES (see
 *             rx_plan_workspace_size) is rejected with RX_ERR_WORKSPACE before anything runs.
 *   others    as for rx_decode_attn (caller-owned device tensors; work enqueued on `stream`).
 * The first call on a device sets up the scratch's device address for that device; make it before
 * any stream capture.  The tables are copied in from the plan's pinned staging buffer, as
 * rx_plan_upload does; like that call, it first waits (on the host) for the plan's previous copy
 * to finish.  All calls share the one array: calls whose work overlaps on the GPU (other streams,
 * other host threads) race on it and must not be issued.
 * Device-side errors (a table entry outside the pool: RX_ERR_RANGE; a bounded wait that ran out:
 * RX_ERR_TIMEOUT) are recorded in the scratch's status word, which the next call resets; read
 * them after the call and before the next one with rx_noalloc_read_status.
 * ------------------------------------------------------------------------------------------- */
#define RX_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
rx_status rx_decode_attn_noalloc(const rx_plan* plan, const rx_kv_desc* desc, const void* k_pool,
                                 const void* v_pool, const void* q, void* o, float* lse,
                                 rx_stream_t stream);
/* rx_noalloc_read_status: as rx_read_status, for the scratch of rx_decode_attn_noalloc on the
 * current device: waits for `stream`, copies the status word of the last call enqueued before it
 * into *status (host; RX_OK or the first device-side error) and clears it.  Allocates nothing. */
rx_status rx_noalloc_read_status(int32_t* status, rx_stream_t stream);
/* rx_noalloc_scratch_bytes: RX_NOALLOC_SCRATCH_BYTES as compiled into the library. */
size_t rx_noalloc_scratch_bytes(void);

/* ---------------------------------------------------------------------------------------------
 * Validation (host; a checking mode for callers and debug builds).  The attention and store
 * calls trust two contracts for speed: the shared prefixes a plan declares really are shared, and
 * the slots a store writes are distinct.  These checks verify them on the host copies of the
 * arrays the caller built (the radix match that fills the table runs on the CPU), before upload.
 * Both are O(total keys); neither touches a GPU.  Each returns RX_OK, or on the first violation
 * its code with a message (rx_last_error) naming the request / token, whose index goes to *bad
 * (nullable; -1 when all is well or the arguments themselves are wrong).
 *
 * rx_check_slots: slots[0..n) (host) for rx_store_kv.  RX_ERR_RANGE for a slot outside
 * [0, pool_size), RX_ERR_INVALID for a slot that repeats an earlier one.
 * rx_check_tables: req_to_token (host) [rows, stride] int32; request b owns row req_idx[b] and
 * reads key_len[b] keys (prefix_len + extend_len for extend, seq_len for decode); groups as for
 * rx_extend_plan_tree / rx_decode_plan_tree (group_of_req and group_parent nullable).
 * RX_ERR_RANGE: a row index, length or slot out of range, a request shorter than its group's
 * prefix, or a forest that is not parent-first with growing prefixes.  RX_ERR_INVALID: the group
 * contract is broken -- for some group g, two requests of g's subtree differ in one of the first
 * group_prefix_len[g] entries of their rows (SGLang explainer, RadixAttention: requests that
 * share a tree node share that node's KV pages; BatchLLM explainer, Global Prefix Sharing: a
 * group's common prefix is one KV context).
 * ------------------------------------------------------------------------------------------- */
rx_status rx_check_slots(const int32_t* slots, int64_t n, int64_t pool_size, int64_t* bad);
rx_status rx_check_tables(const int32_t* req_to_token, int64_t rows, int64_t stride,
                          int64_t pool_size, int32_t batch, const int32_t* req_idx,
                          const int32_t* key_len, const int32_t* group_of_req,
                          int32_t num_groups, const int32_t* group_prefix_len,
                          const int32_t* group_parent, int64_t* bad);

/* Read (synchronously, on `stream`) and clear the device status word of a workspace that a plan
 * was uploaded to.  *status receives RX_OK or the first device-side error recorded. */
rx_status rx_read_status(const void* workspace, int32_t* status, rx_stream_t stream);

/* Self-test of device-side failure detection (no counterpart on the pages).  Launches one CTA
 * that waits, with the bounded wait every tensor-core kernel uses, for an mbarrier phase that
 * nothing completes, giving up after limit_ns (0 < limit_ns <= 2 s); the wait then records
 * RX_ERR_TIMEOUT in *status (device, int32, first error wins: clear it to 0 first).  The GPU and
 * the context stay usable.  For tests of the timeout path. */
rx_status rx_selftest_wait_timeout(int32_t* status, int64_t limit_ns, rx_stream_t stream);
/* rx_selftest_pair_mma: the tensor-core steps of the extend kernel that runs on a pair of SMs (a
 * cluster of two CTAs, tcgen05 .cta_group::2), once, on one cluster, for tests:
 * s_out = q k^T and o_out = p v, fp32 [256, 128] row-major, from bf16 row-major q [256, 128]
 * (query rows), k [128, 128] (keys x head dim), v [128, 128], p [256, 128] (query rows x keys);
 * all device pointers, caller-owned.  info (device, int32[3]): [0] status word, set to RX_OK by
 * the caller (the kernel records RX_ERR_TIMEOUT there when a bounded wait ran out, and then does
 * not write the outputs); [1] and [2] the tensor-memory address each CTA of the pair was given.
 * Enqueued on `stream`. */
rx_status rx_selftest_pair_mma(const void* q, const void* k, const void* v, const void* p,
                               float* s_out, float* o_out, int32_t* info, rx_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * Host radix cache: token sequences -> pool slots, edges labelled with token runs (SGLang
 * explainer, RadixAttention: radix tree whose nodes refer to the pages of their tokens).
 * All arguments (host).  Not thread-safe per object.
 * ------------------------------------------------------------------------------------------- */
typedef struct rx_radix rx_radix;

rx_status rx_radix_create(rx_radix** out);
void rx_radix_destroy(rx_radix* tree);
/* Insert tokens[0..n) whose KV sits in slots[0..n).  Tokens already cached keep their existing
 * slots (the caller's slots for them are not referenced); *new_tokens (nullable) receives how
 * many tokens were added.  A partially matched edge is split. */
rx_status rx_radix_insert(rx_radix* tree, const int32_t* tokens, const int32_t* slots, int64_t n,
                          int64_t* new_tokens);
/* Longest cached prefix of tokens[0..n), floored to match_unit (>= 1): the tokens a prefill can
 * skip (prefix-caching comparison page: 992 of a 1,000-token prefix at unit 16, 1,000 at unit 1).
 * out_slots (nullable, capacity n) receives the slots of the saved tokens. */
rx_status rx_radix_match(const rx_radix* tree, const int32_t* tokens, int64_t n,
                         int32_t match_unit, int64_t* saved, int32_t* out_slots);
/* Number of tokens (= pool slots) the tree holds, and its node count (root excluded). */
rx_status rx_radix_stats(const rx_radix* tree, int64_t* tokens, int64_t* nodes);

/* Memory management (SGLang explainer, "LRU退避": free the least recently used leaves whose
 * reference count is 0, recursively; SGLang paper notes, §3: nodes keep reference counts, and the
 * cache shares one pool with the running requests; Figure 3 walks it through nine steps).
 * Every insert and acquire advances a logical clock and stamps the nodes on its path.
 *
 * rx_radix_acquire: rx_radix_match of tokens[0..n) at match_unit that also stamps the saved
 * prefix's nodes as used now (the edge at its end is split so exactly the saved tokens form
 * nodes) and, with lock != 0, holds them (reference count + 1) until rx_radix_release of the same
 * tokens[0..*saved).  out_slots (nullable, capacity n) receives the saved tokens' slots.
 * rx_radix_release: drops one hold on the nodes spelling tokens[0..n); RX_ERR_INVALID (nothing
 * changed) if they do not end on a node boundary or are not held.
 * rx_radix_evict: frees whole nodes -- each time the least recently used leaf not held by a
 * request (the older node first on a tie) -- until at least n_tokens slots are freed or none is
 * left to free; a parent left without children becomes a candidate.  Freed slots go to out_slots
 * (nullable; with a buffer, eviction stops before a node that would overflow `capacity`);
 * *n_freed receives their number.  Insert's note still applies: the caller's slots for tokens the
 * tree already held (the first n - new_tokens) are not taken and go back to the pool. */
rx_status rx_radix_acquire(rx_radix* tree, const int32_t* tokens, int64_t n, int32_t match_unit,
                           int32_t lock, int64_t* saved, int32_t* out_slots);
rx_status rx_radix_release(rx_radix* tree, const int32_t* tokens, int64_t n);
rx_status rx_radix_evict(rx_radix* tree, int64_t n_tokens, int32_t* out_slots, int64_t capacity,
                         int64_t* n_freed);

/* Slot pool: the pool slots that neither the cache nor a running request holds, handed out oldest
 * freed first (slots 0..pool_size-1 at creation).  rx_slot_pool_alloc takes n slots for new tokens;
 * when fewer are free and `tree` is given, it first evicts from the tree (rx_radix_evict) and
 * takes the freed slots back; RX_ERR_WORKSPACE if still short (no slot taken; evicted nodes stay
 * evicted).  rx_slot_pool_release returns slots (a finished request's tokens that the tree did
 * not take); RX_ERR_RANGE for a slot outside the pool (nothing returned).  (host) */
typedef struct rx_slot_pool rx_slot_pool;
rx_status rx_slot_pool_create(int64_t pool_size, rx_slot_pool** out);
void rx_slot_pool_destroy(rx_slot_pool* pool);
int64_t rx_slot_pool_free_count(const rx_slot_pool* pool);
rx_status rx_slot_pool_alloc(rx_slot_pool* pool, rx_radix* tree, int64_t n, int32_t* out_slots);
rx_status rx_slot_pool_release(rx_slot_pool* pool, const int32_t* slots, int64_t n);

/* Cache-aware order of a batch (SGLang paper notes, §3 cache-aware scheduling and App. A.3,
 * Theorem 3.1: with a cache holding at least the longest request, the depth-first order of the
 * batch's radix tree computes every edge once, which maximises the cache hit rate; serving the
 * longest shared prefix first approximates it).  Request r is tokens[offsets[r] .. offsets[r+1]);
 * order (capacity batch) receives a permutation of 0..batch-1: a pre-order walk of the batch's
 * radix tree, children by first token, each node's ending requests in batch order.  (host) */
rx_status rx_dfs_order(const int32_t* tokens, const int64_t* offsets, int32_t batch,
                       int32_t* order);

/* BatchLLM group formation (BatchLLM explainer, Global Prefix Sharing, merge criterion): one-level
 * groups for a batch from its radix tree.  gain(c') = (leaves(c') - 1) * tokens(c'), with leaves =
 * requests in the subtree and tokens = the node's own tokens; a node c' below a group's node c
 * starts a group of its own when gain(c') > tokens(c) (the penalty).  Reading (the page leaves
 * the merge step open): groups start at the root's children holding >= 2 requests, the rule is
 * applied recursively at every group's node, a request belongs to the deepest group on its path.
 * Outputs: group_of_req[r] (-1 = no group), group_prefix_len[g] (capacity batch; nullable) =
 * tokens from the root through g's node, *num_groups -- ready for rx_extend_plan /
 * rx_decode_plan.  Request r is tokens[offsets[r] .. offsets[r+1]).  (host) */
rx_status rx_gain_groups(const int32_t* tokens, const int64_t* offsets, int32_t batch,
                         int32_t* group_of_req, int32_t* group_prefix_len, int32_t* num_groups);

/* ---------------------------------------------------------------------------------------------
 * Token accounting (host, pure functions).
 * ------------------------------------------------------------------------------------------- */
/* Tokens a prefill skips when `matched` leading tokens hit at match unit `unit`: floor to unit. */
int64_t rx_saved_tokens(int64_t matched, int32_t unit);
/* BatchLLM token-saving ratio, percent: (1 - n_processed / n_logical) * 100 (BatchLLM explainer,
 * Global Prefix Sharing, Equation 2).  Returns NaN if n_logical <= 0. */
double rx_token_saving(int64_t n_processed, int64_t n_logical);
/* Compute removed by a hit: l_prefix / (l_prefix + l_new) (SGLang explainer, RadixAttention,
 * Reduction formula).  NaN if the sum is 0. */
double rx_compute_reduction(int64_t l_prefix, int64_t l_new);

#ifdef __cplusplus
}
#endif

#endif /* RX_H_ */
