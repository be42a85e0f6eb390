// C-ABI of the library: argument checks, the host work planners, the radix cache and the token
// accounting.  Device work is in the .cu files; this file launches nothing itself.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <limits>
#include <memory>
#include <numeric>
#include <queue>
#include <string>
#include <unordered_map>
#include <vector>

#include "rx_internal.h"

using namespace rx;

namespace {

thread_local std::string g_err;

rx_status fail(rx_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return st;
}

rx_status cuda_fail(int e, const char* what) {
  return fail(RX_ERR_CUDA, "%s: %s", what, cudaGetErrorString((cudaError_t)e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

rx_status check_desc(const rx_kv_desc* d, bool need_table) {
  if (!d) return fail(RX_ERR_INVALID, "desc is NULL");
  if (d->head_dim != kHeadDim) return fail(RX_ERR_UNSUPPORTED, "head_dim %d != 128", d->head_dim);
  if (d->num_kv_heads <= 0 || d->num_q_heads <= 0)
    return fail(RX_ERR_INVALID, "head counts must be positive");
  if (d->num_q_heads % d->num_kv_heads)
    return fail(RX_ERR_UNSUPPORTED, "num_q_heads %% num_kv_heads != 0");
  const int gq = d->num_q_heads / d->num_kv_heads;
  if (gq != 1 && gq != 2 && gq != 4 && gq != 8)
    return fail(RX_ERR_UNSUPPORTED, "head ratio %d not in {1,2,4,8}", gq);
  if (d->num_kv_heads > 256) return fail(RX_ERR_UNSUPPORTED, "num_kv_heads > 256");
  if (d->pool_size <= 0 || d->pool_size > (int64_t)INT32_MAX)
    return fail(RX_ERR_INVALID, "pool_size must be in [1, 2^31)");
  if (!(d->softmax_scale > 0.f) || !std::isfinite(d->softmax_scale))
    return fail(RX_ERR_INVALID, "softmax_scale must be finite and > 0");
  if (need_table) {
    if (!d->req_to_token) return fail(RX_ERR_INVALID, "req_to_token is NULL");
    if (d->req_to_token_rows <= 0 || d->req_to_token_stride <= 0 ||
        d->req_to_token_stride > (int64_t)INT32_MAX || d->req_to_token_rows > (int64_t)INT32_MAX)
      return fail(RX_ERR_INVALID, "bad req_to_token shape");
  }
  return RX_OK;
}

// SMs of the current device (plans are sized for it); 152 when no device can be asked
int device_sms() {
  static std::atomic<int> cached[64];
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 152;
  }
  if ((n = cached[dev].load()) > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0) {
    cached[dev].store(n);
    return n;
  }
  cudaGetLastError();
  return 152;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

// ---------------------------------------------------------------------------------------------
// Plans
// ---------------------------------------------------------------------------------------------
struct rx_plan {
  int kind = 0;  // 0 = empty, 1 = extend, 2 = decode
  int32_t ext_kernel = RX_EXTEND_TILES;  // the kernel extend plans built from now on run on
  std::vector<uint8_t> blob;  // header + tables, uploaded verbatim
  size_t ws_bytes = 0;
  int64_t key_reads = 0;  // (key, KV head) rows of the pool the kernels read
  int32_t hq = 0, hkv = 0;
  int64_t rows = 0, stride = 0, pool = 0;
  const int32_t* table = nullptr;
  // rx_plan_upload stages the blob in pinned host memory so that the copy is asynchronous for the
  // host too; `staged` records the copy, and the buffer is reused only once it has completed
  mutable void* pinned = nullptr;
  mutable size_t pinned_bytes = 0;
  mutable cudaEvent_t staged = nullptr;
  mutable int staged_dev = -1;
  mutable bool staged_pending = false;
  // decode: the second stream on which a call runs its mma.sync units beside the tensor-core
  // units, with its fork / join events; created on first use, on that call's device, and owned by
  // the plan (so callers with plans of their own never serialise on a shared stream)
  mutable cudaStream_t aux = nullptr;
  mutable cudaEvent_t aux_fork = nullptr, aux_join = nullptr;
  mutable int aux_dev = -1;
  void drop_aux() const {
    if (aux_fork) cudaEventDestroy(aux_fork);
    if (aux_join) cudaEventDestroy(aux_join);
    if (aux) cudaStreamDestroy(aux);
    aux = nullptr;
    aux_fork = aux_join = nullptr;
    aux_dev = -1;
  }
  ~rx_plan() {
    if (staged) {
      if (staged_pending) cudaEventSynchronize(staged);
      cudaEventDestroy(staged);
    }
    if (pinned) cudaFreeHost(pinned);
    drop_aux();
  }
  PlanHeader hdr() const {
    PlanHeader h;
    std::memcpy(&h, blob.data(), sizeof h);
    return h;
  }
};

namespace {

// Steps of the tensor-core attention kernel over a segment of n keys, and an item's cost in
// fourteenths of a two-tile step.  The weights are a least-squares fit of the per-CTA times of
// the extend, radix-mixed (tree and one-level), chunked-prefill and paged workloads (globaltimer
// at each CTA's entry and exit, 760 CTAs): a two-tile step 1.03 µs, a one-tile step 0.81 µs, and
// 4.9 µs per item beyond its steps (its query tiles in, its rows out, the pipelines' refill).
int32_t attn_steps(int64_t n) { return (int32_t)((n + kAttnKeys - 1) / kAttnKeys); }
int64_t attn_cost(const ExtItem& it) { return (int64_t)it.n_steps * (it.n_tok[1] > 0 ? 14 : 11); }
constexpr int64_t kItemCost = 66;

// SMs of the calling thread's current GPU, the number of per-CTA lists an extend plan for the
// one-SM kernel makes; a GB300's 152 where no GPU can be asked (plans are host work).
int32_t plan_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0)
    return n;
  (void)cudaGetLastError();
  return 152;
}
// On the SM-pair kernel an item takes steps of kPairKeys keys per segment and costs its steps
// whether or not it has a second tile (the other CTA gathers and multiplies anyway).
int32_t pair_steps(int64_t n) { return (int32_t)((n + kPairKeys - 1) / kPairKeys); }
constexpr int64_t kPairCostClass = 2;  // two steps

template <typename T>
void put(std::vector<uint8_t>& blob, int64_t off, const std::vector<T>& v) {
  if (!v.empty()) std::memcpy(blob.data() + off, v.data(), v.size() * sizeof(T));
}

void remember_desc(rx_plan* p, const rx_kv_desc* d) {
  p->hq = d->num_q_heads;
  p->hkv = d->num_kv_heads;
  p->rows = d->req_to_token_rows;
  p->stride = d->req_to_token_stride;
  p->pool = d->pool_size;
  p->table = d->req_to_token;
}

rx_status check_plan_use(const rx_plan* p, int kind, const rx_kv_desc* d, const void* k,
                         const void* v, const void* q, const void* o, const void* lse,
                         const void* ws, size_t ws_bytes) {
  if (!p) return fail(RX_ERR_INVALID, "plan is NULL");
  if (p->kind != kind)
    return fail(RX_ERR_INVALID, "plan was built for %s", p->kind == 1 ? "extend" : p->kind == 2 ? "decode" : "nothing");
  rx_status st = check_desc(d, true);
  if (st) return st;
  if (d->num_q_heads != p->hq || d->num_kv_heads != p->hkv || d->req_to_token_rows != p->rows ||
      d->req_to_token_stride != p->stride || d->pool_size != p->pool)
    return fail(RX_ERR_INVALID, "descriptor differs from the one the plan was built with");
  const PlanHeader h = p->hdr();
  if (h.n_items > 0 || h.batch > 0) {
    if (!k || !v || !q || !o || !lse) return fail(RX_ERR_INVALID, "NULL tensor pointer");
    if (!aligned16(k) || !aligned16(v) || !aligned16(q) || !aligned16(o) || !aligned16(lse))
      return fail(RX_ERR_INVALID, "tensors must be 16-byte aligned");
  }
  if (!ws) return fail(RX_ERR_WORKSPACE, "workspace is NULL");
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return fail(RX_ERR_INVALID, "workspace must be 256-byte aligned");
  if (ws_bytes < p->ws_bytes)
    return fail(RX_ERR_WORKSPACE, "workspace of %zu bytes < %zu needed", ws_bytes, p->ws_bytes);
  return RX_OK;
}

}  // namespace

rx_status rx::set_error(rx_status st, const char* msg) { return fail(st, "%s", msg); }

rx_status rx::plan_aux_stream(const rx_plan* plan, AuxStream* out) {
  out->stream = out->fork = out->join = nullptr;
  const PlanHeader h = plan->hdr();
  if (!(h.n_xitems > 0 && h.n_items > 0)) return RX_OK;  // one kernel: no second stream
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e) return cuda_fail(e, "decode: current device");
  if (plan->aux && plan->aux_dev != dev) plan->drop_aux();  // streams belong to one device
  if (!plan->aux) {
    e = cudaStreamCreateWithFlags(&plan->aux, cudaStreamNonBlocking);
    if (!e) e = cudaEventCreateWithFlags(&plan->aux_fork, cudaEventDisableTiming);
    if (!e) e = cudaEventCreateWithFlags(&plan->aux_join, cudaEventDisableTiming);
    if (e) {
      plan->drop_aux();
      return cuda_fail(e, "decode: second stream");
    }
    plan->aux_dev = dev;
  }
  out->stream = plan->aux;
  out->fork = plan->aux_fork;
  out->join = plan->aux_join;
  return RX_OK;
}

rx_status rx::plan_for_noalloc(const rx_plan* plan, const rx_kv_desc* desc, const void* k,
                               const void* v, const void* q, const void* o, const void* lse,
                               const void* scratch, size_t scratch_bytes, PlanHeader* hdr) {
  if (plan && plan->kind == 2 && plan->ws_bytes > scratch_bytes)
    return fail(RX_ERR_WORKSPACE,
                "rx_decode_attn_noalloc: the plan needs %zu bytes of scratch, the library holds "
                "%zu; use rx_decode_attn with a workspace for batches this large",
                plan->ws_bytes, scratch_bytes);
  rx_status st = check_plan_use(plan, 2, desc, k, v, q, o, lse, scratch, scratch_bytes);
  if (st) return st;
  *hdr = plan->hdr();
  return RX_OK;
}

extern "C" {

const char* rx_status_string(int s) {
  switch (s) {
    case RX_OK: return "ok";
    case RX_ERR_INVALID: return "invalid argument";
    case RX_ERR_RANGE: return "out of range";
    case RX_ERR_UNSUPPORTED: return "unsupported shape";
    case RX_ERR_CUDA: return "CUDA error";
    case RX_ERR_TIMEOUT: return "device wait timed out";
    case RX_ERR_WORKSPACE: return "workspace too small";
    default: return "unknown status";
  }
}

const char* rx_last_error(void) { return g_err.c_str(); }

rx_status rx_store_kv(const rx_kv_desc* desc, void* k_pool, void* v_pool, const void* k_new,
                      const void* v_new, const int32_t* slots, int64_t num_tokens,
                      rx_stream_t stream) {
  rx_status st = check_desc(desc, false);
  if (st) return st;
  if (num_tokens < 0) return fail(RX_ERR_INVALID, "num_tokens < 0");
  if (num_tokens == 0) return RX_OK;
  if (!k_pool || !v_pool || !k_new || !v_new || !slots)
    return fail(RX_ERR_INVALID, "NULL pointer");
  if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(k_new) || !aligned16(v_new))
    return fail(RX_ERR_INVALID, "K/V pointers must be 16-byte aligned");
  if (num_tokens > (int64_t)INT32_MAX) return fail(RX_ERR_RANGE, "num_tokens >= 2^31");
  const int e = launch_store_kv(desc, k_pool, v_pool, k_new, v_new, slots, num_tokens, stream);
  return e ? cuda_fail(e, "store_kv launch") : RX_OK;
}

rx_status rx_plan_create(rx_plan** out) {
  if (!out) return fail(RX_ERR_INVALID, "out is NULL");
  *out = new rx_plan();
  return RX_OK;
}

void rx_plan_destroy(rx_plan* plan) { delete plan; }

rx_status rx_plan_set_extend_kernel(rx_plan* plan, int32_t kernel) {
  if (!plan) return fail(RX_ERR_INVALID, "plan is NULL");
  if (kernel != RX_EXTEND_TILES && kernel != RX_EXTEND_PAIR)
    return fail(RX_ERR_INVALID, "unknown extend kernel");
  plan->ext_kernel = kernel;
  return RX_OK;
}

rx_status rx_plan_key_reads(const rx_plan* plan, int64_t* rows) {
  if (!plan || !rows) return fail(RX_ERR_INVALID, "NULL argument");
  if (!plan->kind) return fail(RX_ERR_INVALID, "plan has not been built");
  *rows = plan->key_reads;
  return RX_OK;
}

rx_status rx_plan_rows(const rx_plan* plan, int64_t* rows) {
  if (!plan || !rows) return fail(RX_ERR_INVALID, "NULL argument");
  if (!plan->kind) return fail(RX_ERR_INVALID, "plan has not been built");
  const PlanHeader h = plan->hdr();
  *rows = plan->kind == 1 ? h.n_rows : h.batch;  // extend: one row per new token
  return RX_OK;
}

rx_status rx_plan_launches(const rx_plan* plan, int32_t* launches) {
  if (!plan || !launches) return fail(RX_ERR_INVALID, "NULL argument");
  if (!plan->kind) return fail(RX_ERR_INVALID, "plan has not been built");
  const PlanHeader h = plan->hdr();
  // the same conditions the launchers test: extend -- the tensor-core kernel when there are
  // items; decode -- the tensor-core kernel for its shared-prefix units, the mma.sync partial
  // kernel for the others, and the merge whenever there are requests
  *launches = plan->kind == 1 ? (h.n_items > 0)
                              : (h.n_xitems > 0) + (h.n_items > 0) + (h.batch > 0);
  return RX_OK;
}

rx_status rx_plan_workspace_size(const rx_plan* plan, size_t* bytes) {
  if (!plan || !bytes) return fail(RX_ERR_INVALID, "NULL argument");
  if (!plan->kind) return fail(RX_ERR_INVALID, "plan has not been built");
  *bytes = plan->ws_bytes;
  return RX_OK;
}

rx_status rx_plan_upload(const rx_plan* plan, void* workspace, size_t workspace_bytes,
                         rx_stream_t stream) {
  if (!plan || !plan->kind) return fail(RX_ERR_INVALID, "plan has not been built");
  if (!workspace) return fail(RX_ERR_WORKSPACE, "workspace is NULL");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(RX_ERR_INVALID, "workspace must be 256-byte aligned");
  if (workspace_bytes < plan->ws_bytes)
    return fail(RX_ERR_WORKSPACE, "workspace of %zu bytes < %zu needed", workspace_bytes,
                plan->ws_bytes);
  // the previous upload's copy out of the staging buffer must be done before it is overwritten
  cudaError_t e = cudaSuccess;
  if (plan->staged_pending) {
    e = cudaEventSynchronize(plan->staged);
    if (e) return cuda_fail(e, "plan upload");
    plan->staged_pending = false;
  }
  const size_t n = plan->blob.size();
  if (plan->pinned_bytes < n) {
    if (plan->pinned) cudaFreeHost(plan->pinned);
    plan->pinned = nullptr;
    plan->pinned_bytes = 0;
    e = cudaHostAlloc(&plan->pinned, n, cudaHostAllocPortable);
    if (e) return cuda_fail(e, "plan upload: pinned staging buffer");
    plan->pinned_bytes = n;
  }
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e) return cuda_fail(e, "plan upload");
  if (plan->staged && plan->staged_dev != dev) {  // events belong to one device
    cudaEventDestroy(plan->staged);
    plan->staged = nullptr;
  }
  if (!plan->staged) {
    e = cudaEventCreateWithFlags(&plan->staged, cudaEventDisableTiming);
    if (e) return cuda_fail(e, "plan upload");
    plan->staged_dev = dev;
  }
  std::memcpy(plan->pinned, plan->blob.data(), n);
  e = cudaMemcpyAsync(workspace, plan->pinned, n, cudaMemcpyHostToDevice, (cudaStream_t)stream);
  if (e) return cuda_fail(e, "plan upload");
  e = cudaEventRecord(plan->staged, (cudaStream_t)stream);
  if (e) return cuda_fail(e, "plan upload");
  plan->staged_pending = true;
  return RX_OK;
}

// ---------------------------------------------------------------------------------------------
// Validates a group forest: parents listed first, a prefix at least as long as its parent's.
rx_status check_tree(int32_t num_groups, const int32_t* group_prefix_len,
                     const int32_t* group_parent) {
  for (int g = 0; g < num_groups; ++g) {
    if (group_prefix_len[g] < 0) return fail(RX_ERR_RANGE, "group_prefix_len[%d] < 0", g);
    if (!group_parent) continue;
    const int pa = group_parent[g];
    if (pa < -1 || pa >= g)
      return fail(RX_ERR_RANGE, "group_parent[%d] = %d: parents must be listed first", g, pa);
    if (pa >= 0 && group_prefix_len[pa] > group_prefix_len[g])
      return fail(RX_ERR_RANGE, "group_prefix_len[%d] < its parent's", g);
  }
  return RX_OK;
}

// Decode planner.  Work units: (group node, member tile, chunk of the node's own keys) -- a node's
// members are all requests of its subtree -- and (request, chunk of its keys past its deepest
// group's prefix); each unit becomes one item per KV-head block.  Chunk
// lengths aim at about three items' worth of bytes per SM so a longest-first launch order
// balances; partial rows are allocated per unit over all KV heads.
// ---------------------------------------------------------------------------------------------
rx_status rx_decode_plan(rx_plan* plan, const rx_kv_desc* desc, int32_t batch,
                         const int32_t* req_idx, const int32_t* seq_len,
                         const int32_t* group_of_req, int32_t num_groups,
                         const int32_t* group_prefix_len) {
  return rx_decode_plan_tree(plan, desc, batch, req_idx, seq_len, group_of_req, num_groups,
                             group_prefix_len, nullptr);
}

rx_status rx_decode_plan_tree(rx_plan* plan, const rx_kv_desc* desc, int32_t batch,
                              const int32_t* req_idx, const int32_t* seq_len,
                              const int32_t* group_of_req, int32_t num_groups,
                              const int32_t* group_prefix_len, const int32_t* group_parent) {
  if (!plan) return fail(RX_ERR_INVALID, "plan is NULL");
  rx_status st = check_desc(desc, true);
  if (st) return st;
  if (batch < 0 || num_groups < 0) return fail(RX_ERR_INVALID, "negative batch or group count");
  if (batch > 0 && (!req_idx || !seq_len)) return fail(RX_ERR_INVALID, "NULL length array");
  if (num_groups > 0 && !group_prefix_len) return fail(RX_ERR_INVALID, "group_prefix_len NULL");
  st = check_tree(num_groups, group_prefix_len, group_parent);
  if (st) return st;
  const int hkv = desc->num_kv_heads, gq = desc->num_q_heads / hkv;
  auto parent = [&](int g) { return group_parent ? group_parent[g] : -1; };
  std::vector<int> grp(batch, -1);
  for (int b = 0; b < batch; ++b) {
    if (req_idx[b] < 0 || req_idx[b] >= desc->req_to_token_rows)
      return fail(RX_ERR_RANGE, "req_idx[%d] = %d outside the table", b, req_idx[b]);
    if (seq_len[b] < 1 || seq_len[b] > desc->req_to_token_stride)
      return fail(RX_ERR_RANGE, "seq_len[%d] = %d outside [1, stride]", b, seq_len[b]);
    if (group_of_req) {
      const int g = group_of_req[b];
      if (g < -1 || g >= num_groups) return fail(RX_ERR_RANGE, "group_of_req[%d] = %d", b, g);
      if (g >= 0) {
        if (group_prefix_len[g] < 0 || group_prefix_len[g] > seq_len[b])
          return fail(RX_ERR_RANGE, "group_prefix_len[%d] = %d exceeds seq_len of member %d", g,
                      group_prefix_len[g], b);
        grp[b] = g;
      }
    }
  }
  // a node's members: every request of its subtree (batch order)
  std::vector<std::vector<int>> members(num_groups);
  for (int b = 0; b < batch; ++b)
    for (int g = grp[b]; g >= 0; g = parent(g)) members[g].push_back(b);
  auto node_lo = [&](int g) { return parent(g) >= 0 ? group_prefix_len[parent(g)] : 0; };

  struct Unit {
    int kind, kv_row, k_begin, k_end, row_begin, n_tok;
    int64_t part;
  };
  std::vector<Unit> units;
  std::vector<int32_t> rows;
  std::vector<std::vector<DecMergeRef>> refs(batch);
  int64_t npart = 0;
  const int max_tok = 64 / gq;
  auto kind_of_rows = [](int r) { return r <= 16 ? 0 : (r <= 32 ? 1 : 2); };
  auto hb_of = [](int kind) { return kind == 0 ? 8 : (kind == 1 ? 4 : 2); };

  // bytes of K+V per key for one KV head
  const double key_bytes = 2.0 * kHeadDim * 2;
  double total = 0;
  for (int g = 0; g < num_groups; ++g)
    if (!members[g].empty() && group_prefix_len[g] > node_lo(g))
      total += (double)(group_prefix_len[g] - node_lo(g)) * hkv * key_bytes *
               ((members[g].size() + max_tok - 1) / max_tok);
  for (int b = 0; b < batch; ++b)
    total += (double)(seq_len[b] - (grp[b] >= 0 ? group_prefix_len[grp[b]] : 0)) * hkv * key_bytes;
  // bytes of K/V per mma.sync item: about three items per SM, but no item under 1 MiB (smaller
  // ones spend more on their own start and partial write-out than on the read)
  const double target = std::min(4.0 * 1048576, std::max(1048576.0, total / (3.0 * device_sms())));

  auto chunks = [&](int len, int kind, std::vector<std::pair<int, int>>& out) {
    const int hb = std::min(hb_of(kind), hkv);
    const int nk = kDecRows / hb_of(kind);
    int max_keys = (int)(target / (hb * key_bytes));
    max_keys = std::max(64, std::min(kDecMaxKeysPerItem, max_keys));
    const int n = (len + max_keys - 1) / max_keys;
    int c = (len + n - 1) / n;
    c = (c + nk - 1) / nk * nk;
    c = std::min(c, kDecMaxKeysPerItem);
    out.clear();
    for (int k = 0; k < len; k += c) out.push_back({k, std::min(len, k + c)});
  };
  std::vector<std::pair<int, int>> ch;

  // Shared-prefix units whose stacked query rows reach 32 per KV head run on the tensor-core
  // attention kernel (128 / gq requests per tile, two tiles per item, one KV head per item, about
  // 2048-key chunks); the rest on the mma.sync kernel above.
  const bool tc_ok = (int64_t)desc->pool_size * hkv < (int64_t)INT32_MAX;
  const int tc_tok = 128 / gq;
  std::vector<ExtItem> xitems;
  std::vector<ExtRow> xrows;
  std::vector<ExtSeg> xsegs;
  int64_t key_reads = 0;
  for (int g = 0; g < num_groups; ++g) {
    const int lo = node_lo(g), hi = group_prefix_len[g];
    const auto& mem = members[g];
    if (mem.empty() || hi <= lo) continue;
    if (tc_ok && (int64_t)mem.size() * gq >= 32) {
      struct XTile {
        int row_begin, n_tok, t0;
      };
      std::vector<XTile> tiles;
      for (size_t t0 = 0; t0 < mem.size(); t0 += tc_tok) {
        const int n_tok = (int)std::min<size_t>(tc_tok, mem.size() - t0);
        tiles.push_back({(int)xrows.size(), n_tok, (int)t0});
        for (int i = 0; i < n_tok; ++i)
          xrows.push_back({mem[t0 + i], INT32_MAX, mem[t0 + i], 0});
      }
      const int n_ch = std::max(1, (hi - lo + 1024) / 2048);
      const int clen = ((hi - lo + n_ch - 1) / n_ch + 63) / 64 * 64;
      for (int c0 = lo; c0 < hi; c0 += clen) {
        const int c1 = std::min(hi, c0 + clen);
        const int seg = (int)xsegs.size();
        xsegs.push_back({req_idx[mem[0]], c0, c1, -1});
        std::vector<int64_t> part(tiles.size());
        for (size_t k = 0; k < tiles.size(); ++k) {
          part[k] = npart;
          npart += (int64_t)hkv * tiles[k].n_tok * gq;
          for (int i = 0; i < tiles[k].n_tok; ++i)
            refs[mem[tiles[k].t0 + i]].push_back(
                {(int32_t)part[k], tiles[k].n_tok * gq, i * gq, 0});
        }
        for (size_t k = 0; k < tiles.size(); k += 2) {
          const bool pair = k + 1 < tiles.size();
          for (int h = 0; h < hkv; ++h) {
            ExtItem it;
            it.row_begin[0] = tiles[k].row_begin;
            it.n_tok[0] = tiles[k].n_tok;
            it.row_begin[1] = pair ? tiles[k + 1].row_begin : 0;
            it.n_tok[1] = pair ? tiles[k + 1].n_tok : 0;
            it.seg_begin = seg;
            it.n_seg = 1;
            it.kv_head = h;
            it.n_steps = attn_steps(c1 - c0);
            it.part[0] = (int32_t)(part[k] + (int64_t)h * tiles[k].n_tok * gq);
            it.part[1] = pair ? (int32_t)(part[k + 1] + (int64_t)h * tiles[k + 1].n_tok * gq) : 0;
            xitems.push_back(it);
          }
          key_reads += (int64_t)(c1 - c0) * hkv;
        }
      }
      continue;
    }
    for (size_t t0 = 0; t0 < mem.size(); t0 += max_tok) {
      const int n_tok = (int)std::min<size_t>(max_tok, mem.size() - t0);
      const int kind = kind_of_rows(n_tok * gq);
      const int row_begin = (int)rows.size();
      for (int i = 0; i < n_tok; ++i) rows.push_back(mem[t0 + i]);
      chunks(hi - lo, kind, ch);
      for (auto& c : ch) {
        const int64_t part = npart;
        npart += (int64_t)hkv * n_tok * gq;
        units.push_back(
            {kind, req_idx[mem[t0]], lo + c.first, lo + c.second, row_begin, n_tok, part});
        for (int i = 0; i < n_tok; ++i)
          refs[mem[t0 + i]].push_back({(int32_t)part, n_tok * gq, i * gq, 0});
      }
    }
  }
  for (int b = 0; b < batch; ++b) {
    const int k0 = grp[b] >= 0 ? group_prefix_len[grp[b]] : 0;
    if (seq_len[b] <= k0) continue;
    const int row_begin = (int)rows.size();
    rows.push_back(b);
    chunks(seq_len[b] - k0, 0, ch);
    for (auto& c : ch) {
      const int64_t part = npart;
      npart += (int64_t)hkv * gq;
      units.push_back({0, req_idx[b], k0 + c.first, k0 + c.second, row_begin, 1, part});
      refs[b].push_back({(int32_t)part, gq, 0, 0});
    }
  }
  if (npart > (int64_t)INT32_MAX) return fail(RX_ERR_RANGE, "plan too large");

  std::vector<DecItem> items;
  for (const Unit& u : units) {
    const int hb = hb_of(u.kind);
    for (int h = 0; h * hb < hkv; ++h)
      items.push_back({u.kind, h, u.kv_row, u.k_begin, u.k_end, u.row_begin, u.n_tok,
                       (int32_t)u.part});
    key_reads += (int64_t)(u.k_end - u.k_begin) * hkv;
  }
  auto cost = [&](const DecItem& it) {
    return (double)(it.k_end - it.k_begin) * std::min(hb_of(it.kind), hkv);
  };
  std::stable_sort(items.begin(), items.end(),
                   [&](const DecItem& a, const DecItem& b) { return cost(a) > cost(b); });

  std::stable_sort(xitems.begin(), xitems.end(), [](const ExtItem& a, const ExtItem& b) {
    return attn_cost(a) > attn_cost(b);
  });

  std::vector<int32_t> midx(batch + 1, 0);
  std::vector<DecMergeRef> mref;
  for (int b = 0; b < batch; ++b) {
    midx[b] = (int32_t)mref.size();
    mref.insert(mref.end(), refs[b].begin(), refs[b].end());
  }
  midx[batch] = (int32_t)mref.size();

  PlanHeader h;
  std::memset(&h, 0, sizeof h);
  h.magic = kPlanMagic;
  h.kind = 2;
  h.n_items = (int32_t)items.size();
  h.num_q_heads = desc->num_q_heads;
  h.num_kv_heads = hkv;
  h.batch = batch;
  h.n_rows = (int32_t)rows.size();
  size_t off = align256(sizeof(PlanHeader));
  h.off_items = off; off = align256(off + items.size() * sizeof(DecItem));
  h.off_rows = off; off = align256(off + rows.size() * 4);
  h.off_segs = off;
  h.off_merge_idx = off; off = align256(off + midx.size() * 4);
  h.off_merge = off; off = align256(off + mref.size() * sizeof(DecMergeRef));
  h.off_xitems = off; off = align256(off + xitems.size() * sizeof(ExtItem));
  h.off_xrows = off; off = align256(off + xrows.size() * sizeof(ExtRow));
  h.off_xsegs = off; off = align256(off + xsegs.size() * sizeof(ExtSeg));
  h.n_xitems = (int32_t)xitems.size();
  const size_t tables = off;
  h.off_part_o = off; off = align256(off + (size_t)npart * kHeadDim * 4);
  h.off_part_lse = off; off = align256(off + (size_t)npart * 4);
  h.n_part_rows = npart;
  h.total_bytes = off;
  plan->blob.assign(tables, 0);
  std::memcpy(plan->blob.data(), &h, sizeof h);
  put(plan->blob, h.off_items, items);
  put(plan->blob, h.off_rows, rows);
  put(plan->blob, h.off_merge_idx, midx);
  put(plan->blob, h.off_merge, mref);
  put(plan->blob, h.off_xitems, xitems);
  put(plan->blob, h.off_xrows, xrows);
  put(plan->blob, h.off_xsegs, xsegs);
  plan->ws_bytes = off;
  plan->key_reads = key_reads;
  plan->kind = 2;
  remember_desc(plan, desc);
  return RX_OK;
}

rx_status rx_decode_attn(const rx_plan* plan, const rx_kv_desc* desc, const void* k_pool,
                         const void* v_pool, const void* q, void* o, float* lse,
                         void* workspace, size_t workspace_bytes, rx_stream_t stream) {
  rx_status st = check_plan_use(plan, 2, desc, k_pool, v_pool, q, o, lse, workspace,
                                workspace_bytes);
  if (st) return st;
  const PlanHeader h = plan->hdr();
  AuxStream aux;
  st = plan_aux_stream(plan, &aux);
  if (st) return st;
  const int e = launch_decode(desc, &h, k_pool, v_pool, q, o, lse, workspace, stream, &aux);
  return e ? cuda_fail(e, "decode launch") : RX_OK;
}

// ---------------------------------------------------------------------------------------------
// Extend planner.  The new tokens of a group's members are packed, member after member, into
// tiles of 128 / gq tokens (128 query rows per KV head).  A tile's segments: the shared prefix
// (read from the first member's row, visible to all rows) and, per member present, its keys from
// the group prefix up to its last row's causal limit.  Ungrouped requests get tiles of their own.
// One item per (tile, KV head).
// ---------------------------------------------------------------------------------------------
rx_status rx_extend_plan(rx_plan* plan, const rx_kv_desc* desc, int32_t batch,
                         const int32_t* req_idx, const int32_t* prefix_len,
                         const int32_t* extend_len, const int32_t* group_of_req,
                         int32_t num_groups, const int32_t* group_prefix_len) {
  return rx_extend_plan_tree(plan, desc, batch, req_idx, prefix_len, extend_len, group_of_req,
                             num_groups, group_prefix_len, nullptr);
}

rx_status rx_extend_plan_tree(rx_plan* plan, const rx_kv_desc* desc, int32_t batch,
                              const int32_t* req_idx, const int32_t* prefix_len,
                              const int32_t* extend_len, const int32_t* group_of_req,
                              int32_t num_groups, const int32_t* group_prefix_len,
                              const int32_t* group_parent) {
  if (!plan) return fail(RX_ERR_INVALID, "plan is NULL");
  rx_status st = check_desc(desc, true);
  if (st) return st;
  if (batch < 0 || num_groups < 0) return fail(RX_ERR_INVALID, "negative batch or group count");
  if (batch > 0 && (!req_idx || !prefix_len || !extend_len))
    return fail(RX_ERR_INVALID, "NULL length array");
  if (num_groups > 0 && !group_prefix_len) return fail(RX_ERR_INVALID, "group_prefix_len NULL");
  st = check_tree(num_groups, group_prefix_len, group_parent);
  if (st) return st;
  const int hkv = desc->num_kv_heads, gq = desc->num_q_heads / hkv;
  std::vector<int64_t> cu(batch + 1, 0);
  std::vector<int> grp(batch, -1);
  for (int b = 0; b < batch; ++b) {
    if (req_idx[b] < 0 || req_idx[b] >= desc->req_to_token_rows)
      return fail(RX_ERR_RANGE, "req_idx[%d] = %d outside the table", b, req_idx[b]);
    if (prefix_len[b] < 0 || extend_len[b] < 0)
      return fail(RX_ERR_INVALID, "negative length for request %d", b);
    if ((int64_t)prefix_len[b] + extend_len[b] > desc->req_to_token_stride)
      return fail(RX_ERR_RANGE, "prefix_len + extend_len of request %d exceeds the stride", b);
    cu[b + 1] = cu[b] + extend_len[b];
    if (group_of_req) {
      const int g = group_of_req[b];
      if (g < -1 || g >= num_groups) return fail(RX_ERR_RANGE, "group_of_req[%d] = %d", b, g);
      if (g >= 0) {
        if (group_prefix_len[g] < 0 || group_prefix_len[g] > prefix_len[b])
          return fail(RX_ERR_RANGE, "group_prefix_len[%d] = %d exceeds prefix_len of member %d",
                      g, group_prefix_len[g], b);
        grp[b] = g;
      }
    }
  }
  if (cu[batch] > (int64_t)INT32_MAX) return fail(RX_ERR_RANGE, "sum of extend_len >= 2^31");
  const int tile_tok = 128 / gq;

  std::vector<ExtRow> rows;
  std::vector<ExtSeg> segs;
  struct Tile {
    int row_begin, n_tok;
    std::vector<ExtSeg> segs;  // shared prefix (owner -1) first, then one per member present
    double cost;
  };
  // A unit is a group (all its tiles read the same prefix KV) or a lone request.
  struct Unit {
    std::vector<Tile> tiles;
    double cost = 0;
  };
  std::vector<Unit> units;

  auto emit_unit = [&](const std::vector<int>& reqs, int gp) {
    Unit un;
    const int first_row = (int)rows.size();
    for (int r : reqs)
      for (int i = 0; i < extend_len[r]; ++i)
        rows.push_back({(int32_t)(cu[r] + i), prefix_len[r] + i + 1, r, 0});
    const int n = (int)rows.size() - first_row;
    for (int t0 = 0; t0 < n; t0 += tile_tok) {
      const int nt = std::min(tile_tok, n - t0);
      Tile tl{first_row + t0, nt, {}, 0.0};
      if (gp > 0) {
        tl.segs.push_back({req_idx[reqs[0]], 0, gp, -1});
        tl.cost += (double)gp;
      }
      int i = 0;
      while (i < nt) {
        const int owner = rows[first_row + t0 + i].owner;
        int j = i;
        while (j + 1 < nt && rows[first_row + t0 + j + 1].owner == owner) ++j;
        const int kend = rows[first_row + t0 + j].kmax;  // last row's causal limit
        if (kend > gp) {
          tl.segs.push_back({req_idx[owner], gp, kend, owner});
          tl.cost += (double)(kend - gp);
        }
        i = j + 1;
      }
      un.cost += tl.cost;
      un.tiles.push_back(std::move(tl));
    }
    std::stable_sort(un.tiles.begin(), un.tiles.end(),
                     [](const Tile& a, const Tile& b) { return a.cost > b.cost; });
    units.push_back(std::move(un));
  };

  // A request's new rows go with the deepest group on its path that holds at least two requests
  // with new tokens (rows that share the most keys share tiles); the tile's shared segment is
  // that group's whole prefix, which is contiguous in every member's row.
  std::vector<int> with_new(num_groups, 0);
  for (int b = 0; b < batch; ++b)
    if (extend_len[b] > 0)
      for (int g = grp[b]; g >= 0; g = group_parent ? group_parent[g] : -1) ++with_new[g];
  std::vector<std::vector<int>> members(num_groups);
  for (int b = 0; b < batch; ++b) {
    if (extend_len[b] <= 0 || grp[b] < 0) continue;
    int g = grp[b];
    while (g >= 0 && with_new[g] < 2) g = group_parent ? group_parent[g] : -1;
    if (g >= 0)
      members[g].push_back(b);
    else
      grp[b] = -1;  // alone on its path: a unit of its own below
  }
  for (int g = 0; g < num_groups; ++g) {
    if (members[g].empty()) continue;
    if (group_prefix_len[g] > 0) {
      emit_unit(members[g], group_prefix_len[g]);
    } else {
      for (int b : members[g]) emit_unit(std::vector<int>{b}, 0);
    }
  }
  for (int b = 0; b < batch; ++b)
    if (grp[b] < 0 && extend_len[b] > 0) emit_unit(std::vector<int>{b}, 0);

  // Pair consecutive tiles of a unit (similar cost after the sort) into one item; the pair walks
  // the union of the two segment lists (same owner: the longer range).  An odd last tile is
  // paired with an empty one.
  struct Pair {
    int a, b;  // tile indices, b = -1 for none
    int seg_begin, n_seg;
  };
  std::vector<std::vector<Pair>> pairs(units.size());
  for (size_t k = 0; k < units.size(); ++k) {
    const auto& tiles = units[k].tiles;
    for (size_t i = 0; i < tiles.size(); i += 2) {
      Pair pr{(int)i, i + 1 < tiles.size() ? (int)i + 1 : -1, (int)segs.size(), 0};
      std::vector<ExtSeg> u = tiles[i].segs;
      if (pr.b >= 0)
        for (const ExtSeg& sg : tiles[pr.b].segs) {
          bool merged = false;
          for (ExtSeg& x : u)
            if (x.owner == sg.owner && x.kv_row == sg.kv_row && x.k_begin == sg.k_begin) {
              x.k_end = std::max(x.k_end, sg.k_end);
              merged = true;
              break;
            }
          if (!merged) u.push_back(sg);
        }
      segs.insert(segs.end(), u.begin(), u.end());
      pr.n_seg = (int)u.size();
      pairs[k].push_back(pr);
    }
  }

  // Launch order: largest unit first (longest-processing-time first across units); inside a
  // unit, KV head outer and pairs inner (for the one-SM kernel then sorted, stably, costliest
  // first), so the tiles that read the same prefix K/V run in the same wave and hit in L2.
  std::vector<size_t> order(units.size());
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(),
                   [&](size_t a, size_t b) { return units[a].cost > units[b].cost; });
  std::vector<ExtItem> items;
  const bool pair_kernel = plan->ext_kernel == RX_EXTEND_PAIR;
  int64_t key_reads = 0;
  for (size_t k : order)
    for (const Pair& pr : pairs[k])
      for (int i = 0; i < pr.n_seg; ++i)
        key_reads += (int64_t)(segs[pr.seg_begin + i].k_end - segs[pr.seg_begin + i].k_begin) * hkv;
  for (size_t k : order) {
    const size_t unit_first = items.size();
    for (int h = 0; h < hkv; ++h)
      for (const Pair& pr : pairs[k]) {
        const Tile& ta = units[k].tiles[pr.a];
        ExtItem it;
        it.row_begin[0] = ta.row_begin;
        it.n_tok[0] = ta.n_tok;
        it.row_begin[1] = pr.b >= 0 ? units[k].tiles[pr.b].row_begin : 0;
        it.n_tok[1] = pr.b >= 0 ? units[k].tiles[pr.b].n_tok : 0;
        it.seg_begin = pr.seg_begin;
        it.n_seg = pr.n_seg;
        it.kv_head = h;
        it.n_steps = 0;
        for (int i = 0; i < pr.n_seg; ++i) {
          const int64_t n = segs[pr.seg_begin + i].k_end - segs[pr.seg_begin + i].k_begin;
          it.n_steps += pair_kernel ? pair_steps(n) : attn_steps(n);
        }
        items.push_back(it);
      }
    // inside a unit the costliest items first (a long causal tile reads all the keys before it)
    if (!pair_kernel)
      std::stable_sort(items.begin() + unit_first, items.end(),
                       [](const ExtItem& a, const ExtItem& b) {
                         return attn_cost(a) > attn_cost(b);
                       });
  }
  if (items.size() > (size_t)INT32_MAX) return fail(RX_ERR_RANGE, "plan too large");
  std::vector<int32_t> cta_begin;
  if (pair_kernel) {
    // The pair kernel deals the list to its clusters in rounds (snake order): sorted by falling
    // cost, every cluster gets a similar total.  The sort is by cost classes two steps wide and
    // keeps the planned order (a unit's KV heads and tiles together) inside a class.
    std::stable_sort(items.begin(), items.end(), [](const ExtItem& a, const ExtItem& b) {
      return a.n_steps / kPairCostClass > b.n_steps / kPairCostClass;
    });
  } else if (!items.empty()) {
    // One list per CTA, made by list scheduling in the planned order (largest unit first; in a
    // unit, costliest item first): each item goes to the CTA whose list ends first under
    // the cost model.  A CTA runs its list in order, so items next to each other in the planned
    // order start at about the same time on different SMs -- the tiles of one unit read its
    // prefix and its causal keys while they are in L2 -- and the lists end at about the same
    // time.  The table is stored CTA by CTA.
    const int32_t G = (int32_t)std::min<int64_t>(plan_sm_count(), (int64_t)items.size());
    using Slot = std::pair<int64_t, int32_t>;  // (end of the list, CTA)
    std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> free_at;
    for (int32_t k = 0; k < G; ++k) free_at.push({0, k});
    std::vector<std::vector<int32_t>> lists(G);
    auto cost_of = [&](int32_t i) { return attn_cost(items[i]) + kItemCost; };
    for (size_t i = 0; i < items.size(); ++i) {
      const Slot s = free_at.top();
      free_at.pop();
      lists[s.second].push_back((int32_t)i);
      free_at.push({s.first + cost_of((int32_t)i), s.second});
    }
    // The lists' ends are left up to one item apart, and the last units' items are large (a
    // branch's 1,700-key tile, a long causal tile).  Balance them: while it lowers the larger of
    // the two, move from the longest list to the shortest the item whose cost best splits their
    // gap (appended at the end, so the longest list's other items only start earlier).
    std::vector<int64_t> load(G, 0);
    for (int32_t k = 0; k < G; ++k)
      for (int32_t i : lists[k]) load[k] += cost_of(i);
    for (int32_t round = 0; round < 8 * G; ++round) {
      const int32_t hi = (int32_t)(std::max_element(load.begin(), load.end()) - load.begin());
      const int32_t lo = (int32_t)(std::min_element(load.begin(), load.end()) - load.begin());
      const int64_t gap = load[hi] - load[lo];
      int64_t best_gain = 0;
      size_t best = 0;
      for (size_t j = 0; j < lists[hi].size(); ++j) {
        const int64_t c = cost_of(lists[hi][j]);
        const int64_t gain = std::min(c, gap - c);  // the longer list shortens by this much
        if (c < gap && gain > best_gain) {
          best_gain = gain;
          best = j;
        }
      }
      if (best_gain <= 0) break;
      const int32_t i = lists[hi][best];
      lists[hi].erase(lists[hi].begin() + (std::ptrdiff_t)best);
      lists[lo].push_back(i);
      load[hi] -= cost_of(i);
      load[lo] += cost_of(i);
    }
    std::vector<ExtItem> by_cta;
    by_cta.reserve(items.size());
    cta_begin.push_back(0);
    for (const auto& l : lists) {
      for (int32_t i : l) by_cta.push_back(items[i]);
      cta_begin.push_back((int32_t)by_cta.size());
    }
    items.swap(by_cta);
  }

  PlanHeader h;
  std::memset(&h, 0, sizeof h);
  h.magic = kPlanMagic;
  h.kind = 1;
  h.ext_kernel = plan->ext_kernel;
  h.n_items = (int32_t)items.size();
  h.num_q_heads = desc->num_q_heads;
  h.num_kv_heads = hkv;
  h.batch = batch;
  h.n_rows = (int32_t)rows.size();
  size_t off = align256(sizeof(PlanHeader));
  h.off_items = off; off = align256(off + items.size() * sizeof(ExtItem));
  h.off_rows = off; off = align256(off + rows.size() * sizeof(ExtRow));
  h.off_segs = off; off = align256(off + segs.size() * sizeof(ExtSeg));
  h.off_cta = off; off = align256(off + cta_begin.size() * sizeof(int32_t));
  h.n_ctas = cta_begin.empty() ? 0 : (int32_t)cta_begin.size() - 1;
  h.off_merge_idx = h.off_merge = h.off_part_o = h.off_part_lse = off;
  h.total_bytes = off;
  plan->blob.assign(off, 0);
  std::memcpy(plan->blob.data(), &h, sizeof h);
  put(plan->blob, h.off_items, items);
  put(plan->blob, h.off_rows, rows);
  put(plan->blob, h.off_segs, segs);
  put(plan->blob, h.off_cta, cta_begin);
  plan->ws_bytes = off;
  plan->key_reads = key_reads;
  plan->kind = 1;
  remember_desc(plan, desc);
  return RX_OK;
}

rx_status rx_extend_attn(const rx_plan* plan, const rx_kv_desc* desc, const void* k_pool,
                         const void* v_pool, const void* q, void* o, float* lse,
                         void* workspace, size_t workspace_bytes, rx_stream_t stream) {
  rx_status st = check_plan_use(plan, 1, desc, k_pool, v_pool, q, o, lse, workspace,
                                workspace_bytes);
  if (st) return st;
  if (desc->pool_size * desc->num_kv_heads >= (int64_t)INT32_MAX)
    return fail(RX_ERR_UNSUPPORTED, "pool_size * num_kv_heads must be < 2^31 for extend");
  const PlanHeader h = plan->hdr();
  const int e = launch_extend(desc, &h, k_pool, v_pool, q, o, lse, workspace, stream);
  return e ? cuda_fail(e, "extend launch") : RX_OK;
}

rx_status rx_read_status(const void* workspace, int32_t* status, rx_stream_t stream) {
  if (!workspace || !status) return fail(RX_ERR_INVALID, "NULL argument");
  const char* w = static_cast<const char*>(workspace) + offsetof(PlanHeader, status);
  cudaError_t e = cudaMemcpyAsync(status, w, 4, cudaMemcpyDeviceToHost, (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  if (*status != 0) {
    e = cudaMemsetAsync(const_cast<char*>(w), 0, 4, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "status clear");
  }
  return RX_OK;
}

// ---------------------------------------------------------------------------------------------
// Validation of the contracts the attention calls trust (host copies of the tables).
// ---------------------------------------------------------------------------------------------
rx_status rx_check_slots(const int32_t* slots, int64_t n, int64_t pool_size, int64_t* bad) {
  if (bad) *bad = -1;
  if (n < 0 || pool_size <= 0) return fail(RX_ERR_INVALID, "negative count or empty pool");
  if (n > 0 && !slots) return fail(RX_ERR_INVALID, "slots is NULL");
  for (int64_t t = 0; t < n; ++t)
    if (slots[t] < 0 || slots[t] >= pool_size) {
      if (bad) *bad = t;
      return fail(RX_ERR_RANGE, "slots[%lld] = %d is outside the pool [0, %lld)", (long long)t,
                  slots[t], (long long)pool_size);
    }
  // (slot, index) pairs in order: within a run of one slot the first index is the original and
  // every later one a repeat; the earliest repeat over all runs is reported
  std::vector<std::pair<int32_t, int64_t>> by(n);
  for (int64_t t = 0; t < n; ++t) by[t] = {slots[t], t};
  std::sort(by.begin(), by.end());
  int64_t rep = -1, orig = -1, run = 0;  // run: start of the current slot's run
  for (int64_t i = 1; i < n; ++i) {
    if (by[i].first != by[i - 1].first) {
      run = i;
    } else if (i == run + 1 && (rep < 0 || by[i].second < rep)) {  // a run's first repeat
      rep = by[i].second;
      orig = by[run].second;
    }
  }
  if (rep >= 0) {
    if (bad) *bad = rep;
    return fail(RX_ERR_INVALID, "slots[%lld] = %d repeats slots[%lld]", (long long)rep,
                slots[rep], (long long)orig);
  }
  return RX_OK;
}

rx_status rx_check_tables(const int32_t* req_to_token, int64_t rows, int64_t stride,
                          int64_t pool_size, int32_t batch, const int32_t* req_idx,
                          const int32_t* key_len, const int32_t* group_of_req,
                          int32_t num_groups, const int32_t* group_prefix_len,
                          const int32_t* group_parent, int64_t* bad) {
  if (bad) *bad = -1;
  if (!req_to_token || rows <= 0 || stride <= 0 || pool_size <= 0 || batch < 0 ||
      num_groups < 0)
    return fail(RX_ERR_INVALID, "bad table shape, pool size or count");
  if (batch > 0 && (!req_idx || !key_len)) return fail(RX_ERR_INVALID, "NULL length array");
  if (num_groups > 0 && !group_prefix_len) return fail(RX_ERR_INVALID, "group_prefix_len NULL");
  rx_status st = check_tree(num_groups, group_prefix_len, group_parent);
  if (st) return st;
  auto parent = [&](int g) { return group_parent ? group_parent[g] : -1; };
  auto row = [&](int b) { return req_to_token + (int64_t)req_idx[b] * stride; };
  // lengths and slots of every request
  for (int b = 0; b < batch; ++b) {
    if (bad) *bad = b;
    if (req_idx[b] < 0 || req_idx[b] >= rows)
      return fail(RX_ERR_RANGE, "req_idx[%d] = %d outside the table", b, req_idx[b]);
    if (key_len[b] < 0 || key_len[b] > stride)
      return fail(RX_ERR_RANGE, "request %d reads %d keys, table rows hold %lld", b, key_len[b],
                  (long long)stride);
    const int g = group_of_req ? group_of_req[b] : -1;
    if (g < -1 || g >= num_groups) return fail(RX_ERR_RANGE, "group_of_req[%d] = %d", b, g);
    if (g >= 0 && group_prefix_len[g] > key_len[b])
      return fail(RX_ERR_RANGE, "request %d reads %d keys, fewer than its group's prefix %d", b,
                  key_len[b], group_prefix_len[g]);
    const int32_t* r = row(b);
    for (int j = 0; j < key_len[b]; ++j)
      if (r[j] < 0 || r[j] >= pool_size)
        return fail(RX_ERR_RANGE, "request %d: key %d has slot %d outside the pool", b, j, r[j]);
  }
  // Every request holds, for each group a on its path, the same entries as a's first request
  // (in batch order, over a's subtree) on a's own keys [prefix of a's parent, prefix of a).  By
  // induction down the path, every request of a's subtree then agrees with every other on
  // [0, prefix of a): the shared prefix the planners read once.
  std::vector<int> rep(num_groups, -1);
  for (int b = 0; b < batch; ++b) {
    const int g = group_of_req ? group_of_req[b] : -1;
    for (int a = g; a >= 0; a = parent(a))
      if (rep[a] < 0) rep[a] = b;
  }
  for (int b = 0; b < batch; ++b) {
    const int g = group_of_req ? group_of_req[b] : -1;
    for (int a = g; a >= 0; a = parent(a)) {
      const int lo = parent(a) >= 0 ? group_prefix_len[parent(a)] : 0;
      const int32_t *x = row(b), *y = row(rep[a]);
      for (int j = lo; j < group_prefix_len[a]; ++j)
        if (x[j] != y[j]) {
          if (bad) *bad = b;
          return fail(RX_ERR_INVALID,
                      "request %d, key %d: slot %d differs from slot %d of request %d, the "
                      "first of group %d (a shared prefix of %d keys)",
                      b, j, x[j], y[j], rep[a], a, group_prefix_len[a]);
        }
    }
  }
  if (bad) *bad = -1;
  return RX_OK;
}

}  // extern "C"
