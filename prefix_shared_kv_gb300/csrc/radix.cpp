// Host radix cache and token accounting.
//
// The cache maps token sequences to the pool slots holding their KV as a radix tree (Patricia
// trie) whose edges carry runs of tokens of any length, so a long shared prefix costs one node
// (SGLang explainer, RadixAttention: radix tree; LMSYS blog translation, RadixAttention backend).
// Matching walks from the root and keeps the slots of every matched token; an edge matched only
// partly contributes its first `common` slots and ends the walk (SGLang explainer, "主要な操作:
// プレフィックスマッチング").  Inserting a finished sequence splits the edge it diverges in and
// hangs the remainder below (same section, insert).  The tree lives on the CPU.
//
// Memory management (SGLang explainer, "LRU退避"; SGLang paper notes, §3 memory management and
// Figure 3): every node records when it was last used (a logical clock that advances on each
// insert / acquire) and how many running requests hold it (reference count).  Eviction frees the
// least recently used leaf whose count is zero, then keeps going -- a parent that becomes a leaf
// is a candidate in turn -- until enough slots are free.  The slot pool hands pool slots to the
// new tokens of running requests and takes back what eviction frees: the cache and the running
// requests share one pool.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <deque>
#include <limits>
#include <memory>
#include <queue>
#include <unordered_map>
#include <vector>

#include "rx.h"

namespace {

struct Node {
  std::vector<int32_t> tokens;  // edge label from the parent
  std::vector<int32_t> slots;   // slot of each label token
  std::unordered_map<int32_t, std::unique_ptr<Node>> children;  // keyed by first label token
  Node* parent = nullptr;
  int64_t last_use = 0;         // logical clock of the last insert / acquire through the node
  int64_t id = 0;               // creation order (ties of last_use: older node first)
  int32_t ref = 0;              // running requests holding the node
};

int64_t common_len(const int32_t* a, int64_t na, const std::vector<int32_t>& b) {
  const int64_t n = std::min<int64_t>(na, (int64_t)b.size());
  int64_t i = 0;
  while (i < n && a[i] == b[i]) ++i;
  return i;
}

}  // namespace

struct rx_radix {
  Node root;
  int64_t tokens = 0;
  int64_t nodes = 0;
  int64_t clock = 0;
  int64_t next_id = 1;
};

namespace {

// Splits `child` (held in parent->children[key]) after its first c tokens: a new inner node takes
// them, with the child's use time and holders; returns the inner node.
Node* split_node(rx_radix* tree, Node* parent, int32_t key, int64_t c) {
  auto& slot = parent->children[key];
  Node* child = slot.get();
  auto inner = std::make_unique<Node>();
  inner->tokens.assign(child->tokens.begin(), child->tokens.begin() + c);
  inner->slots.assign(child->slots.begin(), child->slots.begin() + c);
  inner->parent = parent;
  inner->last_use = child->last_use;
  inner->ref = child->ref;
  inner->id = tree->next_id++;
  std::unique_ptr<Node> old = std::move(slot);
  old->tokens.erase(old->tokens.begin(), old->tokens.begin() + c);
  old->slots.erase(old->slots.begin(), old->slots.begin() + c);
  old->parent = inner.get();
  const int32_t k = old->tokens[0];
  inner->children.emplace(k, std::move(old));
  slot = std::move(inner);
  tree->nodes += 1;
  return slot.get();
}

}  // namespace

extern "C" {

rx_status rx_radix_create(rx_radix** out) {
  if (!out) return RX_ERR_INVALID;
  *out = new rx_radix();
  return RX_OK;
}

void rx_radix_destroy(rx_radix* tree) { delete tree; }

rx_status rx_radix_match(const rx_radix* tree, const int32_t* tokens, int64_t n,
                         int32_t match_unit, int64_t* saved, int32_t* out_slots) {
  if (!tree || !saved || n < 0 || (n > 0 && !tokens)) return RX_ERR_INVALID;
  if (match_unit < 1) return RX_ERR_INVALID;
  const Node* node = &tree->root;
  int64_t pos = 0;
  std::vector<int32_t> slots;
  while (pos < n) {
    auto it = node->children.find(tokens[pos]);
    if (it == node->children.end()) break;
    const Node* child = it->second.get();
    const int64_t c = common_len(tokens + pos, n - pos, child->tokens);
    if (out_slots) slots.insert(slots.end(), child->slots.begin(), child->slots.begin() + c);
    pos += c;
    if (c < (int64_t)child->tokens.size()) break;
    node = child;
  }
  const int64_t s = pos / match_unit * match_unit;
  if (out_slots && s > 0) std::memcpy(out_slots, slots.data(), (size_t)s * sizeof(int32_t));
  *saved = s;
  return RX_OK;
}

rx_status rx_radix_insert(rx_radix* tree, const int32_t* tokens, const int32_t* slots, int64_t n,
                          int64_t* new_tokens) {
  if (!tree || n < 0 || (n > 0 && (!tokens || !slots))) return RX_ERR_INVALID;
  const int64_t now = ++tree->clock;
  Node* node = &tree->root;
  int64_t pos = 0;
  while (pos < n) {
    auto it = node->children.find(tokens[pos]);
    if (it == node->children.end()) {
      auto leaf = std::make_unique<Node>();
      leaf->tokens.assign(tokens + pos, tokens + n);
      leaf->slots.assign(slots + pos, slots + n);
      leaf->parent = node;
      leaf->last_use = now;
      leaf->id = tree->next_id++;
      node->children.emplace(tokens[pos], std::move(leaf));
      tree->tokens += n - pos;
      tree->nodes += 1;
      if (new_tokens) *new_tokens = n - pos;
      return RX_OK;
    }
    Node* child = it->second.get();
    const int64_t c = common_len(tokens + pos, n - pos, child->tokens);
    // split the edge where the sequence diverges: a new inner node takes the common part
    if (c < (int64_t)child->tokens.size()) child = split_node(tree, node, tokens[pos], c);
    child->last_use = now;
    pos += c;
    node = child;
  }
  if (new_tokens) *new_tokens = 0;
  return RX_OK;
}

rx_status rx_radix_acquire(rx_radix* tree, const int32_t* tokens, int64_t n, int32_t match_unit,
                           int32_t lock, int64_t* saved, int32_t* out_slots) {
  if (!tree || !saved || n < 0 || (n > 0 && !tokens) || match_unit < 1) return RX_ERR_INVALID;
  // the floored match first (read-only walk), then split at its end and touch / hold its nodes
  int64_t matched = 0;
  rx_status st = rx_radix_match(tree, tokens, n, 1, &matched, nullptr);
  if (st) return st;
  const int64_t s = matched / match_unit * match_unit;
  const int64_t now = ++tree->clock;
  Node* node = &tree->root;
  int64_t pos = 0;
  while (pos < s) {
    Node* child = node->children.find(tokens[pos])->second.get();
    const int64_t c = std::min<int64_t>(s - pos, (int64_t)child->tokens.size());
    if (c < (int64_t)child->tokens.size()) child = split_node(tree, node, tokens[pos], c);
    child->last_use = now;
    if (lock) child->ref += 1;
    if (out_slots) std::memcpy(out_slots + pos, child->slots.data(), (size_t)c * sizeof(int32_t));
    pos += c;
    node = child;
  }
  *saved = s;
  return RX_OK;
}

rx_status rx_radix_release(rx_radix* tree, const int32_t* tokens, int64_t n) {
  if (!tree || n < 0 || (n > 0 && !tokens)) return RX_ERR_INVALID;
  std::vector<Node*> path;
  Node* node = &tree->root;
  int64_t pos = 0;
  while (pos < n) {
    auto it = node->children.find(tokens[pos]);
    if (it == node->children.end()) return RX_ERR_INVALID;
    Node* child = it->second.get();
    const int64_t c = common_len(tokens + pos, n - pos, child->tokens);
    if (c != (int64_t)child->tokens.size() || child->ref < 1) return RX_ERR_INVALID;
    path.push_back(child);
    pos += c;
    node = child;
  }
  for (Node* x : path) x->ref -= 1;
  return RX_OK;
}

rx_status rx_radix_evict(rx_radix* tree, int64_t n_tokens, int32_t* out_slots, int64_t capacity,
                         int64_t* n_freed) {
  if (!tree || !n_freed || n_tokens < 0 || capacity < 0) return RX_ERR_INVALID;
  // candidates: unheld leaves, least recently used first (older node first on a tie)
  auto later = [](const Node* a, const Node* b) {
    return a->last_use != b->last_use ? a->last_use > b->last_use : a->id > b->id;
  };
  std::priority_queue<Node*, std::vector<Node*>, decltype(later)> heap(later);
  std::vector<Node*> stack{&tree->root};
  while (!stack.empty()) {
    Node* x = stack.back();
    stack.pop_back();
    for (auto& kv : x->children) stack.push_back(kv.second.get());
    if (x != &tree->root && x->children.empty() && x->ref == 0) heap.push(x);
  }
  int64_t freed = 0;
  while (freed < n_tokens && !heap.empty()) {
    Node* x = heap.top();
    const int64_t k = (int64_t)x->slots.size();
    if (out_slots && freed + k > capacity) break;  // would not fit the caller's buffer
    heap.pop();
    if (out_slots) std::memcpy(out_slots + freed, x->slots.data(), (size_t)k * sizeof(int32_t));
    freed += k;
    Node* pa = x->parent;
    tree->tokens -= k;
    tree->nodes -= 1;
    pa->children.erase(x->tokens[0]);  // destroys x
    if (pa != &tree->root && pa->children.empty() && pa->ref == 0) heap.push(pa);
  }
  *n_freed = freed;
  return RX_OK;
}

rx_status rx_radix_stats(const rx_radix* tree, int64_t* tokens, int64_t* nodes) {
  if (!tree) return RX_ERR_INVALID;
  if (tokens) *tokens = tree->tokens;
  if (nodes) *nodes = tree->nodes;
  return RX_OK;
}

}  // extern "C"

struct rx_slot_pool {
  std::deque<int32_t> free;  // oldest freed first
  int64_t size = 0;
};

extern "C" {

rx_status rx_slot_pool_create(int64_t pool_size, rx_slot_pool** out) {
  if (!out || pool_size < 0 || pool_size > (int64_t)INT32_MAX) return RX_ERR_INVALID;
  auto* p = new rx_slot_pool();
  p->size = pool_size;
  for (int64_t i = 0; i < pool_size; ++i) p->free.push_back((int32_t)i);
  *out = p;
  return RX_OK;
}

void rx_slot_pool_destroy(rx_slot_pool* pool) { delete pool; }

int64_t rx_slot_pool_free_count(const rx_slot_pool* pool) {
  return pool ? (int64_t)pool->free.size() : -1;
}

rx_status rx_slot_pool_alloc(rx_slot_pool* pool, rx_radix* tree, int64_t n, int32_t* out_slots) {
  if (!pool || n < 0 || (n > 0 && !out_slots)) return RX_ERR_INVALID;
  if ((int64_t)pool->free.size() < n && tree) {
    std::vector<int32_t> got((size_t)tree->tokens);
    int64_t freed = 0;
    rx_status st = rx_radix_evict(tree, n - (int64_t)pool->free.size(), got.data(),
                                  (int64_t)got.size(), &freed);
    if (st) return st;
    for (int64_t i = 0; i < freed; ++i) pool->free.push_back(got[(size_t)i]);
  }
  if ((int64_t)pool->free.size() < n) return RX_ERR_WORKSPACE;
  for (int64_t i = 0; i < n; ++i) {
    out_slots[i] = pool->free.front();
    pool->free.pop_front();
  }
  return RX_OK;
}

rx_status rx_slot_pool_release(rx_slot_pool* pool, const int32_t* slots, int64_t n) {
  if (!pool || n < 0 || (n > 0 && !slots)) return RX_ERR_INVALID;
  for (int64_t i = 0; i < n; ++i) {
    if (slots[i] < 0 || slots[i] >= pool->size) return RX_ERR_RANGE;
  }
  for (int64_t i = 0; i < n; ++i) pool->free.push_back(slots[i]);
  return RX_OK;
}

// Cache-aware ordering (SGLang paper notes, §3 cache-aware scheduling and App. A.3, Theorem 3.1:
// with a cache at least as large as the longest request, running a batch in the depth-first order
// of its radix tree computes every edge's KV once, which is optimal; longest-shared-prefix-first
// approximates it online).  The batch's sequences go into a scratch radix tree (every sequence
// then ends on a node boundary); a pre-order walk, children by first token, emits the requests
// ending at each node before descending.
rx_status rx_dfs_order(const int32_t* tokens, const int64_t* offsets, int32_t batch,
                       int32_t* order) {
  if (batch < 0 || (batch > 0 && (!tokens || !offsets || !order))) return RX_ERR_INVALID;
  rx_radix tree;
  for (int32_t r = 0; r < batch; ++r) {
    const int64_t n = offsets[r + 1] - offsets[r];
    if (n < 0) return RX_ERR_INVALID;
    std::vector<int32_t> dummy((size_t)n, 0);
    rx_status st = rx_radix_insert(&tree, tokens + offsets[r], dummy.data(), n, nullptr);
    if (st) return st;
  }
  // the node each sequence ends at
  std::unordered_map<const Node*, std::vector<int32_t>> ends;
  for (int32_t r = 0; r < batch; ++r) {
    const int32_t* t = tokens + offsets[r];
    const int64_t n = offsets[r + 1] - offsets[r];
    const Node* node = &tree.root;
    int64_t pos = 0;
    while (pos < n) {
      node = node->children.find(t[pos])->second.get();
      pos += (int64_t)node->tokens.size();
    }
    ends[node].push_back(r);
  }
  int32_t k = 0;
  std::vector<const Node*> stack{&tree.root};
  while (!stack.empty()) {
    const Node* x = stack.back();
    stack.pop_back();
    auto it = ends.find(x);
    if (it != ends.end())
      for (int32_t r : it->second) order[k++] = r;
    std::vector<const Node*> kids;
    for (auto& kv : x->children) kids.push_back(kv.second.get());
    std::sort(kids.begin(), kids.end(),
              [](const Node* a, const Node* b) { return a->tokens[0] > b->tokens[0]; });
    for (const Node* c : kids) stack.push_back(c);  // smallest first token popped first
  }
  return RX_OK;
}

// BatchLLM's group formation (BatchLLM explainer, Global Prefix Sharing: "マージ判定の基準"):
// gain(c') = (leaves(c') - 1) * tokens(c') for a node c' below a group's node c; c' forms a group
// of its own (its members share the longer prefix through c') when the gain exceeds the penalty
// tokens(c).  Reading, as the explainer leaves the merge step open: groups start at the root's
// children holding at least two requests, the rule is applied recursively to every node a group
// starts at, and a request belongs to the deepest group on its path.
rx_status rx_gain_groups(const int32_t* tokens, const int64_t* offsets, int32_t batch,
                         int32_t* group_of_req, int32_t* group_prefix_len, int32_t* num_groups) {
  if (batch < 0 || !num_groups || (batch > 0 && (!tokens || !offsets || !group_of_req)))
    return RX_ERR_INVALID;
  rx_radix tree;
  for (int32_t r = 0; r < batch; ++r) {
    const int64_t n = offsets[r + 1] - offsets[r];
    if (n < 0) return RX_ERR_INVALID;
    std::vector<int32_t> dummy((size_t)n, 0);
    rx_status st = rx_radix_insert(&tree, tokens + offsets[r], dummy.data(), n, nullptr);
    if (st) return st;
  }
  // requests ending in each node's subtree (leaves(c)), and the path of each request
  std::unordered_map<const Node*, int64_t> leaves;
  std::vector<std::vector<const Node*>> paths((size_t)batch);
  for (int32_t r = 0; r < batch; ++r) {
    const int32_t* t = tokens + offsets[r];
    const int64_t n = offsets[r + 1] - offsets[r];
    const Node* node = &tree.root;
    int64_t pos = 0;
    while (pos < n) {
      node = node->children.find(t[pos])->second.get();
      pos += (int64_t)node->tokens.size();
      paths[(size_t)r].push_back(node);
      leaves[node] += 1;
    }
  }
  // nodes where a group starts, with their prefix lengths
  std::unordered_map<const Node*, int32_t> group_at;
  std::vector<int32_t> prefix;
  struct Item {
    const Node* node;
    int64_t depth;  // tokens from the root through node
  };
  std::vector<Item> todo;
  for (auto& kv : tree.root.children)
    if (leaves[kv.second.get()] >= 2)
      todo.push_back({kv.second.get(), (int64_t)kv.second->tokens.size()});
  while (!todo.empty()) {
    const Item it = todo.back();
    todo.pop_back();
    group_at[it.node] = (int32_t)prefix.size();
    prefix.push_back((int32_t)it.depth);
    // every node below it.node is a candidate c' (its path from it.node passes nodes that did
    // not split, as those keep their requests in this group)
    std::vector<Item> below;
    for (auto& kv : it.node->children)
      below.push_back({kv.second.get(), it.depth + (int64_t)kv.second->tokens.size()});
    while (!below.empty()) {
      const Item c = below.back();
      below.pop_back();
      const int64_t gain = (leaves[c.node] - 1) * (int64_t)c.node->tokens.size();
      if (leaves[c.node] >= 2 && gain > (int64_t)it.node->tokens.size()) {
        todo.push_back(c);
      } else {
        for (auto& kv : c.node->children)
          below.push_back({kv.second.get(), c.depth + (int64_t)kv.second->tokens.size()});
      }
    }
  }
  for (int32_t r = 0; r < batch; ++r) {
    int32_t g = -1;
    for (const Node* x : paths[(size_t)r]) {
      auto f = group_at.find(x);
      if (f != group_at.end()) g = f->second;
    }
    group_of_req[r] = g;
  }
  if (group_prefix_len)
    std::memcpy(group_prefix_len, prefix.data(), prefix.size() * sizeof(int32_t));
  *num_groups = (int32_t)prefix.size();
  return RX_OK;
}

int64_t rx_saved_tokens(int64_t matched, int32_t unit) {
  if (unit < 1 || matched < 0) return -1;
  return matched / unit * unit;
}

double rx_token_saving(int64_t n_processed, int64_t n_logical) {
  if (n_logical <= 0) return std::numeric_limits<double>::quiet_NaN();
  return (1.0 - (double)n_processed / (double)n_logical) * 100.0;
}

double rx_compute_reduction(int64_t l_prefix, int64_t l_new) {
  const int64_t s = l_prefix + l_new;
  if (s == 0) return std::numeric_limits<double>::quiet_NaN();
  return (double)l_prefix / (double)s;
}

}  // extern "C"
