// Host radix cache and token accounting.
//
// The cache maps token sequences to the pool slots holding their KV as a radix tree (Patricia
// trie) whose edges carry runs of tokens of any length, so a long shared prefix costs one node
// (SGLang explainer, RadixAttention: radix tree; LMSYS blog translation, RadixAttention backend).
// Matching walks from the root and keeps the slots of every matched token; an edge matched only
// partly contributes its first `common` slots and ends the walk (SGLang explainer, "主要な操作:
// プレフィックスマッチング").  Inserting a finished sequence splits the edge it diverges in and
// hangs the remainder below (same section, insert).  The tree lives on the CPU.
#include <cmath>
#include <cstring>
#include <limits>
#include <memory>
#include <unordered_map>
#include <vector>

#include "rx.h"

namespace {

struct Node {
  std::vector<int32_t> tokens;  // edge label from the parent
  std::vector<int32_t> slots;   // slot of each label token
  std::unordered_map<int32_t, std::unique_ptr<Node>> children;  // keyed by first label token
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
};

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
  Node* node = &tree->root;
  int64_t pos = 0;
  while (pos < n) {
    auto it = node->children.find(tokens[pos]);
    if (it == node->children.end()) {
      auto leaf = std::make_unique<Node>();
      leaf->tokens.assign(tokens + pos, tokens + n);
      leaf->slots.assign(slots + pos, slots + n);
      node->children.emplace(tokens[pos], std::move(leaf));
      tree->tokens += n - pos;
      tree->nodes += 1;
      if (new_tokens) *new_tokens = n - pos;
      return RX_OK;
    }
    Node* child = it->second.get();
    const int64_t c = common_len(tokens + pos, n - pos, child->tokens);
    if (c < (int64_t)child->tokens.size()) {
      // split the edge: a new inner node takes the common part, the old child keeps the rest
      auto inner = std::make_unique<Node>();
      inner->tokens.assign(child->tokens.begin(), child->tokens.begin() + c);
      inner->slots.assign(child->slots.begin(), child->slots.begin() + c);
      std::unique_ptr<Node> old = std::move(it->second);
      old->tokens.erase(old->tokens.begin(), old->tokens.begin() + c);
      old->slots.erase(old->slots.begin(), old->slots.begin() + c);
      const int32_t key = old->tokens[0];
      inner->children.emplace(key, std::move(old));
      it->second = std::move(inner);
      tree->nodes += 1;
      child = it->second.get();
    }
    pos += c;
    node = child;
  }
  if (new_tokens) *new_tokens = 0;
  return RX_OK;
}

rx_status rx_radix_stats(const rx_radix* tree, int64_t* tokens, int64_t* nodes) {
  if (!tree) return RX_ERR_INVALID;
  if (tokens) *tokens = tree->tokens;
  if (nodes) *nodes = tree->nodes;
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
