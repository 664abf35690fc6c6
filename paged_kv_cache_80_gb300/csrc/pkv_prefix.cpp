// Radix prefix cache over the block pool (host control plane).
//
// "KV Cache Management" (cs249r vol. 3 ch. 5), "Prefix Caching Across Turns":
//   * Table 4 / Definition 0.2: a radix tree whose nodes bind a compressed token slice
//     (prefix_tokens) to the ordered physical blocks backing it (block_ids), with children,
//     a parent, a reference count of the active requests reading through the node, and a
//     last-access stamp.
//   * "Longest prefix matching": only fully packed blocks are shared; a match is rounded
//     down to whole blocks (S_usable = floor(S_match / B) * B), the tail is recomputed.
//     The tree is therefore built over whole blocks: an edge holds a whole number of
//     blocks and children are keyed by their first block's B tokens.
//   * "Dynamic radix eviction": dormant leaves (reference count 0, no children) are
//     evicted least recently used first; evicting a leaf releases all of its blocks and
//     may turn its parent into a dormant leaf (cascading eligibility).
//   * Eq. 2: the prefix hit rate, matched prompt tokens over prompt tokens.
//
// The cache owns one reference on every block it indexes, so a finished request's blocks
// stay in HBM (dormant) after the request releases them; eviction drops that reference.
#include <algorithm>
#include <cstring>
#include <map>
#include <memory>
#include <queue>
#include <string>
#include <tuple>
#include <unordered_map>
#include <vector>

#include "pkv_internal.h"

namespace pkv {

struct PrefixNode {
  std::vector<int32_t> tokens;  // prefix_tokens: blocks.size() * B tokens
  std::vector<int32_t> blocks;  // block_ids
  std::map<std::vector<int32_t>, std::unique_ptr<PrefixNode>> children;  // keyed by first block's tokens
  PrefixNode* parent = nullptr;
  int64_t ref = 0;           // active requests whose matched path passes through this node
  uint64_t last_access = 0;  // clock of the last operation that traversed it
  uint64_t serial = 0;       // creation order (breaks LRU ties)
};

struct PrefixCache {
  Pool* pool = nullptr;
  int32_t B = 0;
  PrefixNode root;
  uint64_t clock = 0, next_serial = 1;
  std::unordered_map<int32_t, PrefixNode*> pinned;  // attached sequence -> deepest matched node
  int64_t prompt_tokens = 0, matched_tokens = 0;
};

namespace {

std::vector<int32_t> block_key(const int32_t* tokens, int64_t blk, int32_t B) {
  return std::vector<int32_t>(tokens + blk * B, tokens + (blk + 1) * B);
}

bool same_block(const int32_t* a, const int32_t* b, int32_t B) { return std::memcmp(a, b, sizeof(int32_t) * B) == 0; }

void drop_block(Pool& P, int32_t p) {
  if (--P.ref[p] == 0) P.free.push_back(p);
}

// Split `n` after its first k blocks: a new node takes the first k blocks and sits
// between n's parent and n; it inherits n's reference count and stamp (every request
// pinning n also passes through the new node).
PrefixNode* split(PrefixCache& C, PrefixNode* n, size_t k) {
  const int32_t B = C.B;
  PrefixNode* parent = n->parent;
  auto it = parent->children.find(std::vector<int32_t>(n->tokens.begin(), n->tokens.begin() + B));
  std::unique_ptr<PrefixNode> owned = std::move(it->second);
  parent->children.erase(it);
  auto up = std::make_unique<PrefixNode>();
  up->tokens.assign(n->tokens.begin(), n->tokens.begin() + k * B);
  up->blocks.assign(n->blocks.begin(), n->blocks.begin() + k);
  up->parent = parent;
  up->ref = n->ref;
  up->last_access = n->last_access;
  up->serial = C.next_serial++;
  n->tokens.erase(n->tokens.begin(), n->tokens.begin() + k * B);
  n->blocks.erase(n->blocks.begin(), n->blocks.begin() + k);
  n->parent = up.get();
  PrefixNode* u = up.get();
  u->children.emplace(std::vector<int32_t>(n->tokens.begin(), n->tokens.begin() + B), std::move(owned));
  parent->children.emplace(std::vector<int32_t>(u->tokens.begin(), u->tokens.begin() + B), std::move(up));
  return u;
}

// Longest whole-block prefix of tokens[0, nb * B) in the tree.  Returns the deepest node
// matched in full, the child matched in part (or null) and how many of its blocks matched.
struct Match {
  PrefixNode* full;
  PrefixNode* part;
  size_t part_blocks;
  int64_t blocks;
};

Match walk(PrefixCache& C, const int32_t* tokens, int64_t nb) {
  const int32_t B = C.B;
  Match m{&C.root, nullptr, 0, 0};
  while (m.blocks < nb) {
    auto it = m.full->children.find(block_key(tokens, m.blocks, B));
    if (it == m.full->children.end()) break;
    PrefixNode* c = it->second.get();
    size_t j = 1;  // the key matched the first block
    const size_t cb = c->blocks.size();
    while (j < cb && m.blocks + static_cast<int64_t>(j) < nb &&
           same_block(tokens + (m.blocks + j) * B, c->tokens.data() + j * B, B))
      ++j;
    m.blocks += static_cast<int64_t>(j);
    if (j < cb) {
      m.part = c;
      m.part_blocks = j;
      break;
    }
    m.full = c;
  }
  return m;
}

void collect_blocks(const PrefixNode* n, std::vector<int32_t>& out) {  // root .. n, in order
  std::vector<const PrefixNode*> path;
  for (; n && n->parent; n = n->parent) path.push_back(n);
  for (auto it = path.rbegin(); it != path.rend(); ++it) out.insert(out.end(), (*it)->blocks.begin(), (*it)->blocks.end());
}

void count(const PrefixNode& n, pkv_prefix_stats& s) {
  for (const auto& kv : n.children) {
    const PrefixNode& c = *kv.second;
    s.nodes += 1;
    s.blocks += static_cast<int64_t>(c.blocks.size());
    if (c.ref > 0) s.pinned_nodes += 1;
    if (c.ref == 0 && c.children.empty()) s.dormant_leaves += 1;
    count(c, s);
  }
}

void release_all(Pool& P, PrefixNode& n) {
  for (auto& kv : n.children) {
    for (int32_t b : kv.second->blocks) drop_block(P, b);
    release_all(P, *kv.second);
  }
}

PrefixCache* as_cache(pkv_prefix_cache* c) { return reinterpret_cast<PrefixCache*>(c); }
const PrefixCache* as_cache(const pkv_prefix_cache* c) { return reinterpret_cast<const PrefixCache*>(c); }

}  // namespace
}  // namespace pkv

using pkv::fail;
using pkv::PrefixCache;
using pkv::PrefixNode;

extern "C" {

int pkv_prefix_cache_create(pkv_pool* pool, pkv_prefix_cache** out) {
  pkv::clear_error();
  if (!pool || !out) return fail(PKV_ERR_INVALID_ARG, "NULL argument");
  auto* C = new PrefixCache();
  C->pool = reinterpret_cast<pkv::Pool*>(pool);
  C->B = C->pool->geo.block_size;
  C->pool->n_prefix_caches += 1;
  *out = reinterpret_cast<pkv_prefix_cache*>(C);
  return PKV_OK;
}

int pkv_prefix_cache_destroy(pkv_prefix_cache* cache) {
  pkv::clear_error();
  if (!cache) return fail(PKV_ERR_INVALID_ARG, "cache is NULL");
  PrefixCache* C = pkv::as_cache(cache);
  pkv::release_all(*C->pool, C->root);
  C->pool->n_prefix_caches -= 1;
  delete C;
  return PKV_OK;
}

int pkv_prefix_match(const pkv_prefix_cache* cache, const int32_t* tokens, int64_t n, int64_t* n_matched,
                     int32_t* block_ids) {
  pkv::clear_error();
  if (!cache || n < 0 || (n > 0 && !tokens) || !n_matched) return fail(PKV_ERR_INVALID_ARG, "bad arguments");
  PrefixCache* C = const_cast<PrefixCache*>(pkv::as_cache(cache));  // the walk does not modify
  const pkv::Match m = pkv::walk(*C, tokens, n / C->B);
  *n_matched = m.blocks * C->B;
  if (block_ids) {
    std::vector<int32_t> bl;
    pkv::collect_blocks(m.full, bl);
    if (m.part) bl.insert(bl.end(), m.part->blocks.begin(), m.part->blocks.begin() + m.part_blocks);
    std::copy(bl.begin(), bl.end(), block_ids);
  }
  return PKV_OK;
}

int pkv_prefix_attach(pkv_prefix_cache* cache, const int32_t* tokens, int64_t n, int32_t* seq, int64_t* n_matched) {
  pkv::clear_error();
  if (!cache || n < 0 || (n > 0 && !tokens) || !seq || !n_matched) return fail(PKV_ERR_INVALID_ARG, "bad arguments");
  PrefixCache* C = pkv::as_cache(cache);
  pkv::Pool& P = *C->pool;
  if (P.next_id == INT32_MAX) return fail(PKV_ERR_INVALID_ARG, "sequence ids exhausted");
  pkv::Match m = pkv::walk(*C, tokens, n / C->B);
  PrefixNode* deepest = m.part ? pkv::split(*C, m.part, m.part_blocks) : m.full;
  pkv::SeqState s;
  pkv::collect_blocks(deepest, s.table);
  for (int32_t b : s.table) P.ref[b] += 1;
  s.len = static_cast<int64_t>(s.table.size()) * C->B;
  P.seqs.push_back(std::move(s));
  *seq = P.next_id++;
  C->clock += 1;
  for (PrefixNode* x = deepest; x != &C->root; x = x->parent) {
    x->ref += 1;
    x->last_access = C->clock;
  }
  C->pinned[*seq] = deepest;
  C->prompt_tokens += n;
  C->matched_tokens += m.blocks * C->B;
  *n_matched = m.blocks * C->B;
  return PKV_OK;
}

int pkv_prefix_insert(pkv_prefix_cache* cache, int32_t seq, const int32_t* tokens, int64_t n) {
  pkv::clear_error();
  if (!cache || n < 0 || (n > 0 && !tokens)) return fail(PKV_ERR_INVALID_ARG, "bad arguments");
  PrefixCache* C = pkv::as_cache(cache);
  pkv::Pool& P = *C->pool;
  if (seq < 0 || seq >= P.next_id || P.seqs[seq].state != 0)
    return fail(PKV_ERR_INVALID_ARG, "unknown or released sequence " + std::to_string(seq));
  const pkv::SeqState& s = P.seqs[seq];
  if (s.swapped) return fail(PKV_ERR_INVALID_ARG, "sequence " + std::to_string(seq) + " is swapped out");
  if (n > s.len) return fail(PKV_ERR_INVALID_ARG, "more tokens than the sequence holds");
  const int32_t B = C->B;
  const int64_t nb = n / B;
  C->clock += 1;
  PrefixNode* node = &C->root;
  int64_t i = 0;
  while (i < nb) {
    auto it = node->children.find(pkv::block_key(tokens, i, B));
    if (it == node->children.end()) {
      auto leaf = std::make_unique<PrefixNode>();
      leaf->tokens.assign(tokens + i * B, tokens + nb * B);
      leaf->blocks.assign(s.table.begin() + i, s.table.begin() + nb);
      for (int32_t b : leaf->blocks) P.ref[b] += 1;
      leaf->parent = node;
      leaf->last_access = C->clock;
      leaf->serial = C->next_serial++;
      node->children.emplace(pkv::block_key(tokens, i, B), std::move(leaf));
      break;
    }
    PrefixNode* c = it->second.get();
    size_t j = 1;
    const size_t cb = c->blocks.size();
    while (j < cb && i + static_cast<int64_t>(j) < nb &&
           pkv::same_block(tokens + (i + j) * B, c->tokens.data() + j * B, B))
      ++j;
    if (j < cb) c = pkv::split(*C, c, j);
    c->last_access = C->clock;
    node = c;
    i += static_cast<int64_t>(j);
  }
  return PKV_OK;
}

int pkv_prefix_release(pkv_prefix_cache* cache, int32_t seq) {
  pkv::clear_error();
  if (!cache) return fail(PKV_ERR_INVALID_ARG, "cache is NULL");
  PrefixCache* C = pkv::as_cache(cache);
  auto it = C->pinned.find(seq);
  if (it == C->pinned.end()) return fail(PKV_ERR_INVALID_ARG, "sequence " + std::to_string(seq) + " holds no pins");
  PrefixNode* deepest = it->second;
  C->pinned.erase(it);
  C->clock += 1;
  for (PrefixNode* x = deepest; x != &C->root; x = x->parent) {
    x->ref -= 1;
    x->last_access = C->clock;
  }
  return PKV_OK;
}

int pkv_prefix_evict(pkv_prefix_cache* cache, int64_t target_free, int64_t* n_released) {
  pkv::clear_error();
  if (!cache || !n_released) return fail(PKV_ERR_INVALID_ARG, "bad arguments");
  PrefixCache* C = pkv::as_cache(cache);
  pkv::Pool& P = *C->pool;
  // the LRU queue of dormant leaves, oldest first (ties: older node first)
  using Key = std::tuple<uint64_t, uint64_t, PrefixNode*>;
  std::priority_queue<Key, std::vector<Key>, std::greater<Key>> lru;
  std::vector<PrefixNode*> stack{&C->root};
  while (!stack.empty()) {
    PrefixNode* x = stack.back();
    stack.pop_back();
    for (auto& kv : x->children) {
      PrefixNode* c = kv.second.get();
      if (c->ref == 0 && c->children.empty()) lru.emplace(c->last_access, c->serial, c);
      stack.push_back(c);
    }
  }
  int64_t released = 0;
  while (P.free.size() < target_free && !lru.empty()) {
    PrefixNode* leaf = std::get<2>(lru.top());
    lru.pop();
    for (int32_t b : leaf->blocks) pkv::drop_block(P, b);
    released += static_cast<int64_t>(leaf->blocks.size());
    PrefixNode* parent = leaf->parent;
    parent->children.erase(std::vector<int32_t>(leaf->tokens.begin(), leaf->tokens.begin() + C->B));  // frees leaf
    if (parent != &C->root && parent->children.empty() && parent->ref == 0)
      lru.emplace(parent->last_access, parent->serial, parent);
  }
  *n_released = released;
  return PKV_OK;
}

int pkv_prefix_get_stats(const pkv_prefix_cache* cache, pkv_prefix_stats* out) {
  pkv::clear_error();
  if (!cache || !out) return fail(PKV_ERR_INVALID_ARG, "NULL argument");
  const PrefixCache* C = pkv::as_cache(cache);
  *out = pkv_prefix_stats{};
  pkv::count(C->root, *out);
  out->prompt_tokens = C->prompt_tokens;
  out->matched_tokens = C->matched_tokens;
  return PKV_OK;
}

int pkv_prefix_export(const pkv_prefix_cache* cache, int64_t* nodes, int32_t* tokens, int32_t* blocks,
                      int64_t cap_nodes, int64_t cap_blocks) {
  pkv::clear_error();
  if (!cache || !nodes || !tokens || !blocks) return fail(PKV_ERR_INVALID_ARG, "NULL argument");
  const PrefixCache* C = pkv::as_cache(cache);
  pkv_prefix_stats st{};
  pkv::count(C->root, st);
  if (cap_nodes < st.nodes || cap_blocks < st.blocks) return fail(PKV_ERR_INVALID_ARG, "export buffers too small");
  // preorder, children in key order; row = parent row (-1 = root), blocks, ref, last_access, serial
  int64_t row = 0, boff = 0;
  std::vector<std::pair<const PrefixNode*, int64_t>> stack;
  for (auto it = C->root.children.rbegin(); it != C->root.children.rend(); ++it) stack.emplace_back(it->second.get(), -1);
  while (!stack.empty()) {
    const PrefixNode* x = stack.back().first;
    const int64_t parent_row = stack.back().second;
    stack.pop_back();
    int64_t* r = nodes + row * 5;
    r[0] = parent_row;
    r[1] = static_cast<int64_t>(x->blocks.size());
    r[2] = x->ref;
    r[3] = static_cast<int64_t>(x->last_access);
    r[4] = static_cast<int64_t>(x->serial);
    std::copy(x->blocks.begin(), x->blocks.end(), blocks + boff);
    std::copy(x->tokens.begin(), x->tokens.end(), tokens + boff * C->B);
    boff += static_cast<int64_t>(x->blocks.size());
    for (auto it = x->children.rbegin(); it != x->children.rend(); ++it) stack.emplace_back(it->second.get(), row);
    ++row;
  }
  return PKV_OK;
}

}  // extern "C"
