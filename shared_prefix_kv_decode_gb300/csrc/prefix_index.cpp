// Prefix lifecycle: a radix-tree index of cached prefixes over token-id sequences, with reference
// counts, HOT-first admission and COLD fallback.
//
// GraniKV (arXiv:2608.15584):
//  - "2 Related Work", prefix-aware serving: a radix tree indexes cached KV by token-id
//    sequences for longest-prefix reuse, and reference-counted nodes keep a cached prefix alive
//    while active requests depend on it;
//  - card page: one HOT slab per radix-tree prefix node, the same radix index for both pools;
//  - "B.10 Cross-pool admission and promotion policy": a prefix goes to HOT first and needs a
//    contiguous extent of L_p slots; when HOT has none (pool full, or free fragments too small)
//    it is placed in COLD; HOT prefixes are never demoted to make room.
//
// Readings where the pages leave a step open:
//  - a prefix is used whole: a request reuses the deepest admitted prefix whose full token
//    sequence starts its own (its L_p is that prefix's length).  Nested prefixes each own a
//    slab holding their full token range, so one request reads one contiguous slab;
//  - eviction is the radix cache's: only prefixes that no request holds (refcount 0) may go,
//    least recently used first.  Admission evicts unreferenced HOT prefixes only when releasing
//    every one of them would let the new prefix fit; it then evicts in LRU order until the
//    first-fit allocation succeeds.  Otherwise nothing is evicted and the prefix goes to COLD;
//  - "use" (the LRU clock) advances on insert, on a match that takes a reference, on acquire
//    and on release.
//
// The tree is path-compressed: every edge holds a run of tokens, a node exists only where an
// admitted prefix ends or two admitted prefixes diverge.  Prefix handles are separate from tree
// nodes and never reused, so splitting and merging edges leaves every handle valid.

#include "../../include/granikv.h"
#include "internal.h"

#include <algorithm>
#include <cstdint>
#include <map>
#include <new>
#include <unordered_map>
#include <vector>

using namespace granikv;

namespace {

struct Node {
  std::vector<int32_t> edge;       // tokens on the edge from the parent into this node
  std::map<int32_t, int32_t> kids;  // first token of the child's edge -> node id
  int32_t parent = -1;
  int32_t prefix = -1;             // prefix handle ending here, or -1
};

struct Prefix {
  int32_t node = -1;
  int32_t length = 0;
  int32_t slab = -1;  // HOT slab or -1 (COLD)
  int64_t offset = -1;
  int32_t refs = 0;
  uint64_t used = 0;  // LRU clock at last use
};

}  // namespace

struct granikv_index {
  granikv_ctx* ctx = nullptr;
  std::unordered_map<int32_t, Node> nodes;  // node 0 is the root (empty edge)
  int32_t next_node = 1;
  std::unordered_map<int32_t, Prefix> prefixes;
  int32_t next_prefix = 0;
  uint64_t clock = 0;
};

namespace {

void fill_info(const granikv_index* x, int32_t id, granikv_prefix_info* out) {
  if (!out) return;
  if (id < 0) {
    *out = granikv_prefix_info{-1, 0, -1, 0, -1};
    return;
  }
  const Prefix& p = x->prefixes.at(id);
  *out = granikv_prefix_info{id, p.length, p.slab, p.refs, p.offset};
}

// Deepest admitted prefix along tokens[0..n); -1 if none.
int32_t longest_match(const granikv_index* x, const int32_t* tokens, int32_t n) {
  int32_t cur = 0, pos = 0, best = -1;
  while (pos < n) {
    const Node& nd = x->nodes.at(cur);
    auto it = nd.kids.find(tokens[pos]);
    if (it == nd.kids.end()) break;
    const Node& kid = x->nodes.at(it->second);
    const int32_t len = (int32_t)kid.edge.size();
    if (pos + len > n || !std::equal(kid.edge.begin(), kid.edge.end(), tokens + pos)) break;
    pos += len;
    cur = it->second;
    if (kid.prefix >= 0) best = kid.prefix;
  }
  return best;
}

// Node whose path spells exactly tokens[0..n), created (splitting an edge if needed).
int32_t find_or_make_node(granikv_index* x, const int32_t* tokens, int32_t n) {
  int32_t cur = 0, pos = 0;
  while (pos < n) {
    Node& nd = x->nodes.at(cur);
    auto it = nd.kids.find(tokens[pos]);
    if (it == nd.kids.end()) {
      const int32_t id = x->next_node++;
      Node leaf;
      leaf.edge.assign(tokens + pos, tokens + n);
      leaf.parent = cur;
      nd.kids[tokens[pos]] = id;
      x->nodes.emplace(id, std::move(leaf));
      return id;
    }
    const int32_t kid_id = it->second;
    Node& kid = x->nodes.at(kid_id);
    const int32_t len = (int32_t)kid.edge.size();
    int32_t m = 0;  // tokens of the edge that match
    while (m < len && pos + m < n && kid.edge[m] == tokens[pos + m]) ++m;
    if (m == len) {
      pos += len;
      cur = kid_id;
      continue;
    }
    // split the edge after m tokens: parent -> mid (edge[0..m)) -> kid (edge[m..))
    const int32_t mid_id = x->next_node++;
    Node mid;
    mid.edge.assign(kid.edge.begin(), kid.edge.begin() + m);
    mid.parent = cur;
    mid.kids[kid.edge[m]] = kid_id;
    kid.edge.erase(kid.edge.begin(), kid.edge.begin() + m);
    kid.parent = mid_id;
    x->nodes.at(cur).kids[mid.edge[0]] = mid_id;
    x->nodes.emplace(mid_id, std::move(mid));
    pos += m;
    cur = mid_id;
  }
  return cur;
}

// Drop node id if it no longer marks a prefix end or a divergence, and repeat upwards.
void prune(granikv_index* x, int32_t id) {
  while (id != 0) {
    Node& nd = x->nodes.at(id);
    if (nd.prefix >= 0 || nd.kids.size() >= 2) return;
    const int32_t parent = nd.parent;
    Node& par = x->nodes.at(parent);
    if (nd.kids.empty()) {
      par.kids.erase(nd.edge[0]);
      x->nodes.erase(id);
      id = parent;  // the parent may now be a pass-through node
      continue;
    }
    // exactly one child: fold this node's edge into the child's
    const int32_t kid_id = nd.kids.begin()->second;
    Node& kid = x->nodes.at(kid_id);
    kid.edge.insert(kid.edge.begin(), nd.edge.begin(), nd.edge.end());
    kid.parent = parent;
    par.kids[kid.edge[0]] = kid_id;
    x->nodes.erase(id);
    return;
  }
}

void drop_prefix(granikv_index* x, int32_t id) {
  Prefix& p = x->prefixes.at(id);
  if (p.slab >= 0) granikv_hot_free(x->ctx, p.slab);
  const int32_t node = p.node;
  x->nodes.at(node).prefix = -1;
  x->prefixes.erase(id);
  prune(x, node);
}

}  // namespace

extern "C" {

granikv_status granikv_index_create(granikv_ctx* ctx, granikv_index** out) {
  if (!ctx || !out) return GRANIKV_ERR_INVALID;
  granikv_index* x = new (std::nothrow) granikv_index();
  if (!x) return GRANIKV_ERR_INVALID;
  x->ctx = ctx;
  x->nodes.emplace(0, Node{});
  *out = x;
  return GRANIKV_OK;
}

granikv_status granikv_index_destroy(granikv_index* x) {
  if (!x) return GRANIKV_ERR_INVALID;
  for (auto& kv : x->prefixes)
    if (kv.second.slab >= 0) granikv_hot_free(x->ctx, kv.second.slab);
  delete x;
  return GRANIKV_OK;
}

granikv_status granikv_index_match(granikv_index* x, const int32_t* tokens, int32_t n,
                                   int32_t acquire, granikv_prefix_info* out) {
  if (!x || n < 0 || (n > 0 && !tokens) || !out) return GRANIKV_ERR_INVALID;
  const int32_t id = longest_match(x, tokens, n);
  if (id >= 0 && acquire) {
    Prefix& p = x->prefixes.at(id);
    p.refs += 1;
    p.used = ++x->clock;
  }
  fill_info(x, id, out);
  return GRANIKV_OK;
}

granikv_status granikv_index_insert(granikv_index* x, const int32_t* tokens, int32_t n,
                                    granikv_prefix_info* out, int32_t* evicted,
                                    int32_t max_evicted, int32_t* n_evicted) {
  if (!x || !tokens || n <= 0 || max_evicted < 0) return GRANIKV_ERR_INVALID;
  if (max_evicted > 0 && !evicted) return GRANIKV_ERR_INVALID;
  // already admitted: the same prefix
  {
    int32_t cur = 0, pos = 0;
    bool exact = true;
    while (pos < n) {
      const Node& nd = x->nodes.at(cur);
      auto it = nd.kids.find(tokens[pos]);
      if (it == nd.kids.end()) {
        exact = false;
        break;
      }
      const Node& kid = x->nodes.at(it->second);
      const int32_t len = (int32_t)kid.edge.size();
      if (pos + len > n || !std::equal(kid.edge.begin(), kid.edge.end(), tokens + pos)) {
        exact = false;
        break;
      }
      pos += len;
      cur = it->second;
    }
    const int32_t hit = exact ? x->nodes.at(cur).prefix : -1;
    if (hit >= 0) {
      x->prefixes.at(hit).used = ++x->clock;
      if (n_evicted) *n_evicted = 0;
      fill_info(x, hit, out);
      return GRANIKV_OK;
    }
  }

  // HOT first.  Which unreferenced HOT prefixes would have to go, least recently used first?
  int64_t largest = 0;
  int32_t ids = 0;
  granikv_internal_hot_if_released(x->ctx, nullptr, 0, &largest, &ids);
  std::vector<int32_t> victims;  // prefix handles
  bool hot = largest >= n && ids > 0;
  if (!hot) {
    std::vector<std::pair<uint64_t, int32_t>> idle;
    for (auto& kv : x->prefixes)
      if (kv.second.refs == 0 && kv.second.slab >= 0) idle.push_back({kv.second.used, kv.first});
    std::sort(idle.begin(), idle.end());
    std::vector<int32_t> slabs;
    for (auto& u : idle) {
      victims.push_back(u.second);
      slabs.push_back(x->prefixes.at(u.second).slab);
      granikv_internal_hot_if_released(x->ctx, slabs.data(), (int32_t)slabs.size(), &largest, &ids);
      if (largest >= n && ids > 0) {
        hot = true;
        break;
      }
    }
    if (!hot) victims.clear();  // eviction cannot make room: evict nothing, place in COLD
  }
  if ((int32_t)victims.size() > max_evicted && evicted) return GRANIKV_ERR_INVALID;
  for (size_t i = 0; i < victims.size(); ++i) {
    if (evicted) evicted[i] = victims[i];
    drop_prefix(x, victims[i]);
  }
  if (n_evicted) *n_evicted = (int32_t)victims.size();

  Prefix p;
  p.length = n;
  if (hot) {
    int32_t sid = -1;
    int64_t off = -1;
    if (granikv_hot_alloc(x->ctx, n, &sid, &off) != GRANIKV_OK) return GRANIKV_ERR_INVALID;  // unreachable
    p.slab = sid;
    p.offset = off;
  }
  const int32_t id = x->next_prefix++;
  p.node = find_or_make_node(x, tokens, n);
  p.used = ++x->clock;
  x->nodes.at(p.node).prefix = id;
  x->prefixes.emplace(id, p);
  fill_info(x, id, out);
  return GRANIKV_OK;
}

granikv_status granikv_index_acquire(granikv_index* x, int32_t id) {
  if (!x) return GRANIKV_ERR_INVALID;
  auto it = x->prefixes.find(id);
  if (it == x->prefixes.end()) return GRANIKV_ERR_INVALID;
  it->second.refs += 1;
  it->second.used = ++x->clock;
  return GRANIKV_OK;
}

granikv_status granikv_index_release(granikv_index* x, int32_t id) {
  if (!x) return GRANIKV_ERR_INVALID;
  auto it = x->prefixes.find(id);
  if (it == x->prefixes.end() || it->second.refs <= 0) return GRANIKV_ERR_INVALID;
  it->second.refs -= 1;
  it->second.used = ++x->clock;
  return GRANIKV_OK;
}

granikv_status granikv_index_remove(granikv_index* x, int32_t id) {
  if (!x) return GRANIKV_ERR_INVALID;
  auto it = x->prefixes.find(id);
  if (it == x->prefixes.end() || it->second.refs != 0) return GRANIKV_ERR_INVALID;
  drop_prefix(x, id);
  return GRANIKV_OK;
}

granikv_status granikv_index_info(granikv_index* x, int32_t id, granikv_prefix_info* out) {
  if (!x || !out) return GRANIKV_ERR_INVALID;
  if (x->prefixes.find(id) == x->prefixes.end()) return GRANIKV_ERR_INVALID;
  fill_info(x, id, out);
  return GRANIKV_OK;
}

granikv_status granikv_index_stats(granikv_index* x, int32_t* n_prefixes, int32_t* n_hot,
                                   int32_t* n_nodes) {
  if (!x) return GRANIKV_ERR_INVALID;
  if (n_prefixes) *n_prefixes = (int32_t)x->prefixes.size();
  if (n_hot) {
    int32_t h = 0;
    for (auto& kv : x->prefixes) h += kv.second.slab >= 0 ? 1 : 0;
    *n_hot = h;
  }
  if (n_nodes) *n_nodes = (int32_t)x->nodes.size() - 1;  // not counting the root
  return GRANIKV_OK;
}

}  // extern "C"
