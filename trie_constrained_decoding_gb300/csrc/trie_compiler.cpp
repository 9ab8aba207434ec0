// Host trie compiler: catalog of token-id strings -> CSR trie with control
// edges, live-pointer counts and per-pointer edge paths.
//
// Follows "Constraint made cheaper than no constraint", section "The grammar
// as a trie over tokens" (edge range per node, token and child per edge, two
// sentinel children for the separator and stop edges, each pointer keeps the
// edges on its path), section "Masked sampling inside the sampler" (each edge
// carries the count of live pointers below it) and section "The sparse output
// layer" (the build refuses a node with more edges than the cap).
#include <algorithm>
#include <cstring>
#include <unordered_map>

#include "tcd_internal.h"

namespace tcd {

static thread_local std::string g_error_message;

void set_error_message(const std::string& msg) { g_error_message = msg; }

WalkLayout walk_layout(int32_t n_nodes, int32_t n_edges) {
  WalkLayout L;
  L.n_nodes = n_nodes;
  L.n_edges = n_edges;
  L.off_ptr = n_nodes + 1;
  L.header_words = 2 * n_nodes + 1;
  L.off_edges = (L.header_words + 7) & ~7;  // 32-byte aligned edge records
  L.words = L.off_edges + 8 * n_edges;
  return L;
}

std::vector<int32_t> build_walk_image(const tc_trie& t, const WalkLayout& L) {
  std::vector<int32_t> img((size_t)L.words, 0);
  std::copy(t.node_begin.begin(), t.node_begin.end(), img.begin());
  auto rank_of = [&](int32_t n) { return t.node_ptr[n] >= 0 ? t.ptr_rank[t.node_ptr[n]] : -1; };
  for (int32_t n = 0; n < L.n_nodes; ++n) img[(size_t)L.off_ptr + n] = rank_of(n);
  for (int32_t e = 0; e < L.n_edges; ++e) {
    int32_t* r = img.data() + L.off_edges + 8 * (size_t)e;
    const int32_t c = t.edge_child[e];
    r[0] = t.edge_tok[e];
    r[1] = c;
    r[2] = t.edge_lo[e];
    r[3] = c >= 0 ? t.static_cnt[e] : 1;
    if (c >= 0) {
      r[4] = t.node_begin[c];
      r[5] = t.node_begin[c + 1];
      r[6] = rank_of(c);
    } else if (c == -1) {  // separator: back to the root
      r[4] = t.node_begin[0];
      r[5] = t.node_begin[1];
      r[6] = rank_of(0);
    } else {
      r[6] = -1;
    }
  }
  return img;
}

static uint64_t fnv1a(uint64_t h, const void* p, size_t n) {
  const unsigned char* c = static_cast<const unsigned char*>(p);
  for (size_t i = 0; i < n; ++i) {
    h ^= c[i];
    h *= 1099511628211ull;
  }
  return h;
}

template <class V>
static uint64_t hash_vec(uint64_t h, const V& v) {
  uint64_t n = v.size();
  h = fnv1a(h, &n, sizeof(n));
  return fnv1a(h, v.data(), v.size() * sizeof(v[0]));
}

}  // namespace tcd

using namespace tcd;

extern "C" tc_status tc_compile_trie(const int32_t* ids, const int64_t* offsets, int32_t n_strings,
                                     int32_t sep_id, int32_t stop_id, int32_t vocab,
                                     int32_t max_fanout, tc_trie** out) {
  if (!out) return TC_ERR_INVALID_ARG;
  *out = nullptr;
  if (!offsets || n_strings < 1 || vocab < 2 || max_fanout < 2 || sep_id == stop_id ||
      sep_id < 0 || sep_id >= vocab || stop_id < 0 || stop_id >= vocab) {
    set_error_message("tc_compile_trie: invalid arguments");
    return TC_ERR_INVALID_ARG;
  }
  if (offsets[0] != 0) {
    set_error_message("tc_compile_trie: offsets[0] must be 0");
    return TC_ERR_INVALID_ARG;
  }
  for (int32_t i = 0; i < n_strings; ++i) {
    if (offsets[i + 1] < offsets[i]) {
      set_error_message("tc_compile_trie: offsets must not decrease");
      return TC_ERR_INVALID_ARG;
    }
    if (offsets[i + 1] == offsets[i]) {
      set_error_message("tc_compile_trie: string " + std::to_string(i) + " is empty");
      return TC_ERR_EMPTY_STRING;
    }
  }
  const int64_t total = offsets[n_strings];
  if (total > 0 && !ids) return TC_ERR_INVALID_ARG;
  if (total >= (int64_t)INT32_MAX / 2) return TC_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n_strings; ++i) {
    for (int64_t q = offsets[i]; q < offsets[i + 1]; ++q) {
      const int32_t t = ids[q];
      if (t == sep_id || t == stop_id) {
        set_error_message("tc_compile_trie: string " + std::to_string(i) + " contains a control id");
        return TC_ERR_CONTROL_COLLISION;
      }
      if (t < 0 || t >= vocab) {
        set_error_message("tc_compile_trie: string " + std::to_string(i) + " has an id outside [0, vocab)");
        return TC_ERR_TOKEN_RANGE;
      }
    }
  }

  // 1. Insert every string into a pointer trie keyed by (node, token).
  std::unordered_map<uint64_t, int32_t> child_of;
  child_of.reserve((size_t)total * 2 + 16);
  std::vector<int32_t> term_ptr(1, -1);             // per insertion-order node
  std::vector<std::vector<int32_t>> kids(1);          // child nodes per node
  std::vector<int32_t> node_tok(1, -1);               // token on the edge into a node
  for (int32_t i = 0; i < n_strings; ++i) {
    int32_t n = 0;
    for (int64_t q = offsets[i]; q < offsets[i + 1]; ++q) {
      const uint64_t key = ((uint64_t)(uint32_t)n << 32) | (uint32_t)ids[q];
      auto it = child_of.find(key);
      if (it == child_of.end()) {
        const int32_t c = (int32_t)term_ptr.size();
        term_ptr.push_back(-1);
        kids.emplace_back();
        node_tok.push_back(ids[q]);
        kids[n].push_back(c);
        child_of.emplace(key, c);
        n = c;
      } else {
        n = it->second;
      }
    }
    if (term_ptr[n] >= 0) {
      set_error_message("tc_compile_trie: strings " + std::to_string(term_ptr[n]) + " and " +
                        std::to_string(i) + " are equal");
      return TC_ERR_DUPLICATE;
    }
    term_ptr[n] = i;
  }
  const int32_t N = (int32_t)term_ptr.size();

  // 2. Depth-first (preorder) numbering, children visited in ascending token
  //    order: a node's first child directly follows it, so a chain of nodes
  //    with one edge each gets consecutive ids and, in the CSR below,
  //    consecutive edge records (a forced span can be read in one go).
  for (auto& k : kids)
    std::sort(k.begin(), k.end(), [&](int32_t a, int32_t b) { return node_tok[a] < node_tok[b]; });
  std::vector<int32_t> order;
  order.reserve(N);
  std::vector<int32_t> new_id(N, -1);
  std::vector<int32_t> stack{0};
  while (!stack.empty()) {
    const int32_t n = stack.back();
    stack.pop_back();
    new_id[n] = (int32_t)order.size();
    order.push_back(n);
    for (auto it = kids[n].rbegin(); it != kids[n].rend(); ++it) stack.push_back(*it);
  }

  // 3. Emit the CSR: per node its child edges plus the two control edges of a
  //    terminal, all sorted by token id.
  auto* t = new tc_trie();
  t->vocab = vocab;
  t->sep = sep_id;
  t->stop = stop_id;
  t->fanout_cap = max_fanout;
  t->n_strings = n_strings;
  t->total_tokens = total;
  t->node_begin.assign((size_t)N + 1, 0);
  t->node_ptr.assign((size_t)N, -1);
  std::vector<int32_t> subtree((size_t)N, 0);  // pointers ending at or below a node (new ids)
  struct Edge { int32_t tok, child; };
  std::vector<Edge> edges;
  edges.reserve((size_t)N + 2 * (size_t)n_strings);
  int32_t max_fan = 0;
  for (int32_t ni = 0; ni < N; ++ni) {
    const int32_t old = order[ni];
    t->node_begin[ni] = (int32_t)edges.size();
    std::vector<Edge> mine;
    mine.reserve(kids[old].size() + 2);
    for (int32_t c : kids[old]) mine.push_back({node_tok[c], new_id[c]});
    if (term_ptr[old] >= 0) {
      t->node_ptr[ni] = term_ptr[old];
      mine.push_back({sep_id, -1});
      mine.push_back({stop_id, -2});
    }
    std::sort(mine.begin(), mine.end(), [](const Edge& a, const Edge& b) { return a.tok < b.tok; });
    const int32_t fan = (int32_t)mine.size();
    if (fan > max_fanout) {
      set_error_message("tc_compile_trie: node " + std::to_string(ni) + " has " + std::to_string(fan) +
                        " edges, above the cap of " + std::to_string(max_fanout));
      delete t;
      return TC_ERR_FANOUT;
    }
    max_fan = std::max(max_fan, fan);
    if (ni == 0) t->root_fanout = fan;
    edges.insert(edges.end(), mine.begin(), mine.end());
  }
  t->node_begin[N] = (int32_t)edges.size();
  const int32_t E = (int32_t)edges.size();
  t->max_fanout = max_fan;
  t->edge_tok.resize(E);
  t->edge_child.resize(E);
  for (int32_t e = 0; e < E; ++e) {
    t->edge_tok[e] = edges[e].tok;
    t->edge_child[e] = edges[e].child;
  }

  // 4. Live-pointer counts: children have larger preorder ids, so one reverse
  //    pass accumulates subtree sizes.
  for (int32_t ni = N - 1; ni >= 0; --ni) {
    int32_t s = t->node_ptr[ni] >= 0 ? 1 : 0;
    for (int32_t e = t->node_begin[ni]; e < t->node_begin[ni + 1]; ++e)
      if (t->edge_child[e] >= 0) s += subtree[t->edge_child[e]];
    subtree[ni] = s;
  }
  t->static_cnt.assign((size_t)E, 0);
  for (int32_t e = 0; e < E; ++e)
    if (t->edge_child[e] >= 0) t->static_cnt[e] = subtree[t->edge_child[e]];

  // 5. Depth-first pointer ranks: a node's own pointer first, then its
  //    children's subtrees in token order; each subtree gets one range.
  t->ptr_rank.assign((size_t)n_strings, -1);
  t->edge_lo.assign((size_t)E, -1);
  {
    std::vector<int32_t> lo_of((size_t)N, 0);
    std::vector<std::pair<int32_t, int32_t>> stack;  // (node, next edge to visit)
    int32_t next_rank = 0;
    stack.push_back({0, t->node_begin[0]});
    lo_of[0] = 0;
    if (t->node_ptr[0] >= 0) t->ptr_rank[t->node_ptr[0]] = next_rank++;
    while (!stack.empty()) {
      auto& top = stack.back();
      const int32_t n = top.first;
      if (top.second == t->node_begin[n + 1]) {
        stack.pop_back();
        continue;
      }
      const int32_t e = top.second++;
      const int32_t c = t->edge_child[e];
      if (c < 0) continue;
      lo_of[c] = next_rank;
      if (t->node_ptr[c] >= 0) t->ptr_rank[t->node_ptr[c]] = next_rank++;
      stack.push_back({c, t->node_begin[c]});
    }
    for (int32_t n = 0; n < N; ++n)
      for (int32_t e = t->node_begin[n]; e < t->node_begin[n + 1]; ++e)
        t->edge_lo[e] = t->edge_child[e] >= 0 ? lo_of[t->edge_child[e]] : t->ptr_rank[t->node_ptr[n]];
  }

  // 6. Per-pointer edge paths (root to terminal), found by binary search of
  //    each node's sorted edge range.
  t->path_off.assign((size_t)n_strings + 1, 0);
  t->path.resize((size_t)total);
  int32_t depth = 0;
  for (int32_t i = 0; i < n_strings; ++i) {
    t->path_off[i] = (int32_t)offsets[i];
    int32_t n = 0;
    for (int64_t qq = offsets[i]; qq < offsets[i + 1]; ++qq) {
      const int32_t* b = t->edge_tok.data() + t->node_begin[n];
      const int32_t* e = t->edge_tok.data() + t->node_begin[n + 1];
      const int32_t* f = std::lower_bound(b, e, ids[qq]);
      const int32_t edge = (int32_t)(f - t->edge_tok.data());
      t->path[(size_t)qq] = edge;
      n = t->edge_child[edge];
    }
    depth = std::max<int32_t>(depth, (int32_t)(offsets[i + 1] - offsets[i]));
  }
  t->path_off[n_strings] = (int32_t)total;
  t->max_depth = depth;

  uint64_t h = 1469598103934665603ull;
  int32_t hdr[4] = {vocab, sep_id, stop_id, n_strings};
  h = fnv1a(h, hdr, sizeof(hdr));
  h = hash_vec(h, t->node_begin);
  h = hash_vec(h, t->edge_tok);
  h = hash_vec(h, t->edge_child);
  h = hash_vec(h, t->node_ptr);
  h = hash_vec(h, t->path);
  t->content_hash = h;
  *out = t;
  return TC_OK;
}

extern "C" tc_status tc_trie_info(const tc_trie* t, tc_trie_info_t* out) {
  if (!t || !out) return TC_ERR_INVALID_ARG;
  std::memset(out, 0, sizeof(*out));
  out->n_nodes = t->n_nodes();
  out->n_edges = t->n_edges();
  out->n_strings = t->n_strings;
  out->max_fanout = t->max_fanout;
  out->root_fanout = t->root_fanout;
  out->max_depth = t->max_depth;
  out->vocab = t->vocab;
  out->sep_id = t->sep;
  out->stop_id = t->stop;
  out->total_tokens = t->total_tokens;
  const WalkLayout L = walk_layout(t->n_nodes(), t->n_edges());
  out->walk_image_bytes = (int64_t)L.words * 4;
  out->header_bytes = L.header_words * 4;
  return TC_OK;
}

extern "C" tc_status tc_trie_export(const tc_trie* t, int32_t* node_begin, int32_t* edge_tok,
                                    int32_t* edge_child, int32_t* node_ptr, int32_t* static_cnt,
                                    int32_t* path_off, int32_t* path) {
  if (!t) return TC_ERR_INVALID_ARG;
  auto put = [](int32_t* dst, const std::vector<int32_t>& v) {
    if (dst && !v.empty()) std::memcpy(dst, v.data(), v.size() * sizeof(int32_t));
  };
  put(node_begin, t->node_begin);
  put(edge_tok, t->edge_tok);
  put(edge_child, t->edge_child);
  put(node_ptr, t->node_ptr);
  put(static_cnt, t->static_cnt);
  put(path_off, t->path_off);
  put(path, t->path);
  return TC_OK;
}

extern "C" tc_status tc_trie_export_ranks(const tc_trie* t, int32_t* ptr_rank, int32_t* edge_lo) {
  if (!t) return TC_ERR_INVALID_ARG;
  if (ptr_rank) std::memcpy(ptr_rank, t->ptr_rank.data(), t->ptr_rank.size() * sizeof(int32_t));
  if (edge_lo) std::memcpy(edge_lo, t->edge_lo.data(), t->edge_lo.size() * sizeof(int32_t));
  return TC_OK;
}

extern "C" void tc_trie_free(tc_trie* t) { delete t; }

extern "C" const char* tc_status_str(tc_status s) {
  switch (s) {
    case TC_OK: return "TC_OK";
    case TC_ERR_INVALID_ARG: return "TC_ERR_INVALID_ARG";
    case TC_ERR_FANOUT: return "TC_ERR_FANOUT";
    case TC_ERR_DUPLICATE: return "TC_ERR_DUPLICATE";
    case TC_ERR_CONTROL_COLLISION: return "TC_ERR_CONTROL_COLLISION";
    case TC_ERR_TOKEN_RANGE: return "TC_ERR_TOKEN_RANGE";
    case TC_ERR_EMPTY_STRING: return "TC_ERR_EMPTY_STRING";
    case TC_ERR_K_RANGE: return "TC_ERR_K_RANGE";
    case TC_ERR_CONST_CAPACITY: return "TC_ERR_CONST_CAPACITY";
    case TC_ERR_NOT_BOUND: return "TC_ERR_NOT_BOUND";
    case TC_ERR_CAPACITY: return "TC_ERR_CAPACITY";
    case TC_ERR_UNSUPPORTED: return "TC_ERR_UNSUPPORTED";
    case TC_ERR_EMPTY_MASK: return "TC_ERR_EMPTY_MASK";
    case TC_ERR_NO_LIVE_EDGE: return "TC_ERR_NO_LIVE_EDGE";
    case TC_ERR_MAX_STEPS: return "TC_ERR_MAX_STEPS";
    case TC_ERR_BOUNDS: return "TC_ERR_BOUNDS";
    case TC_ERR_DEVICE_TIMEOUT: return "TC_ERR_DEVICE_TIMEOUT";
    case TC_ERR_CUDA: return "TC_ERR_CUDA";
    case TC_ERR_OOM: return "TC_ERR_OOM";
  }
  return "TC_ERR_UNKNOWN";
}

extern "C" const char* tc_last_error_message(void) { return tcd::g_error_message.c_str(); }
