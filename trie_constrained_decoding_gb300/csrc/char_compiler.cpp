// Host compiler of character-level grammars: catalog strings as bytes, a byte
// vocabulary, and the token-level CSR the decode kernels walk.
//
// Follows the pith.science review of arXiv 2608.12574 (key machinery): a
// character-level trie of the catalog strings; an Aho-Corasick automaton over
// the vocabulary's byte strings; a depth-first walk of the trie that carries
// the automaton state, so that at each trie node the automaton reports every
// token ending there, and each such token becomes an edge from the node where
// it starts (its length above) to this node.  A token never overshoots the
// strings: it is reported only where its last character lies on a trie path.
// The cost is linear in trie size plus vocabulary size, times the token length.
//
// The result has the token compiler's layout: per node its outgoing token
// edges sorted by token id, plus the separator and stop edges at a terminal;
// nodes are numbered depth-first (preorder, children by ascending byte) over
// the character trie, so a run of nodes with one character child each gets
// consecutive ids and consecutive edge records, as in the token compiler
// (a forced run of one-character tokens is read in one round trip).  Live-pointer
// counts are subtree sizes in the character trie, and pointer ranks are
// depth-first over it, so every edge's pointers are one rank range.
#include <algorithm>
#include <cstring>
#include <deque>
#include <unordered_map>

#include "tcd_internal.h"

using namespace tcd;

namespace {

uint64_t key(int32_t node, uint8_t c) { return ((uint64_t)(uint32_t)node << 8) | c; }

struct Automaton {
  std::unordered_map<uint64_t, int32_t> go;  // trie of the token strings
  std::vector<int32_t> fail, out_link, tok, depth;

  int32_t add_state(int32_t d) {
    fail.push_back(0);
    out_link.push_back(-1);
    tok.push_back(-1);
    depth.push_back(d);
    return (int32_t)tok.size() - 1;
  }
  int32_t child(int32_t s, uint8_t c) const {
    auto it = go.find(key(s, c));
    return it == go.end() ? -1 : it->second;
  }
  // delta(s, c): follow failure links until a state has a c-transition.
  int32_t step(int32_t s, uint8_t c) const {
    for (;;) {
      const int32_t n = child(s, c);
      if (n >= 0) return n;
      if (s == 0) return 0;
      s = fail[s];
    }
  }
};

}  // namespace

extern "C" tc_status tc_compile_char_trie(const uint8_t* chars, const int64_t* offsets, int32_t n_strings,
                                          const int32_t* tok_ids, const uint8_t* tok_chars,
                                          const int64_t* tok_offsets, int32_t n_tokens, int32_t sep_id,
                                          int32_t stop_id, int32_t vocab, int32_t max_fanout, tc_trie** out) {
  if (!out) return TC_ERR_INVALID_ARG;
  *out = nullptr;
  if (!chars || !offsets || !tok_ids || !tok_chars || !tok_offsets || n_strings < 1 || n_tokens < 1 ||
      vocab < 2 || max_fanout < 2 || sep_id == stop_id || sep_id < 0 || sep_id >= vocab || stop_id < 0 ||
      stop_id >= vocab || offsets[0] != 0 || tok_offsets[0] != 0) {
    set_error_message("tc_compile_char_trie: invalid arguments");
    return TC_ERR_INVALID_ARG;
  }
  for (int32_t i = 0; i < n_strings; ++i) {
    if (offsets[i + 1] < offsets[i]) return TC_ERR_INVALID_ARG;
    if (offsets[i + 1] == offsets[i]) {
      set_error_message("tc_compile_char_trie: string " + std::to_string(i) + " is empty");
      return TC_ERR_EMPTY_STRING;
    }
  }
  {
    std::vector<int32_t> ids(tok_ids, tok_ids + n_tokens);
    for (int32_t j = 0; j < n_tokens; ++j) {
      if (tok_offsets[j + 1] <= tok_offsets[j]) {
        set_error_message("tc_compile_char_trie: token " + std::to_string(j) + " is empty");
        return TC_ERR_EMPTY_STRING;
      }
      if (ids[j] == sep_id || ids[j] == stop_id) {
        set_error_message("tc_compile_char_trie: a vocabulary token uses a control id");
        return TC_ERR_CONTROL_COLLISION;
      }
      if (ids[j] < 0 || ids[j] >= vocab) {
        set_error_message("tc_compile_char_trie: token id outside [0, vocab)");
        return TC_ERR_TOKEN_RANGE;
      }
    }
    std::sort(ids.begin(), ids.end());
    if (std::adjacent_find(ids.begin(), ids.end()) != ids.end()) {
      set_error_message("tc_compile_char_trie: token ids are not distinct");
      return TC_ERR_DUPLICATE;
    }
  }

  // 1. Character trie of the strings (insertion order), children per byte.
  std::unordered_map<uint64_t, int32_t> kid;
  std::vector<int32_t> term(1, -1);
  std::vector<std::vector<std::pair<uint8_t, int32_t>>> kids(1);
  for (int32_t i = 0; i < n_strings; ++i) {
    int32_t n = 0;
    for (int64_t q = offsets[i]; q < offsets[i + 1]; ++q) {
      const uint8_t c = chars[q];
      auto it = kid.find(key(n, c));
      if (it == kid.end()) {
        const int32_t m = (int32_t)term.size();
        term.push_back(-1);
        kids.emplace_back();
        kids[n].push_back({c, m});
        kid.emplace(key(n, c), m);
        n = m;
      } else {
        n = it->second;
      }
    }
    if (term[n] >= 0) {
      set_error_message("tc_compile_char_trie: strings " + std::to_string(term[n]) + " and " + std::to_string(i) +
                        " are equal");
      return TC_ERR_DUPLICATE;
    }
    term[n] = i;
  }
  const int32_t N = (int32_t)term.size();
  for (auto& k : kids) std::sort(k.begin(), k.end());
  // Depth-first (preorder) numbering, children by ascending byte: order[i]
  // is the trie node numbered i.
  std::vector<int32_t> order, new_id((size_t)N, -1);
  order.reserve(N);
  {
    std::vector<int32_t> stack{0};
    while (!stack.empty()) {
      const int32_t n = stack.back();
      stack.pop_back();
      new_id[(size_t)n] = (int32_t)order.size();
      order.push_back(n);
      for (auto it = kids[(size_t)n].rbegin(); it != kids[(size_t)n].rend(); ++it) stack.push_back(it->second);
    }
  }

  // 2. Aho-Corasick automaton over the token strings.
  Automaton ac;
  ac.add_state(0);
  for (int32_t j = 0; j < n_tokens; ++j) {
    int32_t s = 0;
    for (int64_t q = tok_offsets[j]; q < tok_offsets[j + 1]; ++q) {
      const uint8_t c = tok_chars[q];
      int32_t n = ac.child(s, c);
      if (n < 0) {
        n = ac.add_state(ac.depth[s] + 1);
        ac.go.emplace(key(s, c), n);
      }
      s = n;
    }
    if (ac.tok[s] >= 0) {
      set_error_message("tc_compile_char_trie: two vocabulary tokens have the same bytes");
      return TC_ERR_DUPLICATE;
    }
    ac.tok[s] = tok_ids[j];
  }
  {
    // failure and output links, breadth-first over the automaton's trie
    std::vector<std::vector<std::pair<uint8_t, int32_t>>> akids(ac.tok.size());
    for (auto& kv : ac.go) akids[(size_t)(kv.first >> 8)].push_back({(uint8_t)(kv.first & 0xff), kv.second});
    std::deque<int32_t> q;
    for (auto& ch : akids[0]) {
      ac.fail[ch.second] = 0;
      q.push_back(ch.second);
    }
    while (!q.empty()) {
      const int32_t s = q.front();
      q.pop_front();
      for (auto& ch : akids[s]) {
        const int32_t t = ch.second;
        ac.fail[t] = ac.step(ac.fail[s], ch.first);
        const int32_t f = ac.fail[t];
        ac.out_link[t] = ac.tok[f] >= 0 ? f : ac.out_link[f];
        q.push_back(t);
      }
    }
  }

  // 3. Depth-first walk of the character trie carrying the automaton state:
  //    every token reported at a node is an edge from the node its length above.
  struct Edge { int32_t tok, child; };
  std::vector<std::vector<Edge>> edges_of((size_t)N);
  {
    struct Frame { int32_t node, state, next; };
    std::vector<Frame> stack{{0, 0, 0}};
    std::vector<int32_t> path{0};  // trie nodes by depth along the current walk
    while (!stack.empty()) {
      Frame& f = stack.back();
      if (f.next == (int32_t)kids[f.node].size()) {
        stack.pop_back();
        path.pop_back();
        continue;
      }
      const auto ch = kids[f.node][(size_t)f.next++];
      const int32_t st = ac.step(f.state, ch.first);
      const int32_t c = ch.second;
      path.push_back(c);
      const int32_t d = (int32_t)path.size() - 1;
      for (int32_t x = ac.tok[st] >= 0 ? st : ac.out_link[st]; x >= 0; x = ac.out_link[x]) {
        const int32_t src = path[(size_t)(d - ac.depth[x])];
        edges_of[(size_t)src].push_back({ac.tok[x], c});
      }
      stack.push_back({c, st, 0});  // (f is not used after this push)
    }
  }

  // 4. CSR in depth-first node order with control edges at terminals.
  auto* t = new tc_trie();
  t->vocab = vocab;
  t->sep = sep_id;
  t->stop = stop_id;
  t->fanout_cap = max_fanout;
  t->n_strings = n_strings;
  t->total_tokens = offsets[n_strings];
  t->char_level = true;
  t->node_begin.assign((size_t)N + 1, 0);
  t->node_ptr.assign((size_t)N, -1);
  int32_t max_fan = 0;
  std::vector<Edge> all;
  for (int32_t ni = 0; ni < N; ++ni) {
    const int32_t old = order[(size_t)ni];
    t->node_begin[(size_t)ni] = (int32_t)all.size();
    std::vector<Edge> mine;
    for (const Edge& e : edges_of[(size_t)old]) mine.push_back({e.tok, new_id[(size_t)e.child]});
    if (term[(size_t)old] >= 0) {
      t->node_ptr[(size_t)ni] = term[(size_t)old];
      mine.push_back({sep_id, -1});
      mine.push_back({stop_id, -2});
    }
    std::sort(mine.begin(), mine.end(), [](const Edge& a, const Edge& b) { return a.tok < b.tok; });
    const int32_t fan = (int32_t)mine.size();
    if (fan > max_fanout) {
      set_error_message("tc_compile_char_trie: node " + std::to_string(ni) + " has " + std::to_string(fan) +
                        " edges, above the cap of " + std::to_string(max_fanout));
      delete t;
      return TC_ERR_FANOUT;
    }
    max_fan = std::max(max_fan, fan);
    if (ni == 0) t->root_fanout = fan;
    all.insert(all.end(), mine.begin(), mine.end());
  }
  t->node_begin[(size_t)N] = (int32_t)all.size();
  const int32_t E = (int32_t)all.size();
  t->max_fanout = max_fan;
  t->edge_tok.resize((size_t)E);
  t->edge_child.resize((size_t)E);
  for (int32_t e = 0; e < E; ++e) {
    t->edge_tok[(size_t)e] = all[(size_t)e].tok;
    t->edge_child[(size_t)e] = all[(size_t)e].child;
  }

  // 5. Subtree sizes and depth-first ranks over the character trie (its own
  //    child links, not the token edges), in the new node ids.
  std::vector<std::vector<int32_t>> tree((size_t)N);
  for (int32_t ni = 0; ni < N; ++ni)
    for (auto& ch : kids[(size_t)order[(size_t)ni]]) tree[(size_t)ni].push_back(new_id[(size_t)ch.second]);
  std::vector<int32_t> lo((size_t)N, 0), cnt((size_t)N, 0);
  t->ptr_rank.assign((size_t)n_strings, -1);
  {
    int32_t next_rank = 0;
    std::vector<std::pair<int32_t, int32_t>> stack{{0, 0}};
    lo[0] = 0;
    if (t->node_ptr[0] >= 0) t->ptr_rank[(size_t)t->node_ptr[0]] = next_rank++;
    while (!stack.empty()) {
      auto& top = stack.back();
      const int32_t n = top.first;
      if (top.second == (int32_t)tree[(size_t)n].size()) {
        cnt[(size_t)n] = next_rank - lo[(size_t)n];
        stack.pop_back();
        continue;
      }
      const int32_t c = tree[(size_t)n][(size_t)top.second++];
      lo[(size_t)c] = next_rank;
      if (t->node_ptr[(size_t)c] >= 0) t->ptr_rank[(size_t)t->node_ptr[(size_t)c]] = next_rank++;
      stack.push_back({c, 0});
    }
  }
  t->static_cnt.assign((size_t)E, 0);
  t->edge_lo.assign((size_t)E, -1);
  for (int32_t n = 0; n < N; ++n)
    for (int32_t e = t->node_begin[(size_t)n]; e < t->node_begin[(size_t)n + 1]; ++e) {
      const int32_t c = t->edge_child[(size_t)e];
      if (c >= 0) {
        t->static_cnt[(size_t)e] = cnt[(size_t)c];
        t->edge_lo[(size_t)e] = lo[(size_t)c];
      } else {
        t->edge_lo[(size_t)e] = t->ptr_rank[(size_t)t->node_ptr[(size_t)n]];
      }
    }

  // 6. No pointer paths (count mode does not apply); depth in characters.
  t->path_off.assign((size_t)n_strings + 1, 0);
  int32_t depth = 0;
  for (int32_t i = 0; i < n_strings; ++i) depth = std::max<int32_t>(depth, (int32_t)(offsets[i + 1] - offsets[i]));
  t->max_depth = depth;

  uint64_t h = 1469598103934665603ull ^ 0x63686172ull;  // distinct from token tries with equal arrays
  auto mix = [&h](const void* p, size_t n) {
    const unsigned char* c = static_cast<const unsigned char*>(p);
    for (size_t i = 0; i < n; ++i) {
      h ^= c[i];
      h *= 1099511628211ull;
    }
  };
  int32_t hdr[4] = {vocab, sep_id, stop_id, n_strings};
  mix(hdr, sizeof(hdr));
  mix(t->node_begin.data(), t->node_begin.size() * 4);
  mix(t->edge_tok.data(), t->edge_tok.size() * 4);
  mix(t->edge_child.data(), t->edge_child.size() * 4);
  mix(t->node_ptr.data(), t->node_ptr.size() * 4);
  t->content_hash = h;
  *out = t;
  return TC_OK;
}
