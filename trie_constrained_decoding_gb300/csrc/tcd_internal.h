// Internal definitions shared by the host compiler, the runtime and the kernels.
#pragma once

#include <stdint.h>

#include <string>
#include <vector>

#include "tcd.h"

// Host form of a compiled catalog: the CSR arrays of tc_trie_export.
struct tc_trie {
  int32_t vocab = 0, sep = 0, stop = 0, fanout_cap = 0;
  int32_t n_strings = 0, max_depth = 0, max_fanout = 0, root_fanout = 0;
  int64_t total_tokens = 0;
  std::vector<int32_t> node_begin, edge_tok, edge_child, node_ptr, static_cnt, path_off, path;
  // Depth-first numbering of the pointers (a node's own pointer before those
  // below it, children in token order): every subtree holds a contiguous range
  // of ranks.  edge_lo[e] is the first rank below a token edge's child (the
  // range has static_cnt[e] ranks), or the terminal's own rank for a control edge.
  std::vector<int32_t> ptr_rank, edge_lo;
  // Character-level grammar (tc_compile_char_trie): nodes are characters and a
  // token edge may span several of them, so several edges can lead to one
  // node; pointer paths are not kept and only the read-only no-repeat state
  // (rank ranges) applies.
  bool char_level = false;
  uint64_t content_hash = 0;

  int32_t n_nodes() const { return (int32_t)node_ptr.size(); }
  int32_t n_edges() const { return (int32_t)edge_tok.size(); }
};

namespace tcd {

// Device walk image, int32 words:
//   header:  node_begin[N+1] | node_rank[N]            (the part copied to constant memory)
//   pad to a multiple of 8 words
//   edges:   {tok, child, lo, n, cbeg, cend, cpid, 0}[E]
// {lo, n} is the range of pointer ranks below a token edge (the terminal's own
// rank and 1 for a control edge); {cbeg, cend, cpid} is the header of the
// edge's child (the root's for a separator, zeros for stop), so a walk never
// needs a node header lookup.  node_rank is the rank of the node's pointer or
// -1; on the device a pointer is named by its rank.
struct WalkLayout {
  int32_t n_nodes, n_edges;
  int32_t off_ptr;        // word offset of node_rank
  int32_t header_words;   // words of the header part
  int32_t off_edges;      // word offset of the edge records (multiple of 8: 32-byte records)
  int32_t words;          // total words
};
WalkLayout walk_layout(int32_t n_nodes, int32_t n_edges);
std::vector<int32_t> build_walk_image(const tc_trie& t, const WalkLayout& L);

void set_error_message(const std::string& msg);

}  // namespace tcd
