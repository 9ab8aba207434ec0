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
  uint64_t content_hash = 0;

  int32_t n_nodes() const { return (int32_t)node_ptr.size(); }
  int32_t n_edges() const { return (int32_t)edge_tok.size(); }
};

namespace tcd {

// Device walk image, int32 words: node_begin[N+1] | pad to even | edges {tok, child}[E] | node_ptr[N].
struct WalkLayout {
  int32_t n_nodes, n_edges;
  int32_t off_edges;   // word offset of the edge records (even)
  int32_t off_ptr;     // word offset of node_ptr
  int32_t words;       // total words
};
WalkLayout walk_layout(int32_t n_nodes, int32_t n_edges);
std::vector<int32_t> build_walk_image(const tc_trie& t, const WalkLayout& L);

void set_error_message(const std::string& msg);

}  // namespace tcd
