// Host-visible interface of the tcgen05 GEMM with a masked-argmax epilogue.
#pragma once

#include <cuda.h>  // CUtensorMap (types only; the encoder is fetched through the runtime)
#include <cuda_runtime.h>
#include <stdint.h>

namespace tcd {

// Best candidate of one sequence within one column tile.
struct GemmPartial {
  float logit;
  int32_t col;  // INT32_MAX when the sequence has no candidate in the tile
};

// One sequence's candidates within one 128-column tile of the union GEMM,
// written before the GEMM so that its epilogue reads them with one load.
struct alignas(16) TileCands {
  uint32_t bits[4];  // bit c set: column tile * 128 + c is one of the sequence's candidates
  int32_t start;     // the sequence's candidates in earlier tiles (index of the first one in this tile)
  int32_t pad[3];
};

struct GemmParams {
  const int64_t* xrow;       // [B] >= 0 for sequences that take this step, -1 otherwise; null: all B take it
  const int32_t* row0_ptr;   // device: first activation row of the step in the activation map (null: 0)
  int32_t B;                 // sequences, <= 256
  int32_t H;                 // multiple of 64
  const int32_t* row_list;   // [n_cols] embedding row of each column (gathered), or null (column = row)
  const int32_t* n_cols_ptr; // device column count (read at kernel start), or null
  int32_t n_cols_fixed;      // column count when n_cols_ptr is null
  const int32_t* cand_col;   // [B, C] ascending columns of each sequence's legal candidates
  const int32_t* ncand;      // [B]
  const TileCands* tile_cands;  // [B, max_tiles] per-tile candidate records, or null (search cand_col)
  int32_t uniform;           // 1: every sequence has the same candidates: tile_cands holds one record per tile
  int32_t C;
  GemmPartial* part;         // [B, max_tiles] (ksplit == 1)
  int32_t max_tiles;
  int32_t ksplit;            // K splits per column tile; H / 64 must be a multiple
  int32_t msplit;            // set by the launcher: 128-sequence M tiles taken by separate tasks
  float* split_part;         // [ksplit, B, C] candidate partial sums (ksplit > 1)
  int32_t* err;              // set to 1 when a wait timed out
  long long wait_limit;      // try_wait polls of one wait before it gives up (the launcher fills 0 in)
  int32_t withhold;          // test switch: CTA 0 issues nothing for its first stage, so the waits on
                             // that stage run out (the error path without any fault)
};

// Tensor maps of the embedding: 64 x 128 boxes (contiguous rows) and 64 x 1
// boxes for four-row gathers; both bf16 with the 128-byte swizzle.
struct EmbMaps {
  CUtensorMap tiled;
  CUtensorMap gather;
};

size_t gemm_smem_bytes(int m_tiles);
int gemm_tile_cols();
// Opt in to the GEMM's dynamic shared memory (current device).
cudaError_t prepare_gemm();
cudaError_t encode_emb_maps(const void* emb, int V, int H, EmbMaps* out);
// hidden: bf16 activations with `rows` rows of H elements (the A operand).
cudaError_t launch_union_gemm(const GemmParams& p, const void* hidden, int64_t rows, const EmbMaps& emb,
                              int num_ctas, cudaStream_t s);

}  // namespace tcd
