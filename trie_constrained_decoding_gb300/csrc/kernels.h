// Host-visible parameter blocks and launchers of the decode-step kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace tcd {

constexpr int kThreads = 256;          // threads per CTA of every step kernel (8 warps)
constexpr int kWarps = kThreads / 32;
constexpr int kMaxTiles = 1024;        // upper bound of CTAs per sequence (partials per sequence)
constexpr int kMaxHidden = 16384;
constexpr int kMaxCandCap = 4096;
// Decode steps per iteration of the graph's WHILE body.  Each iteration of a
// conditional node costs a few microseconds of its own; running several step
// kernels per iteration amortises it, at the price of up to kLoopUnroll - 1
// idle step launches after the last sequence stops (an idle launch that sees
// the batch already finished only waits, counts itself and steers the loop).
constexpr int kLoopUnroll = 16;
// Dynamic shared memory a step kernel may request: x staged for the generic
// hidden size, two int32 candidate lists of up to kMaxCandCap entries, and
// (dense head) 128 KiB of row stages or (multi-CTA sampling) 64 KiB of sort
// keys and weights.
constexpr int kMaxDynamicSmem = kMaxHidden * 2 + 2 * kMaxCandCap * 4 + 128 + 128 * 1024;
constexpr int kSampleSmem = kMaxCandCap * 8 + 2 * kMaxCandCap * 4 + 256 * 4 + 64;

// Largest k of the read-only no-repeat state: the banned set is up to kBanMax
// 16-bit pointer ranks, 16 bytes per sequence.
constexpr int kBanMax = 8;
constexpr int kBanMaxStrings = 65535;

// Per-sequence decode state (device memory, one 48-byte record per sequence).
struct alignas(16) SeqState {
  int32_t node;     // current trie node
  int32_t emitted;  // pointers completed so far (j)
  int32_t len;      // tokens emitted so far
  int32_t status;   // TC_OK or the error that stopped the sequence
  int32_t done;     // 1 once the stop token was emitted or an error occurred
  int32_t k;        // pointers owed in total
  int32_t pre_n;    // one-CTA sparse step: size + 1 of the node's precomputed legal set (0: none)
  int32_t pre_pid;  // and the node's pointer rank
  // Read-only no-repeat mode: ranks of the completed pointers, two per word
  // (scalar fields: an array member would keep the state out of registers).
  uint32_t ban0, ban1, ban2, ban3;
};
// 16-byte aligned: a step reads its state as three 16-byte loads.
static_assert(sizeof(SeqState) == 48, "sequence state: three 16-byte loads");

// A legal candidate as kept in candidate lists: {token, edge, child, live
// pointers below} and the child's header {edge begin, edge end, pointer rank, 0}.
struct Cand {
  int4 a;
  int4 h;
};

// One CTA's best candidate, handed to the sequence's last CTA.
struct Partial {
  float logit;
  int32_t tok;
  int32_t edge;
  int32_t err;  // the CTA's error flag (nonzero: its filter or a bounded wait failed)
};

// Device control block of the device-resident loop.
struct Ctrl {
  int32_t live;       // sequences neither stopped nor failed
  uint32_t ticket;    // CTAs of the current launch that have finished (loop-control launches)
  int32_t pad[6];
};

// The bound grammar as the kernels see it.
struct GrammarView {
  const int32_t* img;        // walk image in global memory (its header part is the constant copy)
  int32_t off_edges, off_ptr;
  int32_t root_beg, root_end, root_pid;  // the root's header
  int32_t n_nodes, n_edges, n_strings;
  const int32_t* static_cnt; // [E]
  const int32_t* path_off;   // [K+1] by pointer rank
  const int32_t* path;       // [total tokens]: the token edges of each pointer, in rank order
};

struct GemmPartial;  // gemm_tc.h
struct EmbMaps;      // gemm_tc.h
struct TileCands;    // gemm_tc.h

// Scratch of the GEMM heads (candidate lists in global memory, the union of
// legal rows, per-(sequence, column tile) partial results).
struct HeadScratch {
  int32_t* cand_tok;        // [B, C] legal tokens of each sequence, ascending
  int32_t* cand_edge;       // [B, C] their edges
  int32_t* cand_col;        // [B, C] their GEMM columns (union index, or the token for the dense GEMM)
  int32_t* ncand;           // [B]
  int32_t* errf;            // [B] filter found an out-of-range index
  int64_t* xrow;            // [B] element offset of the sequence's hidden row, -1 if not stepping
  uint32_t* ubits;          // [ceil(V/32)] union bitmap (all zero between steps)
  int32_t* ulist;           // [V] union of legal tokens, ascending
  int32_t* umap;            // [V] token -> union index (valid for members only)
  int32_t* n_union;         // [1]
  TileCands* tile_cands;    // [B, max_tiles] each sequence's candidates per union tile
  GemmPartial* part;        // [B, max_tiles]
  int32_t max_tiles;
  int32_t ksplit;           // K splits of the union GEMM (fixed by the hidden size)
  float* split_part;        // [ksplit, B, C] per-split candidate sums of the union GEMM
  int32_t union_mode;       // 1: columns are the union; 0: every vocabulary row
  int32_t* gemm_err;        // [1] GEMM wait timeout (cleared by every reset)
  long long wait_limit;     // polls of one GEMM wait before it gives up (0: the default)
  int32_t withhold;         // test switch of the GEMM (see GemmParams::withhold)
  int32_t* row0;            // [1] first activation row of the current step
  // Root step (the first step of a decode, every sequence at the root with
  // nothing completed): its candidates are the root's token edges, the same
  // for every sequence, so no filter or union compaction runs.
  int32_t root_mode;        // 1: this GEMM step is the root step
  int32_t n_root;           // the root's token edges
  const int32_t* root_tok;  // [n_root] their tokens, ascending (the GEMM's columns)
  const int32_t* root_edge; // [n_root] their edge indices
  const EmbMaps* emb_maps;  // host: tensor maps of the embedding
};

struct StepParams {
  GrammarView g;
  const uint16_t* emb;      // bf16 [V, H]
  int32_t V, H;
  const uint16_t* hidden;   // bf16 [B, H] (host form) or [S, B, H] (device form: row len_b * B + b)
  int64_t hidden_rows;      // rows of `hidden` (B, or S * B)
  SeqState* st;             // [B]
  int32_t* cnt;             // [B, E] live-pointer counts (count mode)
  uint32_t* spent;          // [B, kw] spent flags by pointer rank (count mode)
  int32_t kw;               // words of spent flags per sequence
  int32_t B;
  int32_t cand_cap;         // C
  Partial* part;            // [B, tiles]
  uint32_t* seq_ticket;     // [B]
  Ctrl* ctrl;               // control block: live count and the loop-control ticket
  int32_t max_steps;        // a live sequence with this many tokens stops with TC_ERR_MAX_STEPS
  int32_t* tok_out;         // host form: [b * out_stride]; device form: toks[b * out_stride + len]
  float* logit_out;         // same indexing as tok_out (may be null in host form)
  int32_t* status_out;      // [B] or null
  int32_t* lens_out;        // [B] or null
  int32_t out_stride;
  unsigned long long cond;  // cudaGraphConditionalHandle of the loop (device form)
  int32_t device_form;      // 1: hidden row and output position follow each sequence's own length
  int32_t loop_ctrl;        // 1: this launch sets the loop's condition (last step of a loop body)
  unsigned long long* stats;  // optional counters, see StatSlot
  HeadScratch hs;           // GEMM heads only
  Cand* pre;                // [B, 32] precomputed candidate lists (sparse head), or null
  int32_t one_cta;          // every node has at most 32 edges: the one-CTA sparse step kernel
  int32_t jump;             // 1: emit forced tokens without the head after each decision (device form only)
  int32_t forced_logits;    // 1: still compute a forced token's logit (one row dot)
  int32_t iv;               // 1: read-only no-repeat state (rank ranges + banned ranks); 0: cnt/spent arrays
  // Sampling instead of the argmax (one-CTA sparse step only)
  int32_t smp;              // 1: sample
  float inv_temp;           // 1 / temperature
  int32_t top_k;            // <= 0: off
  float top_p;              // >= 1: off
  const float* u;           // uniforms: device form [b * out_stride + position], host form [b]
  // Multi-CTA sampling: each CTA leaves its candidates' logits, tokens and
  // edges here by candidate rank, for the sequence's last CTA ([B, cand_cap] each)
  float* smp_lg;
  int32_t* smp_tok;
  int32_t* smp_edge;
  int32_t wide;             // batch above the SM count: the one-CTA step stages x in shared memory
  int32_t multi_xs;         // multi-CTA sparse step: x staged in shared memory (two CTAs per SM)
};

// Cumulative counters kept by the kernels (one atomic per launch / per sequence step).
enum StatSlot {
  kStatStepLaunches = 0,   // step-kernel launches (idle ones included)
  kStatSeqSteps = 1,       // head decisions: one per live sequence per step
  kStatCandRows = 2,       // legal candidates the head evaluated
  kStatResetLaunches = 3,
  kStatForced = 4,         // tokens emitted as forced continuations (no head read)
  kStatUnionRows = 5,      // union head: rows of the union, summed over its steps
  kStatSlots = 6
};

struct ResetParams {
  GrammarView g;
  SeqState* st;
  int32_t* cnt;
  uint32_t* spent;
  int32_t kw;
  int32_t B, k, max_steps;
  int32_t iv;               // 1: read-only no-repeat state (no count arrays to fill)
  uint32_t* seq_ticket;
  Ctrl* ctrl;
  int32_t* gemm_err;        // the GEMM heads' timeout flag, cleared here (null before their first use)
  int32_t* toks;            // optional [B, max_steps] prefill with -1
  float* logits;            // optional [B, max_steps] prefill with 0
  int32_t* lens_out;        // optional
  int32_t* status_out;      // optional
  unsigned long long cond;  // 0: none
  unsigned long long* stats;
};

enum Head { kHeadSparse = 0, kHeadDense = 1, kHeadUnionGemm = 2, kHeadDenseGemm = 3 };

// Number of CTAs per sequence the multi-CTA sparse step uses for a grammar of
// the given largest fan-out at batch B (at most one wave of resident CTAs),
// and the dense step's CTAs per sequence.
// *xs_out: 1 when the step stages x in shared memory for two CTAs per SM.
int sparse_tiles(int max_fanout, int B, int num_sms, int H, int cand_cap, bool const_resident, int* xs_out);
int dense_tiles(int B, int num_sms);

// Opt the step kernels in to kMaxDynamicSmem bytes of dynamic shared memory
// (current device; call once per device before the first launch or capture).
cudaError_t prepare_kernels();
cudaError_t launch_reset(const ResetParams& r, cudaStream_t s);
// pdl: launch as the programmatic dependent of the previous kernel in the stream.
cudaError_t launch_step(const StepParams& p, bool const_resident, int head, int tiles, cudaStream_t s,
                        bool pdl = false);
cudaError_t launch_finalize(const StepParams& p, cudaStream_t s);
// One step of a GEMM head: candidate filter, [union compaction], tcgen05 GEMM
// with masked-argmax epilogue, per-sequence fold and transition.
cudaError_t launch_gemm_step(const StepParams& p, bool const_resident, int head, int gemm_ctas, cudaStream_t s);
cudaError_t launch_root_step(const StepParams& p, bool const_resident, const TileCands* root_tiles, int gemm_ctas,
                             cudaStream_t s);
// Copy a walk image (device memory) into the constant bank, stream-ordered.
cudaError_t const_upload(const void* d_src, size_t bytes, cudaStream_t s);

}  // namespace tcd
