/*
 * tcd.h - C ABI of the trie-constrained greedy decoder for GB300 (sm_103a).
 *
 * The decoder emits exactly k distinct pointers from a finite catalog of
 * token-id strings, separated by a separator token and ended by a stop
 * token, choosing each token greedily by a tied-embedding logit over the
 * legal set only.  It follows "Constraint made cheaper than no constraint"
 * (coreyjames.ai), sections "The grammar as a trie over tokens", "Masked
 * sampling inside the sampler", "The sparse output layer" and "The whole loop
 * on the device"; the legal set is the next-token mask of "GLRMask"
 * (introduction) for that finite language.
 *
 * Conventions for every call:
 *  - Pointers marked (host) are CPU memory, (device) are CUDA device memory of
 *    the context's device.  bf16 values are 16-bit IEEE bfloat16 bit patterns.
 *  - The caller owns every buffer it passes; the library never frees them and
 *    never keeps a host pointer past the call.  Device buffers passed to
 *    tc_decode / tc_decode_graph_create are remembered by the captured graph
 *    and must stay valid while that graph may be launched.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *    that take a stream are asynchronous with respect to the host unless
 *    stated otherwise.
 *  - Argument and compile errors are returned synchronously and leave the
 *    objects unchanged.  Errors found on the device (an empty legal set, a
 *    winner on a dead edge, an index out of range, running out of steps) are
 *    recorded per sequence, stop that sequence only, and are read with
 *    tc_first_error / tc_read_seq_state or the status outputs.
 *  - The library is not thread-safe per object: one host thread at a time
 *    per tc_ctx.  Constant-memory residency is one image per device (see
 *    tc_bind_grammar).
 */
#ifndef TCD_H
#define TCD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum tc_status {
  TC_OK = 0,
  TC_ERR_INVALID_ARG = 1,        /* bad pointer, size or enum value */
  TC_ERR_FANOUT = 2,             /* a node has more edges than max_fanout (control edges count) */
  TC_ERR_DUPLICATE = 3,          /* two catalog strings are equal */
  TC_ERR_CONTROL_COLLISION = 4,  /* a catalog string contains the separator or stop id */
  TC_ERR_TOKEN_RANGE = 5,        /* a token id outside [0, vocab) */
  TC_ERR_EMPTY_STRING = 6,       /* a catalog string has no tokens */
  TC_ERR_K_RANGE = 7,            /* k < 1 or k > number of catalog strings */
  TC_ERR_CONST_CAPACITY = 8,     /* constant residency requested but the walk image's header part does not fit */
  TC_ERR_NOT_BOUND = 9,          /* no grammar bound, or no tc_reset since binding */
  TC_ERR_CAPACITY = 10,          /* batch > max_batch or max fan-out > the candidate buffer */
  TC_ERR_UNSUPPORTED = 11,       /* shape the kernels do not handle (e.g. hidden % 8 != 0) */
  TC_ERR_EMPTY_MASK = 16,        /* device: no legal token at a step */
  TC_ERR_NO_LIVE_EDGE = 17,      /* device: the chosen token sits on no live edge (defensive) */
  TC_ERR_MAX_STEPS = 18,         /* device: the step budget ran out before the stop token */
  TC_ERR_BOUNDS = 19,            /* device: an index of the grammar image or a logit is invalid */
  TC_ERR_DEVICE_TIMEOUT = 20,    /* device: a bounded wait inside a kernel gave up (the kernel returned
                                    without finishing its work; the step fails for every sequence it
                                    served; cleared by tc_reset / the next decode's reset) */
  TC_ERR_CUDA = 32,              /* a CUDA runtime call failed (see tc_last_error_message) */
  TC_ERR_OOM = 33                /* device allocation failed */
} tc_status;

/* Grammar residency (tc_bind_grammar). */
enum {
  TC_RES_AUTO = 0,    /* constant memory when the walk image's header part fits, else global memory */
  TC_RES_CONST = 1,   /* header part (node ranges, pointer ranks) in __constant__ memory, at most
                         TC_CONST_CAPACITY_BYTES; edge records always in global memory */
  TC_RES_GLOBAL = 2   /* the whole walk image in global memory, read through the read-only cache */
};

/*
 * Flag or-ed into the `residency` argument of tc_bind_grammar: keep the
 * per-sequence live-count arrays for every k.  Without it a decode or reset
 * with k <= 8 pointers (and a catalog of at most 65535 strings) uses the
 * read-only no-repeat state ("Constraint made cheaper than no constraint",
 * section "The batched engine": a 16-byte per-sequence banned set against
 * read-only per-edge pointer sets): the pointers below an edge are one range of
 * depth-first ranks stored in the shared edge record, and each sequence keeps
 * the ranks of its completed pointers (at most 8 x 16 bits) in its state, so no
 * per-sequence array is filled at reset or updated on completion.  Both modes
 * give identical results; larger k always uses the count arrays, which are
 * allocated on first use.
 */
#define TC_BIND_LIVE_COUNTS 0x10

/* Output head (tc_step / tc_decode). */
enum {
  TC_HEAD_SPARSE = 0,     /* one embedding-row dot product per legal candidate */
  TC_HEAD_DENSE = 1,      /* every vocabulary row, then the legal mask, then the argmax (cross-check) */
  TC_HEAD_UNION_GEMM = 2, /* batches: the union of all sequences' legal rows as one tcgen05 GEMM,
                             each sequence's argmax over its own candidates (batch <= 256, hidden % 64 == 0) */
  TC_HEAD_DENSE_GEMM = 3  /* batches: every vocabulary row as one tcgen05 GEMM, then each sequence's
                             legal mask and argmax (the dense comparison for TC_HEAD_UNION_GEMM) */
};

/*
 * Flag or-ed into the `head` argument of tc_decode and tc_decode_graph_create:
 * forced continuations ("Understanding Inference for Systems Engineers",
 * section 7.5, forced spans).  After each head decision, while the grammar
 * admits exactly one token at a sequence's node, that token is emitted in the
 * same step without reading the head, and its logit slot is set to NaN; the
 * walk advances through it (pointer completions included).  Emitted tokens
 * are those of the decode without the flag; a sequence's first token always
 * comes from the head, and a forced position's hidden state is not read.  One
 * decode step then covers a decision and the forced span after it, so fewer
 * steps run.  Sparse and dense heads only (the GEMM heads read all sequences'
 * hidden states of one step as one tile, which needs them in lockstep):
 * TC_ERR_UNSUPPORTED otherwise, and from tc_step and tc_decode_host.
 */
#define TC_FLAG_JUMP_FORWARD 0x100

/*
 * Or-ed in together with TC_FLAG_JUMP_FORWARD: forced tokens keep their
 * logits.  Each forced position still takes no head decision, but its token's
 * embedding row is dotted with that position's hidden state (the head's lane
 * map and reduction, so the logit equals the plain decode's bit for bit):
 * tokens and logits are those of the decode without either flag, at one row
 * read per forced token.  Alone: TC_ERR_INVALID_ARG.
 */
#define TC_FLAG_FORCED_LOGITS 0x200

/*
 * Flag or-ed into the `head` argument of tc_decode, tc_decode_graph_create
 * and tc_decode_host together with TC_HEAD_SPARSE (and of tc_step, for the
 * first step after tc_reset): the first step runs on the
 * tcgen05 GEMM ("Constraint made cheaper than no constraint", section "The
 * sparse output layer": in batched form the rows of the legal set are one
 * GEMM).  At that step every sequence is at the root with nothing emitted, so
 * its legal set is the root's token edges, the same for all sequences: one
 * [batch x hidden] x [hidden x root edges] product with each sequence's argmax
 * over all columns (ties to the lower token id), then the transition; later
 * steps use the sparse head.  The first step's logits are fp32 sums of the
 * same bf16 products in the tensor cores' order and K split, so they equal the
 * sparse head's on integer-valued inputs and differ by rounding otherwise (a
 * token may then differ only where two logits are within rounding).  It pays
 * off where the root is wide and the batch large (e.g. a catalog of
 * unstructured strings at 256 sequences) and costs time at small batches.
 * Needs batch <= 256, hidden % 64 == 0 and a root whose edges all lead to
 * pointers (no empty catalog string); TC_ERR_UNSUPPORTED with
 * TC_FLAG_JUMP_FORWARD, sampling or another head.  The device checks that each
 * sequence is at the root with nothing emitted (TC_ERR_BOUNDS otherwise).
 */
#define TC_FLAG_ROOT_GEMM 0x400

/* Bytes of __constant__ memory reserved for the header part of one walk image. */
#define TC_CONST_CAPACITY_BYTES (63 * 1024)

typedef struct tc_trie tc_trie;   /* compiled catalog, host object */
typedef struct tc_ctx tc_ctx;     /* device context: model, bound grammar, per-sequence state */
typedef struct tc_graph tc_graph; /* a captured device-resident decode loop */

typedef struct tc_trie_info_t {
  int32_t n_nodes;          /* N, root is node 0, nodes numbered depth-first (preorder, children in
                               ascending token or byte order) */
  int32_t n_edges;          /* E, token edges plus two control edges per terminal node */
  int32_t n_strings;        /* K, catalog size (pointer ids 0..K-1 in input order) */
  int32_t max_fanout;       /* largest edge count of any node (control edges included) */
  int32_t root_fanout;      /* edge count of the root */
  int32_t max_depth;        /* longest catalog string, in tokens */
  int32_t vocab, sep_id, stop_id;
  int32_t header_bytes;     /* bytes of the walk image's header part (node ranges and pointer
                               ranks): what constant residency places in __constant__ memory */
  int64_t total_tokens;     /* sum of the string lengths */
  int64_t walk_image_bytes; /* bytes of the device walk image: the header part and the 32-byte
                               edge records (token, child, rank range, child header) */
} tc_trie_info_t;

/* ---------------------------------------------------------------- compiler */

/*
 * tc_compile_trie - compile a catalog of token-id strings into a CSR trie
 * ("The grammar as a trie over tokens": an edge range per node, a token and a
 * child per edge, and two sentinel children for the control edges).
 *
 *  ids        (host) int32[offsets[n_strings]]: the strings, concatenated.
 *  offsets    (host) int64[n_strings + 1]: string i is ids[offsets[i] .. offsets[i+1]).
 *  n_strings  K >= 1.  String i becomes pointer id i.
 *  sep_id, stop_id  distinct ids in [0, vocab) used for the two control edges.
 *  vocab      token ids must lie in [0, vocab).
 *  max_fanout refuse any node with more edges than this (the page's cap is
 *             256; control edges count).  Must be >= 2.
 *  out        receives a new tc_trie the caller frees with tc_trie_free.
 *
 * Refusals (nothing is allocated): TC_ERR_EMPTY_STRING, TC_ERR_DUPLICATE,
 * TC_ERR_CONTROL_COLLISION, TC_ERR_TOKEN_RANGE, TC_ERR_FANOUT,
 * TC_ERR_INVALID_ARG.  Host only; needs no GPU.
 */
tc_status tc_compile_trie(const int32_t* ids, const int64_t* offsets, int32_t n_strings,
                          int32_t sep_id, int32_t stop_id, int32_t vocab, int32_t max_fanout,
                          tc_trie** out);

/*
 * tc_trie_info - sizes of a compiled trie into *out (host): node and edge
 * counts, fan-outs, depth and the bytes of its walk image ("The grammar as a
 * trie over tokens": the size of the compiled trie decides whether it fits
 * the constant-memory budget).  Errors: TC_ERR_INVALID_ARG on a NULL argument.
 */
tc_status tc_trie_info(const tc_trie* trie, tc_trie_info_t* out);

/*
 * tc_trie_export - copy the CSR arrays into caller buffers (host), any of
 * which may be NULL.  Sizes from tc_trie_info:
 *  node_begin  int32[N+1]  edges of node n are [node_begin[n], node_begin[n+1])
 *  edge_tok    int32[E]    token of each edge; a node's edges ascend by token
 *  edge_child  int32[E]    child node, or -1 for the separator edge (back to
 *                          the root), -2 for the stop edge
 *  node_ptr    int32[N]    pointer id ending at the node, or -1
 *  static_cnt  int32[E]    pointers ending at or below a token edge's child;
 *                          0 on control edges
 *  path_off    int32[K+1]  pointer p's root-to-terminal token edges are
 *  path        int32[total_tokens]   path[path_off[p] .. path_off[p+1])
 */
tc_status tc_trie_export(const tc_trie* trie, int32_t* node_begin, int32_t* edge_tok,
                         int32_t* edge_child, int32_t* node_ptr, int32_t* static_cnt,
                         int32_t* path_off, int32_t* path);

/*
 * tc_compile_char_trie - compile a character-level grammar: the catalog as
 * byte strings and a byte vocabulary, so that every tokenization of a catalog
 * string is accepted, not only one (the pith.science review of arXiv
 * 2608.12574, key machinery: a character trie of the strings whose nodes carry
 * the vocabulary tokens that can be walked from them without overshooting,
 * found by Aho-Corasick matching of the vocabulary along the trie).
 *
 *  chars, offsets       string i is chars[offsets[i] .. offsets[i+1]) (bytes,
 *                       non-empty, distinct), offsets int64[n_strings + 1]
 *  tok_ids              int32[n_tokens] distinct ids in [0, vocab), none equal
 *                       to sep_id / stop_id
 *  tok_chars, tok_offsets  token j's bytes, non-empty, distinct
 *  max_fanout           cap on any node's edges (token edges + 2 control edges)
 *
 * The result is a tc_trie like tc_compile_trie's: nodes are character-trie
 * nodes numbered depth-first (preorder, children by ascending byte), a node's edges are the tokens that walk from
 * it (a token edge may skip several characters, and several edges may lead to
 * one node) plus the separator and stop edges at a terminal, sorted by token
 * id; static_cnt counts the strings below an edge's target.  It keeps no
 * pointer paths (path_off all 0), so only the read-only no-repeat state
 * applies: k <= 8 pointers, and TC_BIND_LIVE_COUNTS is TC_ERR_UNSUPPORTED.
 * Errors: TC_ERR_INVALID_ARG, TC_ERR_EMPTY_STRING, TC_ERR_DUPLICATE (equal
 * strings, equal token ids or token bytes), TC_ERR_CONTROL_COLLISION,
 * TC_ERR_TOKEN_RANGE, TC_ERR_FANOUT.
 */
tc_status tc_compile_char_trie(const uint8_t* chars, const int64_t* offsets, int32_t n_strings,
                               const int32_t* tok_ids, const uint8_t* tok_chars, const int64_t* tok_offsets,
                               int32_t n_tokens, int32_t sep_id, int32_t stop_id, int32_t vocab,
                               int32_t max_fanout, tc_trie** out);

/*
 * tc_trie_export_ranks - the depth-first pointer numbering behind the
 * read-only no-repeat state ("Constraint made cheaper than no constraint",
 * section "The batched engine": batched sequences share one read-only trie and
 * keep only their own small no-repeat state).  Pointers are ranked in
 * depth-first order (a node's own pointer before those below it, children in
 * token order), so the pointers below any node hold one contiguous range of
 * ranks.  Host buffers, either may be NULL:
 *  ptr_rank  int32[K]  rank of pointer id p
 *  edge_lo   int32[E]  first rank below a token edge's child (the range has
 *                      static_cnt[e] ranks); the terminal's own rank for a
 *                      control edge
 */
tc_status tc_trie_export_ranks(const tc_trie* trie, int32_t* ptr_rank, int32_t* edge_lo);

void tc_trie_free(tc_trie* trie);

/* --------------------------------------------------------------- context */

/*
 * tc_ctx_create - a decoding context on `device` over a tied embedding
 * ("The sparse output layer": the output head is the tied embedding, one row
 * per token; "The batched engine": each sequence of a batch keeps its own
 * small state next to the shared, read-only grammar).
 *
 *  emb_bf16   (device) bf16[vocab, hidden], row-major, 16-byte aligned; the
 *             caller keeps it alive and unchanged while the context is used.
 *  vocab      V >= 2.   hidden  H >= 8 and a multiple of 8.
 *  max_batch  largest batch passed to tc_reset / tc_decode (>= 1).
 *  cand_cap   candidate-buffer capacity C: grammars whose max fan-out exceeds
 *             it are refused at bind (256 for the page's cap; up to 4096).
 *
 * Allocates the context's device scratch (O(max_batch * cand_cap) bytes).
 */
tc_status tc_ctx_create(int32_t device, const void* emb_bf16, int32_t vocab, int32_t hidden,
                        int32_t max_batch, int32_t cand_cap, tc_ctx** out);

/* tc_ctx_destroy - synchronise the device, free every graph, grammar image and buffer. */
void tc_ctx_destroy(tc_ctx* ctx);

/*
 * tc_bind_grammar - make `trie` the context's grammar ("The grammar as a trie
 * over tokens": constant residency is owned by one grammar and re-bound on
 * every switch; a captured graph re-binds at launch).
 *
 * Uploads the trie's image to device memory owned by the context (once per
 * distinct trie content; the trie may be freed afterwards) and allocates its
 * per-sequence state for max_batch sequences.  residency is TC_RES_AUTO,
 * TC_RES_CONST or TC_RES_GLOBAL (optionally or-ed with TC_BIND_LIVE_COUNTS);
 * AUTO picks CONST when the walk image's header part (tc_trie_info's
 * header_bytes) is at most TC_CONST_CAPACITY_BYTES.  With CONST that part is
 * copied into the device's __constant__ bank on `stream` now, before any later tc_step, and
 * as the first node of any graph captured for it.  There is one constant
 * image per device: contexts that use different CONST grammars on
 * concurrently running streams race; use GLOBAL for that.
 *
 * Errors: TC_ERR_TOKEN_RANGE (trie vocab > context vocab), TC_ERR_CAPACITY
 * (max fan-out > cand_cap), TC_ERR_CONST_CAPACITY, TC_ERR_OOM, TC_ERR_CUDA.
 * Binding invalidates the per-sequence state: call tc_reset before tc_step.
 */
tc_status tc_bind_grammar(tc_ctx* ctx, const tc_trie* trie, int32_t residency, void* stream);

/* tc_bound_residency - the residency the bound grammar resolved to (TC_RES_CONST / TC_RES_GLOBAL;
 * "The grammar as a trie over tokens": constant memory for a small catalog, global memory otherwise). */
tc_status tc_bound_residency(const tc_ctx* ctx, int32_t* residency);

/*
 * tc_reset - start `batch` sequences, each owing exactly k pointers, at the
 * root of the bound grammar ("Masked sampling inside the sampler": a query
 * owes exactly k distinct pointers; every pointer starts live, so the live
 * counts start as the static counts and no spent flag is set).  Also clears
 * the GEMM heads' timeout flag (TC_ERR_DEVICE_TIMEOUT).  1 <= batch <= max_batch; 1 <= k <= K (a larger k
 * would make the language empty; TC_ERR_K_RANGE).  Asynchronous on `stream`.
 */
tc_status tc_reset(tc_ctx* ctx, int32_t batch, int32_t k, void* stream);

/*
 * tc_step - one decode step of every sequence of the last tc_reset, driven
 * from the host ("Masked sampling inside the sampler"): mask the current
 * node's edges, one logit per legal token (head = TC_HEAD_SPARSE) or every
 * vocabulary logit then the mask (TC_HEAD_DENSE), argmax with ties to the
 * lower token id, advance the trie, and on a completed pointer decrement the
 * live counts along its path.
 *
 *  hidden_bf16 (device) bf16[batch, hidden]: this step's hidden state per sequence.
 *  tok_out     (device) int32[batch]: the emitted token, or -1 for a sequence
 *              that had already stopped or failed.
 *  logit_out   (device) float[batch]: its fp32 logit (0 for -1 tokens); may be NULL.
 *  status_out  (device) int32[batch]: TC_OK or the sequence's error; may be NULL.
 *
 * The head may change from one call to the next, also inside a captured
 * graph: the sparse step keeps each sequence's next candidate list in its
 * device state, and every other head's step clears it there, so the next
 * sparse step filters that node itself.  TC_HEAD_SPARSE | TC_FLAG_ROOT_GEMM
 * runs the first step after tc_reset as the tensor-core root step (see the
 * flag); a sequence that is not at the root with nothing emitted fails that
 * step with TC_ERR_BOUNDS.
 *
 * Asynchronous on `stream`; a sequence that meets an error stops there.
 */
tc_status tc_step(tc_ctx* ctx, const void* hidden_bf16, int32_t head, int32_t* tok_out,
                  float* logit_out, int32_t* status_out, void* stream);

/*
 * tc_decode - decode `batch` sequences to completion in one device-resident
 * graph ("The whole loop on the device": [re-bind] -> reset -> while (a
 * sequence is live and step < max_steps) { step }, the step counter kept in
 * device memory).  The graph is captured on first use for each distinct
 * argument set and replayed afterwards.
 *
 *  hidden_steps_bf16 (device) bf16[n_steps, batch, hidden]: step t of sequence
 *              b reads hidden_steps[t, b, :].
 *  n_steps     rows available in hidden_steps; 1 <= max_steps <= n_steps.
 *  toks        (device) int32[batch, max_steps]: emitted tokens, -1 after the end.
 *  logits      (device) float[batch, max_steps]: their logits, 0 after the end.
 *  lens        (device) int32[batch]: tokens emitted per sequence.
 *  status      (device) int32[batch]: TC_OK (stopped normally) or the error
 *              (TC_ERR_MAX_STEPS when the budget ran out).
 *
 * Asynchronous on `stream`; the host need not synchronise until it reads the
 * outputs.  Leaves the context's sequences in their final state.
 */
tc_status tc_decode(tc_ctx* ctx, const void* hidden_steps_bf16, int32_t n_steps, int32_t batch,
                    int32_t k, int32_t max_steps, int32_t head, int32_t* toks, float* logits,
                    int32_t* lens, int32_t* status, void* stream);

/*
 * Sampling instead of the greedy argmax ("Understanding Inference for Systems
 * Engineers", section 3.8): the token is drawn from softmax(logit /
 * temperature) over the legal candidates, restricted first to the top_k
 * highest logits - a value threshold, so every candidate tied with the top_k-th
 * largest logit is kept - and then by removing the ascending prefix, in
 * (logit, token id) order, whose probability mass is at most 1 - top_p (the
 * largest is never removed, so among equal probabilities the highest id
 * survives).  The draw is the first kept candidate, in ascending token order,
 * whose cumulative probability exceeds the caller's uniform u in [0, 1).
 * top_k = 0 and top_p = 1 switch the restrictions off.  Sums run in a fixed
 * order, so a draw depends only on the sequence's own inputs.
 */
typedef struct tc_sampling_t {
  float temperature;  /* > 0, finite */
  int32_t top_k;      /* >= 0; 0: no top-k */
  float top_p;        /* in [0, 1]; 1: no top-p */
} tc_sampling_t;

/*
 * tc_decode_sample - tc_decode with sampling.  uniforms (device) float[batch,
 * max_steps]: the uniform of sequence b at output position t is
 * uniforms[b * max_steps + t] (positions filled by forced continuations use
 * none).  Sparse head only (TC_FLAG_JUMP_FORWARD may be or-ed in):
 * TC_ERR_UNSUPPORTED otherwise.  On grammars with a node of more than 32 edges
 * the first call allocates per-context scratch of 12 bytes per candidate slot
 * (max_batch x cand_cap) for the multi-CTA step's candidate logits.  The
 * random numbers are the caller's: the library generates none.
 */
tc_status tc_decode_sample(tc_ctx* ctx, const void* hidden_steps_bf16, int32_t n_steps, int32_t batch,
                           int32_t k, int32_t max_steps, int32_t head, const tc_sampling_t* sampling,
                           const float* uniforms, int32_t* toks, float* logits, int32_t* lens,
                           int32_t* status, void* stream);

/*
 * tc_step_sample - tc_step with sampling; uniforms (device) float[batch], one
 * per sequence for this step.  Same restrictions as tc_decode_sample.
 */
tc_status tc_step_sample(tc_ctx* ctx, const void* hidden_bf16, int32_t head, const tc_sampling_t* sampling,
                         const float* uniforms, int32_t* tok_out, float* logit_out, int32_t* status_out,
                         void* stream);

/*
 * tc_decode_host - the same decode driven from the host: tc_reset, then one
 * tc_step per step with a synchronising read of the live count after each,
 * the comparison loop of "The whole loop on the device".  Same arguments and
 * outputs as tc_decode.  Synchronous.
 */
tc_status tc_decode_host(tc_ctx* ctx, const void* hidden_steps_bf16, int32_t n_steps, int32_t batch,
                         int32_t k, int32_t max_steps, int32_t head, int32_t* toks, float* logits,
                         int32_t* lens, int32_t* status, void* stream);

/*
 * tc_decode_graph_create - capture the tc_decode graph for these arguments
 * without launching it; the caller launches it with tc_graph_launch and frees
 * it with tc_graph_destroy (before tc_ctx_destroy).  The graph keeps using the
 * grammar bound now, even after another grammar is bound: its first node
 * re-binds that grammar's constant image.
 */
tc_status tc_decode_graph_create(tc_ctx* ctx, const void* hidden_steps_bf16, int32_t n_steps,
                                 int32_t batch, int32_t k, int32_t max_steps, int32_t head,
                                 int32_t* toks, float* logits, int32_t* lens, int32_t* status,
                                 tc_graph** out);
tc_status tc_graph_launch(tc_graph* graph, void* stream);
void tc_graph_destroy(tc_graph* graph);

/*
 * tc_first_error - synchronise `stream`, then report the lowest sequence
 * index whose status is not TC_OK (*seq = -1, *code = TC_OK if none)
 * ("Masked sampling inside the sampler": a step with no legal token stops
 * the sequence with an error instead of emitting one; this surfaces it).
 * Errors: TC_ERR_INVALID_ARG, TC_ERR_NOT_BOUND (no reset since binding),
 * TC_ERR_CUDA.
 */
tc_status tc_first_error(tc_ctx* ctx, void* stream, int32_t* seq, int32_t* code);

/*
 * tc_read_seq_state - synchronise `stream` and copy per-sequence state of the
 * last reset's batch into host arrays int32[batch] (any may be NULL): current
 * node, pointers completed, tokens emitted, status, done flag (the walk state
 * of "Masked sampling inside the sampler").
 */
tc_status tc_read_seq_state(tc_ctx* ctx, void* stream, int32_t* node, int32_t* emitted,
                            int32_t* len, int32_t* status, int32_t* done);

/*
 * tc_read_stats - synchronise `stream` and copy the context's cumulative
 * kernel counters into out (host) int64[TC_STAT_SLOTS]: step-kernel launches
 * (idle launches at the end of a graph loop included), head decisions (one
 * per live sequence per step), legal candidates evaluated (rows gathered by
 * the sparse head), reset-kernel launches, tokens emitted as forced
 * continuations (TC_FLAG_JUMP_FORWARD), and the union head's rows (the size
 * of the union of legal rows, summed over its steps).  reset != 0 zeroes them
 * afterwards.
 * Used to count launches and algorithmic bytes.
 */
#define TC_STAT_SLOTS 6
tc_status tc_read_stats(tc_ctx* ctx, void* stream, int64_t* out, int32_t reset);

/*
 * tc_gemm_wait_test - exercise the GEMM heads' error path without any fault
 * ("Constraint made cheaper than no constraint", section "Masked sampling
 * inside the sampler": a step that cannot finish fails loudly).  Every wait
 * of the tcgen05 GEMM kernel on a shared-memory barrier is bounded by a poll
 * count; when one runs out, the kernel stops issuing, waits (again bounded)
 * for the copies and MMAs it started, frees its tensor memory, sets the
 * context's timeout flag and returns; the step then fails every sequence it
 * served with TC_ERR_DEVICE_TIMEOUT, and the next tc_reset (or decode) clears
 * the flag.
 *
 *  withhold    nonzero: in later GEMM-head steps, the kernel's first CTA
 *              issues no copy for its first pipeline stage, so the waits on
 *              that stage run out.  0: normal operation.
 *  wait_polls  polls of one wait before it gives up; 0 restores the default
 *              (2^22).  A small count (e.g. 2000) makes the timeout quick.
 *
 * Test use only; it allocates the GEMM heads' scratch if needed, synchronises
 * the device and drops the context's cached decode graphs (they hold the old
 * settings).  Errors: TC_ERR_INVALID_ARG, TC_ERR_OOM, TC_ERR_CUDA.
 */
tc_status tc_gemm_wait_test(tc_ctx* ctx, int32_t withhold, int64_t wait_polls);

/*
 * tc_dense_argmax_noalloc - the dense head's masked argmax without any device
 * allocation.  The pages have no counterpart: this entry point serves callers
 * that cannot allocate device memory themselves or let a library do it - code
 * running under a framework whose caching allocator owns the device-memory
 * budget, plugin hosts that forbid allocation calls, and latency-critical
 * paths where cudaMalloc or cudaFree may synchronise the device.
 *
 * For each sequence b: logit[v] = sum_h E[v, h] * x[b, h] for every row v
 * (fp32 accumulation, the same lane map and shuffle tree as tc_step, so the
 * result equals tc_step's dense head bit for bit), restricted to the tokens in
 * legal[b, 0 .. n_legal[b]) (ascending ids), then the largest logit with ties
 * to the lower id.
 *
 *  emb_bf16     (device) bf16[vocab, hidden], 16-byte aligned.
 *  hidden_bf16  (device) bf16[batch, hidden], 16-byte aligned; hidden % 8 == 0,
 *               hidden <= TC_NOALLOC_MAX_HIDDEN.
 *  legal        (device) int32[batch, legal_stride]; legal_stride <=
 *               TC_NOALLOC_MAX_LEGAL.  n_legal (device) int32[batch].
 *  tok_out      (device) int32[batch]: the winner, or -1 when no listed token
 *               has a comparable logit (empty list, or NaN logits).
 *  logit_out    (device) float[batch]: its logit (0 with -1).
 *  1 <= batch <= TC_NOALLOC_MAX_BATCH.  Sizes beyond the limits return
 *  TC_ERR_CAPACITY with a message in tc_last_error_message.
 *
 * Memory: it calls no allocating routine.  Its scratch is a file-scope
 * __device__ array of TC_NOALLOC_MAX_SLOTS 8-byte partial results plus
 * TC_NOALLOC_MAX_BATCH counters (about 64 KiB), which every GPU that loads the
 * library holds until the process exits.  The first call on a device looks up
 * the array's device address (once per device, with that device current);
 * make that first call before any stream capture.  Every call shares the
 * array and clears the counters it uses with a stream-ordered memset; calls
 * that overlap on the GPU (for example on two streams) race and give wrong
 * results.  Runs on the current device, asynchronously on `stream`.
 */
#define TC_NOALLOC_MAX_BATCH 64
#define TC_NOALLOC_MAX_SLOTS 8192
#define TC_NOALLOC_MAX_HIDDEN 8192
#define TC_NOALLOC_MAX_LEGAL 4096
tc_status tc_dense_argmax_noalloc(const void* emb_bf16, int32_t vocab, int32_t hidden,
                                  const void* hidden_bf16, int32_t batch, const int32_t* legal,
                                  int32_t legal_stride, const int32_t* n_legal, int32_t* tok_out,
                                  float* logit_out, void* stream);

/*
 * tc_loop_floor - the launch floor of tc_decode's loop ("Constraint made
 * cheaper than no constraint": a do-nothing kernel launched in the sampler's
 * place separates the cost of adding a kernel from the cost of its work).
 * Builds the decode graph's shape - an arming kernel, then a conditional WHILE
 * node whose body chains the step's launches, one CTA of 256 threads per
 * sequence (grid 1 x batch), with programmatic dependent launch - with
 * do-nothing kernels in the steps' place, runs `iterations` body iterations
 * once untimed and once timed (CUDA events on `stream`), and returns the timed
 * launch's milliseconds in *ms_out and its kernel launches in *launches_out.
 * Synchronous; allocates and frees its own 4-byte counter and stream.
 */
tc_status tc_loop_floor(int32_t device, int32_t batch, int32_t iterations, void* stream, float* ms_out,
                        int64_t* launches_out);

/* tc_status_str - a static name for a status code. */
const char* tc_status_str(tc_status status);

/* tc_last_error_message - detail of the last error on this host thread (static storage). */
const char* tc_last_error_message(void);

#ifdef __cplusplus
}
#endif

#endif /* TCD_H */
