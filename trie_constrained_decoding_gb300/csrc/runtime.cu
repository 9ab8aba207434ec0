// Runtime behind the C ABI: contexts, grammar residency, per-sequence state,
// host-driven steps and the device-resident decode loop (CUDA graph with a
// conditional WHILE node).
//
// "Constraint made cheaper than no constraint", section "The grammar as a
// trie over tokens": constant residency is owned by one grammar and re-bound
// on every switch, and a captured graph re-binds at launch because replay
// does not repeat the host upload.  Here the owner of the device's constant
// bank is tracked per device; a host-driven step re-copies the bound image
// when another grammar owns the bank, and every captured graph starts with a
// device-to-device copy node of its own grammar's image.
//
// Section "The whole loop on the device": the loop is one captured graph - a
// reset, then a conditional body that runs the step while the predicate
// holds - with every loop-varying value (step, live count) in device memory;
// the kernels have a host-argument form (tc_step) and a device-pointer form
// (the graph body) sharing one body.  "Understanding Inference for Systems
// Engineers", section 6.2, makes the same choice: a small control block in
// device memory so that the graph is captured once and replayed unchanged.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstddef>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "gemm_tc.h"
#include "kernels.h"
#include "tcd.h"
#include "tcd_internal.h"

using namespace tcd;

namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kGraphCacheSize = 16;

std::mutex g_const_mu;
const void* g_const_owner[kMaxDevices];  // grammar whose image the constant bank holds

tc_status cuda_fail(cudaError_t e, const char* what) {
  set_error_message(std::string(what) + ": " + cudaGetErrorString(e));
  cudaGetLastError();  // clear a sticky-free error so later calls start clean
  return e == cudaErrorMemoryAllocation ? TC_ERR_OOM : TC_ERR_CUDA;
}

#define TC_CUDA(call)                                      \
  do {                                                     \
    cudaError_t e_ = (call);                               \
    if (e_ != cudaSuccess) return cuda_fail(e_, #call);    \
  } while (0)

bool misaligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; }

struct DeviceGuard {
  int prev = -1;
  bool changed = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) == cudaSuccess && prev != dev) {
      changed = cudaSetDevice(dev) == cudaSuccess;
    }
  }
  ~DeviceGuard() {
    if (changed) cudaSetDevice(prev);
  }
};

}  // namespace

// A grammar resident on the device, with the per-sequence state of its batch.
struct DevGrammar {
  uint64_t hash = 0;
  int32_t residency = TC_RES_GLOBAL;  // resolved: CONST or GLOBAL
  int32_t n_nodes = 0, n_edges = 0, n_strings = 0, max_fanout = 0, max_depth = 0;
  WalkLayout layout{};
  int32_t* d_img = nullptr;
  int32_t* d_static_cnt = nullptr;
  int32_t* d_path_off = nullptr;
  int32_t* d_path = nullptr;
  SeqState* d_st = nullptr;
  int32_t* d_cnt = nullptr;
  uint32_t* d_spent = nullptr;
  Cand* d_pre = nullptr;  // [max_batch, 32] next-step candidate lists
  // Root step (TC_FLAG_ROOT_GEMM): the root's token edges as GEMM columns:
  // tokens [n_root], edge indices [n_root], then one TileCands record per 128
  // columns at word root_tiles_off (16-byte aligned).
  int32_t* d_root = nullptr;
  int32_t n_root = 0;  // 0: the root step does not apply (the root has a control edge or an edge without pointers)
  int32_t root_tiles_off = 0;
  int32_t root_beg = 0, root_end = 0, root_pid = -1;
  int32_t kw = 1;
  int32_t batch = 0, k = 0;  // of the last reset (0: none)
  bool force_counts = false;  // TC_BIND_LIVE_COUNTS: per-sequence count arrays for every k
  bool no_counts = false;     // character-level grammar: no pointer paths, read-only state only
  int32_t iv = 0;             // state mode of the last reset (1: read-only no-repeat state)
  size_t cnt_batch = 0;       // sequences the count arrays (allocated on first use) hold

  GrammarView view() const {
    GrammarView v;
    v.img = d_img;
    v.off_edges = layout.off_edges;
    v.off_ptr = layout.off_ptr;
    v.root_beg = root_beg;
    v.root_end = root_end;
    v.root_pid = root_pid;
    v.n_nodes = n_nodes;
    v.n_edges = n_edges;
    v.n_strings = n_strings;
    v.static_cnt = d_static_cnt;
    v.path_off = d_path_off;
    v.path = d_path;
    return v;
  }
  void release() {
    cudaFree(d_img);
    cudaFree(d_static_cnt);
    cudaFree(d_path_off);
    cudaFree(d_path);
    cudaFree(d_st);
    cudaFree(d_cnt);
    cudaFree(d_spent);
    cudaFree(d_pre);
    cudaFree(d_root);
  }
};

// Sampling arguments as the kernels take them (smp = 0: greedy).
struct SampleArgs {
  int32_t smp = 0;
  float inv_temp = 1.f;
  int32_t top_k = 0;
  float top_p = 1.f;
  const float* u = nullptr;
  bool operator==(const SampleArgs& o) const {
    return smp == o.smp && (!smp || (inv_temp == o.inv_temp && top_k == o.top_k && top_p == o.top_p && u == o.u));
  }
};

struct GraphKey {
  const DevGrammar* g;
  const void* hidden;
  int32_t n_steps, batch, k, max_steps, head;
  void *toks, *logits, *lens, *status;
  SampleArgs smp;
  bool operator==(const GraphKey& o) const {
    return g == o.g && hidden == o.hidden && n_steps == o.n_steps && batch == o.batch && k == o.k &&
           max_steps == o.max_steps && head == o.head && toks == o.toks && logits == o.logits &&
           lens == o.lens && status == o.status && smp == o.smp;
  }
};

struct tc_graph {
  tc_ctx* ctx = nullptr;
  DevGrammar* g = nullptr;
  GraphKey key{};
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  bool cached = false;  // owned by the context's cache
};

struct tc_ctx {
  int device = 0;
  int num_sms = 148;
  const uint16_t* emb = nullptr;
  int32_t V = 0, H = 0, max_batch = 0, cand_cap = 0;
  std::vector<DevGrammar*> grammars;
  DevGrammar* bound = nullptr;
  Partial* d_part = nullptr;
  uint32_t* d_seq_ticket = nullptr;
  Ctrl* d_ctrl = nullptr;
  unsigned long long* d_stats = nullptr;
  float* d_smp_lg = nullptr;       // multi-CTA sampling scratch [max_batch, cand_cap], on first use
  int32_t* d_smp_tok = nullptr;
  int32_t* d_smp_edge = nullptr;
  HeadScratch hs{};           // GEMM-head scratch, allocated on first use
  EmbMaps emb_maps{};         // tensor maps of the embedding for the GEMM heads
  bool hs_ready = false;
  int32_t* h_live = nullptr;  // pinned
  cudaStream_t capture_stream = nullptr;
  std::vector<tc_graph*> cache;  // most recently used last
  std::vector<tc_graph*> owned;  // created by tc_decode_graph_create
};

namespace {

// Grammars whose nodes have at most 32 edges take the one-CTA sparse step,
// which also precomputes the next step's candidates.
bool one_cta_sparse(const DevGrammar* g) { return g->max_fanout <= 32; }

int tiles_for(const tc_ctx* c, const DevGrammar* g, int head, int B, int* xs = nullptr) {
  if (xs) *xs = 0;
  if (head == TC_HEAD_SPARSE && one_cta_sparse(g)) return 1;
  return head == TC_HEAD_SPARSE ? sparse_tiles(g->max_fanout, B, c->num_sms, c->H, c->cand_cap,
                                              g->residency == TC_RES_CONST, xs)
                                 : dense_tiles(B, c->num_sms);
}

bool is_gemm_head(int head) { return head == TC_HEAD_UNION_GEMM || head == TC_HEAD_DENSE_GEMM; }

int gemm_ctas(const tc_ctx* c, int head) {
  const int tasks = c->hs.max_tiles * (head == TC_HEAD_UNION_GEMM ? c->hs.ksplit : 1);
  return std::min(c->num_sms, tasks);
}

// Scratch of the GEMM heads, sized for max_batch sequences and the whole vocabulary.
tc_status ensure_gemm_scratch(tc_ctx* c) {
  if (c->hs_ready) return TC_OK;
  HeadScratch& h = c->hs;
  const size_t BC = (size_t)c->max_batch * c->cand_cap, V = (size_t)c->V;
  h.max_tiles = (int32_t)((V + gemm_tile_cols() - 1) / gemm_tile_cols());
  cudaError_t e = cudaMalloc(&h.cand_tok, BC * 4);
  if (e == cudaSuccess) e = cudaMalloc(&h.cand_edge, BC * 4);
  if (e == cudaSuccess) e = cudaMalloc(&h.cand_col, BC * 4);
  if (e == cudaSuccess) e = cudaMalloc(&h.ncand, (size_t)c->max_batch * 4);
  if (e == cudaSuccess) e = cudaMalloc(&h.errf, (size_t)c->max_batch * 4);
  if (e == cudaSuccess) e = cudaMalloc(&h.xrow, (size_t)c->max_batch * 8);
  if (e == cudaSuccess) e = cudaMalloc(&h.ubits, ((V + 31) / 32) * 4);
  if (e == cudaSuccess) e = cudaMemset(h.ubits, 0, ((V + 31) / 32) * 4);
  if (e == cudaSuccess) e = cudaMalloc(&h.ulist, V * 4);
  if (e == cudaSuccess) e = cudaMalloc(&h.umap, V * 4);
  if (e == cudaSuccess) e = cudaMalloc(&h.n_union, 4);
  if (e == cudaSuccess) e = cudaMemset(h.n_union, 0, 4);
  if (e == cudaSuccess) e = cudaMalloc(&h.part, (size_t)c->max_batch * h.max_tiles * sizeof(GemmPartial));
  if (e == cudaSuccess) e = cudaMalloc(&h.tile_cands, (size_t)c->max_batch * h.max_tiles * sizeof(TileCands));
  // The union GEMM splits K into tasks of 4 k-steps (256 elements) when the
  // hidden size allows; the split count depends only on the hidden size, so a
  // sequence's sums never depend on its batch-mates.
  h.ksplit = (c->H / 64) % 4 == 0 ? c->H / 256 : 1;
  if (e == cudaSuccess && h.ksplit > 1) e = cudaMalloc(&h.split_part, (size_t)h.ksplit * BC * 4);
  if (e == cudaSuccess) e = cudaMalloc(&h.gemm_err, 4);
  if (e == cudaSuccess) e = cudaMalloc(&h.row0, 4);
  if (e == cudaSuccess) e = cudaMemset(h.row0, 0, 4);
  if (e == cudaSuccess) e = encode_emb_maps(c->emb, c->V, c->H, &c->emb_maps);
  h.emb_maps = &c->emb_maps;
  if (e == cudaSuccess) e = cudaMemset(h.gemm_err, 0, 4);
  if (e != cudaSuccess) return cuda_fail(e, "GEMM-head scratch");
  c->hs_ready = true;
  return TC_OK;
}

void free_gemm_scratch(tc_ctx* c) {
  HeadScratch& h = c->hs;
  cudaFree(h.cand_tok);
  cudaFree(h.cand_edge);
  cudaFree(h.cand_col);
  cudaFree(h.ncand);
  cudaFree(h.errf);
  cudaFree(h.xrow);
  cudaFree(h.ubits);
  cudaFree(h.ulist);
  cudaFree(h.umap);
  cudaFree(h.n_union);
  cudaFree(h.part);
  cudaFree(h.tile_cands);
  cudaFree(h.split_part);
  cudaFree(h.gemm_err);
  cudaFree(h.row0);
  c->hs_ready = false;
}

// Checks shared by every entry point that runs a step with `head`.
tc_status check_head(tc_ctx* c, int head, int B) {
  if (head != TC_HEAD_SPARSE && head != TC_HEAD_DENSE && !is_gemm_head(head)) return TC_ERR_INVALID_ARG;
  if (is_gemm_head(head)) {
    if (B > 256 || c->H % 64 != 0) {
      set_error_message("GEMM heads need batch <= 256 and hidden % 64 == 0");
      return TC_ERR_UNSUPPORTED;
    }
    return ensure_gemm_scratch(c);
  }
  return TC_OK;
}

// One step of any head.
cudaError_t launch_any_step(tc_ctx* c, DevGrammar* g, const StepParams& p, int head, cudaStream_t s, bool pdl) {
  const bool cst = g->residency == TC_RES_CONST;
  if (is_gemm_head(head)) {
    StepParams q = p;
    q.hs = c->hs;
    return launch_gemm_step(q, cst, head, gemm_ctas(c, head), s);
  }
  StepParams q = p;
  const int tiles = tiles_for(c, g, head, p.B, &q.multi_xs);
  return launch_step(q, cst, head, tiles, s, pdl);
}

// The root step of TC_FLAG_ROOT_GEMM: every sequence at the root (the first
// step after a reset), its candidates the root's token edges, on the tcgen05
// GEMM.  p is the step's parameters as for the sparse head.
cudaError_t launch_root(tc_ctx* c, DevGrammar* g, const StepParams& p, cudaStream_t s) {
  StepParams q = p;
  q.hs = c->hs;
  q.hs.n_root = g->n_root;
  q.hs.root_tok = g->d_root;
  q.hs.root_edge = g->d_root + g->n_root;
  const TileCands* tiles = reinterpret_cast<const TileCands*>(g->d_root + g->root_tiles_off);
  const int tasks = (g->n_root + gemm_tile_cols() - 1) / gemm_tile_cols() * c->hs.ksplit * (p.B > 128 ? 2 : 1);
  return launch_root_step(q, g->residency == TC_RES_CONST, tiles, std::min(c->num_sms, tasks), s);
}

StepParams step_params(const tc_ctx* c, const DevGrammar* g, int B) {
  StepParams p{};
  p.g = g->view();
  p.emb = c->emb;
  p.V = c->V;
  p.H = c->H;
  p.st = g->d_st;
  p.cnt = g->d_cnt;
  p.spent = g->d_spent;
  p.kw = g->kw;
  p.B = B;
  p.cand_cap = c->cand_cap;
  p.part = c->d_part;
  p.seq_ticket = c->d_seq_ticket;
  p.ctrl = c->d_ctrl;
  p.stats = c->d_stats;
  p.max_steps = INT32_MAX;
  p.pre = g->d_pre;
  p.one_cta = one_cta_sparse(g) ? 1 : 0;
  p.iv = g->iv;
  p.smp_lg = c->d_smp_lg;
  p.smp_tok = c->d_smp_tok;
  p.smp_edge = c->d_smp_edge;
  p.wide = B > c->num_sms ? 1 : 0;
  return p;
}

// The read-only no-repeat state serves k <= kBanMax pointers (16-bit ranks);
// larger k, or a grammar bound with TC_BIND_LIVE_COUNTS, uses count arrays.
bool use_iv(const DevGrammar* g, int k) {
  return !g->force_counts && k <= kBanMax && g->n_strings <= kBanMaxStrings;
}

// Count arrays of max_batch sequences, allocated the first time count mode runs.
tc_status ensure_counts(const tc_ctx* c, DevGrammar* g) {
  if (g->no_counts) {
    set_error_message("a character-level grammar keeps no live-count arrays: k must be at most " +
                      std::to_string(kBanMax));
    return TC_ERR_UNSUPPORTED;
  }
  if (g->d_cnt) return TC_OK;
  const size_t n = (size_t)c->max_batch * (size_t)std::max<int32_t>(1, g->n_edges);
  cudaError_t e = cudaMalloc(&g->d_cnt, sizeof(int32_t) * n);
  if (e != cudaSuccess) {
    g->d_cnt = nullptr;
    cudaGetLastError();
    set_error_message("live-count arrays: " + std::string(cudaGetErrorString(e)));
    return TC_ERR_OOM;
  }
  g->cnt_batch = (size_t)c->max_batch;
  return TC_OK;
}

ResetParams reset_params(const tc_ctx* c, const DevGrammar* g, int B, int k, int max_steps) {
  ResetParams r{};
  r.iv = use_iv(g, k) ? 1 : 0;
  r.g = g->view();
  r.st = g->d_st;
  r.cnt = g->d_cnt;
  r.spent = g->d_spent;
  r.kw = g->kw;
  r.B = B;
  r.k = k;
  r.max_steps = max_steps;
  r.seq_ticket = c->d_seq_ticket;
  r.ctrl = c->d_ctrl;
  r.stats = c->d_stats;
  r.gemm_err = c->hs_ready ? c->hs.gemm_err : nullptr;
  return r;
}

// Re-copy g's walk image into the constant bank unless g already owns it.
tc_status ensure_const(tc_ctx* c, DevGrammar* g, cudaStream_t s) {
  if (g->residency != TC_RES_CONST) return TC_OK;
  std::lock_guard<std::mutex> lk(g_const_mu);
  if (g_const_owner[c->device] == g) return TC_OK;
  TC_CUDA(const_upload(g->d_img, (size_t)g->layout.header_words * 4, s));
  g_const_owner[c->device] = g;
  return TC_OK;
}

tc_status check_decode_args(tc_ctx* c, const void* hidden, int32_t n_steps, int32_t batch, int32_t k,
                            int32_t max_steps, int32_t head, int32_t* toks, float* logits, int32_t* lens,
                            int32_t* status) {
  if (!c || !hidden || !toks || !logits || !lens || !status) return TC_ERR_INVALID_ARG;
  if (misaligned(hidden, 16) || misaligned(toks, 4) || misaligned(logits, 4) || misaligned(lens, 4) ||
      misaligned(status, 4)) {
    set_error_message("hidden states must be 16-byte aligned and outputs 4-byte aligned");
    return TC_ERR_INVALID_ARG;
  }
  if (!c->bound) return TC_ERR_NOT_BOUND;
  if (batch < 1 || batch > c->max_batch) return TC_ERR_CAPACITY;
  if (k < 1 || k > c->bound->n_strings) return TC_ERR_K_RANGE;
  if (max_steps < 1 || max_steps > n_steps) return TC_ERR_INVALID_ARG;
  if (head & TC_FLAG_ROOT_GEMM) {
    head &= ~TC_FLAG_ROOT_GEMM;
    if (head != TC_HEAD_SPARSE) {
      set_error_message("TC_FLAG_ROOT_GEMM: the sparse head without forced continuations only");
      return TC_ERR_UNSUPPORTED;
    }
    if (c->bound->n_root == 0) {
      set_error_message("TC_FLAG_ROOT_GEMM: the grammar's root has a control edge or an edge without pointers");
      return TC_ERR_UNSUPPORTED;
    }
    return check_head(c, TC_HEAD_UNION_GEMM, batch);  // the GEMM's limits and scratch
  }
  if ((head & TC_FLAG_FORCED_LOGITS) && !(head & TC_FLAG_JUMP_FORWARD)) {
    set_error_message("TC_FLAG_FORCED_LOGITS needs TC_FLAG_JUMP_FORWARD");
    return TC_ERR_INVALID_ARG;
  }
  head &= ~TC_FLAG_FORCED_LOGITS;
  if (head & TC_FLAG_JUMP_FORWARD) {
    head &= ~TC_FLAG_JUMP_FORWARD;
    if (head != TC_HEAD_SPARSE && head != TC_HEAD_DENSE) {
      set_error_message("TC_FLAG_JUMP_FORWARD: sparse and dense heads only");
      return is_gemm_head(head) ? TC_ERR_UNSUPPORTED : TC_ERR_INVALID_ARG;
    }
  }
  return check_head(c, head, batch);
}

void apply_sampling(StepParams& p, const SampleArgs& a) {
  p.smp = a.smp;
  p.inv_temp = a.inv_temp;
  p.top_k = a.top_k;
  p.top_p = a.top_p;
  p.u = a.u;
}

// Sampling runs in the one-CTA sparse step (grammars whose nodes have at most
// 32 edges); temperature > 0 and finite, top_k >= 0, top_p in [0, 1].
tc_status check_sampling(tc_ctx* c, const DevGrammar* g, int head, const tc_sampling_t* sp, const float* u,
                         SampleArgs* out) {
  if (!sp || !u || misaligned(u, 4)) {
    set_error_message("sampling: parameters and 4-byte aligned uniforms are required");
    return TC_ERR_INVALID_ARG;
  }
  if (!(sp->temperature > 0.f) || !std::isfinite(sp->temperature) || sp->top_k < 0 || !(sp->top_p >= 0.f) ||
      sp->top_p > 1.f) {
    set_error_message("sampling: temperature must be positive and finite, top_k >= 0, 0 <= top_p <= 1");
    return TC_ERR_INVALID_ARG;
  }
  if ((head & ~(TC_FLAG_JUMP_FORWARD | TC_FLAG_FORCED_LOGITS)) != TC_HEAD_SPARSE || !g) {
    set_error_message("sampling: sparse head only (without TC_FLAG_ROOT_GEMM)");
    return TC_ERR_UNSUPPORTED;
  }
  if (!one_cta_sparse(g) && !c->d_smp_lg) {
    // The multi-CTA step hands every candidate's logit to the sequence's last CTA.
    const size_t n = (size_t)c->max_batch * (size_t)c->cand_cap;
    cudaError_t e = cudaMalloc(&c->d_smp_lg, n * sizeof(float));
    if (e == cudaSuccess) e = cudaMalloc(&c->d_smp_tok, n * sizeof(int32_t));
    if (e == cudaSuccess) e = cudaMalloc(&c->d_smp_edge, n * sizeof(int32_t));
    if (e != cudaSuccess) {
      cudaFree(c->d_smp_lg);
      cudaFree(c->d_smp_tok);
      cudaFree(c->d_smp_edge);
      c->d_smp_lg = nullptr;
      c->d_smp_tok = c->d_smp_edge = nullptr;
      cudaGetLastError();
      set_error_message("sampling scratch: " + std::string(cudaGetErrorString(e)));
      return TC_ERR_OOM;
    }
  }
  out->smp = 1;
  out->inv_temp = 1.f / sp->temperature;
  out->top_k = sp->top_k;
  out->top_p = sp->top_p;
  out->u = u;
  return TC_OK;
}

void destroy_graph(tc_graph* gr) {
  if (!gr) return;
  if (gr->exec) cudaGraphExecDestroy(gr->exec);
  if (gr->graph) cudaGraphDestroy(gr->graph);
  delete gr;
}

// Capture: [constant re-bind] -> reset -> WHILE(cond) { step }.
tc_status build_graph(tc_ctx* c, DevGrammar* g, const GraphKey& key, tc_graph** out) {
  if (!use_iv(g, key.k)) {
    tc_status rc0 = ensure_counts(c, g);  // no allocation during capture
    if (rc0 != TC_OK) return rc0;
  }
  auto* gr = new tc_graph();
  gr->ctx = c;
  gr->g = g;
  gr->key = key;
  cudaStream_t cs = c->capture_stream;
  cudaGraphConditionalHandle cond = 0;
  tc_status rc = TC_OK;
  auto fail = [&](cudaError_t e, const char* what) {
    cudaStreamCaptureStatus st;
    if (cudaStreamIsCapturing(cs, &st) == cudaSuccess && st != cudaStreamCaptureStatusNone) {
      cudaGraph_t junk = nullptr;
      cudaStreamEndCapture(cs, &junk);
      if (junk && junk != gr->graph) cudaGraphDestroy(junk);
    }
    rc = cuda_fail(e, what);
    destroy_graph(gr);
    return rc;
  };
  cudaError_t e;
  if ((e = cudaGraphCreate(&gr->graph, 0)) != cudaSuccess) return fail(e, "cudaGraphCreate");
  if ((e = cudaGraphConditionalHandleCreate(&cond, gr->graph, 0, 0)) != cudaSuccess)
    return fail(e, "cudaGraphConditionalHandleCreate");
  if ((e = cudaStreamBeginCaptureToGraph(cs, gr->graph, nullptr, nullptr, 0, cudaStreamCaptureModeThreadLocal)) !=
      cudaSuccess)
    return fail(e, "cudaStreamBeginCaptureToGraph");
  if (g->residency == TC_RES_CONST) {
    if ((e = const_upload(g->d_img, (size_t)g->layout.header_words * 4, cs)) != cudaSuccess)
      return fail(e, "constant re-bind node");
  }
  ResetParams r = reset_params(c, g, key.batch, key.k, key.max_steps);
  r.toks = static_cast<int32_t*>(key.toks);
  r.logits = static_cast<float*>(key.logits);
  r.lens_out = static_cast<int32_t*>(key.lens);
  r.status_out = static_cast<int32_t*>(key.status);
  r.cond = (unsigned long long)cond;
  if ((e = launch_reset(r, cs)) != cudaSuccess) return fail(e, "reset kernel capture");
  StepParams p = step_params(c, g, key.batch);
  p.hidden = static_cast<const uint16_t*>(key.hidden);
  p.hidden_rows = (int64_t)key.n_steps * key.batch;
  p.tok_out = static_cast<int32_t*>(key.toks);
  p.logit_out = static_cast<float*>(key.logits);
  p.status_out = static_cast<int32_t*>(key.status);
  p.lens_out = static_cast<int32_t*>(key.lens);
  p.out_stride = key.max_steps;
  p.max_steps = key.max_steps;
  p.cond = (unsigned long long)cond;
  p.device_form = 1;
  p.jump = (key.head & TC_FLAG_JUMP_FORWARD) ? 1 : 0;
  p.forced_logits = (key.head & TC_FLAG_FORCED_LOGITS) ? 1 : 0;
  p.iv = r.iv;
  apply_sampling(p, key.smp);
  if (key.head & TC_FLAG_ROOT_GEMM) {
    // The first step, every sequence at the root, on the tensor cores; the
    // loop then continues with the sparse head.
    p.loop_ctrl = 0;
    if ((e = launch_root(c, g, p, cs)) != cudaSuccess) return fail(e, "root step capture");
  }
  cudaStreamCaptureStatus cst;
  cudaGraph_t cap_graph = nullptr;
  const cudaGraphNode_t* deps = nullptr;
  const cudaGraphEdgeData* edata = nullptr;
  size_t ndeps = 0;
  if ((e = cudaStreamGetCaptureInfo(cs, &cst, nullptr, &cap_graph, &deps, &edata, &ndeps)) != cudaSuccess)
    return fail(e, "cudaStreamGetCaptureInfo");
  cudaGraphNodeParams np{};
  np.type = cudaGraphNodeTypeConditional;
  np.conditional.handle = cond;
  np.conditional.type = cudaGraphCondTypeWhile;
  np.conditional.size = 1;
  cudaGraphNode_t cnode = nullptr;
  if ((e = cudaGraphAddNode(&cnode, cap_graph, deps, edata, ndeps, &np)) != cudaSuccess)
    return fail(e, "cudaGraphAddNode(conditional)");
  cudaGraph_t body = np.conditional.phGraph_out[0];
  if ((e = cudaStreamUpdateCaptureDependencies(cs, &cnode, nullptr, 1, cudaStreamSetCaptureDependencies)) !=
      cudaSuccess)
    return fail(e, "cudaStreamUpdateCaptureDependencies");
  cudaGraph_t ended = nullptr;
  if ((e = cudaStreamEndCapture(cs, &ended)) != cudaSuccess) return fail(e, "cudaStreamEndCapture");

  if ((e = cudaStreamBeginCaptureToGraph(cs, body, nullptr, nullptr, 0, cudaStreamCaptureModeThreadLocal)) !=
      cudaSuccess)
    return fail(e, "cudaStreamBeginCaptureToGraph(body)");
  const int head = key.head & ~(TC_FLAG_JUMP_FORWARD | TC_FLAG_FORCED_LOGITS | TC_FLAG_ROOT_GEMM);
  // The body runs kLoopUnroll steps; only the last sets the loop condition.
  // A sequence that has stopped makes the remaining steps of the body no-ops.
  for (int u = 0; u < kLoopUnroll; ++u) {
    p.loop_ctrl = (u == kLoopUnroll - 1);
    if ((e = launch_any_step(c, g, p, head, cs, /*pdl=*/u > 0)) != cudaSuccess)
      return fail(e, "step kernel capture");
  }
  cudaGraph_t body_ended = nullptr;
  if ((e = cudaStreamEndCapture(cs, &body_ended)) != cudaSuccess) return fail(e, "cudaStreamEndCapture(body)");
  if ((e = cudaGraphInstantiate(&gr->exec, gr->graph, 0)) != cudaSuccess) return fail(e, "cudaGraphInstantiate");
  *out = gr;
  return TC_OK;
}

tc_status launch_graph(tc_graph* gr, cudaStream_t s) {
  tc_ctx* c = gr->ctx;
  TC_CUDA(cudaGraphLaunch(gr->exec, s));
  if (gr->g->residency == TC_RES_CONST) {
    std::lock_guard<std::mutex> lk(g_const_mu);
    g_const_owner[c->device] = gr->g;
  }
  gr->g->batch = gr->key.batch;
  gr->g->k = gr->key.k;
  gr->g->iv = use_iv(gr->g, gr->key.k) ? 1 : 0;
  return TC_OK;
}

}  // namespace

extern "C" tc_status tc_ctx_create(int32_t device, const void* emb_bf16, int32_t vocab, int32_t hidden,
                                   int32_t max_batch, int32_t cand_cap, tc_ctx** out) {
  if (!out) return TC_ERR_INVALID_ARG;
  *out = nullptr;
  if (device < 0 || device >= kMaxDevices || !emb_bf16 || vocab < 2 || hidden < 8 || max_batch < 1 ||
      cand_cap < 2 || cand_cap > kMaxCandCap) {
    set_error_message("tc_ctx_create: invalid arguments");
    return TC_ERR_INVALID_ARG;
  }
  if (hidden % 8 != 0 || hidden > kMaxHidden || (reinterpret_cast<uintptr_t>(emb_bf16) & 15) != 0) {
    set_error_message("tc_ctx_create: hidden must be a multiple of 8 (<= 16384) and the embedding 16-byte aligned");
    return TC_ERR_UNSUPPORTED;
  }
  DeviceGuard dg(device);
  int cur = -1;
  TC_CUDA(cudaGetDevice(&cur));
  if (cur != device) return TC_ERR_CUDA;
  auto* c = new tc_ctx();
  c->device = device;
  c->emb = static_cast<const uint16_t*>(emb_bf16);
  c->V = vocab;
  c->H = hidden;
  c->max_batch = max_batch;
  c->cand_cap = cand_cap;
  cudaError_t e = cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, device);
  if (e == cudaSuccess) e = prepare_kernels();
  if (e == cudaSuccess) e = prepare_gemm();
  if (e == cudaSuccess) e = cudaMalloc(&c->d_part, sizeof(Partial) * (size_t)max_batch * kMaxTiles);
  if (e == cudaSuccess) e = cudaMalloc(&c->d_seq_ticket, sizeof(uint32_t) * (size_t)max_batch);
  if (e == cudaSuccess) e = cudaMalloc(&c->d_ctrl, sizeof(Ctrl));
  if (e == cudaSuccess) e = cudaMalloc(&c->d_stats, sizeof(unsigned long long) * kStatSlots);
  if (e == cudaSuccess) e = cudaMemset(c->d_stats, 0, sizeof(unsigned long long) * kStatSlots);
  if (e == cudaSuccess) e = cudaMemset(c->d_seq_ticket, 0, sizeof(uint32_t) * (size_t)max_batch);
  if (e == cudaSuccess) e = cudaMemset(c->d_ctrl, 0, sizeof(Ctrl));
  if (e == cudaSuccess) e = cudaMallocHost(&c->h_live, sizeof(int32_t));
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&c->capture_stream, cudaStreamNonBlocking);
  if (e != cudaSuccess) {
    tc_status rc = cuda_fail(e, "tc_ctx_create");
    tc_ctx_destroy(c);
    return rc;
  }
  *out = c;
  return TC_OK;
}

extern "C" void tc_ctx_destroy(tc_ctx* c) {
  if (!c) return;
  DeviceGuard dg(c->device);
  cudaDeviceSynchronize();
  for (tc_graph* g : c->cache) destroy_graph(g);
  for (tc_graph* g : c->owned) destroy_graph(g);
  {
    std::lock_guard<std::mutex> lk(g_const_mu);
    for (DevGrammar* g : c->grammars)
      if (g_const_owner[c->device] == g) g_const_owner[c->device] = nullptr;
  }
  for (DevGrammar* g : c->grammars) {
    g->release();
    delete g;
  }
  free_gemm_scratch(c);
  cudaFree(c->d_part);
  cudaFree(c->d_seq_ticket);
  cudaFree(c->d_ctrl);
  cudaFree(c->d_stats);
  cudaFree(c->d_smp_lg);
  cudaFree(c->d_smp_tok);
  cudaFree(c->d_smp_edge);
  if (c->h_live) cudaFreeHost(c->h_live);
  if (c->capture_stream) cudaStreamDestroy(c->capture_stream);
  delete c;
}

extern "C" tc_status tc_bind_grammar(tc_ctx* c, const tc_trie* t, int32_t residency, void* stream) {
  if (!c || !t) return TC_ERR_INVALID_ARG;
  const bool force_counts = (residency & TC_BIND_LIVE_COUNTS) != 0;
  residency &= ~TC_BIND_LIVE_COUNTS;
  if (force_counts && t->char_level) {
    set_error_message("tc_bind_grammar: a character-level grammar has no live-count arrays");
    return TC_ERR_UNSUPPORTED;
  }
  if (residency != TC_RES_AUTO && residency != TC_RES_CONST && residency != TC_RES_GLOBAL) return TC_ERR_INVALID_ARG;
  if (t->vocab > c->V) {
    set_error_message("tc_bind_grammar: the trie's vocabulary is larger than the context's");
    return TC_ERR_TOKEN_RANGE;
  }
  if (t->max_fanout > c->cand_cap) {
    set_error_message("tc_bind_grammar: max fan-out " + std::to_string(t->max_fanout) +
                      " exceeds the candidate buffer " + std::to_string(c->cand_cap));
    return TC_ERR_CAPACITY;
  }
  const WalkLayout L = walk_layout(t->n_nodes(), t->n_edges());
  const size_t img_bytes = (size_t)L.words * 4;
  const size_t hdr_bytes = (size_t)L.header_words * 4;  // the part constant residency places in __constant__
  int32_t res = residency;
  if (res == TC_RES_AUTO) res = hdr_bytes <= TC_CONST_CAPACITY_BYTES ? TC_RES_CONST : TC_RES_GLOBAL;
  if (res == TC_RES_CONST && hdr_bytes > TC_CONST_CAPACITY_BYTES) {
    set_error_message("tc_bind_grammar: walk image header of " + std::to_string(hdr_bytes) +
                      " bytes exceeds constant capacity");
    return TC_ERR_CONST_CAPACITY;
  }
  DeviceGuard dg(c->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DevGrammar* g = nullptr;
  for (DevGrammar* x : c->grammars)
    if (x->hash == t->content_hash && x->residency == res && x->n_nodes == t->n_nodes() &&
        x->n_edges == t->n_edges() && x->force_counts == force_counts)
      g = x;
  if (!g) {
    g = new DevGrammar();
    g->hash = t->content_hash;
    g->residency = res;
    g->n_nodes = t->n_nodes();
    g->n_edges = t->n_edges();
    g->n_strings = t->n_strings;
    g->max_fanout = t->max_fanout;
    g->max_depth = t->max_depth;
    g->layout = L;
    g->kw = (t->n_strings + 31) / 32;
    g->force_counts = force_counts;
    g->no_counts = t->char_level;
    g->root_beg = t->node_begin[0];
    g->root_end = t->node_begin[1];
    g->root_pid = t->node_ptr[0] >= 0 ? t->ptr_rank[t->node_ptr[0]] : -1;
    const std::vector<int32_t> img = build_walk_image(*t, L);
    // On the device a pointer is named by its depth-first rank: its edge path
    // is stored at its rank.
    std::vector<int32_t> path_off((size_t)t->n_strings + 1, 0), path;
    {
      std::vector<int32_t> by_rank((size_t)t->n_strings);
      for (int32_t q = 0; q < t->n_strings; ++q) by_rank[(size_t)t->ptr_rank[q]] = q;
      path.reserve(t->path.size());
      for (int32_t r = 0; r < t->n_strings; ++r) {
        const int32_t q = by_rank[(size_t)r];
        path_off[(size_t)r] = (int32_t)path.size();
        path.insert(path.end(), t->path.begin() + t->path_off[q], t->path.begin() + t->path_off[q + 1]);
      }
      path_off[(size_t)t->n_strings] = (int32_t)path.size();
    }
    // The root step's columns: the root's token edges in CSR order (ascending
    // tokens).  At the first step of a decode each is legal for every
    // sequence: the root is not a terminal (empty strings are refused) and a
    // token edge has a pointer below it.
    std::vector<int32_t> root_img;
    {
      const int32_t rb = t->node_begin[0], re = t->node_begin[1];
      bool ok = re > rb;
      for (int32_t e = rb; ok && e < re; ++e) ok = t->edge_child[e] >= 0 && t->static_cnt[e] > 0;
      if (ok) {
        const int32_t R = re - rb, cols = gemm_tile_cols(), tiles = (R + cols - 1) / cols;
        const int32_t toff = (2 * R + 3) / 4 * 4;
        root_img.assign((size_t)toff + 8 * (size_t)tiles, 0);
        for (int32_t i = 0; i < R; ++i) {
          root_img[(size_t)i] = t->edge_tok[rb + i];
          root_img[(size_t)R + i] = rb + i;
        }
        for (int32_t col = 0; col < R; ++col) {
          const int32_t j = col % cols;
          root_img[(size_t)toff + 8 * (col / cols) + (j >> 5)] |= (int32_t)(1u << (j & 31));
        }
        for (int32_t tl = 0; tl < tiles; ++tl) root_img[(size_t)toff + 8 * tl + 4] = cols * tl;  // first index
        g->n_root = R;
        g->root_tiles_off = toff;
      }
    }
    const size_t B = (size_t)c->max_batch;
    cudaError_t e = cudaMalloc(&g->d_img, img_bytes);
    if (e == cudaSuccess) e = cudaMalloc(&g->d_static_cnt, sizeof(int32_t) * std::max<size_t>(1, t->static_cnt.size()));
    if (e == cudaSuccess) e = cudaMalloc(&g->d_path_off, sizeof(int32_t) * t->path_off.size());
    if (e == cudaSuccess) e = cudaMalloc(&g->d_path, sizeof(int32_t) * std::max<size_t>(1, t->path.size()));
    if (e == cudaSuccess) e = cudaMalloc(&g->d_st, sizeof(SeqState) * B);
    if (e == cudaSuccess) e = cudaMalloc(&g->d_spent, sizeof(uint32_t) * B * g->kw);
    if (e == cudaSuccess) e = cudaMalloc(&g->d_pre, sizeof(Cand) * B * 32);
    if (e == cudaSuccess) e = cudaMemset(g->d_pre, 0, sizeof(Cand) * B * 32);
    if (e == cudaSuccess) e = cudaMemcpy(g->d_img, img.data(), img_bytes, cudaMemcpyHostToDevice);
    if (e == cudaSuccess)
      e = cudaMemcpy(g->d_static_cnt, t->static_cnt.data(), sizeof(int32_t) * t->static_cnt.size(), cudaMemcpyHostToDevice);
    if (e == cudaSuccess)
      e = cudaMemcpy(g->d_path_off, path_off.data(), sizeof(int32_t) * path_off.size(), cudaMemcpyHostToDevice);
    if (e == cudaSuccess)
      e = cudaMemcpy(g->d_path, path.data(), sizeof(int32_t) * path.size(), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemset(g->d_st, 0, sizeof(SeqState) * B);
    if (e == cudaSuccess && !root_img.empty()) e = cudaMalloc(&g->d_root, root_img.size() * sizeof(int32_t));
    if (e == cudaSuccess && !root_img.empty())
      e = cudaMemcpy(g->d_root, root_img.data(), root_img.size() * sizeof(int32_t), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
      g->release();
      delete g;
      return cuda_fail(e, "tc_bind_grammar upload");
    }
    c->grammars.push_back(g);
  }
  if (res == TC_RES_CONST) {
    std::lock_guard<std::mutex> lk(g_const_mu);
    TC_CUDA(const_upload(g->d_img, hdr_bytes, s));
    g_const_owner[c->device] = g;
  }
  g->batch = 0;
  g->k = 0;
  c->bound = g;
  return TC_OK;
}

extern "C" tc_status tc_bound_residency(const tc_ctx* c, int32_t* residency) {
  if (!c || !residency) return TC_ERR_INVALID_ARG;
  if (!c->bound) return TC_ERR_NOT_BOUND;
  *residency = c->bound->residency;
  return TC_OK;
}

extern "C" tc_status tc_reset(tc_ctx* c, int32_t batch, int32_t k, void* stream) {
  if (!c) return TC_ERR_INVALID_ARG;
  if (!c->bound) return TC_ERR_NOT_BOUND;
  if (batch < 1 || batch > c->max_batch) return TC_ERR_CAPACITY;
  if (k < 1 || k > c->bound->n_strings) return TC_ERR_K_RANGE;
  DeviceGuard dg(c->device);
  DevGrammar* g = c->bound;
  if (!use_iv(g, k)) {
    tc_status rc = ensure_counts(c, g);
    if (rc != TC_OK) return rc;
  }
  ResetParams r = reset_params(c, g, batch, k, 0);
  r.cnt = g->d_cnt;
  TC_CUDA(launch_reset(r, static_cast<cudaStream_t>(stream)));
  g->batch = batch;
  g->k = k;
  g->iv = r.iv;
  return TC_OK;
}

namespace {

tc_status step_impl(tc_ctx* c, const void* hidden, int32_t head, const tc_sampling_t* sp, const float* u,
                    int32_t* tok_out, float* logit_out, int32_t* status_out, void* stream) {
  if (!c || !hidden || !tok_out) return TC_ERR_INVALID_ARG;
  if (misaligned(hidden, 16) || misaligned(tok_out, 4) || misaligned(logit_out, 4) || misaligned(status_out, 4)) {
    set_error_message("tc_step: hidden states must be 16-byte aligned and outputs 4-byte aligned");
    return TC_ERR_INVALID_ARG;
  }
  DevGrammar* g = c->bound;
  if (!g || g->batch < 1) return TC_ERR_NOT_BOUND;
  DeviceGuard dg(c->device);
  const bool root_gemm = (head & TC_FLAG_ROOT_GEMM) != 0;
  if (root_gemm) {
    head &= ~TC_FLAG_ROOT_GEMM;
    if (head != TC_HEAD_SPARSE || sp || u) {
      set_error_message("tc_step: TC_FLAG_ROOT_GEMM with the greedy sparse head only");
      return TC_ERR_UNSUPPORTED;
    }
    if (g->n_root == 0) {
      set_error_message("TC_FLAG_ROOT_GEMM: the grammar's root has a control edge or an edge without pointers");
      return TC_ERR_UNSUPPORTED;
    }
  }
  tc_status rc = check_head(c, root_gemm ? TC_HEAD_UNION_GEMM : head, g->batch);
  if (rc != TC_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  rc = ensure_const(c, g, s);
  if (rc != TC_OK) return rc;
  StepParams p = step_params(c, g, g->batch);
  p.hidden = static_cast<const uint16_t*>(hidden);
  p.hidden_rows = g->batch;
  p.tok_out = tok_out;
  p.logit_out = logit_out;
  p.status_out = status_out;
  p.out_stride = 1;
  if (sp || u) {
    SampleArgs smp;
    rc = check_sampling(c, g, head, sp, u, &smp);
    if (rc != TC_OK) return rc;
    apply_sampling(p, smp);
    p.smp_lg = c->d_smp_lg;  // (allocated by check_sampling on first use)
    p.smp_tok = c->d_smp_tok;
    p.smp_edge = c->d_smp_edge;
  }
  if (root_gemm) TC_CUDA(launch_root(c, g, p, s));
  else TC_CUDA(launch_any_step(c, g, p, head, s, false));
  return TC_OK;
}

}  // namespace

extern "C" tc_status tc_step(tc_ctx* c, const void* hidden, int32_t head, int32_t* tok_out, float* logit_out,
                             int32_t* status_out, void* stream) {
  return step_impl(c, hidden, head, nullptr, nullptr, tok_out, logit_out, status_out, stream);
}

extern "C" tc_status tc_step_sample(tc_ctx* c, const void* hidden, int32_t head, const tc_sampling_t* sampling,
                                    const float* uniforms, int32_t* tok_out, float* logit_out, int32_t* status_out,
                                    void* stream) {
  if (!sampling || !uniforms) return TC_ERR_INVALID_ARG;
  return step_impl(c, hidden, head, sampling, uniforms, tok_out, logit_out, status_out, stream);
}

extern "C" tc_status tc_decode_graph_create(tc_ctx* c, const void* hidden, int32_t n_steps, int32_t batch,
                                            int32_t k, int32_t max_steps, int32_t head, int32_t* toks,
                                            float* logits, int32_t* lens, int32_t* status, tc_graph** out) {
  if (!out) return TC_ERR_INVALID_ARG;
  *out = nullptr;
  tc_status rc = check_decode_args(c, hidden, n_steps, batch, k, max_steps, head, toks, logits, lens, status);
  if (rc != TC_OK) return rc;
  DeviceGuard dg(c->device);
  GraphKey key{c->bound, hidden, n_steps, batch, k, max_steps, head, toks, logits, lens, status, SampleArgs{}};
  tc_graph* gr = nullptr;
  rc = build_graph(c, c->bound, key, &gr);
  if (rc != TC_OK) return rc;
  c->owned.push_back(gr);
  *out = gr;
  return TC_OK;
}

extern "C" tc_status tc_graph_launch(tc_graph* gr, void* stream) {
  if (!gr) return TC_ERR_INVALID_ARG;
  DeviceGuard dg(gr->ctx->device);
  return launch_graph(gr, static_cast<cudaStream_t>(stream));
}

extern "C" void tc_graph_destroy(tc_graph* gr) {
  if (!gr) return;
  tc_ctx* c = gr->ctx;
  DeviceGuard dg(c->device);
  auto it = std::find(c->owned.begin(), c->owned.end(), gr);
  if (it != c->owned.end()) c->owned.erase(it);
  destroy_graph(gr);
}

namespace {

tc_status decode_impl(tc_ctx* c, const void* hidden, int32_t n_steps, int32_t batch, int32_t k, int32_t max_steps,
                      int32_t head, const tc_sampling_t* sp, const float* u, int32_t* toks, float* logits,
                      int32_t* lens, int32_t* status, void* stream) {
  tc_status rc = check_decode_args(c, hidden, n_steps, batch, k, max_steps, head, toks, logits, lens, status);
  if (rc != TC_OK) return rc;
  DeviceGuard dg(c->device);
  SampleArgs smp;
  if (sp || u) {
    rc = check_sampling(c, c->bound, head, sp, u, &smp);
    if (rc != TC_OK) return rc;
  }
  GraphKey key{c->bound, hidden, n_steps, batch, k, max_steps, head, toks, logits, lens, status, smp};
  tc_graph* gr = nullptr;
  for (size_t i = 0; i < c->cache.size(); ++i) {
    if (c->cache[i]->key == key) {
      gr = c->cache[i];
      c->cache.erase(c->cache.begin() + i);
      c->cache.push_back(gr);
      break;
    }
  }
  if (!gr) {
    rc = build_graph(c, c->bound, key, &gr);
    if (rc != TC_OK) return rc;
    gr->cached = true;
    if (c->cache.size() >= kGraphCacheSize) {
      // The evicted graph may still be running on some stream: finish first.
      cudaDeviceSynchronize();
      destroy_graph(c->cache.front());
      c->cache.erase(c->cache.begin());
    }
    c->cache.push_back(gr);
  }
  return launch_graph(gr, static_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" tc_status tc_decode(tc_ctx* c, const void* hidden, int32_t n_steps, int32_t batch, int32_t k,
                               int32_t max_steps, int32_t head, int32_t* toks, float* logits, int32_t* lens,
                               int32_t* status, void* stream) {
  return decode_impl(c, hidden, n_steps, batch, k, max_steps, head, nullptr, nullptr, toks, logits, lens, status,
                     stream);
}

extern "C" tc_status tc_decode_sample(tc_ctx* c, const void* hidden, int32_t n_steps, int32_t batch, int32_t k,
                                      int32_t max_steps, int32_t head, const tc_sampling_t* sampling,
                                      const float* uniforms, int32_t* toks, float* logits, int32_t* lens,
                                      int32_t* status, void* stream) {
  if (!sampling || !uniforms) return TC_ERR_INVALID_ARG;
  return decode_impl(c, hidden, n_steps, batch, k, max_steps, head, sampling, uniforms, toks, logits, lens, status,
                     stream);
}

extern "C" tc_status tc_decode_host(tc_ctx* c, const void* hidden, int32_t n_steps, int32_t batch, int32_t k,
                                    int32_t max_steps, int32_t head, int32_t* toks, float* logits, int32_t* lens,
                                    int32_t* status, void* stream) {
  tc_status rc = check_decode_args(c, hidden, n_steps, batch, k, max_steps, head, toks, logits, lens, status);
  if (rc != TC_OK) return rc;
  if (head & TC_FLAG_JUMP_FORWARD) {
    // Host-form steps read every sequence's hidden state of one step: lockstep only.
    set_error_message("tc_decode_host: TC_FLAG_JUMP_FORWARD needs the device-resident decode (tc_decode)");
    return TC_ERR_UNSUPPORTED;
  }
  DeviceGuard dg(c->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DevGrammar* g = c->bound;
  rc = ensure_const(c, g, s);
  if (rc != TC_OK) return rc;
  if (!use_iv(g, k)) {
    rc = ensure_counts(c, g);
    if (rc != TC_OK) return rc;
  }
  ResetParams r = reset_params(c, g, batch, k, max_steps);
  r.toks = toks;
  r.logits = logits;
  r.lens_out = lens;
  r.status_out = status;
  TC_CUDA(launch_reset(r, s));
  g->batch = batch;
  g->k = k;
  g->iv = r.iv;
  const size_t row = (size_t)batch * (size_t)c->H;
  const bool root_gemm = (head & TC_FLAG_ROOT_GEMM) != 0;
  head &= ~TC_FLAG_ROOT_GEMM;
  for (int32_t t = 0; t < max_steps; ++t) {
    StepParams p = step_params(c, g, batch);
    p.hidden = static_cast<const uint16_t*>(hidden) + (size_t)t * row;
    p.hidden_rows = batch;
    p.tok_out = toks + t;
    p.logit_out = logits + t;
    p.status_out = status;
    p.lens_out = lens;
    p.out_stride = max_steps;
    p.max_steps = max_steps;
    if (root_gemm && t == 0) TC_CUDA(launch_root(c, g, p, s));
    else TC_CUDA(launch_any_step(c, g, p, head, s, false));
    TC_CUDA(cudaMemcpyAsync(c->h_live, &c->d_ctrl->live, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
    TC_CUDA(cudaStreamSynchronize(s));
    if (*c->h_live <= 0) break;
  }
  StepParams p = step_params(c, g, batch);
  p.status_out = status;
  p.lens_out = lens;
  TC_CUDA(launch_finalize(p, s));
  TC_CUDA(cudaStreamSynchronize(s));
  return TC_OK;
}

extern "C" tc_status tc_read_seq_state(tc_ctx* c, void* stream, int32_t* node, int32_t* emitted, int32_t* len,
                                       int32_t* status, int32_t* done) {
  if (!c) return TC_ERR_INVALID_ARG;
  DevGrammar* g = c->bound;
  if (!g || g->batch < 1) return TC_ERR_NOT_BOUND;
  DeviceGuard dg(c->device);
  TC_CUDA(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
  std::vector<SeqState> h((size_t)g->batch);
  TC_CUDA(cudaMemcpy(h.data(), g->d_st, sizeof(SeqState) * h.size(), cudaMemcpyDeviceToHost));
  for (int32_t b = 0; b < g->batch; ++b) {
    if (node) node[b] = h[b].node;
    if (emitted) emitted[b] = h[b].emitted;
    if (len) len[b] = h[b].len;
    if (status) status[b] = h[b].status;
    if (done) done[b] = h[b].done;
  }
  return TC_OK;
}

extern "C" tc_status tc_first_error(tc_ctx* c, void* stream, int32_t* seq, int32_t* code) {
  if (!c || !seq || !code) return TC_ERR_INVALID_ARG;
  DevGrammar* g = c->bound;
  if (!g || g->batch < 1) return TC_ERR_NOT_BOUND;
  std::vector<int32_t> st((size_t)g->batch);
  tc_status rc = tc_read_seq_state(c, stream, nullptr, nullptr, nullptr, st.data(), nullptr);
  if (rc != TC_OK) return rc;
  *seq = -1;
  *code = TC_OK;
  for (int32_t b = 0; b < g->batch; ++b) {
    if (st[b] != TC_OK) {
      *seq = b;
      *code = st[b];
      break;
    }
  }
  return TC_OK;
}

extern "C" tc_status tc_gemm_wait_test(tc_ctx* c, int32_t withhold, int64_t wait_polls) {
  if (!c || wait_polls < 0) return TC_ERR_INVALID_ARG;
  DeviceGuard dg(c->device);
  tc_status rc = ensure_gemm_scratch(c);
  if (rc != TC_OK) return rc;
  // Captured graphs hold the kernels' parameters as they were: drop them.
  TC_CUDA(cudaDeviceSynchronize());
  for (tc_graph* g : c->cache) destroy_graph(g);
  c->cache.clear();
  c->hs.withhold = withhold ? 1 : 0;
  c->hs.wait_limit = wait_polls;
  return TC_OK;
}

extern "C" tc_status tc_read_stats(tc_ctx* c, void* stream, int64_t* out, int32_t reset) {
  if (!c || !out) return TC_ERR_INVALID_ARG;
  DeviceGuard dg(c->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  static_assert(kStatSlots == TC_STAT_SLOTS, "counter slots of the C ABI");
  unsigned long long h[kStatSlots];
  TC_CUDA(cudaMemcpyAsync(h, c->d_stats, sizeof(h), cudaMemcpyDeviceToHost, s));
  TC_CUDA(cudaStreamSynchronize(s));
  for (int i = 0; i < kStatSlots; ++i) out[i] = (int64_t)h[i];
  if (reset) {
    TC_CUDA(cudaMemsetAsync(c->d_stats, 0, sizeof(h), s));
    TC_CUDA(cudaStreamSynchronize(s));
  }
  return TC_OK;
}
