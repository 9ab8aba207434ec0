// Decode-step kernels for sm_103a: reset, sparse step, dense step, finalize.
//
// One launch performs one whole step for every sequence of the batch
// ("Constraint made cheaper than no constraint", section "Masked sampling
// inside the sampler": read the current node's edge range, filter the edges,
// take the argmax over the survivors with a fixed tree and the lower-id
// tie-break, advance; section "The sparse output layer": one tied-embedding
// dot product per legal candidate over a fixed grid).
//
// Two step kernels serve the sparse head.  For grammars whose nodes have at
// most 32 edges, sparse_step1_kernel gives each sequence one CTA: the
// candidates come from a list the previous step computed, each warp gathers a
// candidate's embedding row and meanwhile computes that candidate's child
// legal set, and the winner's set becomes the next step's list.  Otherwise
// sparse_step_kernel gives each sequence up to `tiles` CTAs (one wave); a
// sequence at a narrow node (a precomputed list, or at most 32 edges) is
// served by its first CTA with the same one-CTA body, and at a wide node
// every CTA the node needs filters the node's edges itself (a few hundred bytes of
// cached reads), so no second launch publishes the candidate list; candidate
// rank r belongs to CTA r % active; each CTA leaves its best (logit, token) in
// a fixed slot and the last to arrive (atomic ticket after a fence, no
// waiting) folds the slots in slot order and applies the transition.  Rows
// are gathered with 16-byte loads and each dot product is reduced by a fixed
// shuffle tree.

// Device form (the graph loop body): sequence b at its own step t = len_b
// reads hidden[t, b] and writes toks[b, t]; a live sequence's length equals
// the loop iteration, so no shared step counter is read.  The launch flagged
// loop_ctrl (the last step of a loop body) also sets the conditional node's
// value: directly when the grid is one CTA, else from the live count after a
// grid-wide ticket.
//
// Determinism: a logit is a function of (row, x) only - lane l accumulates
// elements 8*(32*i + l) .. +7 for i = 0, 1, ... in order with fp32 FMAs, then
// a butterfly xor tree over the 32 lanes - so the sparse and the dense head
// produce bit-identical logits, and the winner under (logit desc, token asc),
// a strict total order on distinct tokens, does not depend on fold order.
#include <cuda_runtime.h>
#include <stdint.h>

#include <climits>

#include "gemm_tc.h"
#include "kernels.h"
#include "tcd.h"

namespace tcd {

__constant__ int32_t c_walk[TC_CONST_CAPACITY_BYTES / 4];

// Sampling over one sequence's candidates by a whole CTA (defined below).
__device__ __noinline__ int block_sample(const StepParams& p, const float* lg, const int32_t* tk, int n, float u,
                                         unsigned char* smem, int& nan);

namespace {

constexpr unsigned kFull = 0xffffffffu;

// Candidate slots per CTA of the multi-CTA sparse step with T CTAs per
// sequence: a node using A <= T of them gives each at most
// max(ceil(C / T), kWarps) candidates (A is ceil(fan-out / kWarps) unless T caps it).
__host__ __device__ __forceinline__ int sparse_local_cap(int cand_cap, int T) {
  const int c = (cand_cap + T - 1) / T;
  return c > kWarps ? c : kWarps;
}
constexpr int gemm_tile_cols_dev = 128;  // columns per GEMM tile (gemm_tc.cu)

template <bool kConst>
struct WalkRd {
  const int32_t* img;
  int32_t off_edges, off_ptr;
  __device__ __forceinline__ int32_t begin(int32_t n) const {
    if constexpr (kConst) return c_walk[n];
    else return __ldg(img + n);
  }
  // Edge record, first half: {token, child, first rank below, ranks below}
  // (control edges: the terminal's own rank, 1).  Lanes read different edges,
  // which the constant cache would serialise, so edge records always come
  // through the read-only data cache (measured faster than constant-bank words
  // at B = 1); node ranges and pointer ranks, read alike by a whole warp, come
  // from the constant bank when the grammar is resident there.
  __device__ __forceinline__ int4 edge(int32_t e) const {
    return __ldg(reinterpret_cast<const int4*>(img + off_edges) + 2 * e);
  }
  // Second half: the child's header {edge begin, edge end, pointer rank, 0}.
  __device__ __forceinline__ int4 child_hdr(int32_t e) const {
    return __ldg(reinterpret_cast<const int4*>(img + off_edges) + 2 * e + 1);
  }
  __device__ __forceinline__ int32_t ptr(int32_t n) const {
    if constexpr (kConst) return c_walk[off_ptr + n];
    else return __ldg(img + off_ptr + n);
  }
};


// acc += e0*x0 + e1*x1 for the two bf16 values packed in each word (low half
// first), one FMA at a time: the mixed-precision FMA takes the bf16 operands
// as they are (their fp32 values are exact) and rounds once in fp32, the same
// result as an fp32 FMA of the widened values, without the widening
// instructions.
__device__ __forceinline__ float fma_bf2(uint32_t e, uint32_t x, float acc) {
  asm("{\n .reg .b16 el, eh, xl, xh;\n mov.b32 {el, eh}, %1;\n mov.b32 {xl, xh}, %2;\n"
      " fma.rn.f32.bf16 %0, el, xl, %0;\n fma.rn.f32.bf16 %0, eh, xh, %0;\n}"
      : "+f"(acc)
      : "r"(e), "r"(x));
  return acc;
}

// acc += e[0]*x[0] + ... + e[7]*x[7], one FMA at a time in element order.
__device__ __forceinline__ float dot8(const uint4 e, const uint4 x, float acc) {
  acc = fma_bf2(e.x, x.x, acc);
  acc = fma_bf2(e.y, x.y, acc);
  acc = fma_bf2(e.z, x.z, acc);
  acc = fma_bf2(e.w, x.w, acc);
  return acc;
}

__device__ __forceinline__ float warp_sum(float v) {
  v += __shfl_xor_sync(kFull, v, 16);
  v += __shfl_xor_sync(kFull, v, 8);
  v += __shfl_xor_sync(kFull, v, 4);
  v += __shfl_xor_sync(kFull, v, 2);
  v += __shfl_xor_sync(kFull, v, 1);
  return v;
}

__device__ __forceinline__ uint4 ld_row(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Ask L2 to fetch `bytes` (a multiple of 16) at a 16-byte aligned address; no
// completion to wait for, nothing lands in shared memory.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// x fragment of one lane: chunks 32*i + lane (8 bf16 each).
template <int NCH>
struct XFrag {
  uint4 v[NCH > 0 ? NCH : 1];
  __device__ __forceinline__ void load(const uint16_t* x, int lane) {
    const uint4* x4 = reinterpret_cast<const uint4*>(x);
#pragma unroll
    for (int i = 0; i < NCH; ++i) v[i] = __ldg(x4 + i * 32 + lane);
  }
};

// Row dot products with the fixed lane map.  NCH > 0: H == 256 * NCH and x in
// registers.  NCH == 0: any H % 8 == 0, x staged in shared memory.
template <int NCH>
__device__ __forceinline__ float row_dot(const uint16_t* row, const XFrag<NCH>& xf,
                                         const uint4* xs, int nch, int lane) {
  const uint4* r4 = reinterpret_cast<const uint4*>(row);
  float acc = 0.f;
  if constexpr (NCH > 0) {
    uint4 e[NCH];
#pragma unroll
    for (int i = 0; i < NCH; ++i) e[i] = ld_row(r4 + i * 32 + lane);
#pragma unroll
    for (int i = 0; i < NCH; ++i) acc = dot8(e[i], xf.v[i], acc);
  } else {
    for (int c = lane; c < nch; c += 32) acc = dot8(ld_row(r4 + c), xs[c], acc);
  }
  return warp_sum(acc);
}

// row_dot with x staged in shared memory but the row's NCH chunks all in
// flight at once (the same lane map and order: bit-identical to row_dot).
template <int NCH>
__device__ __forceinline__ float row_dot_xs(const uint16_t* row, const uint4* xs, int lane) {
  const uint4* r4 = reinterpret_cast<const uint4*>(row);
  uint4 e[NCH];
#pragma unroll
  for (int i = 0; i < NCH; ++i) e[i] = ld_row(r4 + i * 32 + lane);
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < NCH; ++i) acc = dot8(e[i], xs[i * 32 + lane], acc);
  return warp_sum(acc);
}

// Two rows at once (more loads in flight); each result is bit-identical to row_dot.
template <int NCH>
__device__ __forceinline__ void row_dot2(const uint16_t* ra, const uint16_t* rb, const XFrag<NCH>& xf,
                                         const uint4* xs, int nch, int lane, float& oa, float& ob) {
  const uint4* a4 = reinterpret_cast<const uint4*>(ra);
  const uint4* b4 = reinterpret_cast<const uint4*>(rb);
  float aa = 0.f, ab = 0.f;
  if constexpr (NCH > 0) {
    uint4 ea[NCH], eb[NCH];
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
      ea[i] = ld_row(a4 + i * 32 + lane);
      eb[i] = ld_row(b4 + i * 32 + lane);
    }
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
      aa = dot8(ea[i], xf.v[i], aa);
      ab = dot8(eb[i], xf.v[i], ab);
    }
  } else {
    for (int c = lane; c < nch; c += 32) {
      const uint4 ea = ld_row(a4 + c), eb = ld_row(b4 + c);
      aa = dot8(ea, xs[c], aa);
      ab = dot8(eb, xs[c], ab);
    }
  }
  oa = warp_sum(aa);
  ob = warp_sum(ab);
}

// (l, t) beats (bl, bt): larger logit, or equal logit and lower token id.
// A NaN logit never beats anything.
__device__ __forceinline__ bool better(float l, int32_t t, float bl, int32_t bt) {
  return l > bl || (l == bl && t < bt);
}

// Shared state of one CTA of a step kernel.
struct StepShared {
  int32_t scan[kWarps];
  float wl[kWarps];
  int32_t wt[kWarps], we[kWarps];
  int32_t ncand, err, last, glast;
  float bl;
  int32_t bt, be, done_after;
};

// The no-repeat state of one sequence as the legality tests read it.
//
// Count mode ("Masked sampling inside the sampler"): every edge carries the
// number of live pointers below it, a per-sequence copy decremented along a
// pointer's path when it completes, and each pointer a spent flag.
// Read-only mode ("The batched engine": a small per-sequence banned set
// against read-only per-edge pointer sets): pointers are numbered in
// depth-first order, so the pointers below an edge are one rank range held in
// the shared edge record; an edge is live while that range holds a rank not in
// the sequence's banned set (the ranks of its completed pointers, at most
// kBanMax, kept in its state).  Both give the same count of live pointers.
struct SeqLive {
  const int32_t* cnt;      // count mode: this sequence's counts; null in read-only mode
  const uint32_t* spent;   // count mode: this sequence's spent flags
  uint32_t ban[kBanMax / 2];
  int32_t nban;
};

// kRO: the read-only mode is known at compile time (no count arrays to read).
template <bool kRO = false>
__device__ __forceinline__ SeqLive seq_live(const StepParams& p, const SeqState& s, int b) {
  SeqLive L;
  L.cnt = (kRO || p.iv) ? nullptr : p.cnt + (size_t)b * p.g.n_edges;
  L.spent = p.spent + (size_t)b * p.kw;
  L.ban[0] = s.ban0;
  L.ban[1] = s.ban1;
  L.ban[2] = s.ban2;
  L.ban[3] = s.ban3;
  L.nban = s.emitted;
  return L;
}

// Banned ranks r with lo <= r < lo + n.
__device__ __forceinline__ int banned_in(const SeqLive& L, int lo, int n) {
  int c = 0;
#pragma unroll
  for (int j = 0; j < kBanMax; ++j) {
    const int r = (int)((L.ban[j >> 1] >> ((j & 1) * 16)) & 0xffffu);
    c += (j < L.nban && (unsigned)(r - lo) < (unsigned)n) ? 1 : 0;
  }
  return c;
}

// Pointer `pid` (a rank) not yet completed by this sequence.
__device__ __forceinline__ bool ptr_free(const StepParams& p, const SeqLive& L, int pid) {
  if (pid < 0 || pid >= p.g.n_strings) return false;
  if (!L.cnt) return banned_in(L, pid, 1) == 0;
  return ((L.spent[pid >> 5] >> (pid & 31)) & 1u) == 0;
}

// Live pointers below token edge e with record ed.
__device__ __forceinline__ int32_t edge_live(const SeqLive& L, int e, const int4& ed, int32_t c) {
  return L.cnt ? c : ed.w - banned_in(L, ed.z, ed.w);
}

// Legality of one edge of the current node (see the filter below); `live`
// receives the live count of a token edge.
// edge_rec_legal takes the edge's record (first half) already read.
__device__ __forceinline__ bool edge_rec_legal(const StepParams& p, const SeqLive& L, int e, bool sep_ok,
                                               bool stop_ok, const int4& ed, int32_t c, int32_t& live, int& bad) {
  live = 0;
  if (ed.x < 0 || ed.x >= p.V) {
    bad = 1;
    return false;
  }
  if (ed.y >= 0) {
    if (ed.y >= p.g.n_nodes) {
      bad = 1;
      return false;
    }
    live = edge_live(L, e, ed, c);
    return live > 0;
  }
  if (ed.y == -1) return sep_ok;
  if (ed.y == -2) return stop_ok;
  bad = 1;
  return false;
}

template <bool kConst>
__device__ __forceinline__ bool edge_legal(const StepParams& p, const WalkRd<kConst>& w, const SeqLive& L,
                                           int e, bool sep_ok, bool stop_ok, int4& ed, int32_t& live, int& bad) {
  ed = w.edge(e);
  const int32_t c = L.cnt ? L.cnt[e] : 0;  // count mode: issued together with the edge record
  return edge_rec_legal(p, L, e, sep_ok, stop_ok, ed, c, live, bad);
}

// A completed pointer leaves the live sets: count mode decrements the counts
// along its path (threads t0, t0 + stride, ...) and sets its spent flag
// (thread t0 == 0); read-only mode records its rank in ns.ban (every caller,
// identically).  ns.emitted is not changed here.
__device__ __forceinline__ void ban_add(SeqState& ns, int pid) {
  const int j = ns.emitted;
  const uint32_t v = (uint32_t)pid << ((j & 1) * 16);
  switch (j >> 1) {
    case 0: ns.ban0 |= v; break;
    case 1: ns.ban1 |= v; break;
    case 2: ns.ban2 |= v; break;
    default: ns.ban3 |= v; break;
  }
}

__device__ __forceinline__ void decrement_path(const StepParams& p, int b, int pid, int t0, int stride) {
  const int32_t q0 = __ldg(p.g.path_off + pid), q1 = __ldg(p.g.path_off + pid + 1);
  int32_t* cnt = p.cnt + (size_t)b * p.g.n_edges;
  for (int32_t q = q0 + t0; q < q1; q += stride) {
    const int32_t e = __ldg(p.g.path + q);
    if (e >= 0 && e < p.g.n_edges) cnt[e] -= 1;
  }
}

__device__ __forceinline__ void complete_pointer(const StepParams& p, int b, int pid, SeqState& ns, int t0,
                                                 int stride) {
  if (p.iv) {
    ban_add(ns, pid);
    return;
  }
  decrement_path(p, b, pid, t0, stride);
  if (t0 == 0) p.spent[(size_t)b * p.kw + (pid >> 5)] |= 1u << (pid & 31);
}

// Edge filter ("Masked sampling inside the sampler"): a token edge is legal
// while a live pointer lies below it; the separator while the terminal's
// pointer is unspent and another pointer is still owed after it; stop while
// it is unspent and it is the last one owed.  The legal candidate of rank r
// (edge order = ascending token order) is stored at s_tok/s_edge[r / T] when
// r % T == t.  Results in sh.ncand / sh.err, visible after the final barrier.
template <bool kConst>
__device__ __forceinline__ void filter_node(const StepParams& p, const WalkRd<kConst>& w, const SeqState& s, int b, int T,
                            int t, int32_t* s_tok, int32_t* s_edge, StepShared& sh) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = s.node;
  const bool n_ok = n >= 0 && n < p.g.n_nodes;
  const int nn = n_ok ? n : 0;
  // Node range and pointer id are independent loads; the spent word and the
  // edge records below are issued before any of them is consumed.
  const int beg = w.begin(nn), end = w.begin(nn + 1), pid = w.ptr(nn);
  const bool ok = n_ok && beg >= 0 && end >= beg && end <= p.g.n_edges && end - beg <= p.cand_cap;
  if (!ok) {
    if (tid == 0) {
      sh.ncand = 0;
      sh.err = 1;
    }
    __syncthreads();
    return;
  }
  int bad = pid >= p.g.n_strings;
  const SeqLive L = seq_live(p, s, b);
  const bool ctl_ok = pid >= 0 && !bad && ptr_free(p, L, pid);
  const bool sep_ok = ctl_ok && (s.emitted + 1 < s.k);
  const bool stop_ok = ctl_ok && (s.emitted + 1 == s.k);
  int32_t live;
  if (end - beg <= 32) {
    // One warp filters a small node; the others wait at the barrier.
    if (warp == 0) {
      const int e = beg + lane;
      int4 ed = make_int4(0, 0, 0, 0);
      const bool legal = e < end && edge_legal<kConst>(p, w, L, e, sep_ok, stop_ok, ed, live, bad);
      const unsigned bal = __ballot_sync(kFull, legal);
      if (legal) {
        const int rank = __popc(bal & ((1u << lane) - 1u));
        if (rank % T == t) {
          s_tok[rank / T] = ed.x;
          s_edge[rank / T] = e;
        }
      }
      const unsigned any_bad = __ballot_sync(kFull, bad);
      if (lane == 0) {
        sh.ncand = __popc(bal);
        sh.err = any_bad != 0u;
      }
    }
    __syncthreads();
    return;
  }
  int running = 0;
  for (int base = beg; base < end; base += kThreads) {
    const int e = base + tid;
    int4 ed = make_int4(0, 0, 0, 0);
    const bool legal = e < end && edge_legal<kConst>(p, w, L, e, sep_ok, stop_ok, ed, live, bad);
    const unsigned bal = __ballot_sync(kFull, legal);
    if (lane == 0) sh.scan[warp] = __popc(bal);
    __syncthreads();
    int woff = 0, tot = 0;
#pragma unroll
    for (int i = 0; i < kWarps; ++i) {
      const int c = sh.scan[i];
      woff += (i < warp) ? c : 0;
      tot += c;
    }
    if (legal) {
      const int rank = running + woff + __popc(bal & ((1u << lane) - 1u));
      if (rank % T == t) {
        s_tok[rank / T] = ed.x;
        s_edge[rank / T] = e;
      }
    }
    running += tot;
    __syncthreads();
  }
  const int any_bad = __syncthreads_or(bad);
  if (tid == 0) {
    sh.ncand = running;
    sh.err = any_bad;
  }
  __syncthreads();
}

// ---------------------------------------------------------------- legal sets of one node, one warp

constexpr int kPreMax = 32;  // largest legal set kept as a precomputed candidate list

// Legal candidates of node `node` into out[] (one warp, node fan-out <= 32).
// Returns the count, or -1 when an index is out of range or the fan-out is larger.
template <bool kConst, bool kRO = false>
__device__ __forceinline__ int warp_legal_set(const StepParams& p, const WalkRd<kConst>& w, const SeqState& s,
                                              int b, int beg, int end, int pid, int lane, Cand* out) {
  if (beg < 0 || end < beg || end > p.g.n_edges || end - beg > kPreMax) return -1;
  int bad = pid >= p.g.n_strings;
  const SeqLive L = seq_live<kRO>(p, s, b);
  const bool ctl_ok = pid >= 0 && !bad && ptr_free(p, L, pid);
  const bool sep_ok = ctl_ok && (s.emitted + 1 < s.k);
  const bool stop_ok = ctl_ok && (s.emitted + 1 == s.k);
  const int e = beg + lane;
  int4 ed = make_int4(0, 0, 0, 0);
  const int4 hd = e < end ? w.child_hdr(e) : make_int4(0, 0, -1, 0);  // issued with the first half
  int32_t c = 0;
  const bool legal = e < end && edge_legal<kConst>(p, w, L, e, sep_ok, stop_ok, ed, c, bad);
  const unsigned bal = __ballot_sync(kFull, legal);
  if (legal) out[__popc(bal & ((1u << lane) - 1u))] = Cand{make_int4(ed.x, e, ed.y, c), hd};
  if (__ballot_sync(kFull, bad)) return -1;
  return __popc(bal);
}

// warp_legal_set with this lane's edge record and child header (edge beg +
// lane, when below end) already read; the read-only no-repeat state only (no
// count array to read).
__device__ __forceinline__ int warp_legal_set_rec(const StepParams& p, const SeqState& s, int b, int beg, int end,
                                                  int pid, int lane, const int4& ed, const int4& hd, Cand* out) {
  if (beg < 0 || end < beg || end > p.g.n_edges || end - beg > kPreMax) return -1;
  int bad = pid >= p.g.n_strings;
  const SeqLive L = seq_live<true>(p, s, b);
  const bool ctl_ok = pid >= 0 && !bad && ptr_free(p, L, pid);
  const bool sep_ok = ctl_ok && (s.emitted + 1 < s.k);
  const bool stop_ok = ctl_ok && (s.emitted + 1 == s.k);
  const int e = beg + lane;
  int32_t c = 0;
  const bool legal = e < end && edge_rec_legal(p, L, e, sep_ok, stop_ok, ed, 0, c, bad);
  const unsigned bal = __ballot_sync(kFull, legal);
  if (legal) out[__popc(bal & ((1u << lane) - 1u))] = Cand{make_int4(ed.x, e, ed.y, c), hd};
  if (__ballot_sync(kFull, bad)) return -1;
  return __popc(bal);
}

// Size of the legal set of node [beg, end), capped at 2, and its first legal
// candidate (live count 0) with its child's header (one warp, any fan-out).
// -1 when an index is out of range.
template <bool kConst>
__device__ __forceinline__ int warp_count_legal(const StepParams& p, const WalkRd<kConst>& w, const SeqState& s,
                                                int b, int beg, int end, int pid, int lane, Cand& first) {
  if (beg < 0 || end < beg || end > p.g.n_edges) return -1;
  int bad = pid >= p.g.n_strings;
  const SeqLive L = seq_live(p, s, b);
  const bool ctl_ok = pid >= 0 && !bad && ptr_free(p, L, pid);
  const bool sep_ok = ctl_ok && (s.emitted + 1 < s.k);
  const bool stop_ok = ctl_ok && (s.emitted + 1 == s.k);
  int count = 0;
  for (int base = beg; base < end && count < 2; base += 32) {
    const int e = base + lane;
    int4 ed = make_int4(0, 0, 0, 0);
    int32_t live;
    const bool legal = e < end && edge_legal<kConst>(p, w, L, e, sep_ok, stop_ok, ed, live, bad);
    const unsigned bal = __ballot_sync(kFull, legal);
    if (__ballot_sync(kFull, bad)) return -1;
    if (bal != 0u && count == 0) {
      const int src = __ffs(bal) - 1;
      const int fe = base + src;
      first = Cand{make_int4(__shfl_sync(kFull, ed.x, src), fe, __shfl_sync(kFull, ed.y, src), 0), w.child_hdr(fe)};
    }
    count += __popc(bal);
  }
  return count < 2 ? count : 2;
}

// Forced continuations ("Understanding Inference for Systems Engineers",
// section 7.5, forced spans): while the grammar admits exactly one token at
// the sequence's node, that token is emitted without reading the head - its
// logit slot holds NaN - and the walk advances, pointer completions included.
// Run by one whole warp after the step's own transition; `ns` is the state
// after that transition, the same in every lane on entry and on return, and
// `hdr` its node's header {edge begin, edge end, pointer rank} (carried from
// edge records, so the chain reads no node headers).  With `list` (grammars
// whose nodes have at most kPreMax edges) the legal set that ends the chain is
// left in list[0, list_n) with its node's pointer rank in list_pid (list_n =
// -1 when the chain ended for another reason); `known` says that list[0]
// already holds the node's only legal candidate.
__device__ __forceinline__ int4 root_hdr(const StepParams& p) {
  return make_int4(p.g.root_beg, p.g.root_end, p.g.root_pid, 0);
}

template <bool kConst>
__device__ __forceinline__ void forced_chain(const StepParams& p, const WalkRd<kConst>& w, int b, SeqState& ns,
                                             int lane, int4 hdr, Cand* list, bool known, int& list_n,
                                             int& list_pid) {
  list_n = -1;
  list_pid = -2;
  unsigned long long forced = 0;
  while (!ns.done && ns.len < p.max_steps && ns.len < p.out_stride) {
    if (!known && !p.forced_logits && hdr.y - hdr.x == 1) {
      // A run of nodes with one edge each.  Nodes are numbered depth-first, so
      // such a run's edge records are consecutive: lane j reads the record that
      // is the run's j-th edge if the run gets that far, and the run is the
      // leading lanes whose edge is a live token edge and whose predecessor's
      // child has exactly that one edge.  One round trip for up to 32 tokens.
      const int e = hdr.x + lane;
      const int room = min(p.max_steps, p.out_stride) - ns.len;
      const SeqLive L = seq_live(p, ns, b);
      bool live = false, link = false;
      int4 ed = make_int4(-1, -1, 0, 0), hd = make_int4(0, 0, -1, 0);
      if (lane < room && e < p.g.n_edges) {
        ed = w.edge(e);
        hd = w.child_hdr(e);
        const int32_t c = L.cnt ? L.cnt[e] : 0;
        live = ed.x >= 0 && ed.x < p.V && ed.y >= 0 && ed.y < p.g.n_nodes && edge_live(L, e, ed, c) > 0;
        link = hd.x == e + 1 && hd.y == e + 2;
      }
      const unsigned run = __ballot_sync(kFull, live) & ((__ballot_sync(kFull, link) << 1) | 1u);
      const int m = run == kFull ? 32 : __ffs(~run) - 1;
      if (m > 0) {
        if (lane < m) {
          p.tok_out[(size_t)b * p.out_stride + ns.len + lane] = ed.x;
          p.logit_out[(size_t)b * p.out_stride + ns.len + lane] = __int_as_float(0x7fc00000);
        }
        ns.len += m;
        forced += (unsigned long long)m;
        ns.node = __shfl_sync(kFull, ed.y, m - 1);
        hdr = make_int4(__shfl_sync(kFull, hd.x, m - 1), __shfl_sync(kFull, hd.y, m - 1),
                        __shfl_sync(kFull, hd.z, m - 1), 0);
        continue;
      }
    }
    int count;
    const int pid = hdr.z;
    Cand only{make_int4(0, -1, 0, 0), make_int4(0, 0, -1, 0)};
    if (known) {
      count = 1;
      only = list[0];
      known = false;
    } else if (list && hdr.y - hdr.x <= kPreMax) {
      count = warp_legal_set<kConst>(p, w, ns, b, hdr.x, hdr.y, pid, lane, list);
      __syncwarp();
      if (count == 1) only = list[0];
    } else {
      // (a node wider than a list: counted, and no list is left for it)
      count = warp_count_legal<kConst>(p, w, ns, b, hdr.x, hdr.y, pid, lane, only);
    }
    if (count != 1) {  // (-1: an index out of range, which the next step reports)
      if (list && hdr.y - hdr.x <= kPreMax) {
        list_n = count;
        list_pid = pid;
      }
      break;
    }
    float v = __int_as_float(0x7fc00000);  // no head read: NaN
    if (p.forced_logits) {
      // Requested anyway: the forced token's own row against this position's
      // hidden state, with the head's lane map (the same value bit for bit).
      const uint4* r4 = reinterpret_cast<const uint4*>(p.emb + (size_t)only.a.x * p.H);
      const uint4* x4 = reinterpret_cast<const uint4*>(p.hidden + ((size_t)ns.len * p.B + b) * p.H);
      float acc = 0.f;
      for (int c = lane; c < (p.H >> 3); c += 32) acc = dot8(ld_row(r4 + c), __ldg(x4 + c), acc);
      v = warp_sum(acc);
    }
    if (lane == 0) {
      p.tok_out[(size_t)b * p.out_stride + ns.len] = only.a.x;
      p.logit_out[(size_t)b * p.out_stride + ns.len] = v;
    }
    ns.len += 1;
    ++forced;
    if (only.a.z >= 0) {
      ns.node = only.a.z;
      hdr = only.h;
    } else {
      // A control edge is legal only at a terminal whose pointer is unspent.
      complete_pointer(p, b, pid, ns, lane, 32);
      ns.emitted += 1;
      ns.node = 0;
      hdr = root_hdr(p);
      if (only.a.z == -2) ns.done = 1;
      __syncwarp();  // decrements and the spent flag are seen by the next legal set
    }
  }
  if (forced && lane == 0 && p.stats) atomicAdd(&p.stats[kStatForced], forced);
}

// Apply the transition of sequence b with winner (best_l, best_t, best_e).
// Called by every thread of the sequence's last CTA; thread 0 returns the
// sequence's done flag afterwards.
template <bool kConst>
__device__ __forceinline__ int finish_sequence(const StepParams& p, const WalkRd<kConst>& w, const SeqState& s, int b,
                               float best_l, int32_t best_t, int32_t best_e, int32_t ncand, int32_t err) {
  const int tid = threadIdx.x;
  int status = TC_OK;
  int32_t new_node = s.node, ptr_done = -1;
  bool stop = false;
  int4 chain_hdr = make_int4(0, 0, -1, 0);  // header of the node after the transition (jump only)
  if (err) {
    // (a wait that gave up reports its own code; any other error flag is an index out of range)
    status = err == TC_ERR_DEVICE_TIMEOUT ? TC_ERR_DEVICE_TIMEOUT : TC_ERR_BOUNDS;
  } else if (ncand == 0) {
    status = TC_ERR_EMPTY_MASK;
  } else if (best_t == INT_MAX || best_e < 0 || best_e >= p.g.n_edges || !(best_l == best_l)) {
    status = TC_ERR_BOUNDS;  // no comparable logit (NaN) or a corrupted slot
  } else {
    const SeqLive L = seq_live(p, s, b);
    const int4 ed = w.edge(best_e);
    if (p.jump) chain_hdr = ed.y == -1 ? root_hdr(p) : w.child_hdr(best_e);
    if (ed.x != best_t) {
      status = TC_ERR_BOUNDS;
    } else if (ed.y >= 0) {
      if (edge_live(L, best_e, ed, L.cnt ? L.cnt[best_e] : 0) <= 0) status = TC_ERR_NO_LIVE_EDGE;
      else new_node = ed.y;
    } else {
      const int32_t pid = w.ptr(s.node);
      if (!ptr_free(p, L, pid)) {
        status = TC_ERR_NO_LIVE_EDGE;
      } else {
        ptr_done = pid;
        stop = (ed.y == -2);
        new_node = 0;
      }
    }
  }
  __syncthreads();  // every thread has decided before the state changes
  // The completed pointer is no longer live below any edge of its path.
  if (ptr_done >= 0 && !p.iv) decrement_path(p, b, ptr_done, tid, kThreads);
  // Forced continuations follow a decision that leaves the sequence live.
  const bool chain = p.jump && status == TC_OK && !stop;
  if (chain) __syncthreads();  // the decrements above are seen by the chain's legal sets
  int done = 0;
  if (tid < 32) {
    const int lane = tid;
    SeqState ns = s;
    // This path keeps no candidate list for the next node: a sparse step
    // after it filters that node itself (whatever head or kernel runs next).
    ns.pre_n = 0;
    ns.pre_pid = -2;
    if (status != TC_OK) {
      ns.status = status;
      ns.done = 1;
    } else {
      ns.node = new_node;
      ns.len = s.len + 1;
      if (ptr_done >= 0) {
        if (p.iv) ban_add(ns, ptr_done);
        else if (lane == 0) p.spent[(size_t)b * p.kw + (ptr_done >> 5)] |= 1u << (ptr_done & 31);
        ns.emitted = s.emitted + 1;
      }
      if (stop) ns.done = 1;
    }
    if (lane == 0) {
      if (p.stats) {
        atomicAdd(&p.stats[kStatSeqSteps], 1ull);
        atomicAdd(&p.stats[kStatCandRows], (unsigned long long)ncand);
      }
      if (p.device_form) {
        if (status == TC_OK && s.len < p.out_stride) {
          p.tok_out[(size_t)b * p.out_stride + s.len] = best_t;
          p.logit_out[(size_t)b * p.out_stride + s.len] = best_l;
        }
      } else {
        p.tok_out[(size_t)b * p.out_stride] = status == TC_OK ? best_t : -1;
        if (p.logit_out) p.logit_out[(size_t)b * p.out_stride] = status == TC_OK ? best_l : 0.f;
      }
    }
    if (chain) {
      __syncwarp();  // the spent flag set above
      int ln, lp;
      forced_chain<kConst>(p, w, b, ns, lane, chain_hdr, nullptr, false, ln, lp);
    }
    if (lane == 0) {
      p.st[b] = ns;
      if (p.status_out) p.status_out[b] = ns.status;
      if (p.lens_out) p.lens_out[b] = ns.len;
      if (ns.done) atomicSub(&p.ctrl->live, 1);
      done = ns.done;
    }
  }
  return done;
}

// A live sequence whose length reached the budget stops here (CTA t == 0, thread 0).
__device__ __forceinline__ void stop_out_of_steps(const StepParams& p, const SeqState& s, int b) {
  SeqState ns = s;
  ns.status = TC_ERR_MAX_STEPS;
  ns.done = 1;
  p.st[b] = ns;
  if (!p.device_form) {
    p.tok_out[(size_t)b * p.out_stride] = -1;
    if (p.logit_out) p.logit_out[(size_t)b * p.out_stride] = 0.f;
  }
  if (p.status_out) p.status_out[b] = ns.status;
  if (p.lens_out) p.lens_out[b] = ns.len;
  atomicSub(&p.ctrl->live, 1);
}

// Byte offset of the multi-CTA step's sampling buffers in its dynamic shared
// memory: after the staged hidden state (generic sizes) and the candidate lists.
__host__ __device__ __forceinline__ size_t sample_smem_offset(const StepParams& p, int tiles) {
  const bool staged = !(p.H == 256 || p.H == 2048 || p.H == 4096);
  const size_t x = staged ? (size_t)(p.H >> 3) * 16 : 0;
  const size_t lists = 3 * (size_t)sparse_local_cap(p.cand_cap, tiles) * sizeof(int32_t);
  return (x + lists + 127) & ~(size_t)127;
}

// Fold the per-warp bests, combine the CTAs of sequence b, let the last CTA
// apply the transition; then, in a loop-control launch, set the loop condition.
// In a loop-control launch (the last step of a graph loop body), set the
// loop condition: every CTA takes a ticket and the last one reads the live
// count; a grid of one CTA decides from its own sequence (`done_after`, read
// by thread 0).  All threads of every CTA call it.
__device__ __forceinline__ void loop_control(const StepParams& p, const int& done_after) {
  if (!p.loop_ctrl) return;
  if (gridDim.x * gridDim.y == 1) {
    if (threadIdx.x == 0) cudaGraphSetConditional((cudaGraphConditionalHandle)p.cond, done_after ? 0u : 1u);
    return;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const uint32_t total = gridDim.x * gridDim.y;
    const uint32_t g = atomicAdd(&p.ctrl->ticket, 1u);
    if (g == total - 1) {
      __threadfence();
      const int32_t live = atomicAdd(&p.ctrl->live, 0);
      p.ctrl->ticket = 0u;
      cudaGraphSetConditional((cudaGraphConditionalHandle)p.cond, live > 0 ? 1u : 0u);
    }
  }
}

template <bool kConst, bool kSmp = false>
__device__ __forceinline__ void step_tail(const StepParams& p, const WalkRd<kConst>& w, const SeqState& s, int b, int mode,
                          float wl, int32_t wt, int32_t we, StepShared& sh, int active) {
  // mode: 0 = idle (stopped or failed before this step), 1 = active, 2 = out of steps now.
  // active: the sequence's CTAs taking part in this step (blockIdx.x < active).
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tiles = active, t = blockIdx.x;
  if (p.stats && tid == 0 && blockIdx.x == 0 && blockIdx.y == 0) atomicAdd(&p.stats[kStatStepLaunches], 1ull);
  if (tid == 0) sh.done_after = 1;
  if (mode == 1 && t >= tiles) {
    // not needed for this node: nothing to fold
  } else if (mode == 1) {
    if (lane == 0) {
      sh.wl[warp] = wl;
      sh.wt[warp] = wt;
      sh.we[warp] = we;
    }
    __syncthreads();
    if (tid == 0) {
      float bl = -INFINITY;
      int32_t bt = INT_MAX, be = -1;
      for (int i = 0; i < kWarps; ++i)
        if (better(sh.wl[i], sh.wt[i], bl, bt)) { bl = sh.wl[i]; bt = sh.wt[i]; be = sh.we[i]; }
      int last = 1;
      if (tiles > 1) {
        // Each CTA's best and its error flag (a CTA whose bounded wait ran out
        // fails the sequence's step, whichever CTA arrives last).
        Partial* slot = p.part + (size_t)b * gridDim.x;
        slot[t] = Partial{bl, bt, be, sh.err};
        __threadfence();
        const uint32_t ticket = atomicAdd(&p.seq_ticket[b], 1u);
        last = (ticket == (uint32_t)tiles - 1);
        if (last) {
          __threadfence();
          bl = -INFINITY;
          bt = INT_MAX;
          be = -1;
          for (int i = 0; i < tiles; ++i) {
            const float l = __ldcg(&slot[i].logit);
            const int32_t tk = __ldcg(&slot[i].tok);
            const int32_t ee = __ldcg(&slot[i].edge);
            if (__ldcg(&slot[i].err) == TC_ERR_DEVICE_TIMEOUT) sh.err = TC_ERR_DEVICE_TIMEOUT;
            if (better(l, tk, bl, bt)) { bl = l; bt = tk; be = ee; }
          }
          p.seq_ticket[b] = 0;
        }
      }
      sh.bl = bl;
      sh.bt = bt;
      sh.be = be;
      sh.last = last;
    }
    __syncthreads();
    if (sh.last) {
      if (kSmp && !sh.err && sh.ncand > 0) {
        // Sampling: the draw replaces the fold's argmax (all candidates' logits
        // were left in the sequence's scratch rows by their CTAs).
        extern __shared__ __align__(128) unsigned char smem_raw[];
        const size_t row = (size_t)b * p.cand_cap;
        const float u = p.device_form ? p.u[(size_t)b * p.out_stride + s.len] : p.u[b];
        int nan = 0;
        const int slot = block_sample(p, p.smp_lg + row, p.smp_tok + row, sh.ncand, u,
                                      smem_raw + sample_smem_offset(p, gridDim.x), nan);
        if (tid == 0) {
          if (slot >= 0) {
            sh.bl = __ldcg(p.smp_lg + row + slot);
            sh.bt = __ldcg(p.smp_tok + row + slot);
            sh.be = __ldcg(p.smp_edge + row + slot);
          } else {
            sh.bl = -INFINITY;
            sh.bt = INT_MAX;
            sh.be = -1;
          }
        }
        __syncthreads();
      }
      const int d = finish_sequence<kConst>(p, w, s, b, sh.bl, sh.bt, sh.be, sh.ncand, sh.err);
      if (tid == 0) sh.done_after = d;
    }
  } else if (t == 0 && tid == 0) {
    if (mode == 2) {
      stop_out_of_steps(p, s, b);
    } else if (!p.device_form) {
      // A stopped or failed sequence reports an idle token.
      p.tok_out[(size_t)b * p.out_stride] = -1;
      if (p.logit_out) p.logit_out[(size_t)b * p.out_stride] = 0.f;
      if (p.status_out) p.status_out[b] = s.status;
      if (p.lens_out) p.lens_out[b] = s.len;
    }
  }

  loop_control(p, sh.done_after);
}

// 0: idle, 1: active, 2: live but out of steps.
__device__ __forceinline__ int seq_mode(const StepParams& p, const SeqState& s) {
  if (s.done) return 0;
  return s.len >= p.max_steps ? 2 : 1;
}

__device__ __forceinline__ const uint16_t* hidden_row(const StepParams& p, const SeqState& s, int b) {
  size_t row = (size_t)b;
  if (p.device_form) row += (size_t)s.len * (size_t)p.B;
  return p.hidden + row * (size_t)p.H;
}

}  // namespace

// Sparse head: one dot product per legal candidate.
// Programmatic dependent launch: a step launched as the programmatic
// dependent of the previous step may be scheduled while that one runs; it
// waits here until the previous grid has completed and its writes are
// visible.  Without a programmatic dependency both instructions are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_enter() {
  pdl_wait();
  pdl_trigger();
}

// Device form: the live count left by the launch before the previous one is
// final when this launch starts (the previous launch let this one start only
// after its own dependency wait returned), so it may be read before this
// launch's wait.  Zero means every sequence has stopped: the launch then does
// nothing but count itself and steer the loop, without reading any state
// (a stale non-zero value takes the normal path, which finds the same).
__device__ __forceinline__ bool idle_launch(const StepParams& p) {
  if (!p.device_form || __ldcg(&p.ctrl->live) != 0) return false;
  pdl_enter();
  if (p.stats && threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) atomicAdd(&p.stats[kStatStepLaunches], 1ull);
  const int done_after = 1;
  loop_control(p, done_after);
  return true;
}

// kSmp: sampling instead of the argmax (a separate instantiation, so the greedy
// kernel carries none of it).
// ---------------------------------------------------------------- one-CTA sparse step
//
// For grammars whose nodes have at most 32 edges each sequence is served by
// one CTA, and the step also prepares the next one.  When the winner is a
// token edge the next node is its child, and the child's legal set depends
// only on state this step does not change (live counts change only when a
// pointer completes, the spent flags and the pointer count likewise), so each
// warp computes its candidate's child legal set while that candidate's
// embedding row is in flight.  The winner's set is stored as the sequence's
// precomputed candidate list; the next step reads it together with the
// sequence state instead of filtering the node (the mask is computed ahead of
// time, as "GLRMask" computes it in parallel with the forward pass).  After a
// separator or a stop, or when a set does not fit, the next step filters.
struct Step1Shared {
  Cand cand[kPreMax];                 // this step's candidates
  Cand spec[kPreMax][kPreMax];        // per candidate: its child's legal candidates
  int32_t spec_n[kPreMax];            // their number, -1 when not available
  float lg[kPreMax];                  // candidate logits (sampling)
  float smp_w[kPreMax];               // sampling weights and kept flags, per candidate
  int32_t smp_k[kPreMax];
  float wl[kWarps];
  int32_t wt[kWarps], wslot[kWarps];
  int32_t ncand, err, pid, done_after, smp_slot, smp_nan;
};

// Sampling over one sequence's candidates ("Understanding Inference for
// Systems Engineers", section 3.8): softmax of logit / temperature, restricted
// first to the top-k highest logits - a value threshold, so tied logits are
// all kept - then by removing the ascending prefix, in (logit, token) order,
// whose probability mass is at most 1 - top-p (the largest is never removed,
// so among equal probabilities the highest id survives); the token is the
// first kept candidate in ascending token order whose cumulative weight
// exceeds u times the kept total.  One warp, n <= 32 candidates in ascending
// token order, lane i holding candidate i; every sum runs in a fixed order.
// Returns the chosen slot, or -1 with nan = 1 when a logit is NaN.
__device__ __forceinline__ int warp_sample(const StepParams& p, const float* lg, const Cand* cand, int n, float u,
                                           int lane, float* wsh, int* ksh, int& nan) {
  const bool act = lane < n;
  const float l = act ? lg[lane] : 0.f;
  const int32_t tok = act ? cand[lane].a.x : INT_MAX;
  nan = __any_sync(kFull, act && !(l == l)) ? 1 : 0;
  if (nan) return -1;
  int kept = act ? 1 : 0;
  if (p.top_k > 0 && p.top_k < n) {
    int greater = 0;
    for (int j = 0; j < n; ++j) greater += lg[j] > l ? 1 : 0;  // shared-memory broadcast reads
    kept = (act && greater < p.top_k) ? 1 : 0;
  }
  float m = kept ? l : -INFINITY;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
  float wgt = kept ? expf((l - m) * p.inv_temp) : 0.f;
  if (p.top_p < 1.f) {
    wsh[lane] = wgt;
    ksh[lane] = kept;
    __syncwarp();
    float total = 0.f, run = 0.f;
    int larger = 0;
    for (int j = 0; j < n; ++j) {  // candidates in token order, a fixed summation order
      const float lj = lg[j], wj = wsh[j];
      const int32_t tj = cand[j].a.x;
      const int kj = ksh[j];
      total += wj;
      if (kj && (lj < l || (lj == l && tj <= tok))) run += wj;
      if (kj && (lj > l || (lj == l && tj > tok))) larger = 1;
    }
    if (kept && larger && run <= (1.f - p.top_p) * total) kept = 0;
    if (!kept) wgt = 0.f;
  }
  float pre = wgt;  // inclusive prefix in lane (ascending token) order
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float v = __shfl_up_sync(kFull, pre, o);
    if (lane >= o) pre += v;
  }
  const float target = u * __shfl_sync(kFull, pre, 31);
  const unsigned hit = __ballot_sync(kFull, kept && pre > target);
  const unsigned any = __ballot_sync(kFull, kept);
  if (hit) return __ffs(hit) - 1;
  return any ? 31 - __clz(any) : -1;
}

// Inclusive prefix sums of v[0, n) in place, in a fixed order for any n:
// thread t sums its contiguous chunk sequentially, warp 0 scans the 256 chunk
// totals (8 per lane, then a shuffle scan), and each chunk adds its offset.
// tot: 256 floats of scratch.  All threads of the CTA call it.
__device__ __forceinline__ void block_scan_inclusive(float* v, int n, float* tot) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int c = (n + kThreads - 1) / kThreads;
  const int i0 = tid * c, i1 = min(n, i0 + c);
  float run = 0.f;
  for (int i = i0; i < i1; ++i) {
    run += v[i];
    v[i] = run;
  }
  tot[tid] = run;
  __syncthreads();
  if (tid < 32) {
    float mine[kThreads / 32];
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < kThreads / 32; ++j) {
      mine[j] = tot[lane * (kThreads / 32) + j];
      s += mine[j];
    }
    float pre = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float x = __shfl_up_sync(kFull, pre, o);
      if (lane >= o) pre += x;
    }
    float off = pre - s;  // exclusive offset of this lane's first chunk
#pragma unroll
    for (int j = 0; j < kThreads / 32; ++j) {
      tot[lane * (kThreads / 32) + j] = off;
      off += mine[j];
    }
  }
  __syncthreads();
  const float off = tot[tid];
  for (int i = i0; i < i1; ++i) v[i] += off;
  __syncthreads();
}

// (Not inlined: a call kept out of line leaves the greedy path's register
// allocation as it was.)
// Sampling over n <= kMaxCandCap candidates by one CTA, with warp_sample's
// rules ("Understanding Inference for Systems Engineers", section 3.8):
// candidates come in ascending token order (lg, tk: logits and tokens in
// global memory).  The (logit, token) keys are sorted ascending by a bitonic
// network; the top-k threshold is the logit k places from the top; weights
// exp((logit - max) / temperature) are prefix-summed in that order and the
// prefix with mass <= 1 - top_p is removed (never the last); the kept weights
// are then prefix-summed in token order and the draw is the first candidate
// whose sum exceeds u times the total.  Every sum has a fixed order.
// Returns the chosen candidate index (all threads), or -1 with nan = 1.
__device__ __noinline__ int block_sample(const StepParams& p, const float* lg, const int32_t* tk, int n, float u,
                                         unsigned char* smem, int& nan) {
  const int tid = threadIdx.x;
  int npad = 1;
  while (npad < n) npad <<= 1;
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(smem);
  float* wsort = reinterpret_cast<float*>(smem + (size_t)kMaxCandCap * 8);
  float* wtok = wsort + kMaxCandCap;
  float* tot = wtok + kMaxCandCap;
  int* pick = reinterpret_cast<int*>(tot + kThreads);
  int bad = 0;
  for (int i = tid; i < npad; i += kThreads) {
    unsigned long long key = ~0ull;
    if (i < n) {
      float l = __ldcg(lg + i);
      if (!(l == l)) bad = 1;
      if (l == 0.f) l = 0.f;  // -0 ties with +0
      uint32_t bits = __float_as_uint(l);
      bits = (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);  // ascending float order
      key = ((unsigned long long)bits << 32) | (uint32_t)__ldcg(tk + i);
    }
    keys[i] = key;
  }
  nan = __syncthreads_or(bad);
  if (nan) return -1;
  for (int k = 2; k <= npad; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < npad; i += kThreads) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const unsigned long long a = keys[i], c = keys[ixj];
          if ((a > c) == ((i & k) == 0)) {
            keys[i] = c;
            keys[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  auto logit_of = [&](unsigned long long key) {
    uint32_t bits = (uint32_t)(key >> 32);
    bits = (bits & 0x80000000u) ? (bits & 0x7fffffffu) : ~bits;
    return __uint_as_float(bits);
  };
  const float m = logit_of(keys[n - 1]);
  const float tau = (p.top_k > 0 && p.top_k < n) ? logit_of(keys[n - p.top_k]) : -INFINITY;
  for (int i = tid; i < n; i += kThreads) {
    const float l = logit_of(keys[i]);
    wsort[i] = l >= tau ? expf((l - m) * p.inv_temp) : 0.f;
  }
  __syncthreads();
  if (p.top_p < 1.f) {
    for (int i = tid; i < n; i += kThreads) wtok[i] = wsort[i];
    __syncthreads();
    block_scan_inclusive(wtok, n, tot);  // ascending (logit, token) order
    const float cut = (1.f - p.top_p) * wtok[n - 1];
    for (int i = tid; i < n - 1; i += kThreads)
      if (wsort[i] > 0.f && wtok[i] <= cut) wsort[i] = 0.f;
    __syncthreads();
  }
  // back to token order: a candidate's index is its token's rank among the candidates
  for (int i = tid; i < n; i += kThreads) {
    const int32_t t = (int32_t)(uint32_t)keys[i];
    int lo = 0, hi = n;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (__ldcg(tk + mid) < t) lo = mid + 1; else hi = mid;
    }
    wtok[lo] = wsort[i];
  }
  __syncthreads();
  for (int i = tid; i < n; i += kThreads) wsort[i] = wtok[i];  // keep the weights; scan a copy
  if (tid == 0) {
    pick[0] = INT_MAX;
    pick[1] = -1;
  }
  __syncthreads();
  block_scan_inclusive(wtok, n, tot);
  const float target = u * wtok[n - 1];
  for (int i = tid; i < n; i += kThreads) {
    if (wsort[i] > 0.f) {
      atomicMax(&pick[1], i);
      if (wtok[i] > target) atomicMin(&pick[0], i);
    }
  }
  __syncthreads();
  const int slot = pick[0] != INT_MAX ? pick[0] : pick[1];
  __syncthreads();
  return slot;
}

// kXs: the hidden state staged in shared memory instead of registers, so two
// CTAs fit an SM (for batches larger than the SM count: one wave, not two).
// One sequence's whole step by one CTA (fan-out of its node at most kPreMax):
// `s` is its state and `pre0` this warp's entry of its precomputed list, both
// read by the caller right after the programmatic-dependency wait; the caller
// does the launch count and the loop control.  Leaves sh.done_after for
// thread 0.
// kLean: greedy steps without forced continuations, the common case, in an
// instantiation that carries neither the sampler nor the forced-span walk
// (a smaller kernel: the step is bound by latency, instruction fetch included).
// kRO (with kLean): the read-only no-repeat state, known at compile time.
template <bool kConst, int NCH, bool kXs, bool kLean = false, bool kRO = false>
__device__ __forceinline__ void step1_body(const StepParams& p, int b, const SeqState& s, const Cand& pre0,
                                           Step1Shared& sh, unsigned char* smem_raw) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool smp = !kLean && p.smp, jump = !kLean && p.jump, iv = kRO || p.iv;
  const WalkRd<kConst> w{p.g.img, p.g.off_edges, p.g.off_ptr};
  const int mode = seq_mode(p, s);
  const int nch = p.H >> 3;
  uint4* xs = reinterpret_cast<uint4*>(smem_raw);

  float wl = -INFINITY;
  int32_t wt = INT_MAX, ws = -1;
  const bool pre = s.pre_n > 0;
  // With a precomputed list every warp knows its candidates from the state
  // alone: the first one's row loads start at once, before the hidden state is
  // read, and no barrier precedes the candidate loop.
  uint4 e[NCH > 0 ? NCH : 1];  // the row of the candidate in flight
  // Lean steps with the read-only state: the first candidate's child edge
  // records (lane i: edge i) are requested before its row, since the child
  // legal set waits on them longer than the dot product waits on the row
  // (A/B: B=1 +2 %, B=64 +4 %, B=256 +1.6 %; in the steps with forced
  // continuations it cost 3.5 %, so only this instantiation does it).
  int4 ped = make_int4(0, 0, 0, 0), phd = make_int4(0, 0, -1, 0);
  if constexpr (NCH > 0) {
    if (mode == 1 && pre && warp < s.pre_n - 1) {
      if constexpr (kRO) {
        const int e0 = pre0.h.x + lane;
        if (pre0.a.z >= 0 && pre0.h.x >= 0 && e0 < pre0.h.y && pre0.h.y <= p.g.n_edges) {
          phd = w.child_hdr(e0);
          ped = w.edge(e0);
        }
      }
      const uint4* r0 = reinterpret_cast<const uint4*>(p.emb + (size_t)pre0.a.x * p.H);
#pragma unroll
      for (int i = 0; i < NCH; ++i) e[i] = ld_row(r0 + i * 32 + lane);
    }
  }
  int n = 0, err = 0;
  if (mode == 1) {
    const uint16_t* x = hidden_row(p, s, b);
    if (p.device_form && tid == 32 && s.len + 1 < p.max_steps)
      prefetch_l2(x + (size_t)p.B * p.H, (uint32_t)p.H * 2u);  // the next step's hidden state
    XFrag<kXs ? 0 : NCH> xf;
    if constexpr (NCH > 0 && !kXs) {
      xf.load(x, lane);
    } else {
      for (int c = tid; c < nch; c += kThreads) xs[c] = __ldg(reinterpret_cast<const uint4*>(x) + c);
    }
    if (!pre) {
      // Filter the node (fan-out <= 32: one warp).
      if (warp == 0) {
        const int nd = s.node;
        const bool n_ok = nd >= 0 && nd < p.g.n_nodes;
        const int nn = n_ok ? nd : 0;
        const int beg = w.begin(nn), end = w.begin(nn + 1), pid = w.ptr(nn);
        const int cnt = n_ok ? warp_legal_set<kConst, kRO>(p, w, s, b, beg, end, pid, lane, sh.cand) : -1;
        if (lane == 0) {
          sh.ncand = cnt < 0 ? 0 : cnt;
          sh.err = cnt < 0;
          sh.pid = pid;
        }
      }
      __syncthreads();  // (pre is the same for the whole CTA)
      n = sh.ncand;
      err = sh.err;
    } else {
      n = s.pre_n - 1;
      if (tid == 0) {
        sh.ncand = n;
        sh.err = 0;
        sh.pid = s.pre_pid;
      }
      if constexpr (NCH == 0 || kXs) __syncthreads();  // x staged in shared memory by all threads
    }
    if (!err) {
      for (int l = warp; l < n; l += kWarps) {
        const Cand cd = pre ? (l == warp ? pre0 : p.pre[(size_t)b * kPreMax + l]) : sh.cand[l];
        // The row, then the child's edges: the candidate carries the child's
        // header, so no node header is read on this path.
        const bool spec = cd.a.z >= 0 && cd.a.z < p.g.n_nodes;
        const int cb = cd.h.x, ce = cd.h.y, cpid = cd.h.z;
        const uint4* r4 = reinterpret_cast<const uint4*>(p.emb + (size_t)cd.a.x * p.H);
        float acc = 0.f;
        if constexpr (NCH > 0) {
          if (!pre || l != warp) {  // (the first precomputed candidate's row is already in flight)
#pragma unroll
            for (int i = 0; i < NCH; ++i) e[i] = ld_row(r4 + i * 32 + lane);
          }
          int sn = -1;
          if (spec) {
            if constexpr (kRO) {
              sn = (pre && l == warp) ? warp_legal_set_rec(p, s, b, cb, ce, cpid, lane, ped, phd, sh.spec[l])
                                      : warp_legal_set<kConst, kRO>(p, w, s, b, cb, ce, cpid, lane, sh.spec[l]);
            } else {
              sn = warp_legal_set<kConst, kRO>(p, w, s, b, cb, ce, cpid, lane, sh.spec[l]);
            }
          }
          if (lane == 0) sh.spec_n[l] = sn;
          __syncwarp();
          if constexpr (kXs) {
#pragma unroll
            for (int i = 0; i < NCH; ++i) acc = dot8(e[i], xs[i * 32 + lane], acc);
          } else {
#pragma unroll
            for (int i = 0; i < NCH; ++i) acc = dot8(e[i], xf.v[i], acc);
          }
        } else {
          const int sn = spec ? warp_legal_set<kConst, kRO>(p, w, s, b, cb, ce, cpid, lane, sh.spec[l]) : -1;
          if (lane == 0) sh.spec_n[l] = sn;
          __syncwarp();
          for (int c = lane; c < nch; c += 32) acc = dot8(ld_row(r4 + c), xs[c], acc);
        }
        const float v = warp_sum(acc);
        if (lane == 0) {
          if (pre) sh.cand[l] = cd;  // the winner's edge data is read from here below
          if (smp) sh.lg[l] = v;
        }
        if (better(v, cd.a.x, wl, wt)) {
          wl = v;
          wt = cd.a.x;
          ws = l;
        }
      }
    }
    if (lane == 0) {
      sh.wl[warp] = wl;
      sh.wt[warp] = wt;
      sh.wslot[warp] = ws;
    }
  }
  __syncthreads();

  // The rest of the step is warp 0's: the fold, the transition, the next list.
  if (mode == 1 && warp == 0) {
    float bl = -INFINITY;
    int32_t bt = INT_MAX, bs = -1;
    if (smp) {
      int nan = 0, slot = -1;
      if (!err && n > 0) {
        const float u = p.device_form ? p.u[(size_t)b * p.out_stride + s.len] : p.u[b];
        slot = warp_sample(p, sh.lg, sh.cand, n, u, lane, sh.smp_w, sh.smp_k, nan);
      }
      bs = slot;
      if (bs >= 0) {
        bl = nan ? __int_as_float(0x7fc00000) : sh.lg[bs];
        bt = sh.cand[bs].a.x;
      }
    } else {
      // Eight warp bests, folded by a fixed butterfly over lanes 0-7 (a strict
      // total order, so every lane ends with the same winner).
      if (lane < kWarps) {
        bl = sh.wl[lane];
        bt = sh.wt[lane];
        bs = sh.wslot[lane];
      }
#pragma unroll
      for (int o = kWarps / 2; o > 0; o >>= 1) {
        const float ol = __shfl_xor_sync(kFull, bl, o);
        const int32_t ot = __shfl_xor_sync(kFull, bt, o);
        const int32_t os = __shfl_xor_sync(kFull, bs, o);
        if (better(ol, ot, bl, bt)) {
          bl = ol;
          bt = ot;
          bs = os;
        }
      }
      bl = __shfl_sync(kFull, bl, 0);
      bt = __shfl_sync(kFull, bt, 0);
      bs = __shfl_sync(kFull, bs, 0);
    }
    const int ncand = n;
    int status = TC_OK;
    int32_t new_node = s.node, ptr_done = -1;
    bool stop = false;
    Cand win{make_int4(0, -1, 0, 0), make_int4(0, 0, -1, 0)};
    if (err) {
      status = TC_ERR_BOUNDS;
    } else if (ncand == 0) {
      status = TC_ERR_EMPTY_MASK;
    } else if (bs < 0 || !(bl == bl)) {
      status = TC_ERR_BOUNDS;  // no comparable logit (NaN)
    } else {
      win = sh.cand[bs];
      if (win.a.z >= 0) {
        if (win.a.w <= 0) status = TC_ERR_NO_LIVE_EDGE;  // live count read this step
        else new_node = win.a.z;
      } else {
        const int32_t pid = pre ? s.pre_pid : sh.pid;
        if (!ptr_free(p, seq_live<kRO>(p, s, b), pid)) {
          status = TC_ERR_NO_LIVE_EDGE;
        } else {
          ptr_done = pid;
          stop = win.a.z == -2;
          new_node = 0;
        }
      }
    }
    // The winner's child legal set becomes the next step's candidate list.
    const int next_n = (status == TC_OK && ptr_done < 0) ? sh.spec_n[bs] : -1;
    // Forced continuations follow when that set is a single token, after a
    // separator (the root's set is not precomputed), or when no set was kept
    // (a child wider than a list, counted by the chain itself).
    const bool chain = jump && status == TC_OK && !stop && (next_n == 1 || next_n < 0 || ptr_done >= 0);
    if (!chain && lane < next_n) {
      // The next step's candidates: their list, and their rows started towards
      // L2 (only these rows: prefetching every candidate's child rows while
      // the rows were in flight cost time at every batch size).
      p.pre[(size_t)b * kPreMax + lane] = sh.spec[bs][lane];
      prefetch_l2(p.emb + (size_t)sh.spec[bs][lane].a.x * p.H, (uint32_t)p.H * 2u);
    }
    if (ptr_done >= 0 && !iv) decrement_path(p, b, ptr_done, lane, 32);
    SeqState ns = s;
    int pre_n = next_n, pre_pid = next_n >= 0 ? win.h.z : -2;  // the child's pointer rank
    if (status != TC_OK) {
      ns.status = status;
      ns.done = 1;
    } else {
      ns.node = new_node;
      ns.len = s.len + 1;
      if (ptr_done >= 0) {
        if (iv) ban_add(ns, ptr_done);
        else if (lane == 0) p.spent[(size_t)b * p.kw + (ptr_done >> 5)] |= 1u << (ptr_done & 31);
        ns.emitted = s.emitted + 1;
      }
      if (stop) ns.done = 1;
    }
    if (lane == 0) {
      if (p.stats) {
        atomicAdd(&p.stats[kStatSeqSteps], 1ull);
        atomicAdd(&p.stats[kStatCandRows], (unsigned long long)ncand);
      }
      if (p.device_form) {
        if (status == TC_OK && s.len < p.out_stride) {
          p.tok_out[(size_t)b * p.out_stride + s.len] = bt;
          p.logit_out[(size_t)b * p.out_stride + s.len] = bl;
        }
      } else {
        p.tok_out[(size_t)b * p.out_stride] = status == TC_OK ? bt : -1;
        if (p.logit_out) p.logit_out[(size_t)b * p.out_stride] = status == TC_OK ? bl : 0.f;
      }
    }
    if (chain) {
      __syncwarp();  // the decrements and the spent flag above are seen by the chain
      // The winner's own (precomputed) list slot serves as the chain's scratch.
      Cand* list = sh.spec[bs];
      const int4 hdr = ptr_done >= 0 ? root_hdr(p) : win.h;
      forced_chain<kConst>(p, w, b, ns, lane, hdr, list, next_n == 1, pre_n, pre_pid);
      if (pre_n > 0 && lane < pre_n) {
        p.pre[(size_t)b * kPreMax + lane] = list[lane];
        prefetch_l2(p.emb + (size_t)list[lane].a.x * p.H, (uint32_t)p.H * 2u);
      }
      if (lane == 0 && !ns.done && ns.len < p.max_steps)
        prefetch_l2(p.hidden + ((size_t)ns.len * p.B + b) * p.H, (uint32_t)p.H * 2u);
    }
    if (ns.status == TC_OK) {
      ns.pre_n = pre_n >= 0 ? pre_n + 1 : 0;
      ns.pre_pid = pre_n >= 0 ? pre_pid : -2;
    } else {
      ns.pre_n = 0;
    }
    if (lane == 0) {
      p.st[b] = ns;
      if (p.status_out) p.status_out[b] = ns.status;
      if (p.lens_out) p.lens_out[b] = ns.len;
      if (ns.done) atomicSub(&p.ctrl->live, 1);
      sh.done_after = ns.done;
    }
  } else if (mode != 1 && tid == 0) {
    if (mode == 2) {
      stop_out_of_steps(p, s, b);
    } else if (!p.device_form) {
      p.tok_out[(size_t)b * p.out_stride] = -1;
      if (p.logit_out) p.logit_out[(size_t)b * p.out_stride] = 0.f;
      if (p.status_out) p.status_out[b] = s.status;
      if (p.lens_out) p.lens_out[b] = s.len;
    }
    sh.done_after = 1;
  }
}

template <bool kConst, int NCH, bool kXs = false, bool kLean = false, bool kRO = false>
__global__ void __launch_bounds__(kThreads, kXs ? 2 : 1) sparse_step1_kernel(const StepParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __shared__ Step1Shared sh;
  if (idle_launch(p)) return;
  pdl_enter();
  const int b = blockIdx.y;
  // The state and this warp's first precomputed candidate are read together.
  const SeqState s = p.st[b];
  const Cand pre0 = p.pre[(size_t)b * kPreMax + (threadIdx.x >> 5)];
  if (p.stats && threadIdx.x == 0 && blockIdx.y == 0) atomicAdd(&p.stats[kStatStepLaunches], 1ull);
  step1_body<kConst, NCH, kXs, kLean, kRO>(p, b, s, pre0, sh, smem_raw);
  loop_control(p, sh.done_after);
}

// ---------------------------------------------------------------- multi-CTA sparse step

// kXs: the hidden state staged in shared memory instead of registers (greedy
// steps at hidden sizes of 2048 and up), so two CTAs share an SM: for batches
// whose nodes' fan-out needs more CTAs than one wave of the register variant holds.
// kLean (greedy steps without forced continuations): the narrow nodes' one-CTA
// body without the sampler or the forced-span walk.
template <bool kConst, int NCH, bool kSmp = false, bool kXs = false, bool kLean = false>
__global__ void __launch_bounds__(kThreads, kXs ? 2 : 1) sparse_step_kernel(const StepParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  // A narrow node's step uses the one-CTA step's shared state instead.
  constexpr size_t kShBytes = sizeof(Step1Shared) < sizeof(StepShared) ? sizeof(StepShared) : sizeof(Step1Shared);
  __shared__ __align__(16) unsigned char sh_raw[kShBytes];
  StepShared& sh = *reinterpret_cast<StepShared*>(sh_raw);
  if (idle_launch(p)) return;
  pdl_enter();
  const int b = blockIdx.y, t = blockIdx.x, T = gridDim.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const WalkRd<kConst> w{p.g.img, p.g.off_edges, p.g.off_ptr};
  const SeqState s = p.st[b];
  // (The first CTA's warps read their precomputed candidates with the state.)
  Cand pre0{make_int4(0, -1, 0, 0), make_int4(0, 0, -1, 0)};
  if (t == 0 && p.pre) pre0 = p.pre[(size_t)b * kPreMax + warp];
  const int mode = seq_mode(p, s);
  const int nch = p.H >> 3;
  const int local_cap = sparse_local_cap(p.cand_cap, T);
  uint4* xs = reinterpret_cast<uint4*>(smem_raw);
  int32_t* s_tok = reinterpret_cast<int32_t*>(smem_raw + (NCH == 0 || kXs ? (size_t)nch * 16 : 0));
  int32_t* s_edge = s_tok + local_cap;
  float* s_lg = reinterpret_cast<float*>(s_edge + local_cap);  // sampling only
  // A node needs one CTA per kWarps of its edges: the others leave at once
  // (deep nodes of a wide catalog have a few edges, its root hundreds).
  int A = T;
  bool narrow = false;
  if (mode == 1) {
    // A node with a precomputed list, or with at most kPreMax edges, takes the
    // one-CTA step: the list is read with the state, the next node's list is
    // computed while the rows are in flight, and the first CTA alone works
    // (drawing with the one-warp sampler when sampling).
    narrow = p.pre && s.pre_n > 0;
    const int nd = s.node;
    if (!narrow && nd >= 0 && nd < p.g.n_nodes) {
      const int fan = w.begin(nd + 1) - w.begin(nd);
      narrow = p.pre && fan <= kPreMax;
      const int need = (fan + kWarps - 1) / kWarps;
      A = need < 1 ? 1 : (need < T ? need : T);
    }
  }
  if (narrow) {
    Step1Shared& sh1 = *reinterpret_cast<Step1Shared*>(sh_raw);
    if (p.stats && tid == 0 && t == 0 && b == 0) atomicAdd(&p.stats[kStatStepLaunches], 1ull);
    if (t == 0) step1_body<kConst, NCH, kXs, kLean>(p, b, s, pre0, sh1, smem_raw);
    loop_control(p, sh1.done_after);
    return;
  }

  float wl = -INFINITY;
  int32_t wt = INT_MAX, we = -1;
  if (mode == 1 && t < A) {
    const uint16_t* x = hidden_row(p, s, b);
    XFrag<kXs ? 0 : NCH> xf;
    if constexpr (NCH > 0 && !kXs) {
      xf.load(x, lane);
    } else {
      // (visible to every warp after the filter's closing barrier)
      for (int c = tid; c < nch; c += kThreads) xs[c] = __ldg(reinterpret_cast<const uint4*>(x) + c);
    }
    filter_node<kConst>(p, w, s, b, A, t, s_tok, s_edge, sh);
    if (!sh.err) {
      const int nc = sh.ncand;
      const int nlocal = nc > t ? (nc - t + A - 1) / A : 0;
      for (int l = warp; l < nlocal; l += kWarps) {
        const int32_t tok = s_tok[l];
        float v;
        if constexpr (kXs) v = row_dot_xs<NCH>(p.emb + (size_t)tok * p.H, xs, lane);
        else v = row_dot<NCH>(p.emb + (size_t)tok * p.H, xf, xs, nch, lane);
        if (better(v, tok, wl, wt)) { wl = v; wt = tok; we = s_edge[l]; }
        if (kSmp && lane == 0) s_lg[l] = v;
      }
      if constexpr (kSmp) {
        // Every candidate's logit, token and edge go to the sequence's scratch
        // rows by candidate rank, for its last CTA (kept out of the loop above).
        __syncthreads();
        for (int i = tid; i < nlocal; i += kThreads) {
          const size_t r = (size_t)b * p.cand_cap + (size_t)i * A + t;
          p.smp_lg[r] = s_lg[i];
          p.smp_tok[r] = s_tok[i];
          p.smp_edge[r] = s_edge[i];
        }
        __threadfence();
      }
    }
  }
  step_tail<kConst, kSmp>(p, w, s, b, mode, wl, wt, we, sh, A);
}

// Dense head: every vocabulary row, then the legal mask, then the argmax.
//
// Each CTA owns a contiguous block of rows and streams it through shared
// memory in stages of up to 8 rows with bulk asynchronous copies (one copy per
// stage, completion counted on the stage's mbarrier), so DRAM sees long
// sequential reads and the bytes in flight do not depend on registers.  Warp w
// computes row w of a stage with the same lane map and reduction tree as the
// sparse head's row_dot, so both heads produce bit-identical logits.
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__host__ __device__ __forceinline__ void dense_rows_per_stage(int H, int& R, int& S) {
  R = (64 * 1024) / (2 * H);
  R = R > kWarps ? kWarps : (R < 1 ? 1 : R);
  S = (128 * 1024) / (R * 2 * H);
  S = S > 4 ? 4 : (S < 2 ? 2 : S);
}

__device__ __forceinline__ bool stage_wait(uint32_t bar, uint32_t parity) {
  for (int i = 0; i < (1 << 20); ++i) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    if (ok) return true;
  }
  return false;
}

template <int NCH>
__device__ __forceinline__ float row_dot_smem(const uint4* row, const XFrag<NCH>& xf, const uint4* xs, int nch,
                                              int lane) {
  float acc = 0.f;
  if constexpr (NCH > 0) {
    uint4 e[NCH];
#pragma unroll
    for (int i = 0; i < NCH; ++i) e[i] = row[i * 32 + lane];
#pragma unroll
    for (int i = 0; i < NCH; ++i) acc = dot8(e[i], xf.v[i], acc);
  } else {
    for (int c = lane; c < nch; c += 32) acc = dot8(row[c], xs[c], acc);
  }
  return warp_sum(acc);
}

template <bool kConst, int NCH>
__global__ void __launch_bounds__(kThreads) dense_step_kernel(const StepParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __shared__ StepShared sh;
  __shared__ __align__(8) uint64_t full[4];
  pdl_wait();  // the next step may launch only near the end: its waiting CTAs would take SM slots
  const int b = blockIdx.y, g = blockIdx.x, G = gridDim.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const WalkRd<kConst> w{p.g.img, p.g.off_edges, p.g.off_ptr};
  const SeqState s = p.st[b];
  const int mode = seq_mode(p, s);
  const int nch = p.H >> 3;
  uint4* xs = reinterpret_cast<uint4*>(smem_raw);
  int32_t* s_tok = reinterpret_cast<int32_t*>(smem_raw + (NCH == 0 ? (size_t)nch * 16 : 0));
  int32_t* s_edge = s_tok + p.cand_cap;
  const size_t lists_end = (size_t)(NCH == 0 ? nch * 16 : 0) + 2 * (size_t)p.cand_cap * sizeof(int32_t);
  unsigned char* stages = smem_raw + ((lists_end + 127) & ~(size_t)127);

  float wl = -INFINITY;
  int32_t wt = INT_MAX, we = -1;
  if (mode == 1) {
    const uint16_t* x = hidden_row(p, s, b);
    XFrag<NCH> xf;
    if constexpr (NCH > 0) {
      xf.load(x, lane);
    } else {
      for (int c = tid; c < nch; c += kThreads) xs[c] = __ldg(reinterpret_cast<const uint4*>(x) + c);
    }
    filter_node<kConst>(p, w, s, b, 1, 0, s_tok, s_edge, sh);
    if (!sh.err) {
      const int n = sh.ncand;
      auto consider = [&](int32_t r, float v) {
        // legal iff r is in the ascending candidate list
        int lo = 0, hi = n;
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (s_tok[mid] < r) lo = mid + 1; else hi = mid;
        }
        if (lo < n && s_tok[lo] == r && better(v, r, wl, wt)) { wl = v; wt = r; we = s_edge[lo]; }
      };
      int R, S;
      dense_rows_per_stage(p.H, R, S);
      const size_t row_bytes = (size_t)p.H * 2;
      const int rpc = (p.V + G - 1) / G;
      const int r_begin = g * rpc;
      const int r_end = min(p.V, r_begin + rpc);
      const int n_chunks = r_end > r_begin ? (r_end - r_begin + R - 1) / R : 0;
      auto issue = [&](int c) {
        const int st = c % S;
        const int r0 = r_begin + c * R;
        const int nr = min(R, r_end - r0);
        const uint32_t bytes = (uint32_t)(nr * row_bytes);
        const uint32_t bar = smem_addr(&full[st]);
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                         smem_addr(stages + (size_t)st * R * row_bytes)),
                     "l"(p.emb + (size_t)r0 * p.H), "r"(bytes), "r"(bar)
                     : "memory");
      };
      if (tid == 0) {
        for (int i = 0; i < S; ++i) asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&full[i])) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        for (int c = 0; c < S && c < n_chunks; ++c) issue(c);
      }
      __syncthreads();
      int failed = 0;
      for (int c = 0; c < n_chunks; ++c) {
        const int st = c % S;
        const bool ok = stage_wait(smem_addr(&full[st]), (uint32_t)((c / S) & 1));
        if (__syncthreads_or(!ok)) {
          failed = 1;
          break;
        }
        const int r0 = r_begin + c * R;
        if (warp < min(R, r_end - r0)) {
          const uint4* row = reinterpret_cast<const uint4*>(stages + (size_t)st * R * row_bytes + (size_t)warp * row_bytes);
          consider(r0 + warp, row_dot_smem<NCH>(row, xf, xs, nch, lane));
        }
        __syncthreads();  // every warp is done with this stage before it is refilled
        if (tid == 0 && c + S < n_chunks) {
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          issue(c + S);
        }
      }
      if (failed) {
        // A copy never completed: wait (bounded) for the ones still in flight, then report.
        if (tid == 0) {
          for (int c = 0; c < n_chunks; ++c) stage_wait(smem_addr(&full[c % S]), (uint32_t)((c / S) & 1));
          sh.err = TC_ERR_DEVICE_TIMEOUT;
        }
        __syncthreads();
      }
    }
  }
  pdl_trigger();
  step_tail<kConst>(p, w, s, b, mode, wl, wt, we, sh, gridDim.x);
}

__global__ void __launch_bounds__(kThreads) reset_kernel(const ResetParams r) {
  const int b = blockIdx.y, tid = threadIdx.x;
  const int E = r.g.n_edges;
  if (!r.iv) {  // count mode: a fresh copy of the live counts and no spent flags
    int32_t* cnt = r.cnt + (size_t)b * E;
    for (int e = blockIdx.x * kThreads + tid; e < E; e += gridDim.x * kThreads) cnt[e] = __ldg(r.g.static_cnt + e);
    if (blockIdx.x == 0)
      for (int i = tid; i < r.kw; i += kThreads) r.spent[(size_t)b * r.kw + i] = 0u;
  }
  if (blockIdx.x == 0) {
    if (r.toks) {
      for (int i = tid; i < r.max_steps; i += kThreads) {
        r.toks[(size_t)b * r.max_steps + i] = -1;
        r.logits[(size_t)b * r.max_steps + i] = 0.f;
      }
    }
    if (tid == 0) {
      SeqState s{};
      s.k = r.k;
      r.st[b] = s;
      r.seq_ticket[b] = 0u;
      if (r.lens_out) r.lens_out[b] = 0;
      if (r.status_out) r.status_out[b] = TC_OK;
    }
    if (b == 0 && tid == 0) {
      if (r.stats) atomicAdd(&r.stats[kStatResetLaunches], 1ull);
      if (r.gemm_err) *r.gemm_err = 0;  // a timed-out GEMM wait fails the steps up to the next reset only
      r.ctrl->live = r.B;
      r.ctrl->ticket = 0u;
      if (r.cond) cudaGraphSetConditional((cudaGraphConditionalHandle)r.cond, r.B > 0 ? 1u : 0u);
    }
  }
}

// End of a host-driven decode: sequences still live ran out of steps.
__global__ void __launch_bounds__(kThreads) finalize_kernel(const StepParams p) {
  for (int b = threadIdx.x; b < p.B; b += kThreads) {
    SeqState s = p.st[b];
    if (!s.done) {
      s.status = TC_ERR_MAX_STEPS;
      s.done = 1;
      p.st[b] = s;
    }
    if (p.status_out) p.status_out[b] = s.status;
    if (p.lens_out) p.lens_out[b] = s.len;
  }
  if (threadIdx.x == 0 && p.ctrl) p.ctrl->live = 0;
}

// ---------------------------------------------------------------- GEMM heads
//
// One step of the union head ("The sparse output layer": in batched form the
// union of legal rows across the batch is bounded by the trie) or of the dense
// GEMM head runs as: candidate filter per sequence -> (union only) compaction
// of the union bitmap into a sorted row list -> tcgen05 GEMM over those rows
// with a masked-argmax epilogue -> per-sequence fold of the column-tile
// partials and the transition.

// Grid (1, B): filter the node of sequence b into global candidate lists.
template <bool kConst>
__global__ void __launch_bounds__(kThreads) cand_filter_kernel(const StepParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __shared__ StepShared sh;
  pdl_enter();
  const int b = blockIdx.y, tid = threadIdx.x;
  const WalkRd<kConst> w{p.g.img, p.g.off_edges, p.g.off_ptr};
  const SeqState s = p.st[b];
  const int mode = seq_mode(p, s);
  int32_t* s_tok = reinterpret_cast<int32_t*>(smem_raw);
  int32_t* s_edge = s_tok + p.cand_cap;
  const HeadScratch& hs = p.hs;
  if (mode != 1) {
    if (tid == 0) {
      hs.xrow[b] = -1;
      hs.ncand[b] = 0;
      hs.errf[b] = 0;
    }
    return;
  }
  filter_node<kConst>(p, w, s, b, 1, 0, s_tok, s_edge, sh);
  const int n = sh.err ? 0 : sh.ncand;
  int32_t* ct = hs.cand_tok + (size_t)b * p.cand_cap;
  int32_t* ce = hs.cand_edge + (size_t)b * p.cand_cap;
  int32_t* cc = hs.cand_col + (size_t)b * p.cand_cap;
  for (int i = tid; i < n; i += kThreads) {
    const int32_t tok = s_tok[i];
    ct[i] = tok;
    ce[i] = s_edge[i];
    if (hs.union_mode) atomicOr(&hs.ubits[tok >> 5], 1u << (tok & 31));
    else cc[i] = tok;
  }
  if (tid == 0) {
    hs.ncand[b] = n;
    hs.errf[b] = sh.err;
    hs.xrow[b] = (int64_t)(((size_t)(p.device_form ? s.len : 0) * (size_t)p.B + (size_t)b) * (size_t)p.H);
    // Every stepping sequence is at the same step: its activation rows start at
    // len * B (identical writes from all of them).
    *hs.row0 = p.device_form ? s.len * p.B : 0;
  }
}

// One CTA of 1024 threads: union bitmap -> ascending row list, token -> index
// map, bitmap cleared for the next step.
constexpr int kCompactThreads = 1024;
__global__ void __launch_bounds__(kCompactThreads) union_compact_kernel(const StepParams p) {
  __shared__ int32_t s_warp[kCompactThreads / 32];
  pdl_enter();
  const HeadScratch& hs = p.hs;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int words = (p.V + 31) >> 5;
  const int per = (words + kCompactThreads - 1) / kCompactThreads;
  const int w0 = tid * per, w1 = min(words, w0 + per);
  int cnt = 0;
  for (int i = w0; i < w1; ++i) cnt += __popc(hs.ubits[i]);
  // block-wide exclusive scan of cnt
  int incl = cnt;
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int v = s_warp[lane];
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(kFull, v, o);
      if (lane >= o) v += u;
    }
    s_warp[lane] = v;  // inclusive per-warp totals
  }
  __syncthreads();
  int idx = (warp > 0 ? s_warp[warp - 1] : 0) + incl - cnt;
  for (int i = w0; i < w1; ++i) {
    uint32_t bits = hs.ubits[i];
    if (bits) hs.ubits[i] = 0u;
    while (bits) {
      const int bit = __ffs(bits) - 1;
      bits &= bits - 1;
      const int tok = i * 32 + bit;
      hs.ulist[idx] = tok;
      hs.umap[tok] = idx;
      ++idx;
    }
  }
  if (tid == 0) {
    *hs.n_union = s_warp[kCompactThreads / 32 - 1];
    if (p.stats) atomicAdd(&p.stats[kStatUnionRows], (unsigned long long)s_warp[kCompactThreads / 32 - 1]);
  }
}

// Grid (1, B): the GEMM column of each of sequence b's candidates, and for
// every 128-column tile of the union the record of sequence b's candidates in
// it (a bitmask of the columns and the index of the first one), so that the
// GEMM's epilogue finds them with one load instead of a search.
__global__ void __launch_bounds__(kThreads) cand_column_kernel(const StepParams p) {
  extern __shared__ __align__(16) int32_t s_col[];  // [cand_cap]
  pdl_enter();
  const HeadScratch& hs = p.hs;
  const int b = blockIdx.y;
  const int n = hs.ncand[b];
  const int32_t* ct = hs.cand_tok + (size_t)b * p.cand_cap;
  int32_t* cc = hs.cand_col + (size_t)b * p.cand_cap;
  for (int i = threadIdx.x; i < n; i += kThreads) {
    const int32_t col = hs.umap[ct[i]];
    s_col[i] = col;
    cc[i] = col;
  }
  __syncthreads();
  // Columns ascend with the candidates (both follow the token order), so the
  // candidates of tile t are the run that starts at the first column >= 128 t.
  const int n_tiles = min((*hs.n_union + gemm_tile_cols_dev - 1) / gemm_tile_cols_dev, hs.max_tiles);
  TileCands* rec = hs.tile_cands + (size_t)b * hs.max_tiles;
  for (int t = threadIdx.x; t < n_tiles; t += kThreads) {
    const int c0 = t * gemm_tile_cols_dev;
    int lo = 0, hi = n;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (s_col[mid] < c0) lo = mid + 1; else hi = mid;
    }
    uint32_t bits[4] = {0u, 0u, 0u, 0u};
    for (int i = lo; i < n; ++i) {
      const int c = s_col[i] - c0;
      if (c >= gemm_tile_cols_dev) break;
      bits[c >> 5] |= 1u << (c & 31);
    }
    int4* r = reinterpret_cast<int4*>(rec + t);
    r[0] = make_int4((int)bits[0], (int)bits[1], (int)bits[2], (int)bits[3]);
    r[1] = make_int4(lo, 0, 0, 0);
  }
}

// Grid (1, B): fold sequence b's column-tile partials, map the winning column
// back to its token and edge, and apply the transition (step_tail).
template <bool kConst>
__global__ void __launch_bounds__(kThreads) gemm_finish_kernel(const StepParams p) {
  __shared__ StepShared sh;
  pdl_enter();
  const int b = blockIdx.y, tid = threadIdx.x;
  const WalkRd<kConst> w{p.g.img, p.g.off_edges, p.g.off_ptr};
  const HeadScratch& hs = p.hs;
  // The step's scalars are read together with the state (one round trip).
  const SeqState s = p.st[b];
  const bool root = hs.root_mode != 0;
  const int n = root ? hs.n_root : hs.ncand[b];
  // A GEMM wait that timed out fails the step of every sequence.  The root
  // step's candidates hold only for a sequence that is at the root with
  // nothing emitted (the first step after a reset).
  const int err = *hs.gemm_err ? TC_ERR_DEVICE_TIMEOUT
                  : root        ? ((s.node != 0 || s.len != 0 || s.emitted != 0) ? 1 : 0)
                                : hs.errf[b];
  const int n_cols = root ? n : hs.union_mode ? *hs.n_union : p.V;
  const int32_t* c_tok = root ? hs.root_tok : hs.cand_tok + (size_t)b * p.cand_cap;
  const int32_t* c_edge = root ? hs.root_edge : hs.cand_edge + (size_t)b * p.cand_cap;
  const int mode = seq_mode(p, s);
  float wl = -INFINITY;
  int32_t wt = INT_MAX, we = -1;
  if (mode == 1) {
    const int n_tiles = (n_cols + gemm_tile_cols_dev - 1) / gemm_tile_cols_dev;
    int32_t bc = INT_MAX;  // winning column (tile partials)
    int32_t bi = INT_MAX;  // winning candidate index (split sums)
    const bool split = (hs.union_mode || root) && hs.ksplit > 1;
    if (!err && n > 0 && split) {
      // Split-K: each candidate's logit is the sum of its per-split partial
      // sums, added in split order (a fixed order, independent of the batch).
      // Candidates ascend by token, so the candidate index orders ties like the token.
      const size_t split_stride = (size_t)p.B * p.cand_cap;
      for (int i = tid; i < n; i += kThreads) {
        const float* sp = hs.split_part + (size_t)b * p.cand_cap + i;
        float v = 0.f;
        // Eight loads in flight, then added in split order.
        for (int s0 = 0; s0 < hs.ksplit; s0 += 8) {
          float x[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) x[j] = s0 + j < hs.ksplit ? __ldcg(sp + (size_t)(s0 + j) * split_stride) : 0.f;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (s0 + j < hs.ksplit) v += x[j];
        }
        if (better(v, i, wl, bi)) {
          wl = v;
          bi = i;
        }
      }
    } else if (!err && n > 0) {
      const GemmPartial* part = hs.part + (size_t)b * hs.max_tiles;
      for (int t = tid; t < n_tiles && t < hs.max_tiles; t += kThreads) {
        const GemmPartial q = part[t];
        if (q.col != INT_MAX && better(q.logit, q.col, wl, bc)) {
          wl = q.logit;
          bc = q.col;
        }
      }
    }
    // warp-wide fold: (logit, column or index) is a total order, so every lane ends with the same best
    int32_t key = split ? bi : bc;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ol = __shfl_xor_sync(kFull, wl, o);
      const int32_t ok = __shfl_xor_sync(kFull, key, o);
      if (better(ol, ok, wl, key)) {
        wl = ol;
        key = ok;
      }
    }
    if (split) {
      if (key != INT_MAX) {
        wt = c_tok[key];
        we = c_edge[key];
      }
    } else if ((bc = key) != INT_MAX) {
      // columns ascend with tokens, so the column order breaks ties like the token order
      int lo = bc;  // (root step: the column is the candidate's index)
      if (!root) {
        const int32_t* cc = hs.cand_col + (size_t)b * p.cand_cap;
        int hi = n;
        lo = 0;
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (cc[mid] < bc) lo = mid + 1; else hi = mid;
        }
        if (!(lo < n && cc[lo] == bc)) lo = -1;
      }
      if (lo >= 0 && lo < n) {
        wt = c_tok[lo];
        we = c_edge[lo];
      } else {
        wl = -INFINITY;  // cannot happen: the column came from this sequence's list
      }
    }
    if (tid == 0) {
      sh.ncand = n;
      sh.err = err;
    }
    __syncthreads();
  }
  step_tail<kConst>(p, w, s, b, mode, wl, wt, we, sh, gridDim.x);
}

// ---------------------------------------------------------------- launchers

namespace {

// Resident CTAs per SM of the multi-CTA sparse step for this hidden size and
// dynamic shared memory (registers usually allow one).
template <bool kConst>
int sparse_occupancy(int H, size_t smem, bool xs) {
  int occ = 0;
  cudaError_t e;
  switch (H) {
    case 256: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, sparse_step_kernel<kConst, 1>, kThreads, smem); break;
    case 2048:
      e = xs ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, sparse_step_kernel<kConst, 8, false, true>,
                                                             kThreads, smem)
             : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, sparse_step_kernel<kConst, 8>, kThreads, smem);
      break;
    case 4096:
      e = xs ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, sparse_step_kernel<kConst, 16, false, true>,
                                                             kThreads, smem)
             : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, sparse_step_kernel<kConst, 16>, kThreads, smem);
      break;
    default: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, sparse_step_kernel<kConst, 0>, kThreads, smem); break;
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return 1;
  }
  return occ < 1 ? 1 : occ;
}

}  // namespace

int sparse_tiles(int max_fanout, int B, int num_sms, int H, int cand_cap, bool const_resident, int* xs_out) {
  // One warp per candidate, but no more CTAs than the GPU holds at once: a
  // second wave would add a whole kernel's latency to every step.
  int by_fan = (max_fanout + kWarps - 1) / kWarps;
  const int b = B > 0 ? B : 1;
  const size_t xbytes = (H == 256 || H == 2048 || H == 4096) ? 0 : (size_t)H * 2;  // x staged for other sizes
  const size_t lists = 2 * (size_t)sparse_local_cap(cand_cap, by_fan > 0 ? by_fan : 1) * sizeof(int32_t);
  const size_t smem = xbytes + lists;
  int occ = const_resident ? sparse_occupancy<true>(H, smem, false) : sparse_occupancy<false>(H, smem, false);
  // When one wave of the register variant cannot give every sequence the
  // CTAs its widest node needs, stage x in shared memory if that fits more
  // CTAs per SM.
  int xs = 0;
  if ((H == 2048 || H == 4096) && (long long)b * by_fan > (long long)num_sms * occ) {
    const size_t smem_xs = (size_t)H * 2 + lists;
    const int occ_xs = const_resident ? sparse_occupancy<true>(H, smem_xs, true)
                                      : sparse_occupancy<false>(H, smem_xs, true);
    if (occ_xs > occ) {
      occ = occ_xs;
      xs = 1;
    }
  }
  if (xs_out) *xs_out = xs;
  int by_grid = (num_sms * occ) / b;
  if (by_grid < 1) by_grid = 1;
  int t = by_fan < by_grid ? by_fan : by_grid;
  if (t < 1) t = 1;
  if (t > kMaxTiles) t = kMaxTiles;
  return t;
}

int dense_tiles(int B, int num_sms) {
  int g = num_sms / (B > 0 ? B : 1);  // one CTA per SM: each streams 128 KB of stages
  if (g < 1) g = 1;
  if (g > kMaxTiles) g = kMaxTiles;
  return g;
}

namespace {

template <bool kConst, int NCH>
cudaError_t launch_one(const StepParams& p, int head, int tiles, bool pdl, cudaStream_t s) {
  const int nch = p.H >> 3;
  const size_t xbytes = NCH == 0 ? (size_t)nch * 16 : 0;
  const int cap = head == kHeadSparse ? sparse_local_cap(p.cand_cap, tiles) : p.cand_cap;
  size_t smem = xbytes + 2 * (size_t)cap * sizeof(int32_t);
  if (head != kHeadSparse) {
    int R, S;
    dense_rows_per_stage(p.H, R, S);
    smem = ((smem + 127) & ~(size_t)127) + (size_t)S * R * 2 * p.H;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(tiles, p.B);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (head == kHeadSparse && p.one_cta) {
    cfg.gridDim = dim3(1, p.B);
    const bool lean = !p.smp && !p.jump;  // greedy without forced continuations
    if constexpr (NCH >= 8) {
      if (p.wide) {
        cfg.dynamicSmemBytes = (size_t)nch * 16;
        if (lean && p.iv) return cudaLaunchKernelEx(&cfg, sparse_step1_kernel<kConst, NCH, true, true, true>, p);
        return lean ? cudaLaunchKernelEx(&cfg, sparse_step1_kernel<kConst, NCH, true, true>, p)
                    : cudaLaunchKernelEx(&cfg, sparse_step1_kernel<kConst, NCH, true>, p);
      }
    }
    cfg.dynamicSmemBytes = xbytes;
    if (lean && p.iv) return cudaLaunchKernelEx(&cfg, sparse_step1_kernel<kConst, NCH, false, true, true>, p);
    return lean ? cudaLaunchKernelEx(&cfg, sparse_step1_kernel<kConst, NCH, false, true>, p)
                : cudaLaunchKernelEx(&cfg, sparse_step1_kernel<kConst, NCH>, p);
  }
  if (head == kHeadSparse && p.smp) {
    cfg.dynamicSmemBytes = sample_smem_offset(p, tiles) + kSampleSmem;
    return cudaLaunchKernelEx(&cfg, sparse_step_kernel<kConst, NCH, true>, p);
  }
  const bool lean = !p.jump;  // (sampling took its own kernel above)
  if constexpr (NCH >= 8) {
    if (head == kHeadSparse && p.multi_xs) {
      cfg.dynamicSmemBytes = (size_t)nch * 16 + 2 * (size_t)cap * sizeof(int32_t);
      return lean ? cudaLaunchKernelEx(&cfg, sparse_step_kernel<kConst, NCH, false, true, true>, p)
                  : cudaLaunchKernelEx(&cfg, sparse_step_kernel<kConst, NCH, false, true>, p);
    }
  }
  if (head == kHeadSparse)
    return lean ? cudaLaunchKernelEx(&cfg, sparse_step_kernel<kConst, NCH, false, false, true>, p)
                : cudaLaunchKernelEx(&cfg, sparse_step_kernel<kConst, NCH>, p);
  return cudaLaunchKernelEx(&cfg, dense_step_kernel<kConst, NCH>, p);
}

template <bool kConst, int NCH>
cudaError_t prepare_one() {
  constexpr int kSmem = kMaxDynamicSmem;
  cudaError_t e = cudaFuncSetAttribute(sparse_step_kernel<kConst, NCH>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(sparse_step_kernel<kConst, NCH, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(sparse_step_kernel<kConst, NCH, false, false, true>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  if constexpr (NCH >= 8) {
    e = cudaFuncSetAttribute(sparse_step_kernel<kConst, NCH, false, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(sparse_step_kernel<kConst, NCH, false, true, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
  }
  return cudaFuncSetAttribute(dense_step_kernel<kConst, NCH>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
}

template <bool kConst>
cudaError_t launch_h(const StepParams& p, int head, int tiles, bool pdl, cudaStream_t s) {
  switch (p.H) {
    case 256: return launch_one<kConst, 1>(p, head, tiles, pdl, s);
    case 2048: return launch_one<kConst, 8>(p, head, tiles, pdl, s);
    case 4096: return launch_one<kConst, 16>(p, head, tiles, pdl, s);
    default: return launch_one<kConst, 0>(p, head, tiles, pdl, s);
  }
}

}  // namespace

cudaError_t prepare_kernels() {
  cudaError_t e;
  if ((e = prepare_one<true, 0>()) != cudaSuccess) return e;
  if ((e = prepare_one<true, 1>()) != cudaSuccess) return e;
  if ((e = prepare_one<true, 8>()) != cudaSuccess) return e;
  if ((e = prepare_one<true, 16>()) != cudaSuccess) return e;
  if ((e = prepare_one<false, 0>()) != cudaSuccess) return e;
  if ((e = prepare_one<false, 1>()) != cudaSuccess) return e;
  if ((e = prepare_one<false, 8>()) != cudaSuccess) return e;
  return prepare_one<false, 16>();
}

cudaError_t launch_step(const StepParams& p, bool const_resident, int head, int tiles, cudaStream_t s, bool pdl) {
  return const_resident ? launch_h<true>(p, head, tiles, pdl, s) : launch_h<false>(p, head, tiles, pdl, s);
}

cudaError_t launch_reset(const ResetParams& r, cudaStream_t s) {
  int bx = r.iv ? 1 : (r.g.n_edges + kThreads * 4 - 1) / (kThreads * 4);
  if (bx < 1) bx = 1;
  if (bx > 64) bx = 64;
  reset_kernel<<<dim3(bx, r.B), kThreads, 0, s>>>(r);
  return cudaGetLastError();
}

template <class... Args>
cudaError_t launch_pdl(void (*kernel)(Args...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// The root step: the GEMM over the root's token rows (the same candidates for
// every sequence: one uniform record per column tile), then the fold and
// transition.  p.hs carries the root arrays; `root_tiles` holds the records.
cudaError_t launch_root_step(const StepParams& p, bool const_resident, const TileCands* root_tiles, int gemm_ctas,
                             cudaStream_t s) {
  StepParams q = p;
  q.hs.root_mode = 1;
  q.hs.union_mode = 0;
  GemmParams gp{};
  gp.xrow = nullptr;     // every sequence takes the root step
  gp.row0_ptr = nullptr; // the step's hidden states are the activation map's first rows
  gp.B = p.B;
  gp.H = p.H;
  gp.row_list = p.hs.root_tok;
  gp.n_cols_ptr = nullptr;
  gp.n_cols_fixed = p.hs.n_root;
  gp.cand_col = nullptr;
  gp.ncand = nullptr;
  gp.tile_cands = root_tiles;
  gp.uniform = 1;
  gp.C = p.cand_cap;
  gp.part = p.hs.part;
  gp.max_tiles = p.hs.max_tiles;
  gp.ksplit = p.hs.ksplit;
  gp.split_part = p.hs.split_part;
  gp.err = p.hs.gemm_err;
  gp.wait_limit = p.hs.wait_limit;
  gp.withhold = p.hs.withhold;
  cudaError_t e = launch_union_gemm(gp, p.hidden, p.hidden_rows, *p.hs.emb_maps, gemm_ctas, s);
  if (e != cudaSuccess) return e;
  return const_resident ? launch_pdl(gemm_finish_kernel<true>, dim3(1, p.B), dim3(kThreads), 0, s, q)
                        : launch_pdl(gemm_finish_kernel<false>, dim3(1, p.B), dim3(kThreads), 0, s, q);
}

cudaError_t launch_gemm_step(const StepParams& p, bool const_resident, int head, int gemm_ctas, cudaStream_t s) {
  StepParams q = p;
  q.hs.union_mode = head == kHeadUnionGemm;
  q.hs.root_mode = 0;
  const size_t fsmem = 2 * (size_t)p.cand_cap * sizeof(int32_t);
  StepParams no_ctrl = q;
  no_ctrl.loop_ctrl = 0;
  no_ctrl.stats = nullptr;
  // Every kernel of the step is a programmatic dependent of the one before
  // (each waits for its predecessor at entry), so launch latency overlaps.
  cudaError_t e = const_resident
                      ? launch_pdl(cand_filter_kernel<true>, dim3(1, p.B), dim3(kThreads), fsmem, s, no_ctrl)
                      : launch_pdl(cand_filter_kernel<false>, dim3(1, p.B), dim3(kThreads), fsmem, s, no_ctrl);
  if (e != cudaSuccess) return e;
  if (q.hs.union_mode) {
    StepParams counted = no_ctrl;
    counted.stats = p.stats;  // (the compaction counts the union's rows)
    if ((e = launch_pdl(union_compact_kernel, dim3(1), dim3(kCompactThreads), 0, s, counted)) != cudaSuccess) return e;
    if ((e = launch_pdl(cand_column_kernel, dim3(1, p.B), dim3(kThreads), (size_t)p.cand_cap * sizeof(int32_t), s,
                        no_ctrl)) != cudaSuccess)
      return e;
  }
  GemmParams gp{};
  gp.xrow = q.hs.xrow;
  gp.row0_ptr = q.hs.row0;
  gp.B = p.B;
  gp.H = p.H;
  gp.row_list = q.hs.union_mode ? q.hs.ulist : nullptr;
  gp.n_cols_ptr = q.hs.union_mode ? q.hs.n_union : nullptr;
  gp.n_cols_fixed = p.V;
  gp.cand_col = q.hs.cand_col;
  gp.ncand = q.hs.ncand;
  gp.tile_cands = q.hs.union_mode ? q.hs.tile_cands : nullptr;
  gp.C = p.cand_cap;
  gp.part = q.hs.part;
  gp.max_tiles = q.hs.max_tiles;
  gp.ksplit = q.hs.union_mode ? q.hs.ksplit : 1;
  gp.split_part = q.hs.split_part;
  gp.err = q.hs.gemm_err;
  gp.wait_limit = q.hs.wait_limit;
  gp.withhold = q.hs.withhold;
  if ((e = launch_union_gemm(gp, p.hidden, p.hidden_rows, *q.hs.emb_maps, gemm_ctas, s)) != cudaSuccess) return e;
  return const_resident ? launch_pdl(gemm_finish_kernel<true>, dim3(1, p.B), dim3(kThreads), 0, s, q)
                        : launch_pdl(gemm_finish_kernel<false>, dim3(1, p.B), dim3(kThreads), 0, s, q);
}

cudaError_t launch_finalize(const StepParams& p, cudaStream_t s) {
  finalize_kernel<<<1, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t const_upload(const void* d_src, size_t bytes, cudaStream_t s) {
  return cudaMemcpyToSymbolAsync(c_walk, d_src, bytes, 0, cudaMemcpyDeviceToDevice, s);
}

}  // namespace tcd
