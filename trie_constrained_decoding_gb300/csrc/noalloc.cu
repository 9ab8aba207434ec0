// tc_dense_argmax_noalloc: the dense head's masked argmax for callers that
// cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: code that runs inside a framework
// whose caching allocator owns the whole device-memory budget, plugin or
// embedded hosts that forbid allocation calls, and latency-critical paths
// where an allocation or a free may synchronise the device.  This entry point
// therefore takes every input and output from the caller and keeps its only
// scratch (per-CTA partial results and per-sequence arrival counters) in the
// file-scope array below, which every GPU that loads the library holds until
// the process exits.
//
// It computes, for each sequence, the fp32 logit of every vocabulary row
// against its hidden state, keeps the rows listed in that sequence's legal
// list, and returns the largest logit with ties broken toward the lower
// token id.  The row dot product uses the same fixed lane map and shuffle
// tree as the library's step kernels, so the results are bit-identical to
// the dense head of tc_step.
#include <cuda_runtime.h>
#include <stdint.h>

#include <climits>
#include <mutex>

#include "tcd.h"
#include "tcd_internal.h"

namespace {

constexpr int kNaThreads = 256;
constexpr int kNaWarps = kNaThreads / 32;
constexpr int kNaMaxDevices = 64;

struct NaPartial {
  float logit;
  int32_t tok;
};

// Scratch shared by every call: TC_NOALLOC_MAX_SLOTS partial results, then
// TC_NOALLOC_MAX_BATCH arrival counters.
constexpr size_t kScratchBytes =
    (size_t)TC_NOALLOC_MAX_SLOTS * sizeof(NaPartial) + (size_t)TC_NOALLOC_MAX_BATCH * sizeof(uint32_t);
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_na_mu;
void* g_na_ptr[kNaMaxDevices];  // device address of g_noalloc_scratch, per device
int g_na_sms[kNaMaxDevices];

// Two bf16 products of a packed word pair (low halves first), each rounded
// once in fp32 (mixed-precision FMA: the same value as an fp32 FMA of the
// widened operands).
__device__ __forceinline__ float na_fma2(uint32_t e, uint32_t x, float acc) {
  asm("{\n .reg .b16 el, eh, xl, xh;\n mov.b32 {el, eh}, %1;\n mov.b32 {xl, xh}, %2;\n"
      " fma.rn.f32.bf16 %0, el, xl, %0;\n fma.rn.f32.bf16 %0, eh, xh, %0;\n}"
      : "+f"(acc)
      : "r"(e), "r"(x));
  return acc;
}

__device__ __forceinline__ float na_dot8(const uint4 e, const uint4 x, float acc) {
  acc = na_fma2(e.x, x.x, acc);
  acc = na_fma2(e.y, x.y, acc);
  acc = na_fma2(e.z, x.z, acc);
  acc = na_fma2(e.w, x.w, acc);
  return acc;
}

__device__ __forceinline__ bool na_better(float l, int32_t t, float bl, int32_t bt) {
  return l > bl || (l == bl && t < bt);
}

// Grid (G, batch).  x is staged in shared memory (any hidden % 8 == 0), the
// legal list after it.  Lane l of a warp accumulates chunks l, l+32, ... of
// 8 elements in order, then a butterfly xor tree.
__global__ void __launch_bounds__(kNaThreads)
dense_argmax_noalloc_kernel(const uint16_t* __restrict__ emb, int32_t V, int32_t H,
                            const uint16_t* __restrict__ hidden, const int32_t* __restrict__ legal,
                            int32_t legal_stride, const int32_t* __restrict__ n_legal, int32_t* tok_out,
                            float* logit_out, NaPartial* part, uint32_t* ticket) {
  extern __shared__ __align__(16) unsigned char na_smem[];
  __shared__ float s_wl[kNaWarps];
  __shared__ int32_t s_wt[kNaWarps];
  __shared__ int32_t s_last;
  const int b = blockIdx.y, g = blockIdx.x, G = gridDim.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nch = H >> 3;
  uint4* xs = reinterpret_cast<uint4*>(na_smem);
  int32_t* s_legal = reinterpret_cast<int32_t*>(na_smem + (size_t)nch * 16);
  const uint4* x4 = reinterpret_cast<const uint4*>(hidden + (size_t)b * H);
  for (int c = tid; c < nch; c += kNaThreads) xs[c] = __ldg(x4 + c);
  int n = __ldg(n_legal + b);
  n = n < 0 ? 0 : (n > legal_stride ? legal_stride : n);
  for (int i = tid; i < n; i += kNaThreads) s_legal[i] = __ldg(legal + (size_t)b * legal_stride + i);
  __syncthreads();

  float wl = -INFINITY;
  int32_t wt = INT_MAX;
  for (int32_t r = g * kNaWarps + warp; r < V; r += G * kNaWarps) {
    const uint4* row = reinterpret_cast<const uint4*>(emb + (size_t)r * H);
    float acc = 0.f;
    for (int c = lane; c < nch; c += 32) acc = na_dot8(__ldg(row + c), xs[c], acc);
    acc += __shfl_xor_sync(0xffffffffu, acc, 16);
    acc += __shfl_xor_sync(0xffffffffu, acc, 8);
    acc += __shfl_xor_sync(0xffffffffu, acc, 4);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    int lo = 0, hi = n;  // r is legal iff it is in the ascending list
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (s_legal[mid] < r) lo = mid + 1; else hi = mid;
    }
    if (lo < n && s_legal[lo] == r && na_better(acc, r, wl, wt)) {
      wl = acc;
      wt = r;
    }
  }
  if (lane == 0) {
    s_wl[warp] = wl;
    s_wt[warp] = wt;
  }
  __syncthreads();
  if (tid == 0) {
    float bl = -INFINITY;
    int32_t bt = INT_MAX;
    for (int i = 0; i < kNaWarps; ++i)
      if (na_better(s_wl[i], s_wt[i], bl, bt)) { bl = s_wl[i]; bt = s_wt[i]; }
    NaPartial* slot = part + (size_t)b * G;
    slot[g] = NaPartial{bl, bt};
    __threadfence();
    const uint32_t arrived = atomicAdd(&ticket[b], 1u);
    s_last = arrived == (uint32_t)G - 1;
    if (s_last) {
      __threadfence();
      bl = -INFINITY;
      bt = INT_MAX;
      for (int i = 0; i < G; ++i) {
        const float l = __ldcg(&slot[i].logit);
        const int32_t t = __ldcg(&slot[i].tok);
        if (na_better(l, t, bl, bt)) { bl = l; bt = t; }
      }
      const bool found = bt != INT_MAX;
      tok_out[b] = found ? bt : -1;
      logit_out[b] = found ? bl : 0.f;
    }
  }
}

// Once per device, with that device current: the device address of the
// scratch array (its name in host code is only a host-side stand-in).
tc_status na_setup(int dev, void** scratch, int* sms) {
  std::lock_guard<std::mutex> lk(g_na_mu);
  if (!g_na_ptr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      tcd::set_error_message(std::string("tc_dense_argmax_noalloc: cudaGetSymbolAddress failed: ") +
                             cudaGetErrorString(e));
      cudaGetLastError();
      return TC_ERR_CUDA;
    }
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess || n <= 0) n = 148;
    cudaGetLastError();
    g_na_sms[dev] = n;
    g_na_ptr[dev] = p;
  }
  *scratch = g_na_ptr[dev];
  *sms = g_na_sms[dev];
  return TC_OK;
}

}  // namespace

extern "C" tc_status tc_dense_argmax_noalloc(const void* emb_bf16, int32_t vocab, int32_t hidden,
                                             const void* hidden_bf16, int32_t batch, const int32_t* legal,
                                             int32_t legal_stride, const int32_t* n_legal, int32_t* tok_out,
                                             float* logit_out, void* stream) {
  if (!emb_bf16 || !hidden_bf16 || !legal || !n_legal || !tok_out || !logit_out || vocab < 1 ||
      hidden < 8 || hidden % 8 != 0 || legal_stride < 1) {
    tcd::set_error_message("tc_dense_argmax_noalloc: invalid arguments");
    return TC_ERR_INVALID_ARG;
  }
  if ((reinterpret_cast<uintptr_t>(emb_bf16) & 15) || (reinterpret_cast<uintptr_t>(hidden_bf16) & 15)) {
    tcd::set_error_message("tc_dense_argmax_noalloc: embedding and hidden states must be 16-byte aligned");
    return TC_ERR_INVALID_ARG;
  }
  if (batch < 1 || batch > TC_NOALLOC_MAX_BATCH || hidden > TC_NOALLOC_MAX_HIDDEN ||
      legal_stride > TC_NOALLOC_MAX_LEGAL) {
    tcd::set_error_message("tc_dense_argmax_noalloc: batch must be 1.." + std::to_string(TC_NOALLOC_MAX_BATCH) +
                           ", hidden at most " + std::to_string(TC_NOALLOC_MAX_HIDDEN) +
                           " and legal_stride at most " + std::to_string(TC_NOALLOC_MAX_LEGAL));
    return TC_ERR_CAPACITY;
  }
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNaMaxDevices) {
    cudaGetLastError();
    tcd::set_error_message("tc_dense_argmax_noalloc: no usable current device");
    return TC_ERR_CUDA;
  }
  void* scratch = nullptr;
  int sms = 0;
  tc_status rc = na_setup(dev, &scratch, &sms);
  if (rc != TC_OK) return rc;
  int G = (2 * sms) / batch;
  if (G < 1) G = 1;
  if (G * batch > TC_NOALLOC_MAX_SLOTS) G = TC_NOALLOC_MAX_SLOTS / batch;
  NaPartial* part = static_cast<NaPartial*>(scratch);
  uint32_t* ticket = reinterpret_cast<uint32_t*>(static_cast<unsigned char*>(scratch) +
                                                 (size_t)TC_NOALLOC_MAX_SLOTS * sizeof(NaPartial));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The counters keep the previous call's values: clear them first.
  cudaError_t e = cudaMemsetAsync(ticket, 0, sizeof(uint32_t) * (size_t)batch, s);
  if (e != cudaSuccess) {
    tcd::set_error_message(std::string("tc_dense_argmax_noalloc: ") + cudaGetErrorString(e));
    cudaGetLastError();
    return TC_ERR_CUDA;
  }
  const size_t smem = (size_t)(hidden / 8) * 16 + (size_t)legal_stride * sizeof(int32_t);
  dense_argmax_noalloc_kernel<<<dim3(G, batch), kNaThreads, smem, s>>>(
      static_cast<const uint16_t*>(emb_bf16), vocab, hidden, static_cast<const uint16_t*>(hidden_bf16), legal,
      legal_stride, n_legal, tok_out, logit_out, part, ticket);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    tcd::set_error_message(std::string("tc_dense_argmax_noalloc launch: ") + cudaGetErrorString(e));
    return TC_ERR_CUDA;
  }
  return TC_OK;
}
