// tcgen05 GEMM with a masked-argmax epilogue: the union-of-legal-rows head and
// the dense head for batches ("Constraint made cheaper than no constraint",
// section "The sparse output layer": in batched form the union of legal rows is
// bounded by the trie; "Understanding Inference for Systems Engineers", section
// 7.5: a sorted row list, then the head over those rows only).
//
//   D[b, n] = sum_h X[b, h] * E[rows[n], h]        b < B (sequences), n < n_cols
//
// A = X (one 128-row tile per 128 sequences, up to two), B = the embedding rows
// listed for the tile's 256 columns (rows[n] = n for the dense head), both bf16
// K-major in shared memory in the 128-byte swizzled layout, staged by cp.async
// (the rows are gathered, so a rectangular TMA box does not describe them).
// One thread issues tcgen05.mma kind::f16 (bf16 in, fp32 accumulate) into TMEM:
// 128 lanes x 256 columns per M tile.  The epilogue reads TMEM with tcgen05.ld;
// thread t of warp w owns sequence 128*m + 32*w + t and keeps, over the columns
// of its own legal candidates only, the largest logit (lowest column on ties;
// columns ascend with token ids) - one (logit, column) partial per sequence and
// column tile.  Persistent CTAs loop over column tiles.
//
// Every wait on an mbarrier is bounded; on a timeout the kernel records an
// error, drains its own copies, frees its TMEM and returns.
#include <cuda_runtime.h>
#include <stdint.h>

#include "gemm_tc.h"

namespace tcd {
namespace {

constexpr int kThreadsG = 128;
constexpr int kTileN = 256;
constexpr int kTileK = 64;         // bf16 elements = one 128-byte swizzle row
constexpr int kStages = 3;
constexpr uint32_t kRowBytes = 128;
constexpr uint32_t kATileBytes = 128 * kRowBytes;    // 16 KiB per 128-row M tile
constexpr uint32_t kBTileBytes = kTileN * kRowBytes;  // 32 KiB
constexpr long long kWaitLimit = 1ll << 20;          // try_wait polls before giving up

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase of the given parity to complete.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (long long i = 0; i < kWaitLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;                  // leading byte offset (unused for swizzled K-major): 16 B
  d |= (uint64_t)(1024u >> 4) << 32;       // stride byte offset: 1024 B
  d |= (uint64_t)1 << 46;                  // version
  d |= (uint64_t)2 << 61;                  // 128-byte swizzle
  return d;
}

// Instruction descriptor of kind::f16: D fp32, A and B bf16, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ bool gbetter(float l, int32_t c, float bl, int32_t bc) {
  return l > bl || (l == bl && c < bc);
}

struct GemmSmemHeader {
  uint64_t empty[kStages];  // one arrival per tcgen05.commit of a k-step
  uint32_t tmem_base;
  int32_t abort;
  int32_t rows[kTileN];     // embedding row of each column of the current tile
  int64_t xoff[256];        // hidden-row offset of each sequence (-1: no row)
  uint32_t cbits[256][kTileN / 32];  // per sequence: its candidate columns in the current tile
  int32_t cpos[256];        // per sequence: index of its first candidate in the current tile
};

template <int MT>
__global__ void __launch_bounds__(kThreadsG, 1) union_gemm_kernel(const GemmParams p) {
  extern __shared__ __align__(1024) unsigned char gsm[];
  // Operand tiles first (1024-byte aligned), header after them.
  const uint32_t stage_bytes = MT * kATileBytes + kBTileBytes;
  unsigned char* tiles = gsm + ((1024 - (smem_u32(gsm) & 1023)) & 1023);
  GemmSmemHeader* hdr = reinterpret_cast<GemmSmemHeader*>(tiles + kStages * stage_bytes);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t tiles_s = smem_u32(tiles);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&hdr->empty[s]), 1);
    hdr->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&hdr->tmem_base)),
                 "r"(MT * kTileN)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  for (int r = tid; r < MT * 128; r += kThreadsG) hdr->xoff[r] = r < p.B ? p.xrow[r] : -1;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = hdr->tmem_base;

  const int n_cols = p.n_cols_ptr ? *p.n_cols_ptr : p.n_cols_fixed;
  const int n_tiles = (n_cols + kTileN - 1) / kTileN;
  const int KS = p.ksplit;              // K splits per column tile (divides H / 64)
  const int KT = p.H / kTileK / KS;     // k-steps per task
  constexpr uint32_t idesc = idesc_bf16(128, kTileN);
  long long g = 0;  // global k-step counter of this CTA (stage = g % kStages)
  bool failed = false;

  for (int task = blockIdx.x; task < n_tiles * KS && !failed; task += gridDim.x) {
    const int tile = task / KS, split = task % KS;
    const int n0 = tile * kTileN;
    const int kbase = split * KT;
    for (int r = tid; r < kTileN; r += kThreadsG) {
      const int col = n0 + r;
      hdr->rows[r] = col < n_cols ? (p.row_list ? p.row_list[col] : col) : -1;
    }
    __syncthreads();

    auto load_stage = [&](int kt, int stage) {
      const uint32_t a_base = tiles_s + stage * stage_bytes;
      const uint32_t b_base = a_base + MT * kATileBytes;
      const int k0 = (kbase + kt) * kTileK;
      for (int i = tid; i < MT * 128 * 8; i += kThreadsG) {
        const int r = i >> 3, c = i & 7;
        const int64_t off = hdr->xoff[r];
        const uint16_t* src = off >= 0 ? p.hidden + off + k0 + c * 8 : p.hidden;
        cp_async16(a_base + r * kRowBytes + ((c ^ (r & 7)) << 4), src, off >= 0 ? 16u : 0u);
      }
      for (int i = tid; i < kTileN * 8; i += kThreadsG) {
        const int r = i >> 3, c = i & 7;
        const int row = hdr->rows[r];
        const uint16_t* src = row >= 0 ? p.emb + (size_t)row * p.H + k0 + c * 8 : p.emb;
        cp_async16(b_base + r * kRowBytes + ((c ^ (r & 7)) << 4), src, row >= 0 ? 16u : 0u);
      }
    };

    // Prologue: the first kStages-1 k-steps of this tile.  Every stage is free:
    // the previous tile ended by waiting for its last MMA.
    for (int s = 0; s < kStages - 1; ++s) {
      if (s < KT) load_stage(s, (int)((g + s) % kStages));
      cp_async_commit();
    }
    // While those copies fly: which columns of this tile are each sequence's
    // candidates (thread t serves sequences t and 128 + t in the epilogue).
    for (int m = 0; m < MT; ++m) {
      const int b = m * 128 + tid;
#pragma unroll
      for (int q = 0; q < kTileN / 32; ++q) hdr->cbits[b][q] = 0u;
      int lo = 0;
      if (hdr->xoff[b] >= 0) {
        const int nc = p.ncand[b];
        const int32_t* cand = p.cand_col + (size_t)b * p.C;
        int hi = nc;
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (cand[mid] < n0) lo = mid + 1; else hi = mid;
        }
        for (int i = lo; i < nc; ++i) {
          const int c = cand[i] - n0;
          if (c >= kTileN) break;
          hdr->cbits[b][c >> 5] |= 1u << (c & 31);
        }
      }
      hdr->cpos[b] = lo;
    }
    for (int kt = 0; kt < KT; ++kt) {
      const long long gk = g + kt;
      const int nxt = kt + kStages - 1;
      if (nxt < KT) {
        // The stage of k-step nxt last held k-step nxt - kStages = kt - 1.
        if (kt >= 1) {
          const long long gp = gk - 1;
          if (!mbar_wait(smem_u32(&hdr->empty[gp % kStages]), (uint32_t)((gp / kStages) & 1))) hdr->abort = 1;
        }
        load_stage(nxt, (int)((gk + kStages - 1) % kStages));
      }
      cp_async_commit();
      cp_async_wait<kStages - 1>();
      fence_proxy_async();
      __syncthreads();
      if (hdr->abort) {
        failed = true;
        break;
      }
      if (tid == 0) {
        tc_fence_after();
        const int stage = (int)(gk % kStages);
        const uint32_t a_base = tiles_s + stage * stage_bytes;
        const uint32_t b_base = a_base + MT * kATileBytes;
#pragma unroll
        for (int m = 0; m < MT; ++m) {
#pragma unroll
          for (int kk = 0; kk < kTileK / 16; ++kk) {
            const uint64_t ad = sw128_desc(a_base + m * kATileBytes + kk * 32);
            const uint64_t bd = sw128_desc(b_base + kk * 32);
            mma_bf16(tmem + m * kTileN, ad, bd, idesc, (kt > 0 || kk > 0) ? 1u : 0u);
          }
        }
        mma_commit(smem_u32(&hdr->empty[stage]));
      }
    }
    if (failed) break;
    // All MMAs of the tile are complete once its last commit has arrived.
    const long long gl = g + KT - 1;
    if (!mbar_wait(smem_u32(&hdr->empty[gl % kStages]), (uint32_t)((gl / kStages) & 1))) {
      hdr->abort = 1;
    }
    __syncthreads();
    if (hdr->abort) {
      failed = true;
      break;
    }
    tc_fence_after();
    g += KT;

    // Epilogue: masked argmax of each sequence over its candidates in this tile.
    for (int m = 0; m < MT; ++m) {
      const int b = m * 128 + warp * 32 + lane;
      const bool has = hdr->xoff[b] >= 0;
      float bl = -INFINITY;
      int32_t bc = INT32_MAX;
      float* sp = KS > 1 && has ? p.split_part + ((size_t)split * p.B + b) * p.C : nullptr;
      int pos = hdr->cpos[b];  // candidate index of the next set bit
#pragma unroll 1
      for (int ch = 0; ch < kTileN / 32; ++ch) {
        uint32_t v[32];
        tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(m * kTileN + ch * 32), v);
        const int c0 = n0 + ch * 32;
        const uint32_t bits = hdr->cbits[b][ch];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if ((bits >> j) & 1u) {
            const float x = __uint_as_float(v[j]);
            if (sp) {
              sp[pos++] = x;  // this split's partial sum of candidate pos
            } else if (gbetter(x, c0 + j, bl, bc)) {
              bl = x;
              bc = c0 + j;
            }
          }
        }
      }
      if (has && KS == 1) p.part[(size_t)b * p.max_tiles + tile] = GemmPartial{bl, bc};
    }
    tc_fence_before();
    __syncthreads();  // TMEM is read before the next tile's MMAs overwrite it
    tc_fence_after();
  }

  if (failed) {
    cp_async_wait_all();
    if (tid == 0) atomicExch(p.err, 1);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(MT * kTileN) : "memory");
  }
}

}  // namespace

size_t gemm_smem_bytes(int mt) {
  return 1024 + (size_t)kStages * (mt * kATileBytes + kBTileBytes) + sizeof(GemmSmemHeader);
}

cudaError_t prepare_gemm() {
  cudaError_t e = cudaFuncSetAttribute(union_gemm_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)gemm_smem_bytes(1));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(union_gemm_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)gemm_smem_bytes(2));
}

int gemm_tile_cols() { return kTileN; }

cudaError_t launch_union_gemm(const GemmParams& p, int num_ctas, cudaStream_t s) {
  if (p.H % kTileK != 0 || p.B < 1 || p.B > 256 || p.ksplit < 1 || (p.H / kTileK) % p.ksplit != 0 ||
      (p.ksplit > 1 && !p.split_part))
    return cudaErrorInvalidValue;
  const int mt = p.B > 128 ? 2 : 1;
  if (mt == 1) union_gemm_kernel<1><<<num_ctas, kThreadsG, gemm_smem_bytes(1), s>>>(p);
  else union_gemm_kernel<2><<<num_ctas, kThreadsG, gemm_smem_bytes(2), s>>>(p);
  return cudaGetLastError();
}

}  // namespace tcd
