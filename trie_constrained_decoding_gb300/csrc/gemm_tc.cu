// tcgen05 GEMM with a masked-argmax epilogue: the union-of-legal-rows head and
// the dense head for batches ("Constraint made cheaper than no constraint",
// section "The sparse output layer": in batched form the union of legal rows is
// bounded by the trie; "Understanding Inference for Systems Engineers", section
// 7.5: a sorted row list, then the head over those rows only).
//
//   D[b, n] = sum_h X[b, h] * E[rows[n], h]        b < B (sequences), n < n_cols
//
// Warp-specialised persistent kernel, 320 threads per CTA:
//  - warp 0 (producer) fills a ring of shared-memory stages with TMA: the
//    activation tiles (128 sequences x 64 K-elements per M tile) with tiled
//    2-D loads and, for the dense head, the embedding tile (128 contiguous
//    rows x 64) with one more; all 128-byte swizzled, completion counted on
//    the stage's "full" mbarrier;
//  - warp 1, one thread, issues tcgen05.mma kind::f16 (bf16 in, fp32 in TMEM,
//    M = 128 per tile, N = 128, K = 16 per instruction) and commits each stage
//    back to its "empty" barrier and each finished task to an accumulator-full
//    barrier; TMEM holds two accumulators so one task's epilogue overlaps the
//    next task's MMAs;
//  - warps 2-9 (epilogue) first issue the union head's row gathers (one
//    four-row gather per lane, four groups per warp per stage: one warp's
//    lanes would issue all 32 one after another), then read the accumulator
//    with tcgen05.ld: the thread on TMEM lane t of M tile m owns sequence
//    128 m + t and keeps, over the columns of its own legal candidates only
//    (a 32-byte record per sequence and tile), the largest logit (lowest column
//    on ties; columns ascend with token ids), or, when K is split, writes its
//    candidates' partial sums through a per-warp 32 x 32 transpose so that one
//    store covers consecutive candidates of one sequence.
// A task is one 128-column tile, one K split and, for the union head above
// 128 sequences, one M tile (the dense head keeps both M tiles in one CTA so
// every embedding tile is read once).  Every wait is bounded; on a timeout the
// kernel records an error, stops issuing and frees its TMEM.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include "gemm_tc.h"

namespace tcd {
namespace {

constexpr int kTileN = 128;
static_assert(sizeof(TileCands) == 32 && kTileN == 32 * 4, "a TileCands record covers one 128-column tile");
constexpr int kTileK = 64;  // bf16 elements = one 128-byte swizzle row
constexpr uint32_t kRowBytes = 128;
constexpr uint32_t kATileBytes = 128 * kRowBytes;     // 16 KiB per 128-row M tile
constexpr uint32_t kBTileBytes = kTileN * kRowBytes;  // 16 KiB
constexpr long long kWaitLimit = 1ll << 22;           // default try_wait polls of one wait before giving up

constexpr int kTbStride = 33;  // floats per row of an epilogue warp's 32 x 32 transpose buffer
// Per epilogue warp: the transpose buffer, then each lane's (candidate bits, first index) pair.
constexpr uint32_t kTbWarpBytes = 32 * kTbStride * 4 + 32 * 8;

// MT: 128-row M tiles (sequences) per CTA.  Warps: TMA producer, MMA issuer,
// then 8 epilogue warps: with two M tiles each takes one lane quarter of one
// tile, with one M tile each takes one lane quarter and half of the columns.
// The two-M-tile configuration serves the full-vocabulary GEMM only, whose K
// is never split (no transpose buffers).  Its tasks are 256 columns wide, so
// each activation tile loaded serves twice as many columns (the activations
// are re-read once per task); the accumulator (two M tiles x 256 columns)
// then fills the 512 TMEM columns, so there is one, not two.
template <int MT>
struct Cfg {
  static constexpr int kTaskN = MT == 2 ? 256 : kTileN;  // columns per task (one MMA's N)
  static constexpr int kStages = MT == 2 ? 3 : 5;
  static constexpr uint32_t kStageBytes = MT * kATileBytes + (uint32_t)kTaskN * kRowBytes;
  static constexpr int kAccCols = MT * kTaskN;  // TMEM columns of one accumulator
  static constexpr int kAccs = MT == 2 ? 1 : 2;  // accumulators in TMEM (512 columns)
  static constexpr int kTmemCols = kAccs * kAccCols;
  static constexpr int kEpiWarps = 8;
  static constexpr int kChunks = 2 * MT;  // 32-column chunks of a tile per epilogue warp
  static constexpr int kThreads = 64 + 32 * kEpiWarps;
  static constexpr size_t kTbBytes = MT == 2 ? 0 : (size_t)kEpiWarps * kTbWarpBytes;
};

struct GemmHdr {
  uint64_t full[6];
  uint64_t empty[6];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;  // after an abort: completion of every MMA the issuer started
  uint32_t tmem_base;
  int32_t abort;
  int32_t row0;
  int32_t n_cols;
  int32_t active[256];  // sequence takes this step
};
// Dynamic shared memory of each configuration (1024 bytes of alignment slack)
// within the 227 KiB a CTA may use.
static_assert(1024 + Cfg<1>::kStages * Cfg<1>::kStageBytes + sizeof(GemmHdr) + Cfg<1>::kTbBytes <= 232448, "smem");
static_assert(1024 + Cfg<2>::kStages * Cfg<2>::kStageBytes + sizeof(GemmHdr) + Cfg<2>::kTbBytes <= 232448, "smem");

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, long long limit) {
  for (long long i = 0; i < limit; ++i) {
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

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void tma_tile_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, int x, int r0, int r1, int r2,
                                            int r3, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
      "%5, %6}], [%7];" ::"r"(dst),
      "l"(map), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;             // leading byte offset (unused for swizzled K-major): 16 B
  d |= (uint64_t)(1024u >> 4) << 32;  // stride byte offset: 1024 B
  d |= (uint64_t)1 << 46;             // version
  d |= (uint64_t)2 << 61;             // 128-byte swizzle
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

// Shared-memory accesses by 32-bit shared address (explicitly in the shared
// state space, so that they are never taken for global accesses).
__device__ __forceinline__ void sts32(uint32_t a, uint32_t v) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ void sts64(uint32_t a, uint32_t x, uint32_t y) {
  asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(a), "r"(x), "r"(y) : "memory");
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a) : "memory");
  return v;
}

__device__ __forceinline__ bool gbetter(float l, int32_t c, float bl, int32_t bc) {
  return l > bl || (l == bl && c < bc);
}

template <int MT>
__global__ void __launch_bounds__(Cfg<MT>::kThreads, 1)
    union_gemm_kernel(const GemmParams p, const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmG) {
  using C = Cfg<MT>;
  constexpr int S = C::kStages;
  extern __shared__ __align__(1024) unsigned char gsm[];
  unsigned char* tiles = gsm + ((1024 - (smem_u32(gsm) & 1023)) & 1023);
  GemmHdr* hdr = reinterpret_cast<GemmHdr*>(tiles + S * C::kStageBytes);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t tiles_s = smem_u32(tiles);
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&hdr->full[s]), 1);
      mbar_init(smem_u32(&hdr->empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&hdr->tfull[a]), 1);
      mbar_init(smem_u32(&hdr->tempty[a]), 32 * C::kEpiWarps);
    }
    mbar_init(smem_u32(&hdr->drain), 1);
    hdr->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmG)) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&hdr->tmem_base)),
                 "r"(C::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // Launched as a programmatic dependent of the step's previous kernel: the
  // setup above touches only shared memory, TMEM and the kernel's own
  // parameters, so it overlaps that kernel's tail; its results are read only
  // from here on.  The next kernel may start launching now.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const long long wl = p.wait_limit;  // polls of one wait before it gives up
  // Test switch: CTA 0 issues nothing for its first stage (issue 0), so every
  // wait on that stage runs out and the error path below is taken.
  const bool held = p.withhold != 0 && blockIdx.x == 0;
  long long prod_it = 0;             // stages the producer armed (read at exit after an abort)
  const int KS = p.ksplit;           // K splits per column tile (divides H / 64)
  const int KT = p.H / kTileK / KS;  // k-steps per task
  // Tasks: (column tile, K split, M tile); the M tiles of one (tile, split)
  // are adjacent, so their shared embedding rows are read while still in L2.
  const int MS = MT == 1 ? p.msplit : 1;
  const bool gather = p.row_list != nullptr;
  // Gathered embedding rows: each four-row gather is one TMA instruction per
  // lane, and one warp's lanes issue theirs one after another, so the 32
  // gathers of a stage are spread over the epilogue warps (idle until the
  // accumulator is ready): groups of four rows, kGroups per warp.
  constexpr int kGroups = 32 / C::kEpiWarps;
  const int g = (warp - 2) * kGroups + lane;  // this lane's group (warp >= 2, lane < kGroups)
  // The first task's gathered rows, read together with the step's scalars
  // (the list holds the whole vocabulary, so the read is in bounds; entries
  // past the union are replaced below).
  int pre[4] = {0, 0, 0, 0};
  if (gather && warp >= 2 && lane < kGroups) {
    const int c = (int)(blockIdx.x / MS / KS) * kTileN + 4 * g;
#pragma unroll
    for (int i = 0; i < 4; ++i) pre[i] = c + i < p.n_cols_fixed ? p.row_list[c + i] : 0;
  }
  if (tid == 0) {
    hdr->row0 = p.row0_ptr ? *p.row0_ptr : 0;
    hdr->n_cols = p.n_cols_ptr ? *p.n_cols_ptr : p.n_cols_fixed;
  }
  for (int r = tid; r < 256; r += C::kThreads) hdr->active[r] = (r < p.B && (!p.xrow || p.xrow[r] >= 0)) ? 1 : 0;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = hdr->tmem_base;
  const int row0 = hdr->row0;
  const int n_cols = hdr->n_cols;
  const int n_tiles = (n_cols + C::kTaskN - 1) / C::kTaskN;
  const int n_tasks = n_tiles * KS * MS;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    long long it = 0;
    for (int task = blockIdx.x; task < n_tasks; task += gridDim.x) {
      const int mt = task % MS, tile = task / MS / KS, split = task / MS % KS;
      const int n0 = tile * C::kTaskN;
      bool stop = false;
      for (int kt = 0; kt < KT; ++kt, ++it) {
        const int stage = (int)(it % S);
        const uint32_t ph = (uint32_t)((it / S) & 1);
        if (!mbar_wait(smem_u32(&hdr->empty[stage]), ph ^ 1u, wl)) {
          hdr->abort = 1;
          stop = true;
          break;
        }
        const uint32_t a_base = tiles_s + stage * C::kStageBytes;
        const uint32_t b_base = a_base + MT * kATileBytes;
        const uint32_t fb = smem_u32(&hdr->full[stage]);
        const int k0 = (split * KT + kt) * kTileK;
        if (lane == 0 && !(held && it == 0)) {
          // The stage's bytes: the activation tiles issued here, and the
          // embedding tile (tiled here, or gathered by the epilogue warps).
          mbar_expect_tx(fb, C::kStageBytes);
          for (int m = 0; m < MT; ++m) tma_tile_2d(a_base + m * kATileBytes, &tmA, k0, row0 + (mt + m) * 128, fb);
          // (rows past the vocabulary are filled with zeros and count in full)
          if (!gather)
            for (int h = 0; h < C::kTaskN / kTileN; ++h)
              tma_tile_2d(b_base + h * kBTileBytes, &tmB, k0, n0 + h * kTileN, fb);
        }
        __syncwarp();
      }
      if (stop || hdr->abort) break;
    }
    prod_it = it;
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(128, C::kTaskN);
      long long it = 0;
      int tl = 0;
      for (int task = blockIdx.x; task < n_tasks; task += gridDim.x, ++tl) {
        const int acc = tl % C::kAccs;
        if (!mbar_wait(smem_u32(&hdr->tempty[acc]), (uint32_t)(((tl / C::kAccs) & 1) ^ 1), wl)) {
          hdr->abort = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + acc * C::kAccCols;
        bool stop = false;
        for (int kt = 0; kt < KT; ++kt, ++it) {
          const int stage = (int)(it % S);
          if (!mbar_wait(smem_u32(&hdr->full[stage]), (uint32_t)((it / S) & 1), wl)) {
            hdr->abort = 1;
            stop = true;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = tiles_s + stage * C::kStageBytes;
          const uint32_t b_base = a_base + MT * kATileBytes;
#pragma unroll
          for (int m = 0; m < MT; ++m) {
#pragma unroll
            for (int kk = 0; kk < kTileK / 16; ++kk) {
              mma_bf16(d + m * C::kTaskN, sw128_desc(a_base + m * kATileBytes + kk * 32),
                       sw128_desc(b_base + kk * 32), idesc, (kt > 0 || kk > 0) ? 1u : 0u);
            }
          }
          mma_commit(smem_u32(&hdr->empty[stage]));
        }
        if (stop) break;
        mma_commit(smem_u32(&hdr->tfull[acc]));
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- epilogue
    // Warp w may read only TMEM lane quarter w % 4; warps 2..4MT+1 cover each
    // quarter of each M tile once, so every thread owns one sequence.
    const int q = warp & 3;
    const int m = MT == 2 ? (warp - 2) >> 2 : 0;             // M tile of this warp
    const int ch_lo = MT == 2 ? 0 : ((warp - 2) >> 2) * 2;   // its first 32-column chunk
    const uint32_t tb = smem_u32(hdr + 1) + (uint32_t)(warp - 2) * kTbWarpBytes;  // this warp's transpose buffer
    const uint32_t tbp = tb + 32 * kTbStride * 4;                                    // and its (bits, index) pairs
    long long it = 0;
    int tl = 0;
    for (int task = blockIdx.x; task < n_tasks; task += gridDim.x, ++tl) {
      const int mt = task % MS, tile = task / MS / KS, split = task / MS % KS;
      const int n0 = tile * C::kTaskN;
      const int acc = tl % C::kAccs;
      const int s0 = (mt + m) * 128 + q * 32;  // this warp's first sequence
      const int b = s0 + lane;
      const bool has = hdr->active[b] != 0;
      if (gather) {
        int rr0 = 0, rr1 = 0, rr2 = 0, rr3 = 0;
        if (lane < kGroups) {
          const int c = n0 + 4 * g;
          if (tl == 0) {
            rr0 = c + 0 < n_cols ? pre[0] : 0;
            rr1 = c + 1 < n_cols ? pre[1] : 0;
            rr2 = c + 2 < n_cols ? pre[2] : 0;
            rr3 = c + 3 < n_cols ? pre[3] : 0;
          } else {
            rr0 = c + 0 < n_cols ? p.row_list[c + 0] : 0;
            rr1 = c + 1 < n_cols ? p.row_list[c + 1] : 0;
            rr2 = c + 2 < n_cols ? p.row_list[c + 2] : 0;
            rr3 = c + 3 < n_cols ? p.row_list[c + 3] : 0;
          }
        }
        bool stop = false;
        for (int kt = 0; kt < KT; ++kt, ++it) {
          const int stage = (int)(it % S);
          if (!mbar_wait(smem_u32(&hdr->empty[stage]), (uint32_t)((it / S) & 1) ^ 1u, wl)) {
            hdr->abort = 1;
            stop = true;
            break;
          }
          // (After an abort nothing more is issued: the exit path waits only
          // for the stages the producer armed.)
          if (*reinterpret_cast<volatile int32_t*>(&hdr->abort)) {
            stop = true;
            break;
          }
          const uint32_t b_base = tiles_s + stage * C::kStageBytes + MT * kATileBytes;
          if (lane < kGroups && !(held && it == 0))
            tma_gather4(b_base + g * 4 * kRowBytes, &tmG, (split * KT + kt) * kTileK, rr0, rr1, rr2, rr3,
                        smem_u32(&hdr->full[stage]));
        }
        if (stop) break;
      }
      // Which columns of this task are this sequence's candidates, and the
      // index of the first one (found while the MMAs of this task run).
      constexpr int NH = C::kTaskN / kTileN;  // 128-column halves of a task
      uint32_t cb[4 * NH];
#pragma unroll
      for (int i = 0; i < 4 * NH; ++i) cb[i] = 0u;
      int cpos = 0;
      if (p.tile_cands) {
        if (has) {
          const int4* r =
              reinterpret_cast<const int4*>(p.tile_cands + (p.uniform ? 0 : (size_t)b * p.max_tiles) + tile);
          const int4 bits = __ldg(r);
          cpos = __ldg(reinterpret_cast<const int*>(r + 1));
          cb[0] = (uint32_t)bits.x;
          cb[1] = (uint32_t)bits.y;
          cb[2] = (uint32_t)bits.z;
          cb[3] = (uint32_t)bits.w;
        }
      } else if (has) {
        const int nc = p.ncand[b];
        const int32_t* cand = p.cand_col + (size_t)b * p.C;
        int lo = 0, hi = nc;
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (cand[mid] < n0) lo = mid + 1; else hi = mid;
        }
        cpos = lo;
        for (int i = lo; i < nc; ++i) {
          const int c = cand[i] - n0;
          if (c >= C::kTaskN) break;
          const uint32_t bit = 1u << (c & 31);  // cb kept in registers: no dynamic index
#pragma unroll
          for (int w = 0; w < 4 * NH; ++w) cb[w] |= (c >> 5) == w ? bit : 0u;
        }
      }
      if (!mbar_wait(smem_u32(&hdr->tfull[acc]), (uint32_t)((tl / C::kAccs) & 1), wl)) {
        hdr->abort = 1;
        break;
      }
      tc_fence_after();
      const uint32_t tacc = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * C::kAccCols + m * C::kTaskN);
      if (MT == 1 && KS > 1) {
        // This split's partial sum of every candidate, at the candidate's
        // index.  Through a 32 x 32 transpose in shared memory, one store
        // instruction writes consecutive candidates of one sequence.
        // This warp's chunks: [ch_lo, ch_lo + kChunks); the candidates of
        // earlier chunks come first.
        int pos = cpos + (ch_lo > 0 ? __popc(cb[0]) : 0) + (ch_lo > 1 ? __popc(cb[1]) : 0);
#pragma unroll 1
        for (int ch = ch_lo; ch < ch_lo + C::kChunks; ++ch) {
          uint32_t v[32];
          tmem_ld32(tacc + ch * 32, v);
          if (ch == ch_lo + C::kChunks - 1) {
            // The sums are in registers: hand the accumulator back to the MMA warp.
            tc_fence_before();
            mbar_arrive(smem_u32(&hdr->tempty[acc]));
          }
          const uint32_t bits = (ch == 0) ? cb[0] : (ch == 1) ? cb[1] : (ch == 2) ? cb[2] : cb[3];
#pragma unroll
          for (int j = 0; j < 32; ++j) sts32(tb + (uint32_t)(lane * kTbStride + j) * 4u, v[j]);
          sts64(tbp + lane * 8u, bits, (uint32_t)pos);
          __syncwarp();
          // Sequence s0 + s's column `lane` and its (bits, index) pair, read as
          // shared-memory broadcasts (warp shuffles here cost far more).
          // In two halves of 16 sequences, every load of a half before any of
          // its stores, so that no store waits on a load.
          float* row = p.split_part + ((size_t)split * p.B + s0) * p.C;
#pragma unroll
          for (int h = 0; h < 32; h += 16) {
            uint32_t tv[16];
            int off[16];
            uint32_t take = 0u;
#pragma unroll
            for (int s = 0; s < 16; ++s) tv[s] = lds32(tb + (uint32_t)((h + s) * kTbStride + lane) * 4u);
#pragma unroll
            for (int s = 0; s < 16; ++s) {
              const uint2 bp = lds64(tbp + (h + s) * 8u);
              take |= ((bp.x >> lane) & 1u) << s;
              off[s] = (int)bp.y + __popc(bp.x & ((1u << lane) - 1u));
            }
#pragma unroll
            for (int s = 0; s < 16; ++s)
              if ((take >> s) & 1u) row[(size_t)(h + s) * p.C + off[s]] = __uint_as_float(tv[s]);
          }
          __syncwarp();
          pos += __popc(bits);
        }
      } else {
        // Masked argmax of each 128-column tile of the task: the warps with
        // the first chunk take all of its columns, the others only hand the
        // accumulator back.  One partial per 128-column tile.
        float bl[NH];
        int32_t bcol[NH];
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          bl[h] = -INFINITY;
          bcol[h] = INT32_MAX;
          const int nh0 = n0 + h * kTileN;
#pragma unroll 1
          for (int ch = 0; ch < (ch_lo == 0 ? kTileN / 32 : 0); ++ch) {
            uint32_t v[32];
            tmem_ld32(tacc + h * kTileN + ch * 32, v);
            const uint32_t bits = (ch == 0) ? cb[4 * h] : (ch == 1) ? cb[4 * h + 1] : (ch == 2) ? cb[4 * h + 2]
                                                                                             : cb[4 * h + 3];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float x = __uint_as_float(v[j]);
              if (((bits >> j) & 1u) && gbetter(x, nh0 + ch * 32 + j, bl[h], bcol[h])) {
                bl[h] = x;
                bcol[h] = nh0 + ch * 32 + j;
              }
            }
          }
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&hdr->tempty[acc]));
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          const int nh0 = n0 + h * kTileN;
          if (has && ch_lo == 0 && nh0 < n_cols)
            p.part[(size_t)b * p.max_tiles + nh0 / kTileN] = GemmPartial{bl[h], bcol[h]};
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (hdr->abort) {
    // A wait ran out.  Before the CTA leaves, everything it started must be
    // finished (each wait again bounded): the MMA issuer's MMAs (one commit
    // tracks all of them), and the loads of every stage the producer armed and
    // no MMA consumed (its last S issues; the epilogue's gathers of those
    // stages land on the same barriers).
    if (warp == 1 && lane == 0) {
      mma_commit(smem_u32(&hdr->drain));
      mbar_wait(smem_u32(&hdr->drain), 0u, wl);
    }
    if (warp == 0 && lane == 0) {
      for (long long j = prod_it > S ? prod_it - S : 0; j < prod_it; ++j)
        if (!(held && j == 0)) mbar_wait(smem_u32(&hdr->full[j % S]), (uint32_t)((j / S) & 1), wl);
    }
    __syncwarp();
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::kTmemCols) : "memory");
  }
  if (tid == 0 && hdr->abort) atomicExch(p.err, 1);
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

cudaError_t encode_2d(CUtensorMap* m, const void* base, int64_t rows, int H, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encoder();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)H * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kTileK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

size_t gemm_smem_bytes(int mt) {
  return mt == 2 ? 1024 + (size_t)Cfg<2>::kStages * Cfg<2>::kStageBytes + sizeof(GemmHdr) + Cfg<2>::kTbBytes
                 : 1024 + (size_t)Cfg<1>::kStages * Cfg<1>::kStageBytes + sizeof(GemmHdr) + Cfg<1>::kTbBytes;
}

cudaError_t prepare_gemm() {
  cudaError_t e = cudaFuncSetAttribute(union_gemm_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)gemm_smem_bytes(1));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(union_gemm_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)gemm_smem_bytes(2));
}

int gemm_tile_cols() { return kTileN; }

cudaError_t encode_emb_maps(const void* emb, int V, int H, EmbMaps* out) {
  cudaError_t e = encode_2d(&out->tiled, emb, V, H, kTileN);
  if (e != cudaSuccess) return e;
  return encode_2d(&out->gather, emb, V, H, 1);
}

cudaError_t launch_union_gemm(const GemmParams& p, const void* hidden, int64_t rows, const EmbMaps& emb,
                              int num_ctas, cudaStream_t s) {
  if (p.H % kTileK != 0 || p.B < 1 || p.B > 256 || p.ksplit < 1 || (p.H / kTileK) % p.ksplit != 0 ||
      (p.ksplit > 1 && !p.split_part))
    return cudaErrorInvalidValue;
  CUtensorMap a;
  cudaError_t e = encode_2d(&a, hidden, rows, p.H, 128);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  // Above 128 sequences the union GEMM takes each M tile as a task of its own
  // (more, shorter tasks for its few column tiles); the full-vocabulary GEMM
  // keeps both M tiles in one CTA so that every embedding tile is read once.
  GemmParams q = p;
  if (q.wait_limit <= 0) q.wait_limit = kWaitLimit;
  const bool two_m = p.B > 128 && p.row_list == nullptr;
  if (two_m && p.ksplit != 1) return cudaErrorInvalidValue;  // (no transpose buffers for split sums)
  q.msplit = p.B > 128 && !two_m ? 2 : 1;
  cfg.gridDim = dim3(num_ctas);
  cfg.blockDim = dim3(two_m ? Cfg<2>::kThreads : Cfg<1>::kThreads);
  cfg.dynamicSmemBytes = gemm_smem_bytes(two_m ? 2 : 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (two_m) return cudaLaunchKernelEx(&cfg, union_gemm_kernel<2>, q, a, emb.tiled, emb.gather);
  return cudaLaunchKernelEx(&cfg, union_gemm_kernel<1>, q, a, emb.tiled, emb.gather);
}

}  // namespace tcd
