// Batch-invariant GEMM on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// C[M,N] = A[M,K] . B[N,K]^T, both operands K-major.  TMA streams
// 128-byte-swizzled K slabs of A and B into a shared-memory ring; one thread
// issues tcgen05.mma (M=128, N=BN) into FP32 accumulators in TMEM; epilogue
// warps read them back (tcgen05.ld), fold and store.
//
// Invariance ("Finish RL Training Faster", section "让训练前向使用推理的数值":
// one batch-invariant GEMM schedule with a fixed K split): K is cut into
// chunks whose boundaries depend on K only (at most 8 for bf16, 128-element
// blocks for FP8); each chunk is accumulated from zero as a fixed sequence of
// K=16 / K=32 MMA steps, and the chunk results are added in ascending chunk
// order in FP32 (FP8: each scaled by its block scales first).  Nothing about
// M enters that arithmetic: rows past M are TMA zero-fill and are not stored,
// and the tile width, the persistent-CTA walk and whether chunks are folded
// inside one CTA or by a second kernel only decide where the same additions
// run.  FAST mode (the
// batch-dependent comparator the pages measure against) does not chunk large
// M and splits K to fill the GPU when M is small.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace biv {
namespace {

constexpr int BM = 128;

template <int BN>
struct Fp8Cfg {
  static constexpr int BK = 128;                      // 128 e4m3 = one 128-byte swizzle row
  static constexpr int A_BYTES = BM * BK;
  static constexpr int B_BYTES = BN * BK;
  static constexpr int STAGE = A_BYTES + B_BYTES;     // one K block of A and of B
  static constexpr int BLOCKS = 4;                    // K blocks in the ring (kpb per stage)
  static constexpr int TMEM_COLS = 2 * BN;            // two accumulator buffers
  static constexpr int MAX_GROUPS = 1024;
  static constexpr int EPI_WARPS = 16;                // lane quarter x 64-column quarter
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  static constexpr int SMEM =
      BLOCKS * STAGE + 1024 + (2 * BLOCKS + 4) * 8 + 16 + (MAX_GROUPS + 1) * 4;
  static_assert(BN == 4 * 64, "each epilogue warp promotes one 64-column quarter");
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Store 32 consecutive FP32 accumulator columns of one row.  bf16 rows whose
// 64 bytes are 32-byte aligned go out as two whole-sector stores.
template <bool F32OUT>
__device__ __forceinline__ void store_row32(void* C, int64_t ldc, int row, int n, int N,
                                            const uint32_t (&r)[32], bool vec_ok) {
  if (F32OUT) {
    float* dst = static_cast<float*>(C) + int64_t(row) * ldc + n;
    if (vec_ok && n + 32 <= N) {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        reinterpret_cast<float4*>(dst)[j] =
            make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                        __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (n + j < N) dst[j] = __uint_as_float(r[j]);
    }
  } else {
    uint16_t* dst = static_cast<uint16_t*>(C) + int64_t(row) * ldc + n;
    if (vec_ok && n + 32 <= N && (reinterpret_cast<uintptr_t>(dst) & 31) == 0) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t w[8];
#pragma unroll
        for (int x = 0; x < 8; ++x)
          w[x] = pack_bf2(__uint_as_float(r[16 * h + 2 * x]), __uint_as_float(r[16 * h + 2 * x + 1]));
        st_global_v8(dst + 16 * h, w);
      }
    } else if (vec_ok && n + 32 <= N) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint4 v;
        v.x = pack_bf2(__uint_as_float(r[8 * j + 0]), __uint_as_float(r[8 * j + 1]));
        v.y = pack_bf2(__uint_as_float(r[8 * j + 2]), __uint_as_float(r[8 * j + 3]));
        v.z = pack_bf2(__uint_as_float(r[8 * j + 4]), __uint_as_float(r[8 * j + 5]));
        v.w = pack_bf2(__uint_as_float(r[8 * j + 6]), __uint_as_float(r[8 * j + 7]));
        reinterpret_cast<uint4*>(dst)[j] = v;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (n + j < N) dst[j] = f2bf(__uint_as_float(r[j]));
    }
  }
}

// Store W consecutive FP32 register values of one row (static indexing only).
template <int W, bool F32OUT>
__device__ __forceinline__ void store_row_regs(void* C, int64_t ldc, int row, int n, int N,
                                               const float (&r)[W], bool vec_ok) {
  if (vec_ok && n + W <= N) {
    if (F32OUT) {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(C) + int64_t(row) * ldc + n);
#pragma unroll
      for (int j = 0; j < W / 4; ++j)
        dst[j] = make_float4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
    } else {
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(C) + int64_t(row) * ldc + n);
#pragma unroll
      for (int j = 0; j < W / 8; ++j)
        dst[j] = make_uint4(pack_bf2(r[8 * j], r[8 * j + 1]), pack_bf2(r[8 * j + 2], r[8 * j + 3]),
                            pack_bf2(r[8 * j + 4], r[8 * j + 5]), pack_bf2(r[8 * j + 6], r[8 * j + 7]));
    }
  } else {
#pragma unroll
    for (int j = 0; j < W; ++j) {
      if (n + j < N) {
        if (F32OUT)
          static_cast<float*>(C)[int64_t(row) * ldc + n + j] = r[j];
        else
          static_cast<uint16_t*>(C)[int64_t(row) * ldc + n + j] = f2bf(r[j]);
      }
    }
  }
}

// ------------------------------------------------------------ bf16 kernel --
// The K schedule of every bf16 GEMM.  K is cut into at most 8 chunks of
// kc_blocks x 64 elements whose boundaries depend on K only.  Each chunk's
// partial P_c is accumulated by tcgen05 from zero in ascending K steps of 16;
// the output is the FP32 left fold r = P_0, r = r + P_1, ..., rounded once to
// the output type.  Two ways of running that schedule give the same bits:
//  - fold mode: a work item is a whole 128 x BN tile; the epilogue warps fold
//    its chunks in registers as the MMA warp finishes them;
//  - partial mode: a work item is one (tile, chunk) pair and its P_c goes to
//    the workspace (row-major per chunk); gemm_fold_kernel, or a consumer op
//    that reads the partials directly, folds every element's partials in
//    chunk order.  This spreads a few output tiles (decode-sized M) over every
//    SM without changing any element's arithmetic.
//
// Persistent CTAs, 320 threads: warp 0 = TMA producer, warp 1 = MMA issuer
// and TMEM owner, warps 2..9 = epilogue.  Epilogue warp w reads TMEM lanes
// 32*(w%4).. (its lane quarter) and columns [h*BN/2, (h+1)*BN/2) with
// h = (w-2)/4.  TMEM holds two BN-column accumulators (chunk double buffer).
// Shared memory: S stages of B (BN x 64) then S stages of A (m_box x 64), and
// a pad after the last A stage: the M=128 MMA reads 128 A rows, the rows past
// m_box never feed a stored output row.
struct GemmArgs {
  void* C;
  int64_t ldc;
  int M, N, K;
  int kc_blocks;        // K blocks of 64 per chunk
  int m_box;            // rows of the A box (multiple of 16, <= 128)
  int stages;           // pipeline depth (<= kMaxStages)
  int partial;          // 1: partial mode
  float* ws;            // partial mode: [chunks][M][ldp] FP32
  int64_t ldp;          // partial row pitch (N rounded up to the tile width)
  int vec_ok;           // C rows 16-byte aligned
  int n_fastest;        // fold mode: walk N tiles first
  int b_after_wait;     // 1: B is written by the previous kernel (no early prefetch)
  int kpb;              // K blocks of 64 per pipeline stage (2: 3-D maps, two panels per copy)
  // log-softmax epilogue (LSE instantiation): per row and 128-column group g
  // of the output, (max, sum of exp(z - max)) to lse[row * ngroups + g]; the
  // logit at target[row] to zt[row]
  const int32_t* target;
  float2* lse;
  float* zt;
  int ngroups;
  int ws_v8;                   // partial mode: the workspace is 32-byte aligned
  int* err;
};

constexpr int kMaxStages = 16;
constexpr int kLseGroup = 128;   // logit columns per (max, sum exp) pair
// The invariant schedule cuts K into at most 8 chunks of at least 8 blocks of
// 64 (shorter chunks make the register fold of wide tiles stall the MMA:
// measured on GB300 at M = 16384, K = 2048, 256-element chunks ran 22% below
// one unchunked pass).
constexpr int kMaxChunks = 8;
constexpr int kMinChunkBlocks = 8;
constexpr int kEpiWarps = 8;
constexpr int kGemmThreads = 64 + 32 * kEpiWarps;

// Epilogue staging: per epilogue warp a 32 x 33 FP32 block, used to turn its
// row-per-lane results into row-contiguous (coalesced) global stores.
constexpr int kStagePitch = 33;
constexpr size_t kStagingBytes = size_t(kEpiWarps) * 32 * kStagePitch * 4;

template <int BN>
struct GemmSmem {
  static constexpr int B_STAGE = BN * 128;
  // bytes of dynamic shared memory for `stages` stages of an m_box-row A box
  // (the store staging blocks only in fold mode)
  static size_t bytes(int stages, int m_box, bool staging, int kpb = 1) {
    return 1024 + size_t(stages) * kpb * (B_STAGE + m_box * 128) + (128 - m_box) * 128 +
           (2 * kMaxStages + 4) * 8 + 16 + (staging ? kStagingBytes : 0);
  }
};

// PARTIAL: the partial-mode instantiation.  Its epilogue keeps no running
// sum, so it is compiled for half the register file; with PDL the next
// kernel's CTAs can then start on the same SMs while it runs.
// LSE: fold mode whose epilogue reduces each 128-column half tile of a row to
// its (max, sum exp) pair instead of storing the FP32 logits.
template <int BN, bool F32OUT, bool PARTIAL, bool LSE = false>
__global__ void __launch_bounds__(kGemmThreads, PARTIAL ? 2 : 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB, const GemmArgs p) {
  constexpr int B_STAGE = GemmSmem<BN>::B_STAGE;
  constexpr int HALF = BN / 2;
  static_assert(HALF % 32 == 0, "epilogue reads 32-column groups");
  // two BN-column accumulators, allocated as a power of two
  constexpr uint32_t kTmemCols = 2 * BN <= 128 ? 128 : (2 * BN <= 256 ? 256 : 512);
  // partial mode runs on tiles of at most 128 columns (register budget)
  constexpr bool kPartialOk = BN <= 128;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int S = p.stages;
  // a stage holds kpb K blocks of 64: [block][rows][128 B] for A and for B
  const int a_blk = p.m_box * 128, b_blk = B_STAGE;
  const int a_stage = a_blk * p.kpb, b_stage = b_blk * p.kpb;
  uint8_t* sB = smem;
  uint8_t* sA = smem + S * b_stage;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sA + S * a_stage + (128 - p.m_box) * 128);
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kMaxStages);
  const uint32_t tfull0 = smem_u32(bars + 2 * kMaxStages);
  const uint32_t tempty0 = smem_u32(bars + 2 * kMaxStages + 2);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kMaxStages + 4);
  float* staging = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) +
                                            (2 * kMaxStages + 4) * 8 + 16);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KB = (p.K + 63) / 64;
  const int chunks = (KB + p.kc_blocks - 1) / p.kc_blocks;
  const int tiles_m = (p.M + BM - 1) / BM, tiles_n = (p.N + BN - 1) / BN;
  const int tiles = tiles_m * tiles_n;
  static_assert(!PARTIAL || kPartialOk, "partial mode needs tiles of at most 128 columns");
  constexpr bool partial = PARTIAL;
  const int items = partial ? tiles * chunks : tiles;
  // item -> tile and chunk range
  auto item_tile = [&](int i) { return partial ? i / chunks : i; };
  auto item_c0 = [&](int i) { return partial ? i % chunks : 0; };
  auto item_c1 = [&](int i) { return partial ? i % chunks + 1 : chunks; };
  auto tile_m0 = [&](int t) { return (p.n_fastest ? t / tiles_n : t % tiles_m) * BM; };
  auto tile_n0 = [&](int t) { return (p.n_fastest ? t % tiles_n : t / tiles_m) * BN; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int j = 0; j < 2; ++j) {
      mbar_init(tfull0 + 8 * j, 1);
      mbar_init(tempty0 + 8 * j, kEpiWarps);
    }
    fence_barrier_init();
  }
  __syncwarp();
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_trigger();  // TMEM is held: the next kernel in the stream may be scheduled

  int issued = 0;
  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      const uint32_t tx = uint32_t(a_stage + b_stage);
      // one stage = K blocks [kb, kb + kpb) of one chunk (a chunk's odd last
      // block leaves the stage's second block unused)
      auto load = [&](const CUtensorMap* map, uint8_t* dst, int kb, int row0, uint32_t bar) {
        if (p.kpb == 2)
          tma_load_3d(smem_u32(dst), map, bar, 0, row0, kb);
        else
          tma_load_2d(smem_u32(dst), map, bar, kb * 64, row0);
      };
      // The weights (B) of the first stages do not depend on the previous
      // kernel: fetch them before waiting for it, then A and the rest.
      int pre = 0;
      if (!p.b_after_wait) {
        const int i = blockIdx.x, n0 = tile_n0(item_tile(i));
        for (int c = item_c0(i); c < item_c1(i) && pre < S; ++c) {
          const int kb1 = min(KB, (c + 1) * p.kc_blocks);
          for (int kb = c * p.kc_blocks; kb < kb1 && pre < S; kb += p.kpb, ++pre) {
            mbar_expect_tx(full0 + 8 * pre, tx);
            load(&tmB, sB + pre * b_stage, kb, n0, full0 + 8 * pre);
          }
        }
      }
      pdl_wait();
      bool ok = true;
      for (int i = blockIdx.x; i < items && ok; i += gridDim.x) {
        const int t = item_tile(i), m0 = tile_m0(t), n0 = tile_n0(t);
        for (int c = item_c0(i); c < item_c1(i) && ok; ++c) {
          const int kb1 = min(KB, (c + 1) * p.kc_blocks);
          for (int kb = c * p.kc_blocks; kb < kb1; kb += p.kpb) {
            const int s = issued % S;
            if (issued >= pre) {
              if (issued >= S && !mbar_wait(empty0 + 8 * s, ((issued / S) - 1) & 1, p.err)) {
                ok = false;
                break;
              }
              mbar_expect_tx(full0 + 8 * s, tx);
              load(&tmB, sB + s * b_stage, kb, n0, full0 + 8 * s);
            }
            load(&tmA, sA + s * a_stage, kb, m0, full0 + 8 * s);
            ++issued;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_mma(1u, BM, BN);
      int it = 0, j = 0;
      bool ok = true;
      for (int i = blockIdx.x; i < items && ok; i += gridDim.x) {
        for (int c = item_c0(i); c < item_c1(i) && ok; ++c, ++j) {
          const int b = j & 1;
          if (j >= 2 && !mbar_wait(tempty0 + 8 * b, ((j >> 1) - 1) & 1, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t dt = tmem + b * BN;
          const int kb0 = c * p.kc_blocks, kb1 = min(KB, kb0 + p.kc_blocks);
          for (int kb = kb0; kb < kb1; kb += p.kpb, ++it) {
            const int s = it % S;
            if (!mbar_wait(full0 + 8 * s, (it / S) & 1, p.err)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const int nb = min(p.kpb, kb1 - kb);
            for (int q = 0; q < nb; ++q) {
              const uint32_t a0 = smem_u32(sA + s * a_stage + q * a_blk);
              const uint32_t b0 = smem_u32(sB + s * b_stage + q * b_blk);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                umma_f16(dt, sdesc_k_sw128(a0 + kk * 32), sdesc_k_sw128(b0 + kk * 32), idesc,
                         (kb + q != kb0 || kk != 0) ? 1u : 0u);
            }
            umma_commit(empty0 + 8 * s);
          }
          if (ok) umma_commit(tfull0 + 8 * b);
        }
      }
    }
  } else {
    // ---------------------------------------------------------- epilogue --
    const int q = warp & 3, col0 = ((warp - 2) >> 2) * HALF;
    constexpr bool kStream1 = F32OUT && !LSE && !PARTIAL;
    float r[PARTIAL ? 1 : HALF];
    int j = 0;
    bool ok = true;
    for (int i = blockIdx.x; i < items && ok; i += gridDim.x) {
      const int t = item_tile(i), m0 = tile_m0(t), n0 = tile_n0(t);
      const int row = m0 + q * 32 + lane;
      const bool live = row < p.M;
      for (int c = item_c0(i); c < item_c1(i); ++c, ++j) {
        const int b = j & 1;
        if (ok && !__all_sync(0xffffffffu, mbar_wait(tfull0 + 8 * b, (j >> 1) & 1, p.err)))
          ok = false;
        if (!ok) break;
        tc_fence_after();
        const uint32_t ta = tmem + b * BN + col0 + (uint32_t(q * 32) << 16);
        float* dst = partial && live ? p.ws + (int64_t(c) * p.M + row) * p.ldp + n0 + col0 : nullptr;
        // tcgen05.ld is warp-collective: every lane issues it, live row or not
        if (partial) {
#pragma unroll
          for (int g = 0; g < HALF / 32; ++g) {
            uint32_t v[32];
            tmem_ld32(ta + g * 32, v);
            tmem_ld_wait();
            if (dst && p.ws_v8) {
              // whole 32-byte sectors per store: half-sector stores slowed
              // the next work item's loads more (measured with a
              // clock-stamped build)
#pragma unroll
              for (int x = 0; x < 32; x += 8) st_global_v8(dst + g * 32 + x, v + x);
            } else if (dst) {
#pragma unroll
              for (int x = 0; x < 32; x += 4)
                *reinterpret_cast<float4*>(dst + g * 32 + x) =
                    make_float4(__uint_as_float(v[x]), __uint_as_float(v[x + 1]),
                                __uint_as_float(v[x + 2]), __uint_as_float(v[x + 3]));
            }
          }
        } else if (kStream1 && item_c1(i) - item_c0(i) == 1) {
          // FP32 output from one chunk: nothing to fold, so 32 columns at a
          // time go from TMEM through the warp's staging block to memory,
          // with no running sums held (the same values the fold path stores;
          // the fold path's 128 sums a thread spill on 256-column tiles)
          constexpr int W = F32OUT ? 4 : 8;
          constexpr int LPR = 32 / W, RPI = 32 / LPR;
          float* stg = staging + (warp - 2) * 32 * kStagePitch;
          const int rows = min(32, p.M - (m0 + q * 32));   // live rows of this warp
          const int sub = lane % LPR, rsub = lane / LPR;
#pragma unroll 1
          for (int blk = 0; blk < HALF / 32; ++blk) {
            uint32_t v32[32];
            tmem_ld32(ta + blk * 32, v32);
            tmem_ld_wait();
            __syncwarp();
#pragma unroll
            for (int x = 0; x < 32; ++x) stg[lane * kStagePitch + x] = __uint_as_float(v32[x]);
            __syncwarp();
            const int n = n0 + col0 + blk * 32 + sub * W;
#pragma unroll
            for (int it = 0; it < 32 / RPI; ++it) {
              const int jr = it * RPI + rsub;
              if (jr >= rows || n >= p.N) continue;
              float v[W];
#pragma unroll
              for (int e = 0; e < W; ++e) v[e] = stg[jr * kStagePitch + sub * W + e];
              const int64_t off = int64_t(m0 + q * 32 + jr) * p.ldc + n;
              if (p.vec_ok && n + W <= p.N) {
                if (F32OUT)
                  *reinterpret_cast<float4*>(static_cast<float*>(p.C) + off) =
                      make_float4(v[0], v[1], v[2], v[3]);
                else
                  *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.C) + off) =
                      make_uint4(pack_bf2(v[0], v[1]), pack_bf2(v[2], v[3]), pack_bf2(v[4], v[5]),
                                 pack_bf2(v[6], v[7]));
              } else {
                for (int e = 0; e < W && n + e < p.N; ++e) {
                  if (F32OUT)
                    static_cast<float*>(p.C)[off + e] = v[e];
                  else
                    static_cast<uint16_t*>(p.C)[off + e] = f2bf(v[e]);
                }
              }
            }
          }
        } else {
          // 16-column loads keep the running sum plus one load in registers
#pragma unroll
          for (int g = 0; g < HALF / 16; ++g) {
            uint32_t v[16];
            tmem_ld16(ta + g * 16, v);
            tmem_ld_wait();
            if (c == 0) {
#pragma unroll
              for (int x = 0; x < 16; ++x) r[g * 16 + x] = __uint_as_float(v[x]);
            } else {
#pragma unroll
              for (int x = 0; x < 16; ++x) r[g * 16 + x] = r[g * 16 + x] + __uint_as_float(v[x]);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty0 + 8 * b);
      }
      if (partial) continue;  // gemm_fold_kernel finishes the tile
      if (!ok) break;
      if (kStream1 && item_c1(i) - item_c0(i) == 1) continue;   // streamed above
      if constexpr (LSE) {
        static_assert(HALF == kLseGroup, "one 128-column group per epilogue thread");
        // the row's logits z[nb .. nb+nv) of this half tile: their max, then
        // sum exp(z - max) over four interleaved chains (x = e mod 4, x
        // ascending) added as (c0 + c1) + (c2 + c3)
        const int nb = n0 + col0, nv = min(HALF, p.N - nb);
        if (live && nv > 0) {
          float gm = -INFINITY;
#pragma unroll
          for (int x = 0; x < HALF; ++x)
            if (x < nv) gm = fmaxf(gm, r[x]);
          float cs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int x = 0; x < HALF; ++x)
            if (x < nv) cs[x & 3] += expf(r[x] - gm);
          p.lse[int64_t(row) * p.ngroups + nb / kLseGroup] =
              make_float2(gm, (cs[0] + cs[1]) + (cs[2] + cs[3]));
          const int tg = p.target[row];
          if (tg >= nb && tg < nb + nv) {
            float z = 0.f;
#pragma unroll
            for (int x = 0; x < HALF; ++x)
              if (nb + x == tg) z = r[x];
            p.zt[row] = z;
          }
        }
        continue;
      }
      // store through the warp's staging block: lane l writes its row, then
      // the warp reads it back as 16-byte row pieces (W columns per lane,
      // LPR lanes per row), so a store instruction writes RPI whole row
      // segments instead of 32 scattered pieces
      constexpr int W = F32OUT ? 4 : 8;
      constexpr int LPR = 32 / W, RPI = 32 / LPR;
      float* stg = staging + (warp - 2) * 32 * kStagePitch;
      const int rows = min(32, p.M - (m0 + q * 32));   // live rows of this warp
      const int sub = lane % LPR, rsub = lane / LPR;
#pragma unroll
      for (int blk = 0; blk < HALF / 32; ++blk) {
        __syncwarp();
#pragma unroll
        for (int x = 0; x < 32; ++x) stg[lane * kStagePitch + x] = r[blk * 32 + x];
        __syncwarp();
        const int n = n0 + col0 + blk * 32 + sub * W;
#pragma unroll
        for (int it = 0; it < 32 / RPI; ++it) {
          const int j = it * RPI + rsub;
          if (j >= rows || n >= p.N) continue;
          float v[W];
#pragma unroll
          for (int e = 0; e < W; ++e) v[e] = stg[j * kStagePitch + sub * W + e];
          const int64_t off = int64_t(m0 + q * 32 + j) * p.ldc + n;
          if (p.vec_ok && n + W <= p.N) {
            if (F32OUT)
              *reinterpret_cast<float4*>(static_cast<float*>(p.C) + off) =
                  make_float4(v[0], v[1], v[2], v[3]);
            else
              *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.C) + off) =
                  make_uint4(pack_bf2(v[0], v[1]), pack_bf2(v[2], v[3]), pack_bf2(v[4], v[5]),
                             pack_bf2(v[6], v[7]));
          } else {
            for (int e = 0; e < W && n + e < p.N; ++e) {
              if (F32OUT)
                static_cast<float*>(p.C)[off + e] = v[e];
              else
                static_cast<uint16_t*>(p.C)[off + e] = f2bf(v[e]);
            }
          }
        }
      }
    }
  }
  // the producer makes sure its copies have landed before the CTA exits
  if (warp == 0 && lane == 0) {
    for (int i = max(0, issued - S); i < issued; ++i)
      mbar_wait(full0 + 8 * (i % S), (i / S) & 1, p.err, 100000000ull);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// Partial mode, second half: every output element's chunk partials folded in
// chunk order, r = P_0, r = r + P_1, ..., rounded once.  One thread per 4
// consecutive columns of a row (coalesced reads of each chunk's rows).
template <bool F32OUT>
__global__ void __launch_bounds__(256) gemm_fold_kernel(const float* __restrict__ ws, void* C,
                                                        int64_t ldc, int M, int N, int64_t ldp,
                                                        int chunks, int vec_ok) {
  pdl_wait();  // the partials of the GEMM kernel before this one
  pdl_trigger();
  const int gpr = (N + 3) / 4;  // 4-column groups per row
  const int64_t groups = int64_t(M) * gpr;
  const int64_t cstride = int64_t(M) * ldp;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < groups;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int row = int(i / gpr), n = int(i % gpr) * 4;
    const float* src = ws + int64_t(row) * ldp + n;
    float4 v[kMaxChunks];
#pragma unroll
    for (int c = 0; c < kMaxChunks; ++c)
      if (c < chunks) v[c] = __ldcg(reinterpret_cast<const float4*>(src + c * cstride));
    float r[4] = {v[0].x, v[0].y, v[0].z, v[0].w};
#pragma unroll
    for (int c = 1; c < kMaxChunks; ++c) {
      if (c < chunks) {
        r[0] = r[0] + v[c].x;
        r[1] = r[1] + v[c].y;
        r[2] = r[2] + v[c].z;
        r[3] = r[3] + v[c].w;
      }
    }
    if (F32OUT) {
      float* dst = static_cast<float*>(C) + int64_t(row) * ldc + n;
      if (vec_ok && n + 4 <= N) {
        *reinterpret_cast<float4*>(dst) = make_float4(r[0], r[1], r[2], r[3]);
      } else {
        for (int j = 0; j < 4 && n + j < N; ++j) dst[j] = r[j];
      }
    } else {
      uint16_t* dst = static_cast<uint16_t*>(C) + int64_t(row) * ldc + n;
      if (vec_ok && n + 4 <= N) {
        *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf2(r[0], r[1]), pack_bf2(r[2], r[3]));
      } else {
        for (int j = 0; j < 4 && n + j < N; ++j) dst[j] = f2bf(r[j]);
      }
    }
  }
}

// ------------------------------------------------------------- FP8 kernel --
// Block-scaled e4m3 GEMM (per 128-wide K block: a scale per A row and one per
// 128 x 128 block of B), optionally grouped (expert g's rows
// [offs[g], offs[g+1]) of A against its weights, rows [g N, g N + N) of B).
// Persistent CTAs walk 128 x 256 tiles, the M tiles of all groups in group
// order, N tiles fastest.
// Pipeline: when K is a whole number of 128-wide blocks, a stage holds
// kpb = 2 K blocks, brought by one 3-D copy per operand (two stages of
// 96 KB; otherwise four stages of one block).  TMA moves about twice the
// bytes per SM clock with two 128-byte panels per row as with one (measured
// on GB300), and one-panel copies left the MMA waiting.
// Warps: 0 = TMA producer, 1 = MMA issuer and TMEM owner, 2..17 =
// promotion/epilogue (lane quarter = warp % 4, 64-column quarter =
// (warp - 2) / 4).  For each K block the MMA writes a fresh FP32 partial into
// one of two TMEM buffers and the epilogue warps fold it into registers as
// acc = fma(sa * sb, partial, acc), blocks in ascending order, while the MMA
// fills the other buffer; a tile's store overlaps the next tile's first
// MMAs.  64 running sums a thread keep the promotion loop in registers (with
// 128, in eight warps, it spilled to local memory).
template <int BN>
__global__ void __launch_bounds__(Fp8Cfg<BN>::THREADS, 1)
    gemm_fp8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    uint16_t* C, int64_t ldc, int M, int N, int K, const float* __restrict__ sa,
                    int64_t ld_sa, const float* __restrict__ sb, const int32_t* __restrict__ offs,
                    int groups, int vec_ok, int kpb, int* err) {
  using Cfg = Fp8Cfg<BN>;
  const int S = Cfg::BLOCKS / kpb;                    // stages of kpb K blocks
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sA = smem;                                 // [S][kpb] A blocks
  uint8_t* sB = smem + Cfg::BLOCKS * Cfg::A_BYTES;    // [S][kpb] B blocks
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::BLOCKS * Cfg::STAGE);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * Cfg::BLOCKS + 4);
  int* tpre = reinterpret_cast<int*>(tmem_slot + 4);   // [groups + 1]: M tiles before group g
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + Cfg::BLOCKS);
  const uint32_t tfull0 = smem_u32(bars + 2 * Cfg::BLOCKS);
  const uint32_t tempty0 = smem_u32(bars + 2 * Cfg::BLOCKS + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KB = (K + Cfg::BK - 1) / Cfg::BK;
  const int NB = (N + 127) / 128;
  const int tiles_n = (N + BN - 1) / BN;
  const int a_stage = kpb * Cfg::A_BYTES, b_stage = kpb * Cfg::B_BYTES;

  if (warp == 0) {   // tile prefix over the groups
    int run = 0;
    for (int g0 = 0; g0 < groups; g0 += 32) {
      const int gg = g0 + lane;
      int nt = 0;
      if (gg < groups)
        nt = groups > 1 ? (max(offs[gg + 1] - offs[gg], 0) + BM - 1) / BM : (M + BM - 1) / BM;
      int incl = nt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (gg < groups) tpre[gg + 1] = run + incl;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) tpre[0] = 0;
  }
  if (threadIdx.x == 32) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int j = 0; j < 2; ++j) {
      mbar_init(tfull0 + 8 * j, 1);
      mbar_init(tempty0 + 8 * j, Cfg::EPI_WARPS);
    }
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int items = tpre[groups] * tiles_n;
  // M tile mt -> its group (the last group whose tiles start at or before
  // mt: empty groups are skipped), first row and row bound
  auto locate = [&](int mt, int& g, int& m0, int& m_end) {
    int lo = 0, hi = groups - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (tpre[mid] <= mt) lo = mid; else hi = mid - 1;
    }
    g = lo;
    m0 = (groups > 1 ? offs[g] : 0) + (mt - tpre[g]) * BM;
    m_end = groups > 1 ? offs[g + 1] : M;
  };

  int issued = 0;
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    bool ok = true;
    for (int t = blockIdx.x; t < items && ok; t += gridDim.x) {
      int g, m0, m_end;
      locate(t / tiles_n, g, m0, m_end);
      const int n0 = (t % tiles_n) * BN;
      for (int kb = 0; kb < KB; kb += kpb) {
        const int s = issued % S;
        if (issued >= S && !mbar_wait(empty0 + 8 * s, ((issued / S) - 1) & 1, err)) {
          ok = false;
          break;
        }
        // a 3-D copy past the last K block fills zeros and counts its bytes
        mbar_expect_tx(full0 + 8 * s, uint32_t(a_stage + b_stage));
        const uint32_t fb = full0 + 8 * s;
        if (kpb == 2) {
          tma_load_3d(smem_u32(sA + s * a_stage), &tmA, fb, 0, m0, kb);
          tma_load_3d(smem_u32(sB + s * b_stage), &tmB, fb, 0, g * N + n0, kb);
        } else {
          tma_load_2d(smem_u32(sA + s * a_stage), &tmA, fb, kb * Cfg::BK, m0);
          tma_load_2d(smem_u32(sB + s * b_stage), &tmB, fb, kb * Cfg::BK, g * N + n0);
        }
        ++issued;
      }
    }
  } else if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc = idesc_mma(0u, BM, BN);
    int it = 0, st = 0;   // K blocks, stages consumed
    bool ok = true;
    for (int t = blockIdx.x; t < items && ok; t += gridDim.x) {
      for (int kb = 0; kb < KB && ok; kb += kpb, ++st) {
        const int s = st % S;
        if (!mbar_wait(full0 + 8 * s, (st / S) & 1, err)) {
          ok = false;
          break;
        }
        for (int b = 0; b < kpb && kb + b < KB; ++b, ++it) {
          const int j = it & 1;
          if (it >= 2 && !mbar_wait(tempty0 + 8 * j, ((it >> 1) - 1) & 1, err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + s * a_stage + b * Cfg::A_BYTES);
          const uint32_t b0 = smem_u32(sB + s * b_stage + b * Cfg::B_BYTES);
#pragma unroll
          for (int kk = 0; kk < Cfg::BK / 32; ++kk)
            umma_f8(tmem + j * BN, sdesc_k_sw128(a0 + kk * 32), sdesc_k_sw128(b0 + kk * 32), idesc,
                    kk != 0 ? 1u : 0u);
          umma_commit(tfull0 + 8 * j);
        }
        umma_commit(empty0 + 8 * s);
      }
    }
  } else if (warp >= 2) {
    const int q = warp & 3, cq = (warp - 2) >> 2;
    int it = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < items && ok; t += gridDim.x) {
      int g, m0, m_end;
      locate(t / tiles_n, g, m0, m_end);
      const int nh = (t % tiles_n) * BN + cq * 64;   // this warp's first column
      const int row = m0 + q * 32 + lane;
      const bool live = row < m_end && row < M;
      const bool hlive = nh < N;
      const float* sbh = sb + (int64_t(g) * NB + (hlive ? nh / 128 : 0)) * KB;
      float acc[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) acc[c] = 0.f;
      for (int kb = 0; kb < KB; ++kb, ++it) {
        const int j = it & 1;
        const float scale = (live ? sa[int64_t(row) * ld_sa + kb] : 0.f) * (hlive ? sbh[kb] : 0.f);
        if (!__all_sync(0xffffffffu, mbar_wait(tfull0 + 8 * j, (it >> 1) & 1, err))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tb = tmem + j * BN + cq * 64 + (uint32_t(q * 32) << 16);
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 16) {
          uint32_t r[16];
          tmem_ld16(tb + c0, r);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 16; ++c) acc[c0 + c] = fmaf(scale, __uint_as_float(r[c]), acc[c0 + c]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty0 + 8 * j);
      }
      if (ok && live && hlive) {
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 32) {
          uint32_t r[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) r[c] = __float_as_uint(acc[c0 + c]);
          if (nh + c0 < N) store_row32<false>(C, ldc, row, nh + c0, N, r, vec_ok != 0);
        }
      }
    }
  }
  if (warp == 0 && lane == 0) {
    for (int i = max(0, issued - S); i < issued; ++i)
      mbar_wait(full0 + 8 * (i % S), (i / S) & 1, err, 100000000ull);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, Cfg::TMEM_COLS);
}

// ------------------------------------------------------- NVFP4 weights --
// Partial-mode GEMM whose B operand is stored as NVFP4: packed e2m1 codes
// [N, K/2] (element 2i in the low nibble of byte i) and one e4m3 scale per 16
// elements [N, K/16], global scale 1.  Each K block of 64 arrives as 4 KB of
// codes and the 16-byte scale group holding its four scales; converter warps
// decode it to bf16 (e2m1 x scale is exact in bf16) straight into TMEM, and
// the MMA runs with the operands swapped: the decoded weight tile (128 weight
// rows in the 128 TMEM lanes) is the A operand, the few activation rows (the
// TMA box in shared memory) the B operand, N = the box's rows.  D'[n][m] is
// the bf16 path's D[m][n]: tcgen05 is operand-symmetric (measured on GB300:
// every element of C1 = A.B^T equals C2^T = (B.A^T)^T), and the K steps run
// in the same order, so every partial, and so every output, has the bits of
// the bf16 GEMM on the decoded weights.  HBM reads 0.5625 bytes per weight
// instead of 2.
// A ring of R raw stages and kFp4Dec decoded tiles in TMEM (32 columns
// each).  A raw stage holds kFp4Sub = 4 K blocks: the codes as one box of
// 128-byte rows, the two 16-byte scale groups around them as one box of
// 32-byte rows, the activations as one 3-D box of four 64-wide panels.  TMA
// moves a few box rows per SM clock whatever their width (measured on
// GB300), so one K block per stage, in 32- and 16-byte rows, ran at about a
// fifth of the HBM rate.
// Warps: 0 = TMA producer, 1 = MMA issuer and TMEM owner, 2..17 = converters
// in four groups of four (lane quarter = warp % 4): group g decodes the K
// blocks whose running index is g mod 4 into decoded tile g, each thread the
// 64 elements of one weight row as 32 columns, so four K blocks are decoded
// at once (one group at a time left the MMA waiting on the store latency);
// 18..21 = epilogue (TMEM lane quarters: one weight row a thread, every
// activation row of the box).  A converter looks each code byte (two elements) up in a
// 256-entry table of bf16 pairs at scale 1 and multiplies the pair by the
// block scale in bf16 (exact: the product has at most 6 significant bits).
// The table is held in 32 interleaved copies so that lane L always reads
// bank L (one shared copy cost about 340 bank conflicts per K block).
constexpr int kFp4Sub = 4;                // K blocks per raw stage
constexpr int kFp4CodeBytes = 128 * 128;  // a stage: 128 rows x 256 codes
constexpr int kFp4SclBytes = 128 * 32;    // a stage: 128 rows x two 16-scale groups (at most)
constexpr int kFp4Conv = 16;              // converter warps: four groups of four
constexpr int kFp4Threads = 64 + 32 * kFp4Conv + 128;
constexpr int kFp4Dec = 4;                // decoded tiles in TMEM, one per converter group
constexpr int kFp4MaxRaw = 32;            // raw stages at most
constexpr uint32_t kFp4DecCol = 0;        // TMEM: decoded tiles at columns [0, 128)
constexpr uint32_t kFp4AccCol = 128;      // two accumulators of <= 64 columns from 128

size_t fp4_smem_bytes(int raw, int m_box) {
  return 1024 + size_t(raw) * (kFp4Sub * m_box * 128 + kFp4CodeBytes + kFp4SclBytes) +
         (2 * kFp4MaxRaw + 2 * kFp4Dec + 4) * 8 + 16 + 256 * 32 * 4;
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, __nv_bfloat162 b) {
  const __nv_bfloat162 r = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&a), b);
  return *reinterpret_cast<const uint32_t*>(&r);
}

__global__ void __launch_bounds__(kFp4Threads, 1)
    gemm_nvfp4_kernel(const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmC,
                      const __grid_constant__ CUtensorMap tmS, const GemmArgs p) {
  constexpr int BN = 128;                 // weight rows per tile (the MMA's M)
  constexpr uint32_t kTmemCols = 256;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int R = p.stages;                                        // raw stages
  const int a_blk = p.m_box * 128, a_stage = kFp4Sub * a_blk;
  const int sw = min(32, p.K / 16);                              // scale bytes a row per stage
  uint8_t* sA = smem;                                            // [R][kFp4Sub] activation boxes
  uint8_t* sCode = sA + R * a_stage;                             // [R] raw codes
  uint8_t* sScl = sCode + R * kFp4CodeBytes;                     // [R] raw scale groups
  uint64_t* bars = reinterpret_cast<uint64_t*>(sScl + R * kFp4SclBytes);
  // full[r]: activations, codes and scales of raw stage r landed.  empty[r]:
  // the MMA (activations) and every converter warp (codes) are done with it.
  // dfull[b] / dempty[b]: decoded tile b written / read by the MMA.
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kFp4MaxRaw);
  const uint32_t dfull0 = smem_u32(bars + 2 * kFp4MaxRaw);
  const uint32_t dempty0 = smem_u32(bars + 2 * kFp4MaxRaw + kFp4Dec);
  const uint32_t tfull0 = smem_u32(bars + 2 * kFp4MaxRaw + 2 * kFp4Dec);
  const uint32_t tempty0 = tfull0 + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kFp4MaxRaw + 2 * kFp4Dec + 4);
  uint32_t* lut = tmem_slot + 4;   // [256][32]: byte (two codes) -> bf16 pair at scale 1

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KB = (p.K + 63) / 64;
  const int chunks = (KB + p.kc_blocks - 1) / p.kc_blocks;
  const int tiles_m = (p.M + BM - 1) / BM, tiles_n = (p.N + BN - 1) / BN;
  const int items = tiles_m * tiles_n * chunks;
  auto tile_m0 = [&](int t) { return (t % tiles_m) * BM; };
  auto tile_n0 = [&](int t) { return (t / tiles_m) * BN; };
  for (int e = threadIdx.x; e < 256 * 32; e += blockDim.x) {
    const __half2_raw hr = __nv_cvt_fp4x2_to_halfraw2(__nv_fp4x2_storage_t(e >> 5), __NV_E2M1);
    const float2 f = __half22float2(__half2(hr));
    lut[e] = pack_bf2(f.x, f.y);
  }

  if (threadIdx.x == 0) {
    for (int r = 0; r < R; ++r) {
      mbar_init(full0 + 8 * r, 1);
      mbar_init(empty0 + 8 * r, 1 + kFp4Conv);
    }
    for (int b = 0; b < kFp4Dec; ++b) {
      mbar_init(dfull0 + 8 * b, 4);        // the four warps of converter group b
      mbar_init(dempty0 + 8 * b, 1);
    }
    for (int j = 0; j < 2; ++j) {
      mbar_init(tfull0 + 8 * j, 1);
      mbar_init(tempty0 + 8 * j, 4);
    }
    fence_barrier_init();
  }
  __syncwarp();
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_trigger();

  int issued = 0;
  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmC);
      tma_prefetch_desc(&tmS);
      // boxes past the end of K fill zeros and count their bytes
      const uint32_t tx = uint32_t(a_stage + kFp4CodeBytes + 128 * sw);
      auto load_b = [&](int r, int kb0, int n0) {
        mbar_expect_tx(full0 + 8 * r, tx);
        tma_load_2d(smem_u32(sCode + r * kFp4CodeBytes), &tmC, full0 + 8 * r, kb0 * 32, n0);
        tma_load_2d(smem_u32(sScl + r * kFp4SclBytes), &tmS, full0 + 8 * r, (kb0 >> 2) * 16, n0);
      };
      // weights of the first stages before waiting for the previous kernel
      int pre = 0;
      if (blockIdx.x < items) {
        const int i = blockIdx.x, t = i / chunks, c = i % chunks;
        const int kb_lo = c * p.kc_blocks, kb_hi = min(KB, kb_lo + p.kc_blocks);
        for (int kb0 = kb_lo; kb0 < kb_hi && pre < R; kb0 += kFp4Sub, ++pre)
          load_b(pre, kb0, tile_n0(t));
      }
      pdl_wait();
      bool ok = true;
      for (int i = blockIdx.x; i < items && ok; i += gridDim.x) {
        const int t = i / chunks, c = i % chunks, m0 = tile_m0(t), n0 = tile_n0(t);
        const int kb1 = min(KB, (c + 1) * p.kc_blocks);
        for (int kb0 = c * p.kc_blocks; kb0 < kb1; kb0 += kFp4Sub) {
          const int r = issued % R;
          if (issued >= pre) {
            if (issued >= R && !mbar_wait(empty0 + 8 * r, ((issued / R) - 1) & 1, p.err)) {
              ok = false;
              break;
            }
            load_b(r, kb0, n0);
          }
          tma_load_3d(smem_u32(sA + r * a_stage), &tmA, full0 + 8 * r, 0, m0, kb0);
          ++issued;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // D'[128 weight rows x m_box activation rows]: A from TMEM, B K-major
      const uint32_t idesc = idesc_mma(1u, BN, p.m_box);
      int it = 0, st = 0, j = 0;   // K blocks, raw stages, work items
      bool ok = true;
      for (int i = blockIdx.x; i < items && ok; i += gridDim.x, ++j) {
        const int c = i % chunks, tb = j & 1;
        if (j >= 2 && !mbar_wait(tempty0 + 8 * tb, ((j >> 1) - 1) & 1, p.err)) break;
        tc_fence_after();
        const uint32_t dt = tmem + kFp4AccCol + tb * 64;
        const int kb_lo = c * p.kc_blocks, kb1 = min(KB, kb_lo + p.kc_blocks);
        for (int kb0 = kb_lo; kb0 < kb1 && ok; kb0 += kFp4Sub, ++st) {
          const int r = st % R;
          if (!mbar_wait(full0 + 8 * r, (st / R) & 1, p.err)) {
            ok = false;
            break;
          }
          for (int kb = kb0; kb < min(kb1, kb0 + kFp4Sub); ++kb, ++it) {
            const int b = it % kFp4Dec;
            if (!mbar_wait(dfull0 + 8 * b, (it / kFp4Dec) & 1, p.err)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a0 = smem_u32(sA + r * a_stage + (kb - kb0) * a_blk);
            const uint32_t w0 = tmem + kFp4DecCol + b * 32;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_f16_ts(dt, w0 + kk * 8, sdesc_k_sw128(a0 + kk * 32), idesc,
                          (kb != kb_lo || kk != 0) ? 1u : 0u);
            umma_commit(dempty0 + 8 * b);
          }
          umma_commit(empty0 + 8 * r);
        }
        if (ok) umma_commit(tfull0 + 8 * tb);
      }
    }
  } else if (warp < 2 + kFp4Conv) {
    // ---------------------------------------------------------- decode --
    // thread: weight row 32 q + lane of the tile; group grp: the K blocks
    // whose running index is grp mod 4, into decoded tile grp
    const int q = warp & 3, grp = (warp - 2) >> 2;
    const int rw = q * 32 + lane;
    const uint32_t dst = tmem + (uint32_t(q * 32) << 16) + kFp4DecCol + grp * 32;
    int it = 0, st = 0;
    bool ok = true;
    for (int i = blockIdx.x; i < items && ok; i += gridDim.x) {
      const int c = i % chunks;
      const int kb1 = min(KB, (c + 1) * p.kc_blocks);
      for (int kb0 = c * p.kc_blocks; kb0 < kb1 && ok; kb0 += kFp4Sub, ++st) {
        const int r = st % R;
        if (!__all_sync(0xffffffffu, mbar_wait(full0 + 8 * r, (st / R) & 1, p.err))) {
          ok = false;
          break;
        }
        for (int kb = kb0; kb < min(kb1, kb0 + kFp4Sub); ++kb, ++it) {
          if (it % kFp4Dec != grp) continue;
          if (it >= kFp4Dec &&
              !__all_sync(0xffffffffu, mbar_wait(dempty0 + 8 * grp, ((it / kFp4Dec) - 1) & 1, p.err))) {
            ok = false;
            break;
          }
          tc_fence_after();
          // codes land 128-byte swizzled (16-byte chunk j of row r at j ^ (r % 8)):
          // a warp's 32 rows then spread over every bank (unswizzled, all 32
          // lanes of a 16-byte load hit the same four banks)
          const uint8_t* crow = sCode + r * kFp4CodeBytes + rw * 128;
          const int j0 = 2 * (kb - kb0), sx = rw & 7;
          const uint4 c0 = *reinterpret_cast<const uint4*>(crow + ((j0 ^ sx) << 4));
          const uint4 c1 = *reinterpret_cast<const uint4*>(crow + (((j0 + 1) ^ sx) << 4));
          // the stage's scale row starts at group (kb0 >> 2): block kb's four
          // scales sit (kb - 4 (kb0 >> 2)) * 4 bytes in
          const uint32_t sc4 = *reinterpret_cast<const uint32_t*>(
              sScl + r * kFp4SclBytes + rw * sw + (kb - 4 * (kb0 >> 2)) * 4);
          const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
          const uint32_t* lt = lut + lane;        // this lane's copy: bank = lane
          uint32_t o[32];
#pragma unroll
          for (int g = 0; g < 4; ++g) {           // 16 elements (two words) per e4m3 scale
            const float sf = __half2float(__ushort_as_half(
                __nv_cvt_fp8_to_halfraw(__nv_fp8_storage_t((sc4 >> (8 * g)) & 0xFFu), __NV_E4M3).x));
            const __nv_bfloat162 s2 = __floats2bfloat162_rn(sf, sf);   // e4m3 is exact in bf16
#pragma unroll
            for (int wi = 2 * g; wi < 2 * g + 2; ++wi)   // 8 elements (4 columns) per word
#pragma unroll
              for (int by = 0; by < 4; ++by)
                o[wi * 4 + by] = bf16x2_mul(lt[((w[wi] >> (8 * by)) & 0xFFu) << 5], s2);
          }
          tmem_st32(dst, o);
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(dfull0 + 8 * grp);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * r);   // this warp is done with raw stage r
      }
    }
  } else {
    // -------------------------------------------------------- epilogue --
    // thread: weight row n0 + 32 q + lane; D' columns = activation rows
    const int q = warp & 3;
    int j = 0;
    bool ok = true;
    for (int i = blockIdx.x; i < items && ok; i += gridDim.x, ++j) {
      const int t = i / chunks, c = i % chunks, m0 = tile_m0(t), n0 = tile_n0(t);
      const int n = n0 + q * 32 + lane;
      const int tb = j & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(tfull0 + 8 * tb, (j >> 1) & 1, p.err))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t ta = tmem + kFp4AccCol + tb * 64 + (uint32_t(q * 32) << 16);
      float* dst = p.ws + (int64_t(c) * p.M + m0) * p.ldp + n;
      const int rows = min(p.m_box, p.M - m0);
      for (int g0 = 0; g0 < p.m_box; g0 += 16) {
        uint32_t v[16];
        tmem_ld16(ta + g0, v);
        tmem_ld_wait();
        if (n < p.N) {
#pragma unroll
          for (int x = 0; x < 16; ++x)
            if (g0 + x < rows) dst[int64_t(g0 + x) * p.ldp] = __uint_as_float(v[x]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty0 + 8 * tb);
    }
  }
  // the producer makes sure its copies have landed before the CTA exits
  if (warp == 0 && lane == 0) {
    for (int i = max(0, issued - R); i < issued; ++i)
      mbar_wait(full0 + 8 * (i % R), (i / R) & 1, p.err, 100000000ull);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------- host --
// 2-D K-major tensor map: dims {K, rows}, box {box_k, box_rows}, 128B swizzle.
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, int elem_bytes, const void* base,
              int64_t K, int64_t rows, int64_t ld, int box_k, int box_rows, bool swizzle = true) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {cuuint64_t(K), cuuint64_t(rows)};
  cuuint64_t strides[1] = {cuuint64_t(ld * elem_bytes)};
  cuuint32_t box[2] = {cuuint32_t(box_k), cuuint32_t(box_rows)};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// A bf16 K-major operand [rows, K] as a 3-D tensor {64, rows, K/64}: a box
// {64, box_rows, 2} brings two consecutive K blocks in one copy, landing as
// [block][row][128 B] with 128-byte swizzling (two ordinary stages back to
// back).  Measured on GB300, one producer thread moves about 25 bytes per SM
// clock in 2-D boxes of 128-byte rows, whatever the pipeline depth, and
// twice that when each row brings two adjacent K blocks.  K % 64 == 0, so no
// block reads past a row.
bool make_map2k(CUtensorMap* m, const void* base, int64_t K, int64_t rows, int64_t ld,
                int box_rows) {
  auto fn = tensor_map_encoder();
  if (!fn || K % 64 != 0) return false;
  cuuint64_t dims[3] = {64, cuuint64_t(rows), cuuint64_t(K / 64)};
  cuuint64_t strides[2] = {cuuint64_t(ld * 2), 128};
  cuuint32_t box[3] = {64, cuuint32_t(box_rows), 2};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A K-major operand [rows, K] as a 3-D tensor {panel, rows, K / panel}
// (elements): a box {panel, box_rows, panels} brings that many consecutive K
// blocks, landing as [block][row][panel] with 128-byte swizzling.
// K % panel == 0.
bool make_map_panels(CUtensorMap* m, CUtensorMapDataType dt, int elem_bytes, const void* base,
                     int64_t K, int64_t rows, int64_t ld, int panel, int box_rows,
                     int panels = 2) {
  auto fn = tensor_map_encoder();
  if (!fn || K % panel != 0) return false;
  cuuint64_t dims[3] = {cuuint64_t(panel), cuuint64_t(rows), cuuint64_t(K / panel)};
  cuuint64_t strides[2] = {cuuint64_t(ld * elem_bytes), cuuint64_t(panel * elem_bytes)};
  cuuint32_t box[3] = {cuuint32_t(panel), cuuint32_t(box_rows), cuuint32_t(panels)};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// FP8: two K blocks of 128 per pipeline stage when K is a whole number of
// blocks (BIV_GEMM_KPB=1 keeps one; the tests check that neither changes a bit).
int fp8_kpb_for(int K) {
  const char* e = getenv("BIV_GEMM_KPB");
  if (e && atoi(e) == 1) return 1;
  return (K % 128 == 0 && K >= 256) ? 2 : 1;
}

struct Plan {
  int bn = 256;
  int kpb = 1;        // K blocks per pipeline stage
  int kc_blocks = 1;  // K blocks (of 64) per chunk
  int chunks = 1;
  bool partial = false;
  int m_box = BM;     // rows of the A TMA box
  int stages = 4;
  int64_t tiles = 0;
  int64_t ldp = 0;    // partial row pitch
  size_t ws_bytes = 0;
};

constexpr size_t kSmemBudget = 227 * 1024;  // the per-CTA maximum
// Partial mode leaves 32 KB of the SM's shared memory free, so that with PDL
// the next kernel's (small) CTAs can start beside the GEMM's.
constexpr size_t kSmemBudgetPartial = kSmemBudget - 32 * 1024;
// At most this many rows, partial mode is taken whenever 128-column tiles
// leave an SM idle (measured on GB300, 12288 x 2048 weights: M = 1 and 64 ran
// 14.5 and 16.6 us as partials, 17.2 and 18.2 us folded in 96 CTAs; at M = 128
// the partials' own traffic made folding faster)
constexpr int kPartialRows = 64;
// The wide tile of the register-fold mode (measured on GB300 at M = 16384:
// 256 columns beat 192 although each epilogue thread then keeps 128 running
// sums and spills a few registers).
constexpr int kWideN = 256;

// Test overrides: BIV_GEMM_TILE_N=64|128|256 forces the tile width and
// BIV_GEMM_FOLD=cta|partial the fold mode; the tests use them to check that
// neither choice changes a result bit.
int env_tile_n() {
  const char* e = getenv("BIV_GEMM_TILE_N");
  const int bn = e ? atoi(e) : 0;
  return (bn == 64 || bn == 128 || bn == 192 || bn == 256) ? bn : 0;
}
int env_fold() {  // 0 = planner, 1 = fold in the CTA, 2 = partials
  const char* e = getenv("BIV_GEMM_FOLD");
  if (!e) return 0;
  if (!strcmp(e, "cta")) return 1;
  if (!strcmp(e, "partial")) return 2;
  return 0;
}

// Two K blocks per stage when K is a whole number of blocks (BIV_GEMM_KPB=1
// keeps one; the tests check that neither changes a bit).
int kpb_for(int K) {
  const char* e = getenv("BIV_GEMM_KPB");
  if (e && atoi(e) == 1) return 1;
  return (K % 64 == 0 && K >= 128) ? 2 : 1;
}

// Tensor maps of a bf16 call: 3-D two-block boxes when the plan takes them.
bool make_bf16_maps(CUtensorMap* ta, CUtensorMap* tb, const void* A, int64_t lda, int64_t M,
                    const void* B, int64_t ldb, int64_t N, int64_t K, const Plan& p) {
  if (p.kpb == 2)
    return make_map2k(ta, A, K, M, lda, p.m_box) && make_map2k(tb, B, K, N, ldb, p.bn);
  return make_map(ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A, K, M, lda, 64, p.m_box) &&
         make_map(tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, K, N, ldb, 64, p.bn);
}

// INVARIANT: K cut into chunks of max(8, ceil(KB/8)) blocks for every M; the
// tile width and the fold mode follow M (neither changes a bit).
// FAST (the batch-dependent comparator): no chunking for large M, and for
// small M a K split sized to fill the GPU.
Plan plan_bf16(const biv_gemm_desc& d) {
  Plan p;
  const int KB = (d.K + 63) / 64;
  const int sms = sm_count() > 0 ? sm_count() : 148;
  const int64_t tiles_m = (d.M + BM - 1) / BM;
  p.m_box = d.M <= BM ? std::max(16, (d.M + 15) / 16 * 16) : BM;
  const int64_t tiles_wide = int64_t((d.N + kWideN - 1) / kWideN) * tiles_m;
  const int64_t tiles128 = int64_t((d.N + 127) / 128) * tiles_m;
  const bool wide = tiles_wide >= sms;   // enough 128 x kWideN tiles to fill the GPU
  // partials when whole 128-column tiles leave most SMs idle, and for the
  // few-row (weight-streaming) shapes whenever they leave any SM idle
  bool partial = !wide && (tiles128 * 2 <= sms || (d.M <= kPartialRows && tiles128 < sms));
  if (d.mode == BIV_MODE_INVARIANT) {
    p.kc_blocks = std::max(kMinChunkBlocks, (KB + kMaxChunks - 1) / kMaxChunks);
  } else if (partial) {
    const int64_t want = (sms + tiles128 - 1) / tiles128;
    const int splits = int(std::max<int64_t>(1, std::min<int64_t>({want, int64_t(kMaxChunks), KB / 2})));
    p.kc_blocks = (KB + splits - 1) / splits;
  } else {
    p.kc_blocks = KB;
  }
  p.chunks = (KB + p.kc_blocks - 1) / p.kc_blocks;
  if (wide) {
    p.bn = kWideN;
  } else if (partial && p.chunks > 1) {
    p.bn = 128;
  } else {
    // fold mode below one full wave of wide tiles: the width with the least
    // A + B rows streamed by the busiest CTA (rounds of tiles x rows per tile)
    int64_t best = -1;
    for (const int bn : {128, 192, 256}) {
      const int64_t t = int64_t((d.N + bn - 1) / bn) * tiles_m;
      const int64_t cost = (t + sms - 1) / sms * (p.m_box + bn);
      if (best < 0 || cost < best) {
        best = cost;
        p.bn = bn;
      }
    }
  }
  if (const int bn = env_tile_n()) p.bn = bn;
  if (const int f = env_fold()) partial = f == 2;
  p.tiles = int64_t((d.N + p.bn - 1) / p.bn) * tiles_m;
  // partial mode: more than one chunk, tiles of at most 128 columns
  p.partial = partial && p.chunks > 1 && p.bn <= 128;
  p.kpb = kpb_for(d.K);
  const int a_stage = p.m_box * 128 * p.kpb, b_stage = p.bn * 128 * p.kpb;
  const size_t fixed = GemmSmem<128>::bytes(0, p.m_box, !p.partial);
  const size_t budget = p.partial ? kSmemBudgetPartial : kSmemBudget;
  p.stages = int(std::min<size_t>(kMaxStages, (budget - fixed) / (a_stage + b_stage)));
  p.ldp = int64_t((d.N + p.bn - 1) / p.bn) * p.bn;
  if (p.partial) p.ws_bytes = size_t(p.chunks) * d.M * p.ldp * sizeof(float);
  return p;
}

template <int BN, bool F32OUT>
biv_status launch_bf16(const CUtensorMap& ta, const CUtensorMap& tb, const biv_gemm_desc& d,
                       const Plan& pl, void* ws, cudaStream_t s, bool b_after_wait) {
  // partial mode writes FP32 partials whatever C's type: one instantiation
  constexpr bool kPartialOk = BN <= 128;
  auto kern = (kPartialOk && pl.partial) ? gemm_bf16_kernel<BN, false, kPartialOk>
                                         : gemm_bf16_kernel<BN, F32OUT, false>;
  static bool attr[2] = {false, false};
  if (!attr[pl.partial]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(kSmemBudget)) != cudaSuccess)
      return set_error(BIV_ERR_CUDA, "gemm: cannot set shared memory size");
    attr[pl.partial] = true;
  }
  const int eb = F32OUT ? 4 : 2;
  GemmArgs a;
  a.C = d.C;
  a.ldc = d.ldc;
  a.M = d.M;
  a.N = d.N;
  a.K = d.K;
  a.kc_blocks = pl.kc_blocks;
  a.m_box = pl.m_box;
  a.stages = pl.stages;
  a.partial = pl.partial ? 1 : 0;
  a.ws = pl.partial ? static_cast<float*>(ws) : nullptr;
  a.ws_v8 = pl.partial && (reinterpret_cast<uintptr_t>(ws) & 31) == 0;
  a.ldp = pl.ldp;
  a.vec_ok = aligned16(d.C) && (d.ldc * eb) % 16 == 0;
  a.n_fastest = !pl.partial && d.N <= d.M;
  a.b_after_wait = b_after_wait ? 1 : 0;
  a.kpb = pl.kpb;
  a.err = device_error_word();
  const int64_t items = pl.partial ? pl.tiles * pl.chunks : pl.tiles;
  const int sms = sm_count() > 0 ? sm_count() : 148;
  const int grid = int(std::min<int64_t>(items, sms));
  const size_t smem = GemmSmem<BN>::bytes(pl.stages, pl.m_box, !pl.partial, pl.kpb);
  launch_pdl(kern, grid, kGemmThreads, smem, s, ta, tb, a);
  biv_status st = check_launch("gemm_bf16");
  if (st != BIV_OK || !pl.partial || d.defer_fold) return st;
  const int64_t groups = int64_t(d.M) * ((d.N + 3) / 4);
  const int blocks = int(std::min<int64_t>((groups + 255) / 256, int64_t(sms) * 8));
  launch_pdl(gemm_fold_kernel<F32OUT>, blocks, 256, 0, s, static_cast<const float*>(ws), d.C,
             d.ldc, d.M, d.N, pl.ldp, pl.chunks, a.vec_ok);
  return check_launch("gemm_fold");
}

template <bool F32OUT>
biv_status dispatch_bf16(const CUtensorMap& ta, const CUtensorMap& tb, const biv_gemm_desc& d,
                         const Plan& p, void* ws, cudaStream_t s, bool b_after_wait = false) {
  switch (p.bn) {
    case 256: return launch_bf16<256, F32OUT>(ta, tb, d, p, ws, s, b_after_wait);
    case 192: return launch_bf16<192, F32OUT>(ta, tb, d, p, ws, s, b_after_wait);
    case 128: return launch_bf16<128, F32OUT>(ta, tb, d, p, ws, s, b_after_wait);
    default: return launch_bf16<64, F32OUT>(ta, tb, d, p, ws, s, b_after_wait);
  }
}

template <int BN>
biv_status launch_fp8(const CUtensorMap& ta, const CUtensorMap& tb, const biv_gemm_desc& d,
                      int kpb, cudaStream_t s) {
  using Cfg = Fp8Cfg<BN>;
  auto kern = gemm_fp8_kernel<BN>;
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM) !=
        cudaSuccess)
      return set_error(BIV_ERR_CUDA, "gemm_fp8: cannot set shared memory size");
    attr = true;
  }
  const int groups = d.groups > 1 ? d.groups : 1;
  const int vec_ok = aligned16(d.C) && (d.ldc * 2) % 16 == 0;
  // persistent grid: at most one CTA per SM, no more than the tiles there
  // can be (each group rounds its rows up to whole tiles)
  const int64_t tiles_m = (d.M + BM - 1) / BM + (groups > 1 ? groups : 0);
  const int64_t items = tiles_m * ((d.N + BN - 1) / BN);
  const int sms = sm_count() > 0 ? sm_count() : 148;
  const int grid = int(std::max<int64_t>(1, std::min<int64_t>(items, sms)));
  kern<<<grid, Cfg::THREADS, Cfg::SMEM, s>>>(ta, tb, static_cast<uint16_t*>(d.C), d.ldc, d.M, d.N,
                                             d.K, d.sa, d.ld_sa, d.sb, d.group_offsets, groups,
                                             vec_ok, kpb, device_error_word());
  return check_launch("gemm_fp8");
}

biv_status validate(const biv_gemm_desc* d) {
  BIV_REQUIRE(d, "gemm: null descriptor");
  BIV_REQUIRE(d->M >= 0 && d->N > 0 && d->K > 0, "gemm: bad sizes M=%d N=%d K=%d", d->M, d->N, d->K);
  BIV_REQUIRE(d->M <= 65535 * 64 && d->N < (1 << 24) && d->K < (1 << 24), "gemm: size too large");
  BIV_REQUIRE(d->mode == BIV_MODE_INVARIANT || d->mode == BIV_MODE_FAST, "gemm: bad mode");
  const bool bf = d->a_dtype == BIV_BF16 && d->b_dtype == BIV_BF16;
  const bool f8 = d->a_dtype == BIV_E4M3 && d->b_dtype == BIV_E4M3;
  if (!bf && !f8) return set_error(BIV_ERR_UNSUPPORTED, "gemm: A/B dtypes must both be bf16 or both e4m3");
  const int eb = bf ? 2 : 1;
  BIV_REQUIRE((int64_t(d->K) * eb) % 16 == 0, "gemm: K*elem_size must be a multiple of 16 (K=%d)", d->K);
  BIV_REQUIRE(aligned16(d->A) && aligned16(d->B), "gemm: A and B must be 16-byte aligned");
  BIV_REQUIRE(d->lda >= d->K && d->ldb >= d->K && (d->lda * eb) % 16 == 0 && (d->ldb * eb) % 16 == 0,
              "gemm: lda/ldb must be >= K and keep rows 16-byte aligned");
  BIV_REQUIRE(d->C && d->ldc >= d->N, "gemm: bad C / ldc");
  if (bf) {
    if (d->c_dtype != BIV_BF16 && d->c_dtype != BIV_F32)
      return set_error(BIV_ERR_UNSUPPORTED, "gemm: bf16 GEMM writes bf16 or f32");
    if (d->groups > 1) return set_error(BIV_ERR_UNSUPPORTED, "gemm: grouped bf16 not supported");
  } else {
    if (d->c_dtype != BIV_BF16) return set_error(BIV_ERR_UNSUPPORTED, "gemm: FP8 GEMM writes bf16");
    BIV_REQUIRE(d->sa && d->sb && d->ld_sa >= (d->K + 127) / 128, "gemm: FP8 needs sa/sb");
    BIV_REQUIRE(d->groups <= 1 || d->group_offsets, "gemm: grouped needs offsets");
    BIV_REQUIRE(d->groups <= Fp8Cfg<256>::MAX_GROUPS, "gemm: at most %d groups",
                Fp8Cfg<256>::MAX_GROUPS);
  }
  return BIV_OK;
}

// The bf16 call that biv_gemm_nvfp4 matches bit for bit (B decoded to bf16).
biv_gemm_desc nvfp4_as_bf16(const uint16_t* A, int64_t lda, const uint16_t* Bdec, int M, int N,
                            int K, void* C, int64_t ldc, int c_dtype, int mode) {
  biv_gemm_desc d;
  memset(&d, 0, sizeof(d));
  d.M = M; d.N = N; d.K = K;
  d.a_dtype = d.b_dtype = BIV_BF16;
  d.c_dtype = c_dtype;
  d.A = A; d.lda = lda;
  d.B = Bdec; d.ldb = K;
  d.C = C; d.ldc = ldc;
  d.mode = mode;
  return d;
}

struct Fp4Plan {
  Plan p;              // the bf16 plan of the same shape
  bool native = false; // NVFP4 partial kernel (else: decode, then the bf16 GEMM)
  int stages = 0;
  size_t dec_bytes = 0, ws_bytes = 0;
};

Fp4Plan plan_nvfp4(const biv_gemm_desc& d) {
  Fp4Plan f;
  f.p = plan_bf16(d);
  // the native kernel reads 16-byte scale groups by TMA: rows of K/16 bytes
  // must be whole 16-byte units.  It runs every weight-streaming shape (at
  // most kPartialRows rows) as partials, also those whose bf16 plan folds in
  // the CTA (wide N, e.g. an LM head): partial and in-CTA fold give the same
  // bits, and only the native kernel reads 4-bit weights.
  const bool stream_rows = d.M <= kPartialRows && d.mode == BIV_MODE_INVARIANT;
  // At most 64 activation rows: the kernel's two accumulators (the box's rows
  // as TMEM columns) and three decoded 32-column tiles share 256 columns.
  f.native = d.K % 256 == 0 && d.M <= kPartialRows &&
             ((f.p.partial && f.p.bn == 128) || stream_rows);
  if (f.native && !(f.p.partial && f.p.bn == 128)) {
    const int64_t tiles_m = (d.M + BM - 1) / BM;
    f.p.partial = true;
    f.p.bn = 128;
    f.p.tiles = int64_t((d.N + 127) / 128) * tiles_m;
    f.p.ldp = int64_t((d.N + 127) / 128) * 128;
    f.p.ws_bytes = size_t(f.p.chunks) * d.M * f.p.ldp * sizeof(float);
  }
  if (f.native) {
    const size_t per = size_t(kFp4Sub) * f.p.m_box * 128 + kFp4CodeBytes + kFp4SclBytes;
    f.stages = int(std::min<size_t>(kFp4MaxRaw, (kSmemBudget - fp4_smem_bytes(0, f.p.m_box)) / per));
    f.ws_bytes = f.p.ws_bytes;
  } else {
    f.dec_bytes = (size_t(d.N) * d.K * 2 + 255) / 256 * 256;
    f.ws_bytes = f.dec_bytes + f.p.ws_bytes;
  }
  return f;
}

}  // namespace
}  // namespace biv

using namespace biv;

extern "C" {

biv_status biv_nvfp4_dequant(const uint8_t* codes, const uint8_t* scales, int N, int K,
                             uint16_t* out, biv_stream_t stream);

static biv_status nvfp4_check(const uint16_t* A, int64_t lda, const uint8_t* codes,
                              const uint8_t* scales, int M, int N, int K, const void* C,
                              int64_t ldc, int c_dtype, int mode) {
  BIV_REQUIRE(M >= 0 && N > 0 && K > 0 && K % 16 == 0,
              "gemm_nvfp4: K=%d must be a multiple of 16", K);
  BIV_REQUIRE(c_dtype == BIV_BF16 || c_dtype == BIV_F32, "gemm_nvfp4: C is bf16 or f32");
  BIV_REQUIRE(mode == BIV_MODE_INVARIANT || mode == BIV_MODE_FAST, "gemm_nvfp4: bad mode");
  if (M == 0) return BIV_OK;
  BIV_REQUIRE(A && codes && scales && C && aligned16(A) && aligned16(codes) && aligned16(scales) &&
                  aligned16(C) && lda >= K && (lda * 2) % 16 == 0 && ldc >= N,
              "gemm_nvfp4: null or misaligned operand");
  return BIV_OK;
}

biv_status biv_gemm_nvfp4_workspace(int M, int N, int K, int c_dtype, int mode, size_t* bytes) {
  BIV_REQUIRE(bytes, "gemm_nvfp4_workspace: null output");
  BIV_REQUIRE(M >= 0 && N > 0 && K > 0 && K % 16 == 0, "gemm_nvfp4: K must be a multiple of 16");
  BIV_REQUIRE(c_dtype == BIV_BF16 || c_dtype == BIV_F32, "gemm_nvfp4: C is bf16 or f32");
  const biv_gemm_desc d = nvfp4_as_bf16(nullptr, K, nullptr, M, N, K, nullptr, N, c_dtype, mode);
  *bytes = M == 0 ? 0 : plan_nvfp4(d).ws_bytes;
  return BIV_OK;
}

biv_status biv_gemm_nvfp4(const uint16_t* A, int64_t lda, const uint8_t* codes,
                          const uint8_t* scales, int M, int N, int K, void* C, int64_t ldc,
                          int c_dtype, int mode, void* ws, size_t ws_bytes, biv_stream_t stream) {
  biv_status st = nvfp4_check(A, lda, codes, scales, M, N, K, C, ldc, c_dtype, mode);
  if (st != BIV_OK || M == 0) return st;
  biv_gemm_desc d = nvfp4_as_bf16(A, lda, nullptr, M, N, K, C, ldc, c_dtype, mode);
  const Fp4Plan f = plan_nvfp4(d);
  if (f.ws_bytes && (!ws || ws_bytes < f.ws_bytes || !aligned16(ws)))
    return set_error(BIV_ERR_WORKSPACE, "gemm_nvfp4: 16-byte aligned workspace of %zu bytes needed",
                     f.ws_bytes);
  cudaStream_t s = as_cuda(stream);
  if (!f.native) {
    // many rows: decode the weights once, then the bf16 GEMM (compute-bound
    // here), its own partials after the decoded weights
    uint16_t* dec = static_cast<uint16_t*>(ws);
    st = biv_nvfp4_dequant(codes, scales, N, K, dec, stream);
    if (st != BIV_OK) return st;
    d.B = dec;
    CUtensorMap ta, tb;
    if (!make_bf16_maps(&ta, &tb, A, lda, M, dec, K, N, K, f.p))
      return set_error(BIV_ERR_CUDA, "gemm_nvfp4: tensor map encoding failed");
    // the decoded weights come from the kernel just before: no early B prefetch
    void* pws = static_cast<uint8_t*>(ws) + f.dec_bytes;
    return c_dtype == BIV_F32 ? dispatch_bf16<true>(ta, tb, d, f.p, pws, s, true)
                              : dispatch_bf16<false>(ta, tb, d, f.p, pws, s, true);
  }
  const Plan& p = f.p;
  CUtensorMap ta, tc, ts;
  if (!make_map_panels(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A, K, M, lda, 64, p.m_box,
                       kFp4Sub) ||
      !make_map(&tc, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, codes, K / 2, N, K / 2, 128, 128, true) ||
      !make_map(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, scales, K / 16, N, K / 16,
                std::min(32, K / 16), 128, false))
    return set_error(BIV_ERR_CUDA, "gemm_nvfp4: tensor map encoding failed");
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(gemm_nvfp4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(kSmemBudget)) != cudaSuccess)
      return set_error(BIV_ERR_CUDA, "gemm_nvfp4: cannot set shared memory size");
    attr = true;
  }
  const int eb = c_dtype == BIV_F32 ? 4 : 2;
  GemmArgs a;
  memset(&a, 0, sizeof(a));
  a.C = C; a.ldc = ldc; a.M = M; a.N = N; a.K = K;
  a.kc_blocks = p.kc_blocks; a.m_box = p.m_box; a.stages = f.stages; a.partial = 1;
  a.ws = static_cast<float*>(ws); a.ldp = p.ldp;
  a.vec_ok = aligned16(C) && (ldc * eb) % 16 == 0;
  a.err = device_error_word();
  const int64_t items = p.tiles * p.chunks;
  const int sms = sm_count() > 0 ? sm_count() : 148;
  launch_pdl(gemm_nvfp4_kernel, int(std::min<int64_t>(items, sms)), kFp4Threads,
             fp4_smem_bytes(f.stages, p.m_box), s, ta, tc, ts, a);
  st = check_launch("gemm_nvfp4");
  if (st != BIV_OK) return st;
  const int64_t groups = int64_t(M) * ((N + 3) / 4);
  const int blocks = int(std::min<int64_t>((groups + 255) / 256, int64_t(sms) * 8));
  if (c_dtype == BIV_F32)
    launch_pdl(gemm_fold_kernel<true>, blocks, 256, 0, s, static_cast<const float*>(ws), C, ldc, M,
               N, p.ldp, p.chunks, a.vec_ok);
  else
    launch_pdl(gemm_fold_kernel<false>, blocks, 256, 0, s, static_cast<const float*>(ws), C, ldc, M,
               N, p.ldp, p.chunks, a.vec_ok);
  return check_launch("gemm_nvfp4_fold");
}

biv_status biv_gemm_workspace(const biv_gemm_desc* d, size_t* bytes) {
  biv_status st = validate(d);
  if (st != BIV_OK) return st;
  BIV_REQUIRE(bytes, "gemm_workspace: null output");
  *bytes = d->a_dtype == BIV_BF16 ? plan_bf16(*d).ws_bytes : 0;
  return BIV_OK;
}

biv_status biv_gemm_partials(const biv_gemm_desc* d, const void* ws, biv_partials* out) {
  biv_status st = validate(d);
  if (st != BIV_OK) return st;
  BIV_REQUIRE(out, "gemm_partials: null output");
  memset(out, 0, sizeof(*out));
  if (d->a_dtype != BIV_BF16) return BIV_OK;
  const Plan p = plan_bf16(*d);
  if (!p.partial) return BIV_OK;
  out->p = static_cast<const float*>(ws);
  out->chunks = p.chunks;
  out->ld = p.ldp;
  out->chunk_stride = int64_t(d->M) * p.ldp;
  return BIV_OK;
}

biv_status biv_gemm(const biv_gemm_desc* d, void* ws, size_t ws_bytes, biv_stream_t stream) {
  biv_status st = validate(d);
  if (st != BIV_OK) return st;
  if (d->M == 0) return BIV_OK;
  cudaStream_t s = as_cuda(stream);
  CUtensorMap ta, tb;
  if (d->a_dtype == BIV_BF16) {
    const Plan p = plan_bf16(*d);
    if (p.ws_bytes && (!ws || ws_bytes < p.ws_bytes))
      return set_error(BIV_ERR_WORKSPACE, "gemm: workspace of %zu bytes needed", p.ws_bytes);
    if (p.ws_bytes && !aligned16(ws))
      return set_error(BIV_ERR_INVALID, "gemm: workspace must be 16-byte aligned");
    if (!make_bf16_maps(&ta, &tb, d->A, d->lda, d->M, d->B, d->ldb, d->N, d->K, p))
      return set_error(BIV_ERR_CUDA, "gemm: tensor map encoding failed");
    return d->c_dtype == BIV_F32 ? dispatch_bf16<true>(ta, tb, *d, p, ws, s)
                                 : dispatch_bf16<false>(ta, tb, *d, p, ws, s);
  }
  // FP8 block-scaled (optionally grouped)
  const int groups = d->groups > 1 ? d->groups : 1;
  constexpr int bn = 256;
  const int kpb = fp8_kpb_for(d->K);
  const bool maps_ok =
      kpb == 2 ? make_map_panels(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, d->A, d->K, d->M, d->lda, 128,
                                 BM) &&
                     make_map_panels(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, d->B, d->K,
                                     int64_t(groups) * d->N, d->ldb, 128, bn)
               : make_map(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, d->A, d->K, d->M, d->lda, 128, BM) &&
                     make_map(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, d->B, d->K,
                              int64_t(groups) * d->N, d->ldb, 128, bn);
  if (!maps_ok) return set_error(BIV_ERR_CUDA, "gemm_fp8: tensor map encoding failed");
  return launch_fp8<bn>(ta, tb, *d, kpb, s);
}

}  // extern "C"


// ------------------------------------------- LM head + log-softmax gather --
// The logprob of every sampled token ("Finish RL Training Faster", section
// "零差异需要一个精确的比较对象") formed without writing the FP32 logits: the
// LM-head GEMM's epilogue reduces each row's logits, in groups of 128
// columns aligned to column 0, to (m_g, s_g) = (max, sum exp(z - m_g)) and
// keeps the target's logit; lse_combine_kernel then forms
// lp = z_t - (M + log S), M = max_g m_g, S = sum_g s_g * exp(m_g - M).
namespace biv {
namespace {

constexpr int kLseWarps = 8;

// One warp per row: lane l takes groups l, l+32, ... in ascending order; the
// lane maxima and sums are combined by xor trees (the order depends on the
// number of groups only).
__global__ void __launch_bounds__(kLseWarps * 32)
    lse_combine_kernel(const float2* __restrict__ lse, int ngroups, const float* __restrict__ zt,
                       const int32_t* __restrict__ target, int M, int N, float* __restrict__ lp,
                       int* err) {
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.x * kLseWarps + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (row >= M) return;
  const float2* g = lse + int64_t(row) * ngroups;
  float mx = -INFINITY;
  for (int i = lane; i < ngroups; i += 32) mx = fmaxf(mx, g[i].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float s = 0.f;
  for (int i = lane; i < ngroups; i += 32) {
    const float2 v = g[i];
    s = fmaf(v.y, expf(v.x - mx), s);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) {
    const int tg = target[row];
    if (tg < 0 || tg >= N) {
      raise_error(err, kErrBadIndex);
      lp[row] = NAN;
      return;
    }
    lp[row] = zt[row] - (mx + logf(s));
  }
}

size_t lse_bytes(int M, int V, int* ngroups) {
  const int ng = (V + kLseGroup - 1) / kLseGroup;
  if (ngroups) *ngroups = ng;
  return (size_t(M) * ng * sizeof(float2) + size_t(M) * sizeof(float) + 15) / 16 * 16;
}

// The fused head always folds in the CTA on 256-column tiles (two 128-column
// groups per tile), whatever M: the groups, and so every bit, stay the same
// for every batch.  K is chunked as in biv_gemm.
Plan plan_lse(const biv_gemm_desc& d) {
  Plan p;
  const int KB = (d.K + 63) / 64;
  p.m_box = d.M <= BM ? std::max(16, (d.M + 15) / 16 * 16) : BM;
  p.kc_blocks = d.mode == BIV_MODE_INVARIANT
                    ? std::max(kMinChunkBlocks, (KB + kMaxChunks - 1) / kMaxChunks)
                    : KB;
  p.chunks = (KB + p.kc_blocks - 1) / p.kc_blocks;
  p.bn = kWideN;
  p.partial = false;
  p.tiles = int64_t((d.N + p.bn - 1) / p.bn) * ((d.M + BM - 1) / BM);
  p.kpb = kpb_for(d.K);
  const size_t fixed = GemmSmem<kWideN>::bytes(0, p.m_box, true);
  p.stages = int(std::min<size_t>(kMaxStages, (kSmemBudget - fixed) /
                                                  ((p.m_box * 128 + GemmSmem<kWideN>::B_STAGE) * p.kpb)));
  return p;
}

}  // namespace
}  // namespace biv

using namespace biv;

extern "C" biv_status biv_lm_head_logprob_workspace(int M, int V, size_t* bytes) {
  BIV_REQUIRE(bytes && M >= 0 && V > 0, "lm_head_logprob_workspace: bad arguments");
  *bytes = lse_bytes(M, V, nullptr);
  return BIV_OK;
}

extern "C" biv_status biv_lm_head_logprob(const uint16_t* h, int64_t ldh, const uint16_t* W,
                                          int64_t ldw, int M, int V, int K,
                                          const int32_t* target, int mode, float* lp,
                                          void* workspace, size_t workspace_bytes,
                                          biv_stream_t stream) {
  BIV_REQUIRE(target && lp, "lm_head_logprob: null target or lp");
  BIV_REQUIRE(V % 4 == 0, "lm_head_logprob: V=%d must be a multiple of 4", V);
  biv_gemm_desc d;
  memset(&d, 0, sizeof(d));
  d.M = M; d.N = V; d.K = K;
  d.a_dtype = BIV_BF16; d.b_dtype = BIV_BF16; d.c_dtype = BIV_F32;
  d.A = h; d.lda = ldh; d.B = W; d.ldb = ldw;
  d.C = lp; d.ldc = V;   // C is not written; validate() wants a non-null target
  d.mode = mode;
  biv_status st = validate(&d);
  if (st != BIV_OK) return st;
  if (M == 0) return BIV_OK;
  int ng = 0;
  const size_t need = lse_bytes(M, V, &ng);
  if (!workspace || workspace_bytes < need)
    return set_error(BIV_ERR_WORKSPACE, "lm_head_logprob: workspace of %zu bytes needed", need);
  if (!aligned16(workspace))
    return set_error(BIV_ERR_INVALID, "lm_head_logprob: workspace must be 16-byte aligned");
  const Plan p = plan_lse(d);
  CUtensorMap ta, tb;
  if (!make_bf16_maps(&ta, &tb, h, ldh, M, W, ldw, V, K, p))
    return set_error(BIV_ERR_CUDA, "lm_head_logprob: tensor map encoding failed");
  auto kern = gemm_bf16_kernel<kWideN, true, false, true>;
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(kSmemBudget)) != cudaSuccess)
      return set_error(BIV_ERR_CUDA, "lm_head_logprob: cannot set shared memory size");
    attr = true;
  }
  GemmArgs a;
  memset(&a, 0, sizeof(a));
  a.M = M; a.N = V; a.K = K;
  a.kc_blocks = p.kc_blocks; a.m_box = p.m_box; a.stages = p.stages; a.kpb = p.kpb;
  a.n_fastest = V <= M;
  a.target = target;
  a.lse = static_cast<float2*>(workspace);
  a.zt = reinterpret_cast<float*>(static_cast<float2*>(workspace) + size_t(M) * ng);
  a.ngroups = ng;
  a.err = device_error_word();
  const int sms = sm_count() > 0 ? sm_count() : 148;
  cudaStream_t s = as_cuda(stream);
  launch_pdl(kern, int(std::min<int64_t>(p.tiles, sms)), kGemmThreads,
             GemmSmem<kWideN>::bytes(p.stages, p.m_box, true, p.kpb), s, ta, tb, a);
  st = check_launch("lm_head_logprob gemm");
  if (st != BIV_OK) return st;
  launch_pdl(lse_combine_kernel, (M + kLseWarps - 1) / kLseWarps, kLseWarps * 32, 0, s,
             static_cast<const float2*>(a.lse), ng, static_cast<const float*>(a.zt), target, M, V,
             lp, a.err);
  return check_launch("lm_head_logprob combine");
}
