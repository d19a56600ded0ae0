// Batch-invariant GEMM on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// C[M,N] = A[M,K] . B[N,K]^T, both operands K-major.  One CTA owns a 128 x BN
// output tile; TMA streams 128-byte-swizzled K-slabs of A and B into a
// shared-memory ring; one thread issues tcgen05.mma (M=128, N=BN) into an FP32
// accumulator in TMEM; the four warps read it back (tcgen05.ld) and store.
//
// Invariance ("Finish RL Training Faster", section "让训练前向使用推理的数值":
// one batch-invariant GEMM schedule): every output element is accumulated over
// K in ascending 64-wide (bf16) / 128-wide (FP8) blocks, each block as a fixed
// sequence of K=16 / K=32 MMA steps, with no split of K in INVARIANT mode.
// Nothing about M enters that sequence: rows past M are TMA zero-fill and are
// not stored.  FAST mode splits K when M is small (batch-dependent), the
// comparator the pages measure against.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdlib>
#include <mutex>

#include "common.cuh"

namespace biv {
namespace {

constexpr int BM = 128;

template <int BN>
struct Bf16Cfg {
  static constexpr int BK = 64;                       // 64 bf16 = one 128-byte swizzle row
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int STAGES = (192 * 1024) / STAGE > 8 ? 8 : (192 * 1024) / STAGE;
  static constexpr int TMEM_COLS = BN < 32 ? 32 : BN;
  static constexpr int SMEM = STAGES * STAGE + 1024 + 256;
};

template <int BN>
struct Fp8Cfg {
  static constexpr int BK = 128;                      // 128 e4m3 = one 128-byte swizzle row
  static constexpr int A_BYTES = BM * BK;
  static constexpr int B_BYTES = BN * BK;
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int STAGES = (160 * 1024) / STAGE > 8 ? 8 : (160 * 1024) / STAGE;
  static constexpr int TMEM_COLS = 2 * BN;            // two accumulator buffers
  static constexpr int SMEM = STAGES * STAGE + 1024 + 256;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Store 32 consecutive FP32 accumulator columns of one row.
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
    if (vec_ok && n + 32 <= N) {
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

// ------------------------------------------------------------ bf16 kernel --
// grid (ceil(N/BN), ceil(M/128), splits).  Split z covers K-blocks
// [z*kb_per_split, min(KB, (z+1)*kb_per_split)); with splits > 1 the FP32
// partial tile goes to partial[z][M][N] instead of C.
template <int BN, bool F32OUT>
__global__ void __launch_bounds__(128, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB, void* C, int64_t ldc, int M, int N,
                     int K, int kb_per_split, float* partial, int vec_ok, int a_box_bytes,
                     int* err) {
  // a_box_bytes: bytes of A that TMA writes per stage (rows of the A box x 128);
  // when M < 128 only the first rows are loaded, rows past them never feed a
  // stored output row.
  using Cfg = Bf16Cfg<BN>;
  constexpr int S = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sA = smem;
  uint8_t* sB = smem + S * Cfg::A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * Cfg::STAGE);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 1);
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + S), done = smem_u32(bars + 2 * S);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BN, m0 = blockIdx.y * BM;
  const int KB = (K + Cfg::BK - 1) / Cfg::BK;
  const int kb0 = blockIdx.z * kb_per_split;
  const int nkb = min(KB, kb0 + kb_per_split) - kb0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    mbar_init(done, 1);
    fence_barrier_init();
  }
  __syncwarp();
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  int issued = 0;
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    for (int i = 0; i < nkb; ++i) {
      const int s = i % S;
      if (i >= S && !mbar_wait(empty0 + 8 * s, ((i / S) - 1) & 1, err)) break;
      mbar_expect_tx(full0 + 8 * s, uint32_t(a_box_bytes + Cfg::B_BYTES));
      const int kx = (kb0 + i) * Cfg::BK;
      tma_load_2d(smem_u32(sA + s * Cfg::A_BYTES), &tmA, full0 + 8 * s, kx, m0);
      tma_load_2d(smem_u32(sB + s * Cfg::B_BYTES), &tmB, full0 + 8 * s, kx, n0);
      issued = i + 1;
    }
  } else if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc = idesc_mma(1u, BM, BN);
    for (int i = 0; i < nkb; ++i) {
      const int s = i % S;
      if (!mbar_wait(full0 + 8 * s, (i / S) & 1, err)) break;
      tc_fence_after();
      const uint32_t a0 = smem_u32(sA + s * Cfg::A_BYTES);
      const uint32_t b0 = smem_u32(sB + s * Cfg::B_BYTES);
#pragma unroll
      for (int kk = 0; kk < Cfg::BK / 16; ++kk)
        umma_f16(tmem, sdesc_k_sw128(a0 + kk * 32), sdesc_k_sw128(b0 + kk * 32), idesc,
                 (i | kk) != 0 ? 1u : 0u);
      umma_commit(empty0 + 8 * s);
    }
    umma_commit(done);
  }
  __syncwarp();
  const bool have = __all_sync(0xffffffffu, mbar_wait(done, 0, err));
  tc_fence_after();

  if (have) {
    const int row = m0 + warp * 32 + lane;
    const uint32_t trow = tmem + (uint32_t(warp * 32) << 16);
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += 32) {
      if (n0 + c0 >= N) break;  // warp-uniform
      uint32_t r[32];
      tmem_ld32(trow + c0, r);
      tmem_ld_wait();
      if (row < M) {
        if (partial) {
          float* dst = partial + (int64_t(blockIdx.z) * M + row) * N + n0 + c0;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (n0 + c0 + j < N) dst[j] = __uint_as_float(r[j]);
        } else {
          store_row32<F32OUT>(C, ldc, row, n0 + c0, N, r, vec_ok != 0);
        }
      }
    }
  }
  // the producer makes sure its copies have landed before the CTA exits
  if (warp == 0 && lane == 0) {
    for (int i = max(0, issued - S); i < issued; ++i)
      mbar_wait(full0 + 8 * (i % S), (i / S) & 1, err, 100000000ull);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, Cfg::TMEM_COLS);
}

// Deterministic split-K reduction: partials summed in ascending split order.
template <bool F32OUT>
__global__ void splitk_reduce_kernel(const float* __restrict__ partial, int splits, int M, int N,
                                     void* C, int64_t ldc) {
  const int64_t total = int64_t(M) * N;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * blockDim.x) {
    float acc = partial[i];
    for (int z = 1; z < splits; ++z) acc += partial[int64_t(z) * total + i];
    const int64_t row = i / N, col = i % N;
    if (F32OUT)
      static_cast<float*>(C)[row * ldc + col] = acc;
    else
      static_cast<uint16_t*>(C)[row * ldc + col] = f2bf(acc);
  }
}

// ----------------------------------------------------- persistent bf16 ----
// Same per-element schedule as gemm_bf16_kernel (ascending 64-wide K blocks,
// four K=16 MMAs each, FP32 accumulator in TMEM), so the two give identical
// bits.  Persistent grid; warp 0 = TMA producer, warp 1 = MMA issuer and TMEM
// owner, warps 2..5 = epilogue.  The accumulator is double-buffered in TMEM so
// the epilogue of tile j overlaps the main loop of tile j+1.  Tiles are walked
// M-fastest so that CTAs running together share the weight tile in L2.
template <int BN>
struct PersistCfg {
  static constexpr int BK = 64;
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int STAGES = (200 * 1024) / STAGE > 8 ? 8 : (200 * 1024) / STAGE;
  static constexpr int TMEM_COLS = 2 * BN;
  static constexpr int SMEM = STAGES * STAGE + 1024 + 256;
};

template <int BN, bool F32OUT>
__global__ void __launch_bounds__(192, 1)
    gemm_bf16_persistent(const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmB, void* C, int64_t ldc, int M,
                         int N, int K, int vec_ok, int n_fastest, int* err) {
  // n_fastest: walk N tiles first (CTAs running together share an A tile and
  // B is re-read from L2) when B is the smaller operand; else M first.
  using Cfg = PersistCfg<BN>;
  constexpr int S = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sA = smem;
  uint8_t* sB = smem + S * Cfg::A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * Cfg::STAGE);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 4);
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + S);
  const uint32_t tfull0 = smem_u32(bars + 2 * S), tempty0 = smem_u32(bars + 2 * S + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KB = (K + Cfg::BK - 1) / Cfg::BK;
  const int tiles_m = (M + BM - 1) / BM, tiles_n = (N + BN - 1) / BN;
  const int tiles = tiles_m * tiles_n;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int j = 0; j < 2; ++j) {
      mbar_init(tfull0 + 8 * j, 1);
      mbar_init(tempty0 + 8 * j, 4);
    }
    fence_barrier_init();
  }
  __syncwarp();
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  int issued = 0;
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    bool ok = true;
    for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
      const int m0 = (n_fastest ? t / tiles_n : t % tiles_m) * BM;
      const int n0 = (n_fastest ? t % tiles_n : t / tiles_m) * BN;
      for (int kb = 0; kb < KB; ++kb) {
        const int it = issued, s = it % S;
        if (it >= S && !mbar_wait(empty0 + 8 * s, ((it / S) - 1) & 1, err)) {
          ok = false;
          break;
        }
        mbar_expect_tx(full0 + 8 * s, Cfg::STAGE);
        tma_load_2d(smem_u32(sA + s * Cfg::A_BYTES), &tmA, full0 + 8 * s, kb * Cfg::BK, m0);
        tma_load_2d(smem_u32(sB + s * Cfg::B_BYTES), &tmB, full0 + 8 * s, kb * Cfg::BK, n0);
        issued = it + 1;
      }
    }
  } else if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc = idesc_mma(1u, BM, BN);
    int it = 0, j = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++j) {
      const int b = j & 1;
      if (j >= 2 && !mbar_wait(tempty0 + 8 * b, ((j >> 1) - 1) & 1, err)) break;
      tc_fence_after();
      const uint32_t dt = tmem + b * BN;
      for (int kb = 0; kb < KB; ++kb, ++it) {
        const int s = it % S;
        if (!mbar_wait(full0 + 8 * s, (it / S) & 1, err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(sA + s * Cfg::A_BYTES);
        const uint32_t b0 = smem_u32(sB + s * Cfg::B_BYTES);
#pragma unroll
        for (int kk = 0; kk < Cfg::BK / 16; ++kk)
          umma_f16(dt, sdesc_k_sw128(a0 + kk * 32), sdesc_k_sw128(b0 + kk * 32), idesc,
                   (kb | kk) != 0 ? 1u : 0u);
        umma_commit(empty0 + 8 * s);
      }
      umma_commit(tfull0 + 8 * b);
    }
  } else if (warp >= 2) {
    const int q = warp & 3;
    int j = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++j) {
      const int b = j & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(tfull0 + 8 * b, (j >> 1) & 1, err))) break;
      tc_fence_after();
      const int m0 = (n_fastest ? t / tiles_n : t % tiles_m) * BM;
      const int n0 = (n_fastest ? t % tiles_n : t / tiles_m) * BN;
      const int row = m0 + q * 32 + lane;
      const uint32_t trow = tmem + b * BN + (uint32_t(q * 32) << 16);
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 32) {
        if (n0 + c0 >= N) break;  // warp-uniform
        uint32_t r[32];
        tmem_ld32(trow + c0, r);
        tmem_ld_wait();
        if (row < M) store_row32<F32OUT>(C, ldc, row, n0 + c0, N, r, vec_ok != 0);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty0 + 8 * b);
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

// ------------------------------------------------------------- FP8 kernel --
// 6 warps: warp 0 = TMA producer, warp 1 = MMA issuer (+TMEM owner),
// warps 2..5 = promotion/epilogue (lane quarter = warp % 4).  For each
// 128-wide K block the MMA writes a fresh FP32 partial into one of two TMEM
// buffers; the epilogue warps fold it into registers as
// acc = fma(sa*sb, partial, acc), blocks in ascending order.
// grid (ceil(N/BN), tiles over groups).
template <int BN>
__global__ void __launch_bounds__(192, 1)
    gemm_fp8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    uint16_t* C, int64_t ldc, int M, int N, int K, const float* __restrict__ sa,
                    int64_t ld_sa, const float* __restrict__ sb, const int32_t* __restrict__ offs,
                    int groups, int vec_ok, int* err) {
  using Cfg = Fp8Cfg<BN>;
  constexpr int S = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  // locate this CTA's (group, row range)
  int g = 0, m0 = blockIdx.y * BM, m_end = M;
  if (groups > 1) {
    int before = 0;
    g = -1;
    for (int gg = 0; gg < groups; ++gg) {
      const int lo = offs[gg], hi = offs[gg + 1];
      const int nt = (hi - lo + BM - 1) / BM;
      if (int(blockIdx.y) < before + nt) {
        g = gg;
        m0 = lo + (int(blockIdx.y) - before) * BM;
        m_end = hi;
        break;
      }
      before += nt;
    }
    if (g < 0) return;  // uniform early exit: nothing allocated yet
  }
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sA = smem;
  uint8_t* sB = smem + S * Cfg::A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * Cfg::STAGE);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 4);
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + S);
  const uint32_t tfull0 = smem_u32(bars + 2 * S), tempty0 = smem_u32(bars + 2 * S + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BN;
  const int KB = (K + Cfg::BK - 1) / Cfg::BK;
  const int NB = (N + 127) / 128;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int j = 0; j < 2; ++j) {
      mbar_init(tfull0 + 8 * j, 1);
      mbar_init(tempty0 + 8 * j, 4);
    }
    fence_barrier_init();
  }
  __syncwarp();
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  int issued = 0;
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    for (int i = 0; i < KB; ++i) {
      const int s = i % S;
      if (i >= S && !mbar_wait(empty0 + 8 * s, ((i / S) - 1) & 1, err)) break;
      mbar_expect_tx(full0 + 8 * s, Cfg::STAGE);
      tma_load_2d(smem_u32(sA + s * Cfg::A_BYTES), &tmA, full0 + 8 * s, i * Cfg::BK, m0);
      tma_load_2d(smem_u32(sB + s * Cfg::B_BYTES), &tmB, full0 + 8 * s, i * Cfg::BK, g * N + n0);
      issued = i + 1;
    }
  } else if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc = idesc_mma(0u, BM, BN);
    for (int i = 0; i < KB; ++i) {
      const int s = i % S, j = i & 1;
      if (i >= 2 && !mbar_wait(tempty0 + 8 * j, ((i >> 1) - 1) & 1, err)) break;
      if (!mbar_wait(full0 + 8 * s, (i / S) & 1, err)) break;
      tc_fence_after();
      const uint32_t a0 = smem_u32(sA + s * Cfg::A_BYTES);
      const uint32_t b0 = smem_u32(sB + s * Cfg::B_BYTES);
#pragma unroll
      for (int kk = 0; kk < Cfg::BK / 32; ++kk)
        umma_f8(tmem + j * BN, sdesc_k_sw128(a0 + kk * 32), sdesc_k_sw128(b0 + kk * 32), idesc,
                kk != 0 ? 1u : 0u);
      umma_commit(empty0 + 8 * s);
      umma_commit(tfull0 + 8 * j);
    }
  } else if (warp >= 2) {
    const int q = warp & 3;
    const int row = m0 + q * 32 + lane;
    const bool live = row < m_end && row < M;
    const float* sbg = sb + int64_t(g) * NB * KB + int64_t(n0 / 128) * KB;
    float acc[BN];
#pragma unroll
    for (int c = 0; c < BN; ++c) acc[c] = 0.f;
    bool ok = true;
    for (int i = 0; i < KB && ok; ++i) {
      const int j = i & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(tfull0 + 8 * j, (i >> 1) & 1, err))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float scale = (live ? sa[int64_t(row) * ld_sa + i] : 0.f) * sbg[i];
      const uint32_t tb = tmem + j * BN + (uint32_t(q * 32) << 16);
#pragma unroll
      for (int c0 = 0; c0 < BN; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(tb + c0, r);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 32; ++c) acc[c0 + c] = fmaf(scale, __uint_as_float(r[c]), acc[c0 + c]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty0 + 8 * j);
    }
    if (ok && live) {
#pragma unroll
      for (int c0 = 0; c0 < BN; c0 += 32) {
        uint32_t r[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) r[c] = __float_as_uint(acc[c0 + c]);
        if (n0 + c0 < N) store_row32<false>(C, ldc, row, n0 + c0, N, r, vec_ok != 0);
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

// ------------------------------------------------------------------- host --
// 2-D K-major tensor map: dims {K, rows}, box {box_k, box_rows}, 128B swizzle.
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, int elem_bytes, const void* base,
              int64_t K, int64_t rows, int64_t ld, int box_k, int box_rows) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {cuuint64_t(K), cuuint64_t(rows)};
  cuuint64_t strides[1] = {cuuint64_t(ld * elem_bytes)};
  cuuint32_t box[2] = {cuuint32_t(box_k), cuuint32_t(box_rows)};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

struct Plan {
  int bn = 128;
  int splits = 1;
  int kb_per_split = 0;
  bool persistent = false;
  int m_box = BM;  // rows of the A TMA box
};

// Few output tiles (decode-sized M): pick the tile width with the best
// modelled weight-streaming rate.  Per 64-wide K block a CTA moves through
// shared memory the A box (m_box rows), the B tile (TMA write) and the MMA's
// operand reads (128 A rows + BN B rows, 4 times 32 bytes each), so the weight
// share of that traffic is BN / (m_box + 2 BN + 128); CTAs beyond the SM
// count add nothing.
int pick_small_m_bn(int M, int N, int m_box, int sms) {
  const int tiles_m = (M + BM - 1) / BM;
  int best = 128;
  double best_score = -1.0;
  for (int bn : {256, 128, 64, 32}) {
    if (bn > 32 && bn / 2 >= N) continue;
    const double rate = double(bn) / double(m_box + 2 * bn + 128);
    const int64_t ctas = int64_t((N + bn - 1) / bn) * tiles_m;
    const double score = double(std::min<int64_t>(ctas, sms)) * rate;
    if (score > best_score * 1.0001) {
      best_score = score;
      best = bn;
    }
  }
  return best;
}

// Test overrides: BIV_GEMM_PERSISTENT=0 forces the one-tile-per-CTA kernel and
// BIV_GEMM_TILE_N=32|64|128|256 forces the tile width; the tests use them to
// check that neither choice changes a result bit.
bool persistent_allowed() {
  const char* e = getenv("BIV_GEMM_PERSISTENT");
  return !(e && e[0] == '0');
}

// INVARIANT: the tile width depends on N only; K is never split.
// FAST: for small M, narrow tiles and a K split sized to fill the GPU.
Plan plan_bf16(const biv_gemm_desc& d) {
  Plan p;
  const int KB = (d.K + 63) / 64;
  p.bn = d.N >= 8192 ? 256 : (d.N >= 128 ? 128 : (d.N > 32 ? 64 : 32));
  p.kb_per_split = KB;
  // The tile width (MMA instruction N) and the one-tile vs persistent kernel
  // do not change any element's K schedule, and tcgen05 gives the same bits
  // for every instruction N, so both may follow M.  Enough 128x256 tiles to
  // fill the GPU: the widest tile on the persistent kernel (least shared-memory
  // traffic per FLOP).
  const int sms = sm_count() > 0 ? sm_count() : 148;
  const int64_t mt = (d.M + BM - 1) / BM;
  if (d.N >= 256 && int64_t((d.N + 255) / 256) * mt >= sms) {
    p.bn = 256;
  } else {
    p.m_box = d.M <= BM ? std::max(16, (d.M + 15) / 16 * 16) : BM;
    p.bn = pick_small_m_bn(d.M, d.N, p.m_box, sms);
  }
  if (const char* e = getenv("BIV_GEMM_TILE_N")) {  // test override of the tile width
    const int bn = atoi(e);
    if (bn == 32 || bn == 64 || bn == 128 || bn == 256) p.bn = bn;
  }
  const int64_t tiles = int64_t((d.N + p.bn - 1) / p.bn) * mt;
  p.persistent = tiles >= 2 * sms && persistent_allowed();
  if (d.mode == BIV_MODE_FAST && d.M <= 256) {
    // the batch-dependent comparator: same modelled tile, plus a K split that
    // fills the GPU (this is what makes its bits depend on M)
    p.persistent = false;
    const int tiles = ((d.N + p.bn - 1) / p.bn) * ((d.M + BM - 1) / BM);
    const int sms = sm_count() > 0 ? sm_count() : 148;
    // split K only when the tiles leave most SMs idle; aim at one wave
    int splits = tiles * 2 <= sms ? (sms + tiles - 1) / tiles : 1;
    splits = std::max(1, std::min(splits, KB / 8));
    p.kb_per_split = (KB + splits - 1) / splits;
    p.splits = (KB + p.kb_per_split - 1) / p.kb_per_split;
  }
  return p;
}

template <int BN, bool F32OUT>
biv_status launch_bf16(const CUtensorMap& ta, const CUtensorMap& tb, const biv_gemm_desc& d,
                       const Plan& p, float* partial, cudaStream_t s) {
  using Cfg = Bf16Cfg<BN>;
  auto kern = gemm_bf16_kernel<BN, F32OUT>;
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM) !=
        cudaSuccess)
      return set_error(BIV_ERR_CUDA, "gemm: cannot set shared memory size");
    attr = true;
  }
  const int eb = F32OUT ? 4 : 2;
  const int vec_ok = aligned16(d.C) && (d.ldc * eb) % 16 == 0;
  dim3 grid((d.N + BN - 1) / BN, (d.M + BM - 1) / BM, p.splits);
  kern<<<grid, 128, Cfg::SMEM, s>>>(ta, tb, d.C, d.ldc, d.M, d.N, d.K, p.kb_per_split,
                                    p.splits > 1 ? partial : nullptr, vec_ok, p.m_box * 128,
                                    device_error_word());
  return check_launch("gemm_bf16");
}

template <int BN, bool F32OUT>
biv_status launch_bf16_persistent(const CUtensorMap& ta, const CUtensorMap& tb,
                                  const biv_gemm_desc& d, cudaStream_t s) {
  using Cfg = PersistCfg<BN>;
  auto kern = gemm_bf16_persistent<BN, F32OUT>;
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM) !=
        cudaSuccess)
      return set_error(BIV_ERR_CUDA, "gemm: cannot set shared memory size");
    attr = true;
  }
  const int eb = F32OUT ? 4 : 2;
  const int vec_ok = aligned16(d.C) && (d.ldc * eb) % 16 == 0;
  const int tiles = ((d.N + BN - 1) / BN) * ((d.M + BM - 1) / BM);
  const int sms = sm_count() > 0 ? sm_count() : 148;
  const int grid = std::min(tiles, sms);
  const int n_fastest = d.N <= d.M;
  kern<<<grid, 192, Cfg::SMEM, s>>>(ta, tb, d.C, d.ldc, d.M, d.N, d.K, vec_ok, n_fastest,
                                    device_error_word());
  return check_launch("gemm_bf16_persistent");
}

template <bool F32OUT>
biv_status dispatch_bf16(const CUtensorMap& ta, const CUtensorMap& tb, const biv_gemm_desc& d,
                         const Plan& p, float* partial, cudaStream_t s) {
  if (p.persistent) {
    switch (p.bn) {
      case 256: return launch_bf16_persistent<256, F32OUT>(ta, tb, d, s);
      case 128: return launch_bf16_persistent<128, F32OUT>(ta, tb, d, s);
      case 64: return launch_bf16_persistent<64, F32OUT>(ta, tb, d, s);
      default: return launch_bf16_persistent<32, F32OUT>(ta, tb, d, s);
    }
  }
  switch (p.bn) {
    case 256: return launch_bf16<256, F32OUT>(ta, tb, d, p, partial, s);
    case 128: return launch_bf16<128, F32OUT>(ta, tb, d, p, partial, s);
    case 64: return launch_bf16<64, F32OUT>(ta, tb, d, p, partial, s);
    default: return launch_bf16<32, F32OUT>(ta, tb, d, p, partial, s);
  }
}

template <int BN>
biv_status launch_fp8(const CUtensorMap& ta, const CUtensorMap& tb, const biv_gemm_desc& d,
                      cudaStream_t s) {
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
  const int tiles_m = (d.M + BM - 1) / BM + (groups > 1 ? groups : 0);
  dim3 grid((d.N + BN - 1) / BN, tiles_m, 1);
  kern<<<grid, 192, Cfg::SMEM, s>>>(ta, tb, static_cast<uint16_t*>(d.C), d.ldc, d.M, d.N, d.K,
                                    d.sa, d.ld_sa, d.sb, d.group_offsets, groups, vec_ok,
                                    device_error_word());
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
  }
  return BIV_OK;
}

}  // namespace
}  // namespace biv

using namespace biv;

extern "C" {

biv_status biv_gemm_workspace(const biv_gemm_desc* d, size_t* bytes) {
  biv_status st = validate(d);
  if (st != BIV_OK) return st;
  BIV_REQUIRE(bytes, "gemm_workspace: null output");
  *bytes = 0;
  if (d->a_dtype == BIV_BF16) {
    const Plan p = plan_bf16(*d);
    if (p.splits > 1) *bytes = size_t(p.splits) * d->M * d->N * sizeof(float);
  }
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
    const size_t need = p.splits > 1 ? size_t(p.splits) * d->M * d->N * sizeof(float) : 0;
    if (need && (!ws || ws_bytes < need))
      return set_error(BIV_ERR_WORKSPACE, "gemm: workspace of %zu bytes needed", need);
    if (!make_map(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d->A, d->K, d->M, d->lda, 64,
                  p.persistent ? BM : p.m_box) ||
        !make_map(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d->B, d->K, d->N, d->ldb, 64, p.bn))
      return set_error(BIV_ERR_CUDA, "gemm: tensor map encoding failed");
    float* partial = static_cast<float*>(ws);
    st = d->c_dtype == BIV_F32 ? dispatch_bf16<true>(ta, tb, *d, p, partial, s)
                               : dispatch_bf16<false>(ta, tb, *d, p, partial, s);
    if (st != BIV_OK || p.splits == 1) return st;
    const int64_t total = int64_t(d->M) * d->N;
    const int blocks = int(std::min<int64_t>((total + 255) / 256, int64_t(sm_count() * 16 + 1)));
    if (d->c_dtype == BIV_F32)
      splitk_reduce_kernel<true><<<blocks, 256, 0, s>>>(partial, p.splits, d->M, d->N, d->C, d->ldc);
    else
      splitk_reduce_kernel<false><<<blocks, 256, 0, s>>>(partial, p.splits, d->M, d->N, d->C, d->ldc);
    return check_launch("gemm_splitk_reduce");
  }
  // FP8 block-scaled (optionally grouped)
  const int groups = d->groups > 1 ? d->groups : 1;
  const int bn = 128;
  if (!make_map(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, d->A, d->K, d->M, d->lda, 128, BM) ||
      !make_map(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, d->B, d->K, int64_t(groups) * d->N, d->ldb,
                128, bn))
    return set_error(BIV_ERR_CUDA, "gemm_fp8: tensor map encoding failed");
  return launch_fp8<128>(ta, tb, *d, s);
}

}  // extern "C"
