// One paged attention operator for prefill, chunked prefill, decode and
// trainer recompute ("Finish RL Training Faster", section "让训练前向使用推理的数值":
// every path gathers, dequantises and enters the same attention operator).
//
// A CTA handles one query block (rows of one sequence), one KV head and one
// KV split.  Its query vectors are (row, q-head-of-the-group) pairs, 16 per
// warp.  Keys are visited in 64-token tiles aligned to absolute positions (one
// cache page), inside splits of kv_split tokens.  Per vector and split:
// online softmax in FP32 in base 2 (x = s * scale * log2 e, rounded once;
// p = 2^(x - m) by ex2.approx; the natural-base softmax up to rounding; m
// moves lazily, see kLazy), P
// split into three bf16 parts hi + mid + lo that add up to the FP32 p exactly
// (three MMAs into one FP32 accumulator, hi first), the denominator summed
// from the FP32 p.  Splits are merged in ascending order.  A vector's arithmetic is the
// same whatever other rows share its CTA and whatever the CTA shape: each warp
// runs one instruction sequence for its 16 vectors, tiles past a vector's own
// position are fully masked and leave (m, l, acc) bitwise unchanged, and
// masked V slots are zero in shared memory.
//
// Loads: dense bf16 pages (D = 64 or 128) arrive by TMA, one 3-D bulk copy
// per page of K and of V (its 64-dim panels back to back), 128-byte
// swizzled, completed on an mbarrier;
// FP8 pages (dequantised on the way in), sparse gathers and D = 80 use
// cp.async / plain loads into padded rows.
#include <algorithm>
#include <climits>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace biv {
namespace {

constexpr int kTile = 64;   // keys per tile = one page
constexpr int kNV = 64;     // most query vectors an attn_kernel CTA takes (4 warps x 16)
constexpr int kNVTc = 128;  // most query vectors a block may hold (attn_tc_kernel)
// Lazy rescaling: a row's running max m (base-2 units) moves only when a tile's
// max exceeds it by more than kLazy, so p = 2^(x - m) stays below 2^kLazy and
// O, l are rescaled rarely.  Every kernel applies the same rule per row.
constexpr float kLazy = 8.f;

// NW warps per CTA, ST-stage K/V pipeline, TMA or thread-issued loads, and
// DS: 1 = each warp owns 16 query vectors (prefill blocks); DS > 1 = DS
// consecutive warps share one group of 16 vectors (NW / DS groups): each
// computes 64/DS keys of the group's score tile, the tile is exchanged
// through shared memory, every warp of the group runs the same softmax on all
// of it and takes 1/DS of the head dimension in P.V (decode blocks, and the
// 32-vector blocks of the sparse path: shorter dependency chains per warp,
// the same arithmetic for every output element).
// F8: FP8 pages; their codes and scales land in a staging area by cp.async one
// tile ahead and are dequantised shared-to-shared into the bf16 K/V tiles.
// One staging buffer: tile t+1's copies are issued once tile t is dequantised
// (a second buffer was never in use, and without it four decode CTAs fit on
// an SM instead of three).
template <int D, int NW, int ST, bool TMA, int DS, bool F8 = false>
struct AttnCfg {
  static_assert(NW % DS == 0 && 4 % DS == 0, "D split: DS warps per vector group");
  static_assert(!(F8 && TMA), "FP8 pages use the thread loader");
  static_assert(!F8 || ST == 2, "FP8 pages: one staged tile in flight");
  static constexpr int LD = D + 8;                   // padded row (elements), thread-loaded tiles
  static constexpr int NV = NW / DS * 16;            // query vectors per CTA
  static constexpr int NT = NW * 32;                 // threads per CTA
  static constexpr int KVB = TMA ? kTile * D * 2 : kTile * LD * 2;  // one K or V stage
  // bf16 K/V tile stages: FP8 keeps one (its staging area holds the prefetch)
  static constexpr int TST = F8 ? 1 : ST;
  // Q is read into registers once; with a D split its area then holds each
  // group's S tile as the warps assemble it (8 n-tiles x 32 lanes x 4 FP32)
  static constexpr int S_BYTES = DS > 1 ? NW / DS * 8 * 32 * 16 : 0;
  static constexpr int Q_BYTES = NV * LD * 2 > S_BYTES ? NV * LD * 2 : S_BYTES;
  static constexpr int F8_CODES = F8 ? 2 * kTile * D : 0;          // K then V codes
  static constexpr int F8_STAGE = F8 ? F8_CODES + 2 * kTile * 4 : 0;  // + K then V scales
  // TMA tiles are 128-byte swizzled (1024-byte aligned); thread-loaded ones
  // need 16 bytes
  static constexpr int ALIGN = TMA ? 1024 : 16;
  static constexpr int SMEM = ALIGN + 2 * TST * KVB + Q_BYTES + F8_STAGE + ST * kTile * 4 +
                              2 * ST * 8 + (TMA ? 0 : kTile * 4);
  // thread-issued copies: how many of a thread's copies read their source
  // rows before any is issued (cp.async is ordered against every other
  // memory access, so one at a time would serialise those reads)
  __host__ __device__ static constexpr int batch(int per) {
    return per <= 8 ? per : per % 8 == 0 ? 8 : per % 5 == 0 ? 5 : per % 4 == 0 ? 4 : 1;
  }
  static constexpr int DK = D / 16;                  // k-steps of Q.K^T
  static constexpr int DT = D / 8;                   // n-tiles of O
  static constexpr int DTW = DT / DS;                // n-tiles of O per warp
  static_assert(DTW % 2 == 0, "P.V runs n-tile pairs");
  // byte offset of (row, dim) inside a K/V stage (dim a multiple of 8)
  __device__ static __forceinline__ uint32_t off(int row, int dim) {
    if (TMA) {
      const int c = (dim & 63) >> 3;
      return uint32_t((dim >> 6) * 8192 + row * 128 + ((c ^ (row & 7)) << 4));
    }
    return uint32_t((row * LD + dim) * 2);
  }
};

// two FP32 values as packed bf16 pairs hi, mid, lo with hi + mid + lo equal to
// each value exactly (x0 in the low halves): hi = bf16(x), mid = bf16(x - hi),
// lo = bf16(x - hi - mid); both differences are exact in FP32
__device__ __forceinline__ uint32_t cvt_bf16x2(float lo_half, float hi_half) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo_half, hi_half);
  return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ void split3(float x0, float x1, uint32_t& hi, uint32_t& mid,
                                       uint32_t& lo) {
  hi = cvt_bf16x2(x0, x1);
  const float r0 = x0 - __uint_as_float(hi << 16), r1 = x1 - __uint_as_float(hi & 0xFFFF0000u);
  mid = cvt_bf16x2(r0, r1);
  lo = cvt_bf16x2(r0 - __uint_as_float(mid << 16), r1 - __uint_as_float(mid & 0xFFFF0000u));
}

// 2^x (PTX ex2.approx.ftz: 2^-inf = +0, results below 2^-126 flush to zero)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 4 : 0)
               : "memory");
}
// two e4m3 codes (first in the low byte) -> their exact values
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t v) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(__nv_fp8x2_storage_t(v), __NV_E4M3);
  return __half22float2(__half2(h));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

struct AttnArgs {
  CUtensorMap tmK, tmV;      // bf16 caches as [pages*64, Hkv*D] (TMA path only)
  CUtensorMap tmQ;           // q as [T][Hq][D], boxes of 64 dims x G heads x 128/G rows (tcgen05 path)
  const uint16_t* q; int64_t q_stride;
  uint16_t* out; int64_t out_stride;
  int T, Hq, Hkv, G;
  const int32_t* row_seq; const int32_t* row_pos;
  const int32_t* qblocks;
  int fp8;
  const void* kc; const void* vc;
  const float* ks; const float* vs;
  const int32_t* bt; int max_pages;
  int kv_split;
  const int32_t* topk_idx; int64_t topk_stride; int topk;
  float scale;               // softmax scale times log2(e): scores in base-2 units
  float* ws_o; float* ws_ml; int nsplit_grid;
  int* err;
};

// Number of splits that hold keys of a row (fixed per row).
__device__ __forceinline__ int row_splits(const AttnArgs& a, int pos) {
  return a.topk_idx ? (a.topk + a.kv_split - 1) / a.kv_split : pos / a.kv_split + 1;
}

// A dense row's position must lie inside the grid's splits (position + 1 <=
// max_ctx rounded up to whole splits) and inside its block-table row.  A row
// outside either bound raises kErrBadIndex, has its output set to NaN and
// takes no part in the loads, the partials or the merge.
__device__ __forceinline__ bool row_pos_ok(const AttnArgs& a, int pos) {
  if (pos < 0) return false;
  if (a.topk_idx) return true;
  return pos < a.nsplit_grid * a.kv_split && pos < a.max_pages * kTile;
}

// The block's largest valid position (rows of a block are one sequence).
// Rows whose position is out of bounds are reported (split 0) and their
// output set to NaN; they take no part in the loads, the partials or the
// merge.  One row per thread, so the positions load in parallel.
template <int D>
__device__ __forceinline__ int block_maxpos(const AttnArgs& a, int r0, int nr, int h, int split,
                                            int* s_max) {
  if (threadIdx.x == 0) *s_max = -1;
  __syncthreads();
  for (int r = threadIdx.x; r < nr; r += blockDim.x) {
    const int p = a.row_pos[r0 + r];
    if (row_pos_ok(a, p)) {
      atomicMax(s_max, p);
    } else if (split == 0) {
      raise_error(a.err, kErrBadIndex);
      uint16_t* dst = a.out + int64_t(r0 + r) * a.out_stride + int64_t(h * a.G) * D;
      for (int i = 0; i < a.G * D; ++i) dst[i] = 0x7FC0;  // bf16 NaN
    }
  }
  __syncthreads();
  return *s_max;
}

// MINB: CTAs per SM the register allocation must allow (0: no bound)
template <int D, int NW, int ST, bool TMA, int DS, int MINB, bool F8>
__global__ void __launch_bounds__(NW * 32, MINB) attn_kernel(const __grid_constant__ AttnArgs a) {
  pdl_wait();     // stream predecessor done, its writes visible
  pdl_trigger();
  using Cfg = AttnCfg<D, NW, ST, TMA, DS, F8>;
  constexpr int LD = Cfg::LD, NV = Cfg::NV, NT = Cfg::NT, KVB = Cfg::KVB;
  constexpr int DTW = Cfg::DTW;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + Cfg::ALIGN - 1) & ~uintptr_t(Cfg::ALIGN - 1));
  constexpr int TST = Cfg::TST;
  uint8_t* sK = base;                                   // [TST] stages of KVB bytes
  uint8_t* sV = base + TST * KVB;
  uint16_t* sQ = reinterpret_cast<uint16_t*>(base + 2 * TST * KVB);
  uint8_t* sF8 = base + 2 * TST * KVB + Cfg::Q_BYTES;   // FP8 staging (F8 only)
  int32_t* sPos = reinterpret_cast<int32_t*>(sF8 + Cfg::F8_STAGE);  // [ST][64]
  // TMA: K of stage s completes on bars[s], V on bars[ST + s], so that K of
  // the next tile streams in while this tile's softmax and P.V run
  uint64_t* bars = reinterpret_cast<uint64_t*>(sPos + ST * kTile);                 // [2 ST]
  // thread loader: the cache slot of each key of the tile being loaded (-1: none)
  int32_t* sSlot = reinterpret_cast<int32_t*>(bars + 2 * ST);                       // [64]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int blk = blockIdx.x, h = blockIdx.y, split = blockIdx.z;
  const int r0 = a.qblocks[2 * blk], nr = a.qblocks[2 * blk + 1];
  const int nv = nr * a.G;
  const int seq = a.row_seq[r0];
  const bool sparse = a.topk_idx != nullptr;

  __shared__ int s_maxpos;
  const int maxpos = block_maxpos<D>(a, r0, nr, h, split, &s_maxpos);

  // key range of this split: [lo, hi) in positions (dense) or list indices (sparse)
  const int lo = split * a.kv_split;
  const int hi = sparse ? min(a.topk, lo + a.kv_split) : min(maxpos + 1, lo + a.kv_split);
  if (lo >= hi) return;  // uniform: nothing of this block lives in this split
  const int ntiles = (hi - lo + kTile - 1) / kTile;

  if (TMA && tid == 0) {
    for (int s = 0; s < 2 * ST; ++s) mbar_init(smem_u32(bars + s), 1);
    fence_barrier_init();
  }

  // ---- load Q (zero for vectors past nv)
  {
    constexpr int CPR = D / 8;  // 16-byte chunks per vector
    for (int i = tid; i < NV * CPR; i += NT) {
      const int v = i / CPR, c = i % CPR;
      uint4 val = make_uint4(0, 0, 0, 0);
      if (v < nv) {
        const int r = v / a.G, j = v % a.G;
        const uint16_t* src = a.q + int64_t(r0 + r) * a.q_stride + int64_t(h * a.G + j) * D;
        val = reinterpret_cast<const uint4*>(src)[c];
      }
      *reinterpret_cast<uint4*>(sQ + v * LD + c * 8) = val;
    }
  }

  // ---- tile loader (dense: the page of absolute tile t; sparse: listed keys)
  const int64_t kv_row = int64_t(a.Hkv) * D;  // elements between consecutive cache slots
  // TMA: K (which = 0) or V (which = 1) of the page of absolute tile t, by
  // thread 0, on that half's barrier of stage buf
  auto load_half = [&](int buf, int t, int which) {
    if (!TMA || tid != 0) return;
    const int tbase = lo + t * kTile;
    const uint32_t bar = smem_u32(bars + which * ST + buf);
    const int page = a.bt[int64_t(seq) * a.max_pages + tbase / kTile];
    uint8_t* dst = (which ? sV : sK) + buf * KVB;
    fence_proxy_async();  // earlier generic accesses to this buffer come first
    mbar_expect_tx(bar, KVB);
    tma_load_3d(smem_u32(dst), which ? &a.tmV : &a.tmK, bar, 0, page * kTile, h * (D / 64));
  };
  auto load_tile = [&](int buf, int t) {
    const int tbase = lo + t * kTile;
    if (TMA) {
      load_half(buf, t, 0);
      load_half(buf, t, 1);
      return;
    }
    int32_t* pos_buf = sPos + buf * kTile;
    for (int j = tid; j < kTile; j += NT) {
      int p;
      if (sparse) {
        const int li = tbase + j;
        p = li < hi ? a.topk_idx[int64_t(r0) * a.topk_stride + li] : -1;
        if (p >= a.max_pages * kTile) {   // a listed key outside the block table
          raise_error(a.err, kErrBadIndex);
          p = -1;
        }
      } else {
        p = tbase + j;
        if (p >= hi) p = -1;
      }
      pos_buf[j] = p;
      int sl = -1;
      if (p >= 0) {
        const int pg = a.bt[int64_t(seq) * a.max_pages + p / kTile];
        if (pg >= 0 && pg <= (INT_MAX - (kTile - 1)) / kTile)
          sl = pg * kTile + p % kTile;
        else
          raise_error(a.err, kErrBadIndex);   // a page index no slot number can hold
      }
      sSlot[j] = sl;
    }
    __syncthreads();
    uint8_t* dK = sK + (buf % TST) * KVB;
    uint8_t* dV = sV + (buf % TST) * KVB;
    if constexpr (!F8) {
      constexpr int CPR = D / 8;
      constexpr int PER = kTile * CPR * 2 / NT, GRP = Cfg::batch(PER);
      static_assert(kTile * CPR * 2 % NT == 0 && PER % GRP == 0, "copies per thread");
#pragma unroll
      for (int g0 = 0; g0 < PER; g0 += GRP) {
        int sl[GRP];
#pragma unroll
        for (int k = 0; k < GRP; ++k) sl[k] = sSlot[((tid + (g0 + k) * NT) % (kTile * CPR)) / CPR];
#pragma unroll
        for (int k = 0; k < GRP; ++k) {
          const int i = tid + (g0 + k) * NT;
          const int which = i / (kTile * CPR);
          const int rem = i % (kTile * CPR);
          const int j = rem / CPR, c = rem % CPR;
          const uint16_t* gp = static_cast<const uint16_t*>(which ? a.vc : a.kc);
          if (sl[k] >= 0) gp += int64_t(sl[k]) * kv_row + int64_t(h) * D + c * 8;
          cp_async16(smem_u32((which ? dV : dK) + Cfg::off(j, c * 8)), gp, sl[k] >= 0);
        }
      }
    } else {
      // raw codes (16 per copy) and scales of the tile's keys into the
      // staging area; missing keys read as zero codes and scales
      uint8_t* stg = sF8;
      constexpr int CPR = D / 16;
      constexpr int PER = kTile * CPR * 2 / NT, GRP = Cfg::batch(PER);
      static_assert(kTile * CPR * 2 % NT == 0 && PER % GRP == 0, "copies per thread");
#pragma unroll
      for (int g0 = 0; g0 < PER; g0 += GRP) {
        int sl[GRP];
#pragma unroll
        for (int k = 0; k < GRP; ++k) sl[k] = sSlot[((tid + (g0 + k) * NT) % (kTile * CPR)) / CPR];
#pragma unroll
        for (int k = 0; k < GRP; ++k) {
          const int i = tid + (g0 + k) * NT;
          const int which = i / (kTile * CPR);
          const int rem = i % (kTile * CPR);
          const int j = rem / CPR, c = rem % CPR;
          const uint8_t* gp = static_cast<const uint8_t*>(which ? a.vc : a.kc);
          if (sl[k] >= 0) gp += int64_t(sl[k]) * kv_row + int64_t(h) * D + c * 16;
          cp_async16(smem_u32(stg + which * kTile * D + j * D + c * 16), gp, sl[k] >= 0);
        }
      }
      constexpr int SPER = 2 * kTile / NT;
      static_assert(2 * kTile % NT == 0, "scale copies per thread");
      int sl[SPER];
#pragma unroll
      for (int k = 0; k < SPER; ++k) sl[k] = sSlot[(tid + k * NT) % kTile];
#pragma unroll
      for (int k = 0; k < SPER; ++k) {
        const int i = tid + k * NT;
        const float* gp = i / kTile ? a.vs : a.ks;
        if (sl[k] >= 0) gp += int64_t(sl[k]) * a.Hkv + h;
        cp_async4(smem_u32(stg + Cfg::F8_CODES + i * 4), gp, sl[k] >= 0);
      }
    }
  };
  // FP8: the staged codes of stage buf -> bf16 K/V tiles, x = bf16(float(code) * s)
  auto dequant_stage = [&](int buf) {
    const uint8_t* stg = sF8;
    const float* scl = reinterpret_cast<const float*>(stg + Cfg::F8_CODES);
    constexpr int CPR = D / 16;
    constexpr int PER = kTile * CPR * 2 / NT, GRP = Cfg::batch(PER);
    // a group's codes and scales are read before any of its stores
#pragma unroll
    for (int g0 = 0; g0 < PER; g0 += GRP) {
      uint4 cvs[GRP];
      float scs[GRP];
#pragma unroll
      for (int k = 0; k < GRP; ++k) {
        const int i = tid + (g0 + k) * NT;
        const int which = i / (kTile * CPR);
        const int rem = i % (kTile * CPR);
        const int j = rem / CPR, c = rem % CPR;
        cvs[k] = *reinterpret_cast<const uint4*>(stg + which * kTile * D + j * D + c * 16);
        scs[k] = scl[which * kTile + j];
      }
#pragma unroll
      for (int k = 0; k < GRP; ++k) {
        const int i = tid + (g0 + k) * NT;
        const int which = i / (kTile * CPR);
        const int rem = i % (kTile * CPR);
        const int j = rem / CPR, c = rem % CPR;
        const uint4 cv = cvs[k];
        const float sc = scs[k];
        const uint32_t w[4] = {cv.x, cv.y, cv.z, cv.w};
        uint32_t packed[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 f01 = e4m3x2_to_float2(uint16_t(w[q] & 0xFFFFu));
          const float2 f23 = e4m3x2_to_float2(uint16_t(w[q] >> 16));
          packed[2 * q] = pack_bf2(f01.x * sc, f01.y * sc);
          packed[2 * q + 1] = pack_bf2(f23.x * sc, f23.y * sc);
        }
        uint8_t* dst = (which ? sV : sK) + (buf % TST) * KVB;
        *reinterpret_cast<uint4*>(dst + Cfg::off(j, c * 16)) =
            make_uint4(packed[0], packed[1], packed[2], packed[3]);
        *reinterpret_cast<uint4*>(dst + Cfg::off(j, c * 16 + 8)) =
            make_uint4(packed[4], packed[5], packed[6], packed[7]);
      }
    }
  };

  // per-thread rows: g and g+8 of the warp's 16 vectors (vw: their group);
  // O n-tiles dt0 .. dt0+DTW-1 of the head dimension
  const int vw = warp / DS;
  const int dt0 = (warp % DS) * DTW;
  const int g = lane >> 2, cq = lane & 3;
  int vpos[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int v = vw * 16 + g + 8 * i;
    vpos[i] = v < nv ? a.row_pos[r0 + v / a.G] : -1;
    if (!row_pos_ok(a, vpos[i])) vpos[i] = -1;   // sees no key; output already NaN
  }

  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  float acc[DTW][4];
#pragma unroll
  for (int i = 0; i < DTW; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

  __syncthreads();  // Q stored, barriers initialised
  // prologue.  TMA: tiles 0 .. ST-1 in flight, a stage is refilled right
  // after the tile that used it.  Threads: tiles 0 .. ST-2 in flight (one
  // cp.async group each, even if empty), refilled at the top of the loop.
#pragma unroll
  for (int s0 = 0; s0 < (TMA ? ST : ST - 1); ++s0) {
    if (s0 < ntiles) load_tile(s0, s0);
    if (!TMA) cp_async_commit();
  }

  // Q fragments (A operand), loaded once
  uint32_t qf[Cfg::DK][4];
  {
    const uint32_t qbase = smem_u32(sQ + (vw * 16 + (lane & 15)) * LD + (lane >> 4) * 8);
#pragma unroll
    for (int kk = 0; kk < Cfg::DK; ++kk)
      ldsm_x4(qbase + kk * 32, qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
  }

  for (int t = 0; t < ntiles; ++t) {
    const int buf = t % ST;
    const int tbase = lo + t * kTile;
    if (TMA) {
      mbar_wait(smem_u32(bars + buf), (t / ST) & 1, a.err);   // K of tile t
    } else {
      cp_async_wait<ST - 2>();  // tile t has landed
    }
    __syncthreads();
    if constexpr (F8) {
      dequant_stage(buf);
      __syncthreads();
    }
    if (!TMA) {
      // refill the stage that tile t-1 used (its compute ended at the last sync)
      if (t + ST - 1 < ntiles) load_tile((t + ST - 1) % ST, t + ST - 1);
      cp_async_commit();
    }
    // a warp with no live vector only takes part in the loads and barriers
    const bool live = vw * 16 < nv;
    const uint32_t tK = smem_u32(sK + (buf % TST) * KVB);
    const uint32_t tV = smem_u32(sV + (buf % TST) * KVB);
    const int32_t* tP = sPos + buf * kTile;

    // S = Q . K^T  (16 x 64 per warp)
    float s[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
    if (DS > 1) {
      // D split: a group's warps share one S tile.  Warp w of the group
      // computes its 64 / DS keys (the same ascending-k chain per element as
      // one warp computing all of them) and publishes them; every warp of
      // the group then reads the whole tile.
      constexpr int NPW = 4 / (DS > 1 ? DS : 1);   // n-tile pairs per warp
      const int wg = warp % DS;                     // the warp's place in its group
      float sw[2 * NPW][4];
#pragma unroll
      for (int i = 0; i < 2 * NPW; ++i) sw[i][0] = sw[i][1] = sw[i][2] = sw[i][3] = 0.f;
      if (live) {
#pragma unroll
        for (int kk = 0; kk < Cfg::DK; ++kk) {
          uint32_t kf[NPW][4];
#pragma unroll
          for (int j = 0; j < NPW; ++j) {
            const int key = (wg * NPW + j) * 16 + (lane & 7) + (lane >> 4) * 8;
            const int dim = kk * 16 + ((lane >> 3) & 1) * 8;
            ldsm_x4(tK + Cfg::off(key, dim), kf[j][0], kf[j][1], kf[j][2], kf[j][3]);
          }
#pragma unroll
          for (int j = 0; j < NPW; ++j) {
            mma_bf16(sw[2 * j], qf[kk], kf[j][0], kf[j][1]);
            mma_bf16(sw[2 * j + 1], qf[kk], kf[j][2], kf[j][3]);
          }
        }
        float4* sS = reinterpret_cast<float4*>(sQ) + vw * 8 * 32;
#pragma unroll
        for (int i = 0; i < 2 * NPW; ++i)
          sS[(wg * 2 * NPW + i) * 32 + lane] = make_float4(sw[i][0], sw[i][1], sw[i][2], sw[i][3]);
      }
      __syncthreads();   // S published; every warp is also done with K of tile t
      if (live) {
        const float4* sS = reinterpret_cast<const float4*>(sQ) + vw * 8 * 32;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          const float4 v = sS[nt * 32 + lane];
          s[nt][0] = v.x; s[nt][1] = v.y; s[nt][2] = v.z; s[nt][3] = v.w;
        }
      }
    } else if (live) {
    // per k-step: all fragment loads first, then the MMAs (independent
    // accumulators back to back; each accumulator still sees ascending k)
#pragma unroll
    for (int kk = 0; kk < Cfg::DK; ++kk) {
      uint32_t kf[4][4];
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        const int key = np * 16 + (lane & 7) + (lane >> 4) * 8;
        const int dim = kk * 16 + ((lane >> 3) & 1) * 8;
        ldsm_x4(tK + Cfg::off(key, dim), kf[np][0], kf[np][1], kf[np][2], kf[np][3]);
      }
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        mma_bf16(s[2 * np], qf[kk], kf[np][0], kf[np][1]);
        mma_bf16(s[2 * np + 1], qf[kk], kf[np][2], kf[np][3]);
      }
    }
    }  // live
    if (TMA) {
      if (DS == 1) __syncthreads();                     // every warp is done with K of tile t
      if (t + ST < ntiles) load_half(buf, t + ST, 0);   // its buffer takes K of tile t+ST
    }
    if (live) {
    // mask, online softmax.  A dense tile that every live row of the warp sees
    // whole needs no per-element test (the result is the same either way).
    float mx[2] = {-INFINITY, -INFINITY};
    const int row_lo = min(vpos[0] < 0 ? INT_MAX : vpos[0], vpos[1] < 0 ? INT_MAX : vpos[1]);
    const bool whole = !sparse && tbase + kTile <= hi &&
                       __all_sync(0xffffffffu, row_lo >= tbase + kTile - 1);
    if (whole) {
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i = e >> 1;
          const float x = vpos[i] >= 0 ? s[nt][e] * a.scale : -INFINITY;
          s[nt][e] = x;
          mx[i] = fmaxf(mx[i], x);
        }
      }
    } else {
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i = e >> 1;
          const int col = nt * 8 + 2 * cq + (e & 1);
          const int kp = sparse ? tP[col] : (tbase + col < hi ? tbase + col : -1);
          const bool vis = kp >= 0 && kp <= vpos[i];
          const float x = vis ? s[nt][e] * a.scale : -INFINITY;
          s[nt][e] = x;
          mx[i] = fmaxf(mx[i], x);
        }
      }
    }
    float alpha[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 1));
      mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 2));
      const float mn = mx[i] > m[i] + kLazy ? mx[i] : m[i];
      alpha[i] = mn == m[i] ? 1.f : ex2(m[i] - mn);
      m[i] = mn;
    }
    // p = exp(x - m) in FP32, kept in s; the denominator sums these FP32 p
    // (per thread and row: one chain over the keys of each tile half, key
    // ascending, the two added; then the quad's four sums as (0+1) + (2+3))
    float rs[2] = {0.f, 0.f}, rb[2] = {0.f, 0.f};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = e >> 1;
        const float pe = (m[i] == -INFINITY) ? 0.f : ex2(s[nt][e] - m[i]);
        s[nt][e] = pe;
        if (nt < 4) rs[i] += pe; else rb[i] += pe;
      }
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      rs[i] = rs[i] + rb[i];
      rs[i] += __shfl_xor_sync(0xffffffffu, rs[i], 1);
      rs[i] += __shfl_xor_sync(0xffffffffu, rs[i], 2);
      l[i] = __fmaf_rn(l[i], alpha[i], rs[i]);
    }
    // rescale only when some row's max moved (a factor of exactly 1 is a no-op)
    if (!__all_sync(0xffffffffu, alpha[0] == 1.f && alpha[1] == 1.f)) {
#pragma unroll
      for (int dt = 0; dt < DTW; ++dt) {
        acc[dt][0] *= alpha[0];
        acc[dt][1] *= alpha[0];
        acc[dt][2] *= alpha[1];
        acc[dt][3] *= alpha[1];
      }
    }
    }  // live
    if (TMA) {
      mbar_wait(smem_u32(bars + ST + buf), (t / ST) & 1, a.err);   // V of tile t
      // slots past the split's end in its last page hold no key of this
      // sequence: zero their V rows (P is 0 there, and 0 * stale must be 0)
      const int first_bad = hi - tbase;
      if (first_bad < kTile) {
        for (int i = tid; i < (kTile - first_bad) * (D / 8); i += NT) {
          const int j = first_bad + i / (D / 8), c = i % (D / 8);
          *reinterpret_cast<uint4*>(sV + buf * KVB + Cfg::off(j, c * 8)) = make_uint4(0, 0, 0, 0);
        }
      }
      __syncthreads();
    }
    if (live) {
    // O += P . V with P = hi + mid + lo: hi = bf16(p), mid = bf16(p - hi),
    // lo = bf16(p - hi - mid).  Both differences are exact in FP32 and the
    // three parts hold p's 24 significant bits, so the products sum the FP32
    // p against exact bf16 V.
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      // A fragment order: (row g, k 0-7), (row g+8, k 0-7), (row g, k 8-15), (row g+8, k 8-15)
      uint32_t af[4], am[4], al[4];
#pragma unroll
      for (int hi2 = 0; hi2 < 2; ++hi2) {
#pragma unroll
        for (int pr = 0; pr < 2; ++pr) {
          const float p0 = s[2 * ks + hi2][2 * pr], p1 = s[2 * ks + hi2][2 * pr + 1];
          split3(p0, p1, af[hi2 * 2 + pr], am[hi2 * 2 + pr], al[hi2 * 2 + pr]);
        }
      }
      // V fragments of this k-step first, then every accumulator's hi MMA,
      // then every mid MMA, then every lo MMA (per accumulator hi, mid, lo,
      // ks ascending)
      constexpr int DPS = DTW / 2;
      uint32_t vf[DPS][4];
#pragma unroll
      for (int dp = 0; dp < DPS; ++dp) {
        const int key = ks * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int dim = (dt0 / 2 + dp) * 16 + (lane >> 4) * 8;
        ldsm_x4_t(tV + Cfg::off(key, dim), vf[dp][0], vf[dp][1], vf[dp][2], vf[dp][3]);
      }
#pragma unroll
      for (int dp = 0; dp < DPS; ++dp) {
        mma_bf16(acc[2 * dp], af, vf[dp][0], vf[dp][1]);
        mma_bf16(acc[2 * dp + 1], af, vf[dp][2], vf[dp][3]);
      }
#pragma unroll
      for (int dp = 0; dp < DPS; ++dp) {
        mma_bf16(acc[2 * dp], am, vf[dp][0], vf[dp][1]);
        mma_bf16(acc[2 * dp + 1], am, vf[dp][2], vf[dp][3]);
      }
#pragma unroll
      for (int dp = 0; dp < DPS; ++dp) {
        mma_bf16(acc[2 * dp], al, vf[dp][0], vf[dp][1]);
        mma_bf16(acc[2 * dp + 1], al, vf[dp][2], vf[dp][3]);
      }
    }
    }  // live
    __syncthreads();
    // TMA: every warp is done with V of tile t: its buffer takes V of tile t+ST
    if (TMA && t + ST < ntiles) load_half(buf, t + ST, 1);
  }

  // ---- epilogue: single-split rows write the final output, others partials
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int v = vw * 16 + g + 8 * i;
    if (v >= nv || vpos[i] < 0) continue;
    const int row = r0 + v / a.G;
    const int head = h * a.G + v % a.G;
    const int ns = row_splits(a, vpos[i]);
    if (split >= ns) continue;
    if (ns == 1) {
      const float inv_l = l[i] > 0.f ? 1.0f / l[i] : 0.f;
      uint16_t* dst = a.out + int64_t(row) * a.out_stride + int64_t(head) * D;
#pragma unroll
      for (int dt = 0; dt < DTW; ++dt) {
        const float o0 = acc[dt][2 * i] * inv_l + 0.0f;
        const float o1 = acc[dt][2 * i + 1] * inv_l + 0.0f;
        *reinterpret_cast<uint32_t*>(dst + (dt0 + dt) * 8 + 2 * cq) = pack_bf2(o0, o1);
      }
    } else {
      const int64_t slot = (int64_t(row) * a.Hq + head) * a.nsplit_grid + split;
      float* wo = a.ws_o + slot * D;
#pragma unroll
      for (int dt = 0; dt < DTW; ++dt)
        *reinterpret_cast<float2*>(wo + (dt0 + dt) * 8 + 2 * cq) =
            make_float2(acc[dt][2 * i], acc[dt][2 * i + 1]);
      if (cq == 0 && dt0 == 0) {
        a.ws_ml[2 * slot] = m[i];
        a.ws_ml[2 * slot + 1] = l[i];
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Prefill attention on tcgen05.  A CTA takes up to 128 query vectors of one
// query block and one KV head (the M = 128 rows of the MMA) over one KV split.
// Per 64-key tile: S = Q . K^T into one of two TMEM buffers (K steps of 16
// over the head dimension, ascending); the online softmax, doing attn_kernel's
// FP32 operations in attn_kernel's order element for element; P's three bf16
// parts into one of two TMEM buffers; and O += P . V accumulated in TMEM with
// P read from TMEM as the A operand (per 16-key step hi, mid, lo).  One K = 16 tcgen05 MMA rounds exactly
// as one mma.sync m16n8k16 on the same operands and accumulator (checked bit
// for bit on GB300, including wide exponent ranges and cancellation), so a
// vector's output has the same bits whichever kernel runs it: prefill rows
// here, decode rows in attn_kernel.
// V is read in place from its TMA tile ([key][dim], 128-byte swizzled) as an
// MN-major operand.  O starts at +0 in TMEM and every P.V MMA accumulates, as
// attn_kernel's register accumulators do.
// Warps: 0 = TMA producer, 1 = MMA issuer and TMEM owner, 2..9 = softmax and
// epilogue.  Softmax warp w reads TMEM lane quarter w % 4 (vector
// 32 * (w % 4) + lane) and tile half hf = (w - 2) / 4: keys [32 hf, 32 hf + 32)
// of S, the same half of P, and head dimensions [hf D/2, (hf + 1) D/2) of O.
// The two warps of a quarter exchange their row maxima and their denominator
// chains through shared memory, with one named barrier per tile.
template <int D>
struct TcCfg {
  static constexpr int NV = 128;                  // query vectors per CTA (MMA rows)
  static constexpr int PANEL = NV * 128;          // one 64-dim panel of Q
  static constexpr int Q_BYTES = NV * D * 2;
  static constexpr int KV_BYTES = kTile * D * 2;  // one K or V tile
  static constexpr int STK = 3, STV = 3;
  static constexpr int NBARS = 21 + 4;   // pipeline barriers + one exchange per lane quarter
  // row exchange between the two halves: [2 tiles][2 halves][NV] maxima and
  // [2 tiles][2 halves][4 chains][NV] denominator chains
  static constexpr int XCH_BYTES = (2 * 2 * NV + 2 * 2 * 4 * NV) * 4;
  static constexpr int SMEM = 1024 + Q_BYTES + (STK + STV) * KV_BYTES + XCH_BYTES + NBARS * 8 + 16;
  // TMEM: S double buffer (2 x 64 columns), O (D), and P as the A operand of
  // P.V: two buffers (the softmax of tile t+1 fills one while P.V of tile t
  // reads the other) of three parts, each 64 bf16 keys packed in 32 columns
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t O_COL = 2 * kTile;
  static constexpr uint32_t P_COL = O_COL + 128;
  static_assert(P_COL + 6 * 32 <= TMEM_COLS, "TMEM budget");
  static constexpr int SOFT_WARPS = 8;
  static constexpr int THREADS = 64 + 32 * SOFT_WARPS;
};

template <int D>
__global__ void __launch_bounds__(TcCfg<D>::THREADS, 1)
    attn_tc_kernel(const __grid_constant__ AttnArgs a) {
  pdl_wait();     // stream predecessor done, its writes visible
  pdl_trigger();
  using Cfg = TcCfg<D>;
  constexpr int KVB = Cfg::KV_BYTES, STK = Cfg::STK, STV = Cfg::STV;
  constexpr int NV = Cfg::NV, SOFTW = Cfg::SOFT_WARPS;
  enum { Q_FULL = 0, K_FULL = 1, K_EMPTY = K_FULL + STK, V_FULL = K_EMPTY + STK,
         V_EMPTY = V_FULL + STV, S_FULL = V_EMPTY + STV, S_EMPTY = S_FULL + 2, P_FULL = S_EMPTY + 2,
         PV_DONE = P_FULL + 2, XCH = PV_DONE + 2 };
  static_assert(XCH + 4 == Cfg::NBARS, "barrier count");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sQ = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  uint8_t* sK = sQ + Cfg::Q_BYTES;
  uint8_t* sV = sK + STK * KVB;
  float* xmax = reinterpret_cast<float*>(sV + STV * KVB);   // [2][2][NV]
  float* xsum = xmax + 2 * 2 * NV;                        // [2][2][4][NV]
  uint64_t* bars = reinterpret_cast<uint64_t*>(xsum + 2 * 2 * 4 * NV);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Cfg::NBARS);
  auto bar = [&](int i) { return smem_u32(bars + i); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int blk = blockIdx.x, h = blockIdx.y, split = blockIdx.z;
  const int r0 = a.qblocks[2 * blk], nr = a.qblocks[2 * blk + 1];
  const int nv = nr * a.G;
  const int seq = a.row_seq[r0];

  __shared__ int s_maxpos;
  const int maxpos = block_maxpos<D>(a, r0, nr, h, split, &s_maxpos);
  const int lo = split * a.kv_split;
  const int hi = min(maxpos + 1, lo + a.kv_split);
  if (lo >= hi) return;  // uniform: nothing of this block lives in this split
  const int ntiles = (hi - lo + kTile - 1) / kTile;

  if (tid == 0) {
    mbar_init(bar(Q_FULL), 1);
    for (int s = 0; s < STK; ++s) {
      mbar_init(bar(K_FULL + s), 1);
      mbar_init(bar(K_EMPTY + s), 1);
    }
    for (int s = 0; s < STV; ++s) {
      mbar_init(bar(V_FULL + s), 1);
      mbar_init(bar(V_EMPTY + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(S_FULL + s), 1);
      mbar_init(bar(S_EMPTY + s), SOFTW);
      mbar_init(bar(P_FULL + s), SOFTW);
      mbar_init(bar(PV_DONE + s), 1);
    }
    for (int q = 0; q < 4; ++q) mbar_init(bar(XCH + q), 2);   // one arrival per half
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
  int issued_k = 0, issued_v = 0;
  if (warp == 0) {
    // ------------------------------------------------------------ producer --
    if (lane == 0) {
      tma_prefetch_desc(&a.tmQ);
      tma_prefetch_desc(&a.tmK);
      tma_prefetch_desc(&a.tmV);
      mbar_expect_tx(bar(Q_FULL), Cfg::Q_BYTES);
#pragma unroll
      for (int hh = 0; hh < D / 64; ++hh)
        tma_load_3d(smem_u32(sQ + hh * Cfg::PANEL), &a.tmQ, bar(Q_FULL), hh * 64, h * a.G, r0);
      // K runs two tiles ahead of V (S(t+2) is issued before P.V(t)), so a K
      // load never queues behind a V stage that P.V still holds
      auto page_of = [&](int t) { return a.bt[int64_t(seq) * a.max_pages + (lo + t * kTile) / kTile]; };
      auto load_k = [&](int t) -> bool {
        const int sk = t % STK;
        if (t >= STK && !mbar_wait(bar(K_EMPTY + sk), ((t / STK) - 1) & 1, a.err)) return false;
        mbar_expect_tx(bar(K_FULL + sk), KVB);
        tma_load_3d(smem_u32(sK + sk * KVB), &a.tmK, bar(K_FULL + sk), 0, page_of(t) * kTile,
                    h * (D / 64));
        ++issued_k;
        return true;
      };
      bool ok = load_k(0) && (ntiles < 2 || load_k(1));
      for (int t = 0; t < ntiles && ok; ++t) {
        if (t + 2 < ntiles && !(ok = load_k(t + 2))) break;
        const int sv = t % STV;
        if (t >= STV && !mbar_wait(bar(V_EMPTY + sv), ((t / STV) - 1) & 1, a.err)) break;
        mbar_expect_tx(bar(V_FULL + sv), KVB);
        tma_load_3d(smem_u32(sV + sv * KVB), &a.tmV, bar(V_FULL + sv), 0, page_of(t) * kTile,
                    h * (D / 64));
        ++issued_v;
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA --
    if (lane == 0) {
      constexpr uint32_t idS = idesc_mma(1u, Cfg::NV, kTile);
      constexpr uint32_t idO = idesc_mma(1u, Cfg::NV, D) | (1u << 16);   // B = V, MN-major
      const uint32_t q0 = smem_u32(sQ);
      // S(t) = Q . K(t)^T into buffer t % 2 (free once the softmax of t-2 read it)
      auto issue_s = [&](int t) -> bool {
        const int sb = t & 1, sk = t % STK;
        if (t >= 2 && !mbar_wait(bar(S_EMPTY + sb), ((t - 2) >> 1) & 1, a.err)) return false;
        if (!mbar_wait(bar(K_FULL + sk), (t / STK) & 1, a.err)) return false;
        tc_fence_after();
        const uint32_t k0 = smem_u32(sK + sk * KVB);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_f16(tmem + sb * kTile, sdesc_k_sw128(q0 + (kk >> 2) * Cfg::PANEL + (kk & 3) * 32),
                   sdesc_k_sw128(k0 + (kk >> 2) * 8192 + (kk & 3) * 32), idS, kk > 0 ? 1u : 0u);
        umma_commit(bar(K_EMPTY + sk));
        umma_commit(bar(S_FULL + sb));
        return true;
      };
      // S runs two tiles ahead of P.V: S(t+2) enters the pipe as soon as the
      // softmax of tile t has read S(t) from the same buffer, ahead of
      // P.V(t), so a tile's softmax never waits behind a P.V
      bool ok = mbar_wait(bar(Q_FULL), 0, a.err) && issue_s(0) && (ntiles < 2 || issue_s(1));
      for (int t = 0; t < ntiles && ok; ++t) {
        if (t + 2 < ntiles && !(ok = issue_s(t + 2))) break;
        // O += P(t) . V(t): per 16-key step the hi, mid and lo parts
        const int pb = t & 1;
        if (!(ok = mbar_wait(bar(P_FULL + pb), (t >> 1) & 1, a.err))) break;
        tc_fence_after();
        const int sv = t % STV;
        const uint32_t v0 = smem_u32(sV + sv * KVB), p0 = tmem + Cfg::P_COL + pb * 3 * 32;
#pragma unroll
        for (int ks = 0; ks < kTile / 16; ++ks) {
          const uint64_t vd = sdesc_mn_sw128(v0 + ks * 2048, 8192, 1024);
#pragma unroll
          for (int part = 0; part < 3; ++part)
            umma_f16_ts(tmem + Cfg::O_COL, p0 + part * 32 + ks * 8, vd, idO, 1u);
        }
        umma_commit(bar(V_EMPTY + sv));
        umma_commit(bar(PV_DONE + pb));
      }
    }
  } else {
    // ------------------------------------------------- softmax, epilogue --
    const int qtr = warp & 3, hf = (warp - 2) >> 2;
    const int v = qtr * 32 + lane;
    const uint32_t lane_off = uint32_t(qtr * 32) << 16;
    constexpr int DH = D / 2;                      // O columns of one half
    const uint32_t o_col = Cfg::O_COL + hf * DH;
    const uint32_t xbar = bar(XCH + qtr);   // the quarter's exchange
    int vpos = v < nv ? a.row_pos[r0 + v / a.G] : -1;
    if (!row_pos_ok(a, vpos)) vpos = -1;   // sees no key; output already NaN
    float m = -INFINITY, l = 0.f, alpha_prev = 1.f;
    float cs[4] = {0.f, 0.f, 0.f, 0.f};    // this half's denominator chains of the last tile
    {
      uint32_t z[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) z[i] = 0u;
#pragma unroll
      for (int c = 0; c < DH / 32; ++c) tmem_st32(tmem + o_col + lane_off + c * 32, z);
      tmem_st_wait();
    }
    // rs of a tile from both halves' chains: c = A_c + B_c, (c0 + c1) + (c2 + c3)
    auto tile_sum = [&](int slot) {
      float c[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float other = xsum[((slot * 2 + (hf ^ 1)) * 4 + k) * NV + v];
        c[k] = hf == 0 ? cs[k] + other : other + cs[k];
      }
      return (c[0] + c[1]) + (c[2] + c[3]);
    };
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
      const int sb = t & 1, tbase = lo + t * kTile, slot = t & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(S_FULL + sb), (t >> 1) & 1, a.err))) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[32];
      {
        uint32_t r[32];
        tmem_ld32(tmem + sb * kTile + hf * 32 + lane_off, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) s[i] = __uint_as_float(r[i]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(S_EMPTY + sb));
      // mask: key tbase + j is seen when it lies below hi and at or before
      // vpos; this half holds keys j = 32 hf + i
      const int lim = (vpos < 0 ? -1 : min(hi - 1, vpos) - tbase) - hf * 32;
      float m8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) m8[i] = -INFINITY;
      if (lim >= 31) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          s[i] = s[i] * a.scale;
          m8[i & 7] = fmaxf(m8[i & 7], s[i]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float x = i <= lim ? s[i] * a.scale : -INFINITY;
          s[i] = x;
          m8[i & 7] = fmaxf(m8[i & 7], x);
        }
      }
      // the row's max over both halves (exact in any order)
      xmax[(slot * 2 + hf) * NV + v] = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                             fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      __syncwarp();
      if (lane == 0) mbar_arrive(xbar);
      if (!__all_sync(0xffffffffu, mbar_wait(xbar, t & 1, a.err))) {
        ok = false;
        break;
      }
      const float mx = fmaxf(xmax[(slot * 2) * NV + v], xmax[(slot * 2 + 1) * NV + v]);
      // the denominator of tile t-1, now that the other half's chains are in
      if (t > 0) l = __fmaf_rn(l, alpha_prev, tile_sum(slot ^ 1));
      const float mn = mx > m + kLazy ? mx : m;
      const float alpha = mn == m ? 1.f : ex2(m - mn);
      m = mn;
      // p = 2^(x - m) in FP32, kept in s (no key seen yet: every x is -inf and
      // p = 0); chain c sums keys 8 nt + 2c, 8 nt + 2c + 1 of this half, nt
      // ascending (attn_kernel: each thread's chain over one tile half)
      const float mm = (m == -INFINITY) ? 0.f : m;
#pragma unroll
      for (int k = 0; k < 4; ++k) cs[k] = 0.f;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int i = nt * 8 + 2 * c;
          s[i] = ex2(s[i] - mm);
          s[i + 1] = ex2(s[i + 1] - mm);
          cs[c] += s[i];
          cs[c] += s[i + 1];
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) xsum[((slot * 2 + hf) * 4 + k) * NV + v] = cs[k];
      alpha_prev = alpha;
      // P buffer t % 2 is free once P.V of tile t-2 is done
      const int pb = t & 1;
      if (t >= 2 &&
          !__all_sync(0xffffffffu, mbar_wait(bar(PV_DONE + pb), ((t - 2) >> 1) & 1, a.err))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int sv = t % STV;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(V_FULL + sv), (t / STV) & 1, a.err))) {
        ok = false;
        break;
      }
      // slots past the split's end in its last page hold no key of this
      // sequence: zero their V rows (P is 0 there, and 0 * stale must be 0)
      const int first_bad = hi - tbase;
      if (first_bad < kTile) {
        uint8_t* vt = sV + sv * KVB;
        for (int i = tid - 64; i < (kTile - first_bad) * (D / 8); i += 32 * SOFTW) {
          const int j = first_bad + i / (D / 8), c = i % (D / 8);
          const int dim = c * 8;
          *reinterpret_cast<uint4*>(vt + (dim >> 6) * 8192 + j * 128 +
                                    ((((dim & 63) >> 3) ^ (j & 7)) << 4)) = make_uint4(0, 0, 0, 0);
        }
      }
      // rescale this half of O when a row's max moved (a factor of exactly 1
      // is a no-op; before the first P.V, O is +0 and stays +0), after P.V of
      // tile t-1
      if (t > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        if (!__all_sync(0xffffffffu,
                        mbar_wait(bar(PV_DONE + (pb ^ 1)), ((t - 1) >> 1) & 1, a.err))) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < DH / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(tmem + o_col + lane_off + c * 32, r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
          tmem_st32(tmem + o_col + lane_off + c * 32, r);
        }
        tmem_st_wait();
      }
      // this half of P's parts into TMEM: lane v, column 16 hf + c holds keys
      // 32 hf + 2c (low half) and 32 hf + 2c + 1
      {
        uint32_t ph[16], pm[16], pl[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) split3(s[2 * c], s[2 * c + 1], ph[c], pm[c], pl[c]);
        const uint32_t pc = tmem + Cfg::P_COL + pb * 3 * 32 + hf * 16 + lane_off;
        tmem_st16(pc, ph);
        tmem_st16(pc + 32, pm);
        tmem_st16(pc + 64, pl);
        tmem_st_wait();
      }
      if (first_bad < kTile) fence_proxy_async();   // zeroed V rows, for the MMA
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(P_FULL + pb));
    }
    // the last tile's denominator (its chains cross once more)
    if (ok) {
      __syncwarp();
      if (lane == 0) mbar_arrive(xbar);
      if (!__all_sync(0xffffffffu, mbar_wait(xbar, ntiles & 1, a.err))) ok = false;
    }
    if (ok) l = __fmaf_rn(l, alpha_prev, tile_sum((ntiles - 1) & 1));
    // ---- epilogue: single-split rows write the final output, others partials
    if (ok && !__all_sync(0xffffffffu, mbar_wait(bar(PV_DONE + ((ntiles - 1) & 1)),
                                                 ((ntiles - 1) >> 1) & 1, a.err)))
      ok = false;
    tc_fence_after();
    if (ok) {
      const int row = r0 + v / a.G, head = h * a.G + v % a.G;
      const int ns = (v < nv && vpos >= 0) ? row_splits(a, vpos) : 0;
      const bool mine = split < ns;
      const float inv_l = l > 0.f ? 1.0f / l : 0.f;
      const int64_t slot = (int64_t(row) * a.Hq + head) * a.nsplit_grid + split;
#pragma unroll
      for (int c = 0; c < DH / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem + o_col + lane_off + c * 32, r);   // warp-collective
        tmem_ld_wait();
        if (!mine) continue;
        const int d0 = hf * DH + c * 32;
        if (ns == 1) {
          uint16_t* orow = a.out + int64_t(row) * a.out_stride + int64_t(head) * D + d0;
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float o0 = __uint_as_float(r[2 * e]) * inv_l + 0.0f;
            const float o1 = __uint_as_float(r[2 * e + 1]) * inv_l + 0.0f;
            pk[e] = pack_bf2(o0, o1);
          }
          if ((reinterpret_cast<uintptr_t>(orow) & 31) == 0) {   // whole sectors
            st_global_v8(orow, pk);
            st_global_v8(orow + 16, pk + 8);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
          }
        } else {
          float* wrow = a.ws_o + slot * D + d0;
          if ((reinterpret_cast<uintptr_t>(wrow) & 31) == 0) {
#pragma unroll
            for (int q = 0; q < 4; ++q) st_global_v8(wrow + 8 * q, r + 8 * q);
          } else {
            float4* wo = reinterpret_cast<float4*>(wrow);
#pragma unroll
            for (int q = 0; q < 8; ++q)
              wo[q] = make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                  __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
          }
        }
      }
      if (mine && ns > 1 && hf == 0) {
        a.ws_ml[2 * slot] = m;
        a.ws_ml[2 * slot + 1] = l;
      }
    }
  }
  // the producer makes sure its copies have landed before the CTA exits
  if (warp == 0 && lane == 0) {
    if (issued_k > 0) {
      const int t = issued_k - 1;
      mbar_wait(bar(K_FULL + t % STK), (t / STK) & 1, a.err, 100000000ull);
    }
    if (issued_v > 0) {
      const int t = issued_v - 1;
      mbar_wait(bar(V_FULL + t % STV), (t / STV) & 1, a.err, 100000000ull);
    }
    mbar_wait(bar(Q_FULL), 0, a.err, 100000000ull);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, Cfg::TMEM_COLS);
}

// Merge the splits of rows that have more than one, in ascending split order:
// w_s = exp(m_s - M), O = sum w_s o_s, L = sum w_s l_s, out = O / L.
template <int D>
__global__ void attn_merge_kernel(const __grid_constant__ AttnArgs a) {
  pdl_wait();     // stream predecessor done, its writes visible
  pdl_trigger();
  const int64_t gw = (blockIdx.x * int64_t(blockDim.x) + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= int64_t(a.T) * a.Hq) return;
  const int row = int(gw / a.Hq), head = int(gw % a.Hq);
  const int pos = a.row_pos[row];
  if (!row_pos_ok(a, pos)) return;   // reported by the attention kernel; output is NaN
  const int ns = row_splits(a, pos);
  if (ns <= 1) return;
  const int64_t base = (int64_t(row) * a.Hq + head) * a.nsplit_grid;
  float M = -INFINITY;
  for (int s = 0; s < ns; ++s) M = fmaxf(M, a.ws_ml[2 * (base + s)]);
  constexpr int PER = (D + 31) / 32;
  float O[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) O[j] = 0.f;
  float L = 0.f;
  for (int s = 0; s < ns; ++s) {
    const float ms = a.ws_ml[2 * (base + s)];
    if (ms == -INFINITY) continue;
    const float w = ex2(ms - M);
    L += w * a.ws_ml[2 * (base + s) + 1];
    const float* o = a.ws_o + (base + s) * D;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int d = lane + 32 * j;
      if (d < D) O[j] += w * o[d];
    }
  }
  uint16_t* dst = a.out + int64_t(row) * a.out_stride + int64_t(head) * D;
  const float inv = L > 0.f ? 1.0f / L : 0.f;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int d = lane + 32 * j;
    if (d < D) dst[d] = f2bf(O[j] * inv + 0.0f);
  }
}

int plan_split(const biv_attn_desc& d) {
  if (d.mode != BIV_MODE_FAST) return d.kv_split;
  // FAST: choose the split from the batch so that the grid fills the GPU
  const int sms = sm_count() > 0 ? sm_count() : 148;
  const int span = d.topk_idx ? d.topk : d.max_ctx;
  const int64_t ctas = int64_t(d.nqblocks) * d.Hkv;
  int split = span;
  while (split > 256 && ctas * ((span + split - 1) / split) < 2 * sms) split /= 2;
  return std::max(64, (split + 63) / 64 * 64);
}

biv_status validate(const biv_attn_desc* d) {
  BIV_REQUIRE(d, "attention: null descriptor");
  BIV_REQUIRE(d->D == 64 || d->D == 80 || d->D == 128, "attention: D=%d unsupported", d->D);
  BIV_REQUIRE(d->T >= 0 && d->Hq > 0 && d->Hkv > 0 && d->Hq % d->Hkv == 0, "attention: bad heads");
  const int G = d->Hq / d->Hkv;
  BIV_REQUIRE(G <= kNV, "attention: q heads per kv head above %d", kNV);
  BIV_REQUIRE(d->page == kTile, "attention: page size must be %d", kTile);
  BIV_REQUIRE(d->kv_split >= kTile && d->kv_split % kTile == 0, "attention: kv_split must be a multiple of 64");
  BIV_REQUIRE(d->kv_dtype == BIV_BF16 || d->kv_dtype == BIV_E4M3, "attention: kv dtype");
  BIV_REQUIRE(d->kv_dtype == BIV_BF16 || (d->k_scale && d->v_scale), "attention: FP8 needs scales");
  BIV_REQUIRE(d->max_rows_per_block >= 1 && d->max_rows_per_block * G <= kNVTc,
              "attention: max_rows_per_block * (Hq/Hkv) must be <= %d", kNVTc);
  BIV_REQUIRE(!d->topk_idx || (d->max_rows_per_block == 1 && d->topk > 0),
              "attention: sparse mode takes one row per block");
  BIV_REQUIRE(d->topk_idx || d->max_ctx >= 1, "attention: max_ctx >= 1 required");
  BIV_REQUIRE(d->nqblocks >= 0 && d->nqblocks <= 0x7fffffff, "attention: bad nqblocks");
  BIV_REQUIRE(d->mode == BIV_MODE_INVARIANT || d->mode == BIV_MODE_FAST, "attention: bad mode");
  return BIV_OK;
}

size_t ws_bytes(const biv_attn_desc& d, int split) {
  const int span = d.topk_idx ? d.topk : d.max_ctx;
  const int64_t ns = (span + split - 1) / split;
  if (ns <= 1) return 0;
  return size_t(d.T) * d.Hq * ns * (d.D + 2) * sizeof(float);
}

template <int D, int NW, int ST, bool TMA, int DS = 1, int MINB = 0, bool F8 = false>
biv_status launch_cfg(const biv_attn_desc& d, const AttnArgs& a, cudaStream_t s) {
  using Cfg = AttnCfg<D, NW, ST, TMA, DS, F8>;
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(attn_kernel<D, NW, ST, TMA, DS, MINB, F8>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM) != cudaSuccess)
      return set_error(BIV_ERR_CUDA, "attention: cannot set shared memory size");
    attr = true;
  }
  dim3 grid(d.nqblocks, d.Hkv, a.nsplit_grid);
  launch_pdl(attn_kernel<D, NW, ST, TMA, DS, MINB, F8>, grid, Cfg::NT, Cfg::SMEM, s, a);
  return check_launch("attention");
}

// Decode CTAs (TMA loads): DS warps split the head dimension, ST stages.
template <int D, int DS>
biv_status launch_decode(const biv_attn_desc& d, const AttnArgs& a, int st, cudaStream_t s) {
  if (st == 1) return launch_cfg<D, DS, 1, true, DS>(d, a, s);
  if (st == 2) return launch_cfg<D, DS, 2, true, DS>(d, a, s);
  return launch_cfg<D, DS, 3, true, DS>(d, a, s);
}

// bf16 cache of one layer as a 3-D tensor {64 dims, num_pages*64 slots,
// Hkv*D/64 panels} (slot stride Hkv*D elements, panel stride 64 elements):
// one box {64, 64, D/64} is one page of one KV head, landing as [panel][slot]
// [128 B] with 128-byte swizzling, in a single copy (a copy per 128-byte row
// segment is what a TMA producer pays for)
bool make_kv_map(CUtensorMap* m, const void* base, int num_pages, int Hkv, int D) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[3] = {64, cuuint64_t(num_pages) * kTile, cuuint64_t(Hkv) * D / 64};
  cuuint64_t strides[2] = {cuuint64_t(Hkv) * D * 2, 128};
  cuuint32_t box[3] = {64, kTile, cuuint32_t(D / 64)};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Decode CTAs (at most 16 query vectors, TMA loads): the pipeline depth and
// the number of warps that split the head dimension change no result bit,
// only speed.  A CTA is latency-bound on its own instruction stream, so many
// shallow one-warp CTAs per SM move the most KV when the grid is large
// (measured on GB300, 256 sequences x 700 tokens: one stage 5.8 TB/s, two
// 4.6, three 3.5); a small grid (few sequences) is faster with two warps
// sharing the head dimension and two stages (4 sequences: 27 vs 30 us).
// BIV_ATTN_DECODE_STAGES (1-3) and BIV_ATTN_DECODE_DSPLIT (1, 2, 4) override
// the choice (tuning and tests).
int env_int(const char* name, int lo, int hi) {
  const char* e = getenv(name);
  const int v = e ? atoi(e) : 0;
  return (v >= lo && v <= hi) ? v : 0;
}
// Decode CTA shape by grid size (GB300, 16 q / 8 kv heads, D 128, 16 to 256
// sequences at 300 to 1400 tokens, graph-replayed over caches larger than
// L2): a second TMA stage pays only below one CTA per SM; four warps on the
// head dimension are fastest from two CTAs per SM up to 1024 CTAs (up to 13%
// over one warp; a whole 64-sequence decode step 2.52 -> 2.40 ms), two below
// that and up to 2048, and one warp beyond, where the kernel runs at the HBM
// rate.
int decode_stages(int64_t ctas) {
  if (const int v = env_int("BIV_ATTN_DECODE_STAGES", 1, 3)) return v;
  const int sms = sm_count() > 0 ? sm_count() : 148;
  return ctas < sms ? 2 : 1;
}
int decode_dsplit(int64_t ctas) {
  const int v = env_int("BIV_ATTN_DECODE_DSPLIT", 1, 4);
  if (v == 1 || v == 2 || v == 4) return v;
  const int sms = sm_count() > 0 ? sm_count() : 148;
  return ctas < 2 * sms ? 2 : ctas <= 1024 ? 4 : ctas <= 2048 ? 2 : 1;
}

// q as a 3-D tensor [T][Hq][D] with boxes of 64 dims x G heads x 128/G rows:
// one box is 128 query vectors (row-major over (row, head of the group)) of
// one 64-dim panel, 128-byte swizzled.  Rows past T read as zero.
bool make_q_map(CUtensorMap* m, const void* q, int T, int Hq, int D, int64_t q_stride, int G) {
  auto fn = tensor_map_encoder();
  if (!fn || kNVTc % G != 0) return false;
  cuuint64_t dims[3] = {cuuint64_t(D), cuuint64_t(Hq), cuuint64_t(T)};
  cuuint64_t strides[2] = {cuuint64_t(D) * 2, cuuint64_t(q_stride) * 2};
  cuuint32_t box[3] = {64, cuuint32_t(G), cuuint32_t(kNVTc / G)};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
biv_status launch_tc(const biv_attn_desc& d, const AttnArgs& a, cudaStream_t s) {
  using Cfg = TcCfg<D>;
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(attn_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg::SMEM) != cudaSuccess)
      return set_error(BIV_ERR_CUDA, "attention: cannot set shared memory size");
    attr = true;
  }
  dim3 grid(d.nqblocks, d.Hkv, a.nsplit_grid);
  launch_pdl(attn_tc_kernel<D>, grid, Cfg::THREADS, Cfg::SMEM, s, a);
  return check_launch("attention_tc");
}

template <int D>
biv_status launch(const biv_attn_desc& d, AttnArgs& a, cudaStream_t s) {
  // The CTA shape, the loader and the tensor-core path follow the call; a
  // vector's arithmetic does not.
  const bool small = d.max_rows_per_block * a.G <= 16;
  const bool wide = d.max_rows_per_block * a.G > kNV;   // only attn_tc_kernel takes these
  biv_status st;
  bool tma = false;
  if constexpr (D % 64 == 0) {
    tma = !a.fp8 && !a.topk_idx && d.num_pages > 0 &&
          make_kv_map(&a.tmK, d.k_cache, d.num_pages, d.Hkv, D) &&
          make_kv_map(&a.tmV, d.v_cache, d.num_pages, d.Hkv, D);
    // prefill blocks on tcgen05 unless BIV_ATTN_PREFILL_TC=0 (tests compare
    // the two kernels bit for bit)
    const char* tc_env = getenv("BIV_ATTN_PREFILL_TC");
    const bool tc = tma && !small && !(tc_env && atoi(tc_env) == 0) &&
                    make_q_map(&a.tmQ, d.q, d.T, d.Hq, D, d.q_stride, a.G);
    if (tc) {
      st = launch_tc<D>(d, a, s);
    } else if (wide) {
      return set_error(BIV_ERR_UNSUPPORTED,
                       "attention: blocks above %d query vectors need a bf16 cache, D 64 or 128, "
                       "dense attention and Hq/Hkv dividing 128", kNV);
    } else if (tma) {
      if (!small) {
        // Prefill CTAs: one TMA stage and registers capped for three CTAs
        // per SM (measured on GB300, 8 sequences x 1024 tokens: 223 us,
        // against 265 us for two stages at two CTAs per SM and 273 us for
        // one stage at two).  BIV_ATTN_PREFILL_STAGES=2 selects the two-stage
        // CTA (tests and tuning; no bit changes).
        st = env_int("BIV_ATTN_PREFILL_STAGES", 2, 2) ? launch_cfg<D, 4, 2, true>(d, a, s)
                                                      : launch_cfg<D, 4, 1, true, 1, 3>(d, a, s);
      } else {
        const int64_t ctas = int64_t(d.nqblocks) * d.Hkv * a.nsplit_grid;
        const int stages = decode_stages(ctas);
        const int dsplit = decode_dsplit(ctas);
        st = dsplit == 1   ? launch_decode<D, 1>(d, a, stages, s)
             : dsplit == 4 ? launch_decode<D, 4>(d, a, stages, s)
                           : launch_decode<D, 2>(d, a, stages, s);
      }
    }
  }
  if (!tma) {
    if (wide)
      return set_error(BIV_ERR_UNSUPPORTED,
                       "attention: blocks above %d query vectors need a bf16 cache, D 64 or 128, "
                       "dense attention and Hq/Hkv dividing 128", kNV);
    if (a.fp8) {
      // FP8 decode CTAs: four warps share the staged dequantisation and split
      // the head dimension in P.V (D = 80 keeps one warp: its 10 output
      // n-tiles do not split four ways)
      // (registers capped so that four of them fit on an SM)
      constexpr int DSF = D % 64 == 0 ? 4 : 1;
      st = small ? launch_cfg<D, DSF, 2, false, DSF, DSF == 4 ? 4 : 0, true>(d, a, s)
                 : launch_cfg<D, 4, 2, false, 1, 0, true>(d, a, s);
    } else if (small) {
      st = launch_cfg<D, 1, 2, false>(d, a, s);
    } else if (D % 64 == 0 && d.max_rows_per_block * a.G <= 32 &&
               !(getenv("BIV_ATTN_GROUP_DSPLIT") && atoi(getenv("BIV_ATTN_GROUP_DSPLIT")) == 0)) {
      // blocks of 17-32 vectors (sparse rows of a 32-head MQA): two vector
      // groups of two warps each, instead of four warps of which two are
      // idle (GB300, a 4096-token block with top-2048 MQA attention and the
      // MoE: 2.82 ms a step against 3.16; two groups of four warps: 3.13).  BIV_ATTN_GROUP_DSPLIT=0
      // keeps the four-warp CTA (tests: no bit changes).
      st = launch_cfg<D, 4, 2, false, D % 64 == 0 ? 2 : 1>(d, a, s);
    } else {
      st = launch_cfg<D, 4, 2, false>(d, a, s);
    }
  }
  if (st != BIV_OK || a.nsplit_grid <= 1) return st;
  const int64_t warps = int64_t(d.T) * d.Hq;
  launch_pdl(attn_merge_kernel<D>, unsigned((warps * 32 + 255) / 256), 256, 0, s, a);
  return check_launch("attention_merge");
}

}  // namespace
}  // namespace biv

using namespace biv;

extern "C" {

biv_status biv_attention_workspace(const biv_attn_desc* d, size_t* bytes) {
  biv_status st = validate(d);
  if (st != BIV_OK) return st;
  BIV_REQUIRE(bytes, "attention_workspace: null output");
  *bytes = ws_bytes(*d, plan_split(*d));
  return BIV_OK;
}

biv_status biv_attention(const biv_attn_desc* d, void* ws, size_t wsb, biv_stream_t stream) {
  biv_status st = validate(d);
  if (st != BIV_OK) return st;
  if (d->T == 0 || d->nqblocks == 0) return BIV_OK;
  BIV_REQUIRE(d->q && d->out && d->row_seq && d->row_pos && d->qblocks && d->k_cache &&
                  d->v_cache && d->block_table,
              "attention: null pointer");
  BIV_REQUIRE(aligned16(d->q) && aligned16(d->out) && (d->q_stride * 2) % 16 == 0 &&
                  (d->out_stride * 2) % 16 == 0 && aligned16(d->k_cache) && aligned16(d->v_cache),
              "attention: q/out/cache must keep rows 16-byte aligned");
  const int split = plan_split(*d);
  const size_t need = ws_bytes(*d, split);
  if (need && (!ws || wsb < need))
    return set_error(BIV_ERR_WORKSPACE, "attention: workspace of %zu bytes needed", need);
  const int span = d->topk_idx ? d->topk : d->max_ctx;
  AttnArgs a;
  memset(&a, 0, sizeof(a));
  a.q = d->q; a.q_stride = d->q_stride;
  a.out = d->out; a.out_stride = d->out_stride;
  a.T = d->T; a.Hq = d->Hq; a.Hkv = d->Hkv; a.G = d->Hq / d->Hkv;
  a.row_seq = d->row_seq; a.row_pos = d->row_pos; a.qblocks = d->qblocks;
  a.fp8 = d->kv_dtype == BIV_E4M3;
  a.kc = d->k_cache; a.vc = d->v_cache; a.ks = d->k_scale; a.vs = d->v_scale;
  a.bt = d->block_table; a.max_pages = d->max_pages;
  a.kv_split = split;
  a.topk_idx = d->topk_idx; a.topk_stride = d->topk_stride; a.topk = d->topk;
  a.scale = float(double(d->scale) * 1.4426950408889634);   // log2(e)
  a.nsplit_grid = (span + split - 1) / split;
  a.ws_o = static_cast<float*>(ws);
  a.ws_ml = a.ws_o ? a.ws_o + size_t(d->T) * d->Hq * a.nsplit_grid * d->D : nullptr;
  a.err = device_error_word();
  BIV_REQUIRE(a.nsplit_grid <= 65535, "attention: too many splits");
  cudaStream_t s = as_cuda(stream);
  switch (d->D) {
    case 64: return launch<64>(*d, a, s);
    case 80: return launch<80>(*d, a, s);
    default: return launch<128>(*d, a, s);
  }
}

}  // extern "C"

// --------------------------------------------------------------------------
// Allocation-free attention.  Some callers cannot call cudaMalloc at all: a
// host process that runs under a memory-budget sandbox, an inference server
// whose allocator is owned by another runtime, or a driver-level hook that
// must not allocate while the caller holds a lock.  For them the split
// partials live in one fixed device array that the library owns.  It is
// reserved on every GPU that loads the library and held until the process
// exits.
namespace biv {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB per device
static __device__ __align__(256) uint8_t g_attn_noalloc_scratch[kNoAllocScratchBytes];

// The host cannot use the array's name as a device address: it is looked up
// with the device current and cached per CUDA context.  Keying the cache on
// the context (not only on the device ordinal) means that a context torn down
// and created again (cudaDeviceReset, which reloads the module and so moves
// the array) gets a fresh lookup instead of a stale address.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);

CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

void* noalloc_scratch_ptr(biv_status* st) {
  struct Entry { CUcontext ctx; int dev; void* ptr; };
  static std::mutex mu;
  static Entry cache[64];
  static int used = 0;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    *st = set_error(BIV_ERR_CUDA, "attention_noalloc: no current CUDA device");
    return nullptr;
  }
  CtxGetCurrentFn get_ctx = ctx_get_current();
  if (!get_ctx) {
    *st = set_error(BIV_ERR_CUDA, "attention_noalloc: cuCtxGetCurrent is not available");
    return nullptr;
  }
  CUcontext ctx = nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (get_ctx(&ctx) == CUDA_SUCCESS && ctx) {
    for (int i = 0; i < used; ++i)
      if (cache[i].ctx == ctx && cache[i].dev == dev) {
        *st = BIV_OK;
        return cache[i].ptr;
      }
  }
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_attn_noalloc_scratch);
  if (e != cudaSuccess || !p) {
    *st = set_error(BIV_ERR_CUDA, "attention_noalloc: cudaGetSymbolAddress failed: %s",
                    cudaGetErrorString(e));
    return nullptr;
  }
  // the lookup makes the device's primary context current if none was
  if (get_ctx(&ctx) == CUDA_SUCCESS && ctx) {
    int slot = -1;
    for (int i = 0; i < used; ++i)
      if (cache[i].dev == dev) slot = i;       // a replaced context of this device
    if (slot < 0 && used < 64) slot = used++;
    if (slot >= 0) cache[slot] = Entry{ctx, dev, p};
  }
  *st = BIV_OK;
  return p;
}

}  // namespace
}  // namespace biv

extern "C" biv_status biv_attention_noalloc(const biv_attn_desc* d, biv_stream_t stream) {
  biv_status st = validate(d);
  if (st != BIV_OK) return st;
  const size_t need = ws_bytes(*d, plan_split(*d));
  if (need > kNoAllocScratchBytes)
    return set_error(BIV_ERR_WORKSPACE,
                     "attention_noalloc: this call needs %zu bytes of scratch, above the fixed "
                     "%zu-byte array; use biv_attention with a caller workspace",
                     need, kNoAllocScratchBytes);
  void* scratch = noalloc_scratch_ptr(&st);
  if (st != BIV_OK) return st;
  // Every slot of the partials that the merge reads is written earlier in the
  // same call, so nothing in the array has to start at zero.
  return biv_attention(d, scratch, kNoAllocScratchBytes, stream);
}
