// Sparse-attention Top-K with a fixed tie-break and a fixed output order
// ("Finish RL Training Faster", section "让训练前向使用推理的数值": equal scores are
// resolved the same way every time and the selection is laid out in position
// order, so the same set is always accumulated in the same order).
//
// Persistent CTAs of 1024 threads, one row at a time.  A row's scores are
// copied to shared memory while the CTA works on the previous row, so the
// HBM read overlaps the selection: by a few bulk copies issued by one thread
// when rows are 16-byte aligned (8192 per-thread 16-byte copies kept the
// load/store unit busy through the whole selection), else by cp.async.  Thread t then keeps 32 keys
// in registers: in round r (0..7) the four consecutive positions
// 4096 r + 4 t + e (e = 0..3).  Scores become order-preserving 32-bit keys:
// +0 and -0 map to one key, and NaN, -inf and the positions past valid_len
// (filled with -inf in shared memory) all map to the key of -inf, which lies
// below every bin the selection can choose and is never selected.
//
// The k-th largest key is bracketed by range refinement.  The first round
// counts every key in a 4096-bin histogram of its top 12 bits while the keys
// are formed; a block scan over the bins in descending order finds the bin
// holding the k-th largest key, which becomes the key range [lo, hi].  Each
// later round cuts the current range into at most 4096 power-of-two-wide
// bins and narrows it the same way (20 -> 8 -> 0 bits of width: at most
// three rounds reach one key value).  When the first bin holds at most 1024
// keys they are copied to a candidate list in shared memory and the later
// rounds run over that list (one candidate per thread) with 256 bins, which
// one warp scans (20 -> 12 -> 4 -> 0 bits); otherwise they run over the
// registers.  Refinement stops once the chosen bin's keys are
// exactly the ones still wanted, or the bin is one key value, whose lowest
// positions then fill the remaining slots.
//
// Output: every key above the final bin plus the chosen keys inside it, in
// ascending position order.  Each thread holds its choice as a 32-bit mask;
// a position's output slot is the number of chosen positions before it,
// from per-(round, warp) counts scanned over the block and per-lane counts
// scanned over the warp.  Only integer counts decide the result, so it is
// unique and independent of scheduling.
//
// The kernel is bound by instruction issue, so the per-row block scans run
// on warp shuffles (one barrier each) and every narrowing step clears the
// histogram it has read, ready for the next round or row.
#include "common.cuh"

namespace biv {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;       // 32: one warp-sum per lane
constexpr int kRounds = 8;                  // float4 rounds per thread
constexpr int kPer = 4 * kRounds;           // keys per thread
constexpr int kRoundSpan = 4 * kThreads;    // positions per round
constexpr int kMaxN = kThreads * kPer;      // 32768
constexpr int kBinBits = 12;
constexpr int kBins = 1 << kBinBits;        // 4096
constexpr int kBinsPerThread = kBins / kThreads;
constexpr uint32_t kNegInfKey = 0x007FFFFFu;   // the key of -inf (and of NaN)
// the first round's bins below this one hold no key but -inf's
constexpr int kFirstValidBin = int((kNegInfKey + 1u) >> (32 - kBinBits));
// Rounds after the first: a 2^20-wide bin needs two more (2^8, then one key);
// the bound only guards the loop.
constexpr int kMaxRefine = 4;
static_assert(kWarps == 32 && kBinsPerThread == 4, "scan and histogram layout");

// Order-preserving key of a score: -0 + 0 = +0 gives -0 the key of +0, and
// the IEEE maximum with -inf turns NaN into -inf (finite values, infinities
// and subnormals pass both unchanged).
__device__ __forceinline__ uint32_t order_key(float s) {
  const uint32_t u = __float_as_uint(fmaxf(s + 0.0f, -INFINITY));
  return u ^ (uint32_t(int32_t(u) >> 31) | 0x80000000u);
}

// position of key slot q (= 4 r + e) of thread t
__device__ __forceinline__ int slot_pos(int q, int t) { return (q >> 2) * kRoundSpan + 4 * t + (q & 3); }

__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

// Exclusive scan of one value per thread over the CTA in thread order; also
// returns the total.  One barrier, after which wsum is read by every warp: a
// caller must pass another barrier before the next scan writes wsum.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* wsum, uint32_t& total) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t x = warp_incl_scan(v, lane);
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  const uint32_t ws = wsum[lane];
  const uint32_t wi = warp_incl_scan(ws, lane);
  total = __shfl_sync(0xffffffffu, wi, 31);
  return __shfl_sync(0xffffffffu, wi - ws, warp) + x - v;
}

struct Range {
  uint32_t lo, hi;   // keys still undecided
  uint32_t rem;      // how many of them are still wanted (1 <= rem <= keys in range)
  uint32_t in_bin;   // keys in [lo, hi]
};

// Bin geometry of a range: bins of 2^shift keys, nb <= 4096 of them.
__device__ __forceinline__ int bin_shift(const Range& g) {
  return max(0, 32 - __clz(g.hi - g.lo) - kBinBits);
}

// After the histogram of the current range is complete in hist[]: find the
// bin holding the rem-th largest key and narrow the range to it (only when
// the range holds at least rem keys).  Every thread returns the same new
// range and the number of keys the histogram held, and hist[] is zero again.
// Barriers: 2; s_sel is free again once the caller has passed one more.
// FIRST: the first round (bins of the top 12 key bits), whose bins below
// kFirstValidBin are not counted.
template <bool FIRST = false>
__device__ __forceinline__ uint32_t narrow(Range& g, int shift, uint32_t* hist, uint32_t* wsum,
                                          uint32_t* s_sel) {
  const int tid = threadIdx.x;
  const int nb = int((g.hi - g.lo) >> shift) + 1;
  // descending bin order: thread t owns bins nb-1-4t .. nb-4-4t
  uint32_t c[kBinsPerThread], sum = 0;
#pragma unroll
  for (int d = 0; d < kBinsPerThread; ++d) {
    const int b = nb - 1 - (kBinsPerThread * tid + d);
    c[d] = b >= (FIRST ? kFirstValidBin : 0) ? hist[b] : 0u;
    sum += c[d];
  }
  uint32_t tot;
  uint32_t above = block_excl_scan(sum, wsum, tot);   // every bin has been read
  reinterpret_cast<uint4*>(hist)[tid] = make_uint4(0u, 0u, 0u, 0u);
  const bool pick = g.rem <= tot;
  if (pick) {
#pragma unroll
    for (int d = 0; d < kBinsPerThread; ++d) {
      if (above < g.rem && g.rem <= above + c[d]) {
        s_sel[0] = uint32_t(nb - 1 - (kBinsPerThread * tid + d));
        s_sel[1] = above;
        s_sel[2] = c[d];
      }
      above += c[d];
    }
  }
  __syncthreads();
  if (pick) {
    const uint32_t b = s_sel[0];
    g.rem -= s_sel[1];
    g.in_bin = s_sel[2];
    const uint32_t nlo = g.lo + (b << shift), width_m1 = (1u << shift) - 1u;
    if (g.hi - nlo > width_m1) g.hi = nlo + width_m1;  // no wrap: nlo + width_m1 < hi
    g.lo = nlo;
  }
  return tot;
}

__device__ __forceinline__ bool range_done(const Range& g) {
  return g.lo == g.hi || g.in_bin == g.rem;
}

// One refinement round over the 32 register keys of every thread.
__device__ __forceinline__ void refine_regs(Range& g, const uint32_t (&key)[kPer], uint32_t* hist,
                                            uint32_t* wsum, uint32_t* s_sel) {
  const int shift = bin_shift(g);
  const uint32_t span = g.hi - g.lo;
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const uint32_t d = key[q] - g.lo;  // keys below lo (-inf's too) wrap above span
    if (d <= span) atomicAdd(hist + (d >> shift), 1u);
  }
  __syncthreads();
  narrow(g, shift, hist, wsum, s_sel);
}

// One refinement round over the candidate list (thread t holds candidate t
// when t < count; ck = its key): at most 256 bins, counted by every thread
// and scanned by warp 0 alone (lane L owns the descending bins nb-1-8L ..
// nb-8-8L), which then clears them.  Barriers: 2.
constexpr int kCandBinBits = 8;
constexpr int kCandBins = 1 << kCandBinBits;
__device__ __forceinline__ void refine_cands(Range& g, bool has, uint32_t ck, uint32_t* hist,
                                             uint32_t* s_sel) {
  const int shift = max(0, 32 - __clz(g.hi - g.lo) - kCandBinBits);
  if (has && ck >= g.lo && ck <= g.hi) atomicAdd(hist + ((ck - g.lo) >> shift), 1u);
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int nb = int((g.hi - g.lo) >> shift) + 1;
    uint32_t c[kCandBins / 32], sum = 0;
#pragma unroll
    for (int d = 0; d < kCandBins / 32; ++d) {
      const int b = nb - 1 - ((kCandBins / 32) * lane + d);
      c[d] = b >= 0 ? hist[b] : 0u;
      sum += c[d];
    }
    const uint32_t incl = warp_incl_scan(sum, lane);
    uint32_t above = incl - sum;
    if (above < g.rem && g.rem <= incl) {
#pragma unroll
      for (int d = 0; d < kCandBins / 32; ++d) {
        if (above < g.rem && g.rem <= above + c[d]) {
          s_sel[0] = uint32_t(nb - 1 - ((kCandBins / 32) * lane + d));
          s_sel[1] = above;
          s_sel[2] = c[d];
        }
        above += c[d];
      }
    }
    __syncwarp();
    reinterpret_cast<uint4*>(hist)[2 * lane] = make_uint4(0u, 0u, 0u, 0u);
    reinterpret_cast<uint4*>(hist)[2 * lane + 1] = make_uint4(0u, 0u, 0u, 0u);
  }
  __syncthreads();
  const uint32_t b = s_sel[0];
  g.rem -= s_sel[1];
  g.in_bin = s_sel[2];
  const uint32_t nlo = g.lo + (b << shift), width_m1 = (1u << shift) - 1u;
  if (g.hi - nlo > width_m1) g.hi = nlo + width_m1;
  g.lo = nlo;
}

// Output slots of the set bits of `mask` (bit q = key slot q of this thread)
// in ascending position order.  tab: kRounds * kWarps words.  On return
// tab[r * kWarps + w] = chosen positions before round r's warp-w block, and
// byte r of the pair pre (rounds 0..3 in pre[0], 4..7 in pre[1]) = chosen
// positions of lanes < this lane in round r.  Also returns the total.
// Barriers: 3 (tab may be rewritten once the caller has passed one more).
__device__ __forceinline__ uint32_t ordered_slots(uint32_t mask, uint32_t* tab, uint32_t* wsum,
                                                  uint32_t (&pre)[2]) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // per-round counts (0..4) packed as 8-bit fields, four rounds per word: a
  // warp prefix is at most 128, so the fields never carry into each other
  uint32_t c[2] = {0u, 0u};
#pragma unroll
  for (int r = 0; r < kRounds; ++r)
    c[r >> 2] |= uint32_t(__popc((mask >> (4 * r)) & 15u)) << (8 * (r & 3));
  uint32_t x[2] = {c[0], c[1]};
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, x[h], o);
      if (lane >= o) x[h] += y;
    }
  }
  // fields never borrow: each inclusive count is at least its own
  pre[0] = x[0] - c[0];
  pre[1] = x[1] - c[1];
  if (lane == 31) {
#pragma unroll
    for (int r = 0; r < kRounds; ++r) tab[r * kWarps + warp] = (x[r >> 2] >> (8 * (r & 3))) & 255u;
  }
  __syncthreads();
  const uint32_t v = tid < kRounds * kWarps ? tab[tid] : 0u;
  uint32_t total;
  const uint32_t before = block_excl_scan(v, wsum, total);
  if (tid < kRounds * kWarps) tab[tid] = before;
  __syncthreads();
  return total;
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}

__device__ __forceinline__ int row_valid(const int32_t* valid_len, int row, int n) {
  return min(max(valid_len[row], 0), n);
}

constexpr int kBulkChunk = 4096;   // floats per bulk copy

// Start the copy of a row's valid scores into buf; the positions past them
// are set to -inf.  VEC (16-byte aligned rows): bulk copies of the first
// nv & ~3 scores by thread 0, completing on mbarrier `bar`, and plain loads
// of the rest; the caller has ordered every read of buf before this call
// with a barrier.  Otherwise: cp.async, 4 or 16 bytes per copy.
template <bool VEC>
__device__ __forceinline__ void prefetch_row(float* buf, const float* __restrict__ scores,
                                             int64_t ld, int row, int nv, uint32_t bar) {
  const float* src = scores + int64_t(row) * ld;
  if constexpr (VEC) {
    const int nv4 = nv & ~3;
    if (threadIdx.x == 0) {
      fence_proxy_async();
      mbar_expect_tx(bar, uint32_t(nv4) * 4u);
      for (int off = 0; off < nv4; off += kBulkChunk)
        bulk_load(smem_u32(buf + off), src + off, uint32_t(min(kBulkChunk, nv4 - off)) * 4u, bar);
    }
    for (int j = nv4 + threadIdx.x; j < kMaxN; j += kThreads) buf[j] = j < nv ? __ldg(src + j) : -INFINITY;
  } else {
    const bool a16 = (reinterpret_cast<uintptr_t>(src) & 15u) == 0;
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
      const int j0 = r * kRoundSpan + 4 * threadIdx.x;
      if (a16 && j0 + 3 < nv) {
        cp_async16(buf + j0, src + j0);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (j0 + e < nv)
            cp_async4(buf + j0 + e, src + j0 + e);
          else
            buf[j0 + e] = -INFINITY;
        }
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
}

template <bool VEC>
__global__ void __launch_bounds__(kThreads, 1)
    topk_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ valid_len,
                int rows, int n, int k, int32_t* __restrict__ idx, int* err) {
  extern __shared__ float4 rowbuf4[];                // one row of scores (kMaxN floats)
  float* rowbuf = reinterpret_cast<float*>(rowbuf4);
  __shared__ __align__(16) uint32_t hist[kBins];     // bin counts, zero between rounds
  __shared__ uint32_t tab[kRounds * kWarps];         // output slot table
  __shared__ uint32_t wsum[kWarps];
  __shared__ uint32_t s_sel[3];
  __shared__ uint32_t s_cnt;                         // candidates gathered
  __shared__ uint32_t cand_key[kThreads];            // candidate list
  __shared__ uint32_t cand_pos[kThreads];
  __shared__ uint32_t tie_bits[kThreads];            // chosen candidates, as thread-slot masks
  __shared__ __align__(8) uint64_t row_bar;          // bulk copies of the next row landed

  const int tid = threadIdx.x, warp = tid >> 5;
  reinterpret_cast<uint4*>(hist)[tid] = make_uint4(0u, 0u, 0u, 0u);
  const uint32_t bar = smem_u32(&row_bar);
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  int row = blockIdx.x;
  int nv_next = row < rows ? row_valid(valid_len, row, n) : 0;
  if (row < rows) prefetch_row<VEC>(rowbuf, scores, ld, row, nv_next, bar);
  uint32_t parity = 0;
  // The first round counts only the bins from lbin up: the bin below the
  // one this CTA's previous row chose (its rows are alike, as the causal
  // rows of one indexer are).  Keys below never reach the histogram, which
  // relieves the shared-memory atomics; a row with fewer than k keys from
  // lbin up is counted again in full.  lbin changes the time, not the result.
  uint32_t lbin = 0;
  for (; row < rows; row += gridDim.x) {
    bool landed = true;
    if (VEC)
      landed = mbar_wait(bar, parity, err);
    else
      asm volatile("cp.async.wait_all;" ::: "memory");
    parity ^= 1u;
    // the row is in shared memory; the previous row's tables are free
    if (!__syncthreads_and(landed)) return;

    // keys, and the first round's histogram of their top 12 bits
    uint32_t key[kPer];
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
      const int j0 = r * kRoundSpan + 4 * tid;
      const float4 f = rowbuf4[j0 / 4];
      const float v[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t kk = order_key(v[e]);
        key[4 * r + e] = kk;
        const uint32_t b = kk >> (32 - kBinBits);
        if (b >= lbin) atomicAdd(hist + b, 1u);
      }
    }
    __syncthreads();  // keys in registers; histogram complete
    // the next row goes to the buffer once this row's candidates are read
    // from it (or at once when no candidate list is built)
    auto start_next = [&]() {
      if (row + int(gridDim.x) < rows) {
        nv_next = row_valid(valid_len, row + gridDim.x, n);
        prefetch_row<VEC>(rowbuf, scores, ld, row + gridDim.x, nv_next, bar);
      }
    };
    if (tid == 0) s_cnt = 0u;
    tie_bits[tid] = 0u;
    Range g{0u, 0xffffffffu, uint32_t(k), 0u};
    uint32_t total_valid = narrow<true>(g, 32 - kBinBits, hist, wsum, s_sel);
    if (total_valid <= uint32_t(k) && lbin > uint32_t(kFirstValidBin)) {
      // at most k keys from lbin up: count every key (the test below must
      // see the whole row's count before it selects every valid key)
#pragma unroll
      for (int q = 0; q < kPer; ++q) atomicAdd(hist + (key[q] >> (32 - kBinBits)), 1u);
      __syncthreads();
      g = Range{0u, 0xffffffffu, uint32_t(k), 0u};   // the filtered pass may have narrowed it
      total_valid = narrow<true>(g, 32 - kBinBits, hist, wsum, s_sel);
    }
    lbin = total_valid >= uint32_t(k) ? (g.lo >> (32 - kBinBits)) - 1u : 0u;

    uint32_t sel = 0;  // bit q: key slot q chosen
    if (total_valid <= uint32_t(k)) {
      start_next();
#pragma unroll
      for (int q = 0; q < kPer; ++q) sel |= uint32_t(key[q] > kNegInfKey) << q;
    } else if (!range_done(g) && g.in_bin <= uint32_t(kThreads)) {
      // the bin's keys as a candidate list (list order is irrelevant: every
      // later decision is by key, then by position); keys above the bin are
      // chosen whatever the later rounds decide
      const uint32_t lo1 = g.lo, hi1 = g.hi, span1 = hi1 - lo1;
      uint32_t cm = 0;   // bit q: key slot q is a candidate
#pragma unroll
      for (int q = 0; q < kPer; ++q) {
        cm |= uint32_t(key[q] - lo1 <= span1) << q;
        sel |= uint32_t(key[q] > hi1) << q;
      }
      if (cm) {   // one slot reservation per thread; keys re-read from the row
        uint32_t s = atomicAdd(&s_cnt, uint32_t(__popc(cm)));
        do {
          const int q = __ffs(cm) - 1;
          cm &= cm - 1u;
          const int pos = slot_pos(q, tid);
          cand_key[s] = order_key(rowbuf[pos]);
          cand_pos[s] = uint32_t(pos);
          ++s;
        } while (cm);
      }
      __syncthreads();
      start_next();
      const uint32_t nc = g.in_bin;
      const bool has = uint32_t(tid) < nc;
      const uint32_t ck = has ? cand_key[tid] : 0u, cp = has ? cand_pos[tid] : 0u;
      for (int it = 0; it < kMaxRefine && !range_done(g); ++it)
        refine_cands(g, has, ck, hist, s_sel);
      bool take = has && ck > g.hi;
      if (has && ck >= g.lo && ck <= g.hi) {
        if (g.in_bin == g.rem) {
          take = true;
        } else {  // one key value: the lowest positions win
          uint32_t before = 0;
          for (uint32_t c = 0; c < nc; ++c) before += (cand_key[c] == ck && cand_pos[c] < cp);
          take = before < g.rem;
        }
      }
      if (take) {
        const uint32_t r = cp / kRoundSpan, w = cp % kRoundSpan;
        atomicOr(tie_bits + w / 4, 1u << (4 * r + (w & 3)));
      }
      __syncthreads();
      sel |= tie_bits[tid];
    } else {
      // more than 1024 keys share the bin (or it is already decided): refine
      // over the registers
      start_next();
      for (int it = 0; it < kMaxRefine && !range_done(g); ++it)
        refine_regs(g, key, hist, wsum, s_sel);
      uint32_t eq = 0;
#pragma unroll
      for (int q = 0; q < kPer; ++q) {
        sel |= uint32_t(key[q] > g.hi) << q;
        eq |= uint32_t(key[q] >= g.lo && key[q] <= g.hi) << q;
      }
      if (g.in_bin == g.rem) {
        sel |= eq;
      } else {  // one key value: its lowest `rem` positions
        uint32_t pre[2];
        ordered_slots(eq, tab, wsum, pre);
#pragma unroll
        for (int r = 0; r < kRounds; ++r) {
          uint32_t rank = tab[r * kWarps + warp] + ((pre[r >> 2] >> (8 * (r & 3))) & 255u);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int q = 4 * r + e;
            if ((eq >> q) & 1u) {
              if (rank < g.rem) sel |= 1u << q;
              ++rank;
            }
          }
        }
        __syncthreads();  // the slot table is rebuilt below
      }
    }

    uint32_t pre[2];
    const uint32_t total_sel = ordered_slots(sel, tab, wsum, pre);
    int32_t* out = idx + int64_t(row) * k;
    for (uint32_t m = sel; m; m &= m - 1u) {   // this thread's chosen slots
      const int q = __ffs(m) - 1, r = q >> 2;
      const uint32_t slot = tab[r * kWarps + warp] + ((pre[r >> 2] >> (8 * (r & 3))) & 255u) +
                            __popc(sel & ((1u << q) - 1u) & (15u << (4 * r)));
      out[slot] = r * kRoundSpan + 4 * tid + (q & 3);
    }
    for (int s2 = int(total_sel) + tid; s2 < k; s2 += kThreads) out[s2] = -1;
  }  // rows
}

}  // namespace
}  // namespace biv

using namespace biv;

extern "C" {

biv_status biv_topk(const float* scores, int64_t ld, const int32_t* valid_len, int rows, int n,
                    int k, int32_t* idx, biv_stream_t stream) {
  BIV_REQUIRE(rows >= 0 && n > 0 && n <= kMaxN && k > 0 && k <= n && ld >= n,
              "topk: need 0 < k <= n <= %d and ld >= n (n=%d k=%d)", kMaxN, n, k);
  if (rows == 0) return BIV_OK;
  BIV_REQUIRE(scores && valid_len && idx, "topk: null pointer");
  // 16-byte copies when every row starts on a 16-byte boundary
  const bool vec = aligned16(scores) && ld % 4 == 0;
  auto kern = vec ? topk_kernel<true> : topk_kernel<false>;
  constexpr int kRowBytes = kMaxN * 4;
  static bool attr[2] = {false, false};
  if (!attr[vec]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kRowBytes) !=
        cudaSuccess)
      return set_error(BIV_ERR_CUDA, "topk: cannot set shared memory size");
    attr[vec] = true;
  }
  const int sms = sm_count() > 0 ? sm_count() : 148;
  kern<<<std::min(rows, sms), kThreads, kRowBytes, as_cuda(stream)>>>(scores, ld, valid_len, rows,
                                                                     n, k, idx, device_error_word());
  return check_launch("topk");
}

}  // extern "C"
