// Sparse-attention Top-K with a fixed tie-break and a fixed output order
// ("Finish RL Training Faster", section "让训练前向使用推理的数值": equal scores are
// resolved the same way every time and the selection is laid out in position
// order, so the same set is always accumulated in the same order).
//
// Persistent CTAs of 1024 threads, one row at a time.  A row's scores are
// copied to shared memory with cp.async while the CTA works on the previous
// row, so the HBM read overlaps the selection.  Thread t then keeps 32 keys
// in registers: in round r (0..7) the four consecutive positions
// 4096 r + 4 t + e (e = 0..3).  Scores become order-preserving 32-bit keys
// (+0 and -0 map to one key; -inf and positions past valid_len are
// excluded).
//
// The k-th largest key is bracketed by range refinement: the current key
// range [lo, hi] is cut into at most 4096 power-of-two-wide bins, a shared
// histogram counts the keys per bin, and a block scan over the bins in
// descending order finds the bin holding the rem-th largest key, which
// becomes the next range (32 -> 20 -> 8 -> 0 bits of width: at most three
// rounds reach one key value).  The first round runs over every key; when
// the chosen bin holds at most 1024 keys they are copied to a candidate list
// in shared memory and the remaining rounds run over that list (one
// candidate per thread).  Refinement stops once the chosen bin's keys are
// exactly the ones still wanted, or the bin is one key value, whose lowest
// positions then fill the remaining slots.
//
// Output: every key above the final bin plus the chosen keys inside it, in
// ascending position order.  Each thread holds its choice as a 32-bit mask;
// a position's output slot is the number of chosen positions before it,
// from per-(round, warp) counts scanned over the block and per-lane counts
// scanned over the warp.  Only integer counts decide the result, so it is
// unique and independent of scheduling.
#include "common.cuh"

namespace biv {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kRounds = 8;                  // float4 rounds per thread
constexpr int kPer = 4 * kRounds;           // keys per thread
constexpr int kRoundSpan = 4 * kThreads;    // positions per round
constexpr int kMaxN = kThreads * kPer;      // 32768
constexpr int kBinBits = 12;
constexpr int kBins = 1 << kBinBits;        // 4096
constexpr int kBinsPerThread = kBins / kThreads;

__device__ __forceinline__ uint32_t order_key(float s) {
  if (s == 0.f) s = 0.f;  // -0 -> +0
  const uint32_t u = __float_as_uint(s);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// position of key slot q (= 4 r + e) of thread t
__device__ __forceinline__ int slot_pos(int q, int t) { return (q >> 2) * kRoundSpan + 4 * t + (q & 3); }

// Exclusive scan of one value per thread over the CTA in thread order; also
// returns the total.  Uses wsum[kWarps]; two barriers.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* wsum, uint32_t& total) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  uint32_t pre = 0, tot = 0;
#pragma unroll 8
  for (int w = 0; w < kWarps; ++w) {
    const uint32_t c = wsum[w];
    pre += w < warp ? c : 0u;
    tot += c;
  }
  __syncthreads();  // wsum may be reused after this
  total = tot;
  return pre + x - v;
}

// Block-wide sum, min and max (a thread without a valid key passes ~0 and 0).
__device__ __forceinline__ void block_count_range(uint32_t cnt, uint32_t mn, uint32_t mx,
                                                  uint32_t* red, uint32_t& tot, uint32_t& kmin,
                                                  uint32_t& kmax) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  if (lane == 0) {
    red[warp] = cnt;
    red[kWarps + warp] = mn;
    red[2 * kWarps + warp] = mx;
  }
  __syncthreads();
  tot = 0;
  kmin = 0xffffffffu;
  kmax = 0;
#pragma unroll 8
  for (int w = 0; w < kWarps; ++w) {
    tot += red[w];
    kmin = min(kmin, red[kWarps + w]);
    kmax = max(kmax, red[2 * kWarps + w]);
  }
  __syncthreads();  // red may be reused after this
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
// bin holding the rem-th largest key and narrow the range to it.  Every
// thread returns the same new range.  Barriers: 3.
__device__ __forceinline__ void narrow(Range& g, int shift, uint32_t* hist, uint32_t* wsum,
                                       uint32_t* s_sel) {
  const int tid = threadIdx.x;
  const int nb = int((g.hi - g.lo) >> shift) + 1;
  // descending bin order: thread t owns bins nb-1-4t .. nb-4-4t
  uint32_t c[kBinsPerThread], sum = 0;
#pragma unroll
  for (int d = 0; d < kBinsPerThread; ++d) {
    const int b = nb - 1 - (kBinsPerThread * tid + d);
    c[d] = b >= 0 ? hist[b] : 0u;
    sum += c[d];
  }
  uint32_t tot;
  uint32_t above = block_excl_scan(sum, wsum, tot);
#pragma unroll
  for (int d = 0; d < kBinsPerThread; ++d) {
    if (above < g.rem && g.rem <= above + c[d]) {
      s_sel[0] = uint32_t(nb - 1 - (kBinsPerThread * tid + d));
      s_sel[1] = above;
      s_sel[2] = c[d];
    }
    above += c[d];
  }
  __syncthreads();
  const uint32_t b = s_sel[0];
  g.rem -= s_sel[1];
  g.in_bin = s_sel[2];
  const uint32_t nlo = g.lo + (b << shift), width_m1 = (1u << shift) - 1u;
  if (g.hi - nlo > width_m1) g.hi = nlo + width_m1;  // no wrap: nlo + width_m1 < hi
  g.lo = nlo;
  __syncthreads();  // s_sel and hist are free again
}

__device__ __forceinline__ bool range_done(const Range& g) {
  return g.lo == g.hi || g.in_bin == g.rem;
}

// One refinement round over the 32 register keys of every thread.
__device__ __forceinline__ void refine_regs(Range& g, const uint32_t (&key)[kPer], uint32_t* hist,
                                            uint32_t* wsum, uint32_t* s_sel) {
  const int shift = bin_shift(g);
#pragma unroll
  for (int b = threadIdx.x; b < kBins; b += kThreads) hist[b] = 0;
  __syncthreads();
  const uint32_t span = g.hi - g.lo;
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const uint32_t d = key[q] - g.lo;  // keys below lo wrap above span
    if (d <= span) atomicAdd(hist + (d >> shift), 1u);
  }
  __syncthreads();
  narrow(g, shift, hist, wsum, s_sel);
}

// One refinement round over the candidate list (thread t holds candidate t
// when t < count; ck = its key).
__device__ __forceinline__ void refine_cands(Range& g, bool has, uint32_t ck, uint32_t* hist,
                                             uint32_t* wsum, uint32_t* s_sel) {
  const int shift = bin_shift(g);
#pragma unroll
  for (int b = threadIdx.x; b < kBins; b += kThreads) hist[b] = 0;
  __syncthreads();
  if (has && ck >= g.lo && ck <= g.hi) atomicAdd(hist + ((ck - g.lo) >> shift), 1u);
  __syncthreads();
  narrow(g, shift, hist, wsum, s_sel);
}

// Output slots of the set bits of `mask` (bit q = key slot q of this thread)
// in ascending position order.  tab: kRounds * kWarps words.  On return
// tab[r * kWarps + w] = chosen positions before round r's warp-w block, and
// lane_pre[r] = chosen positions of lanes < this lane in round r.  Also
// returns the total.  Barriers: 3.
__device__ __forceinline__ uint32_t ordered_slots(uint32_t mask, uint32_t* tab, uint32_t* wsum,
                                                  uint32_t (&lane_pre)[kRounds]) {
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
#pragma unroll
  for (int r = 0; r < kRounds; ++r) {
    const int sh = 8 * (r & 3);
    const uint32_t incl = (x[r >> 2] >> sh) & 255u;
    lane_pre[r] = incl - ((c[r >> 2] >> sh) & 255u);
    if (lane == 31) tab[r * kWarps + warp] = incl;
  }
  __syncthreads();
  const uint32_t v = tid < kRounds * kWarps ? tab[tid] : 0u;
  uint32_t total;
  const uint32_t pre = block_excl_scan(v, wsum, total);
  if (tid < kRounds * kWarps) tab[tid] = pre;
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

// Start the copy of a row's valid scores into buf (16-byte pieces where the
// row allows them).
template <bool VEC>
__device__ __forceinline__ void prefetch_row(float* buf, const float* __restrict__ scores,
                                             int64_t ld, int row, int nv) {
  const float* src = scores + int64_t(row) * ld;
#pragma unroll
  for (int r = 0; r < kRounds; ++r) {
    const int j0 = r * kRoundSpan + 4 * threadIdx.x;
    if (VEC && j0 + 3 < nv) {
      cp_async16(buf + j0, src + j0);
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (j0 + e < nv) cp_async4(buf + j0 + e, src + j0 + e);
    }
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}

template <bool VEC>
__global__ void __launch_bounds__(kThreads, 1)
    topk_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ valid_len,
                int rows, int n, int k, int32_t* __restrict__ idx) {
  extern __shared__ float4 rowbuf4[];         // one row of scores (kMaxN floats)
  float* rowbuf = reinterpret_cast<float*>(rowbuf4);
  __shared__ uint32_t hist[kBins];            // bin counts; reused as the slot table
  __shared__ uint32_t wsum[3 * kWarps];
  __shared__ uint32_t s_sel[4];
  __shared__ uint32_t cand_key[kThreads];     // candidate list
  __shared__ uint32_t cand_pos[kThreads];
  __shared__ uint32_t tie_bits[kThreads];     // chosen candidates, as thread-slot masks

  const int tid = threadIdx.x, warp = tid >> 5;
  int row = blockIdx.x;
  int nv_next = row < rows ? row_valid(valid_len, row, n) : 0;
  if (row < rows) prefetch_row<VEC>(rowbuf, scores, ld, row, nv_next);
  for (; row < rows; row += gridDim.x) {
    const int nv = nv_next;
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();  // the row is in shared memory; the previous row's tables are free

    uint32_t key[kPer];
    uint32_t cnt = 0, mn = 0xffffffffu, mx = 0;
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
      const int j0 = r * kRoundSpan + 4 * tid;
      const float4 f = rowbuf4[j0 / 4];
      const float v[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t kk = (j0 + e < nv && v[e] != -INFINITY) ? order_key(v[e]) : 0u;
        key[4 * r + e] = kk;
        if (kk != 0) {
          ++cnt;
          mn = min(mn, kk);
          mx = max(mx, kk);
        }
      }
    }
    __syncthreads();  // every thread holds its keys: the buffer takes the next row
    if (row + int(gridDim.x) < rows) {
      nv_next = row_valid(valid_len, row + gridDim.x, n);
      prefetch_row<VEC>(rowbuf, scores, ld, row + gridDim.x, nv_next);
    }
    uint32_t total_valid;
    Range g;
    block_count_range(cnt, mn, mx, wsum, total_valid, g.lo, g.hi);
    g.rem = uint32_t(k);
    g.in_bin = total_valid;

    uint32_t sel = 0;  // bit q: key slot q chosen
    if (total_valid <= uint32_t(k)) {
#pragma unroll
      for (int q = 0; q < kPer; ++q) sel |= uint32_t(key[q] != 0) << q;
    } else {
      if (!range_done(g)) refine_regs(g, key, hist, wsum, s_sel);
      if (!range_done(g) && g.in_bin <= uint32_t(kThreads)) {
        // the bin's keys as a candidate list (list order is irrelevant: every
        // later decision is by key, then by position)
        if (tid == 0) s_sel[3] = 0;
        tie_bits[tid] = 0;
        __syncthreads();
        // keys above the bin are chosen whatever the later rounds decide
        const uint32_t lo1 = g.lo, span1 = g.hi - g.lo;
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
          const uint32_t d = key[q] - lo1;
          if (d <= span1) {
            const uint32_t s = atomicAdd(s_sel + 3, 1u);
            cand_key[s] = key[q];
            cand_pos[s] = uint32_t(slot_pos(q, tid));
          }
          sel |= uint32_t(key[q] > lo1 && d > span1) << q;
        }
        __syncthreads();
        const uint32_t nc = g.in_bin;
        const bool has = uint32_t(tid) < nc;
        const uint32_t ck = has ? cand_key[tid] : 0u, cp = has ? cand_pos[tid] : 0u;
        while (!range_done(g)) refine_cands(g, has, ck, hist, wsum, s_sel);
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
        // more than 1024 keys share the bin: refine over the registers
        while (!range_done(g)) refine_regs(g, key, hist, wsum, s_sel);
        uint32_t eq = 0;
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
          sel |= uint32_t(key[q] > g.hi) << q;
          eq |= uint32_t(key[q] >= g.lo && key[q] <= g.hi) << q;
        }
        if (g.in_bin == g.rem) {
          sel |= eq;
        } else {  // one key value: its lowest `rem` positions
          uint32_t lane_pre[kRounds];
          ordered_slots(eq, hist, wsum, lane_pre);
#pragma unroll
          for (int r = 0; r < kRounds; ++r) {
            uint32_t rank = hist[r * kWarps + warp] + lane_pre[r];
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
    }

    uint32_t lane_pre[kRounds];
    const uint32_t total_sel = ordered_slots(sel, hist, wsum, lane_pre);
    int32_t* out = idx + int64_t(row) * k;
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
      const uint32_t nib = (sel >> (4 * r)) & 15u;
      if (nib) {
        uint32_t slot = hist[r * kWarps + warp] + lane_pre[r];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if ((nib >> e) & 1u) out[slot++] = r * kRoundSpan + 4 * tid + e;
      }
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
                                                                     n, k, idx);
  return check_launch("topk");
}

}  // extern "C"
