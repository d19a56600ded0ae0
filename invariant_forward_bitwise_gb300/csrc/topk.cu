// Sparse-attention Top-K with a fixed tie-break and a fixed output order
// ("Finish RL Training Faster", section "让训练前向使用推理的数值": equal scores are
// resolved the same way every time and the selection is laid out in position
// order, so the same set is always accumulated in the same order).
//
// One CTA of 1024 threads per row; thread t keeps keys t, t+1024, ... in
// registers (32 per thread).  Scores become order-preserving 32-bit keys (+0
// and -0 map to one key; -inf and positions past valid_len are excluded).  A
// 4-pass MSB-first radix select (per-warp shared-memory histograms, the
// k-th-largest bin found by a parallel scan) gives the k-th largest key T;
// every key > T is chosen, and among keys == T the lowest indices fill the
// remaining slots.  The chosen indices are written in ascending order: index
// j = i*1024 + 32*w + l is ranked by block-wide scans of per-(i, warp) ballot
// counts.  Only integer counts and ballots decide the result, so it is unique
// and independent of scheduling.
#include "common.cuh"

namespace biv {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kPer = 32;                    // keys per thread
constexpr int kMaxN = kThreads * kPer;      // 32768

__device__ __forceinline__ uint32_t order_key(float s) {
  if (s == 0.f) s = 0.f;  // -0 -> +0
  const uint32_t u = __float_as_uint(s);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

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

__global__ void __launch_bounds__(kThreads, 1)
    topk_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ valid_len,
                int n, int k, int32_t* __restrict__ idx) {
  __shared__ uint32_t whist[kWarps * 256];   // per-warp histograms; reused as scan tables
  __shared__ uint32_t wsum[kWarps];
  __shared__ uint32_t s_sel[2];              // chosen bin prefix, remaining count

  const int row = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nv = min(max(valid_len[row], 0), n);
  const float* src = scores + int64_t(row) * ld;

  uint32_t key[kPer];
  uint32_t cnt = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int j = i * kThreads + tid;
    uint32_t kk = 0;
    if (j < nv) {
      const float sc = __ldg(src + j);
      if (sc != -INFINITY) kk = order_key(sc);
    }
    key[i] = kk;
    cnt += kk != 0;
  }
  uint32_t total_valid;
  block_excl_scan(cnt, wsum, total_valid);
  const bool take_all = total_valid <= uint32_t(k);

  uint32_t want = 0, mask = 0, rem = uint32_t(k);
  if (!take_all) {
    for (int byte = 3; byte >= 0; --byte) {
      const int sh = 8 * byte;
      uint32_t* h = whist + warp * 256;
#pragma unroll
      for (int b = lane; b < 256; b += 32) h[b] = 0;
      __syncwarp();
      // shared-memory atomics into the warp's own histogram (measured faster
      // than warp-aggregating equal bins with match_any first)
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const uint32_t kk = key[i];
        if (kk != 0 && (kk & mask) == want) atomicAdd(h + ((kk >> sh) & 255u), 1u);
      }
      __syncthreads();
      // bins in descending order: thread t < 256 takes bin 255 - t; the bin
      // holding the rem-th largest key has (keys in higher bins) < rem <=
      // (keys in higher bins) + (its own keys)
      uint32_t c = 0;
      if (tid < 256) {
#pragma unroll 8
        for (int w = 0; w < kWarps; ++w) c += whist[w * 256 + 255 - tid];
      }
      __syncthreads();  // all histogram reads done before the scan reuses wsum
      uint32_t tot;
      const uint32_t above = block_excl_scan(c, wsum, tot);
      if (tid < 256 && above < rem && rem <= above + c) {
        s_sel[0] = uint32_t(255 - tid);
        s_sel[1] = rem - above;
      }
      __syncthreads();
      want |= s_sel[0] << sh;
      mask |= 255u << sh;
      rem = s_sel[1];
      __syncthreads();  // everyone has read s_sel and the histograms are free
    }
  }
  const uint32_t T = want;
  const uint32_t need_eq = take_all ? 0u : rem;
  const uint32_t lt = (1u << lane) - 1u;

  // ranks of equal keys: count per (round i, warp), scanned in index order
  // (table entry i*32 + w is owned by thread i*32 + w in the scan)
  uint32_t* tab = whist;  // [kPer][kWarps]
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const bool eq = !take_all && key[i] != 0 && key[i] == T;
    const uint32_t b = __ballot_sync(0xffffffffu, eq);
    if (lane == 0) tab[i * kWarps + warp] = __popc(b);
  }
  __syncthreads();
  uint32_t dummy;
  const uint32_t eq_pre = block_excl_scan(tab[tid], wsum, dummy);
  tab[tid] = eq_pre;
  __syncthreads();
  uint32_t* tab2 = whist + kPer * kWarps;  // [kPer][kWarps] selected counts
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const uint32_t kk = key[i];
    const bool valid = kk != 0;
    const bool eq = !take_all && valid && kk == T;
    const bool gt = valid && (take_all || kk > T);
    const uint32_t beq = __ballot_sync(0xffffffffu, eq);
    const uint32_t rank = tab[i * kWarps + warp] + __popc(beq & lt);
    const bool sel = gt || (eq && rank < need_eq);
    const uint32_t bs = __ballot_sync(0xffffffffu, sel);
    if (lane == 0) tab2[i * kWarps + warp] = __popc(bs);
  }
  __syncthreads();
  uint32_t total_sel;
  const uint32_t sel_pre = block_excl_scan(tab2[tid], wsum, total_sel);
  tab2[tid] = sel_pre;
  __syncthreads();
  int32_t* out = idx + int64_t(row) * k;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const uint32_t kk = key[i];
    const bool valid = kk != 0;
    const bool eq = !take_all && valid && kk == T;
    const bool gt = valid && (take_all || kk > T);
    const uint32_t beq = __ballot_sync(0xffffffffu, eq);
    const uint32_t rank = tab[i * kWarps + warp] + __popc(beq & lt);
    const bool sel = gt || (eq && rank < need_eq);
    const uint32_t bs = __ballot_sync(0xffffffffu, sel);
    if (sel) out[tab2[i * kWarps + warp] + __popc(bs & lt)] = i * kThreads + tid;
  }
  for (int s2 = int(total_sel) + tid; s2 < k; s2 += kThreads) out[s2] = -1;
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
  topk_kernel<<<rows, kThreads, 0, as_cuda(stream)>>>(scores, ld, valid_len, n, k, idx);
  return check_launch("topk");
}

}  // extern "C"
