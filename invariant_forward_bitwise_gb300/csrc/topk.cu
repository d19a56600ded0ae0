// Sparse-attention Top-K with a fixed tie-break and a fixed output order
// ("Finish RL Training Faster", section "让训练前向使用推理的数值": equal scores are
// resolved the same way every time and the selection is laid out in position
// order, so the same set is always accumulated in the same order).
//
// One CTA of 1024 threads per row.  Scores become order-preserving 32-bit keys
// (+0 and -0 map to one key; -inf and positions past valid_len are excluded)
// held in shared memory.  A 4-pass MSB-first radix select finds the k-th
// largest key T; every key > T is chosen, and among keys == T the lowest
// indices fill the remaining slots.  A stable compaction then writes the
// chosen indices in ascending order.  Only integer counts and ballots decide
// the result, so it is unique and independent of scheduling.
#include "common.cuh"

namespace biv {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxN = 40960;  // keys kept in shared memory (160 KB)

__device__ __forceinline__ uint32_t order_key(float s) {
  if (s == 0.f) s = 0.f;  // -0 -> +0
  const uint32_t u = __float_as_uint(s);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__global__ void __launch_bounds__(kThreads, 1)
    topk_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ valid_len,
                int n, int k, int32_t* __restrict__ idx) {
  extern __shared__ uint32_t sm[];
  uint32_t* keys = sm;                       // [n]; 0 = not selectable
  uint32_t* whist = sm + kMaxN;              // [kWarps][256]
  __shared__ uint32_t s_cnt[kWarps];
  __shared__ uint32_t s_cnt2[kWarps];
  __shared__ uint32_t s_sel[3];              // prefix, remaining, valid count

  const int row = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nv = min(max(valid_len[row], 0), n);
  const float* src = scores + int64_t(row) * ld;

  uint32_t cnt = 0;
  for (int j = tid; j < n; j += kThreads) {
    uint32_t key = 0;
    if (j < nv) {
      const float s = src[j];
      if (s != -INFINITY) key = order_key(s);
    }
    keys[j] = key;
    cnt += key != 0;
  }
  // valid count (integer, order-free)
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  if (lane == 0) s_cnt[warp] = cnt;
  __syncthreads();
  if (tid == 0) {
    uint32_t t = 0;
    for (int w = 0; w < kWarps; ++w) t += s_cnt[w];
    s_sel[2] = t;
    s_sel[0] = 0;
    s_sel[1] = uint32_t(k);
  }
  __syncthreads();
  const uint32_t total_valid = s_sel[2];
  const bool take_all = total_valid <= uint32_t(k);

  uint32_t want = 0, mask = 0;
  if (!take_all) {
    for (int byte = 3; byte >= 0; --byte) {
      const int sh = 8 * byte;
      for (int b = lane; b < 256; b += 32) whist[warp * 256 + b] = 0;
      __syncwarp();
      // uniform trip count: every lane of a warp reaches the ballot/match
      for (int base = 0; base < n; base += kThreads) {
        const int j = base + tid;
        const uint32_t key = j < n ? keys[j] : 0u;
        const bool hit = key != 0 && (key & mask) == want;
        const uint32_t bin = (key >> sh) & 255u;
        const uint32_t act = __ballot_sync(0xffffffffu, hit);
        if (hit) {
          const uint32_t peers = __match_any_sync(act, bin);
          if ((peers & ((1u << lane) - 1u)) == 0) whist[warp * 256 + bin] += __popc(peers);
        }
      }
      __syncthreads();
      // fold the per-warp histograms (thread b owns bin b)
      if (tid < 256) {
        uint32_t t = 0;
        for (int w = 0; w < kWarps; ++w) t += whist[w * 256 + tid];
        whist[tid] = t;  // warp 0's row now holds the totals (read below after sync)
      }
      __syncthreads();
      if (tid == 0) {
        uint32_t rem = s_sel[1];
        int chosen = 0;
        for (int b = 255; b >= 0; --b) {
          const uint32_t c = whist[b];
          if (rem <= c) {
            chosen = b;
            break;
          }
          rem -= c;
        }
        s_sel[0] |= uint32_t(chosen) << sh;
        s_sel[1] = rem;
      }
      __syncthreads();
      want = s_sel[0];
      mask |= 255u << sh;
    }
  }
  const uint32_t T = want;
  const uint32_t need_eq = take_all ? 0u : s_sel[1];

  // stable compaction in ascending index order, 1024 indices per round
  uint32_t eq_base = 0, out_base = 0;
  const uint32_t lt = (1u << lane) - 1u;
  for (int base = 0; base < n; base += kThreads) {
    const int j = base + tid;
    const uint32_t key = j < n ? keys[j] : 0u;
    const bool valid = key != 0;
    const bool gt = valid && (take_all || key > T);
    const bool eq = valid && !take_all && key == T;
    const uint32_t beq = __ballot_sync(0xffffffffu, eq);
    if (lane == 0) s_cnt[warp] = __popc(beq);
    __syncthreads();
    uint32_t eq_pre = eq_base, eq_tot = 0;
    for (int w = 0; w < kWarps; ++w) {
      const uint32_t c = s_cnt[w];
      if (w < warp) eq_pre += c;
      eq_tot += c;
    }
    const uint32_t eq_rank = eq_pre + __popc(beq & lt);
    const bool sel = gt || (eq && eq_rank < need_eq);
    const uint32_t bsel = __ballot_sync(0xffffffffu, sel);
    if (lane == 0) s_cnt2[warp] = __popc(bsel);
    __syncthreads();
    uint32_t sel_pre = out_base, sel_tot = 0;
    for (int w = 0; w < kWarps; ++w) {
      const uint32_t c = s_cnt2[w];
      if (w < warp) sel_pre += c;
      sel_tot += c;
    }
    if (sel) idx[int64_t(row) * k + sel_pre + __popc(bsel & lt)] = j;
    eq_base += eq_tot;
    out_base += sel_tot;
    __syncthreads();
  }
  for (int s = int(out_base) + tid; s < k; s += kThreads) idx[int64_t(row) * k + s] = -1;
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
  const int smem = (kMaxN + kWarps * 256) * 4;
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
      return set_error(BIV_ERR_CUDA, "topk: cannot set shared memory size");
    attr = true;
  }
  topk_kernel<<<rows, kThreads, smem, as_cuda(stream)>>>(scores, ld, valid_len, n, k, idx);
  return check_launch("topk");
}

}  // extern "C"
