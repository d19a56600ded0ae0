// Mamba-2 SSD scan whose decode step replays the prefill chunk order
// ("Finish RL Training Faster", section "一致性有多个层面": decode replays the
// prefill's chunked computation order and training reuses the same op).
//
// Chunks of Q positions are aligned to absolute positions.  Inside chunk
// [s0, s0+Q), with a_s = dt_s*A (per head) and L_t = a_{s0} + ... + a_t
// (sequential FP32 prefix sum), the output of row t is
//   y_t[p] = sum_{s=s0..t} (exp(L_t - L_s) * (C_t . B_s)) * (dt_s * x_s[p])
//            + sum_n (exp(L_t) * h_in[p][n]) * C_t[n] + D * x_t[p]
// accumulated in that order in one FP32 register (s ascending, then n
// ascending, then the skip term), and a closed chunk hands on
//   h_out[p][n] = exp(L_last) h_in[p][n] + sum_s (exp(L_last - L_s) * dt_s * x_s[p]) * B_s[n].
// Row t depends only on h_in and rows s0..t, so one code path serves a whole
// prefill, a chunked prefill and a token-by-token decode: the open chunk's
// rows are kept in a per-sequence buffer and re-read, never approximated.
//
// One CTA per (sequence, head); thread t_local owns row s0 + t_local.
#include "common.cuh"

namespace biv {
namespace {

constexpr int kP = 64, kN = 128, kMaxQ = 256;
constexpr int kLDC = kN + 8;  // padded C rows (bank spread for per-row reads)
constexpr int kFewRows = 4;   // at most this many new rows in a chunk: (row, p) threads

struct SsdSmem {
  uint16_t B[kMaxQ][kN];
  uint16_t C[kMaxQ][kLDC];
  uint16_t x[kMaxQ][kP];
  float dt[kMaxQ];
  float L[kMaxQ];
  float h[kP][kN];
  float W[4][kMaxQ];  // term weights of the new rows (few-row path)
};

__global__ void __launch_bounds__(256, 1) ssd_kernel(const biv_ssd_desc d) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SsdSmem& S = *reinterpret_cast<SsdSmem*>(smem_raw);
  const int i = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const int H = d.H, Q = d.chunk;
  const int n = d.n[i];
  if (n <= 0) return;
  const int pos0 = d.pos0[i], row0 = d.row0[i];
  const float A = d.A[h], Dh = d.D[h];
  float* state = d.state + (int64_t(i) * H + h) * kP * kN;
  uint16_t* bx = d.buf_x + int64_t(i) * Q * H * kP;
  uint16_t* bB = d.buf_B + int64_t(i) * Q * kN;
  uint16_t* bC = d.buf_C + int64_t(i) * Q * kN;
  float* bdt = d.buf_dt + int64_t(i) * Q * H;

  for (int e = tid; e < kP * kN; e += 256) S.h[e / kN][e % kN] = state[e];

  bool closed_any = false;
  const int c_first = pos0 / Q, c_last = (pos0 + n - 1) / Q;
  for (int c = c_first; c <= c_last; ++c) {
    const int s0 = c * Q;
    const int first = max(s0, pos0);
    const int last = min(s0 + Q, pos0 + n);  // exclusive
    const int cnt = last - s0;
    __syncthreads();
    // rows of the chunk: buffered (s0 .. first-1) then new (first .. last-1)
    for (int e = tid; e < cnt * (kN / 8); e += 256) {
      const int r = e / (kN / 8), q = e % (kN / 8);
      const int t = s0 + r;
      const uint4* srcB;
      const uint4* srcC;
      if (t < first) {
        srcB = reinterpret_cast<const uint4*>(bB + int64_t(r) * kN) + q;
        srcC = reinterpret_cast<const uint4*>(bC + int64_t(r) * kN) + q;
      } else {
        const int64_t row = row0 + (t - pos0);
        srcB = reinterpret_cast<const uint4*>(d.B + row * d.B_stride) + q;
        srcC = reinterpret_cast<const uint4*>(d.C + row * d.C_stride) + q;
      }
      *reinterpret_cast<uint4*>(&S.B[r][q * 8]) = *srcB;
      *reinterpret_cast<uint4*>(&S.C[r][q * 8]) = *srcC;
    }
    for (int e = tid; e < cnt * (kP / 8); e += 256) {
      const int r = e / (kP / 8), q = e % (kP / 8);
      const int t = s0 + r;
      const uint4* src;
      if (t < first)
        src = reinterpret_cast<const uint4*>(bx + (int64_t(r) * H + h) * kP) + q;
      else
        src = reinterpret_cast<const uint4*>(d.x + int64_t(row0 + (t - pos0)) * d.x_stride + int64_t(h) * kP) + q;
      *reinterpret_cast<uint4*>(&S.x[r][q * 8]) = *src;
    }
    for (int r = tid; r < cnt; r += 256) {
      const int t = s0 + r;
      S.dt[r] = t < first ? bdt[int64_t(r) * H + h] : d.dt[int64_t(row0 + (t - pos0)) * d.dt_stride + h];
    }
    __syncthreads();
    if (tid == 0) {
      float acc = 0.f;
      for (int r = 0; r < cnt; ++r) {
        acc += S.dt[r] * A;
        S.L[r] = acc;
      }
    }
    __syncthreads();

    // outputs of the new rows.  Few new rows (decode): threads over (row, p)
    // with the term weights w(t, s) staged in shared memory; many rows: one
    // thread per row.  Both evaluate every output with the same operations in
    // the same order (the weights, then the s sum, the n sum and the skip
    // term as fma chains), so they give the same bits.
    const int nnew = last - first;
    if (nnew <= kFewRows) {
      for (int e = tid; e < nnew * kMaxQ; e += 256) {
        const int j = e / kMaxQ, sidx = e % kMaxQ;
        const int rj = first - s0 + j;
        if (sidx > rj) continue;
        float cb = 0.f;
#pragma unroll 8
        for (int q = 0; q < kN; ++q) cb = fmaf(bf2f(S.C[rj][q]), bf2f(S.B[sidx][q]), cb);
        S.W[j][sidx] = expf(S.L[rj] - S.L[sidx]) * cb;
      }
      __syncthreads();
      if (tid < nnew * kP) {
        const int j = tid / kP, pp = tid % kP;
        const int rj = first - s0 + j;
        float acc = 0.f;
        for (int sidx = 0; sidx <= rj; ++sidx)
          acc = fmaf(S.W[j][sidx], S.dt[sidx] * bf2f(S.x[sidx][pp]), acc);
        const float eL = expf(S.L[rj]);
        for (int q = 0; q < kN; ++q) acc = fmaf(eL * S.h[pp][q], bf2f(S.C[rj][q]), acc);
        const int t = s0 + rj;
        uint16_t* y = d.y + int64_t(row0 + (t - pos0)) * d.y_stride + int64_t(h) * kP;
        y[pp] = f2bf(fmaf(Dh, bf2f(S.x[rj][pp]), acc));
      }
    }
    const int r = tid;
    if (nnew > kFewRows && r < cnt && s0 + r >= first) {
      const int t = s0 + r;
      const float Lt = S.L[r];
      float acc[kP];
#pragma unroll
      for (int p = 0; p < kP; ++p) acc[p] = 0.f;
      for (int s = 0; s <= r; ++s) {
        float cb = 0.f;
#pragma unroll 8
        for (int q = 0; q < kN; ++q) cb = fmaf(bf2f(S.C[r][q]), bf2f(S.B[s][q]), cb);
        const float w = expf(Lt - S.L[s]) * cb;
        const float dts = S.dt[s];
#pragma unroll
        for (int p = 0; p < kP; ++p) acc[p] = fmaf(w, dts * bf2f(S.x[s][p]), acc[p]);
      }
      const float eL = expf(Lt);
#pragma unroll 2
      for (int q = 0; q < kN; ++q) {
        const float cq = bf2f(S.C[r][q]);
#pragma unroll
        for (int p = 0; p < kP; ++p) acc[p] = fmaf(eL * S.h[p][q], cq, acc[p]);
      }
      uint16_t* y = d.y + int64_t(row0 + (t - pos0)) * d.y_stride + int64_t(h) * kP;
#pragma unroll
      for (int p = 0; p < kP; p += 2) {
        const float o0 = fmaf(Dh, bf2f(S.x[r][p]), acc[p]);
        const float o1 = fmaf(Dh, bf2f(S.x[r][p + 1]), acc[p + 1]);
        *reinterpret_cast<uint32_t*>(y + p) = pack_bf2(o0, o1);
      }
    }
    __syncthreads();
    if (last == s0 + Q) {
      // chunk closes: h_out from h_in and all Q rows
      const float Lend = S.L[Q - 1];
      const float eEnd = expf(Lend);
      for (int e = tid; e < kP * kN; e += 256) {
        const int p = e / kN, q = e % kN;
        float acc = 0.f;
        for (int s = 0; s < Q; ++s)
          acc = fmaf(expf(Lend - S.L[s]) * S.dt[s] * bf2f(S.x[s][p]), bf2f(S.B[s][q]), acc);
        S.h[p][q] = eEnd * S.h[p][q] + acc;
      }
      closed_any = true;
    } else {
      // chunk stays open: keep its new rows for the next call
      for (int e = tid; e < (last - first) * (kP / 8); e += 256) {
        const int rr = (first - s0) + e / (kP / 8), q = e % (kP / 8);
        reinterpret_cast<uint4*>(bx + (int64_t(rr) * H + h) * kP)[q] =
            *reinterpret_cast<const uint4*>(&S.x[rr][q * 8]);
      }
      for (int rr = (first - s0) + tid; rr < cnt; rr += 256) bdt[int64_t(rr) * H + h] = S.dt[rr];
      if (h == 0) {
        for (int e = tid; e < (last - first) * (kN / 8); e += 256) {
          const int rr = (first - s0) + e / (kN / 8), q = e % (kN / 8);
          reinterpret_cast<uint4*>(bB + int64_t(rr) * kN)[q] = *reinterpret_cast<const uint4*>(&S.B[rr][q * 8]);
          reinterpret_cast<uint4*>(bC + int64_t(rr) * kN)[q] = *reinterpret_cast<const uint4*>(&S.C[rr][q * 8]);
        }
      }
    }
  }
  __syncthreads();
  if (closed_any)
    for (int e = tid; e < kP * kN; e += 256) state[e] = S.h[e / kN][e % kN];
}

}  // namespace
}  // namespace biv

using namespace biv;

extern "C" {

biv_status biv_ssd_scan(const biv_ssd_desc* d, biv_stream_t stream) {
  BIV_REQUIRE(d, "ssd_scan: null descriptor");
  BIV_REQUIRE(d->P == kP && d->N == kN, "ssd_scan: supports P=%d, N=%d", kP, kN);
  BIV_REQUIRE(d->chunk == 64 || d->chunk == 128 || d->chunk == 256, "ssd_scan: chunk in {64,128,256}");
  BIV_REQUIRE(d->H > 0 && d->H <= 65535 && d->nseq >= 0 && d->nseq <= 0x7fffffff, "ssd_scan: bad sizes");
  if (d->nseq == 0) return BIV_OK;
  BIV_REQUIRE(d->x && d->dt && d->A && d->B && d->C && d->D && d->y && d->row0 && d->n && d->pos0 &&
                  d->state && d->buf_x && d->buf_B && d->buf_C && d->buf_dt,
              "ssd_scan: null pointer");
  BIV_REQUIRE(aligned16(d->x) && aligned16(d->B) && aligned16(d->C) && aligned16(d->buf_x) &&
                  aligned16(d->buf_B) && aligned16(d->buf_C) && (d->x_stride * 2) % 16 == 0 &&
                  (d->B_stride * 2) % 16 == 0 && (d->C_stride * 2) % 16 == 0,
              "ssd_scan: x/B/C rows must be 16-byte aligned");
  const int smem = int(sizeof(SsdSmem));
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(ssd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
      return set_error(BIV_ERR_CUDA, "ssd_scan: cannot set shared memory size");
    attr = true;
  }
  dim3 grid(d->nseq, d->H);
  ssd_kernel<<<grid, 256, smem, as_cuda(stream)>>>(*d);
  return check_launch("ssd_scan");
}

}  // extern "C"
