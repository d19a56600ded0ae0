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
        acc = fmaf(S.dt[r], A, acc);
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
          acc = fmaf((expf(Lend - S.L[s]) * S.dt[s]) * bf2f(S.x[s][p]), bf2f(S.B[s][q]), acc);
        S.h[p][q] = fmaf(eEnd, S.h[p][q], acc);
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

// --------------------------------------------------- many-row path ----
// The same per-row formulas as ssd_kernel, spread over the GPU for calls with
// many new rows.  Every (sequence, chunk) pair the call touches and every head
// run in parallel; only the chunk-to-chunk state hand-over is sequential, and
// it is an elementwise fma per state entry:
//   ssd_cb_kernel     cb(t, s) = sum_q C_t[q] B_s[q] (fma chain), all heads share it
//   ssd_intra_kernel  intra(t, p) = sum_{s<=t} w(t,s) * (dt_s x_s[p]);  for a closing
//                     chunk dH(p, q) = sum_s ((e^{Lend-L_s} dt_s) x_s[p]) B_s[q], e^{Lend}
//   ssd_state_kernel  start state of each chunk; h <- fma(e^{Lend}, h, dH) per closed chunk
//   ssd_out_kernel    y = fma(D, x, intra + sum_q (e^{L_t} h[p][q]) C_t[q]); buffers of
//                     an open last chunk
// All sums run in the orders ssd_kernel uses, so either path gives the same bits.
struct SsdGeom {
  int n, pos0, row0, c, s0, first, last;  // chunk c = pos0/Q + blockIdx.y
  __device__ bool load(const biv_ssd_desc& d, int i, int cr) {
    n = d.n[i];
    if (n <= 0) return false;
    pos0 = d.pos0[i];
    row0 = d.row0[i];
    c = pos0 / d.chunk + cr;
    s0 = c * d.chunk;
    if (s0 >= pos0 + n) return false;
    first = max(s0, pos0);
    last = min(s0 + d.chunk, pos0 + n);
    return true;
  }
};

struct SsdWs {  // carve-up of the many-row workspace
  float* cb;    // [nseq][maxc][Q][Q]
  float* acc;   // [nseq][max_n][H][P]
  float* dH;    // [nseq][maxc][H][P][N]
  float* eEnd;  // [nseq][maxc][H]
  float* hst;   // [nseq][maxc][H][P][N]
};

__host__ __device__ inline int ssd_max_chunks(int max_n, int Q) { return (max_n + Q - 1) / Q + 1; }

__host__ __device__ inline SsdWs ssd_ws(void* base, const biv_ssd_desc& d) {
  const int64_t mc = ssd_max_chunks(d.max_n, d.chunk), Q = d.chunk;
  float* p = static_cast<float*>(base);
  SsdWs w;
  w.cb = p;
  p += int64_t(d.nseq) * mc * Q * Q;
  w.acc = p;
  p += int64_t(d.nseq) * d.max_n * d.H * kP;
  w.dH = p;
  p += int64_t(d.nseq) * mc * d.H * kP * kN;
  w.eEnd = p;
  p += (int64_t(d.nseq) * mc * d.H + 3) / 4 * 4;
  w.hst = p;
  p += int64_t(d.nseq) * mc * d.H * kP * kN;
  return w;
}

inline size_t ssd_ws_bytes(const biv_ssd_desc& d) {
  const int64_t mc = ssd_max_chunks(d.max_n, d.chunk), Q = d.chunk;
  const int64_t floats = int64_t(d.nseq) * mc * Q * Q + int64_t(d.nseq) * d.max_n * d.H * kP +
                         2 * int64_t(d.nseq) * mc * d.H * kP * kN +
                         (int64_t(d.nseq) * mc * d.H + 3) / 4 * 4;
  return size_t(floats) * sizeof(float);
}

// bf16 row of the chunk, local index r: the open chunk's buffer below `first`,
// the call's input at and above it
__device__ __forceinline__ const uint16_t* chunk_row(const SsdGeom& g, int r, const uint16_t* buf,
                                                     int64_t buf_stride, const uint16_t* in,
                                                     int64_t in_stride) {
  const int t = g.s0 + r;
  return t < g.first ? buf + int64_t(r) * buf_stride : in + int64_t(g.row0 + (t - g.pos0)) * in_stride;
}

constexpr int kCbRows = 32;   // rows t per ssd_cb_kernel CTA
constexpr int kLDB = kN + 2;  // padded B rows: consecutive rows start one bank apart

struct CbSmem {
  uint16_t B[kMaxQ][kLDB];
  uint16_t C[kCbRows][kN];
};

__global__ void __launch_bounds__(256) ssd_cb_kernel(const biv_ssd_desc d, SsdWs w) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  CbSmem& S = *reinterpret_cast<CbSmem*>(smem_raw);
  auto& sB = S.B;
  auto& sC = S.C;
  const int i = blockIdx.x, cr = blockIdx.y, tb = blockIdx.z, tid = threadIdx.x;
  SsdGeom g;
  if (!g.load(d, i, cr)) return;
  const int t_lo = max(g.first - g.s0, tb * kCbRows), t_hi = min(g.last - g.s0, tb * kCbRows + kCbRows);
  if (t_lo >= t_hi) return;
  const uint16_t* bB = d.buf_B + int64_t(i) * d.chunk * kN;
  const uint16_t* bC = d.buf_C + int64_t(i) * d.chunk * kN;
  for (int e = tid; e < t_hi * (kN / 2); e += 256) {
    const int r = e / (kN / 2), q2 = e % (kN / 2);
    const uint16_t* src = chunk_row(g, r, bB, kN, d.B, d.B_stride);
    *reinterpret_cast<uint32_t*>(&sB[r][2 * q2]) = reinterpret_cast<const uint32_t*>(src)[q2];
  }
  for (int e = tid; e < (t_hi - t_lo) * (kN / 8); e += 256) {
    const int r = t_lo + e / (kN / 8), q = e % (kN / 8);
    const uint16_t* src = chunk_row(g, r, bC, kN, d.C, d.C_stride);
    *reinterpret_cast<uint4*>(&sC[r - t_lo][q * 8]) = reinterpret_cast<const uint4*>(src)[q];
  }
  __syncthreads();
  const int sidx = tid;  // thread = key row s
  float* out = w.cb + (int64_t(i) * ssd_max_chunks(d.max_n, d.chunk) + cr) * d.chunk * d.chunk;
  for (int t = t_lo; t < t_hi; ++t) {
    if (sidx > t) continue;
    float cb = 0.f;
#pragma unroll 16
    for (int q = 0; q < kN; q += 2) {
      const uint32_t b2 = *reinterpret_cast<const uint32_t*>(&sB[sidx][q]);
      const uint32_t c2 = *reinterpret_cast<const uint32_t*>(&sC[t - t_lo][q]);
      cb = fmaf(bf2f(uint16_t(c2 & 0xFFFF)), bf2f(uint16_t(b2 & 0xFFFF)), cb);
      cb = fmaf(bf2f(uint16_t(c2 >> 16)), bf2f(uint16_t(b2 >> 16)), cb);
    }
    out[int64_t(t) * d.chunk + sidx] = cb;
  }
}

constexpr int kST = 32;            // key rows s per weight tile
constexpr int kWP = kST + 1;        // padded weight-tile row: rows one bank apart

struct IntraSmem {
  uint16_t x[kMaxQ][kP];
  uint16_t B[kMaxQ][kN];
  float dt[kMaxQ];
  float L[kMaxQ];
  float v[kMaxQ][kP];      // dt_s * x_s[p]; for a closing chunk reused as u[s][p]
  float wt[kMaxQ][kWP];    // w(t, s) of one tile of kST key rows
};

// rows 0 .. cnt-1 of the chunk: dt and x of head h (buffer below `first`)
__device__ void load_dt_x(const biv_ssd_desc& d, const SsdGeom& g, int i, int h, int cnt, float* dt,
                          uint16_t (*x)[kP]) {
  const int H = d.H, tid = threadIdx.x;
  const float* bdt = d.buf_dt + int64_t(i) * d.chunk * H;
  const uint16_t* bx = d.buf_x + int64_t(i) * d.chunk * H * kP;
  for (int r = tid; r < cnt; r += blockDim.x) {
    const int t = g.s0 + r;
    dt[r] = t < g.first ? bdt[int64_t(r) * H + h] : d.dt[int64_t(g.row0 + (t - g.pos0)) * d.dt_stride + h];
  }
  for (int e = tid; e < cnt * (kP / 8); e += blockDim.x) {
    const int r = e / (kP / 8), q = e % (kP / 8);
    const int t = g.s0 + r;
    const uint16_t* src = t < g.first ? bx + (int64_t(r) * H + h) * kP
                                      : d.x + int64_t(g.row0 + (t - g.pos0)) * d.x_stride + int64_t(h) * kP;
    *reinterpret_cast<uint4*>(&x[r][q * 8]) = reinterpret_cast<const uint4*>(src)[q];
  }
}

// the chunk's decay prefix L_r = L_{r-1} + dt_r A (one thread, in order)
__device__ void decay_prefix(const float* dt, float A, int cnt, float* L) {
  if (threadIdx.x == 0) {
    float acc = 0.f;
    for (int r = 0; r < cnt; ++r) {
      acc = fmaf(dt[r], A, acc);
      L[r] = acc;
    }
  }
}

constexpr int kSsdThreads = 512;   // many-row path CTAs: 16 warps per SM hide shared-memory latency

__global__ void __launch_bounds__(kSsdThreads, 1) ssd_intra_kernel(const biv_ssd_desc d, SsdWs w) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  IntraSmem& S = *reinterpret_cast<IntraSmem*>(smem_raw);
  const int i = blockIdx.x, cr = blockIdx.y, h = blockIdx.z, tid = threadIdx.x;
  SsdGeom g;
  if (!g.load(d, i, cr)) return;
  const int Q = d.chunk, cnt = g.last - g.s0, fr = g.first - g.s0;
  const int64_t ci = int64_t(i) * ssd_max_chunks(d.max_n, Q) + cr;
  load_dt_x(d, g, i, h, cnt, S.dt, S.x);
  __syncthreads();
  decay_prefix(S.dt, d.A[h], cnt, S.L);
  for (int e = tid; e < cnt * kP; e += kSsdThreads) {
    const int sidx = e / kP, p = e % kP;
    S.v[sidx][p] = S.dt[sidx] * bf2f(S.x[sidx][p]);
  }
  __syncthreads();
  // intra-chunk sums of the new rows [fr, cnt).  Thread (k, quarter) owns
  // rows fr+k and cnt-1-k (balanced: their key counts add up to the same
  // total) and 16 columns p; keys go by tiles of kST in ascending order, each
  // tile's weights formed once in shared memory.
  constexpr int PC = kP / 4;
  const int nnew = cnt - fr;
  const int k = tid & 127, pc = (tid >> 7) * PC;
  const int ra = fr + k, rb = cnt - 1 - k;
  const bool has_a = k < (nnew + 1) / 2, has_b = has_a && rb != ra;
  float acc_a[PC], acc_b[PC];
#pragma unroll
  for (int c = 0; c < PC; ++c) acc_a[c] = acc_b[c] = 0.f;
  const float* cbase = w.cb + ci * Q * Q;
  for (int s0 = 0; s0 < cnt; s0 += kST) {
    // weights of the tile: the C.B products of rows max(fr, s0) .. cnt-1 come
    // in row by row (one warp reads a row's kST = 32 values, coalesced), then
    // each becomes w = e^{L_r - L_s} * cb in place
    const int rlo = max(fr, s0);
    for (int e = tid; e < (cnt - rlo) * kST; e += kSsdThreads) {
      const int r = rlo + e / kST, c = e % kST, sidx = s0 + c;
      S.wt[r][c] = sidx <= r ? expf(S.L[r] - S.L[sidx]) * cbase[int64_t(r) * Q + sidx] : 0.f;
    }
    __syncthreads();
    const int cmax = min(kST, cnt - s0);
    if (has_a && ra >= s0) {
      const int ce = min(cmax, ra - s0 + 1);
      for (int c = 0; c < ce; ++c) {
        const float wv = S.wt[ra][c];
        const float4* vr = reinterpret_cast<const float4*>(&S.v[s0 + c][pc]);
#pragma unroll
        for (int j = 0; j < PC / 4; ++j) {
          const float4 v4 = vr[j];
          acc_a[4 * j] = fmaf(wv, v4.x, acc_a[4 * j]);
          acc_a[4 * j + 1] = fmaf(wv, v4.y, acc_a[4 * j + 1]);
          acc_a[4 * j + 2] = fmaf(wv, v4.z, acc_a[4 * j + 2]);
          acc_a[4 * j + 3] = fmaf(wv, v4.w, acc_a[4 * j + 3]);
        }
      }
    }
    if (has_b && rb >= s0) {
      const int ce = min(cmax, rb - s0 + 1);
      for (int c = 0; c < ce; ++c) {
        const float wv = S.wt[rb][c];
        const float4* vr = reinterpret_cast<const float4*>(&S.v[s0 + c][pc]);
#pragma unroll
        for (int j = 0; j < PC / 4; ++j) {
          const float4 v4 = vr[j];
          acc_b[4 * j] = fmaf(wv, v4.x, acc_b[4 * j]);
          acc_b[4 * j + 1] = fmaf(wv, v4.y, acc_b[4 * j + 1]);
          acc_b[4 * j + 2] = fmaf(wv, v4.z, acc_b[4 * j + 2]);
          acc_b[4 * j + 3] = fmaf(wv, v4.w, acc_b[4 * j + 3]);
        }
      }
    }
    __syncthreads();
  }
  auto put = [&](int r, const float (&acc)[PC]) {
    float4* dst = reinterpret_cast<float4*>(
        w.acc + ((int64_t(i) * d.max_n + (g.s0 + r - g.pos0)) * d.H + h) * kP + pc);
#pragma unroll
    for (int j = 0; j < PC / 4; ++j)
      dst[j] = make_float4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]);
  };
  if (has_a) put(ra, acc_a);
  if (has_b) put(rb, acc_b);
  if (g.last != g.s0 + Q) return;  // the chunk stays open: no hand-over yet
  // closing chunk: dH and e^{Lend}
  const float Lend = S.L[Q - 1];
  const uint16_t* bB = d.buf_B + int64_t(i) * Q * kN;
  for (int e = tid; e < Q * (kN / 8); e += kSsdThreads) {
    const int rr = e / (kN / 8), q = e % (kN / 8);
    const uint16_t* src = chunk_row(g, rr, bB, kN, d.B, d.B_stride);
    *reinterpret_cast<uint4*>(&S.B[rr][q * 8]) = reinterpret_cast<const uint4*>(src)[q];
  }
  for (int e = tid; e < Q * kP; e += kSsdThreads) {  // u[s][p] = (e^{Lend-L_s} dt_s) x_s[p]
    const int sidx = e / kP, p = e % kP;
    S.v[sidx][p] = (expf(Lend - S.L[sidx]) * S.dt[sidx]) * bf2f(S.x[sidx][p]);
  }
  __syncthreads();
  const int q = tid % kN, pb = (tid / kN) * PC;  // this thread: column q, rows pb .. pb+15
  float acc[PC];
#pragma unroll
  for (int c = 0; c < PC; ++c) acc[c] = 0.f;
  for (int sidx = 0; sidx < Q; ++sidx) {
    const float bq = bf2f(S.B[sidx][q]);
    const float4* ur = reinterpret_cast<const float4*>(&S.v[sidx][pb]);
#pragma unroll
    for (int j = 0; j < PC / 4; ++j) {
      const float4 u4 = ur[j];
      acc[4 * j] = fmaf(u4.x, bq, acc[4 * j]);
      acc[4 * j + 1] = fmaf(u4.y, bq, acc[4 * j + 1]);
      acc[4 * j + 2] = fmaf(u4.z, bq, acc[4 * j + 2]);
      acc[4 * j + 3] = fmaf(u4.w, bq, acc[4 * j + 3]);
    }
  }
  float* dH = w.dH + (ci * d.H + h) * kP * kN;
#pragma unroll
  for (int c = 0; c < PC; ++c) dH[(pb + c) * kN + q] = acc[c];
  if (tid == 0) w.eEnd[ci * d.H + h] = expf(Lend);
}

// chunk start states and the sequence's state after the call
__global__ void __launch_bounds__(256) ssd_state_kernel(const biv_ssd_desc d, SsdWs w) {
  const int i = blockIdx.x, h = blockIdx.y, e = blockIdx.z * 256 + threadIdx.x;
  const int n = d.n[i];
  if (n <= 0 || e >= kP * kN) return;
  const int pos0 = d.pos0[i], Q = d.chunk;
  const int mc = ssd_max_chunks(d.max_n, Q);
  float* state = d.state + (int64_t(i) * d.H + h) * kP * kN;
  float hv = state[e];
  bool closed = false;
  for (int cr = 0; cr < mc; ++cr) {
    const int s0 = (pos0 / Q + cr) * Q;
    if (s0 >= pos0 + n) break;
    const int64_t ci = int64_t(i) * mc + cr;
    w.hst[(ci * d.H + h) * kP * kN + e] = hv;
    if (s0 + Q <= pos0 + n) {
      hv = fmaf(w.eEnd[ci * d.H + h], hv, w.dH[(ci * d.H + h) * kP * kN + e]);
      closed = true;
    }
  }
  if (closed) state[e] = hv;
}

constexpr int kHP = kP + 4;  // transposed state rows (16-byte aligned)

struct OutSmem {
  float hT[kN][kHP];          // chunk start state, transposed: hT[q][p] = h[p][q]
  uint16_t x[kMaxQ][kP];
  uint16_t C[kMaxQ][kLDB];  // rows one bank apart: thread r reads row r
  float dt[kMaxQ];
  float L[kMaxQ];
};

__global__ void __launch_bounds__(kSsdThreads, 1) ssd_out_kernel(const biv_ssd_desc d, SsdWs w) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  OutSmem& S = *reinterpret_cast<OutSmem*>(smem_raw);
  const int i = blockIdx.x, cr = blockIdx.y, h = blockIdx.z, tid = threadIdx.x;
  SsdGeom g;
  if (!g.load(d, i, cr)) return;
  const int Q = d.chunk, H = d.H, cnt = g.last - g.s0;
  const int64_t ci = int64_t(i) * ssd_max_chunks(d.max_n, Q) + cr;
  load_dt_x(d, g, i, h, cnt, S.dt, S.x);
  const float* hs = w.hst + (ci * H + h) * kP * kN;
  for (int e = tid; e < kP * kN; e += kSsdThreads) S.hT[e % kN][e / kN] = hs[e];
  const int fr = g.first - g.s0;
  for (int e = tid; e < (cnt - fr) * (kN / 2); e += kSsdThreads) {
    const int r = fr + e / (kN / 2), q2 = e % (kN / 2);
    const uint32_t* src = reinterpret_cast<const uint32_t*>(d.C + int64_t(g.row0 + (g.s0 + r - g.pos0)) * d.C_stride) + q2;
    *reinterpret_cast<uint32_t*>(&S.C[r][2 * q2]) = *src;
  }
  __syncthreads();
  decay_prefix(S.dt, d.A[h], cnt, S.L);
  __syncthreads();
  // thread (row r, half): the 32 columns p of its half
  constexpr int PH = kP / 2;
  const int r = tid % kMaxQ, p0 = (tid / kMaxQ) * PH;
  if (r < cnt && r >= fr) {
    const int j = g.s0 + r - g.pos0;  // new-row index of the call
    const float4* src = reinterpret_cast<const float4*>(w.acc + ((int64_t(i) * d.max_n + j) * H + h) * kP + p0);
    float acc[PH];
#pragma unroll
    for (int p = 0; p < PH; p += 4) {
      const float4 v = src[p / 4];
      acc[p] = v.x; acc[p + 1] = v.y; acc[p + 2] = v.z; acc[p + 3] = v.w;
    }
    const float eL = expf(S.L[r]);
#pragma unroll 2
    for (int q = 0; q < kN; ++q) {
      const float cq = bf2f(S.C[r][q]);
      const float4* hq = reinterpret_cast<const float4*>(&S.hT[q][p0]);
#pragma unroll
      for (int jj = 0; jj < PH / 4; ++jj) {
        const float4 h4 = hq[jj];
        acc[4 * jj] = fmaf(eL * h4.x, cq, acc[4 * jj]);
        acc[4 * jj + 1] = fmaf(eL * h4.y, cq, acc[4 * jj + 1]);
        acc[4 * jj + 2] = fmaf(eL * h4.z, cq, acc[4 * jj + 2]);
        acc[4 * jj + 3] = fmaf(eL * h4.w, cq, acc[4 * jj + 3]);
      }
    }
    const float Dh = d.D[h];
    uint16_t* y = d.y + int64_t(g.row0 + j) * d.y_stride + int64_t(h) * kP + p0;
#pragma unroll
    for (int p = 0; p < PH; p += 2) {
      const float o0 = fmaf(Dh, bf2f(S.x[r][p0 + p]), acc[p]);
      const float o1 = fmaf(Dh, bf2f(S.x[r][p0 + p + 1]), acc[p + 1]);
      *reinterpret_cast<uint32_t*>(y + p) = pack_bf2(o0, o1);
    }
  }
  if (g.last == g.s0 + Q) return;
  // the chunk stays open: keep its new rows for the next call
  uint16_t* bx = d.buf_x + int64_t(i) * Q * H * kP;
  float* bdt = d.buf_dt + int64_t(i) * Q * H;
  for (int e = tid; e < (cnt - fr) * (kP / 8); e += kSsdThreads) {
    const int rr = fr + e / (kP / 8), q = e % (kP / 8);
    reinterpret_cast<uint4*>(bx + (int64_t(rr) * H + h) * kP)[q] = *reinterpret_cast<const uint4*>(&S.x[rr][q * 8]);
  }
  for (int rr = fr + tid; rr < cnt; rr += kSsdThreads) bdt[int64_t(rr) * H + h] = S.dt[rr];
  if (h == 0) {
    uint16_t* bB = d.buf_B + int64_t(i) * Q * kN;
    uint16_t* bC = d.buf_C + int64_t(i) * Q * kN;
    for (int e = tid; e < (cnt - fr) * (kN / 8); e += kSsdThreads) {
      const int rr = fr + e / (kN / 8), q = e % (kN / 8);
      const int64_t row = g.row0 + (g.s0 + rr - g.pos0);
      reinterpret_cast<uint4*>(bB + int64_t(rr) * kN)[q] = reinterpret_cast<const uint4*>(d.B + row * d.B_stride)[q];
      reinterpret_cast<uint4*>(bC + int64_t(rr) * kN)[q] = reinterpret_cast<const uint4*>(d.C + row * d.C_stride)[q];
    }
  }
}

template <typename Kern>
biv_status set_smem(Kern kern, size_t bytes, bool& done) {
  if (!done) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes)) !=
        cudaSuccess)
      return set_error(BIV_ERR_CUDA, "ssd_scan: cannot set shared memory size");
    done = true;
  }
  return BIV_OK;
}

biv_status validate_ssd(const biv_ssd_desc* d) {
  BIV_REQUIRE(d, "ssd_scan: null descriptor");
  BIV_REQUIRE(d->P == kP && d->N == kN, "ssd_scan: supports P=%d, N=%d", kP, kN);
  BIV_REQUIRE(d->chunk == 64 || d->chunk == 128 || d->chunk == 256, "ssd_scan: chunk in {64,128,256}");
  BIV_REQUIRE(d->H > 0 && d->H <= 65535 && d->nseq >= 0 && d->nseq <= 65535 && d->max_n >= 0,
              "ssd_scan: bad sizes");
  return BIV_OK;
}

// many new rows in some sequence: the parallel path (when given its workspace)
bool many_rows(const biv_ssd_desc& d) { return d.max_n > kFewRows; }

}  // namespace
}  // namespace biv

using namespace biv;

extern "C" {

biv_status biv_ssd_workspace(const biv_ssd_desc* d, size_t* bytes) {
  biv_status st = validate_ssd(d);
  if (st != BIV_OK) return st;
  BIV_REQUIRE(bytes, "ssd_workspace: null output");
  *bytes = many_rows(*d) ? ssd_ws_bytes(*d) : 0;
  return BIV_OK;
}

biv_status biv_ssd_scan(const biv_ssd_desc* d, biv_stream_t stream) {
  biv_status st = validate_ssd(d);
  if (st != BIV_OK) return st;
  if (d->nseq == 0) return BIV_OK;
  BIV_REQUIRE(d->x && d->dt && d->A && d->B && d->C && d->D && d->y && d->row0 && d->n && d->pos0 &&
                  d->state && d->buf_x && d->buf_B && d->buf_C && d->buf_dt,
              "ssd_scan: null pointer");
  BIV_REQUIRE(aligned16(d->x) && aligned16(d->B) && aligned16(d->C) && aligned16(d->buf_x) &&
                  aligned16(d->buf_B) && aligned16(d->buf_C) && (d->x_stride * 2) % 16 == 0 &&
                  (d->B_stride * 2) % 16 == 0 && (d->C_stride * 2) % 16 == 0,
              "ssd_scan: x/B/C rows must be 16-byte aligned");
  cudaStream_t s = as_cuda(stream);
  const size_t need = many_rows(*d) ? ssd_ws_bytes(*d) : 0;
  if (need && d->workspace && d->workspace_bytes >= need && aligned16(d->workspace)) {
    static bool a1 = false, a2 = false, a3 = false;
    if ((st = set_smem(ssd_cb_kernel, sizeof(CbSmem), a1)) != BIV_OK) return st;
    if ((st = set_smem(ssd_intra_kernel, sizeof(IntraSmem), a2)) != BIV_OK) return st;
    if ((st = set_smem(ssd_out_kernel, sizeof(OutSmem), a3)) != BIV_OK) return st;
    const SsdWs w = ssd_ws(d->workspace, *d);
    const int mc = ssd_max_chunks(d->max_n, d->chunk);
    ssd_cb_kernel<<<dim3(d->nseq, mc, d->chunk / kCbRows), 256, sizeof(CbSmem), s>>>(*d, w);
    if ((st = check_launch("ssd_cb")) != BIV_OK) return st;
    ssd_intra_kernel<<<dim3(d->nseq, mc, d->H), kSsdThreads, sizeof(IntraSmem), s>>>(*d, w);
    if ((st = check_launch("ssd_intra")) != BIV_OK) return st;
    ssd_state_kernel<<<dim3(d->nseq, d->H, kP * kN / 256), 256, 0, s>>>(*d, w);
    if ((st = check_launch("ssd_state")) != BIV_OK) return st;
    ssd_out_kernel<<<dim3(d->nseq, mc, d->H), kSsdThreads, sizeof(OutSmem), s>>>(*d, w);
    return check_launch("ssd_out");
  }
  static bool a0 = false;
  if ((st = set_smem(ssd_kernel, sizeof(SsdSmem), a0)) != BIV_OK) return st;
  dim3 grid(d->nseq, d->H);
  ssd_kernel<<<grid, 256, sizeof(SsdSmem), s>>>(*d);
  return check_launch("ssd_scan");
}

}  // extern "C"
