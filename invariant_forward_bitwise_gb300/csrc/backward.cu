// Backward of the fused forward ops, for the trainer side that runs the
// inference ops' own backward ("No More Train-Inference Mismatch", section
// "方法细节") with the FP8 round trip passed straight through ("Finish RL
// Training Faster", section "让训练前向使用推理的数值").  Every reduction has
// one fixed order that depends on the shapes only (fixed per-row trees,
// ascending loops), so a gradient is the same bits run after run; a row's
// dx / dz / dq depends on that row alone.  FP32 on the CUDA cores.
//
//  RMSNorm   dx = inv * (w dy) - x * (inv^3 * sum(x w dy) / d); dw[c] = sum over
//            rows r ascending of dy x inv  (a second kernel, one thread per c)
//  SiLU-mul  dgate = dy * up * s * (1 + gate * (1 - s)), dup = dy * gate * s,
//            s = 1 / (1 + exp(-gate))
//  logprob   dz = dlp * (onehot(target) - exp(z - lse))
//  attention per (row, head): lse and D = do . o from one pass over the keys
//            in ascending order; dq from a second pass; dk, dv per (key, kv
//            head) from a pass over rows ascending, q heads ascending.
#include <algorithm>

#include "common.cuh"

namespace biv {
namespace {

constexpr int kBT = 256;   // threads of a row CTA (the tree depends on d only)

__device__ __forceinline__ float warp_sum_x(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
// sum over the CTA: per-thread value, warp xor tree, warps in order
__device__ __forceinline__ float cta_sum(float v, float* red) {
  v = warp_sum_x(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = 0.f;
  for (int i = 0; i < int(blockDim.x >> 5); ++i) t += red[i];
  return t;
}

__global__ void __launch_bounds__(kBT) rmsnorm_bwd_kernel(
    const uint16_t* __restrict__ x, int64_t xs, const uint16_t* __restrict__ w,
    const float* __restrict__ dy, int64_t dys, float* __restrict__ dx, int64_t dxs,
    float* __restrict__ t, int d, float eps) {
  __shared__ float red[kBT / 32];
  const int row = blockIdx.x;
  const uint16_t* xr = x + int64_t(row) * xs;
  const float* dr = dy + int64_t(row) * dys;
  float ss = 0.f, gx = 0.f;
  for (int c = threadIdx.x; c < d; c += kBT) {
    const float xv = bf2f(xr[c]);
    ss = fmaf(xv, xv, ss);
    gx = fmaf(dr[c] * bf2f(w[c]), xv, gx);
  }
  ss = cta_sum(ss, red);
  gx = cta_sum(gx, red);
  const float inv = 1.0f / sqrtf(ss / float(d) + eps);
  const float corr = inv * inv * inv * (gx / float(d));
  float* dxr = dx + int64_t(row) * dxs;
  float* tr = t + int64_t(row) * d;
  for (int c = threadIdx.x; c < d; c += kBT) {
    const float xv = bf2f(xr[c]);
    dxr[c] = inv * (dr[c] * bf2f(w[c])) - xv * corr;
    tr[c] = dr[c] * xv * inv;
  }
}

// dw[c] = sum over rows, ascending, of t[r, c]
__global__ void colsum_kernel(const float* __restrict__ t, int rows, int d, float* __restrict__ dw) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= d) return;
  float acc = 0.f;
  for (int r = 0; r < rows; ++r) acc += t[int64_t(r) * d + c];
  dw[c] = acc;
}

__global__ void silu_mul_bwd_kernel(const uint16_t* __restrict__ gu, int64_t gs,
                                    const float* __restrict__ dy, int64_t dys,
                                    float* __restrict__ dgu, int64_t dgs, int rows, int I) {
  const int64_t total = int64_t(rows) * I;
  for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < total;
       e += int64_t(gridDim.x) * blockDim.x) {
    const int r = int(e / I), c = int(e % I);
    const float g = bf2f(gu[int64_t(r) * gs + c]), u = bf2f(gu[int64_t(r) * gs + I + c]);
    const float s = 1.0f / (1.0f + expf(-g));
    const float d = dy[int64_t(r) * dys + c];
    dgu[int64_t(r) * dgs + c] = d * u * (s * (1.0f + g * (1.0f - s)));
    dgu[int64_t(r) * dgs + I + c] = d * (g * s);
  }
}

constexpr int kLT = 512;
__global__ void __launch_bounds__(kLT) logprob_bwd_kernel(
    const float* __restrict__ z, int64_t ld, const int32_t* __restrict__ target,
    const float* __restrict__ dlp, int V, float* __restrict__ dz, int64_t ldz, int* err) {
  __shared__ float red[kLT / 32];
  const int row = blockIdx.x;
  const float* zr = z + int64_t(row) * ld;
  float m = -INFINITY;
  for (int v = threadIdx.x; v < V; v += kLT) m = fmaxf(m, zr[v]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  m = -INFINITY;
  for (int i = 0; i < kLT / 32; ++i) m = fmaxf(m, red[i]);
  float se = 0.f;
  for (int v = threadIdx.x; v < V; v += kLT) se += expf(zr[v] - m);
  se = cta_sum(se, red);
  const float lse = m + logf(se);
  const int tg = target[row];
  if (tg < 0 || tg >= V) {
    if (threadIdx.x == 0) raise_error(err, kErrBadIndex);
  }
  const float g = dlp[row];
  float* dr = dz + int64_t(row) * ldz;
  for (int v = threadIdx.x; v < V; v += kLT) dr[v] = g * ((v == tg ? 1.0f : 0.0f) - expf(zr[v] - lse));
}

// ------------------------------------------------------------ attention --
// one warp per (row or key, head); lane l holds dims l, l+32, l+64, l+96 (< D)
struct AttnBwd {
  const uint16_t *q, *k, *v, *dout;
  float *dq, *dk, *dv;
  int Tq, Tk, Hq, Hkv, D;
  const int32_t *q_pos, *k_pos;
  float scale;
  float *lse, *Dr;
};

__device__ __forceinline__ void load4(const uint16_t* p, int D, int lane, float (&f)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int c = lane + 32 * i;
    f[i] = c < D ? bf2f(p[c]) : 0.f;
  }
}
__device__ __forceinline__ float dot4(const float (&a)[4], const float (&b)[4]) {
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) s = fmaf(a[i], b[i], s);
  return warp_sum_x(s);
}

// pass 1: lse and D = do . o per (row, q head), keys ascending (online softmax)
__global__ void attn_bwd_stats_kernel(const __grid_constant__ AttnBwd a) {
  const int64_t gw = (blockIdx.x * int64_t(blockDim.x) + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= int64_t(a.Tq) * a.Hq) return;
  const int i = int(gw / a.Hq), h = int(gw % a.Hq), kvh = h / (a.Hq / a.Hkv);
  float q[4], o[4] = {0.f, 0.f, 0.f, 0.f};
  load4(a.q + (int64_t(i) * a.Hq + h) * a.D, a.D, lane, q);
  float m = -INFINITY, l = 0.f;
  const int qp = a.q_pos[i];
  for (int j = 0; j < a.Tk; ++j) {
    if (a.k_pos[j] > qp) continue;
    float kk[4], vv[4];
    load4(a.k + (int64_t(j) * a.Hkv + kvh) * a.D, a.D, lane, kk);
    load4(a.v + (int64_t(j) * a.Hkv + kvh) * a.D, a.D, lane, vv);
    const float s = dot4(q, kk) * a.scale;
    const float mn = fmaxf(m, s);
    const float alpha = expf(m - mn), p = expf(s - mn);
    l = l * alpha + p;
#pragma unroll
    for (int x = 0; x < 4; ++x) o[x] = o[x] * alpha + p * vv[x];
    m = mn;
  }
  float dov[4];
  load4(a.dout + (int64_t(i) * a.Hq + h) * a.D, a.D, lane, dov);
  const float inv = l > 0.f ? 1.0f / l : 0.f;
#pragma unroll
  for (int x = 0; x < 4; ++x) o[x] *= inv;
  const float Dv = dot4(dov, o);
  if (lane == 0) {
    a.lse[gw] = l > 0.f ? m + logf(l) : INFINITY;   // a row with no key: p = 0 everywhere
    a.Dr[gw] = Dv;
  }
}

// pass 2: dq per (row, q head), keys ascending
__global__ void attn_bwd_dq_kernel(const __grid_constant__ AttnBwd a) {
  const int64_t gw = (blockIdx.x * int64_t(blockDim.x) + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= int64_t(a.Tq) * a.Hq) return;
  const int i = int(gw / a.Hq), h = int(gw % a.Hq), kvh = h / (a.Hq / a.Hkv);
  float q[4], dov[4], acc[4] = {0.f, 0.f, 0.f, 0.f};
  load4(a.q + (int64_t(i) * a.Hq + h) * a.D, a.D, lane, q);
  load4(a.dout + (int64_t(i) * a.Hq + h) * a.D, a.D, lane, dov);
  const float lse = a.lse[gw], Dv = a.Dr[gw];
  const int qp = a.q_pos[i];
  for (int j = 0; j < a.Tk; ++j) {
    if (a.k_pos[j] > qp) continue;
    float kk[4], vv[4];
    load4(a.k + (int64_t(j) * a.Hkv + kvh) * a.D, a.D, lane, kk);
    load4(a.v + (int64_t(j) * a.Hkv + kvh) * a.D, a.D, lane, vv);
    const float p = expf(dot4(q, kk) * a.scale - lse);
    const float ds = p * (dot4(dov, vv) - Dv);
#pragma unroll
    for (int x = 0; x < 4; ++x) acc[x] = fmaf(ds * a.scale, kk[x], acc[x]);
  }
  float* dst = a.dq + (int64_t(i) * a.Hq + h) * a.D;
#pragma unroll
  for (int x = 0; x < 4; ++x)
    if (lane + 32 * x < a.D) dst[lane + 32 * x] = acc[x];
}

// pass 3: dk, dv per (key, kv head), rows ascending, q heads of the group ascending
__global__ void attn_bwd_dkv_kernel(const __grid_constant__ AttnBwd a) {
  const int64_t gw = (blockIdx.x * int64_t(blockDim.x) + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= int64_t(a.Tk) * a.Hkv) return;
  const int j = int(gw / a.Hkv), kvh = int(gw % a.Hkv), G = a.Hq / a.Hkv;
  float kk[4], vv[4], dk[4] = {0.f, 0.f, 0.f, 0.f}, dv[4] = {0.f, 0.f, 0.f, 0.f};
  load4(a.k + (int64_t(j) * a.Hkv + kvh) * a.D, a.D, lane, kk);
  load4(a.v + (int64_t(j) * a.Hkv + kvh) * a.D, a.D, lane, vv);
  const int kp = a.k_pos[j];
  for (int i = 0; i < a.Tq; ++i) {
    if (a.q_pos[i] < kp) continue;
    for (int g = 0; g < G; ++g) {
      const int h = kvh * G + g;
      const int64_t rh = int64_t(i) * a.Hq + h;
      float q[4], dov[4];
      load4(a.q + rh * a.D, a.D, lane, q);
      load4(a.dout + rh * a.D, a.D, lane, dov);
      const float p = expf(dot4(q, kk) * a.scale - a.lse[rh]);
      const float ds = p * (dot4(dov, vv) - a.Dr[rh]);
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        dk[x] = fmaf(ds * a.scale, q[x], dk[x]);
        dv[x] = fmaf(p, dov[x], dv[x]);
      }
    }
  }
  float* dkd = a.dk + gw * a.D;
  float* dvd = a.dv + gw * a.D;
#pragma unroll
  for (int x = 0; x < 4; ++x)
    if (lane + 32 * x < a.D) {
      dkd[lane + 32 * x] = dk[x];
      dvd[lane + 32 * x] = dv[x];
    }
}

unsigned blocks_for_warps(int64_t warps) { return unsigned((warps * 32 + 255) / 256); }

}  // namespace
}  // namespace biv

using namespace biv;

extern "C" {

biv_status biv_rmsnorm_backward(const uint16_t* x, int64_t x_stride, const uint16_t* w,
                                const float* dy, int64_t dy_stride, float* dx, int64_t dx_stride,
                                float* dw, int rows, int d, float eps, void* workspace,
                                size_t workspace_bytes, biv_stream_t stream) {
  BIV_REQUIRE(rows >= 0 && d > 0, "rmsnorm_backward: bad shape");
  if (rows == 0) return BIV_OK;
  BIV_REQUIRE(x && w && dy && dx && dw, "rmsnorm_backward: null pointer");
  if (!workspace || workspace_bytes < size_t(rows) * d * sizeof(float))
    return set_error(BIV_ERR_WORKSPACE, "rmsnorm_backward: workspace of %zu bytes needed",
                     size_t(rows) * d * sizeof(float));
  cudaStream_t s = as_cuda(stream);
  float* t = static_cast<float*>(workspace);
  rmsnorm_bwd_kernel<<<rows, kBT, 0, s>>>(x, x_stride, w, dy, dy_stride, dx, dx_stride, t, d, eps);
  biv_status st = check_launch("rmsnorm_backward");
  if (st != BIV_OK) return st;
  colsum_kernel<<<(d + 255) / 256, 256, 0, s>>>(t, rows, d, dw);
  return check_launch("rmsnorm_backward_dw");
}

biv_status biv_silu_mul_backward(const uint16_t* gate_up, int64_t gs, const float* dy,
                                 int64_t dys, float* dgate_up, int64_t dgs, int rows, int I,
                                 biv_stream_t stream) {
  BIV_REQUIRE(rows >= 0 && I > 0, "silu_mul_backward: bad shape");
  if (rows == 0) return BIV_OK;
  BIV_REQUIRE(gate_up && dy && dgate_up, "silu_mul_backward: null pointer");
  const int64_t total = int64_t(rows) * I;
  const int blocks = int(std::min<int64_t>((total + 255) / 256, 152 * 16));
  silu_mul_bwd_kernel<<<blocks, 256, 0, as_cuda(stream)>>>(gate_up, gs, dy, dys, dgate_up, dgs,
                                                           rows, I);
  return check_launch("silu_mul_backward");
}

biv_status biv_logprob_backward(const float* logits, int64_t ld, const int32_t* target,
                                const float* dlp, int T, int V, float* dz, int64_t ldz,
                                biv_stream_t stream) {
  BIV_REQUIRE(T >= 0 && V > 0 && ld >= V && ldz >= V, "logprob_backward: bad shape");
  if (T == 0) return BIV_OK;
  BIV_REQUIRE(logits && target && dlp && dz, "logprob_backward: null pointer");
  logprob_bwd_kernel<<<T, kLT, 0, as_cuda(stream)>>>(logits, ld, target, dlp, V, dz, ldz,
                                                     device_error_word());
  return check_launch("logprob_backward");
}

biv_status biv_attention_backward(const biv_attn_bwd_desc* d, biv_stream_t stream) {
  BIV_REQUIRE(d, "attention_backward: null descriptor");
  BIV_REQUIRE(d->D > 0 && d->D <= 128 && d->Hq > 0 && d->Hkv > 0 && d->Hq % d->Hkv == 0 &&
                  d->Tq >= 0 && d->Tk >= 0,
              "attention_backward: D <= 128 and Hq a multiple of Hkv");
  if (d->Tq == 0) return BIV_OK;
  BIV_REQUIRE(d->q && d->k && d->v && d->dout && d->dq && d->dk && d->dv && d->q_pos && d->k_pos &&
                  d->workspace,
              "attention_backward: null pointer");
  AttnBwd a;
  a.q = d->q; a.k = d->k; a.v = d->v; a.dout = d->dout;
  a.dq = d->dq; a.dk = d->dk; a.dv = d->dv;
  a.Tq = d->Tq; a.Tk = d->Tk; a.Hq = d->Hq; a.Hkv = d->Hkv; a.D = d->D;
  a.q_pos = d->q_pos; a.k_pos = d->k_pos; a.scale = d->scale;
  a.lse = d->workspace;
  a.Dr = d->workspace + int64_t(d->Tq) * d->Hq;
  cudaStream_t s = as_cuda(stream);
  const int64_t rw = int64_t(d->Tq) * d->Hq, kw = int64_t(d->Tk) * d->Hkv;
  attn_bwd_stats_kernel<<<blocks_for_warps(rw), 256, 0, s>>>(a);
  biv_status st = check_launch("attention_backward_stats");
  if (st != BIV_OK) return st;
  attn_bwd_dq_kernel<<<blocks_for_warps(rw), 256, 0, s>>>(a);
  st = check_launch("attention_backward_dq");
  if (st != BIV_OK || kw == 0) return st;
  attn_bwd_dkv_kernel<<<blocks_for_warps(kw), 256, 0, s>>>(a);
  return check_launch("attention_backward_dkv");
}

}  // extern "C"
