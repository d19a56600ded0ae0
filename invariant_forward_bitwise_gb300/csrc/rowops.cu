// Row-wise memory-bound kernels of the invariant forward.  Each output row is
// computed by one fixed thread/warp arrangement that depends only on the row
// length (never on the number of rows), with reductions in a fixed tree, so a
// row's bits do not depend on the batch it is in.
#include "common.cuh"

namespace biv {

namespace {

constexpr int kNormThreads = 256;  // fixed: the RMSNorm tree depends on d only
constexpr int kLogprobThreads = 512;
constexpr int kLogprobAhead = 8;  // logit chunks a thread loads before using them

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  return make_uint4(pack_bf2(f[0], f[1]), pack_bf2(f[2], f[3]), pack_bf2(f[4], f[5]),
                    pack_bf2(f[6], f[7]));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// ------------------------------------------------------------------ embed --
__global__ void embed_kernel(const int32_t* __restrict__ ids, const uint16_t* __restrict__ table,
                             int vocab, int d, uint16_t* __restrict__ h, int64_t h_stride,
                             int* err) {
  pdl_wait();     // stream predecessor done, its writes visible
  pdl_trigger();
  const int t = blockIdx.x;
  const int id = ids[t];
  uint4* dst = reinterpret_cast<uint4*>(h + int64_t(t) * h_stride);
  const int chunks = d / 8;
  if (id < 0 || id >= vocab) {
    for (int c = threadIdx.x; c < chunks; c += blockDim.x) dst[c] = make_uint4(0, 0, 0, 0);
    if (threadIdx.x == 0) raise_error(err, kErrBadIndex);
    return;
  }
  const uint4* src = reinterpret_cast<const uint4*>(table + int64_t(id) * d);
  for (int c = threadIdx.x; c < chunks; c += blockDim.x) dst[c] = __ldg(src + c);
}

// ------------------------------------------------------- add + RMSNorm ----
// One CTA of kNormThreads per row.  Thread t owns 8-element chunks
// t, t+256, ...; sum of squares: per-thread in chunk order, warp xor tree,
// then the 8 warp sums added in warp order.
// 8 consecutive bf16 outputs of a GEMM whose chunk partials were left for the
// consumer: fold the partials in chunk order, round once (what the GEMM's own
// fold kernel stores)
// GEMM chunk partials hold at most this many chunks (the GEMM's schedule)
constexpr int kMaxPartialChunks = 8;

// 8 consecutive columns of one row folded over the chunks in chunk order and
// rounded to bf16 (what the GEMM's own fold stores).  Every chunk's loads are
// issued before the first add so that the chunks' latencies overlap.
__device__ __forceinline__ void fold8(const biv_partials& xp, int64_t row, int col, float (&f)[8]) {
  const float* src = xp.p + row * xp.ld + col;
  float4 a[kMaxPartialChunks], b[kMaxPartialChunks];
#pragma unroll
  for (int c = 0; c < kMaxPartialChunks; ++c) {
    if (c < xp.chunks) {
      const float* sc = src + c * xp.chunk_stride;
      a[c] = __ldcg(reinterpret_cast<const float4*>(sc));
      b[c] = __ldcg(reinterpret_cast<const float4*>(sc + 4));
    }
  }
  float t[8] = {a[0].x, a[0].y, a[0].z, a[0].w, b[0].x, b[0].y, b[0].z, b[0].w};
#pragma unroll
  for (int c = 1; c < kMaxPartialChunks; ++c) {
    if (c < xp.chunks) {
      t[0] = t[0] + a[c].x; t[1] = t[1] + a[c].y; t[2] = t[2] + a[c].z; t[3] = t[3] + a[c].w;
      t[4] = t[4] + b[c].x; t[5] = t[5] + b[c].y; t[6] = t[6] + b[c].z; t[7] = t[7] + b[c].w;
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) f[j] = bf2f(f2bf(t[j]));
}

// 4 consecutive columns of one row folded like fold8.
__device__ __forceinline__ void fold4(const biv_partials& xp, int64_t row, int col, float (&f)[4]) {
  const float* src = xp.p + row * xp.ld + col;
  float4 a[kMaxPartialChunks];
#pragma unroll
  for (int c = 0; c < kMaxPartialChunks; ++c)
    if (c < xp.chunks) a[c] = __ldcg(reinterpret_cast<const float4*>(src + c * xp.chunk_stride));
  float t[4] = {a[0].x, a[0].y, a[0].z, a[0].w};
#pragma unroll
  for (int c = 1; c < kMaxPartialChunks; ++c) {
    if (c < xp.chunks) {
      t[0] = t[0] + a[c].x; t[1] = t[1] + a[c].y; t[2] = t[2] + a[c].z; t[3] = t[3] + a[c].w;
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) f[j] = bf2f(f2bf(t[j]));
}

template <int CPT, bool PARTIAL>  // chunks per thread (ceil(d/8/256)); x as partials
__global__ void __launch_bounds__(kNormThreads) add_rmsnorm_kernel(
    const uint16_t* __restrict__ x, int64_t xs, const biv_partials xp, uint16_t* __restrict__ r,
    int64_t rs, const uint16_t* __restrict__ w, uint16_t* __restrict__ y, int64_t ys, int d,
    float eps) {
  pdl_wait();     // stream predecessor done, its writes visible
  pdl_trigger();
  __shared__ float warp_ss[kNormThreads / 32];
  const int row = blockIdx.x;
  const int chunks = d / 8;
  const uint4* xr = reinterpret_cast<const uint4*>(x + int64_t(row) * xs);
  uint4* rr = r ? reinterpret_cast<uint4*>(r + int64_t(row) * rs) : nullptr;
  float v[CPT][8];
  float ss = 0.f;
  // the weights go out with the row's loads, not after the reduction
  const uint4* wr = reinterpret_cast<const uint4*>(w);
  uint4 wq[CPT];
#pragma unroll
  for (int i = 0; i < CPT; ++i) {
    const int c = threadIdx.x + i * kNormThreads;
    wq[i] = c < chunks ? __ldg(wr + c) : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int i = 0; i < CPT; ++i) {
    const int c = threadIdx.x + i * kNormThreads;
    if (c < chunks) {
      if (PARTIAL)
        fold8(xp, row, c * 8, v[i]);
      else
        unpack8(xr[c], v[i]);
      if (rr) {
        float rv[8];
        unpack8(rr[c], rv);
#pragma unroll
        for (int j = 0; j < 8; ++j) v[i][j] = bf2f(f2bf(v[i][j] + rv[j]));
        rr[c] = pack8(v[i]);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) ss = fmaf(v[i][j], v[i][j], ss);
    }
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) warp_ss[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < kNormThreads / 32; ++i) tot += warp_ss[i];
  const float inv = 1.0f / sqrtf(tot / float(d) + eps);
  uint4* yr = reinterpret_cast<uint4*>(y + int64_t(row) * ys);
#pragma unroll
  for (int i = 0; i < CPT; ++i) {
    const int c = threadIdx.x + i * kNormThreads;
    if (c < chunks) {
      float wv[8], o[8];
      unpack8(wq[i], wv);
#pragma unroll
      for (int j = 0; j < 8; ++j) o[j] = (v[i][j] * inv) * wv[j];
      yr[c] = pack8(o);
    }
  }
}

// ------------------------------------------------------------- SiLU-mul ----
// gate_up given as bf16 rows: one thread per 8 columns.
__global__ void silu_mul_kernel(const uint16_t* __restrict__ gu, int64_t gs,
                                uint16_t* __restrict__ y, int64_t ys, int rows, int I) {
  pdl_wait();     // stream predecessor done, its writes visible
  pdl_trigger();
  const int cpr = I / 8;
  const int64_t total = int64_t(rows) * cpr;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int row = int(i / cpr), c = int(i % cpr);
    const uint4* g = reinterpret_cast<const uint4*>(gu + int64_t(row) * gs);
    float gv[8], uv[8], o[8];
    unpack8(g[c], gv);
    unpack8(g[cpr + c], uv);
#pragma unroll
    for (int j = 0; j < 8; ++j) o[j] = (gv[j] / (1.0f + expf(-gv[j]))) * uv[j];
    reinterpret_cast<uint4*>(y + int64_t(row) * ys)[c] = pack8(o);
  }
}

// gate_up given as the chunk partials of the GEMM that produced it, folded
// here to the same bf16 values: one thread per 4 columns (the chunk loads of
// both halves stay in registers)
__global__ void silu_mul_partials_kernel(const biv_partials gp, uint16_t* __restrict__ y,
                                         int64_t ys, int rows, int I) {
  pdl_wait();     // stream predecessor done, its writes visible
  pdl_trigger();
  const int cpr = I / 4;
  const int64_t total = int64_t(rows) * cpr;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int row = int(i / cpr), c = int(i % cpr);
    float gv[4], uv[4], o[4];
    fold4(gp, row, c * 4, gv);
    fold4(gp, row, I + c * 4, uv);
#pragma unroll
    for (int j = 0; j < 4; ++j) o[j] = (gv[j] / (1.0f + expf(-gv[j]))) * uv[j];
    reinterpret_cast<uint2*>(y + int64_t(row) * ys)[c] = make_uint2(pack_bf2(o[0], o[1]),
                                                                     pack_bf2(o[2], o[3]));
  }
}

// ------------------------------------------------------------ RoPE table --
__global__ void rope_table_kernel(double theta, int D, int max_pos, float* cos_sin) {
  const int half = D / 2;
  const int64_t n = int64_t(max_pos) * half;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int p = int(i / half), j = int(i % half);
    const double inv_freq = pow(theta, -(2.0 * j) / double(D));
    const double ang = double(p) * inv_freq;
    cos_sin[i] = float(cos(ang));
    cos_sin[n + i] = float(sin(ang));
  }
}

// ------------------------------------------------------- QK-norm + RoPE ----
// The rotation of one pair (a, b) at angle (c, s), rounded to bf16: the one
// instruction sequence every kernel that applies RoPE uses.
__device__ __forceinline__ void rope_pair(float a, float b, float c, float s, uint16_t& oa,
                                          uint16_t& ob) {
  oa = f2bf(fmaf(a, c, -(b * s)));
  ob = f2bf(fmaf(b, c, a * s));
}

// One warp per (token, head).  Lane l owns the rotation pairs p = l, l+32
// (p < D/2) holding elements p and p + D/2.
__global__ void qk_norm_rope_kernel(uint16_t* __restrict__ qkv, int64_t rs, int T, int Hq,
                                    int Hkv, int D, const uint16_t* __restrict__ qw,
                                    const uint16_t* __restrict__ kw,
                                    const float* __restrict__ cos_sin, int max_pos,
                                    const int32_t* __restrict__ pos, float eps, int* err) {
  pdl_wait();     // stream predecessor done, its writes visible
  pdl_trigger();
  const int heads = Hq + Hkv;
  const int64_t gw = (blockIdx.x * int64_t(blockDim.x) + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= int64_t(T) * heads) return;
  const int t = int(gw / heads), h = int(gw % heads);
  const bool is_q = h < Hq;
  const uint16_t* wn = is_q ? qw : kw;
  uint16_t* v = qkv + int64_t(t) * rs + int64_t(h) * D;
  const int half = D / 2;
  int p = pos[t];
  if (p < 0 || p >= max_pos) {
    if (lane == 0) raise_error(err, kErrBadIndex);
    p = 0;
  }
  float a[2], b[2];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int j = lane + 32 * i;
    a[i] = b[i] = 0.f;
    if (j < half) {
      a[i] = bf2f(v[j]);
      b[i] = bf2f(v[j + half]);
      ss = fmaf(a[i], a[i], ss);
      ss = fmaf(b[i], b[i], ss);
    }
  }
  if (wn) {
    ss = warp_sum(ss);
    const float inv = 1.0f / sqrtf(ss / float(D) + eps);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int j = lane + 32 * i;
      if (j < half) {
        a[i] = bf2f(f2bf((a[i] * inv) * bf2f(wn[j])));
        b[i] = bf2f(f2bf((b[i] * inv) * bf2f(wn[j + half])));
      }
    }
  }
  const int64_t n = int64_t(max_pos) * half;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int j = lane + 32 * i;
    if (j < half) {
      const float c = cos_sin[int64_t(p) * half + j];
      const float s = cos_sin[n + int64_t(p) * half + j];
      rope_pair(a[i], b[i], c, s, v[j], v[j + half]);
    }
  }
}

// --------------------------------------------------------------- KV store --
__global__ void kv_store_bf16_kernel(const uint16_t* __restrict__ k,
                                     const uint16_t* __restrict__ v, int64_t rs,
                                     const int64_t* __restrict__ slot, int T, int Hkv, int D,
                                     uint16_t* __restrict__ kc, uint16_t* __restrict__ vc) {
  pdl_wait();     // stream predecessor done, its writes visible
  pdl_trigger();
  const int cpv = D / 8;  // 16-byte chunks per head vector
  const int64_t total = int64_t(T) * Hkv * cpv * 2;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * blockDim.x) {
    int64_t r = i;
    const int c = int(r % cpv); r /= cpv;
    const int h = int(r % Hkv); r /= Hkv;
    const int which = int(r % 2); r /= 2;
    const int t = int(r);
    const int64_t s = slot[t];
    if (s < 0) continue;
    const uint16_t* src = (which ? v : k) + int64_t(t) * rs + int64_t(h) * D;
    uint16_t* dst = (which ? vc : kc) + (s * Hkv + h) * D;
    reinterpret_cast<uint4*>(dst)[c] = reinterpret_cast<const uint4*>(src)[c];
  }
}

// One warp per (token, kv head, K|V): amax, scale, codes.
__global__ void kv_fp8_quant_kernel(const uint16_t* __restrict__ k,
                                    const uint16_t* __restrict__ v, int64_t rs,
                                    const int64_t* __restrict__ slot, int T, int Hkv, int D,
                                    uint8_t* __restrict__ kc, uint8_t* __restrict__ vc,
                                    float* __restrict__ ks, float* __restrict__ vs) {
  pdl_wait();     // stream predecessor done, its writes visible
  pdl_trigger();
  const int64_t gw = (blockIdx.x * int64_t(blockDim.x) + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= int64_t(T) * Hkv * 2) return;
  const int which = int(gw % 2);
  const int h = int((gw / 2) % Hkv);
  const int t = int(gw / 2 / Hkv);
  const int64_t s = slot[t];
  if (s < 0) return;
  const uint16_t* src = (which ? v : k) + int64_t(t) * rs + int64_t(h) * D;
  float x[4];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int j = lane + 32 * i;
    x[i] = j < D ? bf2f(src[j]) : 0.f;
    amax = fmaxf(amax, fabsf(x[i]));
  }
  amax = warp_max(amax);
  const float sc = amax == 0.f ? 1.0f : amax / 448.0f;
  uint8_t* dst = (which ? vc : kc) + (s * Hkv + h) * D;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int j = lane + 32 * i;
    if (j < D) dst[j] = f2e4m3(x[i] / sc);
  }
  if (lane == 0) (which ? vs : ks)[s * Hkv + h] = sc;
}

// QKV finalize: one warp per (token, head) over the q, k and v heads.  It
// computes what the QKV GEMM's fold, qk_norm_rope and kv_store_bf16 /
// kv_fp8_quant compute one after another, with the same operations per
// element, in one pass: fold the GEMM's chunk partials (when given) and round
// to bf16; QK-RMSNorm and RoPE on q and k heads; write q, k, v back into qkv;
// store k and v of rows with a cache slot into the paged cache (bf16, or e4m3
// codes with scale amax/448 per (token, head)).
template <bool PARTIAL>
__global__ void qkv_finalize_kernel(uint16_t* __restrict__ qkv, int64_t rs, const biv_partials xp,
                                    int T, int Hq, int Hkv, int D, const uint16_t* __restrict__ qw,
                                    const uint16_t* __restrict__ kw,
                                    const float* __restrict__ cos_sin, int max_pos,
                                    const int32_t* __restrict__ pos, float eps,
                                    const int64_t* __restrict__ slot, int fp8, void* kc, void* vc,
                                    float* ks, float* vs, int* err) {
  pdl_wait();     // stream predecessor done, its writes visible
  pdl_trigger();
  const int heads = Hq + 2 * Hkv;
  const int64_t gw = (blockIdx.x * int64_t(blockDim.x) + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= int64_t(T) * heads) return;
  const int t = int(gw / heads), h = int(gw % heads);
  const int kind = h < Hq ? 0 : (h < Hq + Hkv ? 1 : 2);  // q, k, v
  uint16_t* v = qkv + int64_t(t) * rs + int64_t(h) * D;
  const int half = D / 2;
  // loads that do not depend on the values go out first, so that their
  // latencies overlap the partials' instead of following them
  const int p_in = kind < 2 ? pos[t] : 0;
  const int64_t sl = kind > 0 ? slot[t] : -1;
  const uint16_t* wn = kind == 0 ? qw : (kind == 1 ? kw : nullptr);
  float wa[2] = {0.f, 0.f}, wb[2] = {0.f, 0.f};
  if (wn) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int j = lane + 32 * i;
      if (j < half) {
        wa[i] = bf2f(wn[j]);
        wb[i] = bf2f(wn[j + half]);
      }
    }
  }
  float a[2], b[2];
  uint16_t oa[2], ob[2];
  if (!PARTIAL) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int j = lane + 32 * i;
      a[i] = j < half ? bf2f(v[j]) : 0.f;
      b[i] = j < half ? bf2f(v[j + half]) : 0.f;
    }
  } else {
    // the GEMM's fold: chunk-order FP32 sum, rounded to bf16; all loads are
    // issued before the first add
    const float* src = xp.p + int64_t(t) * xp.ld + int64_t(h) * D;
    float pa[2][kMaxPartialChunks], pb[2][kMaxPartialChunks];
#pragma unroll
    for (int c = 0; c < kMaxPartialChunks; ++c) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int j = lane + 32 * i;
        if (c < xp.chunks && j < half) {
          pa[i][c] = __ldcg(src + c * xp.chunk_stride + j);
          pb[i][c] = __ldcg(src + c * xp.chunk_stride + j + half);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      a[i] = b[i] = 0.f;
      if (lane + 32 * i < half) {
        a[i] = pa[i][0];
        b[i] = pb[i][0];
#pragma unroll
        for (int c = 1; c < kMaxPartialChunks; ++c) {
          if (c < xp.chunks) {
            a[i] = a[i] + pa[i][c];
            b[i] = b[i] + pb[i][c];
          }
        }
        a[i] = bf2f(f2bf(a[i]));
        b[i] = bf2f(f2bf(b[i]));
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    oa[i] = f2bf(a[i]);
    ob[i] = f2bf(b[i]);
  }
  if (kind < 2) {
    int p = p_in;
    if (p < 0 || p >= max_pos) {
      if (lane == 0) raise_error(err, kErrBadIndex);
      p = 0;
    }
    if (wn) {
      float ss = 0.f;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        if (lane + 32 * i < half) {
          ss = fmaf(a[i], a[i], ss);
          ss = fmaf(b[i], b[i], ss);
        }
      }
      ss = warp_sum(ss);
      const float inv = 1.0f / sqrtf(ss / float(D) + eps);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int j = lane + 32 * i;
        if (j < half) {
          a[i] = bf2f(f2bf((a[i] * inv) * wa[i]));
          b[i] = bf2f(f2bf((b[i] * inv) * wb[i]));
        }
      }
    }
    const int64_t n = int64_t(max_pos) * half;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int j = lane + 32 * i;
      if (j < half) {
        const float c = cos_sin[int64_t(p) * half + j];
        const float s = cos_sin[n + int64_t(p) * half + j];
        rope_pair(a[i], b[i], c, s, oa[i], ob[i]);
      }
    }
  }
  if (PARTIAL || kind < 2) {  // v rows already hold their values unless folded here
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int j = lane + 32 * i;
      if (j < half) {
        v[j] = oa[i];
        v[j + half] = ob[i];
      }
    }
  }
  if (kind == 0) return;
  if (sl < 0) return;
  const int hk = h - Hq - (kind == 2 ? Hkv : 0);
  const int64_t base = (sl * Hkv + hk) * D;
  if (!fp8) {
    uint16_t* dst = static_cast<uint16_t*>(kind == 1 ? kc : vc) + base;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int j = lane + 32 * i;
      if (j < half) {
        dst[j] = oa[i];
        dst[j + half] = ob[i];
      }
    }
    return;
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    if (lane + 32 * i < half) amax = fmaxf(amax, fmaxf(fabsf(bf2f(oa[i])), fabsf(bf2f(ob[i]))));
  }
  amax = warp_max(amax);
  const float sc = amax == 0.f ? 1.0f : amax / 448.0f;
  uint8_t* dst = static_cast<uint8_t*>(kind == 1 ? kc : vc) + base;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int j = lane + 32 * i;
    if (j < half) {
      dst[j] = f2e4m3(bf2f(oa[i]) / sc);
      dst[j + half] = f2e4m3(bf2f(ob[i]) / sc);
    }
  }
  if (lane == 0) (kind == 1 ? ks : vs)[sl * Hkv + hk] = sc;
}

__global__ void kv_fp8_gather_kernel(const uint8_t* __restrict__ codes,
                                     const float* __restrict__ scales,
                                     const int32_t* __restrict__ bt, int max_pages,
                                     const int32_t* __restrict__ ctx,
                                     const int64_t* __restrict__ row0, int Hkv, int D, int page,
                                     uint16_t* __restrict__ out) {
  const int i = blockIdx.y;
  const int n = ctx[i];
  const int per_tok = Hkv * D;
  for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < int64_t(n) * per_tok;
       e += int64_t(gridDim.x) * blockDim.x) {
    const int t = int(e / per_tok);
    const int hd = int(e % per_tok);
    const int64_t s = int64_t(bt[int64_t(i) * max_pages + t / page]) * page + t % page;
    const float sc = scales[s * Hkv + hd / D];
    out[(row0[i] + t) * per_tok + hd] = f2bf(e4m32f(codes[s * per_tok + hd]) * sc);
  }
}

// ---------------------------------------------------- activation quant ----
// Half a warp per (row, 128-wide group), 8 values a lane (16-byte loads):
// amax over the 16 lanes, s = amax / 448 (1 when amax = 0), codes by RNE.
__device__ __forceinline__ float half_warp_max(float v) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Quantise the 8 values of one lane of its group (K % 16 == 0: a lane's
// values are all in the row or none); every lane of the warp calls this for
// the shuffles, and only lanes with `on` store: their codes, and lane % 16 ==
// 0 the group's scale.
__device__ __forceinline__ void quant8_store(const float (&v)[8], bool on, uint8_t* dst,
                                             float* scale_dst, int lane) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
  amax = half_warp_max(amax);
  const float sc = amax == 0.f ? 1.0f : amax / 448.0f;
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 8; ++i) w[i >> 2] |= uint32_t(f2e4m3(v[i] / sc)) << (8 * (i & 3));
  if (!on) return;
  *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
  if ((lane & 15) == 0) *scale_dst = sc;
}

__global__ void act_quant_kernel(const uint16_t* __restrict__ x, int64_t xs, int rows, int K,
                                 uint8_t* __restrict__ codes, float* __restrict__ scales) {
  const int groups = (K + 127) / 128;
  const int64_t hw = (blockIdx.x * int64_t(blockDim.x) + threadIdx.x) >> 4;   // half warp
  const int lane = threadIdx.x & 31;
  const bool on = hw < int64_t(rows) * groups;   // both halves of a warp reach the shuffles
  const int row = on ? int(hw / groups) : 0, g = on ? int(hw % groups) : 0;
  const int c0 = g * 128 + (lane & 15) * 8;
  const bool live = on && c0 < K;
  float v[8];
  if (live) {
    unpack8(*reinterpret_cast<const uint4*>(x + int64_t(row) * xs + c0), v);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = 0.f;
  }
  quant8_store(v, live, codes + int64_t(row) * K + c0, scales + int64_t(row) * groups + g, lane);
}

// SiLU-mul and the activation quantisation of its result in one pass: each
// value is the bf16 silu_mul_kernel stores, quantised as act_quant_kernel
// quantises it (the bf16 activation itself is not written).  Half a warp per
// (row, 128-wide group), 8 values a lane.
__global__ void silu_mul_quant_kernel(const uint16_t* __restrict__ gu, int64_t gs, int rows, int I,
                                      uint8_t* __restrict__ codes, float* __restrict__ scales) {
  pdl_wait();     // stream predecessor done, its writes visible
  pdl_trigger();
  const int groups = (I + 127) / 128;
  const int64_t hw = (blockIdx.x * int64_t(blockDim.x) + threadIdx.x) >> 4;   // half warp
  const int lane = threadIdx.x & 31;
  const bool on = hw < int64_t(rows) * groups;   // both halves of a warp reach the shuffles
  const int row = on ? int(hw / groups) : 0, g = on ? int(hw % groups) : 0;
  const int c0 = g * 128 + (lane & 15) * 8;
  const bool live = on && c0 < I;
  float v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = 0.f;
  if (live) {
    const uint16_t* gr = gu + int64_t(row) * gs;
    float gv[8], uv[8];
    unpack8(*reinterpret_cast<const uint4*>(gr + c0), gv);
    unpack8(*reinterpret_cast<const uint4*>(gr + I + c0), uv);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = bf2f(f2bf((gv[i] / (1.0f + expf(-gv[i]))) * uv[i]));
  }
  quant8_store(v, live, codes + int64_t(row) * I + c0, scales + int64_t(row) * groups + g, lane);
}

// -------------------------------------------------------------- logprob ----
// One CTA of 512 threads per row.  Thread t folds float4 chunks t, t+512, ...
// into an online (max, sumexp) pair; pairs are then merged by a warp xor tree
// and the 16 warp results in warp order.
__device__ __forceinline__ void lse_merge(float& m, float& s, float m2, float s2) {
  const float mn = fmaxf(m, m2);
  const float a = (m == -INFINITY) ? 0.f : s * expf(m - mn);
  const float b = (m2 == -INFINITY) ? 0.f : s2 * expf(m2 - mn);
  m = mn;
  s = a + b;
}

__global__ void __launch_bounds__(kLogprobThreads) logprob_kernel(
    const float* __restrict__ z, int64_t ld, const int32_t* __restrict__ target, int V,
    float* __restrict__ lp, int* err) {
  pdl_wait();     // stream predecessor done, its writes visible
  pdl_trigger();
  __shared__ float sm_m[kLogprobThreads / 32], sm_s[kLogprobThreads / 32];
  const int row = blockIdx.x;
  const float4* zr = reinterpret_cast<const float4*>(z + int64_t(row) * ld);
  const int chunks = V / 4;
  float m = -INFINITY, s = 0.f;
  auto update = [&](const float4& q) {
    const float cm = fmaxf(fmaxf(q.x, q.y), fmaxf(q.z, q.w));
    if (cm > m) {
      s = (m == -INFINITY) ? 0.f : s * expf(m - cm);
      m = cm;
    }
    s += expf(q.x - m);
    s += expf(q.y - m);
    s += expf(q.z - m);
    s += expf(q.w - m);
  };
  // the thread's chunks c, c + T, c + 2T, ... in that order; the loads of
  // kLogprobAhead of them are issued before the first update
  constexpr int kStep = kLogprobThreads * kLogprobAhead;
  for (int c0 = threadIdx.x; c0 < chunks; c0 += kStep) {
    float4 q[kLogprobAhead];
#pragma unroll
    for (int u = 0; u < kLogprobAhead; ++u)
      if (c0 + u * kLogprobThreads < chunks) q[u] = __ldcs(zr + c0 + u * kLogprobThreads);
#pragma unroll
    for (int u = 0; u < kLogprobAhead; ++u)
      if (c0 + u * kLogprobThreads < chunks) update(q[u]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    lse_merge(m, s, m2, s2);
  }
  if ((threadIdx.x & 31) == 0) {
    sm_m[threadIdx.x >> 5] = m;
    sm_s[threadIdx.x >> 5] = s;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float M = sm_m[0], S = sm_s[0];
    for (int i = 1; i < kLogprobThreads / 32; ++i) lse_merge(M, S, sm_m[i], sm_s[i]);
    int tg = target[row];
    if (tg < 0 || tg >= V) {
      raise_error(err, kErrBadIndex);
      lp[row] = NAN;
      return;
    }
    lp[row] = z[int64_t(row) * ld + tg] - (M + logf(S));
  }
}

// ---------------------------------------------------------------- router --
// One warp per row; logits staged in shared memory.
constexpr int kRouterWarps = 4;
__global__ void router_kernel(const float* __restrict__ logits, int64_t ld, int rows, int E,
                              int k, int32_t* __restrict__ idx, float* __restrict__ w) {
  extern __shared__ float sm_router[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kRouterWarps + warp;
  if (row >= rows) return;
  float* z = sm_router + warp * E;
  const float* src = logits + int64_t(row) * ld;
  float m = -INFINITY;
  for (int e = lane; e < E; e += 32) {
    z[e] = src[e];
    m = fmaxf(m, z[e]);
  }
  m = warp_max(m);
  float den = 0.f;
  for (int e = lane; e < E; e += 32) den += expf(z[e] - m);
  den = warp_sum(den);
  __syncwarp();
  for (int s = 0; s < k; ++s) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int e = lane; e < E; e += 32) {
      const float v = z[e];
      if (isnan(v)) continue;  // chosen entries are marked NaN
      if (v > bv || (v == bv && e < bi)) {
        bv = v;
        bi = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
      const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
      if (v2 > bv || (v2 == bv && i2 < bi)) {
        bv = v2;
        bi = i2;
      }
    }
    if (lane == 0) {
      idx[int64_t(row) * k + s] = bi;
      w[int64_t(row) * k + s] = expf(bv - m) / den;
    }
    __syncwarp();
    if (lane == (bi & 31)) z[bi] = NAN;
    __syncwarp();
  }
}

// ------------------------------------------------------------- dispatch ----
// One CTA per expert e.  e's first slot is the number of entries routed to
// an expert below e (a per-thread count, then one block sum: order-free
// integers).  Then e's entries are placed in ascending (t, s) order, 4096 per
// round (4 consecutive entries a thread) by a block-wide scan of the hit
// counts, so the layout is unique.
__device__ __forceinline__ int warp_incl_scan_i(int x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

__global__ void __launch_bounds__(1024) moe_dispatch_kernel(const int32_t* __restrict__ idx,
                                                            int n, int E,
                                                            int32_t* __restrict__ offsets,
                                                            int32_t* __restrict__ perm,
                                                            int32_t* __restrict__ src_row) {
  __shared__ int wsum[32];
  __shared__ int s_start;
  const int e = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int below = 0;
  for (int i = tid; i < n; i += blockDim.x) {
    const int v = idx[i];
    below += (v >= 0 && v < e) ? 1 : 0;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) below += __shfl_xor_sync(0xffffffffu, below, o);
  if (lane == 0) wsum[warp] = below;
  __syncthreads();
  if (warp == 0) {
    int x = wsum[lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    if (lane == 0) s_start = x;
  }
  __syncthreads();
  const int start = s_start;
  int at = start;
  for (int base = 0; base < n; base += 4 * int(blockDim.x)) {
    const int i0 = base + 4 * tid;
    bool hit[4];
    int c = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      hit[j] = i0 + j < n && idx[i0 + j] == e;
      c += hit[j] ? 1 : 0;
    }
    const int incl = warp_incl_scan_i(c, lane);
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    const int ws = wsum[lane];
    const int wi = warp_incl_scan_i(ws, lane);
    const int tot = __shfl_sync(0xffffffffu, wi, 31);
    int r = at + __shfl_sync(0xffffffffu, wi - ws, warp) + incl - c;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (hit[j]) {
        perm[r] = i0 + j;
        src_row[i0 + j] = r;
        ++r;
      }
    }
    at += tot;
    __syncthreads();   // wsum is rewritten next round
  }
  if (tid == 0) {
    offsets[e] = start;
    if (e == E - 1) offsets[E] = at;
  }
}

__global__ void gather_rows_kernel(const uint8_t* __restrict__ src, int64_t ss,
                                   const int32_t* __restrict__ perm, int k_div, int n,
                                   int row_bytes, uint8_t* __restrict__ dst, int64_t ds) {
  pdl_wait();     // stream predecessor done, its writes visible
  pdl_trigger();
  const int cpr = row_bytes / 16;
  const int64_t total = int64_t(n) * cpr;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int r = int(i / cpr), c = int(i % cpr);
    const int64_t s = perm[r] / k_div;
    reinterpret_cast<uint4*>(dst + r * ds)[c] = reinterpret_cast<const uint4*>(src + s * ss)[c];
  }
}

// --------------------------------------------------------------- combine --
__global__ void moe_combine_kernel(const uint16_t* __restrict__ y,
                                   const int32_t* __restrict__ src_row,
                                   const float* __restrict__ w, const uint16_t* __restrict__ sh,
                                   uint16_t* __restrict__ out, int T, int k, int d) {
  const int cpr = d / 8;
  const int64_t total = int64_t(T) * cpr;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int t = int(i / cpr), c = int(i % cpr);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int s = 0; s < k; ++s) {
      const int64_t e = int64_t(t) * k + s;
      const int64_t r = src_row ? int64_t(src_row[e]) : e;
      float v[8];
      unpack8(reinterpret_cast<const uint4*>(y + r * d)[c], v);
      const float ws = w[e];
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = fmaf(ws, v[j], acc[j]);
    }
    if (sh) {
      float v[8];
      unpack8(reinterpret_cast<const uint4*>(sh + int64_t(t) * d)[c], v);
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] += v[j];
    }
    reinterpret_cast<uint4*>(out + int64_t(t) * d)[c] = pack8(acc);
  }
}

int grid_for(int64_t work, int threads) {
  const int64_t want = (work + threads - 1) / threads;
  const int64_t cap = int64_t(sm_count() > 0 ? sm_count() : 148) * 16;
  return int(want < 1 ? 1 : (want > cap ? cap : want));
}

bool row_ok(const void* p, int64_t stride_elems, int elem_bytes) {
  return aligned16(p) && ((stride_elems * elem_bytes) % 16 == 0);
}

}  // namespace
}  // namespace biv

using namespace biv;

extern "C" {

biv_status biv_embed(const int32_t* ids, const uint16_t* table, int vocab, int T, int d,
                     uint16_t* h, int64_t h_stride, biv_stream_t stream) {
  BIV_REQUIRE(T >= 0 && d > 0 && d % 8 == 0 && vocab > 0, "embed: bad sizes T=%d d=%d", T, d);
  if (T == 0) return BIV_OK;
  BIV_REQUIRE(ids && aligned16(table) && row_ok(h, h_stride, 2), "embed: bad pointer/stride");
  launch_pdl(embed_kernel, T, 128, 0, as_cuda(stream), ids, table, vocab, d, h, h_stride,
             device_error_word());
  return check_launch("embed");
}

}  // extern "C"

namespace biv {
namespace {
template <bool PARTIAL>
biv_status launch_add_rmsnorm(int cpt, const uint16_t* x, int64_t xs, const biv_partials& xp,
                              uint16_t* r, int64_t rs, const uint16_t* w, uint16_t* y, int64_t ys,
                              int rows, int d, float eps, biv_stream_t stream) {
  cudaStream_t s = as_cuda(stream);
  switch (cpt) {
    case 1: launch_pdl(add_rmsnorm_kernel<1, PARTIAL>, rows, kNormThreads, 0, s, x, xs, xp, r, rs, w, y, ys, d, eps); break;
    case 2: launch_pdl(add_rmsnorm_kernel<2, PARTIAL>, rows, kNormThreads, 0, s, x, xs, xp, r, rs, w, y, ys, d, eps); break;
    case 3: launch_pdl(add_rmsnorm_kernel<3, PARTIAL>, rows, kNormThreads, 0, s, x, xs, xp, r, rs, w, y, ys, d, eps); break;
    default: launch_pdl(add_rmsnorm_kernel<4, PARTIAL>, rows, kNormThreads, 0, s, x, xs, xp, r, rs, w, y, ys, d, eps); break;
  }
  return check_launch("add_rmsnorm");
}

biv_status add_rmsnorm_impl(const uint16_t* x, int64_t xs, const biv_partials& xp, uint16_t* r,
                            int64_t rs, const uint16_t* w, uint16_t* y, int64_t ys, int rows, int d,
                            float eps, biv_stream_t stream) {
  BIV_REQUIRE(rows >= 0 && d > 0 && d % 8 == 0 && d <= 8192, "add_rmsnorm: bad d=%d", d);
  if (rows == 0) return BIV_OK;
  BIV_REQUIRE((xp.chunks > 0 || row_ok(x, xs, 2)) && row_ok(y, ys, 2) && aligned16(w) &&
                  (!r || row_ok(r, rs, 2)),
              "add_rmsnorm: pointers/strides must keep rows 16-byte aligned");
  BIV_REQUIRE(xp.chunks == 0 || (xp.chunks <= kMaxPartialChunks && aligned16(xp.p) && xp.ld % 4 == 0 &&
                                 xp.chunk_stride % 4 == 0),
              "add_rmsnorm: bad partials");
  const int cpt = (d / 8 + kNormThreads - 1) / kNormThreads;
  if (xp.chunks > 0) return launch_add_rmsnorm<true>(cpt, x, xs, xp, r, rs, w, y, ys, rows, d, eps, stream);
  return launch_add_rmsnorm<false>(cpt, x, xs, xp, r, rs, w, y, ys, rows, d, eps, stream);
}
}  // namespace
}  // namespace biv

extern "C" {

biv_status biv_add_rmsnorm(const uint16_t* x, int64_t xs, uint16_t* r, int64_t rs,
                           const uint16_t* w, uint16_t* y, int64_t ys, int rows, int d, float eps,
                           biv_stream_t stream) {
  const biv_partials none = {nullptr, 0, 0, 0};
  return add_rmsnorm_impl(x, xs, none, r, rs, w, y, ys, rows, d, eps, stream);
}

biv_status biv_add_rmsnorm_partials(const biv_partials* x, uint16_t* r, int64_t rs,
                                    const uint16_t* w, uint16_t* y, int64_t ys, int rows, int d,
                                    float eps, biv_stream_t stream) {
  BIV_REQUIRE(x && x->p && x->chunks > 0, "add_rmsnorm_partials: no partials");
  return add_rmsnorm_impl(nullptr, 0, *x, r, rs, w, y, ys, rows, d, eps, stream);
}

biv_status biv_silu_mul(const uint16_t* gu, int64_t gs, uint16_t* y, int64_t ys, int rows, int I,
                        biv_stream_t stream) {
  BIV_REQUIRE(rows >= 0 && I > 0 && I % 8 == 0, "silu_mul: I=%d must be a multiple of 8", I);
  if (rows == 0) return BIV_OK;
  BIV_REQUIRE(row_ok(gu, gs, 2) && row_ok(y, ys, 2), "silu_mul: misaligned rows");
  const int64_t work = int64_t(rows) * (I / 8);
  launch_pdl(silu_mul_kernel, grid_for(work, 256), 256, 0, as_cuda(stream), gu, gs, y, ys, rows,
             I);
  return check_launch("silu_mul");
}

biv_status biv_silu_mul_partials(const biv_partials* gu, uint16_t* y, int64_t ys, int rows, int I,
                                 biv_stream_t stream) {
  BIV_REQUIRE(rows >= 0 && I > 0 && I % 8 == 0, "silu_mul: I=%d must be a multiple of 8", I);
  BIV_REQUIRE(gu && gu->p && gu->chunks > 0 && gu->chunks <= kMaxPartialChunks &&
                  aligned16(gu->p) && gu->ld % 4 == 0 && gu->chunk_stride % 4 == 0 &&
                  gu->ld >= 2 * int64_t(I),
              "silu_mul_partials: bad partials");
  if (rows == 0) return BIV_OK;
  BIV_REQUIRE(row_ok(y, ys, 2), "silu_mul: misaligned rows");
  const int64_t work = int64_t(rows) * (I / 4);
  launch_pdl(silu_mul_partials_kernel, grid_for(work, 256), 256, 0, as_cuda(stream), *gu, y, ys,
             rows, I);
  return check_launch("silu_mul");
}

biv_status biv_rope_table(double theta, int D, int max_pos, float* cos_sin, biv_stream_t stream) {
  BIV_REQUIRE(D > 0 && D % 2 == 0 && max_pos > 0 && cos_sin && theta > 0, "rope_table: bad args");
  const int64_t n = int64_t(max_pos) * (D / 2);
  rope_table_kernel<<<grid_for(n, 256), 256, 0, as_cuda(stream)>>>(theta, D, max_pos, cos_sin);
  return check_launch("rope_table");
}

biv_status biv_qk_norm_rope(uint16_t* qkv, int64_t rs, int T, int Hq, int Hkv, int D,
                            const uint16_t* q_w, const uint16_t* k_w, const float* cos_sin,
                            int max_pos, const int32_t* pos, float eps, biv_stream_t stream) {
  BIV_REQUIRE(D == 64 || D == 80 || D == 128, "qk_norm_rope: D=%d unsupported", D);
  BIV_REQUIRE(T >= 0 && Hq > 0 && Hkv > 0 && max_pos > 0, "qk_norm_rope: bad sizes");
  BIV_REQUIRE((q_w == nullptr) == (k_w == nullptr), "qk_norm_rope: give both gains or neither");
  if (T == 0) return BIV_OK;
  BIV_REQUIRE(qkv && cos_sin && pos, "qk_norm_rope: null pointer");
  const int64_t warps = int64_t(T) * (Hq + Hkv);
  const int threads = 256;
  const int64_t blocks = (warps * 32 + threads - 1) / threads;
  launch_pdl(qk_norm_rope_kernel, unsigned(blocks), threads, 0, as_cuda(stream), qkv, rs, T, Hq,
             Hkv, D, q_w, k_w, cos_sin, max_pos, pos, eps, device_error_word());
  return check_launch("qk_norm_rope");
}

biv_status biv_qkv_finalize(uint16_t* qkv, int64_t rs, const biv_partials* qkv_partials, int T,
                            int Hq, int Hkv, int D, const uint16_t* q_w, const uint16_t* k_w,
                            const float* cos_sin, int max_pos, const int32_t* pos, float eps,
                            const int64_t* slot, int kv_dtype, void* k_cache, void* v_cache,
                            float* k_scale, float* v_scale, biv_stream_t stream) {
  BIV_REQUIRE(D == 64 || D == 80 || D == 128, "qkv_finalize: D=%d unsupported", D);
  BIV_REQUIRE(T >= 0 && Hq > 0 && Hkv > 0 && max_pos > 0, "qkv_finalize: bad sizes");
  BIV_REQUIRE((q_w == nullptr) == (k_w == nullptr), "qkv_finalize: give both gains or neither");
  BIV_REQUIRE(kv_dtype == BIV_BF16 || kv_dtype == BIV_E4M3, "qkv_finalize: kv dtype");
  if (T == 0) return BIV_OK;
  BIV_REQUIRE(qkv && cos_sin && pos && slot && k_cache && v_cache, "qkv_finalize: null pointer");
  BIV_REQUIRE(kv_dtype == BIV_BF16 || (k_scale && v_scale), "qkv_finalize: FP8 needs scales");
  biv_partials xp = {nullptr, 0, 0, 0};
  if (qkv_partials && qkv_partials->chunks > 0) {
    xp = *qkv_partials;
    BIV_REQUIRE(xp.p && xp.chunks <= kMaxPartialChunks, "qkv_finalize: bad partials");
  }
  const int64_t warps = int64_t(T) * (Hq + 2 * Hkv);
  const int threads = 256;
  const int64_t blocks = (warps * 32 + threads - 1) / threads;
  launch_pdl(xp.chunks > 0 ? qkv_finalize_kernel<true> : qkv_finalize_kernel<false>,
             unsigned(blocks), threads, 0, as_cuda(stream), qkv, rs, xp, T, Hq, Hkv, D, q_w, k_w,
             cos_sin, max_pos, pos, eps, slot, kv_dtype == BIV_E4M3 ? 1 : 0, k_cache, v_cache,
             k_scale, v_scale, device_error_word());
  return check_launch("qkv_finalize");
}

biv_status biv_kv_store_bf16(const uint16_t* k, const uint16_t* v, int64_t rs, const int64_t* slot,
                             int T, int Hkv, int D, uint16_t* kc, uint16_t* vc,
                             biv_stream_t stream) {
  BIV_REQUIRE(T >= 0 && Hkv > 0 && D % 8 == 0, "kv_store_bf16: bad sizes");
  if (T == 0) return BIV_OK;
  BIV_REQUIRE(row_ok(k, rs, 2) && row_ok(v, rs, 2) && aligned16(kc) && aligned16(vc) && slot,
              "kv_store_bf16: misaligned");
  const int64_t work = int64_t(T) * Hkv * (D / 8) * 2;
  launch_pdl(kv_store_bf16_kernel, grid_for(work, 256), 256, 0, as_cuda(stream), k, v, rs, slot, T,
             Hkv, D, kc, vc);
  return check_launch("kv_store_bf16");
}

biv_status biv_kv_fp8_quant(const uint16_t* k, const uint16_t* v, int64_t rs, const int64_t* slot,
                            int T, int Hkv, int D, uint8_t* kc, uint8_t* vc, float* ks, float* vs,
                            biv_stream_t stream) {
  BIV_REQUIRE(T >= 0 && Hkv > 0 && D > 0 && D <= 128, "kv_fp8_quant: bad sizes");
  if (T == 0) return BIV_OK;
  BIV_REQUIRE(k && v && slot && kc && vc && ks && vs, "kv_fp8_quant: null pointer");
  const int64_t warps = int64_t(T) * Hkv * 2;
  const int64_t blocks = (warps * 32 + 255) / 256;
  launch_pdl(kv_fp8_quant_kernel, unsigned(blocks), 256, 0, as_cuda(stream), k, v, rs, slot, T, Hkv,
             D, kc, vc, ks, vs);
  return check_launch("kv_fp8_quant");
}

biv_status biv_kv_fp8_gather(const uint8_t* codes, const float* scales, const int32_t* bt,
                             int max_pages, const int32_t* ctx, const int64_t* row0, int nseq,
                             int Hkv, int D, int page, uint16_t* out, biv_stream_t stream) {
  BIV_REQUIRE(nseq >= 0 && Hkv > 0 && D > 0 && page > 0 && max_pages > 0,
              "kv_fp8_gather: bad sizes");
  if (nseq == 0) return BIV_OK;
  BIV_REQUIRE(nseq <= 65535, "kv_fp8_gather: nseq above 65535");
  BIV_REQUIRE(codes && scales && bt && ctx && row0 && out, "kv_fp8_gather: null pointer");
  dim3 grid(64, nseq);
  kv_fp8_gather_kernel<<<grid, 256, 0, as_cuda(stream)>>>(codes, scales, bt, max_pages, ctx, row0,
                                                          Hkv, D, page, out);
  return check_launch("kv_fp8_gather");
}

biv_status biv_act_quant_fp8(const uint16_t* x, int64_t xs, int rows, int K, uint8_t* codes,
                             float* scales, biv_stream_t stream) {
  BIV_REQUIRE(rows >= 0 && K > 0 && K % 16 == 0, "act_quant_fp8: K=%d must be a multiple of 16", K);
  if (rows == 0) return BIV_OK;
  BIV_REQUIRE(x && codes && scales, "act_quant_fp8: null pointer");
  BIV_REQUIRE(row_ok(x, xs, 2), "act_quant_fp8: x rows must be 16-byte aligned");
  const int64_t halves = int64_t(rows) * ((K + 127) / 128);
  act_quant_kernel<<<unsigned((halves * 16 + 255) / 256), 256, 0, as_cuda(stream)>>>(
      x, xs, rows, K, codes, scales);
  return check_launch("act_quant_fp8");
}

biv_status biv_silu_mul_quant_fp8(const uint16_t* gu, int64_t gs, int rows, int I, uint8_t* codes,
                                  float* scales, biv_stream_t stream) {
  BIV_REQUIRE(rows >= 0 && I > 0 && I % 16 == 0, "silu_mul_quant_fp8: I=%d must be a multiple of 16",
              I);
  if (rows == 0) return BIV_OK;
  BIV_REQUIRE(gu && codes && scales && gs >= 2 * int64_t(I) && row_ok(gu, gs, 2),
              "silu_mul_quant_fp8: bad arguments (rows must be 16-byte aligned)");
  const int64_t halves = int64_t(rows) * ((I + 127) / 128);
  launch_pdl(silu_mul_quant_kernel, unsigned((halves * 16 + 255) / 256), 256, 0, as_cuda(stream),
             gu, gs, rows, I, codes, scales);
  return check_launch("silu_mul_quant_fp8");
}

biv_status biv_logprob(const float* z, int64_t ld, const int32_t* target, int T, int V, float* lp,
                       biv_stream_t stream) {
  BIV_REQUIRE(T >= 0 && V > 0 && V % 4 == 0, "logprob: V=%d must be a multiple of 4", V);
  if (T == 0) return BIV_OK;
  BIV_REQUIRE(row_ok(z, ld, 4) && target && lp, "logprob: logits rows must be 16-byte aligned");
  launch_pdl(logprob_kernel, T, kLogprobThreads, 0, as_cuda(stream), z, ld, target, V, lp,
             device_error_word());
  return check_launch("logprob");
}

biv_status biv_router_topk(const float* logits, int64_t ld, int rows, int E, int k, int32_t* idx,
                           float* w, biv_stream_t stream) {
  BIV_REQUIRE(rows >= 0 && E > 0 && E <= 1024 && k > 0 && k <= 32 && k <= E,
              "router_topk: bad sizes E=%d k=%d", E, k);
  if (rows == 0) return BIV_OK;
  BIV_REQUIRE(logits && idx && w, "router_topk: null pointer");
  const int blocks = (rows + kRouterWarps - 1) / kRouterWarps;
  router_kernel<<<blocks, 32 * kRouterWarps, kRouterWarps * E * sizeof(float), as_cuda(stream)>>>(
      logits, ld, rows, E, k, idx, w);
  return check_launch("router_topk");
}

biv_status biv_moe_dispatch(const int32_t* idx, int T, int k, int E, int32_t* offsets,
                            int32_t* perm, int32_t* src_row, biv_stream_t stream) {
  BIV_REQUIRE(T >= 0 && k > 0 && E > 0 && E <= 4096 && int64_t(T) * k <= (1 << 20),
              "moe_dispatch: bad sizes");
  BIV_REQUIRE(idx && offsets && perm && src_row, "moe_dispatch: null pointer");
  moe_dispatch_kernel<<<E, 1024, 0, as_cuda(stream)>>>(idx, T * k, E, offsets, perm, src_row);
  return check_launch("moe_dispatch");
}

biv_status biv_gather_rows(const void* src, int64_t ss, const int32_t* perm, int k_div, int n,
                           int row_bytes, void* dst, int64_t ds, biv_stream_t stream) {
  BIV_REQUIRE(n >= 0 && k_div > 0 && row_bytes > 0 && row_bytes % 16 == 0,
              "gather_rows: bad sizes");
  if (n == 0) return BIV_OK;
  BIV_REQUIRE(aligned16(src) && aligned16(dst) && ss % 16 == 0 && ds % 16 == 0 && perm,
              "gather_rows: misaligned");
  const int64_t work = int64_t(n) * (row_bytes / 16);
  launch_pdl(gather_rows_kernel, grid_for(work, 256), 256, 0, as_cuda(stream),
             static_cast<const uint8_t*>(src), ss, perm, k_div, n, row_bytes,
             static_cast<uint8_t*>(dst), ds);
  return check_launch("gather_rows");
}

biv_status biv_moe_combine(const uint16_t* y, const int32_t* src_row, const float* w,
                           const uint16_t* sh, uint16_t* out, int T, int k, int d,
                           biv_stream_t stream) {
  BIV_REQUIRE(T >= 0 && k > 0 && d > 0 && d % 8 == 0, "moe_combine: bad sizes");
  if (T == 0) return BIV_OK;
  BIV_REQUIRE(aligned16(y) && aligned16(out) && w && (!sh || aligned16(sh)),
              "moe_combine: misaligned");
  const int64_t work = int64_t(T) * (d / 8);
  moe_combine_kernel<<<grid_for(work, 256), 256, 0, as_cuda(stream)>>>(y, src_row, w, sh, out, T,
                                                                       k, d);
  return check_launch("moe_combine");
}

}  // extern "C"
