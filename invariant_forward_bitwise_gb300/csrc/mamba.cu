// The Mamba-2 mixer's element-wise and row-wise steps around the SSD scan,
// and the NVFP4 weight decoder of the hybrid stack ("Finish RL Training
// Faster", section "两组结果，要连同分母一起读": a Mamba-2 hybrid with NVFP4
// weights; section "一致性有多个层面": decode replays the prefill order).
//
//  * causal conv1d (width 4, depthwise) + SiLU over the xBC columns of the
//    in-projection, and dt = softplus(dt_raw + dt_bias) over its dt columns.
//    An output row's arithmetic is one fixed FP32 sequence, acc = bias, then
//    acc = acc + w[j] * x[t-3+j] for j = 0..3 (product and sum each rounded:
//    no contraction into fma), whatever rows share the call: its earlier
//    inputs come from the call's own rows or, before the call's first row,
//    from the sequence's conv state, which holds the three inputs that
//    preceded it.  Prefill, chunked prefill and decode therefore give the
//    same bits.  A second kernel then replaces the state with the last three
//    inputs.
//  * gated RMSNorm: g = y * silu(z) in FP32, out = bf16((g * inv) * w) with
//    the same per-row reduction tree as the other norms (256 threads, per
//    thread in chunk order, warp xor tree, warps in order).
//  * NVFP4 decode: packed e2m1 codes times their block's e4m3 scale, exact in
//    bf16 (the same conversion the NVFP4 GEMM runs in shared memory).
#include "common.cuh"

namespace biv {
namespace {

constexpr int kConvW = 4;
constexpr int kGNThreads = 256;

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
__device__ __forceinline__ float silu_f(float x) { return x / (1.0f + expf(-x)); }
__device__ __forceinline__ float softplus_f(float x) {
  return x > 20.0f ? x : log1pf(expf(x));
}

struct ConvArgs {
  const uint16_t* u; int64_t us;
  int col_x, col_dt, ch, heads;
  const uint16_t* w; const uint16_t* b; const float* dt_bias;
  uint16_t* out; int64_t os;
  float* dt; int64_t dts;
  int T;
  const int32_t* row_seq; const int32_t* row_pos;
  int nseq;
  const int32_t* row0; const int32_t* n; const int32_t* pos0;
  uint16_t* state;                  // [nseq, 3, ch]
  int* err;
};

// the input x[q, c..c+7] of sequence i: from the call's rows when q is at or
// after the sequence's first row in the call, from the conv state before it,
// zero before position 0
__device__ __forceinline__ void conv_input(const ConvArgs& a, int i, int q, int c, float (&f)[8]) {
  const int p0 = a.pos0[i];
  if (q < 0) {
#pragma unroll
    for (int j = 0; j < 8; ++j) f[j] = 0.f;
  } else if (q >= p0) {
    const int64_t r = int64_t(a.row0[i]) + (q - p0);
    unpack8(*reinterpret_cast<const uint4*>(a.u + r * a.us + a.col_x + c), f);
  } else {
    const int s = q - p0 + (kConvW - 1);           // 0 .. 2
    unpack8(*reinterpret_cast<const uint4*>(a.state + (int64_t(i) * (kConvW - 1) + s) * a.ch + c), f);
  }
}

// one thread per (row, 8 channels); the last heads/8 chunks of a row are dt
__global__ void conv_silu_kernel(const __grid_constant__ ConvArgs a) {
  pdl_wait();
  pdl_trigger();
  const int cx = a.ch / 8, cd = a.heads / 8, cpr = cx + cd;
  const int64_t total = int64_t(a.T) * cpr;
  for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < total;
       e += int64_t(gridDim.x) * blockDim.x) {
    const int r = int(e / cpr), k = int(e % cpr);
    if (k >= cx) {                                 // dt = softplus(dt_raw + dt_bias)
      const int h = (k - cx) * 8;
      float raw[8];
      unpack8(*reinterpret_cast<const uint4*>(a.u + int64_t(r) * a.us + a.col_dt + h), raw);
      float* dst = a.dt + int64_t(r) * a.dts + h;
#pragma unroll
      for (int j = 0; j < 8; ++j) dst[j] = softplus_f(__fadd_rn(raw[j], a.dt_bias[h + j]));
      continue;
    }
    const int c = k * 8;
    const int i = a.row_seq[r], p = a.row_pos[r];
    if (i < 0 || i >= a.nseq || p < a.pos0[i] || p - a.pos0[i] >= a.n[i]) {
      if (c == 0) raise_error(a.err, kErrBadIndex);
      *reinterpret_cast<uint4*>(a.out + int64_t(r) * a.os + c) = make_uint4(0, 0, 0, 0);
      continue;
    }
    float acc[8], wv[kConvW][8];
    {
      float bv[8];
      unpack8(*reinterpret_cast<const uint4*>(a.b + c), bv);
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = bv[j];
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {                  // weights [ch, 4]: 4 per channel
      const uint2 w2 = *reinterpret_cast<const uint2*>(a.w + int64_t(c + j) * kConvW);
      wv[0][j] = __uint_as_float(w2.x << 16);
      wv[1][j] = __uint_as_float(w2.x & 0xFFFF0000u);
      wv[2][j] = __uint_as_float(w2.y << 16);
      wv[3][j] = __uint_as_float(w2.y & 0xFFFF0000u);
    }
#pragma unroll
    for (int t = 0; t < kConvW; ++t) {
      float x[8];
      conv_input(a, i, p - (kConvW - 1) + t, c, x);
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = __fadd_rn(acc[j], __fmul_rn(wv[t][j], x[j]));
    }
    float o[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) o[j] = silu_f(acc[j]);
    *reinterpret_cast<uint4*>(a.out + int64_t(r) * a.os + c) = pack8(o);
  }
}

// after the conv: state[i] = the inputs at positions pos0+n-3 .. pos0+n-1
// (one thread per (sequence, 8 channels) reads all three, then writes them)
__global__ void conv_state_kernel(const __grid_constant__ ConvArgs a) {
  pdl_wait();
  pdl_trigger();
  const int cx = a.ch / 8;
  const int64_t total = int64_t(a.nseq) * cx;
  for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < total;
       e += int64_t(gridDim.x) * blockDim.x) {
    const int i = int(e / cx), c = int(e % cx) * 8;
    const int n = a.n[i];
    if (n <= 0) continue;
    float v[kConvW - 1][8];
#pragma unroll
    for (int s = 0; s < kConvW - 1; ++s) conv_input(a, i, a.pos0[i] + n - (kConvW - 1) + s, c, v[s]);
#pragma unroll
    for (int s = 0; s < kConvW - 1; ++s)
      *reinterpret_cast<uint4*>(a.state + (int64_t(i) * (kConvW - 1) + s) * a.ch + c) = pack8(v[s]);
  }
}

// ------------------------------------------------------- gated RMSNorm ----
template <int CPT>
__global__ void __launch_bounds__(kGNThreads) gated_rmsnorm_kernel(
    const uint16_t* __restrict__ y, int64_t ys, const uint16_t* __restrict__ z, int64_t zs,
    const uint16_t* __restrict__ w, uint16_t* __restrict__ out, int64_t os, int d, float eps) {
  pdl_wait();
  pdl_trigger();
  __shared__ float warp_ss[kGNThreads / 32];
  const int row = blockIdx.x;
  const int chunks = d / 8;
  const uint4* yr = reinterpret_cast<const uint4*>(y + int64_t(row) * ys);
  const uint4* zr = reinterpret_cast<const uint4*>(z + int64_t(row) * zs);
  float g[CPT][8];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < CPT; ++i) {
    const int c = threadIdx.x + i * kGNThreads;
    if (c < chunks) {
      float yv[8], zv[8];
      unpack8(yr[c], yv);
      unpack8(zr[c], zv);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        g[i][j] = __fmul_rn(yv[j], silu_f(zv[j]));
        ss = fmaf(g[i][j], g[i][j], ss);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) warp_ss[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < kGNThreads / 32; ++i) tot += warp_ss[i];
  const float inv = 1.0f / sqrtf(tot / float(d) + eps);
  const uint4* wr = reinterpret_cast<const uint4*>(w);
  uint4* orow = reinterpret_cast<uint4*>(out + int64_t(row) * os);
#pragma unroll
  for (int i = 0; i < CPT; ++i) {
    const int c = threadIdx.x + i * kGNThreads;
    if (c < chunks) {
      float wv[8], o[8];
      unpack8(__ldg(wr + c), wv);
#pragma unroll
      for (int j = 0; j < 8; ++j) o[j] = (g[i][j] * inv) * wv[j];
      orow[c] = pack8(o);
    }
  }
}

// ------------------------------------------------------------ NVFP4 ----
// one thread per 16-element block: 8 bytes of packed e2m1 codes (element 2i in
// the low nibble of byte i) and the block's e4m3 scale -> 16 bf16 values.
// e2m1 x e4m3 has at most 6 significant bits: exact in f16 and in bf16.
__global__ void nvfp4_dequant_kernel(const uint8_t* __restrict__ codes,
                                     const uint8_t* __restrict__ scales, int N, int K,
                                     uint16_t* __restrict__ out) {
  const int kb = K / 16;
  const int64_t total = int64_t(N) * kb;
  for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < total;
       e += int64_t(gridDim.x) * blockDim.x) {
    const int64_t n = e / kb;
    const int b = int(e % kb);
    const __half s = __ushort_as_half(
        __nv_cvt_fp8_to_halfraw(__nv_fp8_storage_t(scales[n * kb + b]), __NV_E4M3).x);
    const __half2 s2 = __halves2half2(s, s);
    const uint2 cv = *reinterpret_cast<const uint2*>(codes + n * (K / 2) + b * 8);
    const uint32_t w[2] = {cv.x, cv.y};
    uint32_t o[8];
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const __half2_raw hr =
            __nv_cvt_fp4x2_to_halfraw2(__nv_fp4x2_storage_t((w[q] >> (8 * j)) & 0xFFu), __NV_E2M1);
        const float2 f = __half22float2(__hmul2(__half2(hr), s2));
        o[4 * q + j] = pack_bf2(f.x, f.y);
      }
    uint4* dst = reinterpret_cast<uint4*>(out + n * K + b * 16);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

int grid_of(int64_t work, int threads) {
  const int64_t want = (work + threads - 1) / threads;
  const int64_t cap = int64_t(sm_count() > 0 ? sm_count() : 148) * 16;
  return int(want < 1 ? 1 : (want > cap ? cap : want));
}
bool rows16(const void* p, int64_t stride, int elem) {
  return aligned16(p) && (stride * elem) % 16 == 0;
}

}  // namespace
}  // namespace biv

using namespace biv;

extern "C" {

biv_status biv_causal_conv1d(const biv_conv_desc* d, biv_stream_t stream) {
  BIV_REQUIRE(d, "causal_conv1d: null descriptor");
  BIV_REQUIRE(d->T >= 0 && d->nseq >= 0 && d->channels > 0 && d->channels % 8 == 0 &&
                  d->heads >= 0 && d->heads % 8 == 0 && d->width == kConvW,
              "causal_conv1d: channels and heads must be multiples of 8, width 4");
  if (d->T == 0 && d->nseq == 0) return BIV_OK;
  BIV_REQUIRE(d->u && d->conv_w && d->conv_b && d->out && d->row_seq && d->row_pos && d->row0 &&
                  d->n && d->pos0 && d->state && (d->heads == 0 || (d->dt_out && d->dt_bias)),
              "causal_conv1d: null pointer");
  BIV_REQUIRE(rows16(d->u, d->u_stride, 2) && d->col_x % 8 == 0 && d->col_dt % 8 == 0 &&
                  rows16(d->out, d->out_stride, 2) && aligned16(d->conv_b) && aligned16(d->state) &&
                  (reinterpret_cast<uintptr_t>(d->conv_w) & 7u) == 0,
              "causal_conv1d: rows, columns and weights must stay 16-byte aligned");
  ConvArgs a;
  a.u = d->u; a.us = d->u_stride; a.col_x = d->col_x; a.col_dt = d->col_dt;
  a.ch = d->channels; a.heads = d->heads;
  a.w = d->conv_w; a.b = d->conv_b; a.dt_bias = d->dt_bias;
  a.out = d->out; a.os = d->out_stride; a.dt = d->dt_out; a.dts = d->dt_stride;
  a.T = d->T; a.row_seq = d->row_seq; a.row_pos = d->row_pos;
  a.nseq = d->nseq; a.row0 = d->row0; a.n = d->n; a.pos0 = d->pos0;
  a.state = d->state; a.err = device_error_word();
  cudaStream_t s = as_cuda(stream);
  if (d->T > 0) {
    const int64_t work = int64_t(d->T) * (d->channels / 8 + d->heads / 8);
    launch_pdl(conv_silu_kernel, grid_of(work, 256), 256, 0, s, a);
    biv_status st = check_launch("causal_conv1d");
    if (st != BIV_OK) return st;
  }
  if (d->nseq > 0) {
    launch_pdl(conv_state_kernel, grid_of(int64_t(d->nseq) * (d->channels / 8), 256), 256, 0, s, a);
    return check_launch("causal_conv1d_state");
  }
  return BIV_OK;
}

biv_status biv_gated_rmsnorm(const uint16_t* y, int64_t ys, const uint16_t* z, int64_t zs,
                             const uint16_t* w, uint16_t* out, int64_t os, int rows, int d,
                             float eps, biv_stream_t stream) {
  BIV_REQUIRE(rows >= 0 && d > 0 && d % 8 == 0 && d <= 8 * kGNThreads * 4,
              "gated_rmsnorm: d=%d must be a multiple of 8 and at most 8192", d);
  if (rows == 0) return BIV_OK;
  BIV_REQUIRE(rows16(y, ys, 2) && rows16(z, zs, 2) && rows16(out, os, 2) && aligned16(w),
              "gated_rmsnorm: misaligned rows");
  const int cpt = (d / 8 + kGNThreads - 1) / kGNThreads;
  cudaStream_t s = as_cuda(stream);
  switch (cpt) {
    case 1: launch_pdl(gated_rmsnorm_kernel<1>, rows, kGNThreads, 0, s, y, ys, z, zs, w, out, os, d, eps); break;
    case 2: launch_pdl(gated_rmsnorm_kernel<2>, rows, kGNThreads, 0, s, y, ys, z, zs, w, out, os, d, eps); break;
    case 3: launch_pdl(gated_rmsnorm_kernel<3>, rows, kGNThreads, 0, s, y, ys, z, zs, w, out, os, d, eps); break;
    default: launch_pdl(gated_rmsnorm_kernel<4>, rows, kGNThreads, 0, s, y, ys, z, zs, w, out, os, d, eps); break;
  }
  return check_launch("gated_rmsnorm");
}

biv_status biv_nvfp4_dequant(const uint8_t* codes, const uint8_t* scales, int N, int K,
                             uint16_t* out, biv_stream_t stream) {
  BIV_REQUIRE(N >= 0 && K > 0 && K % 16 == 0, "nvfp4_dequant: K=%d must be a multiple of 16", K);
  if (N == 0) return BIV_OK;
  BIV_REQUIRE(codes && scales && out && aligned16(codes) && aligned16(out),
              "nvfp4_dequant: codes and out must be 16-byte aligned");
  nvfp4_dequant_kernel<<<grid_of(int64_t(N) * (K / 16), 256), 256, 0, as_cuda(stream)>>>(
      codes, scales, N, K, out);
  return check_launch("nvfp4_dequant");
}

}  // extern "C"
