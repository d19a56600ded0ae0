/*
 * libbiv -- batch-invariant transformer forward for one GB300 (sm_103a).
 *
 * Every call computes each output row from that row's own inputs (and its own
 * sequence's KV cache or SSM state) with one fixed reduction order, so a
 * token's logprob does not change with batch size, batch mix, prefill vs
 * chunked prefill vs decode, eager vs CUDA-Graph replay, or rollout vs
 * trainer recompute.  The requirement and the rules that achieve it (one
 * computation path, one quantisation rule, one tie-break, one accumulation
 * order per op) come from "Finish RL Training Faster: Bitwise-Consistent,
 * High-Performance, Agent-Driven", sections "零差异需要一个精确的比较对象" and
 * "让训练前向使用推理的数值", and from "No More Train-Inference Mismatch:
 * Bitwise Consistent On-Policy Reinforcement Learning with vLLM and
 * TorchTitan", section "方法细节".
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library
 *    never allocates, frees or synchronises (except biv_poll_error), and only
 *    launches kernels on the given stream.  Weights may be updated in place
 *    between calls (captured graphs keep reading the same addresses).
 *  - bf16 tensors are passed as uint16_t* (raw bfloat16 payloads); FP8 tensors
 *    as uint8_t* (OCP E4M3FN codes).  Row-major; *_stride arguments are in
 *    ELEMENTS between consecutive rows.
 *  - Pointers used with 16-byte vector or TMA access must be 16-byte aligned
 *    and row strides must keep rows 16-byte aligned; the host check returns
 *    BIV_ERR_INVALID otherwise, without launching anything.
 *  - Zero-sized work (rows == 0, T == 0 ...) returns BIV_OK and launches nothing.
 *  - On error the status is returned and biv_last_error() describes it.
 *  - mode BIV_MODE_FAST switches the split-K / split-KV choice to one that
 *    depends on the batch (the non-invariant comparator); results then change
 *    with batch size.  BIV_MODE_INVARIANT never lets the batch enter a
 *    reduction.
 */
#ifndef BIV_H
#define BIV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* biv_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
  BIV_OK = 0,
  BIV_ERR_INVALID = 1,     /* bad argument: nothing was launched */
  BIV_ERR_UNSUPPORTED = 2, /* valid but not implemented shape/dtype combination */
  BIV_ERR_WORKSPACE = 3,   /* workspace pointer NULL or smaller than required */
  BIV_ERR_CUDA = 4,        /* a CUDA runtime/driver call or launch failed */
  BIV_ERR_TIMEOUT = 5      /* a device-side wait gave up (see biv_poll_error) */
} biv_status;

typedef enum { BIV_MODE_INVARIANT = 0, BIV_MODE_FAST = 1 } biv_mode;
typedef enum { BIV_BF16 = 0, BIV_F32 = 1, BIV_E4M3 = 2 } biv_dtype;

/* Chunk partials that a bf16 biv_gemm left in its workspace: the output
 * element (row, col) is RN(((p[0] + p[1]) + p[2]) + ...) with p[c] =
 * p + c*chunk_stride + row*ld + col, rounded once to the GEMM's output type;
 * chunks == 0 means the call wrote C itself. */
typedef struct {
  const float* p;
  int chunks;
  int64_t ld;
  int64_t chunk_stride;
} biv_partials;


/* Library version (major*10000 + minor*100 + patch). */
int biv_version(void);

/* Thread-local description of the last error on this thread; never NULL. */
const char* biv_last_error(void);

/* Number of SMs of the current device (0 if no device). */
int biv_device_sm_count(void);

/* Reads and clears the device error word that bounded device-side waits set
 * when they give up.  Synchronises the given stream.  *code receives the word
 * (0 = no timeout).  Returns BIV_ERR_TIMEOUT when the word was non-zero. */
biv_status biv_poll_error(biv_stream_t stream, int* code);

/* Test hook for the timeout path: launches one CTA that waits on an mbarrier
 * nothing will ever arrive on, for at most `limit_ns` nanoseconds, then sets
 * the device error word and returns.  Never hangs, never traps. */
biv_status biv_selftest_timeout(uint64_t limit_ns, biv_stream_t stream);

/* ---------------------------------------------------------------- embed --
 * h[t, :] = table[ids[t], :]   ids int32 [T] (0 <= id < vocab, checked on the
 * device: an out-of-range id writes a zero row and sets the error word);
 * table bf16 [vocab, d]; h bf16 [T, d] with row stride h_stride. */
biv_status biv_embed(const int32_t* ids, const uint16_t* table, int vocab, int T, int d,
                     uint16_t* h, int64_t h_stride, biv_stream_t stream);

/* ------------------------------------------------------------ RMSNorm ----
 * Fused residual add + RMSNorm ("No More Train-Inference Mismatch", section
 * "方法细节": fused RMSNorm with residual).  With residual != NULL:
 *   r' = bf16(x + r) (written back to residual), y = bf16(r' * inv * w);
 * with residual == NULL: y = bf16(x * inv * w); inv = 1/sqrt(mean(v^2) + eps)
 * where v is r' (or x), summed in FP32 in a fixed tree that depends on d
 * only.  x, residual, y bf16 [rows, d] with their own row strides; w bf16 [d].
 * d must be a multiple of 8 and <= 8192; y may alias x. */
biv_status biv_add_rmsnorm(const uint16_t* x, int64_t x_stride, uint16_t* residual,
                           int64_t r_stride, const uint16_t* w, uint16_t* y, int64_t y_stride,
                           int rows, int d, float eps, biv_stream_t stream);

/* The same, with x given as the chunk partials of the GEMM that produced it
 * (biv_gemm with defer_fold): x = the GEMM's rounded output, formed here
 * instead of by the GEMM's fold kernel, so the result is the same bit for
 * bit and one launch and one round trip of x are saved.  The partials stay
 * the caller's (the GEMM workspace) and are only read.  BIV_ERR_INVALID on
 * x NULL or chunks outside 1..8, a partial base not 16-byte aligned, or
 * ld / chunk_stride not multiples of 4. */
biv_status biv_add_rmsnorm_partials(const biv_partials* x, uint16_t* residual, int64_t r_stride,
                                    const uint16_t* w, uint16_t* y, int64_t y_stride, int rows,
                                    int d, float eps, biv_stream_t stream);

/* ------------------------------------------------------------ SiLU-mul ----
 * y = bf16(silu(g) * u), silu(g) = g / (1 + exp(-g)) in FP32, for
 * gate_up = [g | u] bf16 [rows, 2I] ("No More Train-Inference Mismatch",
 * section "方法细节": fused SiLU MLP).  y bf16 [rows, I].  I % 8 == 0. */
biv_status biv_silu_mul(const uint16_t* gate_up, int64_t gu_stride, uint16_t* y,
                        int64_t y_stride, int rows, int I, biv_stream_t stream);

/* The same, with gate_up given as the chunk partials of the GEMM that
 * produced it (biv_gemm with defer_fold; partial columns [0, I) are g and
 * [I, 2I) are u): folded here to the GEMM's bf16 output, so y is the same bit
 * for bit.  BIV_ERR_INVALID on chunks outside 1..8, a partial base not
 * 16-byte aligned, or ld / chunk_stride not multiples of 4 or ld < 2I. */
biv_status biv_silu_mul_partials(const biv_partials* gate_up, uint16_t* y, int64_t y_stride,
                                 int rows, int I, biv_stream_t stream);

/* --------------------------------------------------------- RoPE table ----
 * cos_sin float32 [2, max_pos, D/2]: cos then sin of pos * theta^(-2i/D),
 * computed in double precision on the device and rounded to FP32. */
biv_status biv_rope_table(double theta, int D, int max_pos, float* cos_sin,
                          biv_stream_t stream);

/* ---------------------------------------------------- QK-norm + RoPE ----
 * In place on the q and k heads of a packed qkv buffer [T, (Hq+2Hkv)*D]:
 * q at columns [0, Hq*D), k at [Hq*D, (Hq+Hkv)*D).  For each (token, head):
 * optional per-head RMSNorm with gain q_w / k_w bf16 [D] (NULL = skip, the
 * norm output rounded to bf16), then rotate-half RoPE with pairs
 * (i, i+D/2) at position pos[t] (int32 [T], 0 <= pos < max_pos), FP32
 * arithmetic, bf16 result.  D in {64, 80, 128}. */
biv_status biv_qk_norm_rope(uint16_t* qkv, int64_t row_stride, int T, int Hq, int Hkv, int D,
                            const uint16_t* q_w, const uint16_t* k_w, const float* cos_sin,
                            int max_pos, const int32_t* pos, float eps, biv_stream_t stream);

/* ------------------------------------------------------- KV cache store --
 * Paged KV cache, page size `page` tokens: slot s = page_id*page + offset.
 * k, v rows: bf16 [T, Hkv, D] at k + t*row_stride, v + t*row_stride.
 * slot int64 [T] (slot < 0 = skip the row).
 *
 * biv_kv_store_bf16: k_cache/v_cache bf16 [pages, page, Hkv, D].
 * biv_kv_fp8_quant ("Finish RL Training Faster", section
 *   "让训练前向使用推理的数值": the cache stays FP8 and every path makes the same
 *   round trip): per (token, kv head), separately for K and V,
 *   s = amax/448 (IEEE division; 1 when amax = 0),
 *   code = e4m3_rne_satfinite(x / s); codes uint8 [pages, page, Hkv, D],
 *   scales float32 [pages, page, Hkv]. */
biv_status biv_kv_store_bf16(const uint16_t* k, const uint16_t* v, int64_t row_stride,
                             const int64_t* slot, int T, int Hkv, int D, uint16_t* k_cache,
                             uint16_t* v_cache, biv_stream_t stream);
biv_status biv_kv_fp8_quant(const uint16_t* k, const uint16_t* v, int64_t row_stride,
                            const int64_t* slot, int T, int Hkv, int D, uint8_t* k_codes,
                            uint8_t* v_codes, float* k_scales, float* v_scales,
                            biv_stream_t stream);

/* QKV finalize: biv_qk_norm_rope followed by biv_kv_store_bf16 (kv_dtype
 * BIV_BF16) or biv_kv_fp8_quant (BIV_E4M3) of the k and v heads, in one
 * pass with the same per-element operations, so the same bits.  When
 * qkv_partials is non-NULL with chunks > 0, the packed qkv [T, (Hq+2Hkv)*D]
 * is first formed from the QKV GEMM's chunk partials (biv_gemm with
 * defer_fold) and written to qkv; otherwise qkv holds it already.  After the
 * call qkv holds roped q and k and the plain v; k/v of rows with slot >= 0
 * are in the cache (bf16 [slots, Hkv, D], or e4m3 codes with per-(token,
 * head) scales).  Sizes and the error behaviour are those of the separate
 * ops (D in {64, 80, 128}; an out-of-range position is reported through
 * biv_poll_error and read as 0); BIV_ERR_INVALID also on partials with
 * more than 8 chunks. */
biv_status biv_qkv_finalize(uint16_t* qkv, int64_t row_stride, const biv_partials* qkv_partials,
                            int T, int Hq, int Hkv, int D, const uint16_t* q_w, const uint16_t* k_w,
                            const float* cos_sin, int max_pos, const int32_t* pos, float eps,
                            const int64_t* slot, int kv_dtype, void* k_cache, void* v_cache,
                            float* k_scale, float* v_scale, biv_stream_t stream);

/* Gather + dequantise: for each sequence i, tokens [0, ctx_len[i]) of its
 * pages (block_table int32 [nseq, max_pages]) are written as
 * bf16(float(code) * s) to out bf16 [sum ctx, Hkv, D] starting at row
 * out_row0[i] (int64 [nseq]).  Same formula as the attention loader. */
biv_status biv_kv_fp8_gather(const uint8_t* codes, const float* scales,
                             const int32_t* block_table, int max_pages, const int32_t* ctx_len,
                             const int64_t* out_row0, int nseq, int Hkv, int D, int page,
                             uint16_t* out, biv_stream_t stream);

/* ----------------------------------------------------------- attention --
 * One paged GQA attention kernel for prefill, chunked prefill and decode rows
 * ("Finish RL Training Faster", section "让训练前向使用推理的数值": every path
 * gathers, dequantises and enters the same attention operator).
 * Row t (a token of sequence row_seq[t] at absolute position row_pos[t])
 * attends to keys at positions <= row_pos[t] of its sequence, read from the
 * paged cache through block_table.  Keys are visited in 64-token tiles aligned
 * to absolute positions, grouped into splits of kv_split tokens (a model
 * constant); each split keeps an online softmax (FP32), P enters P.V as
 * three bf16 parts hi + mid + lo that add up to the FP32 p exactly, and the
 * splits are merged in ascending order in FP32.  With topk_idx != NULL (sparse attention) the
 * keys of row t are the positions topk_idx[t, 0..topk) (ascending, -1 =
 * none) and splits run over that list.
 * qblocks int32 [nqblocks, 2] = (first row, row count): rows of a block must
 * belong to one sequence (sparse: one row per block).  The grouping into
 * blocks does not change any result bit.  Output bf16 [T, Hq, D]. */
typedef struct {
  const uint16_t* q;        /* [T, Hq, D] rows at q + t*q_stride */
  int64_t q_stride;
  uint16_t* out;            /* [T, Hq, D] rows at out + t*out_stride */
  int64_t out_stride;
  int T, Hq, Hkv, D;        /* D in {64, 80, 128}; Hq % Hkv == 0 */
  const int32_t* row_seq;   /* [T] */
  const int32_t* row_pos;   /* [T] */
  const int32_t* qblocks;   /* [nqblocks, 2] */
  int nqblocks;
  int max_rows_per_block;   /* host bound on the row count of any block */
  int kv_dtype;             /* BIV_BF16 or BIV_E4M3 */
  const void* k_cache;      /* [pages, page, Hkv, D] bf16 or e4m3 */
  const void* v_cache;
  const float* k_scale;     /* [pages, page, Hkv] (E4M3 only) */
  const float* v_scale;
  const int32_t* block_table; /* [nseq, max_pages]: page indices, 0 <= page < 2^31 / 64
                                 (the thread loader raises the device error word on a
                                 negative or larger entry, reads zeros for that page's
                                 keys and leaves the outputs that see them undefined) */
  int max_pages;
  int page;                 /* must be 64 */
  int kv_split;             /* tokens per split, multiple of 64 (INVARIANT: model constant) */
  int max_ctx;              /* host bound: max over rows of row_pos+1 (dense) */
  const int32_t* topk_idx;  /* optional [T, topk] */
  int64_t topk_stride;
  int topk;
  float scale;              /* softmax scale, usually 1/sqrt(D) */
  int mode;                 /* biv_mode; FAST picks kv_split from the batch */
  int num_pages;            /* pages the cache arrays hold (bf16 caches: lets the
                               kernel fetch whole pages by TMA); 0 = unknown */
} biv_attn_desc;

biv_status biv_attention_workspace(const biv_attn_desc* desc, size_t* bytes);
biv_status biv_attention(const biv_attn_desc* desc, void* workspace, size_t workspace_bytes,
                         biv_stream_t stream);

/* Allocation-free variant of biv_attention (the paper has no counterpart: it
 * exists for callers that cannot call cudaMalloc, e.g. code running inside
 * another runtime's memory budget or a hook that must not allocate).  Same
 * arguments and results as biv_attention, but the split partials go to a
 * fixed 64 MiB device array inside the library instead of a caller
 * workspace.  Every GPU that loads the library holds that array until the
 * process exits.  The first call in a CUDA context looks the array's address
 * up (with that context's device current) and caches it for that context;
 * make that first call before any stream capture, and again after a device
 * reset (a new context gets a fresh lookup on its first call).  A call whose scratch need (biv_attention_workspace)
 * exceeds 64 MiB returns BIV_ERR_WORKSPACE and launches nothing.  All calls
 * share the one array: calls whose work can overlap on the GPU (different
 * streams, no ordering between them) race and must not be issued.  Nothing
 * in the array needs to start at zero. */
biv_status biv_attention_noalloc(const biv_attn_desc* desc, biv_stream_t stream);

/* ---------------------------------------------------------------- GEMM --
 * C[M, N] = A[M, K] . B[N, K]^T on the tcgen05 tensor cores, FP32
 * accumulation in TMEM ("Finish RL Training Faster", section
 * "让训练前向使用推理的数值": one batch-invariant GEMM schedule with a fixed K
 * split).  A and B are K-major (row-major with K contiguous).  INVARIANT
 * mode, whatever M is:
 *  - bf16 x bf16 -> bf16 or f32 (c_dtype): with KB = ceil(K/64), K is cut
 *    into chunks of max(8, ceil(KB/8)) blocks of 64 (at most 8 chunks, the
 *    last may be shorter); each chunk P_c is accumulated in FP32 from zero in
 *    ascending K steps of 16; the output is the left fold r = P_0,
 *    r = r + P_1, ... in FP32, rounded once to c_dtype.
 *  - e4m3 x e4m3 -> bf16 with block scales: per 128-wide K block kb,
 *    acc += (sa[m,kb]*sb[g][n/128,kb]) * (FP8 products summed over the
 *    block), promoted to FP32 every block, blocks in ascending order.
 * Grouped (MoE) when groups > 1: rows [off[g], off[g+1]) of A use weight
 * group g (B rows g*N .. g*N+N-1, sb + g*ceil(N/128)*ceil(K/128)).
 * K % 8 == 0 (bf16) / K % 16 == 0 (e4m3); lda, ldb keep rows 16-byte
 * aligned; ldc keeps rows 16-byte aligned for vector stores.
 * FAST mode (bf16): no K chunks when M fills the GPU, a K split sized to the
 * GPU when it does not (results depend on M; the comparator).
 * Workspace (bf16, when biv_gemm_workspace reports > 0: few output tiles,
 * where the chunks of one tile run on different SMs and a second kernel
 * folds them): device memory, 16-byte aligned, owned by the caller, no
 * initial value needed.  Calls that can overlap on the GPU need separate
 * workspaces.
 * Returns BIV_ERR_WORKSPACE when the workspace is missing or too small. */
typedef struct {
  int M, N, K;
  int a_dtype, b_dtype, c_dtype;
  const void* A; int64_t lda;
  const void* B; int64_t ldb;
  void* C; int64_t ldc;
  const float* sa; int64_t ld_sa;   /* FP8: [M, ld_sa >= ceil(K/128)] */
  const float* sb;                  /* FP8: [groups, ceil(N/128), ceil(K/128)] */
  const int32_t* group_offsets;     /* optional device [groups+1] */
  int groups;                       /* 0/1 = plain */
  int mode;                         /* biv_mode */
  int defer_fold;                   /* 1: when the call leaves chunk partials in the
                                       workspace (biv_gemm_partials says so), skip the
                                       fold: a consumer op reads them; C is not written */
} biv_gemm_desc;

/* Fills *out with the partials layout of a call (chunks = 0 when the plan
 * folds inside the GEMM).  Pure host computation, no launch. */
biv_status biv_gemm_partials(const biv_gemm_desc* desc, const void* workspace, biv_partials* out);

biv_status biv_gemm_workspace(const biv_gemm_desc* desc, size_t* bytes);
biv_status biv_gemm(const biv_gemm_desc* desc, void* workspace, size_t workspace_bytes,
                    biv_stream_t stream);

/* Per-token activation quantisation for the FP8 GEMM: groups of 128 along K,
 * s = amax/448 (1 when amax = 0), code = e4m3_rne_satfinite(x/s).
 * x bf16 [rows, K]; codes uint8 [rows, K] (row stride K); scales float32
 * [rows, ceil(K/128)].  K % 16 == 0. */
biv_status biv_act_quant_fp8(const uint16_t* x, int64_t x_stride, int rows, int K,
                             uint8_t* codes, float* scales, biv_stream_t stream);

/* biv_silu_mul followed by biv_act_quant_fp8 of its result, in one pass:
 * gate_up = [g | u] bf16 [rows, 2I] (row stride gu_stride >= 2I); codes
 * uint8 [rows, I] and scales float32 [rows, ceil(I/128)] are bit for bit what
 * the two calls write (the bf16 activation is not stored).  I % 16 == 0. */
biv_status biv_silu_mul_quant_fp8(const uint16_t* gate_up, int64_t gu_stride, int rows, int I,
                                  uint8_t* codes, float* scales, biv_stream_t stream);

/* -------------------------------------------------------------- Top-K ---
 * Sparse-attention selection ("Finish RL Training Faster", section
 * "让训练前向使用推理的数值": fixed tie-break and fixed position order): per row
 * r, among indices j < valid_len[r] with scores[r, j] > -inf, the k largest
 * scores, equal scores resolved toward the LOWER index; the chosen indices
 * are written to idx int32 [rows, k] in ASCENDING index order, padded with
 * -1.  -0.0 and +0.0 compare equal; a NaN score is never chosen.
 * 0 < k <= n <= 32768, ld >= n. */
biv_status biv_topk(const float* scores, int64_t ld, const int32_t* valid_len, int rows, int n,
                    int k, int32_t* idx, biv_stream_t stream);

/* MoE router: per row, the k largest of E logits (ties -> lower expert id),
 * written in rank order (logit descending, id ascending) to idx int32
 * [rows, k]; w float32 [rows, k] = softmax probability of each chosen expert
 * over all E (not renormalised).  E <= 1024, k <= 32. */
biv_status biv_router_topk(const float* logits, int64_t ld, int rows, int E, int k, int32_t* idx,
                           float* w, biv_stream_t stream);

/* Deterministic dispatch: experts idx int32 [T, k] -> offsets int32 [E+1]
 * (rows of expert e = [offsets[e], offsets[e+1])) and perm int32 [T*k]
 * (entry t*k+s of expert e placed at offsets[e] + rank of (t, s) among that
 * expert's entries in ascending (t, s) order); src_row int32 [T, k] is the
 * inverse (row of entry (t, s) in the grouped layout).  T*k <= 1<<20. */
biv_status biv_moe_dispatch(const int32_t* idx, int T, int k, int E, int32_t* offsets,
                            int32_t* perm, int32_t* src_row, biv_stream_t stream);

/* Row gather for grouped GEMM inputs: dst[i, :] = src[perm[i] / k_div, :] for
 * byte rows of `row_bytes` (multiple of 16), i < n. */
biv_status biv_gather_rows(const void* src, int64_t src_stride_bytes, const int32_t* perm,
                           int k_div, int n, int row_bytes, void* dst, int64_t dst_stride_bytes,
                           biv_stream_t stream);

/* FP32 fixed-slot combine ("Finish RL Training Faster", section
 * "让训练前向使用推理的数值": expert outputs merged in FP32 in slot order):
 * out[t] = bf16( sum_{s=0..k-1, in order} w[t,s]*float(y_row(t,s)) + float(shared[t]) )
 * with y_row(t,s) = y[src_row[t*k+s]] when src_row != NULL, else y[t*k+s];
 * y bf16 [*, d], shared bf16 [T, d] or NULL, out bf16 [T, d]. */
biv_status biv_moe_combine(const uint16_t* y, const int32_t* src_row, const float* w,
                           const uint16_t* shared, uint16_t* out, int T, int k, int d,
                           biv_stream_t stream);

/* ------------------------------------------------------------ log-prob --
 * lp[t] = z[t, target[t]] - (m + log sum_v exp(z[t, v] - m)), m = max_v z,
 * in FP32 with a reduction order that depends on V only (the logprob of
 * every sampled token, "Finish RL Training Faster", section
 * "零差异需要一个精确的比较对象").  logits float32 [T, V] rows at ld. */
biv_status biv_logprob(const float* logits, int64_t ld, const int32_t* target, int T, int V,
                       float* lp, biv_stream_t stream);

/* LM head with the log-softmax gather in its epilogue: lp[t] = z[t, target[t]]
 * - logsumexp_v z[t, v] for z = h . W^T, without writing the FP32 logits
 * (same source as biv_logprob).  The GEMM is biv_gemm's bf16 schedule (K
 * chunks in INVARIANT mode), folded in the CTA on 256-column tiles for every
 * M.  Its epilogue reduces each row's logits in groups of 128 columns
 * (group g = columns [128g, 128g+128) of V) to m_g = max z and
 * s_g = sum exp(z - m_g), summed as four interleaved chains (column mod 4,
 * ascending) added as (c0 + c1) + (c2 + c3); a second kernel forms
 * M = max_g m_g and S = sum_g s_g * exp(m_g - M) (lane l of a warp takes
 * groups l, l+32, ... in order, then a xor tree) and lp = z_t - (M + log S).
 * Every step depends on V and the row only, so a row's lp has the same bits
 * in every batch.
 * h bf16 [M, K] rows at ldh; W bf16 [V, K] rows at ldw (K-major, 16-byte
 * aligned rows); target int32 [M]; lp float32 [M].  V % 4 == 0, K % 8 == 0.
 * A target outside [0, V) gives lp = NaN and the device error code 2.
 * Workspace: device memory of biv_lm_head_logprob_workspace(M, V) bytes,
 * 16-byte aligned, owned by the caller, no initial value needed; calls that
 * can overlap on the GPU need separate workspaces. */
biv_status biv_lm_head_logprob_workspace(int M, int V, size_t* bytes);
biv_status biv_lm_head_logprob(const uint16_t* h, int64_t ldh, const uint16_t* W, int64_t ldw,
                               int M, int V, int K, const int32_t* target, int mode, float* lp,
                               void* workspace, size_t workspace_bytes, biv_stream_t stream);

/* ------------------------------------------------------------- SSD scan --
 * Mamba-2 SSD over chunks of `chunk` positions aligned to absolute positions
 * ("Finish RL Training Faster", section "一致性有多个层面": decode replays the
 * prefill chunk order).  For each sequence i, rows [row0[i], row0[i]+n[i])
 * of x/dt/B/C are its next n[i] tokens, starting at absolute position pos0[i].
 * Per sequence the library keeps, in caller memory:
 *   state  float32 [nseq, H, P, N]: the state at the start of the open chunk;
 *   buf_x  bf16 [nseq, chunk, H, P], buf_B/buf_C bf16 [nseq, chunk, N],
 *   buf_dt float32 [nseq, chunk, H]: the open chunk's rows so far.
 * Every output row y_t is computed from its chunk's start state and the
 * chunk's rows <= t with one code path, so prefill, chunked prefill and
 * token-by-token decode give the same bits.  When a chunk closes its end
 * state replaces `state`.  Set state to zero for a new sequence (pos0 = 0).
 * H*P, N: P in {64}, N in {128}; chunk in {64, 128, 256}. */
typedef struct {
  const uint16_t* x; int64_t x_stride;   /* [rows, H, P] */
  const float* dt;   int64_t dt_stride;  /* [rows, H] (after softplus) */
  const float* A;                        /* [H], negative */
  const uint16_t* B; int64_t B_stride;   /* [rows, N] */
  const uint16_t* C; int64_t C_stride;   /* [rows, N] */
  const float* D;                        /* [H] */
  uint16_t* y; int64_t y_stride;         /* [rows, H, P] */
  int H, P, N, chunk;
  int nseq;
  const int32_t* row0;                   /* [nseq] */
  const int32_t* n;                      /* [nseq] */
  const int32_t* pos0;                   /* [nseq] */
  int max_n;                             /* host bound on n[i] */
  float* state;
  uint16_t* buf_x;
  uint16_t* buf_B;
  uint16_t* buf_C;
  float* buf_dt;
  void* workspace;                       /* optional, biv_ssd_workspace bytes, 16-byte aligned */
  size_t workspace_bytes;
} biv_ssd_desc;

/* Workspace of the parallel path (0 when no sequence has more than 4 new rows,
 * where one CTA per (sequence, head) runs the chunk).  With a large enough
 * workspace a call with many new rows runs every (sequence, chunk, head) in
 * parallel and hands states on chunk to chunk; without one it runs the
 * per-(sequence, head) path.  Both evaluate every row with the same FP32
 * operations in the same order, so the choice changes no bit.  The workspace
 * needs no initial value. */
biv_status biv_ssd_workspace(const biv_ssd_desc* desc, size_t* bytes);
biv_status biv_ssd_scan(const biv_ssd_desc* desc, biv_stream_t stream);

/* ------------------------------------------------- Mamba-2 mixer steps --
 * The steps of a Mamba-2 layer around biv_ssd_scan ("Finish RL Training
 * Faster", section "两组结果，要连同分母一起读": the Mamba-2 hybrid; section
 * "一致性有多个层面": decode replays the prefill order bit for bit).
 *
 * biv_causal_conv1d: depthwise causal convolution of width 4 over the
 * `channels` xBC columns of the in-projection output u (columns col_x ..),
 * then SiLU, rounded to bf16 into out [T, channels]:
 *   out[t, c] = bf16(silu(acc)), acc = b[c]; acc = acc + w[c, j] * x[t-3+j, c]
 *   for j = 0..3 in FP32, product and sum each rounded (no fma);
 * and, over the `heads` dt columns (col_dt ..), dt_out[t, h] =
 * softplus(dt_raw + dt_bias[h]) in FP32 (x > 20 gives x).  Rows of sequence
 * i (0 <= i < nseq) are rows row0[i] .. row0[i]+n[i]-1 of this call, at
 * consecutive positions from pos0[i]; row_seq / row_pos give each row's i
 * and position.  Inputs before a sequence's first row in the call come from
 * state [nseq, 3, channels] bf16 (the three inputs that preceded it; zero for
 * a new sequence, pos0 = 0), so prefill, chunked prefill and decode give the
 * same bits.  After the call state[i] holds the last three inputs of every
 * sequence with n[i] > 0.  conv_w bf16 [channels, 4], conv_b bf16
 * [channels], dt_bias fp32 [heads].  channels and heads multiples of 8;
 * u, out rows and state 16-byte aligned.  A row whose (row_seq, row_pos) is
 * not one of its sequence's rows is reported through biv_poll_error and
 * written as zeros. */
typedef struct {
  const uint16_t* u; int64_t u_stride;
  int col_x, col_dt, channels, heads, width;   /* width must be 4 */
  const uint16_t* conv_w; const uint16_t* conv_b; const float* dt_bias;
  uint16_t* out; int64_t out_stride;
  float* dt_out; int64_t dt_stride;
  int T;
  const int32_t* row_seq; const int32_t* row_pos;
  int nseq;
  const int32_t* row0; const int32_t* n; const int32_t* pos0;
  uint16_t* state;
} biv_conv_desc;
biv_status biv_causal_conv1d(const biv_conv_desc* desc, biv_stream_t stream);

/* Gated RMSNorm of the Mamba-2 output: g = y * silu(z) in FP32 (not
 * rounded), out = bf16((g * inv) * w), inv = 1/sqrt(mean(g^2) + eps), the
 * same per-row reduction tree as biv_add_rmsnorm.  y, z, out bf16 rows of d
 * (d a multiple of 8, at most 8192), w bf16 [d]. */
biv_status biv_gated_rmsnorm(const uint16_t* y, int64_t y_stride, const uint16_t* z,
                             int64_t z_stride, const uint16_t* w, uint16_t* out,
                             int64_t out_stride, int rows, int d, float eps, biv_stream_t stream);

/* NVFP4 weights to bf16 ("Finish RL Training Faster", section
 * "两组结果，要连同分母一起读": NVFP4 weights): out[n, k] = e2m1(code[n, k])
 * * e4m3(scales[n, k/16]), global scale 1.  codes uint8 [N, K/2] packed two
 * per byte (element 2i in the low nibble of byte i), scales uint8 [N, K/16]
 * (e4m3), out bf16 [N, K]; the product is exact in bf16.  K a multiple of
 * 16, codes and out 16-byte aligned. */
biv_status biv_nvfp4_dequant(const uint8_t* codes, const uint8_t* scales, int N, int K,
                             uint16_t* out, biv_stream_t stream);

/* GEMM with NVFP4 weights (W4A16): C[M, N] = A[M, K] . W^T with W = the
 * biv_nvfp4_dequant of (codes, scales), every output bit equal to biv_gemm
 * on that bf16 W (same K-chunk schedule, same tcgen05 MMAs; "Finish RL
 * Training Faster", section "两组结果，要连同分母一起读": NVFP4 weights, and
 * section "让训练前向使用推理的数值": one schedule for every batch).  When
 * the bf16 plan would spread a few output tiles' K chunks over the SMs
 * (decode-sized M), the kernel streams the packed codes and scales by TMA
 * and decodes them in shared memory: 0.5625 bytes of HBM per weight instead
 * of 2 (K a multiple of 256).  Otherwise (many rows: compute-bound; or
 * another K) the weights are decoded once into the workspace and the bf16
 * GEMM runs.  A bf16 [M, K] row-major
 * (lda >= K); codes/scales as for biv_nvfp4_dequant; C bf16 or f32 (c_dtype)
 * [M, ldc].  K a multiple of 16; every pointer 16-byte aligned.  Workspace:
 * biv_gemm_nvfp4_workspace bytes (0 possible), caller-owned, 16-byte
 * aligned, no initial value; BIV_ERR_WORKSPACE when missing or too small. */
biv_status biv_gemm_nvfp4_workspace(int M, int N, int K, int c_dtype, int mode, size_t* bytes);
biv_status biv_gemm_nvfp4(const uint16_t* A, int64_t lda, const uint8_t* codes,
                          const uint8_t* scales, int M, int N, int K, void* C, int64_t ldc,
                          int c_dtype, int mode, void* workspace, size_t workspace_bytes,
                          biv_stream_t stream);

/* ------------------------------------------------------------ backward --
 * Backward of the fused forward ops for a trainer that runs the inference
 * ops' own backward ("No More Train-Inference Mismatch", section "方法细节"),
 * the FP8 KV round trip passing gradients straight through ("Finish RL
 * Training Faster", section "让训练前向使用推理的数值").  FP32 on the CUDA
 * cores; every reduction has one order fixed by the shapes (per-row trees,
 * ascending loops), so results repeat bit for bit, and a row's dx / dz / dq
 * depends on that row (and, for dq, its keys) only.
 *
 * RMSNorm of x (bf16 rows of d, gain w bf16 [d]): dy, dx float32 rows;
 * dx = inv*(w*dy) - x*(inv^3*sum(x*w*dy)/d), inv = 1/sqrt(mean(x^2)+eps);
 * dw float32 [d] = sum over rows in ascending order of dy*x*inv.  Workspace:
 * rows*d*4 bytes (caller-owned, no initial value). */
biv_status biv_rmsnorm_backward(const uint16_t* x, int64_t x_stride, const uint16_t* w,
                                const float* dy, int64_t dy_stride, float* dx, int64_t dx_stride,
                                float* dw, int rows, int d, float eps, void* workspace,
                                size_t workspace_bytes, biv_stream_t stream);

/* SiLU-mul: gate_up bf16 [rows, 2I] ([gate | up]), dy float32 [rows, I] ->
 * dgate_up float32 [rows, 2I]: dgate = dy*up*s*(1+gate*(1-s)), dup =
 * dy*gate*s, s = 1/(1+exp(-gate)). */
biv_status biv_silu_mul_backward(const uint16_t* gate_up, int64_t gate_up_stride, const float* dy,
                                 int64_t dy_stride, float* dgate_up, int64_t dgate_up_stride,
                                 int rows, int I, biv_stream_t stream);

/* logprob: logits float32 [T, V] (ld), target int32 [T], dlp float32 [T] ->
 * dz float32 [T, V] (ldz) = dlp*(onehot(target) - exp(z - lse)); lse from a
 * per-row max and sum in a fixed order.  A target outside [0, V) is reported
 * through biv_poll_error. */
biv_status biv_logprob_backward(const float* logits, int64_t ld, const int32_t* target,
                                const float* dlp, int T, int V, float* dz, int64_t ldz,
                                biv_stream_t stream);

/* Causal GQA attention of one sequence: q, dout bf16 [Tq, Hq, D]; k, v bf16
 * [Tk, Hkv, D] (the cache's dequantised values: an FP8 round trip passes dk,
 * dv through unchanged); key j is visible to row i iff k_pos[j] <= q_pos[i].
 * dq float32 [Tq, Hq, D], dk, dv float32 [Tk, Hkv, D]: with p = softmax(s),
 * s = q.k*scale, D_i = dout_i . o_i, ds = p*(dout.v - D): dq = sum_j ds k
 * scale (keys ascending), dk = sum ds q scale and dv = sum p dout (rows
 * ascending, q heads of the group ascending).  D <= 128.  workspace float32
 * [2*Tq*Hq] (row statistics, no initial value). */
typedef struct {
  const uint16_t* q; const uint16_t* k; const uint16_t* v; const uint16_t* dout;
  float* dq; float* dk; float* dv;
  int Tq, Tk, Hq, Hkv, D;
  const int32_t* q_pos; const int32_t* k_pos;
  float scale;
  float* workspace;
} biv_attn_bwd_desc;
biv_status biv_attention_backward(const biv_attn_bwd_desc* desc, biv_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* BIV_H */
