"""Python binding of libbiv: the C-ABI entry points of ``include/biv.h`` under
the same names, taking torch CUDA tensors.  Argument marshalling only: every
step runs in the library's CUDA kernels.  There is no CPU fallback; a missing
or unloadable library raises.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Dict, Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libbiv.so")

BIV_OK, BIV_ERR_INVALID, BIV_ERR_UNSUPPORTED, BIV_ERR_WORKSPACE, BIV_ERR_CUDA, BIV_ERR_TIMEOUT = range(6)
MODE_INVARIANT, MODE_FAST = 0, 1
BF16, F32, E4M3 = 0, 1, 2

EXPORTS = [
    "biv_version", "biv_last_error", "biv_device_sm_count", "biv_poll_error",
    "biv_selftest_timeout", "biv_embed", "biv_add_rmsnorm", "biv_add_rmsnorm_partials", "biv_silu_mul",
    "biv_rope_table", "biv_qk_norm_rope", "biv_kv_store_bf16", "biv_kv_fp8_quant", "biv_qkv_finalize", "biv_silu_mul_partials",
    "biv_kv_fp8_gather", "biv_attention_workspace", "biv_attention", "biv_attention_noalloc",
    "biv_gemm_workspace", "biv_gemm_partials", "biv_gemm",
    "biv_act_quant_fp8", "biv_silu_mul_quant_fp8", "biv_topk", "biv_router_topk", "biv_moe_dispatch", "biv_gather_rows",
    "biv_moe_combine", "biv_logprob", "biv_lm_head_logprob_workspace", "biv_lm_head_logprob",
    "biv_ssd_workspace", "biv_ssd_scan",
    "biv_causal_conv1d", "biv_gated_rmsnorm", "biv_nvfp4_dequant",
    "biv_gemm_nvfp4_workspace", "biv_gemm_nvfp4",
    "biv_rmsnorm_backward", "biv_silu_mul_backward", "biv_logprob_backward", "biv_attention_backward",
]


class BivError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"libbiv status {status}: {msg}")
        self.status = status


class GemmDesc(C.Structure):
    _fields_ = [("M", C.c_int), ("N", C.c_int), ("K", C.c_int),
                ("a_dtype", C.c_int), ("b_dtype", C.c_int), ("c_dtype", C.c_int),
                ("A", C.c_void_p), ("lda", C.c_int64),
                ("B", C.c_void_p), ("ldb", C.c_int64),
                ("C", C.c_void_p), ("ldc", C.c_int64),
                ("sa", C.c_void_p), ("ld_sa", C.c_int64),
                ("sb", C.c_void_p),
                ("group_offsets", C.c_void_p), ("groups", C.c_int),
                ("mode", C.c_int), ("defer_fold", C.c_int)]


class Partials(C.Structure):
    """Chunk partials a GEMM left for its consumer (see include/biv.h)."""
    _fields_ = [("p", C.c_void_p), ("chunks", C.c_int), ("ld", C.c_int64),
                ("chunk_stride", C.c_int64)]


class AttnDesc(C.Structure):
    _fields_ = [("q", C.c_void_p), ("q_stride", C.c_int64),
                ("out", C.c_void_p), ("out_stride", C.c_int64),
                ("T", C.c_int), ("Hq", C.c_int), ("Hkv", C.c_int), ("D", C.c_int),
                ("row_seq", C.c_void_p), ("row_pos", C.c_void_p),
                ("qblocks", C.c_void_p), ("nqblocks", C.c_int),
                ("max_rows_per_block", C.c_int),
                ("kv_dtype", C.c_int),
                ("k_cache", C.c_void_p), ("v_cache", C.c_void_p),
                ("k_scale", C.c_void_p), ("v_scale", C.c_void_p),
                ("block_table", C.c_void_p), ("max_pages", C.c_int),
                ("page", C.c_int), ("kv_split", C.c_int), ("max_ctx", C.c_int),
                ("topk_idx", C.c_void_p), ("topk_stride", C.c_int64), ("topk", C.c_int),
                ("scale", C.c_float), ("mode", C.c_int), ("num_pages", C.c_int)]


class SSDDesc(C.Structure):
    _fields_ = [("x", C.c_void_p), ("x_stride", C.c_int64),
                ("dt", C.c_void_p), ("dt_stride", C.c_int64),
                ("A", C.c_void_p),
                ("B", C.c_void_p), ("B_stride", C.c_int64),
                ("C", C.c_void_p), ("C_stride", C.c_int64),
                ("D", C.c_void_p),
                ("y", C.c_void_p), ("y_stride", C.c_int64),
                ("H", C.c_int), ("P", C.c_int), ("N", C.c_int), ("chunk", C.c_int),
                ("nseq", C.c_int),
                ("row0", C.c_void_p), ("n", C.c_void_p), ("pos0", C.c_void_p),
                ("max_n", C.c_int),
                ("state", C.c_void_p), ("buf_x", C.c_void_p), ("buf_B", C.c_void_p),
                ("buf_C", C.c_void_p), ("buf_dt", C.c_void_p),
                ("workspace", C.c_void_p), ("workspace_bytes", C.c_size_t)]


class ConvDesc(C.Structure):
    _fields_ = [("u", C.c_void_p), ("u_stride", C.c_int64),
                ("col_x", C.c_int), ("col_dt", C.c_int), ("channels", C.c_int), ("heads", C.c_int),
                ("width", C.c_int),
                ("conv_w", C.c_void_p), ("conv_b", C.c_void_p), ("dt_bias", C.c_void_p),
                ("out", C.c_void_p), ("out_stride", C.c_int64),
                ("dt_out", C.c_void_p), ("dt_stride", C.c_int64),
                ("T", C.c_int),
                ("row_seq", C.c_void_p), ("row_pos", C.c_void_p),
                ("nseq", C.c_int),
                ("row0", C.c_void_p), ("n", C.c_void_p), ("pos0", C.c_void_p),
                ("state", C.c_void_p)]


class AttnBwdDesc(C.Structure):
    _fields_ = [("q", C.c_void_p), ("k", C.c_void_p), ("v", C.c_void_p), ("dout", C.c_void_p),
                ("dq", C.c_void_p), ("dk", C.c_void_p), ("dv", C.c_void_p),
                ("Tq", C.c_int), ("Tk", C.c_int), ("Hq", C.c_int), ("Hkv", C.c_int), ("D", C.c_int),
                ("q_pos", C.c_void_p), ("k_pos", C.c_void_p), ("scale", C.c_float),
                ("workspace", C.c_void_p)]


_lib: Optional[C.CDLL] = None


def load(path: str = LIB_PATH) -> C.CDLL:
    """Load libbiv.so (built by ``build.build()``); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libbiv.so not found at {path}: run invariant_forward_bitwise_gb300.build.build()")
    lib = C.CDLL(path)
    P, I, I64, F, D_ = C.c_void_p, C.c_int, C.c_int64, C.c_float, C.c_double
    sig = {
        "biv_version": ([], I), "biv_last_error": ([], C.c_char_p),
        "biv_device_sm_count": ([], I), "biv_poll_error": ([P, P], I),
        "biv_selftest_timeout": ([C.c_uint64, P], I),
        "biv_embed": ([P, P, I, I, I, P, I64, P], I),
        "biv_add_rmsnorm": ([P, I64, P, I64, P, P, I64, I, I, F, P], I),
        "biv_add_rmsnorm_partials": ([P, P, I64, P, P, I64, I, I, F, P], I),
        "biv_qkv_finalize": ([P, I64, P, I, I, I, I, P, P, P, I, P, F, P, I, P, P, P, P, P], I),
        "biv_gemm_partials": ([P, P, P], I),
        "biv_silu_mul": ([P, I64, P, I64, I, I, P], I),
        "biv_silu_mul_partials": ([P, P, I64, I, I, P], I),
        "biv_rope_table": ([D_, I, I, P, P], I),
        "biv_qk_norm_rope": ([P, I64, I, I, I, I, P, P, P, I, P, F, P], I),
        "biv_kv_store_bf16": ([P, P, I64, P, I, I, I, P, P, P], I),
        "biv_kv_fp8_quant": ([P, P, I64, P, I, I, I, P, P, P, P, P], I),
        "biv_kv_fp8_gather": ([P, P, P, I, P, P, I, I, I, I, P, P], I),
        "biv_attention_workspace": ([P, P], I), "biv_attention": ([P, P, C.c_size_t, P], I),
        "biv_attention_noalloc": ([P, P], I),
        "biv_gemm_workspace": ([P, P], I), "biv_gemm": ([P, P, C.c_size_t, P], I),
        "biv_act_quant_fp8": ([P, I64, I, I, P, P, P], I),
        "biv_silu_mul_quant_fp8": ([P, I64, I, I, P, P, P], I),
        "biv_topk": ([P, I64, P, I, I, I, P, P], I),
        "biv_router_topk": ([P, I64, I, I, I, P, P, P], I),
        "biv_moe_dispatch": ([P, I, I, I, P, P, P, P], I),
        "biv_gather_rows": ([P, I64, P, I, I, I, P, I64, P], I),
        "biv_moe_combine": ([P, P, P, P, P, I, I, I, P], I),
        "biv_logprob": ([P, I64, P, I, I, P, P], I),
        "biv_lm_head_logprob_workspace": ([I, I, P], I),
        "biv_lm_head_logprob": ([P, I64, P, I64, I, I, I, P, I, P, P, C.c_size_t, P], I),
        "biv_ssd_workspace": ([P, P], I), "biv_ssd_scan": ([P, P], I),
        "biv_causal_conv1d": ([P, P], I),
        "biv_gated_rmsnorm": ([P, I64, P, I64, P, P, I64, I, I, F, P], I),
        "biv_nvfp4_dequant": ([P, P, I, I, P, P], I),
        "biv_gemm_nvfp4_workspace": ([I, I, I, I, I, P], I),
        "biv_gemm_nvfp4": ([P, I64, P, P, I, I, I, P, I64, I, I, P, C.c_size_t, P], I),
        "biv_rmsnorm_backward": ([P, I64, P, P, I64, P, I64, P, I, I, F, P, C.c_size_t, P], I),
        "biv_silu_mul_backward": ([P, I64, P, I64, P, I64, I, I, P], I),
        "biv_logprob_backward": ([P, I64, P, P, I, I, P, I64, P], I),
        "biv_attention_backward": ([P, P], I),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name, None)
        if fn is None:
            continue
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def missing_exports(path: str = LIB_PATH) -> list:
    lib = C.CDLL(path)
    return [n for n in EXPORTS if not hasattr(lib, n)]


# ------------------------------------------------------------- helpers ----
def _p(t: Optional[torch.Tensor]):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream) -> C.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream)


def _check(st: int, what: str):
    if st != BIV_OK:
        raise BivError(st, f"{what}: {load().biv_last_error().decode()}")


def _rs(t: torch.Tensor) -> int:
    """row stride (elements) of a 2-D view."""
    return t.stride(0) if t.dim() >= 2 else t.shape[-1]


def _bf16_ok(*ts):
    for t in ts:
        if t is not None:
            assert t.is_cuda and t.dtype == torch.bfloat16, "expected a CUDA bf16 tensor"


# ------------------------------------------------------------ entry points --
def biv_version() -> int:
    return load().biv_version()


def biv_device_sm_count() -> int:
    return load().biv_device_sm_count()


def biv_poll_error(stream=None) -> int:
    code = C.c_int(0)
    st = load().biv_poll_error(_stream(stream), C.byref(code))
    if st not in (BIV_OK, BIV_ERR_TIMEOUT, BIV_ERR_INVALID):
        _check(st, "biv_poll_error")
    return code.value


def biv_selftest_timeout(limit_ns: int, stream=None):
    _check(load().biv_selftest_timeout(int(limit_ns), _stream(stream)), "biv_selftest_timeout")


def biv_embed(ids, table, h, stream=None):
    _bf16_ok(table, h)
    _check(load().biv_embed(_p(ids), _p(table), table.shape[0], ids.shape[0], table.shape[1],
                            _p(h), _rs(h), _stream(stream)), "biv_embed")


def biv_add_rmsnorm(x, residual, w, y, eps, stream=None):
    """residual may be None; rows = x.shape[0]."""
    _bf16_ok(x, residual, w, y)
    rows, d = x.shape[0], x.shape[-1]
    _check(load().biv_add_rmsnorm(_p(x), _rs(x), _p(residual), _rs(residual) if residual is not None else 0,
                                  _p(w), _p(y), _rs(y), rows, d, float(eps), _stream(stream)),
           "biv_add_rmsnorm")


def biv_silu_mul(gate_up, y, stream=None):
    _bf16_ok(gate_up, y)
    _check(load().biv_silu_mul(_p(gate_up), _rs(gate_up), _p(y), _rs(y), gate_up.shape[0],
                               y.shape[-1], _stream(stream)), "biv_silu_mul")


def biv_rope_table(theta, D, max_pos, out, stream=None):
    assert out.dtype == torch.float32 and out.numel() >= 2 * max_pos * (D // 2)
    _check(load().biv_rope_table(float(theta), D, max_pos, _p(out), _stream(stream)), "biv_rope_table")


def biv_add_rmsnorm_partials(xp: "Partials", residual, w, y, rows, eps, stream=None):
    """x given as GEMM chunk partials; rows/d from the arguments."""
    _bf16_ok(residual, w, y)
    d = y.shape[-1]
    _check(load().biv_add_rmsnorm_partials(C.byref(xp), _p(residual),
                                           _rs(residual) if residual is not None else 0, _p(w), _p(y),
                                           _rs(y), rows, d, float(eps), _stream(stream)),
           "biv_add_rmsnorm_partials")


def biv_silu_mul_partials(gp: "Partials", y, rows, stream=None):
    """gate_up given as GEMM chunk partials; I = y.shape[-1]."""
    _bf16_ok(y)
    _check(load().biv_silu_mul_partials(C.byref(gp), _p(y), _rs(y), rows, y.shape[-1],
                                        _stream(stream)), "biv_silu_mul_partials")


def biv_qkv_finalize(qkv, T, Hq, Hkv, D, q_w, k_w, cos_sin, max_pos, pos, eps, slot, kv_dtype,
                     k_cache, v_cache, k_scale=None, v_scale=None, partials: Optional["Partials"] = None,
                     stream=None):
    _check(load().biv_qkv_finalize(_p(qkv), _rs(qkv), C.byref(partials) if partials is not None else None,
                                   T, Hq, Hkv, D, _p(q_w), _p(k_w), _p(cos_sin), max_pos, _p(pos),
                                   float(eps), _p(slot), kv_dtype, _p(k_cache), _p(v_cache), _p(k_scale),
                                   _p(v_scale), _stream(stream)), "biv_qkv_finalize")


def biv_gemm_partials(desc: GemmDesc, ws: Optional[torch.Tensor]) -> "Partials":
    out = Partials()
    _check(load().biv_gemm_partials(C.byref(desc), _p(ws), C.byref(out)), "biv_gemm_partials")
    return out


def biv_qk_norm_rope(qkv, T, Hq, Hkv, D, q_w, k_w, cos_sin, max_pos, pos, eps, stream=None):
    _check(load().biv_qk_norm_rope(_p(qkv), _rs(qkv), T, Hq, Hkv, D, _p(q_w), _p(k_w), _p(cos_sin),
                                   max_pos, _p(pos), float(eps), _stream(stream)), "biv_qk_norm_rope")


def biv_kv_store_bf16(k, v, row_stride, slot, T, Hkv, D, k_cache, v_cache, stream=None):
    _check(load().biv_kv_store_bf16(_p(k), _p(v), row_stride, _p(slot), T, Hkv, D, _p(k_cache),
                                    _p(v_cache), _stream(stream)), "biv_kv_store_bf16")


def biv_kv_fp8_quant(k, v, row_stride, slot, T, Hkv, D, kc, vc, ks, vs, stream=None):
    _check(load().biv_kv_fp8_quant(_p(k), _p(v), row_stride, _p(slot), T, Hkv, D, _p(kc), _p(vc),
                                   _p(ks), _p(vs), _stream(stream)), "biv_kv_fp8_quant")


def biv_kv_fp8_gather(codes, scales, block_table, ctx_len, out_row0, Hkv, D, page, out, stream=None):
    _check(load().biv_kv_fp8_gather(_p(codes), _p(scales), _p(block_table), block_table.shape[1],
                                    _p(ctx_len), _p(out_row0), ctx_len.shape[0], Hkv, D, page,
                                    _p(out), _stream(stream)), "biv_kv_fp8_gather")


def biv_attention_workspace(desc: AttnDesc) -> int:
    n = C.c_size_t(0)
    _check(load().biv_attention_workspace(C.byref(desc), C.byref(n)), "biv_attention_workspace")
    return n.value


def biv_attention(desc: AttnDesc, ws: Optional[torch.Tensor], stream=None):
    _check(load().biv_attention(C.byref(desc), _p(ws), 0 if ws is None else ws.numel() * ws.element_size(),
                                _stream(stream)), "biv_attention")


def biv_attention_noalloc(desc: AttnDesc, stream=None):
    """biv_attention without a caller workspace (see include/biv.h)."""
    _check(load().biv_attention_noalloc(C.byref(desc), _stream(stream)), "biv_attention_noalloc")


def gemm_desc(A, B, Cout, mode=MODE_INVARIANT, sa=None, sb=None, group_offsets=None, groups=0,
              M=None) -> GemmDesc:
    dt = {torch.bfloat16: BF16, torch.float32: F32, torch.uint8: E4M3, torch.float8_e4m3fn: E4M3}
    d = GemmDesc()
    d.M = A.shape[0] if M is None else M
    d.N = Cout.shape[1] if groups <= 1 else B.shape[0] // groups
    d.K = A.shape[1]
    d.a_dtype, d.b_dtype, d.c_dtype = dt[A.dtype], dt[B.dtype], dt[Cout.dtype]
    d.A, d.lda = A.data_ptr(), A.stride(0)
    d.B, d.ldb = B.data_ptr(), B.stride(0)
    d.C, d.ldc = Cout.data_ptr(), Cout.stride(0)
    d.sa = sa.data_ptr() if sa is not None else None
    d.ld_sa = sa.stride(0) if sa is not None else 0
    d.sb = sb.data_ptr() if sb is not None else None
    d.group_offsets = group_offsets.data_ptr() if group_offsets is not None else None
    d.groups = groups
    d.mode = mode
    return d


def biv_gemm_workspace(desc: GemmDesc) -> int:
    n = C.c_size_t(0)
    _check(load().biv_gemm_workspace(C.byref(desc), C.byref(n)), "biv_gemm_workspace")
    return n.value


_gemm_scratch: Dict[int, torch.Tensor] = {}


def gemm_scratch(nbytes: int, device=None) -> torch.Tensor:
    """A scratch workspace of at least nbytes (GEMM chunk partials, SSD
    intermediates), cached per device (for callers on one stream)."""
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
    t = _gemm_scratch.get(dev.index)
    if t is None or t.numel() < nbytes:
        t = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
        _gemm_scratch[dev.index] = t
    return t


def biv_gemm(desc: GemmDesc, ws: Optional[torch.Tensor] = None, stream=None):
    """ws: a workspace of biv_gemm_workspace(desc) bytes; when None and the
    plan needs one, a cached per-device scratch buffer is used."""
    if ws is None:
        need = biv_gemm_workspace(desc)
        if need:
            ws = gemm_scratch(need)
    _check(load().biv_gemm(C.byref(desc), _p(ws), 0 if ws is None else ws.numel() * ws.element_size(),
                           _stream(stream)), "biv_gemm")


def biv_act_quant_fp8(x, codes, scales, stream=None):
    _check(load().biv_act_quant_fp8(_p(x), _rs(x), x.shape[0], x.shape[1], _p(codes), _p(scales),
                                    _stream(stream)), "biv_act_quant_fp8")


def biv_silu_mul_quant_fp8(gate_up, codes, scales, stream=None):
    _check(load().biv_silu_mul_quant_fp8(_p(gate_up), _rs(gate_up), gate_up.shape[0],
                                         codes.shape[1], _p(codes), _p(scales), _stream(stream)),
           "biv_silu_mul_quant_fp8")


def biv_topk(scores, valid_len, k, idx, stream=None):
    _check(load().biv_topk(_p(scores), scores.stride(0), _p(valid_len), scores.shape[0],
                           scores.shape[1], k, _p(idx), _stream(stream)), "biv_topk")


def biv_router_topk(logits, k, idx, w, stream=None):
    _check(load().biv_router_topk(_p(logits), logits.stride(0), logits.shape[0], logits.shape[1], k,
                                  _p(idx), _p(w), _stream(stream)), "biv_router_topk")


def biv_moe_dispatch(idx, E, offsets, perm, src_row, stream=None):
    _check(load().biv_moe_dispatch(_p(idx), idx.shape[0], idx.shape[1], E, _p(offsets), _p(perm),
                                   _p(src_row), _stream(stream)), "biv_moe_dispatch")


def biv_gather_rows(src, perm, k_div, n, dst, stream=None):
    rb = src.shape[1] * src.element_size()
    _check(load().biv_gather_rows(_p(src), src.stride(0) * src.element_size(), _p(perm), k_div, n, rb,
                                  _p(dst), dst.stride(0) * dst.element_size(), _stream(stream)),
           "biv_gather_rows")


def biv_moe_combine(y, src_row, w, shared, out, stream=None):
    T, k = w.shape
    _check(load().biv_moe_combine(_p(y), _p(src_row), _p(w), _p(shared), _p(out), T, k, out.shape[1],
                                  _stream(stream)), "biv_moe_combine")


def biv_logprob(logits, target, lp, T=None, stream=None):
    T = logits.shape[0] if T is None else T
    _check(load().biv_logprob(_p(logits), logits.stride(0), _p(target), T, logits.shape[1], _p(lp),
                              _stream(stream)), "biv_logprob")


def biv_lm_head_logprob_workspace(M: int, V: int) -> int:
    n = C.c_size_t(0)
    _check(load().biv_lm_head_logprob_workspace(M, V, C.byref(n)), "biv_lm_head_logprob_workspace")
    return n.value


def biv_lm_head_logprob(h, W, target, lp, workspace, M=None, mode=0, stream=None):
    """lp[:M] = log-softmax of (h[:M] . W^T) at target[:M], without FP32 logits."""
    M = h.shape[0] if M is None else M
    _check(load().biv_lm_head_logprob(_p(h), h.stride(0), _p(W), W.stride(0), M, W.shape[0], h.shape[1],
                                      _p(target), mode, _p(lp), _p(workspace),
                                      workspace.numel() * workspace.element_size(), _stream(stream)),
           "biv_lm_head_logprob")


def biv_ssd_workspace(desc: SSDDesc) -> int:
    n = C.c_size_t(0)
    _check(load().biv_ssd_workspace(C.byref(desc), C.byref(n)), "biv_ssd_workspace")
    return n.value


def biv_ssd_scan(desc: SSDDesc, stream=None):
    """When desc.workspace is unset and the call has many new rows, a cached
    per-device scratch buffer serves as the workspace (callers on one stream)."""
    if not desc.workspace:
        need = biv_ssd_workspace(desc)
        if need:
            ws = gemm_scratch(need)
            desc.workspace, desc.workspace_bytes = ws.data_ptr(), ws.numel()
    _check(load().biv_ssd_scan(C.byref(desc), _stream(stream)), "biv_ssd_scan")


def biv_causal_conv1d(desc: ConvDesc, stream=None):
    _check(load().biv_causal_conv1d(C.byref(desc), _stream(stream)), "biv_causal_conv1d")


def biv_gated_rmsnorm(y, z, w, out, eps, rows=None, stream=None):
    """y, z, out: 2-D bf16 views (rows of d); w bf16 [d]."""
    _bf16_ok(y, z, w, out)
    n = y.shape[0] if rows is None else rows
    _check(load().biv_gated_rmsnorm(_p(y), _rs(y), _p(z), _rs(z), _p(w), _p(out), _rs(out), n,
                                    y.shape[-1], eps, _stream(stream)), "biv_gated_rmsnorm")


def biv_nvfp4_dequant(codes, scales, out, stream=None):
    """codes uint8 [N, K/2] (packed), scales uint8 [N, K/16] (e4m3) -> out bf16 [N, K]."""
    N, K = out.shape
    _check(load().biv_nvfp4_dequant(_p(codes), _p(scales), N, K, _p(out), _stream(stream)),
           "biv_nvfp4_dequant")


def biv_gemm_nvfp4_workspace(M, N, K, c_dtype=BF16, mode=MODE_INVARIANT) -> int:
    n = C.c_size_t(0)
    _check(load().biv_gemm_nvfp4_workspace(M, N, K, c_dtype, mode, C.byref(n)),
           "biv_gemm_nvfp4_workspace")
    return n.value


def biv_gemm_nvfp4(A, codes, scales, Cout, M=None, mode=MODE_INVARIANT, ws=None, stream=None):
    """Cout[M, N] = A[M, K] . dequant(codes, scales)^T; ws: a workspace of
    biv_gemm_nvfp4_workspace bytes (a cached per-device scratch when None)."""
    M = A.shape[0] if M is None else M
    N, K = codes.shape[0], A.shape[1]
    cdt = F32 if Cout.dtype == torch.float32 else BF16
    need = biv_gemm_nvfp4_workspace(M, N, K, cdt, mode)
    if ws is None and need:
        ws = gemm_scratch(need)
    _check(load().biv_gemm_nvfp4(_p(A), A.stride(0), _p(codes), _p(scales), M, N, K, _p(Cout),
                                 Cout.stride(0), cdt, mode, _p(ws), ws.numel() if ws is not None else 0,
                                 _stream(stream)), "biv_gemm_nvfp4")


# ------------------------------------------------------------- backward --
def biv_rmsnorm_backward(x, w, dy, dx, dw, eps, ws=None, stream=None):
    """x bf16 [R, d], w bf16 [d], dy float32 [R, d] -> dx float32 [R, d], dw float32 [d]."""
    R, d = x.shape
    if ws is None:
        ws = gemm_scratch(R * d * 4)
    _check(load().biv_rmsnorm_backward(_p(x), x.stride(0), _p(w), _p(dy), dy.stride(0), _p(dx),
                                       dx.stride(0), _p(dw), R, d, float(eps), _p(ws), ws.numel(),
                                       _stream(stream)), "biv_rmsnorm_backward")


def biv_silu_mul_backward(gate_up, dy, dgate_up, stream=None):
    R, I = dy.shape
    _check(load().biv_silu_mul_backward(_p(gate_up), gate_up.stride(0), _p(dy), dy.stride(0),
                                        _p(dgate_up), dgate_up.stride(0), R, I, _stream(stream)),
           "biv_silu_mul_backward")


def biv_logprob_backward(logits, target, dlp, dz, stream=None):
    T, V = logits.shape
    _check(load().biv_logprob_backward(_p(logits), logits.stride(0), _p(target), _p(dlp), T, V, _p(dz),
                                       dz.stride(0), _stream(stream)), "biv_logprob_backward")


def biv_attention_backward(q, k, v, dout, q_pos, k_pos, scale, dq, dk, dv, stream=None):
    """One sequence: q, dout bf16 [Tq, Hq, D]; k, v bf16 [Tk, Hkv, D]."""
    Tq, Hq, D = q.shape
    ws = gemm_scratch(2 * Tq * Hq * 4)
    d = AttnBwdDesc()
    d.q, d.k, d.v, d.dout = (t.data_ptr() for t in (q, k, v, dout))
    d.dq, d.dk, d.dv = dq.data_ptr(), dk.data_ptr(), dv.data_ptr()
    d.Tq, d.Tk, d.Hq, d.Hkv, d.D = Tq, k.shape[0], Hq, k.shape[1], D
    d.q_pos, d.k_pos, d.scale, d.workspace = q_pos.data_ptr(), k_pos.data_ptr(), float(scale), ws.data_ptr()
    _check(load().biv_attention_backward(C.byref(d), _stream(stream)), "biv_attention_backward")
