"""bf16 and FP8 E4M3 codecs of the oracle (numpy, independent of the CUDA path).

bf16: the upper 16 bits of an IEEE binary32, rounded to nearest, ties to even.
e4m3: OCP 8-bit floating point "E4M3FN": sign, 4 exponent bits (bias 7),
3 mantissa bits, no infinities, a single NaN pattern per sign (S.1111.111),
largest finite value 448, smallest subnormal 2^-9.  The quantisers round to
nearest with ties to even and saturate to +-448 ("satfinite").

These carry the "same quantisation rules" that the pages require for every
path ("Finish RL Training Faster", section "零差异需要一个精确的比较对象").
"""
from __future__ import annotations

import numpy as np

# ----------------------------------------------------------------- bf16 ----


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Decode bf16 payloads (uint16) to float32 exactly."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """Encode float32 to bf16 payloads, round to nearest even; NaN stays NaN."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        r = r.copy()
        r[nan] = ((u[nan] >> np.uint64(16)).astype(np.uint16) | np.uint16(0x0040))
    return r


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float32 values onto the bf16 grid (result stays float32)."""
    return bf16_to_f32(f32_to_bf16(x))


# ----------------------------------------------------------------- e4m3 ----

E4M3_MAX = 448.0


def _e4m3_value(code: int) -> float:
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


E4M3_TABLE = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)
# non-negative finite codes 0x00..0x7E in increasing order of value
_POS = E4M3_TABLE[:0x7F]


def e4m3_to_f32(codes: np.ndarray) -> np.ndarray:
    """Decode e4m3 codes (uint8) to float32 exactly."""
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8)].astype(np.float32)


def f32_to_e4m3(x: np.ndarray) -> np.ndarray:
    """Quantise float32 to e4m3: nearest finite value, ties to the even code,
    magnitudes beyond 448 saturate to 448, NaN -> 0x7F (sign kept)."""
    x = np.asarray(x, dtype=np.float32)
    a = np.abs(x.astype(np.float64))
    neg = np.signbit(x)
    nan = np.isnan(x)
    a = np.where(nan, 0.0, a)
    # index of the largest representable value <= a
    i = np.clip(np.searchsorted(_POS, a, side="right") - 1, 0, 0x7E)
    j = np.minimum(i + 1, 0x7E)
    lo, hi = _POS[i], _POS[j]
    d_lo, d_hi = a - lo, hi - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (j % 2 == 0) & (j != i))
    code = np.where(pick_hi, j, i)
    code = np.where(a >= E4M3_MAX, 0x7E, code).astype(np.uint8)
    code = np.where(nan, np.uint8(0x7F), code).astype(np.uint8)
    return (code | np.where(neg, np.uint8(0x80), np.uint8(0))).astype(np.uint8)


# ----------------------------------------------------------------- e2m1 ----
# OCP 4-bit floating point "E2M1": sign, 2 exponent bits (bias 1), 1 mantissa
# bit, no infinities or NaN.  Exponent field 0 is subnormal (0 and 0.5).

def _e2m1_value(code: int) -> float:
    s = -1.0 if code & 0x8 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        return s * m * 0.5
    return s * (1.0 + m / 2.0) * 2.0 ** (e - 1)


E2M1_TABLE = np.array([_e2m1_value(c) for c in range(16)], dtype=np.float64)


def e2m1_to_f32(codes: np.ndarray) -> np.ndarray:
    """Decode e2m1 codes (low 4 bits of uint8) to float32 exactly."""
    return E2M1_TABLE[np.asarray(codes, dtype=np.uint8) & 0xF].astype(np.float32)


def nvfp4_unpack(packed: np.ndarray) -> np.ndarray:
    """Packed NVFP4 codes [N, K/2] -> one e2m1 code per element [N, K]:
    element 2i is the low nibble of byte i, element 2i+1 the high nibble."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def nvfp4_dequant(packed: np.ndarray, scale_codes: np.ndarray, block: int = 16) -> np.ndarray:
    """NVFP4 weights [N, K]: packed e2m1 codes [N, K/2] (nvfp4_unpack) times
    one e4m3 scale per block of 16 consecutive K elements (scale codes
    [N, K/16]), global scale 1.
    A 2-significant-bit value times a 4-significant-bit scale has at most 6
    significant bits, so the product is exact in FP32 and lies on the bf16
    grid (unless it leaves bf16's exponent range, which e4m3 scales cannot
    reach)."""
    v = e2m1_to_f32(nvfp4_unpack(packed)).astype(np.float64)
    s = np.repeat(e4m3_to_f32(scale_codes).astype(np.float64), block, axis=-1)[..., :v.shape[-1]]
    return (v * s).astype(np.float32)
