"""Pins for the oracle's bf16 / e4m3 codecs (CPU only)."""
import os

import numpy as np
import pytest
import torch

from oracle.codecs import (E4M3_TABLE, bf16_round, bf16_to_f32, e2m1_to_f32, e4m3_to_f32,
                           f32_to_bf16, f32_to_e4m3, nvfp4_dequant, nvfp4_unpack)
from oracle import ops

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLD, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                yield line.split()


def test_e4m3_table_matches_ocp_fixture():
    for code, val in _rows("e4m3_ocp_values.txt"):
        c = int(code, 16)
        got = E4M3_TABLE[c]
        if val == "nan":
            assert np.isnan(got)
        else:
            assert got == float(val), (code, got, val)
            assert np.signbit(got) == val.startswith("-")


def test_e4m3_table_structure():
    pos = E4M3_TABLE[:0x7F]
    assert np.all(np.diff(pos) > 0)                 # strictly increasing codes
    assert pos.max() == 448.0 and pos[1] == 2.0 ** -9
    assert np.array_equal(E4M3_TABLE[0x80:0xFF], -pos)
    assert np.isnan(E4M3_TABLE[0x7F]) and np.isnan(E4M3_TABLE[0xFF])
    assert int(np.isnan(E4M3_TABLE).sum()) == 2


def test_e4m3_encode_matches_torch_cast_in_range():
    g = np.random.default_rng(0)
    x = np.concatenate([
        g.standard_normal(200000).astype(np.float32) * 50,
        g.standard_normal(50000).astype(np.float32) * 0.01,
        # exact midpoints between neighbouring codes (ties -> even code)
        ((E4M3_TABLE[1:0x7E] + E4M3_TABLE[2:0x7F]) / 2).astype(np.float32),
        -((E4M3_TABLE[1:0x7E] + E4M3_TABLE[2:0x7F]) / 2).astype(np.float32),
        np.array([0.0, -0.0, 448.0, -448.0, 2 ** -10, 2 ** -11], np.float32),
    ])
    x = x[np.abs(x) <= 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(f32_to_e4m3(x), ref)


def test_e4m3_satfinite_and_roundtrip():
    assert f32_to_e4m3(np.array([1e6, -1e6, 449.0, 470.0, np.inf, -np.inf], np.float32)).tolist() == \
        [0x7E, 0xFE, 0x7E, 0x7E, 0x7E, 0xFE]
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    assert np.array_equal(f32_to_e4m3(e4m3_to_f32(finite)), finite)


def test_bf16_fixture():
    for f_hex, b_hex in _rows("bf16_values.txt"):
        x = np.array([int(f_hex, 16)], np.uint32).view(np.float32)
        assert int(f32_to_bf16(x)[0]) == int(b_hex, 16), (f_hex, b_hex)


def test_bf16_exhaustive_roundtrip():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = bf16_to_f32(bits)
    ok = ~np.isnan(vals)
    assert np.array_equal(f32_to_bf16(vals)[ok], bits[ok])
    assert np.all(np.isnan(bf16_to_f32(f32_to_bf16(vals[~ok]))))


def test_bf16_encode_matches_torch_and_nearest():
    g = np.random.default_rng(1)
    raw = g.integers(0, 2 ** 32, size=400000, dtype=np.uint64).astype(np.uint32)
    x = raw.view(np.float32)
    x = x[np.isfinite(x)]
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = f32_to_bf16(x)
    assert np.array_equal(got, ref)
    # nearest-value check by brute force on the two neighbours (float64)
    y = x[:20000]
    lo = (y.view(np.uint32) >> 16).astype(np.uint16)
    a = bf16_to_f32(lo).astype(np.float64)
    b = bf16_to_f32((lo.astype(np.uint32) + 1).astype(np.uint16)).astype(np.float64)
    r = bf16_to_f32(f32_to_bf16(y)).astype(np.float64)
    fin = np.isfinite(b) & np.isfinite(r)
    d = np.abs(r - y.astype(np.float64))
    assert np.all(d[fin] <= np.minimum(np.abs(a - y), np.abs(b - y))[fin])


def test_fp8_scale_roundtrip_idempotent():
    """Quantising a dequantised row with the same scale returns the same codes,
    for the FP32 product and for the bf16-rounded product of the KV path."""
    g = np.random.default_rng(2)
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    for s in np.exp2(g.uniform(-20, 8, size=40)).astype(np.float32):
        xf = (e4m3_to_f32(finite) * s).astype(np.float32)
        assert np.array_equal(f32_to_e4m3(xf / s), finite)
        xb = bf16_round(xf)
        assert np.array_equal(f32_to_e4m3(xb / s), finite)


def test_fp8_quant_rows_rules():
    x = np.zeros((3, 16), np.float32)
    x[1] = np.linspace(-3, 5, 16, dtype=np.float32)
    x[2, 3] = -7.0
    c, s = ops.fp8_quant_rows(x)
    assert s[0] == 1.0 and np.all(c[0] == 0)
    assert s[1] == np.float32(5.0) / np.float32(448.0)
    assert c[1, 15] == 0x7E and c[2, 3] == 0xFE
    # quantise -> dequantise -> quantise is stable
    xq = ops.fp8_dequant_rows(c, s)
    c2, s2 = ops.fp8_quant_rows(xq)
    assert np.array_equal(ops.fp8_dequant_rows(c2, s2), ops.fp8_dequant_rows(c, s)) or \
        np.max(np.abs(ops.fp8_dequant_rows(c2, s2) - xq)) <= 2 ** -6 * np.max(np.abs(xq))


def test_e2m1_matches_ocp_fixture():
    got = e2m1_to_f32(np.arange(16, dtype=np.uint8))
    n = 0
    for code, val in _rows("e2m1_ocp_values.txt"):
        c = int(code, 16)
        assert got[c] == float(val) and np.signbit(got[c]) == val.startswith("-"), (code, got[c])
        n += 1
    assert n == 16
    # only the low nibble is a code
    assert np.array_equal(e2m1_to_f32(np.arange(256, dtype=np.uint8)), np.tile(got, 16))


def test_nvfp4_unpack_low_nibble_first():
    packed = np.array([[0x21, 0x0F, 0xA5]], np.uint8)
    assert np.array_equal(nvfp4_unpack(packed), np.array([[1, 2, 15, 0, 5, 10]], np.uint8))


def test_nvfp4_dequant_exact_products_on_the_bf16_grid():
    """Every (e2m1 code, finite e4m3 scale) product is exact in FP32 and a
    bf16 value; scale j covers the 16 elements 16j .. 16j+15 of its row."""
    codes = np.arange(16, dtype=np.uint8)
    scales = np.array([c for c in range(256) if np.isfinite(E4M3_TABLE[c])], np.uint8)
    for sc in scales:
        packed = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)[None, :]   # one block of 16
        w = nvfp4_dequant(packed, np.array([[sc]], np.uint8))[0]
        want = e2m1_to_f32(codes).astype(np.float64) * float(E4M3_TABLE[sc])
        assert np.array_equal(w.astype(np.float64), want)
        assert np.array_equal(bf16_round(w), w)
    # block mapping: three blocks with scales 1, 2, 0.5 on the same codes
    packed = np.tile((codes[0::2] | (codes[1::2] << 4)).astype(np.uint8), 3)[None, :]
    s = f32_to_e4m3(np.array([[1.0, 2.0, 0.5]], np.float32))
    w = nvfp4_dequant(packed, s)[0]
    base = e2m1_to_f32(codes)
    assert np.array_equal(w, np.concatenate([base, 2 * base, 0.5 * base]).astype(np.float32))
