"""Pins of the oracle's format conversions against the format definitions and
independent library routines (no GPU).

E2M1 / E4M3 are the element and block-scale formats of NVFP4 as the pages use
them (fast-path PR: "the FP4/E4M3 casts and their exact decodes"); FP16 is the
candidate-error precision of the FP16-error mode and, with BF16, an output
type of the fused quantize-dequantize (Megatron fused-QDQ PR, numerical
contract).
"""
import os
from fractions import Fraction as F

import numpy as np
import pytest
import torch

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _read_table(name):
    rows = []
    for line in open(os.path.join(GOLD, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        c, v = line.split()
        rows.append((int(c, 16), float(v)))
    return rows


def _same(a, b):
    if np.isnan(a) and np.isnan(b):
        return True
    return a == b and np.signbit(a) == np.signbit(b)


def test_e2m1_decode_table(orc):
    rows = _read_table("e2m1_decode.txt")
    assert len(rows) == 16
    for code, val in rows:
        assert _same(orc.e2m1_value(code), val), (code, val)


def test_e4m3_decode_special_codes(orc):
    for code, val in _read_table("e4m3_special.txt"):
        assert _same(orc.e4m3_value(code), val), (hex(code), val)


def test_e4m3_decode_all_codes_vs_torch(orc):
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).float()
    for code in range(256):
        assert _same(orc.e4m3_value(code), ref[code].item()), hex(code)


def _bf16_patterns_upto(limit):
    """Every float32 whose low 16 bits are zero and |v| <= limit, both signs."""
    hi = np.arange(0, 0x8000, dtype=np.uint32) << 16
    v = hi.view(np.float32)
    v = v[np.isfinite(v) & (np.abs(v) <= limit)]
    return np.concatenate([v, -v])


def _around(points, ulps=3):
    p = np.asarray(points, np.float32)
    out = [p]
    up, dn = p.copy(), p.copy()
    for _ in range(ulps):
        up = np.nextafter(up, np.float32(np.inf))
        dn = np.nextafter(dn, np.float32(-np.inf))
        out += [up, dn]
    return np.concatenate(out)


def test_e4m3_encode_vs_torch_in_range(orc):
    rng = np.random.default_rng(1)
    mags = np.array([orc.e4m3_value(c) for c in range(127)], np.float64)
    mids = (mags[:-1] + mags[1:]) / 2
    pts = np.concatenate([
        _bf16_patterns_upto(464.0),
        _around(np.concatenate([mids, -mids, mags, -mags]).astype(np.float32)),
        rng.uniform(-464, 464, 200000).astype(np.float32),
        (rng.standard_normal(200000) * 2.0 ** rng.integers(-20, 8, 200000)).astype(np.float32),
        np.array([0.0, -0.0, 464.0, -464.0, 2.0 ** -10, 2.0 ** -11, 1e-30, -1e-30], np.float32),
    ]).astype(np.float32)
    pts = pts[np.abs(pts) <= 464.0]
    got = orc.e4m3_encode(pts)
    ref = torch.from_numpy(pts).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(pts[i]), hex(got[i]), hex(ref[i])) for i in bad[:10]]


def test_e4m3_encode_saturates_and_nan(orc):
    big = np.array([464.001, 480.0, 1e6, 3e38, np.inf], np.float32)
    assert (orc.e4m3_encode(big) == 0x7E).all()
    assert (orc.e4m3_encode(-big) == 0xFE).all()
    assert orc.e4m3_encode(np.array([np.nan], np.float32))[0] & 0x7F == 0x7F


def _brute_e2m1(y):
    """Nearest magnitude on the E2M1 grid by exhaustive search, ties to the
    even code; sign kept; values past 6 take 6 (the largest finite code)."""
    if np.isnan(y):
        return None
    mags = [F(0), F(1, 2), F(1), F(3, 2), F(2), F(3), F(4), F(6)]
    a = F(abs(float(y))) if np.isfinite(y) else F(10 ** 9)
    best, bd = 0, abs(a)
    for c in range(1, 8):
        d = abs(a - mags[c])
        if d < bd or (d == bd and c % 2 == 0):
            best, bd = c, d
    return best | (8 if np.signbit(y) else 0)


def test_e2m1_encode_vs_bruteforce(orc):
    rng = np.random.default_rng(2)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    pts = np.concatenate([
        _bf16_patterns_upto(8.0),
        _around(np.concatenate([mids, -mids])),
        rng.uniform(-8, 8, 20000).astype(np.float32),
        np.array([0.0, -0.0, np.inf, -np.inf, 7.0, 1e30, -1e30, 1e-45, -1e-45], np.float32),
    ]).astype(np.float32)
    got = orc.e2m1_encode(pts)
    for y, g in zip(pts, got):
        assert g == _brute_e2m1(y), (float(y), hex(g))


def test_e2m1_encode_nan_is_plus_six(orc):
    # Fast-path PR: NaN inputs encode to +6 codes.
    nans = np.array([np.nan, -np.nan], np.float32)
    nans[1] = np.float32(np.copysign(np.nan, -1.0))
    assert (orc.e2m1_encode(nans) == 0x7).all()


def _sample_f32(rng, n):
    bits = rng.integers(0, 2 ** 32, n, dtype=np.uint64).astype(np.uint32)
    return bits.view(np.float32)


def test_f16_round_vs_numpy(orc):
    rng = np.random.default_rng(3)
    h = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float32)
    with np.errstate(over="ignore"):
        nxt = np.nextafter(h.astype(np.float16), np.float16(np.inf)).astype(np.float32)
    mids = ((h.astype(np.float64) + nxt.astype(np.float64)) / 2).astype(np.float32)
    pts = np.concatenate([
        _sample_f32(rng, 2_000_000), _around(mids, 2), -_around(mids, 2),
        np.array([65504, 65519.99, 65520, 65536, 1e5, 2.0 ** -25, 2.0 ** -24, 3 * 2.0 ** -26,
                  np.inf, -np.inf, 0.0, -0.0], np.float32)]).astype(np.float32)
    pts = pts[~np.isnan(pts)]
    got = orc.f16_round(pts)
    with np.errstate(over="ignore"):
        ref = pts.astype(np.float16).astype(np.float32)
        ref_bits = pts.astype(np.float16).view(np.uint16)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    assert np.array_equal(orc.f16_bits(pts), ref_bits)


def test_bf16_round_vs_torch(orc):
    rng = np.random.default_rng(4)
    hi = np.arange(0, 0x7F80, dtype=np.uint32) << 16
    lo = hi + (1 << 15)  # exact midpoints between adjacent bf16 values
    pts = np.concatenate([
        _sample_f32(rng, 2_000_000), _around(lo.view(np.float32), 2),
        -_around(lo.view(np.float32), 2),
        np.array([3.4e38, np.finfo(np.float32).max, np.inf, -np.inf, 0.0, -0.0, 1e-40],
                 np.float32)]).astype(np.float32)
    pts = pts[~np.isnan(pts)]
    got = orc.bf16_round(pts)
    ref = torch.from_numpy(pts).to(torch.bfloat16).float().numpy()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    ref_bits = torch.from_numpy(pts).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(orc.bf16_bits(pts), ref_bits)
