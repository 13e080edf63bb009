"""The CPU oracle run over row slices of a large input on every host core.

Test infrastructure, like the oracle itself.  Given the global amax, rows
(and 16-row tile bands for 16x16 blocks) are independent: each block's
codes, scale and decoded values depend only on its own elements and on the
global encode scale S of its row.  So the oracle is called once per
contiguous slice of rows, each call on its own thread (ctypes releases the
GIL while the C code runs), and the slices' outputs are stitched back in
row order.  Nothing is reordered inside a call; a slice is exactly the
oracle's own computation on those rows.

The global amax of a tensor is the NaN-dropping maximum of |x| with initial
+0; the maximum of the slices' maxima is the same number (max is
associative and commutative, and no slice maximum is NaN).
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

import oracle


def threads():
    return max(1, min(64, os.cpu_count() or 1))


def _slices(rows, align, parts):
    units = rows // align
    parts = max(1, min(parts, units))
    cuts = [(units * i // parts) * align for i in range(parts + 1)]
    cuts[-1] = rows
    return [(cuts[i], cuts[i + 1]) for i in range(parts) if cuts[i + 1] > cuts[i]]


def _run(fn, rows, align, per_thread=4):
    sl = _slices(rows, align, threads() * per_thread)
    with ThreadPoolExecutor(threads()) as ex:
        for f in [ex.submit(fn, lo, hi) for lo, hi in sl]:
            f.result()


def amax_tensor(x):
    """Per-tensor amax of float32 [R, C] (all cores)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    R = x.shape[0]
    part = {}

    def work(lo, hi):
        part[lo] = float(oracle.amax_tensor(x[lo:hi])[0])

    _run(work, R, 1, per_thread=1)
    return np.array([max([0.0] + list(part.values()))], np.float32)


def amax_rows(x):
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape[0], np.float32)

    def work(lo, hi):
        out[lo:hi] = oracle.amax_rows(x[lo:hi])

    _run(work, x.shape[0], 1)
    return out


def quantize(x, cfg, amax):
    """oracle.quantize with the amax given ([1] per tensor, [R] per row);
    returns (codes, scales)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    R, C = x.shape
    assert cfg.amax_is_input
    b = 16 if cfg.block16x16 else 1
    amax = np.ascontiguousarray(amax, dtype=np.float32).ravel()
    codes = np.empty((R, C // 2), np.uint8)
    scales = np.empty((R // b, C // 16), np.uint8)

    def work(lo, hi):
        a = amax[lo:hi] if cfg.row_scaled else amax
        c, s, _ = oracle.quantize(x[lo:hi], cfg, amax=a)
        codes[lo:hi] = c
        scales[lo // b:hi // b] = s

    _run(work, R, b)
    return codes, scales


def qdq(x, cfg, out_dtype, amax):
    """oracle.qdq with the amax given; returns the output bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    R, C = x.shape
    assert cfg.amax_is_input
    amax = np.ascontiguousarray(amax, dtype=np.float32).ravel()
    out = np.empty((R, C), np.float32 if out_dtype == "f32" else np.uint16)

    def work(lo, hi):
        a = amax[lo:hi] if cfg.row_scaled else amax
        out[lo:hi] = oracle.qdq(x[lo:hi], cfg, out_dtype, amax=a)[0]

    _run(work, R, 1)
    return out


def dequantize(codes, scales, amax, cfg, out_dtype):
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    R, C2 = codes.shape
    b = 16 if cfg.block16x16 else 1
    amax = np.ascontiguousarray(amax, dtype=np.float32).ravel()
    out = np.empty((R, 2 * C2), np.float32 if out_dtype == "f32" else np.uint16)

    def work(lo, hi):
        a = amax[lo:hi] if cfg.row_scaled else amax
        out[lo:hi] = oracle.dequantize(codes[lo:hi], scales[lo // b:hi // b], a, cfg, out_dtype)

    _run(work, R, b)
    return out
