"""Exact-rational model of one block of the four-over-six quantizer.

An independent pin for the oracle, not a second copy of it: every quantity is
a Fraction, grids come from the format definitions (E2M1 from the OCP MX
table, E4M3 from torch's float8_e4m3fn decode), rounding to a grid is a
brute-force argmin with the even-code tie-break, and sums are exact.  The model
applies only where binary32 arithmetic is exact, so it asserts that every
intermediate is representable and flags elements whose encode could be decided
by the rounding of an inexact common scale (those blocks are skipped).

Method (grouped-GEMM PR, first commit; fast-path PR description): block amax
maps to 6 (standard) or to 4 under a 1.5x scale; both candidates are encoded,
decoded and compared by MAE or MSE; the lower error is stored, ties keep
map-to-6.
"""
from fractions import Fraction as F

import numpy as np
import torch

E2M1_MAG = [F(0), F(1, 2), F(1), F(3, 2), F(2), F(3), F(4), F(6)]


def _e4m3_mags():
    codes = torch.arange(0, 127, dtype=torch.uint8)
    vals = codes.view(torch.float8_e4m3fn).float().tolist()
    return [F(v) for v in vals]


E4M3_MAG = _e4m3_mags()


def f32_exact(v: F) -> bool:
    return F(float(np.float32(float(v)))) == v and abs(v) <= F(float(np.finfo(np.float32).max))


def nearest(value: F, grid):
    """Brute-force nearest grid index; equal distances go to the even index."""
    best = None
    bestd = None
    for i, g in enumerate(grid):
        d = abs(value - g)
        if bestd is None or d < bestd or (d == bestd and i % 2 == 0 and best % 2 == 1):
            best, bestd = i, d
    return best


def _near_midpoint(y: F, rel=F(1, 2**20)):
    a = abs(y)
    for lo, hi in zip(E2M1_MAG[:-1], E2M1_MAG[1:]):
        mid = (lo + hi) / 2
        if abs(a - mid) <= rel * mid:
            return True
    return False


class Inexact(Exception):
    pass


def candidate(rows, S: F, k: int, mse: bool, f16: bool):
    """rows: list of lists of 16 Fractions.  Returns dict with codes (list of
    lists of 4-bit codes), sc (E4M3 code), err (Fraction), ambiguous (bool)."""
    c = candidate_terms(rows, S, k, mse, f16)
    partials = c.pop("terms")
    # Every partial sum of the nonnegative dyadic terms is a multiple of the
    # finest grain and at most the total; below 2^24 grains all are exact in
    # binary32, so the reduction order cannot matter for these blocks.
    allterms = [t for ts in partials for t in ts]
    grain = max((t.denominator for t in allterms), default=1)
    if grain & (grain - 1):
        raise Inexact("non-dyadic term")
    total = sum(allterms, F(0))
    if total * grain >= 2**24:
        raise Inexact("error sum not exact")
    c["err"] = total
    return c


def candidate_terms(rows, S: F, k: int, mse: bool, f16: bool):
    """Like candidate() but stops before the reduction: returns codes, sc,
    ambiguous and terms (per row, the 16 exact error terms, each exactly a
    binary32 value), for blocks whose per-element arithmetic is exact even
    when their sum is not."""
    a_b = max(abs(v) for r in rows for v in r)
    t = a_b * S
    s = t / k
    if not (f32_exact(t) and f32_exact(s)):
        raise Inexact("scale product not exact")
    sc = nearest(s, E4M3_MAG)
    sigma = E4M3_MAG[sc]
    if sigma == 0:
        r_exact, d = F(0), F(0)
    else:
        r_exact, d = S / sigma, sigma / S
    if not f32_exact(d):
        raise Inexact("decode scale not exact")
    r_is_exact = f32_exact(r_exact)
    ambiguous = False
    codes, partials = [], []
    for row in rows:
        crow, terms = [], []
        for x in row:
            y = x * r_exact
            if not r_is_exact and _near_midpoint(y):
                ambiguous = True
            q = nearest(abs(y), E2M1_MAG)
            neg = y < 0 or (y == 0 and x < 0)
            code = q | (8 if neg else 0)
            crow.append(code)
            deq = E2M1_MAG[q] * d * (-1 if code & 8 else 1)
            if f16:
                deq = F(float(np.float16(float(deq))))
            e = x - deq
            term = e * e if mse else abs(e)
            if not (f32_exact(deq) and f32_exact(e) and f32_exact(term)):
                raise Inexact("element arithmetic not exact")
            terms.append(term)
        codes.append(crow)
        partials.append(terms)
    return {"codes": codes, "sc": sc, "terms": partials, "ambiguous": ambiguous}


def block(rows, S: F, four_over_six=True, mse=True, f16=False):
    """Selected candidate of one block under the method: map-to-4 only when
    its error is strictly lower."""
    c6 = candidate(rows, S, 6, mse, f16)
    if not four_over_six:
        return c6, c6, None
    c4 = candidate(rows, S, 4, mse, f16)
    sel = c4 if c4["err"] < c6["err"] else c6
    return sel, c6, c4


def pack_row(codes16):
    return bytes((codes16[2 * j] | (codes16[2 * j + 1] << 4)) for j in range(8))
