"""Pins of the oracle's method steps (no GPU).

Each test checks the oracle against something other than itself: closed-form
values, the exact-rational block model in ``exact_model.py`` (brute-force
grids, exact sums), hand-derived golden fixtures under ``golden/``, and
invariants the pages state (grouped == per-group, NaN -> +6, ...).
"""
import os
import struct
from fractions import Fraction as F

import numpy as np
import pytest
import torch

import exact_model as em
import workloads

GOLD = os.path.join(os.path.dirname(__file__), "golden")
FLT_MAX = float(np.finfo(np.float32).max)


def _numbers(name):
    out = []
    for line in open(os.path.join(GOLD, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            out.append(line.split())
    return out


# ---------------------------------------------------------------- global scale
@pytest.mark.parametrize("A,bound,S", [
    (5.25, 448, 512.0), (2688.0, 448, 1.0), (1536.0, 256, 1.0), (6.0, 256, 256.0),
    (7.0, 448, 384.0), (3.0, 448, 896.0), (0.75, 256, 2048.0),
])
def test_global_scale_closed_forms(orc, A, bound, S):
    # FP32 global scale that maps the amax to 6 x the E4M3 bound (reading R2).
    assert orc.global_scale(A, bound) == S


@pytest.mark.parametrize("A", [0.0, -0.0, -1.0, float("inf"), float("nan")])
def test_global_scale_degenerate_amax(orc, A):
    assert orc.global_scale(A, 448) == 1.0


def test_global_scale_overflow_clamps(orc):
    assert orc.global_scale(1e-45, 448) == FLT_MAX


# ---------------------------------------------------------------- golden cases
def test_pack_order_golden(orc):
    vals, codes_hex, scale_hex = _numbers("pack_order.txt")
    x = np.array([float(v) for v in vals], np.float32).reshape(1, 16)
    cfg = orc.Config(four_over_six=False, amax_is_input=True, bound=448)
    codes, scales, _ = orc.quantize(x, cfg, amax=[2688.0])
    assert bytes(codes.ravel()) == bytes(int(h, 16) for h in codes_hex)
    assert scales.ravel()[0] == int(scale_hex[0], 16)


def test_tree_order_golden(orc):
    (bits_hex,) = _numbers("tree_order.txt")[0]
    x = np.full((1, 16), np.float32(0.5) + np.float32(2.0 ** -24), np.float32)
    x[0, 0] = 5.0
    x[0, 15] = 6.0
    cfg = orc.Config(four_over_six=True, mse=False, err_f16=False, amax_is_input=True)
    _, _, _, e6, _ = orc.quantize(x, cfg, amax=[2688.0], with_errors=True)
    assert struct.pack(">f", float(e6[0, 0])).hex().upper() == bits_hex


def test_seq_order_golden(orc):
    (bits_hex,) = _numbers("seq_order.txt")[0]
    x = np.full((1, 16), np.float32(0.5) + np.float32(2.0 ** -24), np.float32)
    x[0, 0] = 5.0
    x[0, 15] = 6.0
    cfg = orc.Config(four_over_six=True, mse=False, err_f16=False, amax_is_input=True,
                     seq_order=True)
    _, _, _, e6, _ = orc.quantize(x, cfg, amax=[2688.0], with_errors=True)
    assert struct.pack(">f", float(e6[0, 0])).hex().upper() == bits_hex


def _fold_seq(terms):
    acc = np.float32(float(terms[0]))
    for t in terms[1:]:
        acc = np.float32(acc + np.float32(float(t)))
    return acc


def _fold_tree(terms):
    t = [np.float32(float(v)) for v in terms]
    w = 8
    while w >= 1:
        for i in range(w):
            t[i] = np.float32(t[i] + t[i + w])
        w //= 2
    return t[0]


@pytest.mark.parametrize("mse", [False, True])
def test_seq_order_against_binary32_folds(orc, mse):
    """Blocks whose element errors are exact but whose sums are not: the
    exact-rational model gives the 16 terms; numpy binary32 additions fold
    them in element order (and, as a control, in the pinned tree order).  The
    oracle's sequential-order errors, codes and scales must follow the
    sequential fold."""
    rng = np.random.default_rng(53 + mse)
    grid = [F(1, 2), F(1), F(3, 2), F(2), F(3), F(4)]
    rows, want = [], []
    differs = 0
    for _ in range(4000):
        if len(rows) == 64:
            break
        row = []
        for _ in range(16):
            g = grid[int(rng.integers(len(grid)))]
            if mse:  # errors of at most 12 significant bits, so that e*e is exact
                step = F(1, 2 ** 13)
            else:    # errors down to one unit in the last place of x
                step = F(2) ** (int(np.floor(np.log2(float(g)))) - 23)
            v = g + int(rng.integers(-40, 41)) * step * 2 ** int(rng.integers(0, 6))
            row.append(-v if rng.random() < 0.5 else v)
        # one element on a grid midpoint (a large error term next to the small
        # ones, so that sums need more than 24 bits) and the block amax 6
        i5, i6 = rng.choice(16, 2, replace=False)
        row[int(i5)] = F(5) if rng.random() < 0.5 else F(-5)
        row[int(i6)] = F(6)
        try:
            c6 = em.candidate_terms([row], F(1), 6, mse, False)
            c4 = em.candidate_terms([row], F(1), 4, mse, False)
        except em.Inexact:
            continue
        if c6["ambiguous"] or c4["ambiguous"]:
            continue
        e6, e4 = _fold_seq(c6["terms"][0]), _fold_seq(c4["terms"][0])
        differs += int(e6 != _fold_tree(c6["terms"][0]) or e4 != _fold_tree(c4["terms"][0]))
        sel = c4 if e4 < e6 else c6
        rows.append(row)
        want.append((e6, e4, sel))
    assert len(rows) == 64
    assert differs >= 8  # the draw really separates the two orders
    x = np.array([[float(v) for v in r] for r in rows], np.float32)
    cfg = orc.Config(four_over_six=True, mse=mse, amax_is_input=True, seq_order=True)
    codes, scales, _, e6, e4 = orc.quantize(x, cfg, amax=[2688.0], with_errors=True)
    for i, (w6, w4, sel) in enumerate(want):
        assert e6[i, 0] == w6 and e4[i, 0] == w4, i
        assert bytes(codes[i]) == em.pack_row(sel["codes"][0]), i
        assert scales[i, 0] == sel["sc"], i


def test_seq_order_rejects_16x16(orc):
    x = np.zeros((16, 16), np.float32)
    with pytest.raises(ValueError):
        orc.quantize(x, orc.Config(block16x16=True, seq_order=True))


# ------------------------------------------------------- exact-rational model
NICE_SIGMA = [F(1), F(9, 8), F(5, 4), F(11, 8), F(3, 2), F(13, 8), F(7, 4), F(15, 8)]


def _draw_block(rng, S, nrows, mse, f16, four, tries=200):
    """Rows of 16 dyadic values whose block amax maps to 6 under an E4M3
    scale, drawn until the exact model applies and no element sits on a
    rounding decision of an inexact common scale."""
    for _ in range(tries):
        sig = NICE_SIGMA[rng.integers(len(NICE_SIGMA))] * F(2) ** int(rng.integers(-3, 4))
        a_b = 6 * sig / S
        grain = a_b / 32
        rows = []
        for _r in range(nrows):
            n = rng.integers(-32, 33, 16)
            rows.append([int(v) * grain for v in n])
        r0, c0 = int(rng.integers(nrows)), int(rng.integers(16))
        rows[r0][c0] = a_b if rng.random() < 0.5 else -a_b
        for r in rows:
            for j in range(16):
                if abs(r[j]) > a_b:
                    r[j] = a_b
        try:
            sel, c6, c4 = em.block(rows, S, four_over_six=four, mse=mse, f16=f16)
        except em.Inexact:
            continue
        if c6["ambiguous"] or (c4 is not None and c4["ambiguous"]):
            continue
        return rows, sel, c6, c4
    raise RuntimeError("could not draw an exact block")


def _to_f32(rows):
    return np.array([[float(v) for v in r] for r in rows], np.float32)


@pytest.mark.parametrize("four,mse,f16", [(False, True, False), (True, False, False),
                                          (True, True, False), (True, False, True),
                                          (True, True, True)])
@pytest.mark.parametrize("bound", [448, 256])
def test_exact_model_1x16_tensor_scale(orc, four, mse, f16, bound):
    rng = np.random.default_rng(100 + 7 * bound + 3 * four + 2 * mse + f16)
    S = F(2) ** int(rng.integers(-2, 6))
    A = F(6 * bound) / S
    blocks = [_draw_block(rng, S, 1, mse, f16, four) for _ in range(48)]
    x = np.concatenate([_to_f32(b[0]) for b in blocks])
    cfg = orc.Config(four_over_six=four, mse=mse, err_f16=f16, bound=bound, amax_is_input=True)
    codes, scales, _, e6, e4 = orc.quantize(x, cfg, amax=[float(A)], with_errors=True)
    for i, (_, sel, c6, c4) in enumerate(blocks):
        assert bytes(codes[i]) == em.pack_row(sel["codes"][0]), i
        assert scales[i, 0] == sel["sc"], i
        assert F(float(e6[i, 0])) == c6["err"], i
        if four:
            assert F(float(e4[i, 0])) == c4["err"], i


@pytest.mark.parametrize("mse,f16", [(True, False), (False, False), (True, True)])
def test_exact_model_1x16_row_scale(orc, mse, f16):
    rng = np.random.default_rng(7 + 2 * mse + f16)
    xs, amax, exp = [], [], []
    for _ in range(40):
        S = F(2) ** int(rng.integers(-4, 8))
        rows, sel, _, _ = _draw_block(rng, S, 1, mse, f16, True)
        xs.append(_to_f32(rows))
        amax.append(float(F(6 * 448) / S))
        exp.append(sel)
    x = np.concatenate(xs)
    cfg = orc.Config(four_over_six=True, mse=mse, err_f16=f16, row_scaled=True,
                     amax_is_input=True)
    codes, scales, _ = orc.quantize(x, cfg, amax=amax)
    for i, sel in enumerate(exp):
        assert bytes(codes[i]) == em.pack_row(sel["codes"][0])
        assert scales[i, 0] == sel["sc"]


def _draw_tile(rng, S, mse, f16):
    """16x16 tile with a power-of-two map-to-6 scale (exact common scales for
    map-to-6, so its ties are real ties) on a grain of amax/24; the two
    multipliers whose map-to-4 value would sit on an E2M1 midpoint (15, 21)
    are left out, so no element depends on the rounding of 2/3."""
    allowed = np.array([n for n in range(-24, 25) if abs(n) not in (15, 21)])
    for _ in range(100):
        sig = F(2) ** int(rng.integers(-2, 3))
        a_b = 6 * sig / S
        grain = a_b / 24
        rows = [[int(v) * grain for v in rng.choice(allowed, 16)] for _ in range(16)]
        rows[int(rng.integers(16))][int(rng.integers(16))] = a_b
        sel, c6, c4 = em.block(rows, S, four_over_six=True, mse=mse, f16=f16)
        if not (c6["ambiguous"] or c4["ambiguous"]):
            return rows, sel, c6, c4
    raise RuntimeError("could not draw an exact tile")


@pytest.mark.parametrize("mse,f16", [(True, False), (False, False), (False, True)])
def test_exact_model_16x16_tiles(orc, mse, f16):
    rng = np.random.default_rng(31 + 2 * mse + f16)
    S = F(2) ** 3
    tiles = [_draw_tile(rng, S, mse, f16) for _ in range(6)]
    # lay the tiles side by side: one band of 16 rows, 6 tiles wide
    x = np.concatenate([_to_f32(t[0]) for t in tiles], axis=1)
    cfg = orc.Config(block16x16=True, four_over_six=True, mse=mse, err_f16=f16,
                     amax_is_input=True)
    codes, scales, _, e6, e4 = orc.quantize(x, cfg, amax=[float(F(2688) / S)], with_errors=True)
    for j, (_, sel, c6, c4) in enumerate(tiles):
        assert scales[0, j] == sel["sc"]
        assert F(float(e6[0, j])) == c6["err"]
        assert F(float(e4[0, j])) == c4["err"]
        for r in range(16):
            assert bytes(codes[r, 8 * j:8 * j + 8]) == em.pack_row(sel["codes"][r]), (j, r)
    assert len({t[0][0][0] for t in tiles}) > 1


def test_exact_model_fp16_error_mode_changes_errors(orc):
    """Tiny magnitudes: the candidate decode falls in FP16's subnormal range,
    so the FP16-error mode must differ from the exact mode and match the
    exact model's FP16 rounding (numpy binary16)."""
    rng = np.random.default_rng(5)
    S = F(2) ** 27
    differs = 0
    for _ in range(20):
        rows, sel, c6, c4 = _draw_block(rng, S, 1, True, True, True)
        x = _to_f32(rows)
        cfg16 = orc.Config(mse=True, err_f16=True, amax_is_input=True)
        cfgex = orc.Config(mse=True, err_f16=False, amax_is_input=True)
        A = [float(F(2688) / S)]
        _, _, _, e6, e4 = orc.quantize(x, cfg16, amax=A, with_errors=True)
        _, _, _, x6, x4 = orc.quantize(x, cfgex, amax=A, with_errors=True)
        assert F(float(e6[0, 0])) == c6["err"] and F(float(e4[0, 0])) == c4["err"]
        differs += int(e6[0, 0] != x6[0, 0] or e4[0, 0] != x4[0, 0])
    assert differs > 0


# ------------------------------------------------------------- round trips
def test_round_trip_map_to_6_grid(orc):
    """Blocks already on the map-to-6 grid (S = 2^k, scale 2^j): zero error,
    codes equal the grid codes, dequantize returns the input bits."""
    rng = np.random.default_rng(11)
    mags = np.array([0, .5, 1, 1.5, 2, 3, 4, 6])
    k = 6
    S = 2.0 ** k
    blocks = []
    for _ in range(64):
        j = int(rng.integers(-3, 5))
        v = rng.choice(mags, 16) * rng.choice([-1, 1], 16)
        v[rng.integers(16)] = 6.0
        blocks.append(v * 2.0 ** j / S)
    x = np.array(blocks, np.float32)
    cfg = orc.Config(four_over_six=True, mse=True, amax_is_input=True)
    A = [2688.0 / S]
    codes, scales, _, e6, e4 = orc.quantize(x, cfg, amax=A, with_errors=True)
    assert (e6 == 0).all()
    back = orc.dequantize(codes, scales, A, cfg, "f32")
    assert np.array_equal(back.view(np.uint32), x.view(np.uint32))
    bf = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    assert np.array_equal(bf, x)  # these values are exact in bf16 too
    qb, _ = orc.qdq(x, cfg, "bf16", amax=A)
    assert np.array_equal(qb, torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy()
                          .view(np.uint16))


def test_round_trip_map_to_4_grid_selects_4(orc):
    """Blocks on the 1.5x-scale map-to-4 grid containing 4 and a value the
    map-to-6 grid cannot hold: map-to-4 has zero error and is selected."""
    rng = np.random.default_rng(12)
    mags = np.array([0, .5, 1, 1.5, 2, 3, 4])
    S = 2.0 ** 5
    blocks, js = [], []
    for _ in range(64):
        j = int(rng.integers(-3, 4))
        v = rng.choice(mags, 16) * rng.choice([-1, 1], 16)
        v[0] = 4.0
        v[1] = 0.5  # 1.5 * 0.5 = 0.75 is off the map-to-6 grid
        blocks.append(v * 1.5 * 2.0 ** j / S)
        js.append(j)
    x = np.array(blocks, np.float32)
    A = [2688.0 / S]
    for mse in (False, True):
        cfg = orc.Config(four_over_six=True, mse=mse, amax_is_input=True)
        codes, scales, _, e6, e4 = orc.quantize(x, cfg, amax=A, with_errors=True)
        assert (e4 == 0).all() and (e6 > 0).all()
        for i, j in enumerate(js):
            assert orc.e4m3_value(int(scales[i, 0])) == 1.5 * 2.0 ** j
        back = orc.dequantize(codes, scales, A, cfg, "f32")
        assert np.array_equal(back.view(np.uint32), x.view(np.uint32))


# ------------------------------------------------------------- special blocks
def test_zero_blocks(orc):
    x = np.zeros((3, 16), np.float32)
    x[1] = -0.0
    x[2, ::2] = -0.0
    cfg = orc.Config(amax_is_input=True)
    codes, scales, _ = orc.quantize(x, cfg, amax=[1.0])
    assert (scales == 0).all()
    assert (codes[0] == 0x00).all() and (codes[1] == 0x88).all() and (codes[2] == 0x08).all()


def test_tiny_block_underflows_scale(orc):
    # S = 1, block amax 1e-7: 1e-7 / 6 is far below half the smallest E4M3
    # subnormal (2^-10), so both candidate scales are zero.
    x = np.array([[1e-7, -1e-7] * 8], np.float32)
    cfg = orc.Config(amax_is_input=True)
    codes, scales, _ = orc.quantize(x, cfg, amax=[2688.0])
    assert scales[0, 0] == 0
    assert (codes[0] == 0x80).all()


def test_nan_element(orc):
    # Fast-path PR: NaN-dropping block amax, NaN encodes to +6; the errors of
    # both candidates are NaN so the block keeps map-to-6.
    x = np.array([[6.0, np.nan] + [1.0] * 14], np.float32)
    cfg = orc.Config(amax_is_input=True)
    codes, scales, _, e6, e4 = orc.quantize(x, cfg, amax=[2688.0], with_errors=True)
    assert scales[0, 0] == 0x38  # block amax 6 -> map-to-6 scale 1.0
    assert codes[0, 0] == (0x7 | (0x7 << 4))  # 6 -> code 7; NaN -> code 7
    assert np.isnan(e6[0, 0]) and np.isnan(e4[0, 0])


def test_all_nan_block_has_zero_amax(orc):
    x = np.full((1, 16), np.nan, np.float32)
    cfg = orc.Config(amax_is_input=False)
    codes, scales, amax = orc.quantize(x, cfg)
    assert amax[0] == 0.0 and scales[0, 0] == 0 and (codes == 0x77).all()


def test_inf_element(orc):
    # Tensor amax Inf -> S = 1 (R2); block amax Inf -> scale saturates to 448
    # (R4); Inf encodes to 6; both errors are Inf, map-to-6 is kept.
    x = np.array([[np.inf] + [1.0] * 15, [2.0] * 16], np.float32)
    cfg = orc.Config(amax_is_input=False)
    codes, scales, amax = orc.quantize(x, cfg)
    assert np.isinf(amax[0])
    assert scales[0, 0] == 0x7E
    assert codes[0, 0] & 0xF == 0x7


# ------------------------------------------------------------- invariants
def _acts(seed, rows=64, cols=256):
    xs = [workloads.activation(rows, cols, f, seed=seed) for f in workloads.FAMILIES]
    return [x.float().numpy() for x in xs]


@pytest.mark.parametrize("bound", [448, 256])
@pytest.mark.parametrize("mse,f16", [(True, False), (False, False), (True, True), (False, True)])
def test_selected_error_not_above_other(orc, bound, mse, f16):
    for x in _acts(1):
        cfg = orc.Config(mse=mse, err_f16=f16, bound=bound)
        codes, scales, amax, e6, e4 = orc.quantize(x, cfg, with_errors=True)
        std, sstd, _ = orc.quantize(x, orc.Config(four_over_six=False, bound=bound))
        switched = (scales != sstd)
        # a block differs from standard only when map-to-4 won strictly
        same_codes = (codes.reshape(x.shape[0], -1, 8) == std.reshape(x.shape[0], -1, 8)).all(-1)
        changed = switched | ~same_codes
        assert (e4[changed] < e6[changed]).all()
        # an unchanged block kept map-to-6, so map-to-4 was not strictly better
        assert not (e4[~changed] < e6[~changed]).any()


def test_standard_equals_map_to_6_candidate(orc):
    for x in _acts(2):
        c4o6, s4o6, _, e6, e4 = orc.quantize(x, orc.Config(), with_errors=True)
        cst, sst, _ = orc.quantize(x, orc.Config(four_over_six=False))
        kept6 = ~(e4 < e6)
        rows_b = np.repeat(kept6, 8, axis=1)
        assert np.array_equal(c4o6[rows_b], cst[rows_b])
        assert np.array_equal(s4o6[kept6], sst[kept6])


def test_row_scale_with_equal_rows_equals_tensor(orc):
    x = _acts(3)[0]
    A = orc.amax_tensor(x)
    ct, st, _ = orc.quantize(x, orc.Config(amax_is_input=True), amax=A)
    cr, sr, _ = orc.quantize(x, orc.Config(amax_is_input=True, row_scaled=True),
                             amax=np.repeat(A, x.shape[0]))
    assert np.array_equal(ct, cr) and np.array_equal(st, sr)


def test_amax_scopes(orc):
    x = _acts(4)[1]
    assert orc.amax_tensor(x)[0] == np.abs(x).max()
    assert np.array_equal(orc.amax_rows(x), np.abs(x).max(1))
    offs = np.array([10, 10, 40, 50], np.int32)
    ga = orc.amax_groups(x, offs)
    ref = [np.abs(x[0:10]).max(), 0.0, np.abs(x[10:40]).max(), np.abs(x[40:50]).max()]
    assert np.array_equal(ga, np.array(ref, np.float32))


@pytest.mark.parametrize("block16", [False, True])
def test_grouped_equals_per_group_calls(orc, block16):
    # Grouped PR: the whole packed tensor quantizes in one call, bitwise equal
    # to quantizing each group separately; rows past offs[-1] are zero-filled.
    rng = np.random.default_rng(9)
    x = np.concatenate(_acts(5, rows=64, cols=128))  # 256 rows
    mult = 16 if block16 else 1
    offs = np.array([32, 32, 96, 160, 208], np.int32) if block16 else \
        np.array([7, 7, 50, 51, 130, 201], np.int32)
    x = x * rng.uniform(0.1, 10, (x.shape[0], 1)).astype(np.float32)
    cfg = orc.Config(block16x16=block16, mse=True)
    codes, scales, ga = orc.quantize_grouped(x, offs, cfg)
    lo = 0
    for g, hi in enumerate(offs):
        if hi > lo:
            c, s, a = orc.quantize(x[lo:hi], orc.Config(block16x16=block16, mse=True))
            assert a[0] == ga[g]
            assert np.array_equal(codes[lo:hi], c)
            assert np.array_equal(scales[lo // mult:hi // mult], s)
        else:
            assert ga[g] == 0.0
        lo = hi
    assert (codes[offs[-1]:] == 0).all() and (scales[offs[-1] // mult:] == 0).all()


@pytest.mark.parametrize("out", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("four,mse,f16", [(False, True, False), (True, False, True),
                                          (True, True, False)])
def test_qdq_equals_dequantize_of_quantize(orc, out, four, mse, f16):
    for x in _acts(6):
        cfg = orc.Config(four_over_six=four, mse=mse, err_f16=f16)
        q, amax = orc.qdq(x, cfg, out)
        codes, scales, a2 = orc.quantize(x, cfg)
        assert a2[0] == amax[0]
        d = orc.dequantize(codes, scales, amax, cfg, out)
        assert np.array_equal(q.view(np.uint16 if out != "f32" else np.uint32),
                              d.view(np.uint16 if out != "f32" else np.uint32))


def test_16x16_identical_rows_equal_1x16(orc):
    """A tile whose 16 rows repeat one 1x16 block has the block's amax, the
    block's codes in every row, and 16x the row error (exact power-of-two
    tree), hence the same selection and scale."""
    base = _acts(8, rows=16, cols=256)[0][:1]
    x = np.repeat(base, 16, axis=0)
    A = [float(np.abs(base).max())]
    c1, s1, _ = orc.quantize(base, orc.Config(amax_is_input=True), amax=A)
    c16, s16, _ = orc.quantize(x, orc.Config(block16x16=True, amax_is_input=True), amax=A)
    assert np.array_equal(s16[0], s1[0])
    for r in range(16):
        assert np.array_equal(c16[r], c1[0])


def test_row_scaled_16x16_uses_first_row_amax(orc):
    x = _acts(10, rows=32, cols=64)[0]
    ra = orc.amax_rows(x)
    cfg = orc.Config(block16x16=True, row_scaled=True, amax_is_input=True)
    c1, s1, _ = orc.quantize(x, cfg, amax=ra)
    uni = np.repeat(ra[::16], 16)
    c2, s2, _ = orc.quantize(x, cfg, amax=uni)
    assert np.array_equal(c1, c2) and np.array_equal(s1, s2)


def test_bad_shapes_rejected(orc):
    with pytest.raises(ValueError):
        orc.quantize(np.zeros((2, 24), np.float32), orc.Config())
    with pytest.raises(ValueError):
        orc.quantize(np.zeros((8, 16), np.float32), orc.Config(block16x16=True))
    with pytest.raises(ValueError):
        orc.quantize(np.zeros((2, 16), np.float32), orc.Config(bound=300))


def test_scale_order_golden(orc):
    bits_hex, amax, code_hex = _numbers("scale_order.txt")[0]
    x = np.zeros((1, 16), np.float32)
    x[0, 0] = np.array([int(bits_hex, 16)], np.uint32).view(np.float32)[0]
    cfg = orc.Config(four_over_six=False, amax_is_input=True, bound=448)
    _, scales, _ = orc.quantize(x, cfg, amax=[float(amax)])
    assert scales[0, 0] == int(code_hex, 16)


# ---------------------------------------------------------------- column-wise operand
def test_colwise_is_the_quantization_of_each_column(orc):
    """Row c of the column-wise result equals the quantization of column c
    of x taken on its own as one row (same global amax given), and the
    scales follow the same blocks (16 consecutive rows)."""
    x = workloads.activation(64, 48, "F2", seed=9, dtype=torch.float32).numpy()
    A = orc.amax_tensor(x)
    cfg = orc.Config(four_over_six=True, mse=True, amax_is_input=True)
    ct, st, _ = orc.quantize_colwise(x, cfg, amax=A)
    assert ct.shape == (48, 32) and st.shape == (48, 4)
    for c in (0, 7, 47):
        cc, sc, _ = orc.quantize(x[:, c].reshape(1, 64).copy(), cfg, amax=A)
        assert np.array_equal(ct[c], cc[0]) and np.array_equal(st[c], sc[0])


def test_colwise_of_a_symmetric_matrix_is_the_rowwise_result(orc):
    a = workloads.activation(32, 32, "F1", seed=10, dtype=torch.float32).numpy()
    x = (a + a.T).astype(np.float32)
    cfg = orc.Config(four_over_six=True, mse=False, err_f16=True)
    assert all(np.array_equal(p, q) for p, q in zip(orc.quantize_colwise(x, cfg),
                                                      orc.quantize(x, cfg)))


# ---------------------------------------------------------------- tiled scale layout
def test_swizzled_scale_layout_offsets(orc):
    """Hand-placed bytes of a 200 x 9 scale matrix (2 tile rows, 3 tile
    columns after padding to 256 x 12) land where the layout puts them, the
    layout is a permutation, and the padding is zero."""
    s = np.zeros((200, 9), np.uint8)
    marks = {(0, 0): 0, (1, 0): 16, (31, 0): 496, (32, 0): 4, (96, 0): 12, (127, 3): 511,
             (0, 1): 1, (0, 4): 512, (5, 6): 512 + 5 * 16 + 2, (128, 0): 3 * 512,
             (199, 8): (3 + 2) * 512 + (71 % 32) * 16 + (71 // 32) * 4 + 0}
    for i, (rc, _) in enumerate(marks.items()):
        s[rc] = i + 1
    out = orc.swizzle_scales(s)
    assert out.size == 256 * 12
    for i, (rc, off) in enumerate(marks.items()):
        assert out[off] == i + 1, (rc, off)
    assert np.count_nonzero(out) == len(marks)
    full = np.arange(256 * 12, dtype=np.int64).reshape(256, 12)
    # a bijection on the padded matrix: every byte of a distinct-valued input appears once
    vals = (full % 251 + 1).astype(np.uint8)
    assert np.array_equal(np.sort(orc.swizzle_scales(vals)), np.sort(vals.ravel()))


def test_tile_uniform_count_hand_cases(orc):
    """The tile-uniform contract of 16x16 blocks with row-scaled amax
    (grouped PR): counts built by hand.  Equal rows give 0; one differing
    row, two differing rows in one tile, and +0 against -0 (bitwise reading)
    each add one tile."""
    a = np.ones(96, np.float32)
    assert orc.count_nonuniform_tiles(a) == 0
    a[17] = 2.0                      # tile 1
    assert orc.count_nonuniform_tiles(a) == 1
    a[40] = 3.0
    a[47] = 3.0                      # tile 2, two rows
    assert orc.count_nonuniform_tiles(a) == 2
    a[48:64] = 0.0
    a[63] = -0.0                     # tile 3: equal as floats, not as bits
    assert orc.count_nonuniform_tiles(a) == 3
    a[0] = 5.0                       # tile 0, first row differs from the rest
    assert orc.count_nonuniform_tiles(a) == 4
    assert orc.count_nonuniform_tiles(np.zeros(0, np.float32)) == 0
    with pytest.raises(ValueError):
        orc.count_nonuniform_tiles(np.ones(17, np.float32))


@pytest.mark.parametrize("row", [False, True])
def test_mm_reference_hand_operands(orc, row):
    """The product reference on operands written by hand: a[0,0] = 1.0 and
    a[1,17] = 6 under a block scale of 2 (code 0x40); b[0,0] = 1.5 and
    b[1,17] = -1.0; every other element 0, every other scale 1.0 (0x38).
    amax 2688 gives S = 1 (g = 1); with a row scale, row 1 of a has amax
    1344, S = 2, g = 0.5.  Expected out[0,0] = 1.5 and out[1,1] = -12
    (-6 row-scaled), zeros elsewhere; the bound is gamma_(K+2) times the
    absolute sum of the terms."""
    M = N = 16
    K = 64
    ac = np.zeros((M, K // 2), np.uint8)
    bc = np.zeros((N, K // 2), np.uint8)
    as_ = np.full((M, K // 16), 0x38, np.uint8)
    bs = np.full((N, K // 16), 0x38, np.uint8)
    ac[0, 0] = 0x02          # element 0 (low nibble): 1.0
    ac[1, 8] = 0x70          # element 17 (high nibble of byte 8): 6
    as_[1, 1] = 0x40         # block 1 of row 1: scale 2.0
    bc[0, 0] = 0x03          # 1.5
    bc[1, 8] = 0xA0          # element 17: -1.0
    a_amax = np.full(M if row else 1, 2688.0, np.float32)
    if row:
        a_amax[1] = 1344.0
    cfg = orc.Config(row_scaled=row)
    ref, bound = orc.mm_reference(ac, as_, a_amax, bc, bs, np.array([2688.0], np.float32), cfg)
    want = np.zeros((M, N))
    want[0, 0] = 1.5
    want[1, 1] = -6.0 if row else -12.0
    assert np.array_equal(ref, want)
    n = K + 2
    gamma = n * 2.0 ** -24 / (1 - n * 2.0 ** -24)
    assert bound[0, 0] == gamma * 1.5 and bound[1, 1] == gamma * abs(want[1, 1])
    assert np.count_nonzero(bound) == 2
