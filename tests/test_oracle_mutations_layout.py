"""Plant plausible mistakes in the oracle's layout and contract functions (the
tiled scale layout, the column-wise operand, the tile-uniform count) and
check that their pins catch each one.  Each mutant replaces one function of
the oracle for the duration of a test; the pins are the ones in
test_oracle_method.py, run unchanged."""
import numpy as np
import pytest

import oracle
import test_oracle_method as pins


def _swizzle(scales, tile_of, byte_of, pad_cols=True):
    s = np.ascontiguousarray(scales, dtype=np.uint8)
    R, NB = s.shape
    PR = -(-R // 128) * 128
    PC = -(-NB // 4) * 4 if pad_cols else NB
    pad = np.zeros((PR, PC), np.uint8)
    pad[:R, :NB] = s
    r = np.arange(PR)[:, None]
    c = np.arange(PC)[None, :]
    off = tile_of(r, c, PR, PC) * 512 + byte_of(r, c)
    out = np.zeros(PR * max(PC, 4), np.uint8)
    out[np.clip(off, 0, out.size - 1).ravel()] = pad.ravel()
    return out


SWIZZLE_MUTANTS = {
    # row groups and rows inside a tile exchanged
    "ij_swapped": lambda s: _swizzle(
        s, lambda r, c, PR, PC: (r // 128) * (PC // 4) + c // 4,
        lambda r, c: ((r % 128) // 32) * 16 + (r % 32) * 4 + c % 4),
    # tiles stored column by column instead of tile-row by tile-row
    "tiles_column_major": lambda s: _swizzle(
        s, lambda r, c, PR, PC: (c // 4) * (PR // 128) + r // 128,
        lambda r, c: (r % 32) * 16 + ((r % 128) // 32) * 4 + c % 4),
    # scale columns not padded to a multiple of 4
    "no_column_padding": lambda s: _swizzle(
        s, lambda r, c, PR, PC: (r // 128) * -(-PC // 4) + c // 4,
        lambda r, c: (r % 32) * 16 + ((r % 128) // 32) * 4 + c % 4, pad_cols=False),
}


@pytest.mark.parametrize("name", sorted(SWIZZLE_MUTANTS))
def test_swizzle_mutants_are_caught(orc, monkeypatch, name):
    monkeypatch.setattr(oracle, "swizzle_scales", SWIZZLE_MUTANTS[name])
    with pytest.raises(AssertionError):
        pins.test_swizzled_scale_layout_offsets(orc)


def _count_float_equal(amax):
    a = np.ascontiguousarray(amax, dtype=np.float32).ravel()
    return sum(1 for t in range(a.size // 16) if np.any(a[16 * t:16 * t + 16] != a[16 * t]))


def _count_ignores_first_row(amax):
    a = np.ascontiguousarray(amax, dtype=np.float32).view(np.uint32).ravel()
    return sum(1 for t in range(a.size // 16)
               if np.any(a[16 * t + 1:16 * t + 16] != a[16 * t + 1]))


@pytest.mark.parametrize("mutant", [_count_float_equal, _count_ignores_first_row])
def test_tile_count_mutants_are_caught(orc, monkeypatch, mutant):
    monkeypatch.setattr(oracle, "count_nonuniform_tiles", mutant)
    with pytest.raises(AssertionError):
        pins.test_tile_uniform_count_hand_cases(orc)


def _colwise_without_transpose(x, cfg, amax=None):
    return oracle.quantize(np.ascontiguousarray(np.asarray(x, np.float32)), cfg, amax=amax)


def _colwise_row_scaled(x, cfg, amax=None):
    c = oracle.Config(**{**cfg.__dict__, "row_scaled": True, "amax_is_input": False})
    return oracle.quantize(np.ascontiguousarray(np.asarray(x, np.float32).T), c)


@pytest.mark.parametrize("mutant", [_colwise_without_transpose, _colwise_row_scaled])
def test_colwise_mutants_are_caught(orc, monkeypatch, mutant):
    monkeypatch.setattr(oracle, "quantize_colwise", mutant)
    with pytest.raises(AssertionError):
        pins.test_colwise_is_the_quantization_of_each_column(orc)
