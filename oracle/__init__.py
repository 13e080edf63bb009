"""CPU oracle for the NVFP4 four-over-six block quantizer (ctypes front end).

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the benchmark's CPU-baseline / reference leg may import this package.  It never
touches the CUDA library and the CUDA library never touches it.

Inputs are numpy arrays.  Floating inputs are passed as float32 (a bf16/fp16
tensor widens to float32 exactly); codes and scales are uint8; bf16/fp16
outputs come back as uint16 bit patterns so that comparisons are bit-exact.
"""
import ctypes
import os
from dataclasses import dataclass

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(os.environ.get("ORACLE_LIB_OVERRIDE") or _build.build())
        _declare(_lib)
    return _lib


def use_library(path):
    """Swap the loaded oracle for another build of it (the mutation tests load
    copies with a planted mistake); returns the previous handle."""
    global _lib
    prev = _lib
    if path is None:
        _lib = None
    elif isinstance(path, ctypes.CDLL):
        _lib = path
    else:
        _lib = ctypes.CDLL(path)
        _declare(_lib)
    return prev


class OrcConfig(ctypes.Structure):
    _fields_ = [("block16x16", ctypes.c_int), ("four_over_six", ctypes.c_int),
                ("mse", ctypes.c_int), ("err_f16", ctypes.c_int), ("bound", ctypes.c_int),
                ("row_scaled", ctypes.c_int), ("amax_is_input", ctypes.c_int),
                ("seq_order", ctypes.c_int)]


OUT_F32, OUT_BF16, OUT_F16 = 0, 1, 2
_P = ctypes.c_void_p
_I64 = ctypes.c_int64


def _declare(L):
    L.orc_e2m1_value.restype = ctypes.c_float
    L.orc_e2m1_value.argtypes = [ctypes.c_uint32]
    L.orc_e4m3_value.restype = ctypes.c_float
    L.orc_e4m3_value.argtypes = [ctypes.c_uint32]
    L.orc_e2m1_encode.restype = ctypes.c_uint32
    L.orc_e2m1_encode.argtypes = [ctypes.c_float]
    L.orc_e4m3_encode.restype = ctypes.c_uint32
    L.orc_e4m3_encode.argtypes = [ctypes.c_float]
    L.orc_global_scale.restype = ctypes.c_float
    L.orc_global_scale.argtypes = [ctypes.c_float, ctypes.c_int]
    for name in ("orc_e2m1_encode_array", "orc_e4m3_encode_array", "orc_f16_round_array",
                 "orc_bf16_round_array", "orc_f16_bits_array", "orc_bf16_bits_array"):
        f = getattr(L, name)
        f.restype = None
        f.argtypes = [_P, _P, _I64]
    L.orc_amax_tensor.argtypes = [_P, _I64, _P]
    L.orc_amax_rows.argtypes = [_P, _I64, _I64, _P]
    L.orc_amax_groups.argtypes = [_P, _I64, _I64, _P, ctypes.c_int, _P]
    L.orc_quantize.restype = ctypes.c_int
    L.orc_quantize.argtypes = [_P, _I64, _I64, ctypes.POINTER(OrcConfig), _P, _P, _P, _P, _P]
    L.orc_qdq.restype = ctypes.c_int
    L.orc_qdq.argtypes = [_P, _I64, _I64, ctypes.POINTER(OrcConfig), _P, _P, ctypes.c_int]
    L.orc_quantize_grouped.restype = ctypes.c_int
    L.orc_quantize_grouped.argtypes = [_P, _I64, _I64, _P, ctypes.c_int,
                                       ctypes.POINTER(OrcConfig), _P, _P, _P]
    L.orc_dequantize.restype = ctypes.c_int
    L.orc_dequantize.argtypes = [_P, _P, _P, _I64, _I64, ctypes.POINTER(OrcConfig), _P,
                                 ctypes.c_int]


@dataclass
class Config:
    """Knobs of the method: block shape, standard vs four-over-six, error
    metric and precision, E4M3 bound, scale granularity, and the order in
    which a block's 16 error terms are summed (pinned tree, or sequential
    with seq_order, 1x16 only)."""
    block16x16: bool = False
    four_over_six: bool = True
    mse: bool = True
    err_f16: bool = False
    bound: int = 448
    row_scaled: bool = False
    amax_is_input: bool = False
    seq_order: bool = False

    def c(self):
        return OrcConfig(int(self.block16x16), int(self.four_over_six), int(self.mse),
                         int(self.err_f16), int(self.bound), int(self.row_scaled),
                         int(self.amax_is_input), int(self.seq_order))


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _f32(x):
    return np.ascontiguousarray(x, dtype=np.float32)


# ---- format conversions -----------------------------------------------------
def e2m1_value(code):
    return lib().orc_e2m1_value(int(code))


def e4m3_value(code):
    return lib().orc_e4m3_value(int(code))


def e2m1_encode(a):
    a = _f32(a).ravel()
    out = np.empty(a.size, np.uint8)
    lib().orc_e2m1_encode_array(_ptr(a), _ptr(out), a.size)
    return out


def e4m3_encode(a):
    a = _f32(a).ravel()
    out = np.empty(a.size, np.uint8)
    lib().orc_e4m3_encode_array(_ptr(a), _ptr(out), a.size)
    return out


def f16_round(a):
    a = _f32(a).ravel()
    out = np.empty(a.size, np.float32)
    lib().orc_f16_round_array(_ptr(a), _ptr(out), a.size)
    return out


def bf16_round(a):
    a = _f32(a).ravel()
    out = np.empty(a.size, np.float32)
    lib().orc_bf16_round_array(_ptr(a), _ptr(out), a.size)
    return out


def f16_bits(a):
    a = _f32(a).ravel()
    out = np.empty(a.size, np.uint16)
    lib().orc_f16_bits_array(_ptr(a), _ptr(out), a.size)
    return out


def bf16_bits(a):
    a = _f32(a).ravel()
    out = np.empty(a.size, np.uint16)
    lib().orc_bf16_bits_array(_ptr(a), _ptr(out), a.size)
    return out


def global_scale(A, bound):
    return lib().orc_global_scale(float(A), int(bound))


# ---- method ------------------------------------------------------------------
def amax_tensor(x):
    x = _f32(x)
    out = np.zeros(1, np.float32)
    lib().orc_amax_tensor(_ptr(x), x.size, _ptr(out))
    return out


def amax_rows(x):
    x = _f32(x)
    out = np.zeros(x.shape[0], np.float32)
    lib().orc_amax_rows(_ptr(x), x.shape[0], x.shape[1], _ptr(out))
    return out


def amax_groups(x, offs):
    x = _f32(x)
    offs = np.ascontiguousarray(offs, dtype=np.int32)
    out = np.zeros(max(offs.size, 1), np.float32)
    lib().orc_amax_groups(_ptr(x), x.shape[0], x.shape[1], _ptr(offs), offs.size, _ptr(out))
    return out[:offs.size]


def _amax_buf(x, cfg, amax):
    n = x.shape[0] if cfg.row_scaled else 1
    if cfg.amax_is_input:
        a = np.ascontiguousarray(amax, dtype=np.float32).ravel()
        assert a.size == n
        return a.copy()
    return np.zeros(n, np.float32)


def quantize(x, cfg: Config, amax=None, with_errors=False):
    """Returns (codes [R, C/2] u8, scales u8, amax f32[, err6, err4])."""
    x = _f32(x)
    R, C = x.shape
    a = _amax_buf(x, cfg, amax)
    codes = np.zeros((R, C // 2), np.uint8)
    srows = R // 16 if cfg.block16x16 else R
    scales = np.zeros((srows, C // 16), np.uint8)
    e6 = np.zeros(scales.shape, np.float32) if with_errors else None
    e4 = np.zeros(scales.shape, np.float32) if with_errors else None
    cc = cfg.c()
    rc = lib().orc_quantize(_ptr(x), R, C, ctypes.byref(cc), _ptr(a), _ptr(codes), _ptr(scales),
                            _ptr(e6), _ptr(e4))
    if rc:
        raise ValueError("oracle: bad shape/config")
    if with_errors:
        return codes, scales, a, e6, e4
    return codes, scales, a


def quantize_colwise(x, cfg: Config, amax=None):
    """The column-wise operand: the quantization of x^T (blocks of 16
    consecutive rows of one column of x), by definition quantize(x.T).  The
    per-tensor amax of x^T is that of x."""
    return quantize(np.ascontiguousarray(_f32(x).T), cfg, amax=amax)


def swizzle_scales(scales):
    """Scales [R, C/16] in the tiled layout of block-scaled FP4 GEMMs: padded
    with zeros to a multiple of 128 rows and 4 columns, cut into 128 x 4
    tiles of 512 bytes stored tile-row by tile-row; inside a tile, scale
    (32 i + j, k) is byte 16 j + 4 i + k."""
    s = np.ascontiguousarray(scales, dtype=np.uint8)
    R, NB = s.shape
    PR, PC = -(-R // 128) * 128, -(-NB // 4) * 4
    pad = np.zeros((PR, PC), np.uint8)
    pad[:R, :NB] = s
    r = np.arange(PR)[:, None]
    c = np.arange(PC)[None, :]
    off = ((r // 128) * (PC // 4) + c // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + c % 4
    out = np.zeros(PR * PC, np.uint8)
    out[off.ravel()] = pad.ravel()
    return out


def block_values(codes, scales):
    """The value v * sigma of every element of 1x16 codes [R, C/2] and E4M3
    block scales [R, C/16] (the standard NVFP4 decode without the global
    scale), exact in binary64: an E2M1 value times an E4M3 value has at most
    seven significant bits."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    R, C2 = codes.shape
    q = np.empty((R, 2 * C2), np.uint32)
    q[:, 0::2], q[:, 1::2] = codes & 0xF, codes >> 4
    v = np.vectorize(e2m1_value, otypes=[np.float64])(q)
    sig = np.vectorize(e4m3_value, otypes=[np.float64])(np.asarray(scales, np.uint32))
    return v * np.repeat(sig, 16, axis=1)


def mm_reference(a_codes, a_scales, a_amax, b_codes, b_scales, b_amax, cfg: Config):
    """The product of quantized operands, out = a . b^T (grouped PR, the
    four_over_six_mm forward), as the binary64 product of the block values
    (its rounding far below the bound) times the FP32 global decode scales
    g = rn(1 / S) (S from the amax
    as quantization computed it; per row of a when cfg.row_scaled), together
    with the bound any FP32 evaluation must meet: K products summed in any
    order plus the two epilogue multiplies, gamma_(K+2) * sum |terms| * |g_a g_b|
    with gamma_n = n u / (1 - n u), u = 2^-24.  Returns (ref, bound)."""
    pa, pb = block_values(a_codes, a_scales), block_values(b_codes, b_scales)
    K = pa.shape[1]
    ga = np.float32(1.0) / np.array([global_scale(float(v), cfg.bound)
                                     for v in np.ravel(a_amax)], np.float32)
    gb = np.float32(1.0) / np.float32(global_scale(float(np.ravel(b_amax)[0]), cfg.bound))
    ga = ga.astype(np.float64).reshape(-1, 1) if cfg.row_scaled else np.float64(ga[0])
    g = ga * np.float64(gb)
    n = K + 2
    gamma = n * 2.0 ** -24 / (1.0 - n * 2.0 ** -24)
    return (pa @ pb.T) * g, gamma * (np.abs(pa) @ np.abs(pb).T) * np.abs(g)


def count_nonuniform_tiles(amax):
    """The tile-uniform contract of 16x16 blocks with a row-scaled global
    scale (grouped PR: the 16 rows of a tile share one amax): the number of
    16-row tiles of a per-row amax [rows] whose 16 entries are not all
    bitwise equal.  rows must be a multiple of 16."""
    bits = np.ascontiguousarray(amax, dtype=np.float32).view(np.uint32).ravel()
    if bits.size % 16:
        raise ValueError("rows must be a multiple of 16")
    count = 0
    for t in range(bits.size // 16):
        tile = bits[16 * t:16 * t + 16]
        if any(int(v) != int(tile[0]) for v in tile):
            count += 1
    return count


_OUTK = {"f32": (OUT_F32, np.float32), "bf16": (OUT_BF16, np.uint16), "f16": (OUT_F16, np.uint16)}


def qdq(x, cfg: Config, out_dtype, amax=None):
    """Fused quantize-dequantize; returns (out, amax).  out is float32 for
    'f32' and uint16 bit patterns for 'bf16' / 'f16'."""
    x = _f32(x)
    R, C = x.shape
    a = _amax_buf(x, cfg, amax)
    kind, npdt = _OUTK[out_dtype]
    out = np.zeros((R, C), npdt)
    cc = cfg.c()
    rc = lib().orc_qdq(_ptr(x), R, C, ctypes.byref(cc), _ptr(a), _ptr(out), kind)
    if rc:
        raise ValueError("oracle: bad shape/config")
    return out, a


def quantize_grouped(x, offs, cfg: Config, group_amax=None):
    x = _f32(x)
    R, C = x.shape
    offs = np.ascontiguousarray(offs, dtype=np.int32)
    G = offs.size
    if cfg.amax_is_input:
        ga = np.ascontiguousarray(group_amax, dtype=np.float32).copy()
    else:
        ga = np.zeros(max(G, 1), np.float32)
    codes = np.zeros((R, C // 2), np.uint8)
    srows = R // 16 if cfg.block16x16 else R
    scales = np.zeros((srows, C // 16), np.uint8)
    cc = cfg.c()
    rc = lib().orc_quantize_grouped(_ptr(x), R, C, _ptr(offs), G, ctypes.byref(cc), _ptr(ga),
                                    _ptr(codes), _ptr(scales))
    if rc:
        raise ValueError("oracle: bad shape/config")
    return codes, scales, ga[:G]


def dequantize(codes, scales, amax, cfg: Config, out_dtype):
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    a = np.ascontiguousarray(amax, dtype=np.float32).ravel()
    R, C2 = codes.shape
    C = C2 * 2
    kind, npdt = _OUTK[out_dtype]
    out = np.zeros((R, C), npdt)
    cc = cfg.c()
    rc = lib().orc_dequantize(_ptr(codes), _ptr(scales), _ptr(a), R, C, ctypes.byref(cc),
                              _ptr(out), kind)
    if rc:
        raise ValueError("oracle: bad shape/config")
    return out
