"""NVFP4 four-over-six block quantizer for GB300 -- Python binding.

Argument marshalling only: every step of the quantizer runs in the CUDA
kernels of ``libfos.so`` (C ABI in ``include/fos.h``).  PyTorch supplies the
device memory and the current stream.  There is no CPU path: if the library
is not built, or a tensor is not on a CUDA device, the call raises.

Entry points (names follow the C ABI):
  amax(x, granularity)                      -> float32 amax
  quantize(x, ...)                          -> (codes, scales, amax)
  check_tile_amax(amax)                     -> number of non-uniform 16-row tiles
  quantize_list(xs, ...)                    -> ([codes], [scales], [amax])
  quantize_overlap(x, amax, codes, scales, x_next, amax_next)
  dequantize(codes, scales, amax, ...)      -> tensor
  qdq(xs, ...)                              -> list of tensors (one launch)
  qdq_fused(xs, ...)                        -> (outs, amaxes), every amax in the same launch
  workspace_error(workspace)                -> error word of a fused launch
  quantize_grouped(x, offs, ...)            -> (codes, scales, group_amax)
  quantize_colwise(x, ...)                  -> (codes_t, scales_t, amax[, codes, scales])
  swizzle_scales(scales, rows, cols)        -> scales in the tiled GEMM layout
  mm(a_codes, a_tiled, a_amax, b_codes, b_tiled, b_amax) -> fp32 a . b^T
"""
import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfos.so")

(FOS_OK, FOS_ERR_INVALID_ARG, FOS_ERR_UNSUPPORTED, FOS_ERR_MISALIGNED, FOS_ERR_CUDA,
 FOS_ERR_NONUNIFORM_TILE_AMAX) = range(6)
FOS_BF16, FOS_FP16, FOS_FP32 = 0, 1, 2
QDQ_MAX_LIST = 64
GROUPED_MAX_GROUPS = 8192

_DT = {torch.bfloat16: FOS_BF16, torch.float16: FOS_FP16, torch.float32: FOS_FP32}
_NAMES = ("fos_amax", "fos_quantize", "fos_quantize_list", "fos_quantize_overlap",
          "fos_dequantize", "fos_qdq", "fos_quantize_grouped",
          "fos_status_string", "fos_version", "fos_diag_convert")


class FosError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__("%s failed: %s (status %d)" % (what, status_string(status), status))


class FosConfig(ctypes.Structure):
    _fields_ = [("block", ctypes.c_int), ("mode", ctypes.c_int), ("err_metric", ctypes.c_int),
                ("err_precision", ctypes.c_int), ("e4m3_bound", ctypes.c_int),
                ("granularity", ctypes.c_int), ("amax_is_input", ctypes.c_int),
                ("err_order", ctypes.c_int), ("scale_layout", ctypes.c_int)]


@dataclass(frozen=True)
class Config:
    """Knobs of the quantizer (see include/fos.h)."""
    block16x16: bool = False
    four_over_six: bool = True
    mse: bool = True
    err_f16: bool = False
    bound: int = 448
    row_scaled: bool = False
    seq_order: bool = False  # sum a block's error terms in element order (1x16 only)
    scale_tiled: bool = False  # write scales in the tiled GEMM layout (1x16 only)

    def c(self, amax_is_input):
        return FosConfig(int(self.block16x16), int(self.four_over_six), int(self.mse),
                         int(self.err_f16), int(self.bound), int(self.row_scaled),
                         int(bool(amax_is_input)), int(self.seq_order),
                         int(self.scale_tiled))


_lib = None


def lib():
    """The loaded libfos.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libfos.so is not built (run __graft_entry__.build() or "
                               "python -m nvfp4_quantization_precision_gb300.build)")
        L = ctypes.CDLL(LIB_PATH)
        P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        CFG = ctypes.POINTER(FosConfig)
        L.fos_amax.argtypes = [P, I, I64, I64, I, P, P]
        L.fos_quantize.argtypes = [P, I, I64, I64, CFG, P, P, P, P]
        L.fos_quantize_list.argtypes = [I, P, I, P, P, CFG, P, P, P, P]
        L.fos_quantize_overlap.argtypes = [P, I, I64, I64, CFG, P, P, P, P, I64, I64, P, P]
        L.fos_dequantize.argtypes = [P, P, P, I64, I64, CFG, P, I, P]
        L.fos_qdq.argtypes = [I, P, P, P, P, P, I, CFG, P]
        L.fos_quantize_grouped.argtypes = [P, I, I64, I64, P, I, CFG, P, P, P, P]
        L.fos_diag_convert.argtypes = [I, P, P, I64, P]
        L.fos_qdq_fused_workspace_bytes.argtypes = [I]
        L.fos_qdq_fused_workspace_bytes.restype = ctypes.c_size_t
        L.fos_qdq_fused.argtypes = [I, P, P, P, P, P, I, CFG, P, ctypes.c_size_t, P]
        L.fos_workspace_error.argtypes = [P, P, ctypes.POINTER(I)]
        L.fos_check_tile_amax.argtypes = [P, I64, P, P]
        L.fos_tile_amax_status.argtypes = [P, P]
        L.fos_swizzled_scales_bytes.argtypes = [I64, I64]
        L.fos_swizzled_scales_bytes.restype = ctypes.c_int64
        for n in ("fos_check_tile_amax", "fos_tile_amax_status", "fos_amax", "fos_quantize", "fos_quantize_list", "fos_quantize_overlap",
                  "fos_dequantize", "fos_qdq", "fos_qdq_fused", "fos_workspace_error",
                  "fos_quantize_grouped", "fos_diag_convert"):
            getattr(L, n).restype = ctypes.c_int
        L.fos_status_string.argtypes = [I]
        L.fos_status_string.restype = ctypes.c_char_p
        L.fos_version.restype = ctypes.c_int
        _lib = L
    return _lib


def status_string(s):
    return lib().fos_status_string(int(s)).decode()


def _check(rc, what):
    if rc != FOS_OK:
        raise FosError(rc, what)


def _stream(t):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _cuda(t, name):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def amax(x, row_scaled=False, out=None):
    """NaN-dropping max|x| per tensor ([1]) or per row ([rows]), float32."""
    _cuda(x, "x")
    R, C = x.shape
    n = R if row_scaled else 1
    if out is None:
        out = torch.empty(n, dtype=torch.float32, device=x.device)
    _check(lib().fos_amax(_p(x), _DT[x.dtype], R, C, int(row_scaled), _p(out), _stream(x)),
           "fos_amax")
    return out


def scales_shape(rows, cols, block16x16):
    return (rows // 16 if block16x16 else rows, cols // 16)


def _scales_buffer(rows, cols, cfg, dev):
    """The scale output of a quantize of [rows, cols] under cfg: [rows, cols/16]
    (plain), or the flat tiled buffer of fos_swizzled_scales_bytes bytes."""
    if cfg.scale_tiled:
        nbytes = lib().fos_swizzled_scales_bytes(rows, cols)
        if nbytes < 0:
            raise ValueError("bad shape for tiled scales")
        return torch.empty(nbytes, dtype=torch.uint8, device=dev)
    return torch.empty(scales_shape(rows, cols, cfg.block16x16), dtype=torch.uint8, device=dev)


def check_tile_amax(amax, bad=None):
    """Number of 16-row tiles of a per-row amax [rows] whose entries are not
    all bitwise equal (fos_check_tile_amax); reads the count back, so it
    waits for the stream."""
    _cuda(amax, "amax")
    if bad is None:
        bad = torch.empty(1, dtype=torch.int64, device=amax.device)
    _check(lib().fos_check_tile_amax(_p(amax), amax.numel(), _p(bad), _stream(amax)),
           "fos_check_tile_amax")
    return int(bad.item())


def quantize(x, cfg=Config(), amax=None, codes=None, scales=None, amax_given=None,
             validate=False):
    """Quantize x [rows, cols] (bf16 / fp16 / fp32).  amax is read when
    given (the default when a tensor is passed); with amax_given=False it is
    an output buffer the library fills.  With amax=None it is allocated,
    computed and returned.  validate=True checks a given per-row amax of a
    16x16 quantize for tile uniformity first (fos_check_tile_amax and
    fos_tile_amax_status, which wait for the stream) and raises FosError
    with FOS_ERR_NONUNIFORM_TILE_AMAX when a tile's rows differ."""
    _cuda(x, "x")
    R, C = x.shape
    dev = x.device
    given = (amax is not None) if amax_given is None else bool(amax_given)
    if validate and given and cfg.block16x16 and cfg.row_scaled:
        _cuda(amax, "amax")
        bad = torch.empty(1, dtype=torch.int64, device=dev)
        _check(lib().fos_check_tile_amax(_p(amax), amax.numel(), _p(bad), _stream(amax)),
               "fos_check_tile_amax")
        _check(lib().fos_tile_amax_status(_p(bad), _stream(amax)), "fos_quantize")
    if amax is None:
        amax = torch.empty(R if cfg.row_scaled else 1, dtype=torch.float32, device=dev)
    if codes is None:
        codes = torch.empty((R, C // 2), dtype=torch.uint8, device=dev)
    if scales is None:
        scales = _scales_buffer(R, C, cfg, dev)
    cc = cfg.c(given)
    _check(lib().fos_quantize(_p(x), _DT[x.dtype], R, C, ctypes.byref(cc), _p(amax), _p(codes),
                              _p(scales), _stream(x)), "fos_quantize")
    return codes, scales, amax


def quantize_list(xs, cfg=Config(), amaxes=None, codes=None, scales=None, amax_given=None):
    """fos_quantize over a list of tensors of one dtype (see fos_quantize_list:
    with per-tensor scale and amax computed, the amax pass of tensor i+1 runs
    inside the encode launch of tensor i).  Returns (codes, scales, amaxes)
    lists."""
    n = len(xs)
    if n == 0:
        return [], [], []
    for x in xs:
        _cuda(x, "x")
    dt = xs[0].dtype
    given = (amaxes is not None) if amax_given is None else bool(amax_given)
    dev = xs[0].device
    if amaxes is None:
        amaxes = [torch.empty(x.shape[0] if cfg.row_scaled else 1, dtype=torch.float32,
                              device=dev) for x in xs]
    if codes is None:
        codes = [torch.empty((x.shape[0], x.shape[1] // 2), dtype=torch.uint8, device=dev)
                 for x in xs]
    if scales is None:
        scales = [_scales_buffer(x.shape[0], x.shape[1], cfg, dev) for x in xs]
    P = ctypes.c_void_p * n
    xp = P(*[x.data_ptr() for x in xs])
    ap = P(*[a.data_ptr() for a in amaxes])
    cp = P(*[c.data_ptr() for c in codes])
    sp = P(*[s.data_ptr() for s in scales])
    rows = (ctypes.c_int64 * n)(*[x.shape[0] for x in xs])
    cols = (ctypes.c_int64 * n)(*[x.shape[1] for x in xs])
    cc = cfg.c(given)
    _check(lib().fos_quantize_list(n, xp, _DT[dt], rows, cols, ctypes.byref(cc), ap, cp, sp,
                                   _stream(xs[0])), "fos_quantize_list")
    return codes, scales, amaxes


def quantize_overlap(x, amax, codes, scales, x_next=None, amax_next=None, cfg=Config()):
    """Quantize x with its per-tensor amax given (1x16) and compute the amax
    of x_next in the same launch (fos_quantize_overlap)."""
    _cuda(x, "x")
    R, C = x.shape
    if x_next is not None:
        _cuda(x_next, "x_next")
        Rn, Cn = x_next.shape
    else:
        Rn = Cn = 0
    cc = cfg.c(True)
    _check(lib().fos_quantize_overlap(_p(x), _DT[x.dtype], R, C, ctypes.byref(cc), _p(amax),
                                      _p(codes), _p(scales), _p(x_next), Rn, Cn, _p(amax_next),
                                      _stream(x)), "fos_quantize_overlap")
    return codes, scales


def dequantize(codes, scales, amax, cfg=Config(), out_dtype=torch.bfloat16, out=None):
    _cuda(codes, "codes")
    R, C2 = codes.shape
    C = 2 * C2
    if out is None:
        out = torch.empty((R, C), dtype=out_dtype, device=codes.device)
    cc = cfg.c(True)
    _check(lib().fos_dequantize(_p(codes), _p(scales), _p(amax), R, C, ctypes.byref(cc), _p(out),
                                _DT[out.dtype], _stream(codes)), "fos_dequantize")
    return out


def qdq(xs, cfg=Config(), amaxes=None, outs=None, amax_given=None):
    """Fused quantize-dequantize of a list of rank-2 bf16/fp16 tensors in one
    launch.  amaxes: list of 1-element float32 tensors, read when given (the
    default when passed) or filled when amax_given=False; None allocates and
    computes them.  Returns the list of outputs."""
    n = len(xs)
    if n == 0:
        return []
    for x in xs:
        _cuda(x, "x")
    dt = xs[0].dtype
    given = (amaxes is not None) if amax_given is None else bool(amax_given)
    if amaxes is None:
        amaxes = [torch.empty(1, dtype=torch.float32, device=x.device) for x in xs]
    if outs is None:
        outs = [torch.empty_like(x) for x in xs]
    P = ctypes.c_void_p * n
    xp = P(*[x.data_ptr() for x in xs])
    op = P(*[o.data_ptr() for o in outs])
    ap = P(*[a.data_ptr() for a in amaxes])
    rows = (ctypes.c_int64 * n)(*[x.shape[0] for x in xs])
    cols = (ctypes.c_int64 * n)(*[x.shape[1] for x in xs])
    cc = cfg.c(given)
    _check(lib().fos_qdq(n, xp, op, rows, cols, ap, _DT[dt], ctypes.byref(cc), _stream(xs[0])),
           "fos_qdq")
    return outs


def quantize_colwise(x, cfg=Config(), amax=None, codes_t=None, scales_t=None, rowwise=False,
                     codes=None, scales=None, amax_given=None):
    """fos_quantize_colwise: the quantization of x.T from x (1x16, per-tensor
    scale).  With rowwise=True (or codes/scales passed) the row-wise result
    of x comes from the same read.  Returns (codes_t, scales_t, amax) or
    (codes_t, scales_t, amax, codes, scales)."""
    _cuda(x, "x")
    R, C = x.shape
    dev = x.device
    given = (amax is not None) if amax_given is None else bool(amax_given)
    if amax is None:
        amax = torch.empty(1, dtype=torch.float32, device=dev)
    if codes_t is None:
        codes_t = torch.empty((C, R // 2), dtype=torch.uint8, device=dev)
    if scales_t is None:
        scales_t = _scales_buffer(C, R, cfg, dev)
    dual = rowwise or codes is not None or scales is not None
    if dual and codes is None:
        codes = torch.empty((R, C // 2), dtype=torch.uint8, device=dev)
    if dual and scales is None:
        scales = _scales_buffer(R, C, cfg, dev)
    L = lib()
    if not getattr(L, "_colwise_declared", False):
        P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.fos_quantize_colwise.argtypes = [P, I, I64, I64, ctypes.POINTER(FosConfig), P, P, P, P,
                                           P, P]
        L.fos_quantize_colwise.restype = I
        L._colwise_declared = True
    cc = cfg.c(given)
    _check(L.fos_quantize_colwise(_p(x), _DT[x.dtype], R, C, ctypes.byref(cc), _p(amax),
                                  _p(codes_t), _p(scales_t), _p(codes), _p(scales), _stream(x)),
           "fos_quantize_colwise")
    if dual:
        return codes_t, scales_t, amax, codes, scales
    return codes_t, scales_t, amax


def swizzle_scales(scales, rows, cols, out=None):
    """fos_swizzle_scales: 1x16 scales [rows, cols/16] in the tiled layout of
    block-scaled FP4 GEMMs (a flat uint8 tensor, zero padded)."""
    _cuda(scales, "scales")
    L = lib()
    if not getattr(L, "_swizzle_declared", False):
        L.fos_swizzled_scales_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64]
        L.fos_swizzled_scales_bytes.restype = ctypes.c_int64
        L.fos_swizzle_scales.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                         ctypes.c_void_p, ctypes.c_void_p]
        L.fos_swizzle_scales.restype = ctypes.c_int
        L._swizzle_declared = True
    nbytes = L.fos_swizzled_scales_bytes(rows, cols)
    if nbytes < 0:
        raise ValueError("bad shape for swizzled scales")
    if out is None:
        out = torch.empty(nbytes, dtype=torch.uint8, device=scales.device)
    _check(L.fos_swizzle_scales(_p(scales), rows, cols, _p(out), _stream(scales)),
           "fos_swizzle_scales")
    return out


def mm(a_codes, a_scales_tiled, a_amax, b_codes, b_scales_tiled, b_amax, cfg=Config(),
       out=None):
    """fos_mm: a . b^T (fp32 [M, N]) from a's and b's 1x16 codes, tiled scales
    (swizzle_scales) and amaxes; cfg.row_scaled when a was quantized with a
    per-row scale."""
    _cuda(a_codes, "a_codes")
    M, K2 = a_codes.shape
    N = b_codes.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=a_codes.device)
    L = lib()
    if not getattr(L, "_mm_declared", False):
        P = ctypes.c_void_p
        L.fos_mm.argtypes = [P, P, P, P, P, P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                             ctypes.POINTER(FosConfig), P, P]
        L.fos_mm.restype = ctypes.c_int
        L._mm_declared = True
    cc = cfg.c(True)
    _check(L.fos_mm(_p(a_codes), _p(a_scales_tiled), _p(a_amax), _p(b_codes), _p(b_scales_tiled),
                    _p(b_amax), M, N, 2 * K2, ctypes.byref(cc), _p(out), _stream(a_codes)),
           "fos_mm")
    return out


def qdq_fused_workspace(n, device):
    """A workspace for fos_qdq_fused over n tensors (caller-side allocation)."""
    nb = lib().fos_qdq_fused_workspace_bytes(int(n))
    return torch.empty(max(nb, 256), dtype=torch.uint8, device=device)


def qdq_fused(xs, cfg=Config(), amaxes=None, outs=None, workspace=None):
    """fos_qdq_fused: amax of every tensor and the fused quantize-dequantize
    of the list in one persistent launch.  amaxes (outputs) and outs are
    allocated when None; workspace too (see qdq_fused_workspace).  Returns
    (outs, amaxes)."""
    n = len(xs)
    if n == 0:
        return [], []
    for x in xs:
        _cuda(x, "x")
    dev = xs[0].device
    if amaxes is None:
        amaxes = [torch.empty(1, dtype=torch.float32, device=dev) for _ in xs]
    if outs is None:
        outs = [torch.empty_like(x) for x in xs]
    if workspace is None:
        workspace = qdq_fused_workspace(n, dev)
    P = ctypes.c_void_p * n
    xp = P(*[x.data_ptr() for x in xs])
    op = P(*[o.data_ptr() for o in outs])
    ap = P(*[a.data_ptr() for a in amaxes])
    rows = (ctypes.c_int64 * n)(*[x.shape[0] for x in xs])
    cols = (ctypes.c_int64 * n)(*[x.shape[1] for x in xs])
    cc = cfg.c(False)
    _check(lib().fos_qdq_fused(n, xp, op, rows, cols, ap, _DT[xs[0].dtype], ctypes.byref(cc),
                               _p(workspace), workspace.numel(), _stream(xs[0])),
           "fos_qdq_fused")
    return outs, amaxes


def workspace_error(workspace):
    """The error word of a fused-launch workspace (waits for the stream)."""
    code = ctypes.c_int(0)
    _check(lib().fos_workspace_error(_p(workspace), _stream(workspace), ctypes.byref(code)),
           "fos_workspace_error")
    return code.value


def quantize_grouped(x, offs, cfg=Config(), group_amax=None, codes=None, scales=None,
                     amax_given=None):
    """One call over a packed token tensor split into groups by cumulative
    ends offs (int32, device).  Rows past offs[-1] get zero codes/scales."""
    _cuda(x, "x")
    _cuda(offs, "offs")
    if offs.dtype != torch.int32:
        raise ValueError("offs must be int32")
    R, C = x.shape
    G = offs.numel()
    dev = x.device
    given = (group_amax is not None) if amax_given is None else bool(amax_given)
    if group_amax is None:
        group_amax = torch.empty(G, dtype=torch.float32, device=dev)
    if codes is None:
        codes = torch.empty((R, C // 2), dtype=torch.uint8, device=dev)
    if scales is None:
        scales = torch.empty(scales_shape(R, C, cfg.block16x16), dtype=torch.uint8, device=dev)
    cc = cfg.c(given)
    _check(lib().fos_quantize_grouped(_p(x), _DT[x.dtype], R, C, _p(offs), G, ctypes.byref(cc),
                                      _p(group_amax), _p(codes), _p(scales), _stream(x)),
           "fos_quantize_grouped")
    return codes, scales, group_amax


DIAG_E2M1_ENCODE, DIAG_E2M1_DECODE, DIAG_E4M3_ENCODE, DIAG_E4M3_DECODE = 0, 1, 2, 3
DIAG_F16_ROUND, DIAG_BF16_BITS, DIAG_F16_BITS, DIAG_DIV6 = 4, 5, 6, 7
DIAG_SCALE_CODES = 8


def diag_convert(op, inp, out):
    """Element-wise access to one device conversion primitive (fos_diag.h)."""
    _cuda(inp, "inp")
    _cuda(out, "out")
    _check(lib().fos_diag_convert(int(op), _p(inp), _p(out), inp.numel(), _stream(inp)),
           "fos_diag_convert")
    return out
