"""C-ABI library checks that need no GPU: it builds, loads, exports every
function the public headers declare, and rejects bad arguments on the host
before touching the CUDA runtime."""
import ctypes
import os
import re

import pytest

import nvfp4_quantization_precision_gb300 as fos
from nvfp4_quantization_precision_gb300 import build as fos_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    fos_build.build()
    return fos.lib()


def _declared():
    names = set()
    for h in ("fos.h", "fos_diag.h"):
        src = open(os.path.join(ROOT, "include", h)).read()
        names |= set(re.findall(r"FOS_API\s+[\w\s\*]+?\b(fos_\w+)\s*\(", src))
    return names


def test_headers_declare_the_entry_points():
    d = _declared()
    for n in ("fos_amax", "fos_quantize", "fos_quantize_list", "fos_quantize_overlap",
              "fos_dequantize", "fos_qdq", "fos_quantize_grouped",
              "fos_status_string", "fos_version", "fos_diag_convert"):
        assert n in d


def test_library_exports_every_declared_symbol(L):
    for n in _declared():
        assert hasattr(L, n), n
    # nothing else leaks out of the library's C namespace
    out = os.popen("nm -D --defined-only %s" % fos.LIB_PATH).read()
    exported = set(re.findall(r" T (fos_\w+)", out))
    assert exported == _declared()


def test_status_strings(L):
    assert fos.status_string(fos.FOS_OK) == "ok"
    assert "misaligned" in fos.status_string(fos.FOS_ERR_MISALIGNED)
    assert L.fos_version() == 10000


def _cfg(**kw):
    base = dict(block=0, mode=1, err_metric=1, err_precision=0, e4m3_bound=448, granularity=0,
                amax_is_input=1)
    base.update(kw)
    return fos.FosConfig(**base)


FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: every call below fails validation


@pytest.mark.parametrize("kw,rc", [
    (dict(block=2), fos.FOS_ERR_INVALID_ARG),
    (dict(mode=7), fos.FOS_ERR_INVALID_ARG),
    (dict(err_metric=-1), fos.FOS_ERR_INVALID_ARG),
    (dict(err_precision=3), fos.FOS_ERR_INVALID_ARG),
    (dict(granularity=2), fos.FOS_ERR_INVALID_ARG),
    (dict(amax_is_input=5), fos.FOS_ERR_INVALID_ARG),
    (dict(e4m3_bound=300), fos.FOS_ERR_UNSUPPORTED),
    (dict(err_order=2), fos.FOS_ERR_INVALID_ARG),
    (dict(block=1, err_order=1), fos.FOS_ERR_UNSUPPORTED),  # sequential order: 1x16 only
    (dict(scale_layout=2), fos.FOS_ERR_INVALID_ARG),
    (dict(scale_layout=-1), fos.FOS_ERR_INVALID_ARG),
    (dict(block=1, scale_layout=1), fos.FOS_ERR_UNSUPPORTED),  # tiled scales: 1x16 only
])
def test_quantize_rejects_bad_config(L, kw, rc):
    c = _cfg(**kw)
    assert L.fos_quantize(FAKE, 0, 16, 16, ctypes.byref(c), FAKE, FAKE, FAKE, None) == rc


@pytest.mark.parametrize("rows,cols,block,rc", [
    (-1, 16, 0, fos.FOS_ERR_INVALID_ARG),
    (16, -16, 0, fos.FOS_ERR_INVALID_ARG),
    (16, 24, 0, fos.FOS_ERR_UNSUPPORTED),
    (8, 16, 1, fos.FOS_ERR_UNSUPPORTED),
    (1 << 40, 1 << 20, 0, fos.FOS_ERR_UNSUPPORTED),
])
def test_quantize_rejects_bad_shape(L, rows, cols, block, rc):
    c = _cfg(block=block)
    assert L.fos_quantize(FAKE, 0, rows, cols, ctypes.byref(c), FAKE, FAKE, FAKE, None) == rc


def test_quantize_rejects_null_and_misaligned(L):
    c = _cfg()
    assert L.fos_quantize(None, 0, 16, 16, ctypes.byref(c), FAKE, FAKE, FAKE, None) == \
        fos.FOS_ERR_INVALID_ARG
    assert L.fos_quantize(FAKE, 9, 16, 16, ctypes.byref(c), FAKE, FAKE, FAKE, None) == \
        fos.FOS_ERR_INVALID_ARG
    assert L.fos_quantize(ctypes.c_void_p(0x10010), 0, 16, 16, ctypes.byref(c), FAKE, FAKE, FAKE,
                          None) == fos.FOS_ERR_MISALIGNED
    assert L.fos_quantize(FAKE, 0, 16, 16, ctypes.byref(c), FAKE, ctypes.c_void_p(0x10004), FAKE,
                          None) == fos.FOS_ERR_MISALIGNED
    assert L.fos_quantize(FAKE, 0, 16, 16, None, FAKE, FAKE, FAKE, None) == fos.FOS_ERR_INVALID_ARG


def test_grouped_rejects_bad_groups(L):
    c = _cfg()
    args = (FAKE, 0, 64, 64, FAKE)
    assert L.fos_quantize_grouped(*args, 0, ctypes.byref(c), FAKE, FAKE, FAKE, None) == \
        fos.FOS_ERR_INVALID_ARG
    assert L.fos_quantize_grouped(*args, fos.GROUPED_MAX_GROUPS + 1, ctypes.byref(c), FAKE, FAKE,
                                  FAKE, None) == fos.FOS_ERR_UNSUPPORTED
    assert L.fos_quantize_grouped(FAKE, 0, 64, 64, ctypes.c_void_p(0x10002), 4, ctypes.byref(c),
                                  FAKE, FAKE, FAKE, None) == fos.FOS_ERR_MISALIGNED


def test_qdq_rejects_unsupported(L):
    P = ctypes.c_void_p * 1
    xs, outs, am = P(FAKE.value), P(FAKE.value), P(FAKE.value)
    rows = (ctypes.c_int64 * 1)(16)
    cols = (ctypes.c_int64 * 1)(16)
    for kw in (dict(block=1), dict(granularity=1)):
        c = _cfg(**kw)
        assert L.fos_qdq(1, xs, outs, rows, cols, am, 0, ctypes.byref(c), None) == \
            fos.FOS_ERR_UNSUPPORTED
    c = _cfg()
    assert L.fos_qdq(1, xs, outs, rows, cols, am, 2, ctypes.byref(c), None) == \
        fos.FOS_ERR_UNSUPPORTED  # fp32 fused QDQ is not offered
    assert L.fos_qdq(-1, xs, outs, rows, cols, am, 0, ctypes.byref(c), None) == \
        fos.FOS_ERR_INVALID_ARG
    assert L.fos_qdq(0, None, None, None, None, None, 0, ctypes.byref(c), None) == fos.FOS_OK
    bad = (ctypes.c_int64 * 1)(24)
    assert L.fos_qdq(1, xs, outs, rows, bad, am, 0, ctypes.byref(c), None) == \
        fos.FOS_ERR_UNSUPPORTED


def test_dequantize_and_amax_and_diag_reject(L):
    c = _cfg()
    assert L.fos_dequantize(FAKE, FAKE, FAKE, 16, 16, ctypes.byref(c), FAKE, 7, None) == \
        fos.FOS_ERR_INVALID_ARG
    assert L.fos_dequantize(FAKE, FAKE, FAKE, 16, 16, ctypes.byref(c), ctypes.c_void_p(0x10008),
                            0, None) == fos.FOS_ERR_MISALIGNED
    assert L.fos_amax(FAKE, 0, 16, 16, 3, FAKE, None) == fos.FOS_ERR_INVALID_ARG
    assert L.fos_amax(FAKE, 0, 16, 17, 0, FAKE, None) == fos.FOS_ERR_UNSUPPORTED
    assert L.fos_diag_convert(99, FAKE, FAKE, 4, None) == fos.FOS_ERR_INVALID_ARG
    assert L.fos_diag_convert(0, FAKE, FAKE, 0, None) == fos.FOS_OK


def test_tiled_scales_only_where_the_quantize_writes_them(L):
    """The tiled layout is an output option of the 1x16 quantize calls; the
    grouped quantize and the dequantize take plain scales and refuse it on
    the host."""
    c = _cfg(scale_layout=1)
    assert L.fos_quantize_grouped(FAKE, 0, 32, 32, FAKE, 1, ctypes.byref(c), FAKE, FAKE, FAKE,
                                  None) == fos.FOS_ERR_UNSUPPORTED
    assert L.fos_dequantize(FAKE, FAKE, FAKE, 32, 32, ctypes.byref(c), FAKE, 0,
                            None) == fos.FOS_ERR_UNSUPPORTED
    c16 = _cfg(block=1, scale_layout=1)
    P = ctypes.c_void_p * 1
    rows, cols = (ctypes.c_int64 * 1)(32), (ctypes.c_int64 * 1)(32)
    assert L.fos_quantize_list(1, P(FAKE), 0, rows, cols, ctypes.byref(c16), P(FAKE), P(FAKE),
                               P(FAKE), None) == fos.FOS_ERR_UNSUPPORTED
    # block positions are 32-bit: tiled scales for fewer than 2^30 rows
    c = _cfg(scale_layout=1)
    assert L.fos_quantize(FAKE, 0, 1 << 30, 16, ctypes.byref(c), FAKE, FAKE, FAKE,
                          None) == fos.FOS_ERR_UNSUPPORTED
    assert fos.Config(scale_tiled=True).c(True).scale_layout == 1
    assert fos.Config().c(True).scale_layout == 0


def test_python_binding_refuses_cpu_tensors():
    import torch
    with pytest.raises(ValueError):
        fos.quantize(torch.zeros(16, 16, dtype=torch.bfloat16))


def test_quantize_list_rejects_before_launching(L):
    P = ctypes.c_void_p * 2
    xs, am, cs, ss = P(FAKE.value, FAKE.value), P(FAKE.value, FAKE.value), \
        P(FAKE.value, FAKE.value), P(FAKE.value, FAKE.value)
    rows = (ctypes.c_int64 * 2)(16, 16)
    cols = (ctypes.c_int64 * 2)(16, 24)  # the second entry is invalid
    c = _cfg(amax_is_input=0)
    assert L.fos_quantize_list(2, xs, 0, rows, cols, ctypes.byref(c), am, cs, ss, None) == \
        fos.FOS_ERR_UNSUPPORTED
    assert L.fos_quantize_list(-1, xs, 0, rows, cols, ctypes.byref(c), am, cs, ss, None) == \
        fos.FOS_ERR_INVALID_ARG
    assert L.fos_quantize_list(0, None, 0, None, None, ctypes.byref(c), None, None, None,
                               None) == fos.FOS_OK


def test_quantize_overlap_requires_given_per_tensor_1x16(L):
    for kw in (dict(block=1), dict(granularity=1), dict(amax_is_input=0)):
        c = _cfg(**kw)
        assert L.fos_quantize_overlap(FAKE, 0, 16, 16, ctypes.byref(c), FAKE, FAKE, FAKE, FAKE,
                                      16, 16, FAKE, None) == fos.FOS_ERR_UNSUPPORTED
    c = _cfg()
    assert L.fos_quantize_overlap(FAKE, 0, 16, 16, ctypes.byref(c), FAKE, FAKE, FAKE,
                                  ctypes.c_void_p(0x10010), 16, 16, FAKE, None) == \
        fos.FOS_ERR_MISALIGNED
    assert L.fos_quantize_overlap(FAKE, 0, 16, 16, ctypes.byref(c), FAKE, FAKE, FAKE, FAKE,
                                  16, 20, FAKE, None) == fos.FOS_ERR_UNSUPPORTED


def test_qdq_fused_workspace_size(L):
    assert L.fos_qdq_fused_workspace_bytes(0) == 0
    assert L.fos_qdq_fused_workspace_bytes(1) == 256
    assert L.fos_qdq_fused_workspace_bytes(64) == 768  # (1 + 2 * 64) words, rounded to 256 B


def test_qdq_fused_rejects_before_any_cuda_call(L):
    P1 = ctypes.c_void_p * 1
    x, o, a = P1(FAKE), P1(FAKE), P1(FAKE)
    rows, cols = (ctypes.c_int64 * 1)(16), (ctypes.c_int64 * 1)(16)
    ws = ctypes.c_void_p(0x100000)

    def call(n=1, cfg=None, w=ws, nbytes=256, dt=0):
        c = cfg or _cfg(amax_is_input=0)
        return L.fos_qdq_fused(n, x, o, rows, cols, a, dt, ctypes.byref(c), w, nbytes, None)
    assert call(cfg=_cfg(amax_is_input=1)) == fos.FOS_ERR_UNSUPPORTED  # the amax is computed
    assert call(cfg=_cfg(amax_is_input=0, block=1)) == fos.FOS_ERR_UNSUPPORTED
    assert call(cfg=_cfg(amax_is_input=0, granularity=1)) == fos.FOS_ERR_UNSUPPORTED
    assert call(dt=2) == fos.FOS_ERR_UNSUPPORTED                      # fp32
    assert call(n=65) == fos.FOS_ERR_UNSUPPORTED                       # above FOS_QDQ_MAX_LIST
    assert call(n=-1) == fos.FOS_ERR_INVALID_ARG
    assert call(w=None) == fos.FOS_ERR_INVALID_ARG
    assert call(nbytes=255) == fos.FOS_ERR_INVALID_ARG                 # workspace too small
    assert call(w=ctypes.c_void_p(0x100080)) == fos.FOS_ERR_MISALIGNED
    assert call(n=0) == fos.FOS_OK


def test_qdq_fused_static_rejects_like_the_workspace_form_before_any_cuda_call(L):
    """fos_qdq_fused_static runs the host checks of fos_qdq_fused in the same
    order (dtype and configuration before the list length), before it
    resolves a device or its fixed array."""
    P1 = ctypes.c_void_p * 1
    x, o, a = P1(FAKE), P1(FAKE), P1(FAKE)
    rows, cols = (ctypes.c_int64 * 1)(16), (ctypes.c_int64 * 1)(16)

    def call(n=1, cfg=None, dt=0, amax=a, nullcfg=False):
        c = cfg or _cfg(amax_is_input=0)
        return L.fos_qdq_fused_static(n, x, o, rows, cols, amax, dt,
                                      None if nullcfg else ctypes.byref(c), None)
    assert call(cfg=_cfg(amax_is_input=1)) == fos.FOS_ERR_UNSUPPORTED
    assert call(cfg=_cfg(amax_is_input=0, block=1)) == fos.FOS_ERR_UNSUPPORTED
    assert call(cfg=_cfg(amax_is_input=0, granularity=1)) == fos.FOS_ERR_UNSUPPORTED
    assert call(dt=2) == fos.FOS_ERR_UNSUPPORTED
    assert call(n=65) == fos.FOS_ERR_UNSUPPORTED
    assert call(n=-1) == fos.FOS_ERR_INVALID_ARG
    # bad dtype / config win over the list length, like fos_qdq_fused
    assert call(n=0, dt=7) == fos.FOS_ERR_INVALID_ARG
    assert call(n=0, nullcfg=True) == fos.FOS_ERR_INVALID_ARG
    assert call(n=65, dt=7) == fos.FOS_ERR_INVALID_ARG
    assert call(n=0, cfg=_cfg(amax_is_input=0, e4m3_bound=100)) == fos.FOS_ERR_UNSUPPORTED
    assert call(amax=P1(None)) == fos.FOS_ERR_INVALID_ARG
    c2 = (ctypes.c_int64 * 1)(24)
    assert L.fos_qdq_fused_static(1, x, o, rows, c2, a, 0, ctypes.byref(_cfg(amax_is_input=0)),
                                  None) == fos.FOS_ERR_UNSUPPORTED
    mis = P1(ctypes.c_void_p(0x10010))
    assert L.fos_qdq_fused_static(1, mis, o, rows, cols, a, 0,
                                  ctypes.byref(_cfg(amax_is_input=0)), None) == \
        fos.FOS_ERR_MISALIGNED
    assert call(n=0) == fos.FOS_OK
    for n in (0, 1, 65):
        for dt in (0, 1, 2, 7):
            want = L.fos_qdq_fused(n, x, o, rows, cols, a, dt,
                                   ctypes.byref(_cfg(amax_is_input=0)),
                                   ctypes.c_void_p(0x100000), 1 << 20, None)
            got = call(n=n, dt=dt)
            if want != fos.FOS_OK or n == 0:
                assert got == want, (n, dt, got, want)


def test_workspace_error_rejects_null(L):
    code = ctypes.c_int(7)
    assert L.fos_workspace_error(None, None, ctypes.byref(code)) == fos.FOS_ERR_INVALID_ARG


def test_quantize_colwise_rejects_before_any_cuda_call(L):
    L.fos_quantize_colwise.restype = ctypes.c_int
    c = _cfg()

    def call(rows=32, cols=32, cfg=c, codes=FAKE, scales=FAKE):
        return L.fos_quantize_colwise(FAKE, 0, ctypes.c_int64(rows), ctypes.c_int64(cols),
                                      ctypes.byref(cfg), FAKE, FAKE, FAKE, codes, scales, None)
    assert call(rows=24) == fos.FOS_ERR_UNSUPPORTED          # blocks of x^T run down the rows
    assert call(cols=24) == fos.FOS_ERR_UNSUPPORTED
    assert call(cfg=_cfg(block=1)) == fos.FOS_ERR_UNSUPPORTED
    assert call(cfg=_cfg(granularity=1)) == fos.FOS_ERR_UNSUPPORTED
    assert call(codes=None) == fos.FOS_ERR_INVALID_ARG        # codes and scales go together


def test_diag_wait_timeout_rejects_bad_arguments(L):
    L.fos_diag_wait_timeout.restype = ctypes.c_int
    assert L.fos_diag_wait_timeout(2, FAKE, None) == fos.FOS_ERR_INVALID_ARG
    assert L.fos_diag_wait_timeout(0, None, None) == fos.FOS_ERR_INVALID_ARG
    assert L.fos_diag_wait_timeout(0, ctypes.c_void_p(0x10002), None) == fos.FOS_ERR_MISALIGNED


def test_mm_rejects_before_any_cuda_call(L):
    L.fos_mm.restype = ctypes.c_int
    c = _cfg()
    i64 = ctypes.c_int64

    def call(M=16, N=16, K=64, cfg=c, a=FAKE):
        return L.fos_mm(a, FAKE, FAKE, FAKE, FAKE, FAKE, i64(M), i64(N), i64(K), ctypes.byref(cfg),
                        FAKE, None)
    assert call(K=48) == fos.FOS_ERR_UNSUPPORTED
    assert call(M=8) == fos.FOS_ERR_UNSUPPORTED
    assert call(cfg=_cfg(block=1)) == fos.FOS_ERR_UNSUPPORTED
    assert call(M=-16) == fos.FOS_ERR_INVALID_ARG
    assert call(a=None) == fos.FOS_ERR_INVALID_ARG
    assert call(a=ctypes.c_void_p(0x10008)) == fos.FOS_ERR_MISALIGNED
    assert call(M=0) == fos.FOS_OK


def test_check_tile_amax_rejects_before_any_cuda_call(L):
    i64 = ctypes.c_int64
    assert "tile" in fos.status_string(fos.FOS_ERR_NONUNIFORM_TILE_AMAX)
    assert L.fos_check_tile_amax(FAKE, i64(24), FAKE, None) == fos.FOS_ERR_UNSUPPORTED
    assert L.fos_check_tile_amax(FAKE, i64(-16), FAKE, None) == fos.FOS_ERR_INVALID_ARG
    assert L.fos_check_tile_amax(None, i64(16), FAKE, None) == fos.FOS_ERR_INVALID_ARG
    assert L.fos_check_tile_amax(FAKE, i64(16), None, None) == fos.FOS_ERR_INVALID_ARG
    assert L.fos_check_tile_amax(ctypes.c_void_p(0x10002), i64(16), FAKE,
                                 None) == fos.FOS_ERR_MISALIGNED
    assert L.fos_check_tile_amax(FAKE, i64(16), ctypes.c_void_p(0x10004),
                                 None) == fos.FOS_ERR_MISALIGNED
    assert L.fos_tile_amax_status(None, None) == fos.FOS_ERR_INVALID_ARG


C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "fos.h"
#include "fos_diag.h"
int main(void) {
    fos_config cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.e4m3_bound = 448;
    /* host validation only: a 24-column tensor is rejected before any CUDA call */
    fos_status st = fos_quantize((const void*)0x10000, FOS_BF16, 32, 24, &cfg, 0, 0, 0, 0);
    printf("%d %d %s\n", fos_version(), (int)st, fos_status_string(st));
    return st == FOS_ERR_UNSUPPORTED ? 0 : 1;
}
"""


@pytest.mark.parametrize("lang", ["c", "c++"])
def test_headers_compile_and_link_from_plain_c(L, tmp_path, lang):
    """The public headers stand alone in C99 and C++17, and a plain C program
    links against the library and calls it (host-side calls only)."""
    import subprocess
    src = tmp_path / ("prog.c" if lang == "c" else "prog.cpp")
    src.write_text(C_PROGRAM)
    exe = tmp_path / "prog"
    cc = ["gcc", "-std=c99"] if lang == "c" else ["g++", "-std=c++17"]
    libdir = os.path.dirname(fos.LIB_PATH)
    r = subprocess.run(cc + ["-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                             str(src), "-o", str(exe), "-L", libdir, "-lfos",
                             "-Wl,-rpath," + libdir], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.split()[0] == "10000"


def test_swizzled_scales_bytes_matches_the_oracle_layout(L):
    """The host-side size of the tiled scale layout equals the size of the
    oracle's layout for the same scale matrix; bad shapes give -1."""
    import numpy as np

    import oracle
    L.fos_swizzled_scales_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64]
    L.fos_swizzled_scales_bytes.restype = ctypes.c_int64
    for rows, cols in [(1, 16), (127, 48), (128, 64), (129, 80), (300, 144), (8192, 4096)]:
        want = oracle.swizzle_scales(np.zeros((rows, cols // 16), np.uint8)).size
        assert L.fos_swizzled_scales_bytes(rows, cols) == want, (rows, cols)
    assert L.fos_swizzled_scales_bytes(0, 64) == 0
    for rows, cols in [(-1, 16), (16, -16), (16, 24)]:
        assert L.fos_swizzled_scales_bytes(rows, cols) == -1


def test_host_validation_fuzz_never_crashes(L):
    """Seeded random argument sets (negative, zero, ragged and huge sizes,
    invalid enums, null, fake and misaligned pointers) for every data entry
    point: each call returns a defined status and nothing crashes.  No GPU is
    present, so a call that passes validation stops at the pointer check."""
    import random
    rng = random.Random(12345)
    i64 = ctypes.c_int64
    sizes = [-16, -1, 0, 1, 15, 16, 17, 32, 48, 4096, 1 << 40, (1 << 62)]
    ptrs = [None, FAKE, ctypes.c_void_p(0x10001), ctypes.c_void_p(0x10010)]
    for n in ("fos_quantize", "fos_dequantize", "fos_quantize_grouped", "fos_quantize_colwise",
              "fos_swizzle_scales", "fos_check_tile_amax", "fos_mm", "fos_amax",
              "fos_qdq_fused", "fos_qdq_fused_static"):
        getattr(L, n).restype = ctypes.c_int
    valid = set(range(6))
    for _ in range(400):
        cfg = _cfg(block=rng.choice([0, 1, 2]), mode=rng.choice([0, 1, 3]),
                   err_metric=rng.choice([0, 1, -1]), err_precision=rng.choice([0, 1, 2]),
                   e4m3_bound=rng.choice([448, 256, 100]), granularity=rng.choice([0, 1, 5]),
                   amax_is_input=rng.choice([0, 1, 2]), err_order=rng.choice([0, 1, 9]))
        R, C = i64(rng.choice(sizes)), i64(rng.choice(sizes))
        p = [rng.choice(ptrs) for _ in range(6)]
        dt = rng.choice([0, 1, 2, 7])
        rcs = [
            L.fos_quantize(p[0], dt, R, C, ctypes.byref(cfg), p[1], p[2], p[3], None),
            L.fos_dequantize(p[0], p[1], p[2], R, C, ctypes.byref(cfg), p[3], dt, None),
            L.fos_quantize_grouped(p[0], dt, R, C, p[1], rng.choice([-1, 0, 1, 64, 9000]),
                                   ctypes.byref(cfg), p[2], p[3], p[4], None),
            L.fos_quantize_colwise(p[0], dt, R, C, ctypes.byref(cfg), p[1], p[2], p[3], p[4],
                                   p[5], None),
            L.fos_swizzle_scales(p[0], R, C, p[1], None),
            L.fos_check_tile_amax(p[0], R, p[1], None),
            L.fos_mm(p[0], p[1], p[2], p[3], p[4], p[5], R, C, i64(rng.choice(sizes)),
                     ctypes.byref(cfg), p[0], None),
            L.fos_amax(p[0], dt, R, C, rng.choice([0, 1, 4]), p[1], None),
        ]
        n = rng.choice([-1, 0, 1, 2, 64, 65])
        k = max(n, 1)
        P = ctypes.c_void_p * k
        xs, os_, am = (P(*[rng.choice(ptrs) for _ in range(k)]) for _ in range(3))
        rr = (i64 * k)(*[rng.choice(sizes) for _ in range(k)])
        cc = (i64 * k)(*[rng.choice(sizes) for _ in range(k)])
        rcs.append(L.fos_qdq_fused_static(n, xs, os_, rr, cc, am, dt, ctypes.byref(cfg), None))
        rcs.append(L.fos_qdq_fused(n, xs, os_, rr, cc, am, dt, ctypes.byref(cfg), p[5],
                                   rng.choice([0, 256, 1 << 20]), None))
        assert all(rc in valid for rc in rcs), rcs
