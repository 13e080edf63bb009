"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle on
identical seeded bytes.  Tolerance 0 everywhere: codes, scales, amax and
outputs are compared as integer views, so signed zeros and NaN payloads of
the outputs count."""
import ctypes
import itertools

import numpy as np
import pytest
import torch

import nvfp4_quantization_precision_gb300 as fos
import oracle
import workloads

pytestmark = pytest.mark.gpu

DEV = "cuda"
DTYPES = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}
MODES = {  # name -> (four_over_six, mse, err_f16)
    "std": (False, True, False),
    "mae": (True, False, False),
    "mse": (True, True, False),
    "mae_f16": (True, False, True),
    "mse_f16": (True, True, True),
}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _cfgs(mode, bound=448, row=False, b16=False, seq=False):
    f, m, h = MODES[mode]
    return (fos.Config(block16x16=b16, four_over_six=f, mse=m, err_f16=h, bound=bound,
                       row_scaled=row, seq_order=seq),
            oracle.Config(block16x16=b16, four_over_six=f, mse=m, err_f16=h, bound=bound,
                          row_scaled=row, seq_order=seq))


def _u16(t):
    return t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _u32(t):
    return t.cpu().contiguous().view(torch.int32).numpy().view(np.uint32)


def _x(rows, cols, fam, seed, dt):
    return workloads.activation(rows, cols, fam, seed=seed, dtype=DTYPES[dt])


def _check_quant(x, gcfg, ocfg, amax_given):
    """Run both sides; amax either computed by each side or given (oracle's)."""
    xf = x.float().numpy()
    if amax_given:
        a = oracle.amax_rows(xf) if ocfg.row_scaled else oracle.amax_tensor(xf)
        ocfg = oracle.Config(**{**ocfg.__dict__, "amax_is_input": True})
        oc, os_, oa = oracle.quantize(xf, ocfg, amax=a)
        gc, gs, ga = fos.quantize(x.to(DEV), gcfg, amax=torch.from_numpy(a).to(DEV))
    else:
        oc, os_, oa = oracle.quantize(xf, ocfg)
        gc, gs, ga = fos.quantize(x.to(DEV), gcfg)
    torch.cuda.synchronize()
    assert np.array_equal(_u32(ga), oa.view(np.uint32)), "amax"
    gcn, gsn = gc.cpu().numpy(), gs.cpu().numpy()
    if not np.array_equal(gsn, os_):
        bad = np.argwhere(gsn != os_)
        raise AssertionError("scales differ at %d places, first %s: gpu %#x oracle %#x" % (
            len(bad), bad[0], gsn[tuple(bad[0])], os_[tuple(bad[0])]))
    if not np.array_equal(gcn, oc):
        bad = np.argwhere(gcn != oc)
        raise AssertionError("codes differ at %d places, first %s" % (len(bad), bad[0]))
    return gc, gs, ga


# ------------------------------------------------------------------ 1x16
@pytest.mark.parametrize("dt,mode,bound,row", list(itertools.product(
    ["bf16", "f16", "f32"], list(MODES), [448, 256], [False, True])))
def test_quantize_1x16_knobs(dt, mode, bound, row):
    gcfg, ocfg = _cfgs(mode, bound, row)
    for i, (fam, shape) in enumerate(zip(workloads.FAMILIES,
                                         [(256, 1024), (48, 272), (7, 1040), (33, 528)])):
        x = _x(*shape, fam, seed=i, dt=dt)
        _check_quant(x, gcfg, ocfg, amax_given=(i % 2 == 1))


@pytest.mark.parametrize("shape", [(1, 16), (3, 16), (1, 512), (5, 496), (2, 8192), (129, 32)])
def test_quantize_1x16_ragged_shapes(shape):
    for mode in ("std", "mse", "mae_f16"):
        for row in (False, True):
            gcfg, ocfg = _cfgs(mode, 448, row)
            _check_quant(_x(*shape, "F4", 3, "bf16"), gcfg, ocfg, amax_given=False)


def test_quantize_pr1_config():
    # one 256x1024 bf16 tensor, N(0,1), per-tensor amax, E4M3 448, MSE exact
    gcfg, ocfg = _cfgs("mse", 448, False)
    for seed in (0, 1, 2):
        _check_quant(_x(256, 1024, "F1", seed, "bf16"), gcfg, ocfg, amax_given=False)


# ------------------------------------------------------------------ 16x16
@pytest.mark.parametrize("dt,mode,bound,row", list(itertools.product(
    ["bf16", "f16", "f32"], list(MODES), [448, 256], [False, True])))
def test_quantize_16x16_knobs(dt, mode, bound, row):
    gcfg, ocfg = _cfgs(mode, bound, row, b16=True)
    for i, shape in enumerate([(64, 272), (32, 1024), (16, 16)]):
        x = workloads.weight(*shape, seed=i, dtype=DTYPES[dt])
        if row:  # per-row amax made tile-uniform (the contract for 16x16)
            xf = x.float().numpy()
            a = np.repeat(oracle.amax_rows(xf).reshape(-1, 16).max(1), 16)
            ocfg2 = oracle.Config(**{**ocfg.__dict__, "amax_is_input": True})
            oc, os_, _ = oracle.quantize(xf, ocfg2, amax=a)
            gc, gs, _ = fos.quantize(x.to(DEV), gcfg, amax=torch.from_numpy(a).to(DEV))
            torch.cuda.synchronize()
            assert np.array_equal(gs.cpu().numpy(), os_)
            assert np.array_equal(gc.cpu().numpy(), oc)
        else:
            _check_quant(x, gcfg, ocfg, amax_given=(i == 1))


def test_16x16_row_amax_uses_first_tile_row():
    # non-uniform per-row amax: every tile takes its first row's value
    x = workloads.weight(64, 256, seed=5, dtype=torch.bfloat16)
    xf = x.float().numpy()
    a = oracle.amax_rows(xf)
    gcfg, ocfg = _cfgs("mse", 448, True, b16=True)
    ocfg = oracle.Config(**{**ocfg.__dict__, "amax_is_input": True})
    oc, os_, _ = oracle.quantize(xf, ocfg, amax=a)
    gc, gs, _ = fos.quantize(x.to(DEV), gcfg, amax=torch.from_numpy(a).to(DEV))
    torch.cuda.synchronize()
    assert np.array_equal(gs.cpu().numpy(), os_) and np.array_equal(gc.cpu().numpy(), oc)



@pytest.mark.parametrize("rows", [0, 16, 4096, 16 * 200003])
def test_check_tile_amax_counts_like_the_oracle(rows):
    """fos_check_tile_amax against the oracle's count on seeded per-row
    amaxes: uniform tiles with a seeded set of tiles broken (a changed row,
    a row of -0 in a tile of +0), over a grid larger than one pass."""
    rng = np.random.default_rng(rows)
    tiles = rows // 16
    a = np.repeat(rng.uniform(0.5, 4.0, tiles).astype(np.float32), 16)
    if tiles:
        a[:16] = 0.0
        broken = rng.choice(tiles, size=max(1, tiles // 7), replace=False)
        for t in broken:
            r = 16 * int(t) + int(rng.integers(16))
            a[r] = -0.0 if a[r] == 0.0 else np.nextafter(a[r], np.float32(9))
    want = oracle.count_nonuniform_tiles(a)
    assert fos.check_tile_amax(torch.from_numpy(a).to(DEV)) == want
    bad = torch.empty(1, dtype=torch.int64, device=DEV)
    L = fos.lib()
    assert L.fos_check_tile_amax(ctypes.c_void_p(torch.from_numpy(a).to(DEV).data_ptr()) if rows
                                 else ctypes.c_void_p(0), ctypes.c_int64(rows),
                                 ctypes.c_void_p(bad.data_ptr()), None) == fos.FOS_OK
    assert L.fos_tile_amax_status(ctypes.c_void_p(bad.data_ptr()), None) == (
        fos.FOS_OK if want == 0 else fos.FOS_ERR_NONUNIFORM_TILE_AMAX)


def test_quantize_validate_rejects_a_nonuniform_tile_amax():
    """quantize(validate=True) of 16x16 blocks with a given per-row amax:
    raises FOS_ERR_NONUNIFORM_TILE_AMAX when one tile's rows differ and
    writes nothing; with tile-uniform amax it equals the oracle."""
    x = workloads.weight(64, 256, seed=5, dtype=torch.bfloat16)
    xf = x.float().numpy()
    gcfg, ocfg = _cfgs("mse", 448, True, b16=True)
    a = np.repeat(oracle.amax_rows(xf).reshape(4, 16).max(axis=1), 16).astype(np.float32)
    ocfg = oracle.Config(**{**ocfg.__dict__, "amax_is_input": True})
    oc, os_, _ = oracle.quantize(xf, ocfg, amax=a)
    gc, gs, _ = fos.quantize(x.to(DEV), gcfg, amax=torch.from_numpy(a).to(DEV), validate=True)
    torch.cuda.synchronize()
    assert np.array_equal(gs.cpu().numpy(), os_) and np.array_equal(gc.cpu().numpy(), oc)
    a[37] *= 2
    codes = torch.full((64, 128), 0x5A, dtype=torch.uint8, device=DEV)
    with pytest.raises(fos.FosError) as e:
        fos.quantize(x.to(DEV), gcfg, amax=torch.from_numpy(a).to(DEV), codes=codes,
                     validate=True)
    assert e.value.status == fos.FOS_ERR_NONUNIFORM_TILE_AMAX
    assert bool((codes == 0x5A).all())

# ------------------------------------------------------------------ special values
def _special_tensor(dt):
    rng = np.random.default_rng(0)
    x = rng.standard_normal((64, 64)).astype(np.float32)
    x[0, :16] = np.nan                     # all-NaN block
    x[1, 3] = np.nan                       # one NaN
    x[2, 0] = np.inf
    x[3, 5] = -np.inf
    x[4, :16] = 0.0
    x[5, :16] = -0.0
    x[6, :16] *= 1e-7                      # scale underflows E4M3
    x[7, :16] = np.float32(2.0 ** -130)    # subnormal f32 (bf16 keeps it)
    x[8, :16] = 6.0                        # exact grid values
    x[9, :16] = np.array([0.5, 1, 1.5, 2, 3, 4, 6, 0] * 2, np.float32)
    x[10, :] = 1e30 if dt != "f16" else 6e4
    x[11, 16:32] = -x[11, 16:32]
    return torch.from_numpy(x).to(DTYPES[dt])


@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("row", [False, True])
def test_special_values(dt, mode, row):
    gcfg, ocfg = _cfgs(mode, 448, row)
    _check_quant(_special_tensor(dt), gcfg, ocfg, amax_given=False)
    # the same rows with amax given as extreme values
    x = _special_tensor(dt)
    n = x.shape[0] if row else 1
    for aval in (0.0, float("inf"), 1e-38, 3e38, float("nan"), -1.0):
        a = np.full(n, aval, np.float32)
        ocfg2 = oracle.Config(**{**ocfg.__dict__, "amax_is_input": True})
        oc, os_, _ = oracle.quantize(x.float().numpy(), ocfg2, amax=a)
        gc, gs, _ = fos.quantize(x.to(DEV), gcfg, amax=torch.from_numpy(a).to(DEV))
        torch.cuda.synchronize()
        assert np.array_equal(gs.cpu().numpy(), os_), aval
        assert np.array_equal(gc.cpu().numpy(), oc), aval


# ------------------------------------------------------------------ dequantize
@pytest.mark.parametrize("out", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("b16", [False, True])
@pytest.mark.parametrize("row", [False, True])
def test_dequantize(out, b16, row):
    rng = np.random.default_rng(3)
    R, C = 48, 272
    codes = rng.integers(0, 256, (R, C // 2), dtype=np.uint8)
    srows = R // 16 if b16 else R
    scales = rng.integers(0, 0x7F, (srows, C // 16), dtype=np.uint8)
    a = rng.uniform(0.01, 100, R if row else 1).astype(np.float32)
    if row and b16:
        a = np.repeat(a[::16], 16)
    ocfg = oracle.Config(block16x16=b16, row_scaled=row, bound=256)
    gcfg = fos.Config(block16x16=b16, row_scaled=row, bound=256)
    ref = oracle.dequantize(codes, scales, a, ocfg, out)
    got = fos.dequantize(torch.from_numpy(codes).to(DEV), torch.from_numpy(scales).to(DEV),
                         torch.from_numpy(a).to(DEV), gcfg, out_dtype=DTYPES[out])
    torch.cuda.synchronize()
    g = _u32(got) if out == "f32" else _u16(got)
    assert np.array_equal(g, ref.view(g.dtype))


def test_dequantize_all_scale_codes():
    codes = np.tile(np.arange(256, dtype=np.uint8).reshape(1, 256)[:, :8], (256, 1))
    scales = np.arange(256, dtype=np.uint8).reshape(256, 1)
    a = np.array([7.0], np.float32)
    ocfg, gcfg = oracle.Config(), fos.Config()
    ref = oracle.dequantize(codes, scales, a, ocfg, "f32")
    got = fos.dequantize(torch.from_numpy(codes).to(DEV), torch.from_numpy(scales).to(DEV),
                         torch.from_numpy(a).to(DEV), gcfg, out_dtype=torch.float32).cpu().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


# ------------------------------------------------------------------ fused QDQ
@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("bound", [448, 256])
def test_qdq_list(dt, mode, bound):
    gcfg, ocfg = _cfgs(mode, bound)
    shapes = [(64, 1024), (0, 64), (7, 1040), (48, 272), (1, 16)]
    xs = [workloads.qdq_weights(1, r, c, seed=i, dtype=DTYPES[dt])[0] if r else
          torch.zeros(0, c, dtype=DTYPES[dt]) for i, (r, c) in enumerate(shapes)]
    outs = fos.qdq([x.to(DEV) for x in xs], gcfg)
    torch.cuda.synchronize()
    for x, o in zip(xs, outs):
        if x.numel() == 0:
            continue
        ref, _ = oracle.qdq(x.float().numpy(), ocfg, dt)
        assert np.array_equal(_u16(o), ref)


def test_qdq_equals_dequantize_of_quantize_on_gpu():
    gcfg, _ = _cfgs("mse_f16", 256)
    x = workloads.qdq_weights(1, 128, 7168, seed=4)[0].to(DEV)
    a = fos.amax(x)
    q = fos.qdq([x], gcfg, amaxes=[a])[0]
    c, s, _ = fos.quantize(x, gcfg, amax=a)
    d = fos.dequantize(c, s, a, gcfg, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(q.view(torch.int16), d.view(torch.int16))


def test_qdq_long_list_splits_launches():
    gcfg, ocfg = _cfgs("mae", 448)
    xs = [workloads.qdq_weights(1, 2, 32, seed=i)[0] for i in range(fos.QDQ_MAX_LIST + 5)]
    outs = fos.qdq([x.to(DEV) for x in xs], gcfg)
    torch.cuda.synchronize()
    for x, o in zip(xs, outs):
        ref, _ = oracle.qdq(x.float().numpy(), ocfg, "bf16")
        assert np.array_equal(_u16(o), ref)


# ------------------------------------------------------------------ grouped
@pytest.mark.parametrize("b16", [False, True])
@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("mode", ["std", "mse", "mae_f16"])
@pytest.mark.parametrize("given", [False, True])
def test_grouped(b16, dt, mode, given):
    R, C = 512, 272
    offs = workloads.moe_offsets(R, 12, seed=1, n_empty=3, multiple=16 if b16 else 1)
    x = workloads.moe_activations(R, C, offs, seed=2, dtype=DTYPES[dt])
    gcfg, ocfg = _cfgs(mode, 448, b16=b16)
    xf = x.float().numpy()
    on = offs.numpy()
    if given:
        ga_in = oracle.amax_groups(xf, on)
        ocfg = oracle.Config(**{**ocfg.__dict__, "amax_is_input": True})
        oc, os_, oa = oracle.quantize_grouped(xf, on, ocfg, group_amax=ga_in)
        gc, gs, ga = fos.quantize_grouped(x.to(DEV), offs.to(DEV), gcfg,
                                          group_amax=torch.from_numpy(ga_in).to(DEV))
    else:
        oc, os_, oa = oracle.quantize_grouped(xf, on, ocfg)
        gc, gs, ga = fos.quantize_grouped(x.to(DEV), offs.to(DEV), gcfg)
    torch.cuda.synchronize()
    assert np.array_equal(_u32(ga), oa.view(np.uint32))
    assert np.array_equal(gs.cpu().numpy(), os_)
    assert np.array_equal(gc.cpu().numpy(), oc)


def test_grouped_bad_offs_are_clamped_like_the_oracle():
    R, C = 64, 64
    x = _x(R, C, "F1", 9, "bf16")
    offs = np.array([10, 5, 40, 200, 30], np.int32)  # non-monotone and past the end
    gcfg, ocfg = _cfgs("mse")
    oc, os_, oa = oracle.quantize_grouped(x.float().numpy(), offs, ocfg)
    gc, gs, ga = fos.quantize_grouped(x.to(DEV), torch.from_numpy(offs).to(DEV), gcfg)
    torch.cuda.synchronize()
    assert np.array_equal(_u32(ga), oa.view(np.uint32))
    assert np.array_equal(gs.cpu().numpy(), os_) and np.array_equal(gc.cpu().numpy(), oc)


def test_grouped_equals_per_group_gpu_calls():
    R, C = 1024, 512
    offs = workloads.moe_offsets(R, 16, seed=3)
    x = workloads.moe_activations(R, C, offs, seed=4).to(DEV)
    gcfg, _ = _cfgs("mse")
    gc, gs, ga = fos.quantize_grouped(x, offs.to(DEV), gcfg)
    lo = 0
    for g, hi in enumerate(offs.tolist()):
        if hi > lo:
            c, s, a = fos.quantize(x[lo:hi].contiguous(), gcfg)
            torch.cuda.synchronize()
            assert torch.equal(a[0], ga[g])
            assert torch.equal(c, gc[lo:hi]) and torch.equal(s, gs[lo:hi])
        lo = hi
    assert bool((gc[lo:] == 0).all()) and bool((gs[lo:] == 0).all())


# ------------------------------------------------------------------ amax
@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
def test_amax(dt):
    x = _special_tensor(dt)
    xf = x.float().numpy()
    g = fos.amax(x.to(DEV))
    r = fos.amax(x.to(DEV), row_scaled=True)
    torch.cuda.synchronize()
    assert np.array_equal(_u32(g), oracle.amax_tensor(xf).view(np.uint32))
    assert np.array_equal(_u32(r), oracle.amax_rows(xf).view(np.uint32))


# ------------------------------------------------------------------ primitives
def _dense_f32(n_random=1 << 22, seed=0):
    rng = np.random.default_rng(seed)
    top = (np.arange(0, 1 << 16, dtype=np.uint32) << 16)
    lows = np.array([0, 1, 0x7FFF, 0x8000, 0x8001, 0xFFFF], np.uint32)
    dense = (top[:, None] | lows[None, :]).ravel()
    rand = rng.integers(0, 1 << 32, n_random, dtype=np.uint64).astype(np.uint32)
    return np.concatenate([dense, rand]).view(np.float32)


def _run_diag(op, arr, out_dtype):
    inp = torch.from_numpy(arr).to(DEV)
    out = torch.empty(arr.size, dtype=out_dtype, device=DEV)
    fos.diag_convert(op, inp, out)
    torch.cuda.synchronize()
    return out.cpu()


def test_diag_e2m1_encode_matches_oracle():
    v = _dense_f32()
    got = _run_diag(fos.DIAG_E2M1_ENCODE, v, torch.uint8).numpy()
    ref = oracle.e2m1_encode(v)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(hex(v.view(np.uint32)[i]), hex(got[i]), hex(ref[i])) for i in bad[:8]]


def test_diag_e2m1_decode_all_codes():
    codes = np.arange(16, dtype=np.uint8)
    got = _run_diag(fos.DIAG_E2M1_DECODE, codes, torch.float32).numpy()
    ref = np.array([oracle.e2m1_value(c) for c in range(16)], np.float32)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_diag_e4m3_encode_matches_oracle():
    v = _dense_f32(1 << 20, seed=1)
    got = _run_diag(fos.DIAG_E4M3_ENCODE, v, torch.uint8).numpy()
    ref = oracle.e4m3_encode(v)
    nan = np.isnan(v)
    # NaN inputs never reach the E4M3 cast on the quantize path; compare NaN-ness only
    assert ((got[nan] & 0x7F) == 0x7F).all()
    bad = np.nonzero((got != ref) & ~nan)[0]
    assert bad.size == 0, [(float(v[i]), hex(got[i]), hex(ref[i])) for i in bad[:8]]


def test_diag_e4m3_decode_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    got = _run_diag(fos.DIAG_E4M3_DECODE, codes, torch.float32).numpy()
    ref = np.array([oracle.e4m3_value(c) for c in range(256)], np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_diag_f16_and_bf16_rounding():
    v = _dense_f32(1 << 20, seed=2)
    v = v[~np.isnan(v)]
    v = v[: v.size // 2 * 2]
    got = _run_diag(fos.DIAG_F16_ROUND, v, torch.float32).numpy()
    assert np.array_equal(got.view(np.uint32), oracle.f16_round(v).view(np.uint32))
    got = _run_diag(fos.DIAG_F16_BITS, v, torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, oracle.f16_bits(v))
    got = _run_diag(fos.DIAG_BF16_BITS, v, torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, oracle.bf16_bits(v))


def test_diag_div6_exhaustive_against_ieee_division():
    """The kernels' t / 6 against correctly rounded division for every one of
    the 2^32 float32 bit patterns.  Reference: the quotient in binary64 rounded
    once to binary32.  That single rounding is exact here: t / 6 is either
    representable or has a repeating 01 binary expansion, which is never
    within 2^-52 of a binary32 midpoint, so neither the binary64 rounding
    nor a reciprocal-multiply inside the double division can move it across
    one."""
    chunk = 1 << 28
    mism = 0
    for start in range(0, 1 << 32, chunk):
        bits = torch.arange(start, start + chunk, dtype=torch.int64, device=DEV)
        v = (bits - (bits >= 2 ** 31).to(torch.int64) * 2 ** 32).to(torch.int32).view(torch.float32)
        out = torch.empty_like(v)
        fos.diag_convert(fos.DIAG_DIV6, v, out)
        ref = (v.double() / 6.0).float()
        same = (out.view(torch.int32) == ref.view(torch.int32)) | (torch.isnan(out) & torch.isnan(ref))
        mism += int((~same).sum().item())
    assert mism == 0


def test_diag_scale_codes_exhaustive():
    """The two block-scale codes the kernels derive from t = block amax * S
    (a branch-free t / 6 that is correctly rounded wherever the quotient is
    normal, and the exact t / 4) equal the E4M3 codes of the correctly
    rounded quotients t / 6 and t / 4, for every non-negative float32 t and
    +Inf.  The quotient t / 6 comes from binary64 division rounded once to
    binary32 (exact, see the division test above); both quotients are
    encoded by the pinned E4M3 conversion."""
    chunk = 1 << 28
    end = 0x7F800001  # +0 .. +Inf
    mism = 0
    for start in range(0, end, chunk):
        stop = min(end, start + chunk)
        t = torch.arange(start, stop, dtype=torch.int64, device=DEV).to(torch.int32).view(
            torch.float32)
        got = torch.empty(t.numel(), dtype=torch.int16, device=DEV)
        fos.diag_convert(fos.DIAG_SCALE_CODES, t, got)
        q = torch.empty(2 * t.numel(), dtype=torch.float32, device=DEV)
        q[0::2] = (t.double() / 6.0).float()
        q[1::2] = t * 0.25
        codes = torch.empty(2 * t.numel(), dtype=torch.uint8, device=DEV)
        fos.diag_convert(fos.DIAG_E4M3_ENCODE, q, codes)
        ref = codes[0::2].to(torch.int32) | (codes[1::2].to(torch.int32) << 8)
        mism += int(((got.to(torch.int32) & 0xFFFF) != ref).sum().item())
        del t, got, q, codes, ref
    assert mism == 0


def test_diag_div6_is_correctly_rounded():
    v = _dense_f32(1 << 22, seed=3)
    got = _run_diag(fos.DIAG_DIV6, v, torch.float32).numpy()
    with np.errstate(all="ignore"):
        ref = (v / np.float32(6.0)).astype(np.float32)  # IEEE binary32 division
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


# ------------------------------------------------------------------ full size
def test_activation_full_size_sampled():
    """8192x4096 bf16, per-tensor amax computed on the device, launched exactly
    as the benchmark launches it; the oracle checks a sample of rows (the
    global amax and therefore S come from the whole tensor)."""
    gen_dev = torch.device(DEV)
    for fam in workloads.FAMILIES:
        x = workloads.activation(8192, 4096, fam, seed=0, dtype=torch.bfloat16, device=gen_dev)
        for mode in ("mse", "mae_f16", "std"):
            for row in (False, True):
                gcfg, ocfg = _cfgs(mode, 448 if mode != "mae_f16" else 256, row)
                gc, gs, ga = fos.quantize(x, gcfg)
                torch.cuda.synchronize()
                xs = x.cpu()
                rows = np.random.default_rng(5).choice(8192, 48, replace=False)
                if row:
                    ref_a = oracle.amax_rows(xs[rows].float().numpy())
                    assert np.array_equal(_u32(ga[torch.from_numpy(rows).to(DEV)]),
                                          ref_a.view(np.uint32))
                else:
                    ref_a = oracle.amax_tensor(xs.float().numpy())
                    assert np.array_equal(_u32(ga), ref_a.view(np.uint32))
                ocfg2 = oracle.Config(**{**ocfg.__dict__, "amax_is_input": True})
                oc, os_, _ = oracle.quantize(xs[rows].float().numpy(), ocfg2, amax=ref_a)
                assert np.array_equal(gc.cpu().numpy()[rows], oc), (fam, mode, row)
                assert np.array_equal(gs.cpu().numpy()[rows], os_), (fam, mode, row)


# ------------------------------------------------------------------ one-pass row scale
@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("shape", [(5, 2048), (3, 4096), (9, 4800), (4, 7168), (2, 8192),
                                   (300, 2064)])
def test_row_scaled_one_pass_shapes(dt, mode, shape):
    """Row lengths served by the one-pass row kernel (128..512 blocks per row,
    ragged last thread, more rows than a CTA handles at once)."""
    gcfg, ocfg = _cfgs(mode, 448 if mode != "mse_f16" else 256, True)
    for i, fam in enumerate(("F2", "F4")):
        _check_quant(_x(*shape, fam, seed=11 + i, dt=dt), gcfg, ocfg, amax_given=(i == 1))


# ------------------------------------------------------------------ quantize list
@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("row", [False, True])
def test_quantize_list(dt, mode, row):
    """fos_quantize_list equals the oracle entry by entry; with per-tensor
    scale and amax computed it runs the pipelined launches (empty and ragged
    entries included)."""
    gcfg, ocfg = _cfgs(mode, 448, row)
    shapes = [(64, 1024), (0, 64), (7, 1040), (256, 2048), (48, 272), (1, 16)]
    xs = [_x(r, c, fam, i, dt) if r else torch.zeros(0, c, dtype=DTYPES[dt])
          for i, ((r, c), fam) in enumerate(zip(shapes, workloads.FAMILIES * 2))]
    gc, gs, ga = fos.quantize_list([x.to(DEV) for x in xs], gcfg)
    torch.cuda.synchronize()
    for x, c, s_, a in zip(xs, gc, gs, ga):
        if x.numel() == 0:
            if not row:
                assert float(a[0]) == 0.0
            continue
        oc, os_, oa = oracle.quantize(x.float().numpy(), ocfg)
        assert np.array_equal(_u32(a), oa.view(np.uint32))
        assert np.array_equal(s_.cpu().numpy(), os_)
        assert np.array_equal(c.cpu().numpy(), oc)


def test_quantize_list_equals_single_calls_full_size():
    gcfg, _ = _cfgs("mse")
    xs = [workloads.activation(8192, 4096, f, seed=i, device=DEV)
          for i, f in enumerate(workloads.FAMILIES)]
    gc, gs, ga = fos.quantize_list(xs, gcfg)
    for x, c, s_, a in zip(xs, gc, gs, ga):
        c1, s1, a1 = fos.quantize(x, gcfg)
        torch.cuda.synchronize()
        assert torch.equal(a, a1) and torch.equal(c, c1) and torch.equal(s_, s1)


@pytest.mark.parametrize("mode", list(MODES))
def test_quantize_overlap_stage(mode):
    gcfg, ocfg = _cfgs(mode)
    x = _x(96, 2048, "F2", 21, "bf16")
    xn = _x(40, 528, "F4", 22, "bf16")
    xf, xnf = x.float().numpy(), xn.float().numpy()
    a = torch.from_numpy(oracle.amax_tensor(xf)).to(DEV)
    an = torch.full((1,), 123.0, device=DEV)  # overwritten by the call
    c = torch.empty(96, 1024, dtype=torch.uint8, device=DEV)
    s_ = torch.empty(96, 128, dtype=torch.uint8, device=DEV)
    fos.quantize_overlap(x.to(DEV), a, c, s_, xn.to(DEV), an, gcfg)
    torch.cuda.synchronize()
    ocfg2 = oracle.Config(**{**ocfg.__dict__, "amax_is_input": True})
    oc, os_, _ = oracle.quantize(xf, ocfg2, amax=a.cpu().numpy())
    assert np.array_equal(c.cpu().numpy(), oc) and np.array_equal(s_.cpu().numpy(), os_)
    assert np.array_equal(_u32(an), oracle.amax_tensor(xnf).view(np.uint32))


# ------------------------------------------------------------------ sequential term order
SEQ_MODES = ["mae", "mse", "mae_f16", "mse_f16"]


@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("mode", SEQ_MODES)
@pytest.mark.parametrize("row", [False, True])
def test_quantize_1x16_seq_order(dt, mode, row):
    """Error terms summed in element order (the Transformer Engine order):
    per-tensor and per-row scale (the one-pass row kernel for the 4096-column
    case), amax computed and given, all four families."""
    gcfg, ocfg = _cfgs(mode, 448, row, seq=True)
    for i, (shape, fam) in enumerate(zip([(33, 4096), (70, 528), (5, 2048), (128, 1040)],
                                         workloads.FAMILIES)):
        _check_quant(_x(*shape, fam, seed=40 + i, dt=dt), gcfg, ocfg, amax_given=(i % 2 == 1))


def test_seq_order_changes_choices_on_gpu():
    """On this input the two orders select differently in some blocks (the
    oracle gives 8 differing scale bytes for MAE), so the sequential tests
    are not satisfied by the tree order by accident."""
    x = _x(256, 4096, "F2", 7, "bf16")
    a = torch.from_numpy(oracle.amax_tensor(x.float().numpy())).to(DEV)
    ct, st, _ = fos.quantize(x.to(DEV), fos.Config(mse=False), amax=a)
    cs, ss, _ = fos.quantize(x.to(DEV), fos.Config(mse=False, seq_order=True), amax=a)
    torch.cuda.synchronize()
    assert not torch.equal(ss, st)


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("mode", SEQ_MODES)
def test_qdq_list_seq_order(dt, mode):
    gcfg, ocfg = _cfgs(mode, 256, seq=True)
    shapes = [(64, 1024), (7, 1040), (48, 272), (1, 16)]
    xs = [workloads.qdq_weights(1, r, c, seed=60 + i, dtype=DTYPES[dt])[0]
          for i, (r, c) in enumerate(shapes)]
    outs = fos.qdq([x.to(DEV) for x in xs], gcfg)
    torch.cuda.synchronize()
    for x, o in zip(xs, outs):
        ref, _ = oracle.qdq(x.float().numpy(), ocfg, dt)
        assert np.array_equal(_u16(o), ref)


@pytest.mark.parametrize("mode", SEQ_MODES)
def test_quantize_list_seq_order(mode):
    """The pipelined list launches (encode of tensor i with the amax pass of
    tensor i+1) with the sequential order."""
    gcfg, ocfg = _cfgs(mode, 448, seq=True)
    xs = [_x(r, c, fam, 80 + i, "bf16") for i, ((r, c), fam) in
          enumerate(zip([(64, 1024), (7, 1040), (256, 2048)], workloads.FAMILIES))]
    gc, gs, ga = fos.quantize_list([x.to(DEV) for x in xs], gcfg)
    torch.cuda.synchronize()
    for x, c, s_, a in zip(xs, gc, gs, ga):
        oc, os_, oa = oracle.quantize(x.float().numpy(), ocfg)
        assert np.array_equal(_u32(a), oa.view(np.uint32))
        assert np.array_equal(s_.cpu().numpy(), os_) and np.array_equal(c.cpu().numpy(), oc)


def test_grouped_seq_order():
    R, C = 512, 272
    offs = workloads.moe_offsets(R, 12, seed=5, n_empty=3)
    x = workloads.moe_activations(R, C, offs, seed=6)
    gcfg, ocfg = _cfgs("mse_f16", 448, seq=True)
    oc, os_, oa = oracle.quantize_grouped(x.float().numpy(), offs.numpy(), ocfg)
    gc, gs, ga = fos.quantize_grouped(x.to(DEV), offs.to(DEV), gcfg)
    torch.cuda.synchronize()
    assert np.array_equal(_u32(ga), oa.view(np.uint32))
    assert np.array_equal(gc.cpu().numpy(), oc) and np.array_equal(gs.cpu().numpy(), os_)


def test_seq_order_with_16x16_is_unsupported():
    x = torch.zeros(16, 16, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(fos.FosError):
        fos.quantize(x, fos.Config(block16x16=True, seq_order=True))
    # standard mode has no candidate errors, so the order is moot and accepted
    fos.quantize(x, fos.Config(block16x16=True, four_over_six=False, seq_order=True))


# ------------------------------------------------------------------ fused amax + QDQ
@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("mode,seq", [("std", False), ("mse", False), ("mae_f16", False),
                                      ("mse_f16", False), ("mae_f16", True), ("mse", True)])
def test_qdq_fused(dt, mode, seq):
    """One persistent launch computes every amax and the QDQ of the list
    (empty and ragged entries included); two calls in a row on the same
    workspace give the oracle's bytes both times."""
    gcfg, ocfg = _cfgs(mode, 448, seq=seq)
    shapes = [(64, 1024), (0, 64), (7, 1040), (300, 2064), (48, 272), (1, 16)]
    xs = [workloads.qdq_weights(1, r, c, seed=90 + i, dtype=DTYPES[dt])[0] if r else
          torch.zeros(0, c, dtype=DTYPES[dt]) for i, (r, c) in enumerate(shapes)]
    xd = [x.to(DEV) for x in xs]
    ws = fos.qdq_fused_workspace(len(xd), DEV)
    for _ in range(2):
        outs, amaxes = fos.qdq_fused(xd, gcfg, workspace=ws)
        assert fos.workspace_error(ws) == 0
        for x, o, a in zip(xs, outs, amaxes):
            ref, oa = oracle.qdq(x.float().numpy(), ocfg, dt)
            assert np.array_equal(_u32(a), oa.view(np.uint32))
            if x.numel():
                assert np.array_equal(_u16(o), ref)


def test_qdq_fused_equals_separate_amax_passes_full_size():
    """8 x 2048x7168 bf16 (the fake-QAT weight list): the fused launch gives
    the bytes of fos_qdq with the amax computed by separate passes."""
    xs = workloads.qdq_weights(8, 2048, 7168, seed=3, device=DEV)
    for mode in ("mse_f16", "std"):
        gcfg, _ = _cfgs(mode, 448, seq=(mode != "std"))
        outs, amaxes = fos.qdq_fused(xs, gcfg)
        ref = fos.qdq(xs, gcfg, amax_given=False)
        a2 = [fos.amax(x) for x in xs]
        torch.cuda.synchronize()
        for o, r, a, b in zip(outs, ref, amaxes, a2):
            assert torch.equal(o.view(torch.int16), r.view(torch.int16))
            assert torch.equal(a, b)


# ------------------------------------------------------------------ column-wise operand
@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("mode", ["std", "mse", "mae_f16"])
@pytest.mark.parametrize("dual", [False, True])
def test_quantize_colwise(dt, mode, dual):
    """x^T quantized from x: whole and ragged 64 x 256 tiles, amax computed
    (first two shapes) and given; with dual the row-wise result of the same
    read equals fos_quantize's oracle result."""
    gcfg, ocfg = _cfgs(mode, 448)
    for i, (shape, fam) in enumerate(zip([(64, 256), (80, 272), (16, 16), (1024, 4096),
                                          (48, 4112)], list(workloads.FAMILIES) + ["F2"])):
        x = _x(*shape, fam, seed=120 + i, dt=dt)
        xf = x.float().numpy()
        given = i >= 2
        if given:
            a = oracle.amax_tensor(xf)
            ocfg2 = oracle.Config(**{**ocfg.__dict__, "amax_is_input": True})
            oct_, ost, oa = oracle.quantize_colwise(xf, ocfg2, amax=a)
            orc_, ors, _ = oracle.quantize(xf, ocfg2, amax=a)
            res = fos.quantize_colwise(x.to(DEV), gcfg, amax=torch.from_numpy(a).to(DEV),
                                       rowwise=dual)
        else:
            oct_, ost, oa = oracle.quantize_colwise(xf, ocfg)
            orc_, ors, _ = oracle.quantize(xf, ocfg)
            res = fos.quantize_colwise(x.to(DEV), gcfg, rowwise=dual)
        torch.cuda.synchronize()
        assert np.array_equal(_u32(res[2]), oa.view(np.uint32)), shape
        assert np.array_equal(res[0].cpu().numpy(), oct_), shape
        assert np.array_equal(res[1].cpu().numpy(), ost), shape
        if dual:
            assert np.array_equal(res[3].cpu().numpy(), orc_), shape
            assert np.array_equal(res[4].cpu().numpy(), ors), shape


def test_quantize_colwise_full_size_sampled():
    """8192x4096 bf16, both layouts from one read, amax computed: the
    row-wise result equals fos_quantize's, sampled columns equal the oracle."""
    x = workloads.activation(8192, 4096, "F2", seed=3, device=DEV)
    gcfg, ocfg = _cfgs("mse", 448)
    ct, st, a, c, s_ = fos.quantize_colwise(x, gcfg, rowwise=True)
    c1, s1, a1 = fos.quantize(x, gcfg)
    torch.cuda.synchronize()
    assert torch.equal(a, a1) and torch.equal(c, c1) and torch.equal(s_, s1)
    oa = oracle.amax_tensor(x.cpu().float().numpy())  # the whole tensor, on the host
    assert np.array_equal(_u32(a), oa.view(np.uint32))
    cols = np.random.default_rng(4).choice(4096, 24, replace=False)
    xc = x[:, torch.from_numpy(cols).to(DEV)].cpu().float().numpy()  # [8192, 24]
    ocfg2 = oracle.Config(**{**ocfg.__dict__, "amax_is_input": True})
    oct_, ost, _ = oracle.quantize_colwise(xc, ocfg2, amax=oa)
    assert np.array_equal(ct.cpu().numpy()[cols], oct_)
    assert np.array_equal(st.cpu().numpy()[cols], ost)


def test_quantize_colwise_unaligned_outputs():
    """Output buffers only 8-byte (codes) and 1-byte (scales) aligned take
    the per-block stores instead of the wide ones; same bytes."""
    gcfg, ocfg = _cfgs("mse", 448)
    for dt in ("bf16", "f32"):
        x = _x(128, 512, "F3", 140, dt)
        R, C = x.shape
        cb = torch.zeros(C * R // 2 + 64, dtype=torch.uint8, device=DEV)
        sb = torch.zeros(C * R // 16 + 64, dtype=torch.uint8, device=DEV)
        ct = cb[8:8 + C * R // 2].view(C, R // 2)
        st = sb[1:1 + C * R // 16].view(C, R // 16)
        _, _, a = fos.quantize_colwise(x.to(DEV), gcfg, codes_t=ct, scales_t=st)
        torch.cuda.synchronize()
        oc, os_, oa = oracle.quantize_colwise(x.float().numpy(), ocfg)
        assert np.array_equal(ct.cpu().numpy(), oc) and np.array_equal(st.cpu().numpy(), os_)


# ------------------------------------------------------------------ bounded waits
@pytest.mark.parametrize("which", [0, 1])
def test_bounded_waits_give_up_and_report(which):
    """A wait whose condition never comes true (a counter nothing increments,
    an mbarrier phase no copy completes) gives up after about a second and
    reports it; the device keeps working afterwards."""
    L = fos.lib()
    L.fos_diag_wait_timeout.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    L.fos_diag_wait_timeout.restype = ctypes.c_int
    word = torch.full((2,), 7, dtype=torch.int32, device=DEV)
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert L.fos_diag_wait_timeout(which, word.data_ptr(), s) == fos.FOS_OK
    torch.cuda.synchronize()
    assert int(word[0]) == 1
    x = _x(64, 256, "F1", 150, "bf16")
    _check_quant(x, *_cfgs("mse"), amax_given=False)


# ------------------------------------------------------------------ tiled scale layout
@pytest.mark.parametrize("shape", [(1, 16), (128, 64), (200, 144), (8192, 4096)])
def test_swizzle_scales(shape):
    R, C = shape
    s = np.random.default_rng(R + C).integers(0, 0x7F, (R, C // 16), dtype=np.uint8)
    got = fos.swizzle_scales(torch.from_numpy(s).to(DEV), R, C)
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy(), oracle.swizzle_scales(s))



@pytest.mark.parametrize("shape", [(300, 64), (130, 48)])
def test_swizzle_scales_unaligned_pointers(shape):
    """Scales that start one byte into a buffer and an output that starts 4
    bytes into one take the byte-load and 4-byte-store forms of the kernel;
    the bytes are those of the oracle's layout."""
    R, C = shape
    s = np.random.default_rng(R).integers(0, 0x7F, (R, C // 16), dtype=np.uint8)
    src = torch.zeros(s.size + 16, dtype=torch.uint8, device=DEV)
    src[1:1 + s.size] = torch.from_numpy(s.ravel()).to(DEV)
    n = -(-R // 128) * 128 * (-(-(C // 16) // 4) * 4)
    dst = torch.full((n + 16,), 0xEE, dtype=torch.uint8, device=DEV)
    fos.swizzle_scales(src[1:1 + s.size], R, C, out=dst[4:4 + n])
    torch.cuda.synchronize()
    got = dst.cpu().numpy()
    assert np.array_equal(got[4:4 + n], oracle.swizzle_scales(s))
    assert (got[:4] == 0xEE).all() and (got[4 + n:] == 0xEE).all()

@pytest.mark.parametrize("mode", ["std", "mse"])
def test_swizzled_scales_feed_an_fp4_gemm(mode):
    """Codes and tiled scales from this library, handed to PyTorch's NVFP4
    scaled matmul, give the product of the dequantized operands: the tiled
    layout is the one such a GEMM reads."""
    if not hasattr(torch, "float4_e2m1fn_x2"):
        pytest.skip("no FP4 dtype in this PyTorch")
    M, N, K = 256, 128, 512
    gcfg, _ = _cfgs(mode)
    a = workloads.activation(M, K, "F1", seed=31, device=DEV)
    b = workloads.activation(N, K, "F3", seed=32, device=DEV)
    ca, sa, aa = fos.quantize(a, gcfg)
    cb, sb, ab = fos.quantize(b, gcfg)
    swa, swb = fos.swizzle_scales(sa, M, K), fos.swizzle_scales(sb, N, K)
    try:
        got = torch._scaled_mm(ca.view(torch.float4_e2m1fn_x2), cb.view(torch.float4_e2m1fn_x2).t(),
                               swa.view(torch.float8_e4m3fn), swb.view(torch.float8_e4m3fn),
                               out_dtype=torch.float32)
    except (RuntimeError, TypeError) as e:
        pytest.skip("no NVFP4 scaled matmul here: %s" % str(e)[:80])
    da = fos.dequantize(ca, sa, aa, gcfg, out_dtype=torch.float32).double()
    db = fos.dequantize(cb, sb, ab, gcfg, out_dtype=torch.float32).double()
    Sa = float(oracle.global_scale(float(aa[0]), 448))
    Sb = float(oracle.global_scale(float(ab[0]), 448))
    ref = (da * Sa) @ (db * Sb).t()
    err = (got.double() - ref).abs().max().item()
    assert err <= 1e-5 * ref.abs().max().item() + 1e-6, err


# ------------------------------------------------------------------ product of quantized operands
@pytest.mark.parametrize("mode", ["std", "mse"])
@pytest.mark.parametrize("row", [False, True])
def test_mm_of_quantized_operands(mode, row):
    """a . b^T from this library's codes and tiled scales equals the oracle's
    product reference (block values of the same inputs times the global
    decode scales) within its fp32 bound gamma_(K+2) * sum |terms|."""
    M, N, K = 256, 128, 512
    gcfg_a, ocfg_a = _cfgs(mode, 448, row)
    gcfg_b, ocfg_b = _cfgs(mode, 448)
    a = _x(M, K, "F2", 51, "bf16")
    b = _x(N, K, "F1", 52, "bf16")
    ca, sa, aa = fos.quantize(a.to(DEV), gcfg_a)
    cb, sb, ab = fos.quantize(b.to(DEV), gcfg_b)
    out = fos.mm(ca, fos.swizzle_scales(sa, M, K), aa, cb, fos.swizzle_scales(sb, N, K), ab,
                 gcfg_a)
    torch.cuda.synchronize()
    oca, osa, oaa = oracle.quantize(a.float().numpy(), ocfg_a)
    ocb, osb, oab = oracle.quantize(b.float().numpy(), ocfg_b)
    assert np.array_equal(ca.cpu().numpy(), oca) and np.array_equal(cb.cpu().numpy(), ocb)
    ref, bound = oracle.mm_reference(oca, osa, oaa, ocb, osb, oab, ocfg_a)
    err = np.abs(out.cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= bound + 1e-30), float((err / (bound + 1e-30)).max())


@pytest.mark.parametrize("M,N,K", [(16, 16, 64), (304, 208, 320), (128, 400, 1024),
                                   (1040, 592, 256), (144, 1344, 2112)])
def test_mm_tile_edges(M, N, K):
    """Shapes that put the edges of the 128 x 192 output tiles everywhere: N
    below one tile, b tiles starting at row 0 and row 64 of a 128-row scale
    tile, with and without a next scale tile, ragged M, K not a multiple of
    the 256-element stage (partial last stage), several tiles per CTA; every
    entry against the oracle's product reference within its fp32 bound."""
    gcfg, ocfg = _cfgs("mse", 448, False)
    a = _x(M, K, "F3", 71, "bf16")
    b = _x(N, K, "F2", 72, "bf16")
    ca, sa, aa = fos.quantize(a.to(DEV), gcfg)
    cb, sb, ab = fos.quantize(b.to(DEV), gcfg)
    out = fos.mm(ca, fos.swizzle_scales(sa, M, K), aa, cb, fos.swizzle_scales(sb, N, K), ab, gcfg)
    torch.cuda.synchronize()
    oca, osa, oaa = oracle.quantize(a.float().numpy(), ocfg)
    ocb, osb, oab = oracle.quantize(b.float().numpy(), ocfg)
    assert np.array_equal(ca.cpu().numpy(), oca) and np.array_equal(cb.cpu().numpy(), ocb)
    ref, bound = oracle.mm_reference(oca, osa, oaa, ocb, osb, oab, ocfg)
    err = np.abs(out.cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= bound + 1e-30), float((err / (bound + 1e-30)).max())


def _at16(t):
    """A copy of t whose storage starts 16 bytes into a larger buffer: 16-byte
    but not 256-byte aligned."""
    nb = t.numel() * t.element_size()
    buf = torch.zeros(nb + 256, dtype=torch.uint8, device=t.device)
    v = buf[16:16 + nb].view(t.dtype).view(t.shape)
    v.copy_(t)
    return v


def test_mm_many_tiles_with_16_byte_aligned_operands():
    """A wide product (17 x 64 output tiles, more than one per SM, so each
    CTA of the persistent kernel walks several and its accumulator is
    reused); operands and output placed 16 bytes into their buffers.  Sampled
    rows of every 768-row band, row-scaled a, against the oracle's block
    values within the fp32 accumulation bound."""
    M, N, K = 2176, 16384, 128
    gcfg_a, ocfg_a = _cfgs("mse", 448, True)
    gcfg_b, ocfg_b = _cfgs("mse", 448)
    a = _x(M, K, "F4", 61, "bf16")
    b = workloads.weight(N, K, seed=62, dtype=torch.bfloat16)
    ca, sa, aa = fos.quantize(a.to(DEV), gcfg_a)
    cb, sb, ab = fos.quantize(b.to(DEV), gcfg_b)
    ta, tb = fos.swizzle_scales(sa, M, K), fos.swizzle_scales(sb, N, K)
    out = _at16(torch.zeros((M, N), dtype=torch.float32, device=DEV))
    got = fos.mm(_at16(ca), _at16(ta), aa, _at16(cb), _at16(tb), ab, gcfg_a, out=out)
    torch.cuda.synchronize()
    assert got.data_ptr() % 256 == 16
    oca, osa, oaa = oracle.quantize(a.float().numpy(), ocfg_a)
    ocb, osb, oab = oracle.quantize(b.float().numpy(), ocfg_b)
    assert np.array_equal(ca.cpu().numpy(), oca) and np.array_equal(cb.cpu().numpy(), ocb)
    rows = np.unique(np.concatenate([np.arange(0, M, 97), [M - 1, M - 16, 767, 768, 1536]]))
    ref, bound = oracle.mm_reference(oca[rows], osa[rows], oaa[rows], ocb, osb, oab, ocfg_a)
    err = np.abs(got.cpu().numpy()[rows].astype(np.float64) - ref)
    assert np.all(err <= bound + 1e-30), float((err / (bound + 1e-30)).max())
