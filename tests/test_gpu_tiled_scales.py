"""Block scales written straight into the tiled GEMM layout by the encoders.

With Config(scale_tiled=True) (fos_config.scale_layout = FOS_SCALES_TILED)
fos_quantize, fos_quantize_list, fos_quantize_overlap and
fos_quantize_colwise store each E4M3 block scale at its place in the 128 x 4
tile layout of block-scaled FP4 GEMMs, padding zeroed.  The result must be,
byte for byte, the oracle's plain scales put through the oracle's layout
function (swizzle_scales), and the codes must be those of the plain layout.
Every encode path is covered: the per-tensor stream, the per-row walker and
the row-pass kernel (one and two passes per row), the list pipeline and the
overlapped launch, the column-wise kernel alone and with its row-wise twin,
on shapes whose rows and block columns are and are not multiples of the
tile (128 rows, 4 blocks), then at the activation size the GEMM consumes.
"""
import dataclasses

import numpy as np
import pytest
import torch

import nvfp4_quantization_precision_gb300 as fos
import oracle
import workloads

import oracle_slices as S

pytestmark = pytest.mark.gpu

DEV = "cuda"

MODES = {
    "std": (False, True, False, False),
    "mse": (True, True, False, False),
    "mae_f16": (True, False, True, False),
    "mse_seq": (True, True, False, True),
}

# (rows, cols): the last block column and row tile are ragged in most of them;
# cols 2064 / 4112 have 129 / 257 blocks per row (the row-pass kernel with one
# and two passes), 272 and below go to the per-row walker
SHAPES = [(16, 16), (48, 48), (128, 64), (300, 272), (256, 4096), (300, 2064), (136, 4112),
          (1000, 1040)]
DTYPES = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _cfgs(mode, row=False, bound=448):
    f, m, h, s = MODES[mode]
    g = fos.Config(four_over_six=f, mse=m, err_f16=h, bound=bound, row_scaled=row,
                   seq_order=s, scale_tiled=True)
    o = oracle.Config(four_over_six=f, mse=m, err_f16=h, bound=bound, row_scaled=row,
                      seq_order=s, amax_is_input=True)
    return g, o


def _u(t):
    t = t.cpu().contiguous()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.view(torch.int32).numpy().view(np.uint32)
    return t.numpy()


def _same(got, ref, what):
    got = _u(got)
    ref = np.asarray(ref)
    if ref.dtype == np.float32:
        ref = ref.view(np.uint32)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    if not np.array_equal(got, ref):
        bad = np.argwhere(got != ref)
        first = tuple(bad[0])
        raise AssertionError("%s: %d of %d differ, first at %s: device %#x oracle %#x" % (
            what, len(bad), got.size, first, int(got[first]), int(ref[first])))


def _input(R, C, dt, seed):
    x = workloads.activation(R, C, "F2", seed=seed, dtype=torch.float32, device="cpu")
    return x.to(DTYPES[dt]).to(DEV)


def _poisoned(R, C):
    """A tiled scale buffer full of 0xFF, so that padding the encoder failed
    to clear shows up."""
    n = fos.lib().fos_swizzled_scales_bytes(R, C)
    return torch.full((n,), 0xFF, dtype=torch.uint8, device=DEV)


@pytest.mark.parametrize("dt", list(DTYPES))
@pytest.mark.parametrize("R,C", SHAPES)
@pytest.mark.parametrize("mode", list(MODES))
def test_quantize_writes_the_tiled_layout(R, C, dt, mode):
    x = _input(R, C, dt, seed=R * 7 + C)
    h = x.cpu().float().numpy()
    for row in (False, True):
        gcfg, ocfg = _cfgs(mode, row)
        ref_a = oracle.amax_rows(h) if row else oracle.amax_tensor(h)
        oc, os_, _ = oracle.quantize(h, ocfg, ref_a)
        want = oracle.swizzle_scales(os_)
        tag = "%dx%d %s %s %s" % (R, C, dt, mode, "row" if row else "tensor")
        # amax computed on the device, then given
        gc, gs, ga = fos.quantize(x, gcfg, scales=_poisoned(R, C))
        kc, ks, _ = fos.quantize(x, gcfg, amax=torch.from_numpy(ref_a).to(DEV),
                                 scales=_poisoned(R, C))
        torch.cuda.synchronize()
        _same(ga, ref_a, tag + " amax")
        for name, c, s in (("computed", gc, gs), ("given", kc, ks)):
            _same(s, want, "%s %s tiled scales" % (tag, name))
            _same(c, oc, "%s %s codes" % (tag, name))


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("row", [False, True], ids=["tensor", "row"])
def test_quantize_list_writes_the_tiled_layout(dt, row):
    """The list call (with per-tensor amax computed: the pipelined launches,
    encode of tensor i with the amax pass of tensor i+1)."""
    shapes = [(300, 272), (128, 64), (136, 4112), (16, 16), (256, 4096)]
    xs = [_input(R, C, dt, seed=i) for i, (R, C) in enumerate(shapes)]
    gcfg, ocfg = _cfgs("mse", row)
    lc, ls, la = fos.quantize_list(xs, gcfg, scales=[_poisoned(R, C) for R, C in shapes])
    torch.cuda.synchronize()
    for i, x in enumerate(xs):
        h = x.cpu().float().numpy()
        a = oracle.amax_rows(h) if row else oracle.amax_tensor(h)
        oc, os_, _ = oracle.quantize(h, ocfg, a)
        _same(la[i], a, "list %d amax" % i)
        _same(ls[i], oracle.swizzle_scales(os_), "list %d tiled scales" % i)
        _same(lc[i], oc, "list %d codes" % i)


def test_quantize_overlap_writes_the_tiled_layout():
    x = _input(300, 2064, "bf16", seed=3)
    xn = _input(136, 4112, "bf16", seed=4)
    h, hn = x.cpu().float().numpy(), xn.cpu().float().numpy()
    gcfg, ocfg = _cfgs("mae_f16")
    a = oracle.amax_tensor(h)
    codes = torch.empty((300, 2064 // 2), dtype=torch.uint8, device=DEV)
    scales = _poisoned(300, 2064)
    an = torch.empty(1, dtype=torch.float32, device=DEV)
    fos.quantize_overlap(x, torch.from_numpy(a).to(DEV), codes, scales, xn, an, gcfg)
    torch.cuda.synchronize()
    oc, os_, _ = oracle.quantize(h, ocfg, a)
    _same(scales, oracle.swizzle_scales(os_), "overlap tiled scales")
    _same(codes, oc, "overlap codes")
    _same(an, oracle.amax_tensor(hn), "overlap next amax")


@pytest.mark.parametrize("dt", list(DTYPES))
@pytest.mark.parametrize("R,C", [(16, 16), (48, 80), (64, 128), (304, 272), (256, 4096),
                                 (1040, 1000 // 16 * 16)])
def test_colwise_writes_the_tiled_layout(R, C, dt):
    """x^T's scales ([cols, rows/16]) tiled; with the row-wise twin both."""
    x = _input(R, C, dt, seed=R + 5 * C)
    h = x.cpu().float().numpy()
    gcfg, ocfg = _cfgs("mse")
    a = oracle.amax_tensor(h)
    otc, ots, _ = oracle.quantize_colwise(h, ocfg, a)
    oc, os_, _ = oracle.quantize(h, ocfg, a)
    ct, st, ca = fos.quantize_colwise(x, gcfg, scales_t=_poisoned(C, R))
    dt_, ds_, da, dc, dsr = fos.quantize_colwise(x, gcfg, scales_t=_poisoned(C, R),
                                                 codes=torch.empty((R, C // 2), dtype=torch.uint8,
                                                                   device=DEV),
                                                 scales=_poisoned(R, C))
    torch.cuda.synchronize()
    tag = "colwise %dx%d %s" % (R, C, dt)
    _same(ca, a, tag + " amax")
    _same(da, a, tag + " dual amax")
    _same(st, oracle.swizzle_scales(ots), tag + " tiled scales")
    _same(ct, otc, tag + " codes")
    _same(ds_, oracle.swizzle_scales(ots), tag + " dual tiled scales")
    _same(dt_, otc, tag + " dual codes")
    _same(dsr, oracle.swizzle_scales(os_), tag + " dual row-wise tiled scales")
    _same(dc, oc, tag + " dual row-wise codes")


@pytest.mark.parametrize("mode", list(MODES))
def test_full_size_activation_tiled_every_row(mode):
    """8192x4096 bf16 (the activation operand of the GEMM) per tensor and per
    row, and its column-wise operand: every tiled byte against the oracle."""
    xs = [workloads.activation(8192, 4096, fam, seed=0, dtype=torch.bfloat16, device=DEV)
          for fam in ("F1", "F2")]
    for x in xs:
        h = x.cpu().float().numpy()
        for row in (False, True):
            gcfg, ocfg = _cfgs(mode, row)
            a = S.amax_rows(h) if row else S.amax_tensor(h)
            gc, gs, _ = fos.quantize(x, gcfg)
            lc, ls, _ = fos.quantize_list([x], gcfg)
            torch.cuda.synchronize()
            oc, os_ = S.quantize(h, ocfg, a)
            want = oracle.swizzle_scales(os_)
            _same(gs, want, "full %s row=%d tiled scales" % (mode, row))
            _same(gc, oc, "full %s row=%d codes" % (mode, row))
            _same(ls[0], want, "full %s row=%d list tiled scales" % (mode, row))
            _same(lc[0], oc, "full %s row=%d list codes" % (mode, row))
        if mode == "mse":
            gcfg, ocfg = _cfgs(mode)
            a = S.amax_tensor(h)
            ct, st, _, dc, ds = fos.quantize_colwise(x, gcfg, rowwise=True)
            torch.cuda.synchronize()
            otc, ots = S.quantize(np.ascontiguousarray(h.T), ocfg, a)
            _same(st, oracle.swizzle_scales(ots), "full colwise tiled scales")
            _same(ct, otc, "full colwise codes")
            oc, os_ = S.quantize(h, ocfg, a)
            _same(ds, oracle.swizzle_scales(os_), "full colwise row-wise tiled scales")


def test_mm_consumes_the_tiled_output_directly():
    """fos_mm on operands whose scales the encoder wrote tiled equals fos_mm on
    the same operands' plain scales put through fos_swizzle_scales."""
    M, N, K = 304, 272, 512
    a = _input(M, K, "bf16", seed=11)
    b = _input(N, K, "bf16", seed=12)
    tcfg, _ = _cfgs("mse")
    pcfg = dataclasses.replace(tcfg, scale_tiled=False)
    ac, at, aa = fos.quantize(a, tcfg)
    bc, bt, ba = fos.quantize(b, tcfg)
    pac, pas, _ = fos.quantize(a, pcfg)
    pbc, pbs, _ = fos.quantize(b, pcfg)
    direct = fos.mm(ac, at, aa, bc, bt, ba, tcfg)
    via = fos.mm(pac, fos.swizzle_scales(pas, M, K), aa, pbc, fos.swizzle_scales(pbs, N, K), ba,
                 pcfg)
    torch.cuda.synchronize()
    _same(ac, _u(pac), "codes tiled vs plain")
    _same(at, _u(fos.swizzle_scales(pas, M, K)), "tiled scales vs swizzled plain")
    _same(direct, _u(via), "mm direct vs swizzled")


def test_mm_row_scaled_from_tiled_output():
    """A row-scaled a (the row pass, scales written tiled) times a per-tensor
    b (list pipeline, tiled): fos_mm equals the oracle's product reference of
    the same operands within its fp32 bound, and the tiled scales equal the
    oracle's."""
    M, N, K = 320, 400, 2048  # 128 blocks per row of a: the one-pass row kernel
    a = _input(M, K, "bf16", seed=21)
    b = _input(N, K, "bf16", seed=22)
    ga, oa = _cfgs("mse", row=True)
    gb, ob = _cfgs("mse")
    ca, sa, aa = fos.quantize(a, ga, scales=_poisoned(M, K))
    (cb,), (sb,), (ab,) = fos.quantize_list([b], gb, scales=[_poisoned(N, K)])
    out = fos.mm(ca, sa, aa, cb, sb, ab, ga)
    torch.cuda.synchronize()
    ha, hb = a.cpu().float().numpy(), b.cpu().float().numpy()
    ra, tb = oracle.amax_rows(ha), oracle.amax_tensor(hb)
    oca, osa, _ = oracle.quantize(ha, oa, ra)
    ocb, osb, _ = oracle.quantize(hb, ob, tb)
    _same(sa, oracle.swizzle_scales(osa), "a tiled scales")
    _same(sb, oracle.swizzle_scales(osb), "b tiled scales")
    _same(ca, oca, "a codes")
    _same(cb, ocb, "b codes")
    ref, bound = oracle.mm_reference(oca, osa, ra, ocb, osb, tb, oa)
    err = np.abs(out.cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= bound + 1e-30), float((err / (bound + 1e-30)).max())
