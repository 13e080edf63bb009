"""Bit-exact parity at the full workload sizes over the whole knob matrix,
every row compared.

The workloads are the ones the benchmark times: the activation batch
(8192x4096 bf16, four families), the weight (14336x4096 bf16 and fp32,
16x16 tiles, then dequantized), the fake-QAT QDQ list (8 x 2048x7168 bf16 and
fp16), the packed MoE activations (65536x7168 bf16 in 64 token groups) and
the flattened expert stack (64 x 2048x7168 bf16, 16x16).  At these sizes the
per-tensor, per-row and 16x16 kernels spend most of the launch in their
steady-state loops (no bounds checks), which small inputs never enter; a
medium-size sweep covers the fp16 / fp32 instantiations of the same loops.

Each configuration runs on the device through the C ABI, then the CPU
oracle recomputes every row from the same bytes (its calls spread over row
slices on every host core, see oracle_slices.py) with the global amax it
computes itself, and codes, scales, amaxes and outputs must agree as integer
views (tolerance 0).
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

# name -> (four_over_six, mse, err_f16, seq_order)
MODES = {
    "std": (False, True, False, False),
    "mae": (True, False, False, False),
    "mse": (True, True, False, False),
    "mae_f16": (True, False, True, False),
    "mse_f16": (True, True, True, False),
    "mae_seq": (True, False, False, True),
    "mse_seq": (True, True, False, True),
    "mae_f16_seq": (True, False, True, True),
    "mse_f16_seq": (True, True, True, True),
}
TREE = ["std", "mae", "mse", "mae_f16", "mse_f16"]
SEQ = ["mae_seq", "mse_seq", "mae_f16_seq", "mse_f16_seq"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _cfgs(mode, bound=448, row=False, b16=False):
    f, m, h, s = MODES[mode]
    g = fos.Config(block16x16=b16, four_over_six=f, mse=m, err_f16=h, bound=bound,
                   row_scaled=row, seq_order=s)
    o = oracle.Config(block16x16=b16, four_over_six=f, mse=m, err_f16=h, bound=bound,
                      row_scaled=row, seq_order=s, amax_is_input=True)
    return g, o


def _np(t):
    t = t.cpu().contiguous()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.view(torch.int32).numpy().view(np.uint32)
    return t.numpy()


def _same(got, ref, what):
    got = _np(got) if isinstance(got, torch.Tensor) else got
    ref = np.asarray(ref)
    if ref.dtype == np.float32:
        ref = ref.view(np.uint32)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    if not np.array_equal(got, ref):
        bad = np.argwhere(got != ref)
        first = tuple(bad[0])
        raise AssertionError("%s: %d of %d differ, first at %s: device %#x oracle %#x" % (
            what, len(bad), got.size, first, int(got[first]), int(ref[first])))


def _host(x):
    return x.cpu().float().numpy()


# ------------------------------------------------------------ activation batch
ACT_CASES = ([(m, b, r) for m in TREE for b in (448, 256) for r in (False, True)] +
             [(m, 448, r) for m in SEQ for r in (False, True)])


@pytest.fixture(scope="module")
def act():
    xs = [workloads.activation(8192, 4096, fam, seed=0, dtype=torch.bfloat16, device=DEV)
          for fam in workloads.FAMILIES]
    host = [_host(x) for x in xs]
    return xs, host, [S.amax_tensor(h) for h in host], [S.amax_rows(h) for h in host]


@pytest.mark.parametrize("mode,bound,row", ACT_CASES)
def test_activation_batch_every_row(act, mode, bound, row):
    """The four 8192x4096 bf16 families through fos_quantize (amax computed,
    and amax given) and through fos_quantize_list (with per-tensor scale the
    pipelined launches: encode of tensor i with the amax pass of i+1)."""
    xs, host, ta, ra = act
    gcfg, ocfg = _cfgs(mode, bound, row)
    lc, ls, la = fos.quantize_list(xs, gcfg)
    for i, fam in enumerate(workloads.FAMILIES):
        a = ra[i] if row else ta[i]
        gc, gs, ga = fos.quantize(xs[i], gcfg)
        kc, ks, _ = fos.quantize(xs[i], gcfg, amax=torch.from_numpy(a).to(DEV))
        torch.cuda.synchronize()
        oc, os_ = S.quantize(host[i], ocfg, a)
        tag = "%s %s %d %s" % (fam, mode, bound, "row" if row else "tensor")
        _same(ga, a, tag + " amax")
        _same(la[i], a, tag + " list amax")
        for name, c, s in (("computed", gc, gs), ("given", kc, ks), ("list", lc[i], ls[i])):
            _same(s, os_, "%s %s scales" % (tag, name))
            _same(c, oc, "%s %s codes" % (tag, name))
        if mode in ("std", "mse") and bound == 448:
            deq = fos.dequantize(gc, gs, ga, gcfg, out_dtype=torch.bfloat16)
            torch.cuda.synchronize()
            _same(deq, S.dequantize(oc, os_, a, ocfg, "bf16"), tag + " dequantize")


COLWISE_CASES = [("std", 448), ("mse", 448), ("mae_f16", 256), ("mse_f16_seq", 448)]


@pytest.mark.parametrize("mode,bound", COLWISE_CASES)
def test_activation_colwise_every_row(act, mode, bound):
    """The column-wise operand of each 8192x4096 family (x^T quantized from
    x, per-tensor amax computed), alone and with the row-wise result of the
    same read, every row of both layouts."""
    xs, host, ta, _ = act
    gcfg, ocfg = _cfgs(mode, bound)
    for i, fam in enumerate(workloads.FAMILIES):
        ct, st, ca = fos.quantize_colwise(xs[i], gcfg)
        dt_, ds_, da, dc, dsr = fos.quantize_colwise(xs[i], gcfg, rowwise=True)
        torch.cuda.synchronize()
        a = ta[i]
        tag = "colwise %s %s %d" % (fam, mode, bound)
        _same(ca, a, tag + " amax")
        _same(da, a, tag + " dual amax")
        otc, ots = S.quantize(np.ascontiguousarray(host[i].T), ocfg, a)
        _same(st, ots, tag + " scales")
        _same(ct, otc, tag + " codes")
        _same(ds_, ots, tag + " dual scales")
        _same(dt_, otc, tag + " dual codes")
        oc, os_ = S.quantize(host[i], ocfg, a)
        _same(dsr, os_, tag + " dual row-wise scales")
        _same(dc, oc, tag + " dual row-wise codes")


# ------------------------------------------------------------ weight, 16x16
WEIGHT_CASES = [(m, b) for m in TREE for b in (448, 256)]


@pytest.fixture(scope="module")
def weights():
    out = {}
    for dt in (torch.bfloat16, torch.float32):
        w = workloads.weight(14336, 4096, seed=0, dtype=dt, device=DEV)
        h = _host(w)
        out[dt] = (w, h, S.amax_tensor(h))
    return out


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("mode,bound", WEIGHT_CASES)
def test_weight_16x16_every_row(weights, dt, mode, bound):
    """14336x4096 weight in 16x16 tiles, per-tensor amax computed on the
    device, then dequantized to bf16 on the device."""
    w, h, a = weights[dt]
    gcfg, ocfg = _cfgs(mode, bound, b16=True)
    gc, gs, ga = fos.quantize(w, gcfg)
    deq = fos.dequantize(gc, gs, ga, gcfg, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    oc, os_ = S.quantize(h, ocfg, a)
    tag = "weight %s %s %d" % (dt, mode, bound)
    _same(ga, a, tag + " amax")
    _same(gs, os_, tag + " scales")
    _same(gc, oc, tag + " codes")
    _same(deq, S.dequantize(oc, os_, a, ocfg, "bf16"), tag + " dequantize")


# ------------------------------------------------------------ fake-QAT QDQ list
QDQ_CASES = [(m, 448) for m in TREE + SEQ] + [(m, 256) for m in TREE if m != "std"]


@pytest.fixture(scope="module")
def qdq_lists():
    out = {}
    for dt in (torch.bfloat16, torch.float16):
        ws = workloads.qdq_weights(8, 2048, 7168, seed=0, dtype=dt, device=DEV)
        host = [_host(w) for w in ws]
        out[dt] = (ws, host, [S.amax_tensor(h) for h in host])
    return out


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16], ids=["bf16", "f16"])
@pytest.mark.parametrize("mode,bound", QDQ_CASES)
def test_qdq_list_every_row(qdq_lists, dt, mode, bound):
    """Eight 2048x7168 weights: fos_qdq with the caller's FP32 amax (one
    launch for the list) and fos_qdq_fused (every amax and the QDQ in one
    launch), every output element against the oracle."""
    ws, host, am = qdq_lists[dt]
    gcfg, ocfg = _cfgs(mode, bound)
    outs = fos.qdq(ws, gcfg, amaxes=[torch.from_numpy(a).to(DEV) for a in am])
    fouts, famax = fos.qdq_fused(ws, gcfg)
    torch.cuda.synchronize()
    kind = "bf16" if dt == torch.bfloat16 else "f16"
    for i, (h, a) in enumerate(zip(host, am)):
        ref = S.qdq(h, ocfg, kind, a)
        tag = "qdq %s %s %d tensor %d" % (kind, mode, bound, i)
        _same(famax[i], a, tag + " fused amax")
        _same(outs[i], ref, tag)
        _same(fouts[i], ref, tag + " fused")


# ------------------------------------------------------------ MoE grouped 1x16
MOE_MODES = [("std", 448), ("mae", 448), ("mse", 448), ("mae_f16", 448), ("mse_f16", 448),
             ("mse", 256), ("mse_seq", 448)]


@pytest.fixture(scope="module")
def moe():
    R, C, G = 65536, 7168, 64
    offs = workloads.moe_offsets(R, G, seed=0)
    x = workloads.moe_activations(R, C, offs, seed=0, device=DEV)
    ends = offs.numpy().astype(np.int64)
    live = int(ends[-1])
    h = _host(x[:live])
    ga = np.zeros(G, np.float32)
    lo = 0
    for g, hi in enumerate(ends):
        if hi > lo:
            ga[g] = S.amax_tensor(h[lo:hi])[0]
        lo = max(lo, hi)
    rows_group = np.searchsorted(ends, np.arange(live), side="right")
    return x, offs, h, ga, ga[rows_group], live


@pytest.mark.parametrize("mode,bound", MOE_MODES)
def test_grouped_moe_every_row(moe, mode, bound):
    """65536x7168 bf16 tokens in 64 lognormal groups (4 empty, the last end
    below the row count): group amax computed on the device, every live row
    against the oracle with its group's amax, every tail row zero."""
    x, offs, h, ga_ref, rowamax, live = moe
    gcfg, ocfg = _cfgs(mode, bound, row=True)
    gcfg = dataclasses.replace(gcfg, row_scaled=False)
    gc, gs, ga = fos.quantize_grouped(x, offs.to(DEV), gcfg)
    torch.cuda.synchronize()
    _same(ga, ga_ref, "moe group amax")
    oc, os_ = S.quantize(h, ocfg, rowamax)
    gcn, gsn = _np(gc), _np(gs)
    _same(gsn[:live], os_, "moe %s %d scales" % (mode, bound))
    _same(gcn[:live], oc, "moe %s %d codes" % (mode, bound))
    assert not gcn[live:].any() and not gsn[live:].any(), "tail not zero"


# ------------------------------------------------------------ MoE expert stack, 16x16
EXPERT_CASES = [(m, b) for m in TREE for b in (448, 256)]


@pytest.fixture(scope="module")
def experts():
    E, R, C = 64, 2048, 7168
    x = workloads.moe_experts(E, R, C, seed=0, device=DEV).view(E * R, C)
    h = _host(x)
    ea = np.array([S.amax_tensor(h[e * R:(e + 1) * R])[0] for e in range(E)], np.float32)
    return x, h, ea, np.repeat(ea, R), E, R


@pytest.mark.parametrize("mode,bound", EXPERT_CASES)
def test_moe_experts_16x16_every_row(experts, mode, bound):
    """64 experts x 2048x7168 bf16 in one flattened call, 16x16 tiles: per-row
    amax (each expert's amax expanded to its rows) and the grouped entry point
    (one group per expert, amax computed), every tile band against the
    oracle."""
    x, h, ea, rowamax, E, R = experts
    gcfg, ocfg = _cfgs(mode, bound, row=True, b16=True)
    gc, gs, _ = fos.quantize(x, gcfg, amax=torch.from_numpy(rowamax).to(DEV))
    offs = torch.arange(1, E + 1, dtype=torch.int32, device=DEV) * R
    qc, qs, qa = fos.quantize_grouped(x, offs, dataclasses.replace(gcfg, row_scaled=False))
    torch.cuda.synchronize()
    _same(qa, ea, "expert amax")
    oc, os_ = S.quantize(h, ocfg, rowamax)
    tag = "experts %s %d" % (mode, bound)
    _same(gs, os_, tag + " scales")
    _same(gc, oc, tag + " codes")
    _same(qs, os_, tag + " grouped scales")
    _same(qc, oc, tag + " grouped codes")


# ------------------------------------------------------------ medium sizes, fp16 / fp32
MED_DT = {"f16": torch.float16, "f32": torch.float32}


@pytest.fixture(scope="module")
def medium():
    out = {}
    for name, dt in MED_DT.items():
        xs = [workloads.activation(4096, 4096, fam, seed=5, dtype=dt, device=DEV)
              for fam in ("F2", "F4")]
        narrow = workloads.activation(16384, 1024, "F4", seed=6, dtype=dt, device=DEV)
        host = [_host(x) for x in xs]
        out[name] = (xs, host, narrow, _host(narrow))
    return out


@pytest.mark.parametrize("dt", list(MED_DT))
@pytest.mark.parametrize("mode", list(MODES))
def test_medium_1x16_steady_state(medium, dt, mode):
    """4096x4096 fp16 / fp32 (two families): per-tensor amax (given, and
    computed in the list pipeline), per-row one-pass (4096 columns) and the
    per-row walk (16384x1024), every row; these sizes run the steady-state
    loops of every input type."""
    xs, host, narrow, nh = medium[dt]
    gcfg, ocfg = _cfgs(mode)
    rcfg, rocfg = _cfgs(mode, row=True)
    lc, ls, la = fos.quantize_list(xs, gcfg)
    for i, (x, h) in enumerate(zip(xs, host)):
        a = S.amax_tensor(h)
        kc, ks, _ = fos.quantize(x, gcfg, amax=torch.from_numpy(a).to(DEV))
        rc, rs, ra = fos.quantize(x, rcfg)
        torch.cuda.synchronize()
        oc, os_ = S.quantize(h, ocfg, a)
        tag = "medium %s %s %d" % (dt, mode, i)
        _same(la[i], a, tag + " list amax")
        for name, c, s in (("given", kc, ks), ("list", lc[i], ls[i])):
            _same(s, os_, "%s %s scales" % (tag, name))
            _same(c, oc, "%s %s codes" % (tag, name))
        r_a = S.amax_rows(h)
        _same(ra, r_a, tag + " row amax")
        roc, ros = S.quantize(h, rocfg, r_a)
        _same(rs, ros, tag + " row scales")
        _same(rc, roc, tag + " row codes")
    n_a = S.amax_rows(nh)
    nc, ns, na = fos.quantize(narrow, rcfg)
    torch.cuda.synchronize()
    _same(na, n_a, "narrow row amax")
    noc, nos = S.quantize(nh, rocfg, n_a)
    _same(ns, nos, "narrow %s %s scales" % (dt, mode))
    _same(nc, noc, "narrow %s %s codes" % (dt, mode))


@pytest.mark.parametrize("dt", list(MED_DT))
@pytest.mark.parametrize("mode", TREE)
def test_medium_16x16_and_grouped_steady_state(medium, dt, mode):
    """4096x4096 fp16 / fp32: 16x16 per tensor, 16x16 per row (tile-uniform
    amax of 256-row groups), and 1x16 grouped (8 groups of 512 rows), every
    row."""
    xs, host, _, _ = medium[dt]
    x, h = xs[0], host[0]
    tcfg, tocfg = _cfgs(mode, b16=True)
    a = S.amax_tensor(h)
    tc, ts, ta = fos.quantize(x, tcfg)
    ra_groups = np.array([S.amax_tensor(h[g * 256:(g + 1) * 256])[0] for g in range(16)],
                         np.float32)
    rowamax = np.repeat(ra_groups, 256)
    rcfg, rocfg = _cfgs(mode, row=True, b16=True)
    rc, rs, _ = fos.quantize(x, rcfg, amax=torch.from_numpy(rowamax).to(DEV))
    offs = torch.arange(1, 9, dtype=torch.int32) * 512
    gcfg, gocfg = _cfgs(mode, row=True)
    gcfg = dataclasses.replace(gcfg, row_scaled=False)
    gc, gs, ga = fos.quantize_grouped(x, offs.to(DEV), gcfg)
    torch.cuda.synchronize()
    tag = "medium %s %s" % (dt, mode)
    _same(ta, a, tag + " amax")
    oc, os_ = S.quantize(h, tocfg, a)
    _same(ts, os_, tag + " 16x16 scales")
    _same(tc, oc, tag + " 16x16 codes")
    roc, ros = S.quantize(h, rocfg, rowamax)
    _same(rs, ros, tag + " 16x16 row scales")
    _same(rc, roc, tag + " 16x16 row codes")
    g_a = np.array([S.amax_tensor(h[g * 512:(g + 1) * 512])[0] for g in range(8)], np.float32)
    _same(ga, g_a, tag + " group amax")
    goc, gos = S.quantize(h, gocfg, np.repeat(g_a, 512))
    _same(gs, gos, tag + " grouped scales")
    _same(gc, goc, tag + " grouped codes")
