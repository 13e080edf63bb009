"""GPU parity at the full workload sizes, launched the way the benchmark
launches them: the weight tiles (14336x4096, 16x16), the fake-QAT QDQ list
(8 x 2048x7168), the packed MoE activations (65536x7168 in 64 groups) and the
flattened expert stack (64 x 2048x7168, 16x16).  The device computes every
output; the oracle recomputes sampled rows (or 16-row tile bands) from the
same bytes, with the global amax it computes itself over the whole tensor,
and the two must agree bit for bit."""
import numpy as np
import pytest
import torch

import nvfp4_quantization_precision_gb300 as fos
import oracle
import workloads

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _u16(a):
    return a.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _u32(a):
    return a.cpu().contiguous().view(torch.int32).numpy().view(np.uint32)


def _bands(n_bands, k, seed):
    """k distinct 16-row tile bands out of n_bands, always including the last."""
    b = np.random.default_rng(seed).choice(n_bands - 1, k - 1, replace=False)
    return np.sort(np.append(b, n_bands - 1))


def _band_rows(bands):
    return (bands[:, None] * 16 + np.arange(16)[None, :]).ravel()


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
def test_weight_16x16_full_size_sampled(dt):
    """14336x4096 weight, N(0, 0.02) with 0.05 % x50 outliers, 16x16 tiles,
    per-tensor amax computed on the device, MSE exact, E4M3 448; then the
    codes are dequantized back to bf16 on the device."""
    R, C = 14336, 4096
    w = workloads.weight(R, C, seed=0, dtype=dt, device=DEV)
    gcfg = fos.Config(block16x16=True)
    gc, gs, ga = fos.quantize(w, gcfg)
    deq = fos.dequantize(gc, gs, ga, gcfg, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    wf = w.cpu().float().numpy()
    a = oracle.amax_tensor(wf)
    assert np.array_equal(_u32(ga), a.view(np.uint32))
    bands = _bands(R // 16, 12, seed=1)
    rows = _band_rows(bands)
    ocfg = oracle.Config(block16x16=True, amax_is_input=True)
    oc, os_, _ = oracle.quantize(wf[rows], ocfg, amax=a)
    assert np.array_equal(gc.cpu().numpy()[rows], oc)
    assert np.array_equal(gs.cpu().numpy()[bands], os_)
    od = oracle.dequantize(oc, os_, a, ocfg, "bf16")
    assert np.array_equal(_u16(deq)[rows], od)


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("mode", ["std", "mae_f16", "mse_f16", "mse", "mae_f16_seq",
                                  "mse_f16_seq"])
def test_qdq_list_full_size_sampled(dt, mode):
    """Eight 2048x7168 weights, N(0, 0.02) with 0.1 % x30 outliers, with the
    caller's FP32 per-tensor amax, fused QDQ of the whole list in one call
    (the *_seq modes sum error terms in element order)."""
    four = mode != "std"
    mse = not mode.startswith("mae")
    f16 = "f16" in mode
    seq = mode.endswith("_seq")
    gcfg = fos.Config(four_over_six=four, mse=mse, err_f16=f16, seq_order=seq)
    ocfg = oracle.Config(four_over_six=four, mse=mse, err_f16=f16, amax_is_input=True,
                         seq_order=seq)
    ws = workloads.qdq_weights(8, 2048, 7168, seed=0, dtype=dt, device=DEV)
    host = [t.cpu().float().numpy() for t in ws]
    am = [oracle.amax_tensor(h) for h in host]
    outs = fos.qdq(ws, gcfg, amaxes=[torch.from_numpy(a).to(DEV) for a in am])
    torch.cuda.synchronize()
    kind = "bf16" if dt == torch.bfloat16 else "f16"
    rng = np.random.default_rng(2)
    for h, a, o in zip(host, am, outs):
        rows = np.sort(np.append(rng.choice(2047, 15, replace=False), 2047))
        ref, _ = oracle.qdq(h[rows], ocfg, kind, amax=a)
        assert np.array_equal(_u16(o)[rows], ref), mode


def test_grouped_moe_full_size_sampled():
    """65536x7168 bf16 tokens in 64 lognormal groups (4 empty, the last end
    below the row count), per-group amax computed on the device, 4/6 MSE:
    group amax over the whole tensor, sampled live rows, zero tail rows."""
    R, C, G = 65536, 7168, 64
    offs = workloads.moe_offsets(R, G, seed=0)
    x = workloads.moe_activations(R, C, offs, seed=0, device=DEV)
    gcfg = fos.Config()
    gc, gs, ga = fos.quantize_grouped(x, offs.to(DEV), gcfg)
    torch.cuda.synchronize()
    ends = offs.numpy().astype(np.int64)
    live = int(ends[-1])
    # the oracle's group amax, one group at a time (bounded host memory)
    ref = np.zeros(G, np.float32)
    lo = 0
    for g, hi in enumerate(ends):
        if hi > lo:
            ref[g] = oracle.amax_tensor(x[lo:hi].cpu().float().numpy())[0]
        lo = max(lo, hi)
    assert np.array_equal(_u32(ga), ref.view(np.uint32))
    rng = np.random.default_rng(3)
    rows = np.sort(np.concatenate([rng.choice(live, 64, replace=False), [0, live - 1]]))
    grp = np.searchsorted(ends, rows, side="right")
    ocfg = oracle.Config(row_scaled=True, amax_is_input=True)
    oc, os_, _ = oracle.quantize(x[torch.from_numpy(rows).to(DEV)].cpu().float().numpy(), ocfg,
                                 amax=ref[grp])
    assert np.array_equal(gc.cpu().numpy()[rows], oc)
    assert np.array_equal(gs.cpu().numpy()[rows], os_)
    tail = np.arange(live, R)
    assert not gc.cpu().numpy()[tail].any() and not gs.cpu().numpy()[tail].any()


def test_moe_experts_16x16_full_size_sampled():
    """64 experts x 2048x7168 bf16, each with its own amax, 16x16 tiles, in one
    flattened call with the expert amax expanded to its rows; the grouped
    entry point over the same stack (one group per expert) gives the same
    bytes."""
    E, R, C = 64, 2048, 7168
    x = workloads.moe_experts(E, R, C, seed=0, device=DEV).view(E * R, C)
    ea = torch.stack([fos.amax(x[e * R:(e + 1) * R])[0] for e in range(E)])
    rowamax = ea.repeat_interleave(R)
    gcfg = fos.Config(block16x16=True, row_scaled=True)
    gc, gs, _ = fos.quantize(x, gcfg, amax=rowamax)
    offs = torch.arange(1, E + 1, dtype=torch.int32, device=DEV) * R
    qc, qs, qa = fos.quantize_grouped(x, offs, fos.Config(block16x16=True), group_amax=ea)
    torch.cuda.synchronize()
    assert torch.equal(gc, qc) and torch.equal(gs, qs)
    eh = np.zeros(E, np.float32)
    for e in range(E):
        eh[e] = oracle.amax_tensor(x[e * R:(e + 1) * R].cpu().float().numpy())[0]
    assert np.array_equal(_u32(ea), eh.view(np.uint32))
    bands = _bands(E * R // 16, 16, seed=4)
    rows = _band_rows(bands)
    ocfg = oracle.Config(block16x16=True, row_scaled=True, amax_is_input=True)
    oc, os_, _ = oracle.quantize(x[torch.from_numpy(rows).to(DEV)].cpu().float().numpy(), ocfg,
                                 amax=eh[rows // R])
    assert np.array_equal(gc.cpu().numpy()[rows], oc)
    assert np.array_equal(gs.cpu().numpy()[bands], os_)


def test_mm_full_size_sampled():
    """The benchmark's product, 8192x4096 activation times a 14336x4096
    weight (4/6 MSE, per-tensor scales): the amaxes the oracle computes over
    the whole tensors equal the device's, and sampled entries of out meet the
    oracle's product reference of the sampled rows within its fp32 bound."""
    M, N, K = 8192, 14336, 4096
    c = fos.Config()
    a = workloads.activation(M, K, "F1", seed=0, device=DEV)
    w = workloads.weight(N, K, seed=0, device=DEV)
    ca, sa, aa = fos.quantize(a, c)
    cw, sw, aw = fos.quantize(w, c)
    out = fos.mm(ca, fos.swizzle_scales(sa, M, K), aa, cw, fos.swizzle_scales(sw, N, K), aw, c)
    torch.cuda.synchronize()
    oa = oracle.amax_tensor(a.cpu().float().numpy())
    ow = oracle.amax_tensor(w.cpu().float().numpy())
    assert np.array_equal(_u32(aa), oa.view(np.uint32)) and np.array_equal(_u32(aw),
                                                                             ow.view(np.uint32))
    rng = np.random.default_rng(6)
    ra = np.sort(rng.choice(M, 8, replace=False))
    rw = np.sort(rng.choice(N, 16, replace=False))
    ocfg = oracle.Config(amax_is_input=True)
    oca, osa, _ = oracle.quantize(a[torch.from_numpy(ra).to(DEV)].cpu().float().numpy(), ocfg,
                                  amax=oa)
    ocw, osw, _ = oracle.quantize(w[torch.from_numpy(rw).to(DEV)].cpu().float().numpy(), ocfg,
                                  amax=ow)
    ref, bound = oracle.mm_reference(oca, osa, oa, ocw, osw, ow, oracle.Config())
    got = out.cpu().numpy()[np.ix_(ra, rw)].astype(np.float64)
    assert np.all(np.abs(got - ref) <= bound + 1e-30)


def test_past_2_to_31_elements_sampled():
    """A bf16 tensor of 524352 x 4096 = 2^31 + 2^18 elements (element 2^31 is
    row 524288, column 0), amax 5.0 by construction: the per-tensor and
    per-row 1x16 quantize, the 16x16 quantize, the dequantize, the fused QDQ
    and the column-wise operand, each on rows (or columns) on both sides of
    the 2^31 boundary and at the end, against the oracle bit for bit."""
    R, C = 524352, 4096
    x = workloads.large_activation(R, C, seed=3, device=DEV)
    rows = np.array([0, 1, 524272, 524287, 524288, 524289, 524303, R - 16, R - 1])
    ridx = torch.from_numpy(rows).to(DEV)
    xs = x[ridx].cpu().float().numpy()
    five = np.array([5.0], np.float32)
    given = oracle.Config(amax_is_input=True)

    codes, scales, amax = fos.quantize(x, fos.Config())
    torch.cuda.synchronize()
    assert np.array_equal(_u32(amax), five.view(np.uint32))
    oc, os_, _ = oracle.quantize(xs, given, amax=five)
    assert np.array_equal(codes[ridx].cpu().numpy(), oc)
    assert np.array_equal(scales[ridx].cpu().numpy(), os_)
    deq = fos.dequantize(codes, scales, amax, fos.Config(), out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    od = oracle.dequantize(oc, os_, five, given, "bf16")
    assert np.array_equal(_u16(deq[ridx]), od)
    del codes, scales, deq

    out = fos.qdq([x], fos.Config(), amaxes=[amax])[0]
    torch.cuda.synchronize()
    oq, _ = oracle.qdq(xs, given, "bf16", amax=five)
    assert np.array_equal(_u16(out[ridx]), oq)
    del out

    rc, rs, ra = fos.quantize(x, fos.Config(row_scaled=True))
    torch.cuda.synchronize()
    orc_, ors, ora = oracle.quantize(xs, oracle.Config(row_scaled=True))
    assert np.array_equal(_u32(ra[ridx]), ora.view(np.uint32))
    assert np.array_equal(rc[ridx].cpu().numpy(), orc_)
    assert np.array_equal(rs[ridx].cpu().numpy(), ors)
    del rc, rs, ra

    bands = np.array([0, 524288 // 16 - 1, 524288 // 16, R // 16 - 1])
    brows = torch.from_numpy(_band_rows(bands)).to(DEV)
    tc, ts, _ = fos.quantize(x, fos.Config(block16x16=True), amax=amax)
    torch.cuda.synchronize()
    otc, ots, _ = oracle.quantize(x[brows].cpu().float().numpy(),
                                  oracle.Config(block16x16=True, amax_is_input=True), amax=five)
    assert np.array_equal(tc[brows].cpu().numpy(), otc)
    assert np.array_equal(ts[torch.from_numpy(bands).to(DEV)].cpu().numpy(), ots)
    del tc, ts

    cols = np.array([0, 2047, C - 2, C - 1])
    ct, st, _ = fos.quantize_colwise(x, fos.Config(), amax=amax)
    torch.cuda.synchronize()
    xc = x[:, torch.from_numpy(cols).to(DEV)].cpu().float().numpy()
    octc, octs, _ = oracle.quantize_colwise(xc, given, amax=five)
    cidx = torch.from_numpy(cols).to(DEV)
    assert np.array_equal(ct[cidx].cpu().numpy(), octc)
    assert np.array_equal(st[cidx].cpu().numpy(), octs)
