"""fos_qdq_fused_static, the allocation-free form of the fused amax + QDQ
list call, for callers that cannot obtain device memory when they call in
(code running under another framework's allocator, or a runtime that allows
no allocations after start-up).  It keeps the counters of the fused launch in
a fixed array of the library instead of a caller workspace.

Checked through the C ABI against fos_qdq_fused (with a workspace of its own)
on the same inputs, bit for bit, on two calls in a row: the second call finds
the array as the first one left it and must clear it itself.  This file is
collected last so that a run stopping at its first failure has already run
every other test; it also passes alone in a fresh process."""
import ctypes

import pytest
import torch

import nvfp4_quantization_precision_gb300 as fos
import workloads

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _static(xs, outs, amaxes, cfg):
    L = fos.lib()
    f = L.fos_qdq_fused_static
    P = ctypes.c_void_p
    f.argtypes = [ctypes.c_int, P, P, P, P, P, ctypes.c_int, ctypes.POINTER(fos.FosConfig), P]
    f.restype = ctypes.c_int
    n = len(xs)
    A = P * max(n, 1)
    xp = A(*[x.data_ptr() for x in xs])
    op = A(*[o.data_ptr() for o in outs])
    ap = A(*[a.data_ptr() for a in amaxes])
    rows = (ctypes.c_int64 * max(n, 1))(*[x.shape[0] for x in xs])
    cols = (ctypes.c_int64 * max(n, 1))(*[x.shape[1] for x in xs])
    cc = cfg.c(False)
    dt = 0 if (n == 0 or xs[0].dtype == torch.bfloat16) else 1
    stream = P(torch.cuda.current_stream().cuda_stream)
    return f(n, xp, op, rows, cols, ap, dt, ctypes.byref(cc), stream)


@pytest.mark.parametrize("dt,cfg", [
    (torch.bfloat16, fos.Config(err_f16=True, seq_order=True)),
    (torch.float16, fos.Config(four_over_six=False)),
    (torch.bfloat16, fos.Config(mse=False)),
])
def test_static_form_matches_the_workspace_form_twice(dt, cfg):
    shapes = [(64, 1024), (0, 64), (7, 1040), (2048, 7168), (48, 272), (1, 16)]
    xs = [workloads.qdq_weights(1, r, c, seed=200 + i, dtype=dt, device=DEV)[0] if r else
          torch.zeros(0, c, dtype=dt, device=DEV) for i, (r, c) in enumerate(shapes)]
    ref_out, ref_amax = fos.qdq_fused(xs, cfg)
    for _ in range(2):
        outs = [torch.full_like(x, 7.0) for x in xs]
        amaxes = [torch.full((1,), -1.0, device=DEV) for _ in xs]
        assert _static(xs, outs, amaxes, cfg) == fos.FOS_OK
        torch.cuda.synchronize()
        for o, r, a, b in zip(outs, ref_out, amaxes, ref_amax):
            assert torch.equal(o.view(torch.int16), r.view(torch.int16))
            assert torch.equal(a, b)


def test_static_form_rejects_lists_beyond_its_array():
    xs = [torch.zeros(16, 16, dtype=torch.bfloat16, device=DEV) for _ in range(65)]
    outs = [torch.empty_like(x) for x in xs]
    amaxes = [torch.empty(1, device=DEV) for _ in xs]
    assert _static(xs, outs, amaxes, fos.Config()) == fos.FOS_ERR_UNSUPPORTED
