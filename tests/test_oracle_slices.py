"""The row-slice front end of the oracle (oracle_slices.py), used by the
full-size GPU tests, gives exactly what one oracle call over the whole input
gives: same amaxes, codes, scales, QDQ and dequantized outputs."""
import numpy as np
import pytest
import torch

import oracle
import oracle_slices as S
import workloads


def _x(rows, cols, fam, seed):
    return workloads.activation(rows, cols, fam, seed=seed, dtype=torch.bfloat16).float().numpy()


@pytest.mark.parametrize("b16", [False, True])
@pytest.mark.parametrize("row", [False, True])
@pytest.mark.parametrize("mode", [(False, True, False), (True, False, True), (True, True, False)])
def test_slices_equal_one_call(orc, b16, row, mode):
    four, mse, f16 = mode
    x = _x(400 if b16 else 389, 272, "F4", 3)
    if b16:
        x = x[:384]
    cfg = oracle.Config(block16x16=b16, four_over_six=four, mse=mse, err_f16=f16,
                        row_scaled=row, amax_is_input=True)
    if row:
        a = oracle.amax_rows(x)
        if b16:
            a = np.repeat(a.reshape(-1, 16).max(1), 16)
    else:
        a = oracle.amax_tensor(x)
    oc, os_, _ = oracle.quantize(x, cfg, amax=a)
    sc, ss = S.quantize(x, cfg, a)
    assert np.array_equal(sc, oc) and np.array_equal(ss, os_)
    od = oracle.dequantize(oc, os_, a, cfg, "bf16")
    assert np.array_equal(S.dequantize(oc, os_, a, cfg, "bf16"), od)
    if not b16:
        oq, _ = oracle.qdq(x, cfg, "f16", amax=a)
        assert np.array_equal(S.qdq(x, cfg, "f16", a), oq)


def test_slice_amaxes(orc):
    x = _x(300, 64, "F2", 4)
    x[17, 5] = np.nan
    assert np.array_equal(S.amax_tensor(x).view(np.uint32),
                          oracle.amax_tensor(x).view(np.uint32))
    assert np.array_equal(S.amax_rows(x).view(np.uint32), oracle.amax_rows(x).view(np.uint32))
    z = np.zeros((5, 16), np.float32)
    assert S.amax_tensor(z)[0] == 0.0
