"""Seeded synthetic inputs shaped like the workloads on the pages.

This module holds no step of the quantizer: it only draws random tensors
(float32, then one round-to-nearest-even cast to the storage dtype) so that the
CUDA library and the CPU oracle see identical bytes.  Both the tests and the
benchmark draw from here.

Families (activation rows, 1x16 blocks along the last axis):
  F1  N(0, 1)
  F2  N(0, 1) with round(0.001 * n) entries, chosen without replacement, x100
  F3  U(-1, 1)
  F4  N(0, 1) with 25 % of the 16-element row blocks replaced: one third all
      zero (half +0, half -0), one third scaled by 1e-4, one third by 1e-7
Large activation (past 2^31 elements): N(0, 1) clipped to [-4, 4] plus one
planted 5.0, so that its amax is known without reading it.
Weights: N(0, 0.02) with 0.05 % of entries x50.
Fake-QAT weight list: N(0, 0.02) with 0.1 % of entries x30.
MoE: token-group sizes ~ round(lognormal(0, 1)) scaled to about 94 % of the
rows (a padded tail stays past the last offset), four groups forced empty,
group values N(0, 1) times a per-group lognormal(0, 1) factor; expert
weights N(0, 0.02) times a per-expert lognormal(0, 0.5) factor.
"""
import math

import torch

FAMILIES = ("F1", "F2", "F3", "F4")


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _finish(x32, dtype):
    return x32 if dtype == torch.float32 else x32.to(dtype)


def activation(rows, cols, family="F1", seed=0, dtype=torch.bfloat16, device="cpu"):
    g = _gen(seed, device)
    n = rows * cols
    if family == "F3":
        x = torch.rand(rows, cols, generator=g, device=device, dtype=torch.float32) * 2.0 - 1.0
        return _finish(x, dtype)
    x = torch.randn(rows, cols, generator=g, device=device, dtype=torch.float32)
    if family == "F2":
        k = int(round(0.001 * n))
        if k:
            idx = torch.randperm(n, generator=g, device=device)[:k]
            x.view(-1)[idx] *= 100.0
    elif family == "F4":
        nblk = n // 16
        blocks = x.view(nblk, 16)
        k = nblk // 4
        pick = torch.randperm(nblk, generator=g, device=device)[:k]
        third = k // 3
        zeros = pick[:third]
        half = zeros.numel() // 2
        blocks[zeros[:half]] = 0.0
        blocks[zeros[half:]] = -0.0
        blocks[pick[third:2 * third]] *= 1e-4
        blocks[pick[2 * third:]] *= 1e-7
    elif family != "F1":
        raise ValueError(family)
    return _finish(x, dtype)


def _sparse_outliers(x, frac, factor, g, device):
    n = x.numel()
    k = int(round(frac * n))
    if k:
        idx = torch.randperm(n, generator=g, device=device)[:k]
        x.view(-1)[idx] *= factor
    return x


def weight(rows, cols, seed=0, dtype=torch.bfloat16, device="cpu"):
    g = _gen(seed, device)
    x = torch.randn(rows, cols, generator=g, device=device, dtype=torch.float32) * 0.02
    return _finish(_sparse_outliers(x, 0.0005, 50.0, g, device), dtype)


def qdq_weights(n=8, rows=2048, cols=7168, seed=0, dtype=torch.bfloat16, device="cpu"):
    out = []
    for i in range(n):
        g = _gen(seed * 1000 + i, device)
        x = torch.randn(rows, cols, generator=g, device=device, dtype=torch.float32) * 0.02
        out.append(_finish(_sparse_outliers(x, 0.001, 30.0, g, device), dtype))
    return out


def moe_offsets(rows=65536, groups=64, seed=0, n_empty=4, fill=0.94, multiple=1):
    """Cumulative group ends (int32, CPU).  The last end stays below `rows`."""
    g = _gen(seed, "cpu")
    w = torch.exp(torch.randn(groups, generator=g, dtype=torch.float64))
    empty = torch.randperm(groups, generator=g)[:n_empty]
    w[empty] = 0.0
    target = fill * rows
    sizes = torch.floor(w / w.sum() * target / multiple).to(torch.int64) * multiple
    offs = torch.cumsum(sizes, 0)
    assert int(offs[-1]) < rows
    return offs.to(torch.int32)


def moe_activations(rows, cols, offs, seed=0, dtype=torch.bfloat16, device="cpu"):
    g = _gen(seed, device)
    x = torch.randn(rows, cols, generator=g, device=device, dtype=torch.float32)
    gc = _gen(seed + 7919, "cpu")
    factors = torch.exp(torch.randn(len(offs), generator=gc, dtype=torch.float32))
    lo = 0
    for gi, hi in enumerate(offs.tolist()):
        if hi > lo:
            x[lo:hi] *= float(factors[gi])
        lo = hi
    return _finish(x, dtype)


def moe_experts(experts, rows, cols, seed=0, dtype=torch.bfloat16, device="cpu"):
    g = _gen(seed, device)
    x = torch.randn(experts, rows, cols, generator=g, device=device, dtype=torch.float32) * 0.02
    gc = _gen(seed + 104729, "cpu")
    f = torch.exp(0.5 * torch.randn(experts, generator=gc, dtype=torch.float32))
    x *= f.to(device).view(experts, 1, 1)
    return _finish(x, dtype)


def large_activation(rows, cols, seed=0, dtype=torch.bfloat16, device="cpu", chunk_rows=65536):
    """N(0, 1) clipped to [-4, 4], drawn in row chunks of float32 (so a tensor
    of several GB needs little staging), with one planted 5.0 in the last
    element: the tensor amax is 5.0 by construction."""
    g = _gen(seed, device)
    x = torch.empty(rows, cols, dtype=dtype, device=device)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        x[r0:r1] = _finish(torch.randn(r1 - r0, cols, generator=g, device=device,
                                       dtype=torch.float32).clamp_(-4.0, 4.0), dtype)
    x[rows - 1, cols - 1] = 5.0
    return x


def ceil_div(a, b):
    return -(-a // b)


def l2_rotation_copies(bytes_per_copy, l2_bytes=129 * 2**20, factor=2.0, minimum=3):
    """How many input copies to rotate so that the copies exceed factor x L2."""
    return max(minimum, int(math.ceil(factor * l2_bytes / max(1, bytes_per_copy))) + 1)
