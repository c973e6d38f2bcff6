"""Seeded random cases of the forward and backward passes against the fp64
oracle: random B, H, Nq, Nk (1..600), head dimension, mask, scale and memory
layout of every tensor (contiguous, [B, N, H, d], rows padded to a wider
stride).  Each case is small; together they cover combinations the explicit
parity tests do not list one by one."""
import numpy as np
import pytest
import torch

import bwd_util
import oracle
from parity_util import compare
from tiled_attention_fwd_gb300 import backward, check_status, forward
from tiled_attention_fwd_gb300.inputs import as_f64_numpy

pytestmark = pytest.mark.gpu

LAYOUTS = ("bhnd", "bnhd", "padded")


def _placed(x: torch.Tensor, layout: str, dev, fill=None):
    """x [B, H, N, d] copied into a tensor of the given layout on dev, returned as a [B, H, N, d] view."""
    B, H, N, d = x.shape
    if layout == "bhnd":
        t = torch.empty((B, H, N, d), device=dev, dtype=x.dtype)
    elif layout == "bnhd":
        t = torch.empty((B, N, H, d), device=dev, dtype=x.dtype).permute(0, 2, 1, 3)
    else:  # each row padded by 8 elements, each head by one row
        store = torch.empty((B, H, N + 1, d + 8), device=dev, dtype=x.dtype)
        t = store[:, :, :N, :d]
    if fill is None:
        t.copy_(x.to(dev))
    else:
        t.fill_(fill)
    return t


def _case(rng):
    B, H = int(rng.integers(1, 3)), int(rng.integers(1, 4))
    nq = int(rng.choice([1, 2, 63, 64, 65, 127, 128, 129, 200, 255, 256, 257, 383, 511, 600]))
    nk = nq if rng.random() < 0.4 else int(rng.integers(1, 601))
    d = int(rng.choice([32, 64, 128, 256]))
    causal = bool(rng.random() < 0.5)
    scale = float(rng.uniform(0.05, 0.3))
    std = float(rng.choice([1.0, 2.0]))
    layouts = [LAYOUTS[int(rng.integers(0, 3))] for _ in range(8)]
    return B, H, nq, nk, d, causal, scale, std, layouts


def _rand(shape, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * std).to(torch.bfloat16)


@pytest.mark.parametrize("case", range(24))
def test_forward_random_case(case):
    rng = np.random.default_rng(1000 + case)
    B, H, nq, nk, d, causal, scale, std, lay = _case(rng)
    dev = torch.device("cuda", 0)
    q = _rand((B, H, nq, d), 10 * case + 1, std)
    k = _rand((B, H, nk, d), 10 * case + 2, std)
    v = _rand((B, H, nk, d), 10 * case + 3)
    qd, kd, vd = (_placed(t, lay[i], dev) for i, t in enumerate((q, k, v)))
    o = _placed(torch.empty((B, H, nq, d), dtype=torch.bfloat16), lay[3], dev, fill=float("nan"))
    lse = torch.full((B, H, nq), float("nan"), device=dev, dtype=torch.float32)
    forward(qd, kd, vd, causal=causal, scale=scale, out=o, lse=lse)
    check_status(dev)
    o_ref, l_ref = oracle.attention(as_f64_numpy(q), as_f64_numpy(k), as_f64_numpy(v), scale, causal)
    r = compare(as_f64_numpy(o.cpu()), lse.cpu().double().numpy(), o_ref, l_ref, "bf16")
    assert r["ok"], (B, H, nq, nk, d, causal, scale, lay[:4], r)


@pytest.mark.parametrize("case", range(16))
def test_backward_random_case(case):
    rng = np.random.default_rng(2000 + case)
    B, H, nq, nk, d, causal, scale, std, lay = _case(rng)
    dev = torch.device("cuda", 0)
    q = _rand((B, H, nq, d), 10 * case + 4, std)
    k = _rand((B, H, nk, d), 10 * case + 5, std)
    v = _rand((B, H, nk, d), 10 * case + 6)
    do = _rand((B, H, nq, d), 10 * case + 7)
    qd, kd, vd, dod = (_placed(t, lay[i], dev) for i, t in enumerate((q, k, v, do)))
    o = _placed(torch.empty((B, H, nq, d), dtype=torch.bfloat16), lay[4], dev, fill=float("nan"))
    lse = torch.empty((B, H, nq), device=dev, dtype=torch.float32)
    forward(qd, kd, vd, causal=causal, scale=scale, out=o, lse=lse)
    grads = tuple(_placed(torch.empty(t.shape, dtype=torch.bfloat16), lay[5 + i], dev, fill=float("nan"))
                  for i, t in enumerate((q, k, v)))
    backward(qd, kd, vd, o, lse, dod, causal=causal, scale=scale, out=grads)
    check_status(dev)
    qn, kn, vn, don = (as_f64_numpy(t) for t in (q, k, v, do))
    on = as_f64_numpy(o.cpu())
    got = [as_f64_numpy(g.cpu()) for g in grads]
    worst = 0.0
    for b in range(B):
        for h in range(H):
            ref, mag = bwd_util.head_bounds(qn[b, h], kn[b, h], vn[b, h], don[b, h], on[b, h], scale, causal)
            ok, r = bwd_util.compare_head((got[0][b, h], got[1][b, h], got[2][b, h]), ref, mag)
            worst = max(worst, r)
            assert ok, (B, H, nq, nk, d, causal, scale, lay, b, h, r)
