"""The backward parity bound (tests/bwd_util.py) is neither too loose nor too tight.

On the CPU: an emulation of the kernel's rounding (bf16 inputs and O, P and dS
rounded to bf16 before their products, fp32 D from the bf16 O, bf16 outputs)
stays inside the bound, and the same emulation with plausible kernel mistakes
falls outside it.
"""
import math

import numpy as np
import pytest
import torch

import bwd_util
import oracle


def _bf16(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float64)).to(torch.bfloat16).double().numpy()


def _emulated_kernel(q, k, v, do, scale, causal, mistake=None):
    """Gradients the way the kernel rounds them (fp64 stands in for fp32 accumulation)."""
    p = oracle.probabilities(oracle.scores(q, k, scale, causal))
    o = _bf16(p @ v)                                  # forward output, bf16
    dsum = (do * o).sum(1, keepdims=True)             # D from the bf16 O
    if mistake == "no_d":
        dsum = 0 * dsum
    dp = do @ v.T
    if mistake == "dp_uses_k":
        dp = do @ k.T
    ds = p * (dp - dsum)
    if mistake == "mask_off" and causal:
        p2 = oracle.probabilities(oracle.scores(q, k, scale, False))
        ds = p2 * (dp - dsum)
        p = p2
    pb, dsb = _bf16(p), _bf16(ds)
    dv = _bf16(pb.T @ do)
    dk = _bf16(scale * (dsb.T @ q))
    dq = _bf16(scale * (dsb @ k))
    if mistake == "dk_unscaled":
        dk = _bf16(dsb.T @ q)
    return (dq, dk, dv), o


@pytest.mark.parametrize("n,d,causal", [(64, 32, False), (96, 64, True), (200, 128, True), (130, 64, False)])
def test_emulated_kernel_is_inside_the_bound(n, d, causal):
    rng = np.random.default_rng(n + d)
    q, k, v, do = (_bf16(rng.standard_normal((n, d)) * s) for s in (3.0, 3.0, 1.0, 1.0))
    scale = 1 / math.sqrt(d)
    got, o = _emulated_kernel(q, k, v, do, scale, causal)
    ref, mag = bwd_util.head_bounds(q, k, v, do, o, scale, causal)
    ok, worst = bwd_util.compare_head(got, ref, mag)
    assert ok, worst
    assert worst > 1e-3  # the bound is not vacuous: rounding uses a visible part of it


@pytest.mark.parametrize("mistake", ["no_d", "dp_uses_k", "mask_off", "dk_unscaled"])
def test_plausible_kernel_mistakes_are_outside_the_bound(mistake):
    n, d = 96, 64
    causal = True
    rng = np.random.default_rng(5)
    q, k, v, do = (_bf16(rng.standard_normal((n, d)) * s) for s in (1.0, 1.0, 1.0, 1.0))
    scale = 1 / math.sqrt(d)
    got, o = _emulated_kernel(q, k, v, do, scale, causal, mistake)
    ref, mag = bwd_util.head_bounds(q, k, v, do, o, scale, causal)
    ok, worst = bwd_util.compare_head(got, ref, mag)
    assert not ok and worst > 10
