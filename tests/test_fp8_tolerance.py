"""The fp8 oracle and the fp8 parity bound (tests/fp8_util.py), on the CPU.

The oracle of the fp8 forward is standard attention on the dequantised
inputs; closed forms pin each dequantisation factor's role.  The bound is
neither too loose nor too tight: an emulation of the kernel's arithmetic
(online softmax over 128-key tiles, P rounded to e4m3 against the running
max, l from the unrounded P, bf16 output) stays inside both the per-element
and the root-mean-square bounds, and the same emulation with plausible
kernel mistakes falls outside them.
"""
import math

import numpy as np
import pytest
import torch

import fp8_util
import oracle


def _e4m3(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float64)).float().to(torch.float8_e4m3fn).double().numpy()


def _bf16(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float64)).to(torch.bfloat16).double().numpy()


def _quantised(rng, n, d, std):
    x = rng.standard_normal((n, d)) * std
    f = 2.0 ** math.ceil(math.log2(np.abs(x).max() / 448.0))
    return _e4m3(x / f), f


# ------------------------------------------------------------------ oracle pins
def test_constant_v_rows_give_that_row_times_the_v_factor():
    rng = np.random.default_rng(0)
    for causal in (False, True):
        q8, qd = _quantised(rng, 9, 8, 1.0)
        k8, kd = _quantised(rng, 9, 8, 1.0)
        row = _e4m3(rng.standard_normal(8))
        v8 = np.tile(row, (9, 1))
        o, _ = oracle.attention_fp8_head(q8, k8, v8, qd, kd, 0.375, 0.3, causal)
        assert np.allclose(o, np.tile(row * 0.375, (9, 1)), rtol=0, atol=1e-13)


def test_zero_queries_give_the_mean_of_dequantised_values():
    rng = np.random.default_rng(1)
    n, d = 12, 4
    k8, kd = _quantised(rng, n, d, 1.0)
    v8, vd = _quantised(rng, n, d, 1.0)
    o, lse = oracle.attention_fp8_head(np.zeros((n, d)), k8, v8, 0.5, kd, vd, 0.5, False)
    assert np.allclose(o, np.tile(v8.mean(0) * vd, (n, 1)), atol=1e-13)
    assert np.allclose(lse, math.log(n), atol=1e-13)
    o, lse = oracle.attention_fp8_head(np.zeros((n, d)), k8, v8, 0.5, kd, vd, 0.5, True)
    for i in range(n):
        assert np.allclose(o[i], v8[:i + 1].mean(0) * vd, atol=1e-13)
        assert abs(lse[i] - math.log(i + 1)) < 1e-13


def test_query_and_key_factors_multiply_the_logits():
    """S = (qd Q8)(kd K8)^T * scale: the factors act exactly like a larger scale."""
    rng = np.random.default_rng(2)
    q8, k8, v8 = (_e4m3(rng.standard_normal((7, 16))) for _ in range(3))
    for causal in (False, True):
        o, lse = oracle.attention_fp8_head(q8, k8, v8, 0.25, 3.0, 1.0, 0.2, causal)
        o2, lse2 = oracle.attention_head(q8, k8, v8, 0.2 * 0.25 * 3.0, causal)
        assert np.allclose(o, o2, atol=1e-13) and np.allclose(lse, lse2, atol=1e-13)
        o3, _ = oracle.attention_fp8_head(q8, k8, v8, 1.0, 1.0, 1.0, 0.2, causal)
        assert not np.allclose(o, o3, atol=1e-3)


# ------------------------------------------------------------------ emulation of the kernel's arithmetic
def _emulate(q8, qd, k8, kd, v8, vd, scale, causal, bk=128, mistake=None):
    """O, L of one head the way the kernel rounds (fp64 stands in for fp32)."""
    n, d = q8.shape
    q = q8 * qd
    k = k8 * (1.0 if mistake == "no_k_factor" else kd)
    m = np.full(n, -np.inf)
    l = np.zeros(n)
    acc = np.zeros((n, d))
    rows = np.arange(n)
    for k0 in range(0, n, bk):
        cols = np.arange(k0, min(n, k0 + bk))
        s = (q @ k[cols].T) * scale
        if causal:
            lead = 1 if mistake == "mask_leak" else 0  # mistake: one future key visible
            vis = cols[None, :] <= rows[:, None] + lead
            s = np.where(vis, s, -np.inf)
        m_new = np.maximum(m, s.max(axis=1))
        base = np.where(np.isfinite(m_new), m_new, 0.0)
        alpha = np.where(np.isfinite(m), np.exp(m - base), 0.0)
        p = np.exp(s - base[:, None])
        p8 = _e4m3(p)
        l = l * alpha + p.sum(axis=1)
        if mistake == "no_rescale":
            alpha = np.ones_like(alpha)
        acc = acc * alpha[:, None] + p8 @ v8[cols]
        m = m_new
    vf = 1.0 if mistake == "no_v_factor" else vd
    with np.errstate(divide="ignore", invalid="ignore"):
        o = _bf16(acc * vf / l[:, None])
    return o, m + np.log(l)


def _case(n, d, causal, std, seed):
    rng = np.random.default_rng(seed)
    q8, qd = _quantised(rng, n, d, std)
    k8, kd = _quantised(rng, n, d, std)
    v8, vd = _quantised(rng, n, d, 1.0)
    return q8, qd, k8, kd, v8, vd, 1.0 / math.sqrt(d)


def _grade(case, causal, mistake=None):
    q8, qd, k8, kd, v8, vd, scale = case
    o, lse = _emulate(q8, qd, k8, kd, v8, vd, scale, causal, mistake=mistake)
    o_ref, l_ref = oracle.attention_fp8_head(q8, k8, v8, qd, kd, vd, scale, causal)
    e, sig2 = fp8_util.head_bounds(q8 * qd, k8 * kd, v8 * vd, scale, causal)
    return fp8_util.compare_head(o, lse, o_ref, l_ref, e, sig2)


@pytest.mark.parametrize("n,d,causal,std", [(300, 128, True, 1.0), (300, 128, False, 1.0), (520, 64, True, 3.0),
                                            (257, 128, False, 3.0), (1100, 128, True, 1.0)])
def test_emulated_kernel_is_inside_both_bounds(n, d, causal, std):
    r = _grade(_case(n, d, causal, std, n + d), causal)
    assert r["ok"], r
    # not vacuous: the rounding uses a visible share of the statistical bound
    # (least on the nearly one-hot rows of the std-3 logits, whose dominant weight rounds exactly)
    assert r["rms_ratio"] > 0.05, r


@pytest.mark.parametrize("mistake", ["no_v_factor", "no_k_factor", "mask_leak", "no_rescale"])
def test_plausible_kernel_mistakes_are_outside_the_bounds(mistake):
    causal = mistake in ("mask_leak", "no_rescale")
    r = _grade(_case(400, 128, causal, 1.0, 7), causal, mistake=mistake)
    assert not r["ok"], r
    assert r["rms_ratio"] > 3 or r["worst_err_over_elem_bound"] > 3 or r["max_err_L"] > 1e-2, r


def test_quantised_inputs_follow_the_recipe():
    """make_qkv_fp8: power-of-two factors, amax just inside e4m3's range, the same draws as make_qkv."""
    from tiled_attention_fwd_gb300.inputs import Workload, make_qkv, make_qkv_fp8

    w = Workload("fp8_recipe", 1, 2, 64, 32, "fp8", True, seed=5, qk_std=3.0)
    (q8, k8, v8), scales = make_qkv_fp8(w)
    ref = make_qkv(w.with_(dtype="f32"))
    for x8, f, x in zip((q8, k8, v8), scales, ref):
        assert x8.dtype == torch.float8_e4m3fn
        assert math.log2(f) == int(math.log2(f))
        deq = x8.double() * f
        assert 224.0 < float(x8.double().abs().max()) <= 448.0
        assert torch.allclose(deq, x.double(), rtol=2.0 ** -4, atol=2.0 ** -10 * f)
