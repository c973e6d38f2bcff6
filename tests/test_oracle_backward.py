"""Pins for the fp64 backward oracle, independent of its formula.

Each pin checks an implementation impl(q, k, v, do, scale, causal) -> (dQ, dK, dV)
on one head ([N, d] fp64) against something fixed outside it: torch's fp64
autograd through its own scaled_dot_product_attention, central finite
differences of the (separately pinned) forward oracle, and invariants that hold
exactly.  The last test plants plausible mistakes in copies of the backward
oracle and requires every one of them to fail at least one pin.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _rand(shape, seed, std=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * std


def oracle_impl(q, k, v, do, scale, causal):
    return oracle.attention_backward_head(q, k, v, do, scale, causal)


def _close(a, b, tol):
    return np.allclose(a, b, atol=tol, rtol=0)


# ----------------------------------------------------------------------------- pins
def pin_autograd(impl):
    """Brute force on tiny inputs against torch fp64 autograd of its own SDPA."""
    bad = []
    seed = 0
    for n in (1, 2, 3, 5, 8, 17):
        for d in (1, 2, 4):
            for causal in (False, True):
                seed += 1
                q, k, v, do = (_rand((n, d), seed + 100 * i) for i in range(4))
                scale = 1.0 / math.sqrt(d) * 1.7
                dq, dk, dv = impl(q, k, v, do, scale, causal)
                tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
                o = torch.nn.functional.scaled_dot_product_attention(
                    tq[None, None], tk[None, None], tv[None, None], is_causal=causal, scale=scale)[0, 0]
                o.backward(torch.from_numpy(do))
                for name, mine, ref in (("dQ", dq, tq.grad), ("dK", dk, tk.grad), ("dV", dv, tv.grad)):
                    if not _close(mine, ref.numpy(), 1e-11):
                        bad.append(f"autograd {name} n={n} d={d} causal={causal}")
    return bad


def pin_finite_differences(impl):
    """Directional derivatives of L(Q,K,V) = sum(O * dO) by central differences of the forward oracle."""
    bad = []
    rng = np.random.default_rng(11)
    for n, d, causal in ((6, 3, False), (6, 3, True), (13, 5, True), (9, 8, False)):
        q, k, v, do = (rng.standard_normal((n, d)) for _ in range(4))
        scale = 0.6

        def loss(q_, k_, v_):
            o, _ = oracle.attention_head(q_, k_, v_, scale, causal)
            return float((o * do).sum())

        dq, dk, dv = impl(q, k, v, do, scale, causal)
        h = 1e-5
        for trial in range(3):
            e = [rng.standard_normal((n, d)) for _ in range(3)]
            fd = (loss(q + h * e[0], k + h * e[1], v + h * e[2]) - loss(q - h * e[0], k - h * e[1], v - h * e[2])) / (2 * h)
            an = float((dq * e[0]).sum() + (dk * e[1]).sum() + (dv * e[2]).sum())
            if abs(fd - an) > 1e-7 * max(1.0, abs(fd)):
                bad.append(f"finite difference n={n} d={d} causal={causal} trial={trial}: {fd} vs {an}")
    return bad


def pin_invariants(impl):
    """Identities that hold exactly for the true gradients."""
    bad = []
    rng = np.random.default_rng(7)
    for n, d, causal in ((1, 4, False), (16, 4, False), (16, 4, True), (33, 8, True), (40, 2, False)):
        q, k, v, do = (rng.standard_normal((n, d)) * s for s in (2.0, 2.0, 1.0, 1.0))
        scale = 1.0 / math.sqrt(d)
        dq, dk, dv = impl(q, k, v, do, scale, causal)
        # Rows of P sum to 1, so the dV rows add up to the dO rows.
        if not _close(dv.sum(0), do.sum(0), 1e-10):
            bad.append(f"sum dV != sum dO n={n} causal={causal}")
        # Rows of dS sum to 0, so the dK rows add up to zero.
        if not _close(dk.sum(0), np.zeros(d), 1e-10):
            bad.append(f"sum dK != 0 n={n} causal={causal}")
        # Zero upstream gradient gives zero gradients.
        z = impl(q, k, v, np.zeros_like(do), scale, causal)
        if any(np.abs(x).max() > 0 for x in z):
            bad.append(f"dO = 0 gives nonzero gradients n={n}")
        # Shifting every key by one vector leaves each row's P unchanged: all gradients unchanged.
        c = rng.standard_normal(d)
        dq2, dk2, dv2 = impl(q, k + c[None, :], v, do, scale, causal)
        if not (_close(dq, dq2, 1e-9) and _close(dk, dk2, 1e-9) and _close(dv, dv2, 1e-9)):
            bad.append(f"key shift changed the gradients n={n} causal={causal}")
        # Identical keys: P uniform over the visible keys and dQ = 0.
        ke = np.repeat(rng.standard_normal((1, d)), n, axis=0)
        dq3, _, dv3 = impl(q, ke, v, do, scale, causal)
        if not _close(dq3, np.zeros_like(dq3), 1e-10):
            bad.append(f"identical keys give nonzero dQ n={n} causal={causal}")
        if not causal:
            if not _close(dv3, np.repeat(do.sum(0, keepdims=True) / n, n, axis=0), 1e-10):
                bad.append(f"identical keys: dV is not mean dO n={n}")
        if causal:
            # Query 0 sees only key 0 (P = 1): its dQ row is zero; key n-1 is seen
            # only by query n-1: its dV row is P[n-1, n-1] * dO[n-1].
            if not _close(dq[0], np.zeros(d), 1e-12):
                bad.append(f"causal dQ[0] != 0 n={n}")
            p_last = oracle.probabilities(oracle.scores(q, k, scale, True, [n - 1]))[0, n - 1]
            if not _close(dv[n - 1], p_last * do[n - 1], 1e-12):
                bad.append(f"causal dV[last] n={n}")
        # D = sum_j P dP equals rowsum(dO * O): the identity a fast backward uses.
        o, _ = oracle.attention_head(q, k, v, scale, causal)
        p = oracle.probabilities(oracle.scores(q, k, scale, causal))
        ds = p * (do @ v.T - (do * o).sum(1, keepdims=True))
        if not (_close(dq, scale * ds @ k, 1e-10) and _close(dk, scale * ds.T @ q, 1e-10)):
            bad.append(f"gradients disagree with D = rowsum(dO * O) n={n} causal={causal}")
    return bad


PINS = [pin_autograd, pin_finite_differences, pin_invariants]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_backward_oracle_passes_pin(pin):
    assert pin(oracle_impl) == []


def test_backward_batched_and_row_blocks():
    """The [B,H,N,d] driver matches the per-head core; row blocking changes nothing."""
    rng = np.random.default_rng(3)
    q, k, v, do = (rng.standard_normal((2, 2, 37, 8)) for _ in range(4))
    dq, dk, dv = oracle.attention_backward(q, k, v, do, 0.4, True)
    for b in range(2):
        for h in range(2):
            r = oracle.attention_backward_head(q[b, h], k[b, h], v[b, h], do[b, h], 0.4, True)
            for x, y in zip((dq[b, h], dk[b, h], dv[b, h]), r):
                assert np.array_equal(x, y)
    r1 = oracle.attention_backward_head(q[0, 0], k[0, 0], v[0, 0], do[0, 0], 0.4, False, row_block=5)
    r2 = oracle.attention_backward_head(q[0, 0], k[0, 0], v[0, 0], do[0, 0], 0.4, False)
    for x, y in zip(r1, r2):
        assert np.allclose(x, y, atol=1e-13, rtol=0)
    part = oracle.attention_backward(q, k, v, do, 0.4, True, heads=[(1, 0)])
    assert np.isnan(part[0][0, 0]).all() and np.array_equal(part[0][1, 0], dq[1, 0])


# -------------------------------------------------------------------- planted mistakes
def _parts(q, k, v, do, scale, causal):
    p = oracle.probabilities(oracle.scores(q, k, scale, causal))
    dp = do @ v.T
    return p, dp, (p * dp).sum(1, keepdims=True)


def _mut_no_d_term(q, k, v, do, scale, causal):
    p, dp, _ = _parts(q, k, v, do, scale, causal)
    ds = p * dp
    return scale * ds @ k, scale * ds.T @ q, p.T @ do


def _mut_d_sign(q, k, v, do, scale, causal):
    p, dp, dsum = _parts(q, k, v, do, scale, causal)
    ds = p * (dsum - dp)
    return scale * ds @ k, scale * ds.T @ q, p.T @ do


def _mut_dk_unscaled(q, k, v, do, scale, causal):
    dq, dk, dv = oracle.attention_backward_head(q, k, v, do, scale, causal)
    return dq, dk / scale, dv


def _mut_dq_transposed(q, k, v, do, scale, causal):
    p, dp, dsum = _parts(q, k, v, do, scale, causal)
    ds = p * (dp - dsum)
    return scale * ds.T @ k, scale * ds.T @ q, p.T @ do


def _mut_dv_untransposed(q, k, v, do, scale, causal):
    dq, dk, _ = oracle.attention_backward_head(q, k, v, do, scale, causal)
    p, _, _ = _parts(q, k, v, do, scale, causal)
    return dq, dk, p @ do


def _mut_mask_ignored(q, k, v, do, scale, causal):
    return oracle.attention_backward_head(q, k, v, do, scale, False)


def _mut_d_over_columns(q, k, v, do, scale, causal):
    p, dp, _ = _parts(q, k, v, do, scale, causal)
    ds = p * (dp - (p * dp).sum(0, keepdims=True))
    return scale * ds @ k, scale * ds.T @ q, p.T @ do


def _mut_dk_wrong_operand(q, k, v, do, scale, causal):
    p, dp, dsum = _parts(q, k, v, do, scale, causal)
    ds = p * (dp - dsum)
    return scale * ds @ k, scale * ds.T @ k, p.T @ do


def _mut_scale_twice(q, k, v, do, scale, causal):
    dq, dk, dv = oracle.attention_backward_head(q, k, v, do, scale, causal)
    return dq * scale, dk * scale, dv


def _mut_dp_uses_k(q, k, v, do, scale, causal):
    p = oracle.probabilities(oracle.scores(q, k, scale, causal))
    dp = do @ k.T
    ds = p * (dp - (p * dp).sum(1, keepdims=True))
    return scale * ds @ k, scale * ds.T @ q, p.T @ do


MUTANTS = [_mut_no_d_term, _mut_d_sign, _mut_dk_unscaled, _mut_dq_transposed, _mut_dv_untransposed,
           _mut_mask_ignored, _mut_d_over_columns, _mut_dk_wrong_operand, _mut_scale_twice, _mut_dp_uses_k]


@pytest.mark.parametrize("mutant", MUTANTS, ids=lambda m: m.__name__)
def test_planted_backward_mistake_fails_a_pin(mutant):
    failures = []
    with np.errstate(all="ignore"):
        for pin in PINS:
            try:
                failures += pin(mutant)
            except Exception as e:  # a crash also counts as caught
                failures.append(f"{pin.__name__} raised {type(e).__name__}")
    assert failures, f"no pin caught {mutant.__name__}"


def test_backward_with_different_query_and_key_lengths():
    """Nq != Nk (top-left causal alignment, as the forward): against torch fp64 autograd of its SDPA."""
    rng = np.random.default_rng(23)
    for nq, nk in ((3, 8), (8, 3), (1, 6), (7, 1), (33, 70)):
        for causal in (False, True):
            d = 4
            q = rng.standard_normal((nq, d))
            k = rng.standard_normal((nk, d)) * 1.5
            v = rng.standard_normal((nk, d))
            do = rng.standard_normal((nq, d))
            scale = 0.8
            dq, dk, dv = oracle.attention_backward_head(q, k, v, do, scale, causal)
            tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
            o = torch.nn.functional.scaled_dot_product_attention(
                tq[None, None], tk[None, None], tv[None, None], is_causal=causal, scale=scale)[0, 0]
            o.backward(torch.from_numpy(do))
            for mine, ref in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
                assert np.allclose(mine, ref.numpy(), atol=1e-11, rtol=0), (nq, nk, causal)
