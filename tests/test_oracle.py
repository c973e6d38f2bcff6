"""Pins for the fp64 oracle, independent of the oracle itself.

Each pin checks the oracle against something the pages or mathematics fix:
an independent library implementation (torch's fp64 scaled_dot_product_attention,
scipy's logsumexp), closed forms, invariants, the pages' worked split of a
softmax row, and the tiled online-softmax recurrence the pages derive.  The
last test plants plausible mistakes in copies of the oracle and requires every
one of them to fail at least one pin.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed, std=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * std


def oracle_impl(q, k, v, scale, causal):
    return oracle.attention_head(q, k, v, scale, causal)


# ----------------------------------------------------------------------------- pins
# Every pin takes an implementation impl(q, k, v, scale, causal) -> (O, L) on a
# single head ([N, d] fp64 arrays) and returns a list of failure strings.


def pin_library(impl):
    """Brute force on tiny inputs against torch's fp64 SDPA and scipy's logsumexp.

    Definition pinned: standard attention ("Writing a FlashAttention kernel in
    Metal", "Standard attention"), the causal mask of the same page's
    "Blockwise attention and causal masking", and L = logsumexp of the scaled
    row ("FlashAttention-2 from PyTorch to Triton", "What We Are Building").
    """
    bad = []
    seed = 0
    for n in (1, 2, 3, 5, 8):
        for d in (1, 2, 4):
            for causal in (False, True):
                seed += 1
                q, k, v = _rand((n, d), seed), _rand((n, d), seed + 100), _rand((n, d), seed + 200)
                scale = 1.0 / math.sqrt(d) * 1.3
                o, lse = impl(q, k, v, scale, causal)
                tq, tk, tv = (torch.from_numpy(x)[None, None] for x in (q, k, v))
                o_ref = torch.nn.functional.scaled_dot_product_attention(
                    tq, tk, tv, is_causal=causal, scale=scale)[0, 0].numpy()
                s_lib = (q @ k.T) * scale
                if causal:
                    s_lib = np.where(np.tri(n, n, dtype=bool), s_lib, -np.inf)
                l_ref = scipy.special.logsumexp(s_lib, axis=1)
                if not np.allclose(o, o_ref, rtol=0, atol=1e-12):
                    bad.append(f"O vs SDPA n={n} d={d} causal={causal}")
                if not np.allclose(lse, l_ref, rtol=0, atol=1e-12):
                    bad.append(f"L vs scipy logsumexp n={n} d={d} causal={causal}")
    return bad


def pin_golden_split(impl):
    """The pages' worked split of a score row into blocks [a, b] and [c, d].

    Source: "Writing a FlashAttention kernel in Metal", "Online softmax":
    l1 = e^a + e^b, l2 = l1 + e^c + e^d, p_a = e^a / l2.  A single query with
    q = [1], scale = 1 and keys k_j = [x_j] makes the score row x exactly; with
    v_j = e_j (one-hot) the output row is the probability row.
    """
    bad = []
    with open(os.path.join(GOLDEN, "online_softmax_split.json")) as f:
        g = json.load(f)
    for row in g["rows"]:
        a, b, c, d = row
        l1 = math.exp(a) + math.exp(b)
        l2 = l1 + math.exp(c) + math.exp(d)
        p = [math.exp(x) / l2 for x in row]
        q = np.array([[1.0]])
        k = np.array(row, dtype=np.float64)[:, None]
        v = np.eye(4)
        # Pad the query to four rows (the extra rows are ignored) so that the
        # causal flag can also be exercised on the last row, which sees all keys.
        q4 = np.ones((4, 1))
        for causal in (False, True):
            o, lse = impl(q4, k, v, 1.0, causal)
            if not np.allclose(o[3], p, rtol=0, atol=1e-14):
                bad.append(f"split row {row} causal={causal}: O {o[3]} != {p}")
            if not abs(lse[3] - math.log(l2)) < 1e-13:
                bad.append(f"split row {row} causal={causal}: L {lse[3]} != log l2")
        o, _ = impl(q, k[:2], np.eye(2), 1.0, False)
        # The first block alone: its local softmax, which the page says is wrong for the row.
        if not np.allclose(o[0], [math.exp(a) / l1, math.exp(b) / l1], atol=1e-14):
            bad.append("first block local softmax")
        if abs(math.exp(a) / l1 - p[0]) < 1e-6:
            bad.append("fixture does not separate local from global softmax")
    return bad


def pin_closed_forms(impl):
    """Closed forms of standard attention."""
    bad = []
    rng = np.random.default_rng(7)
    n, d = 37, 6
    q, k = rng.standard_normal((n, d)) * 2, rng.standard_normal((n, d)) * 2
    scale = 0.4
    # All V rows equal c: every output row is c, causal or not.
    c = rng.standard_normal(d)
    v_const = np.tile(c, (n, 1))
    for causal in (False, True):
        o, _ = impl(q, k, v_const, scale, causal)
        if not np.allclose(o, v_const, atol=1e-12):
            bad.append(f"constant V causal={causal}")
    # Q = 0: all scores 0, so O is the mean of the visible V rows and L = log(count).
    v = rng.standard_normal((n, d))
    o, lse = impl(np.zeros((n, d)), k, v, scale, False)
    if not np.allclose(o, np.tile(v.mean(0), (n, 1)), atol=1e-12):
        bad.append("Q=0 non-causal mean")
    if not np.allclose(lse, math.log(n), atol=1e-12):
        bad.append("Q=0 non-causal L=log N")
    o, lse = impl(np.zeros((n, d)), k, v, scale, True)
    prefix = np.cumsum(v, axis=0) / np.arange(1, n + 1)[:, None]
    if not np.allclose(o, prefix, atol=1e-12):
        bad.append("Q=0 causal prefix mean")
    if not np.allclose(lse, np.log(np.arange(1, n + 1)), atol=1e-12):
        bad.append("Q=0 causal L=log(q+1)")
    # Causal row 0 sees only key 0.
    o, lse = impl(q, k, v, scale, True)
    if not np.allclose(o[0], v[0], atol=1e-13):
        bad.append("causal row 0 = V[0]")
    if not abs(lse[0] - scale * float(q[0] @ k[0])) < 1e-12:
        bad.append("causal L[0] = scale q0.k0")
    # Two keys with scores 0 and log 3: weights 1/4 and 3/4 exactly, L = log 4.
    q2 = np.array([[math.log(3.0) / scale, 0.0]])
    k2 = np.array([[0.0, 5.0], [1.0, 0.0]])
    v2 = np.array([[4.0, -8.0], [8.0, 4.0]])
    o, lse = impl(q2, k2, v2, scale, False)
    if not np.allclose(o[0], [0.25 * 4 + 0.75 * 8, 0.25 * -8 + 0.75 * 4], atol=1e-12):
        bad.append("two-key 1/4,3/4")
    if not abs(lse[0] - math.log(4.0)) < 1e-12:
        bad.append("two-key L = log 4")
    return bad


def pin_invariants(impl):
    """Invariants: L = logsumexp, exp(S - L) reproduces P, key permutation,
    independence of future keys under the causal mask, scale covariance."""
    bad = []
    rng = np.random.default_rng(11)
    n, d = 29, 5
    q, k, v = rng.standard_normal((n, d)), rng.standard_normal((n, d)), rng.standard_normal((n, d))
    scale = 0.7
    for causal in (False, True):
        o, lse = impl(q, k, v, scale, causal)
        # exp(S - L) reproduces the probabilities, so (exp(S - L)) V == O and its rows sum to 1
        # ("FlashAttention-2 from PyTorch to Triton": P = exp(S - L)).
        s = (q @ k.T) * scale
        if causal:
            s = np.where(np.tri(n, n, dtype=bool), s, -np.inf)
        p = np.exp(s - lse[:, None])
        if not np.allclose(p.sum(1), 1.0, atol=1e-12):
            bad.append(f"rows of exp(S-L) sum to 1 causal={causal}")
        if not np.allclose(p @ v, o, atol=1e-12):
            bad.append(f"exp(S-L) V == O causal={causal}")
    # Non-causal: a joint permutation of key/value rows changes nothing.
    perm = rng.permutation(n)
    o1, l1 = impl(q, k, v, scale, False)
    o2, l2 = impl(q, k[perm], v[perm], scale, False)
    if not (np.allclose(o1, o2, atol=1e-12) and np.allclose(l1, l2, atol=1e-12)):
        bad.append("key permutation invariance")
    # Causal: changing key/value row j leaves rows q < j unchanged, and changes row j.
    j = 17
    k2, v2 = k.copy(), v.copy()
    k2[j] += 3.0
    v2[j] -= 5.0
    o1, l1 = impl(q, k, v, scale, True)
    o2, l2 = impl(q, k2, v2, scale, True)
    if not (np.allclose(o1[:j], o2[:j], atol=1e-13) and np.allclose(l1[:j], l2[:j], atol=1e-13)):
        bad.append("causal rows before j depend on key j")
    if np.allclose(o1[j], o2[j], atol=1e-6):
        bad.append("causal row j ignores key j")
    # Scale covariance: (Q * t, scale / t) gives the same result.
    o1, l1 = impl(q, k, v, scale, True)
    o2, l2 = impl(q * 4.0, k, v, scale / 4.0, True)
    if not (np.allclose(o1, o2, atol=1e-12) and np.allclose(l1, l2, atol=1e-12)):
        bad.append("scale covariance")
    return bad


def tiled_recurrence(q, k, v, scale, causal, bq, bk):
    """fp64 FA2 recurrence, written from the pages' algorithm; used only here.

    Running row max m (from -inf), rescaled sum l and unnormalised output u;
    alpha = exp(m - m_new) rescales the old state, the division by l happens
    once at the end, L = m + log l ("Writing a FlashAttention kernel in Metal",
    "One-query attention" and "Blockwise attention and causal masking";
    "FlashAttention-2 from PyTorch to Triton", "What We Are Building").
    Fully-future key blocks are skipped.
    """
    n, dv = q.shape[0], v.shape[1]
    out = np.zeros((n, dv))
    lse = np.zeros(n)
    for qs in range(0, n, bq):
        rows = np.arange(qs, min(qs + bq, n))
        m = np.full((len(rows), 1), -np.inf)
        l = np.zeros((len(rows), 1))
        u = np.zeros((len(rows), dv))
        for ks in range(0, n, bk):
            if causal and ks >= qs + len(rows):
                break
            keys = np.arange(ks, min(ks + bk, n))
            s = (q[rows] @ k[keys].T) * scale
            if causal:
                s = np.where(keys[None, :] > rows[:, None], -np.inf, s)
            m_new = np.maximum(m, s.max(1, keepdims=True))
            alpha = np.exp(m - m_new)
            w = np.exp(s - m_new)
            l = alpha * l + w.sum(1, keepdims=True)
            u = alpha * u + w @ v[keys]
            m = m_new
        out[rows] = u / l
        lse[rows] = (m + np.log(l))[:, 0]
    return out, lse


def pin_recurrence(impl):
    """The tiled recurrence equals the plain definition for every tile size."""
    bad = []
    rng = np.random.default_rng(5)
    for n, d in ((1, 3), (7, 4), (45, 8), (300, 16)):
        q, k, v = rng.standard_normal((n, d)) * 2, rng.standard_normal((n, d)) * 2, rng.standard_normal((n, d))
        scale = 1 / math.sqrt(d)
        for causal in (False, True):
            o, lse = impl(q, k, v, scale, causal)
            for bq, bk in ((1, 1), (16, 16), (128, 128), (7, 13)):
                if n > 64 and bq == 1:
                    continue  # tile size 1 is covered by the smaller cases
                o2, l2 = tiled_recurrence(q, k, v, scale, causal, bq, bk)
                if not (np.allclose(o, o2, atol=1e-12) and np.allclose(lse, l2, atol=1e-12)):
                    bad.append(f"recurrence n={n} bq={bq} bk={bk} causal={causal}")
    return bad


PINS = [pin_library, pin_golden_split, pin_closed_forms, pin_invariants, pin_recurrence]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_passes_pin(pin):
    assert pin(oracle_impl) == []


def test_batched_matches_per_head_and_row_subsets():
    """The [B,H,N,d] driver evaluates each head and row subset like the single-head core."""
    rng = np.random.default_rng(3)
    q, k, v = (rng.standard_normal((2, 3, 50, 8)) for _ in range(3))
    o, lse = oracle.attention(q, k, v, 0.3, True)
    for b in range(2):
        for h in range(3):
            o1, l1 = oracle.attention_head(q[b, h], k[b, h], v[b, h], 0.3, True)
            assert np.array_equal(o[b, h], o1) and np.array_equal(lse[b, h], l1)
    rows = [0, 1, 17, 49]
    o2, l2 = oracle.attention(q, k, v, 0.3, True, rows=rows, heads=[(1, 2)])
    assert np.allclose(o2[1, 2], o[1, 2, rows], atol=1e-14, rtol=0)
    assert np.allclose(l2[1, 2], lse[1, 2, rows], atol=1e-14, rtol=0)
    assert np.isnan(o2[0, 0]).all()
    # Row blocking inside a head changes nothing.
    o3, l3 = oracle.attention_head(q[0, 0], k[0, 0], v[0, 0], 0.3, False, row_block=7)
    o4, l4 = oracle.attention_head(q[0, 0], k[0, 0], v[0, 0], 0.3, False)
    assert np.allclose(o3, o4, atol=1e-14) and np.allclose(l3, l4, atol=1e-14)


def test_memory_figures_of_the_pages():
    """Byte accounting pinned to the pages' N=4096 figures (score matrix never stored)."""
    with open(os.path.join(GOLDEN, "memory_figures.json")) as f:
        g = json.load(f)
    n = g["N"]
    tol = g["rel_tolerance"]
    assert abs(n * n - g["S_entries_approx"]) / g["S_entries_approx"] < tol
    assert abs(n * n * 2 - g["S_bytes_bf16_approx"]) / g["S_bytes_bf16_approx"] < tol
    assert n == g["L_entries"]
    assert abs(n * 4 - g["L_bytes_approx"]) / g["L_bytes_approx"] < tol


# -------------------------------------------------------------------- planted mistakes
def _mut_no_scale(q, k, v, scale, causal):
    return oracle.attention_head(q, k, v, 1.0, causal)


def _mut_mask_flipped(q, k, v, scale, causal):
    if not causal:
        return oracle.attention_head(q, k, v, scale, causal)
    o, lse = oracle.attention_head(q[::-1], k[::-1], v[::-1], scale, True)
    return o[::-1], lse[::-1]


def _mut_mask_excludes_diagonal(q, k, v, scale, causal):
    n = q.shape[0]
    s = (q @ k.T) * scale
    if causal:
        s = np.where(np.arange(n)[None, :] >= np.arange(n)[:, None], -np.inf, s)
    with np.errstate(invalid="ignore"):
        return oracle.probabilities(s) @ v, oracle.logsumexp_rows(s)


def _mut_kv_swapped(q, k, v, scale, causal):
    if k.shape != v.shape:
        return oracle.attention_head(q, k, v, scale, causal)
    return oracle.attention_head(q, v, k, scale, causal)


def _mut_transposed_scores(q, k, v, scale, causal):
    n = q.shape[0]
    s = (k @ q.T) * scale
    if causal:
        s = np.where(np.tri(n, n, dtype=bool), s, -np.inf)
    return oracle.probabilities(s) @ v, oracle.logsumexp_rows(s)


def _mut_lse_without_max(q, k, v, scale, causal):
    o, _ = oracle.attention_head(q, k, v, scale, causal)
    s = oracle.scores(q, k, scale, causal)
    return o, np.log(np.exp(s - s.max(1, keepdims=True)).sum(1))


def _mut_lse_log2(q, k, v, scale, causal):
    o, lse = oracle.attention_head(q, k, v, scale, causal)
    return o, lse / math.log(2.0)


def _mut_softmax_wrong_axis(q, k, v, scale, causal):
    s = oracle.scores(q, k, scale, causal)
    e = np.exp(s - s.max(0, keepdims=True))
    p = e / e.sum(0, keepdims=True)
    return p @ v, oracle.logsumexp_rows(s)


def _mut_not_normalised(q, k, v, scale, causal):
    s = oracle.scores(q, k, scale, causal)
    e = np.exp(s - s.max(1, keepdims=True))
    return e @ v, oracle.logsumexp_rows(s)


def _mut_scale_sqrt_missing(q, k, v, scale, causal):
    return oracle.attention_head(q, k, v, scale * scale, causal)


MUTANTS = [_mut_no_scale, _mut_mask_flipped, _mut_mask_excludes_diagonal, _mut_kv_swapped,
           _mut_transposed_scores, _mut_lse_without_max, _mut_lse_log2, _mut_softmax_wrong_axis,
           _mut_not_normalised, _mut_scale_sqrt_missing]


@pytest.mark.parametrize("mutant", MUTANTS, ids=lambda m: m.__name__)
def test_planted_mistake_fails_a_pin(mutant):
    failures = []
    with np.errstate(all="ignore"):
        for pin in PINS:
            try:
                failures += pin(mutant)
            except Exception as e:  # a crash also counts as caught
                failures.append(f"{pin.__name__} raised {type(e).__name__}")
    assert failures, f"no pin caught {mutant.__name__}"


def test_oracle_with_different_query_and_key_lengths():
    """Nq != Nk: the pages' kernel takes N_QUERIES and N_KEYS separately and keeps key k for
    query i iff k < N_KEYS and, when causal, k <= i ("FlashAttention-2 from PyTorch to Triton",
    the Triton kernel).  torch's SDPA uses the same top-left alignment for non-square causal masks."""
    rng = np.random.default_rng(17)
    for nq, nk in ((3, 7), (7, 3), (1, 5), (9, 1), (40, 65)):
        for d in (2, 8):
            for causal in (False, True):
                q = rng.standard_normal((nq, d)) * 2
                k = rng.standard_normal((nk, d)) * 2
                v = rng.standard_normal((nk, d))
                scale = 0.7 / math.sqrt(d)
                o, lse = oracle.attention_head(q, k, v, scale, causal)
                tq, tk, tv = (torch.from_numpy(x)[None, None] for x in (q, k, v))
                o_ref = torch.nn.functional.scaled_dot_product_attention(
                    tq, tk, tv, is_causal=causal, scale=scale)[0, 0].numpy()
                s = (q @ k.T) * scale
                if causal:
                    s = np.where(np.arange(nk)[None, :] <= np.arange(nq)[:, None], s, -np.inf)
                assert np.allclose(o, o_ref, atol=1e-12, rtol=0), (nq, nk, d, causal)
                assert np.allclose(lse, scipy.special.logsumexp(s, axis=1), atol=1e-12, rtol=0), (nq, nk, d, causal)
