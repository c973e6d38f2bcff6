"""Plain fp64 CPU oracle for the FlashAttention-2 forward pass.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or
links this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` use it.  It shares no code with
the CUDA path.

What it computes is standard scaled-dot-product attention, written out the
obvious way (it materialises the score matrix S and the probability matrix P
of every head), not the tiled online-softmax recurrence.  The recurrence
reaches this result exactly up to rounding, so the plain definition is the
oracle:

* S = (Q K^T) * scale
    -- "Writing a FlashAttention kernel in Metal", section "Standard attention".
* causal: S[q, k] = -inf where key position k > query position q; positions
  are absolute indices in the sequence (top-left alignment), and masked
  entries contribute exactly zero after exponentiation
    -- same page, section "Blockwise attention and causal masking".
* P = row softmax of S (subtract the row max, exponentiate, divide by the row
  sum); every row of P sums to 1
    -- same page, "Standard attention" (torch.softmax over dim=1).
* O = P V
    -- same page, "Standard attention".
* L[q] = logsumexp over k of S[q, k] = max_k S[q,k] + log sum_k exp(S[q,k] - max)
  in natural-log units; the tiled method's m + log(l) equals this
    -- "FlashAttention-2 from PyTorch to Triton", section "What We Are Building".

Rows are independent in this definition, so the function evaluates them in
blocks of ``row_block`` query rows (and can be restricted to a subset of rows);
this changes nothing in any row's arithmetic.  Every function here is pinned by
the ``-m "not gpu"`` tests in ``tests/test_oracle.py`` (library routine,
closed forms, invariants, the pages' worked split of a softmax row, and the
tiled recurrence at several tile sizes).
"""
from __future__ import annotations

import numpy as np


def scores(q: np.ndarray, k: np.ndarray, scale: float, causal: bool, rows=None) -> np.ndarray:
    """Scaled, optionally causally masked logits S for one head.

    q, k: fp64 arrays of shape [N, d].  ``rows`` (optional) selects query rows;
    their absolute positions are used for the causal comparison.
    Returns S of shape [len(rows) or N, N].
    """
    n = k.shape[0]
    qpos = np.arange(q.shape[0]) if rows is None else np.asarray(rows)
    s = (q[qpos] @ k.T) * scale
    if causal:
        kpos = np.arange(n)
        future = kpos[None, :] > qpos[:, None]
        s = np.where(future, -np.inf, s)
    return s


def probabilities(s: np.ndarray) -> np.ndarray:
    """Row softmax of S: exp(S - rowmax) / rowsum."""
    mx = s.max(axis=-1, keepdims=True)
    e = np.exp(s - mx)
    return e / e.sum(axis=-1, keepdims=True)


def logsumexp_rows(s: np.ndarray) -> np.ndarray:
    """L = rowmax + log(sum exp(S - rowmax)), natural log."""
    mx = s.max(axis=-1)
    return mx + np.log(np.exp(s - mx[:, None]).sum(axis=-1))


def attention_head(q, k, v, scale: float, causal: bool, rows=None, row_block: int = 1024):
    """O and L for one head.  q, k, v: fp64 [N, d].  Returns (O [R, d], L [R])."""
    rows = np.arange(q.shape[0]) if rows is None else np.asarray(rows)
    o = np.empty((rows.shape[0], v.shape[1]), dtype=np.float64)
    lse = np.empty(rows.shape[0], dtype=np.float64)
    for a in range(0, rows.shape[0], row_block):
        r = rows[a:a + row_block]
        s = scores(q, k, scale, causal, r)
        p = probabilities(s)
        o[a:a + row_block] = p @ v
        lse[a:a + row_block] = logsumexp_rows(s)
    return o, lse


def attention(q, k, v, scale: float, causal: bool, rows=None, heads=None):
    """Standard attention over [B, H, N, d] fp64 inputs.

    ``rows``: optional query-row subset applied to every head.
    ``heads``: optional list of (b, h) pairs to evaluate (default: all).
    Returns O [B, H, R, d] and L [B, H, R] (fp64); heads that were not
    evaluated are left as NaN.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, N, _ = q.shape
    R = N if rows is None else len(rows)
    o = np.full((B, H, R, v.shape[-1]), np.nan)
    lse = np.full((B, H, R), np.nan)
    todo = [(b, h) for b in range(B) for h in range(H)] if heads is None else heads
    for b, h in todo:
        o[b, h], lse[b, h] = attention_head(q[b, h], k[b, h], v[b, h], scale, causal, rows)
    return o, lse
