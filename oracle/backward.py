"""Plain fp64 CPU oracle for the attention backward pass.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or
links this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU legs of ``bench.py`` use it.  It shares no code with the CUDA path.

The function differentiated is the forward pass of ``oracle.attention``
(standard attention: S = Q K^T * scale, optional causal mask, P = row softmax
of S, O = P V -- "Writing a FlashAttention kernel in Metal", sections
"Standard attention" and "Blockwise attention and causal masking").  Given the
upstream gradient dO of a scalar loss with respect to O, the gradients follow
from the chain rule, written out plainly (S and P are materialised, one block
of query rows at a time):

* dV = P^T dO
* dP = dO V^T
* dS = P * (dP - D), D[i] = sum_j P[i, j] dP[i, j]  (the row-softmax Jacobian
  dP[i,j]/dS[i,l] = P[i,j] (delta_jl - P[i,l]) applied to dP; masked entries
  have P = 0 and receive dS = 0)
* dQ = scale * dS K,  dK = scale * dS^T Q.

The pages fix how a fast backward gets P without storing it: recompute
P = exp(S - L) from the forward's logsumexp L ("FlashAttention-2 from PyTorch
to Triton", "What We Are Building"), and split the work into a dQ kernel and a
dK/dV kernel that each own their outputs ("Case Study: metal-flash-attention").
Neither changes the result, so the oracle is the definition above.

Every function here is pinned by ``tests/test_oracle_backward.py`` (torch
fp64 autograd, central finite differences of the forward oracle, invariants
that hold exactly, and planted mistakes that must fail a pin).
"""
from __future__ import annotations

import numpy as np

from .attention import probabilities, scores


def attention_backward_head(q, k, v, do, scale: float, causal: bool, row_block: int = 1024):
    """dQ, dK, dV for one head.  q, k, v, do: fp64 [N, d].  Returns (dQ, dK, dV), each [N, d]."""
    n = q.shape[0]
    dq = np.zeros_like(q, dtype=np.float64)
    dk = np.zeros_like(k, dtype=np.float64)
    dv = np.zeros_like(v, dtype=np.float64)
    for a in range(0, n, row_block):
        r = np.arange(a, min(n, a + row_block))
        p = probabilities(scores(q, k, scale, causal, r))  # [R, N]
        dv += p.T @ do[r]
        dp = do[r] @ v.T
        dsum = (p * dp).sum(axis=1, keepdims=True)
        ds = p * (dp - dsum)
        dq[r] = scale * (ds @ k)
        dk += scale * (ds.T @ q[r])
    return dq, dk, dv


def attention_backward(q, k, v, do, scale: float, causal: bool, heads=None):
    """dQ, dK, dV over [B, H, N, d] fp64 inputs.

    ``heads``: optional list of (b, h) pairs to evaluate (default: all); heads
    that were not evaluated are left as NaN.
    """
    q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, do))
    B, H = q.shape[:2]
    dq = np.full(q.shape, np.nan)
    dk = np.full(k.shape, np.nan)
    dv = np.full(v.shape, np.nan)
    todo = [(b, h) for b in range(B) for h in range(H)] if heads is None else heads
    for b, h in todo:
        dq[b, h], dk[b, h], dv[b, h] = attention_backward_head(q[b, h], k[b, h], v[b, h], do[b, h], scale, causal)
    return dq, dk, dv
