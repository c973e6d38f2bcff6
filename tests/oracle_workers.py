"""Per-head oracle work for the whole-tensor parity tests, run in worker
processes of a spawn pool (one head per task).  Imports only numpy and the
oracle, so that the workers start quickly and never touch a GPU."""
from __future__ import annotations

import numpy as np

import fp8_util
import oracle


def forward_head(args):
    """(b, h, O, L) of one head by the fp64 oracle."""
    b, h, q, k, v, scale, causal = args
    o, lse = oracle.attention_head(q, k, v, scale, causal)
    return b, h, o, lse


def head_bounds(q, k, v, do, o_gpu, scale, causal):
    """Reference gradients of one head (fp64 oracle) and the per-element
    magnitudes M of the backward bound (the gradient's own products over
    absolute values; see tests/bwd_util.py)."""
    dq, dk, dv = oracle.attention_backward_head(q, k, v, do, scale, causal)
    p = oracle.probabilities(oracle.scores(q, k, scale, causal))
    o = p @ v
    ds = p * (do @ v.T - (do * o).sum(1, keepdims=True))
    e = np.abs(do * o_gpu).sum(1, keepdims=True)
    pe = p * e
    m_v = np.abs(p).T @ np.abs(do)
    m_k = scale * (np.abs(ds).T @ np.abs(q) + pe.T @ np.abs(q))
    m_q = scale * (np.abs(ds) @ np.abs(k) + pe @ np.abs(k))
    return (dq, dk, dv), (m_q, m_k, m_v)


def backward_head(args):
    """(b, h, reference gradients, magnitudes) of one head."""
    b, h, q, k, v, do, o_gpu, scale, causal = args
    ref, mag = head_bounds(q, k, v, do, o_gpu, scale, causal)
    return b, h, ref, mag


def fp8_head(args):
    """(b, h, O, L, E, sigma^2) of one head of an e4m3 problem: the oracle on the
    dequantised inputs and the per-element bounds of tests/fp8_util.py."""
    b, h, q8, k8, v8, qd, kd, vd, scale, causal = args
    o, lse = oracle.attention_fp8_head(q8, k8, v8, qd, kd, vd, scale, causal)
    e, sig2 = fp8_util.head_bounds(q8 * qd, k8 * kd, v8 * vd, scale, causal)
    return b, h, o, lse, e, sig2
