"""Parity of the fp8 (e4m3) forward pass: the bound derived from its arithmetic.

The kernel computes S from the e4m3 Q and K exactly (products of e4m3 values
are exact in fp32), runs the online softmax in fp32 like the bf16 path, and
rounds P to e4m3 (the dtype of V, as the Triton kernel of "FlashAttention-2
from PyTorch to Triton" casts P to V's dtype) before O += P V; l is summed
from the fp32 P; O = (P V) * v_descale / l is stored in bf16.  P is rounded
relative to the running max at its key tile, p~ = exp(s - m_run) in [0, 1];
e4m3 keeps 3 mantissa bits (half-ulp 2^-4 relative above 2^-6) and spaces its
subnormals 2^-9 apart (values below 2^-10 round to 0).  In units of the final
row max (p = exp(s - m), l = sum p) the rounding error of each weight is
therefore at most

    dp = max(2^-4 p, min(p, 2^-10)),

so, per output element (row i, column c),

    |O - O_ref| <= 1.1 * E + 2^-8 |O_ref| + 1e-5,   E = sum_j dp_ij |v_jc| / l_i,

where 1.1 covers fp32 accumulation and the exponential's rounding, and 2^-8
|O_ref| the bf16 rounding of the output.  This worst case adds every weight's
error with the same sign; round-to-nearest errors are unbiased and
independent, so a second, statistical check holds the root-mean-square error
over all elements of a head to the predicted standard deviation:

    rms(O - O_ref) <= 1.5 * sqrt(mean(sigma^2)),
    sigma^2 = sum_j dp_ij^2 v_jc^2 / (3 l_i^2) + (2^-9 O_ref)^2 / 3

(a uniform error on [-dp, dp] has variance dp^2 / 3).  A systematic mistake
(a missing factor, a shifted mask, a skipped rescale) moves every element
the same way and fails it by orders of magnitude.  L is graded at 1e-3 as in
the bf16 path: the logits, the max and l are not rounded to e4m3.
"""
from __future__ import annotations

import numpy as np

import oracle

ELEM_FACTOR = 1.1
RMS_FACTOR = 1.5
TOL_L = 1e-3


def weight_error(s: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """(dp, l) of logits s [R, N] (masked entries -inf): the bound on the
    rounding error of each e4m3 weight in final-max units, and the row sums."""
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    dp = np.maximum(2.0 ** -4 * p, np.minimum(p, 2.0 ** -10))
    return dp, p.sum(axis=1)


def head_bounds(q, k, v, scale: float, causal: bool, row_block: int = 1024):
    """E (worst case) and sigma^2 (predicted variance of the P rounding) per
    output element of one head; q, k, v are the dequantised fp64 inputs.
    Rows are independent; they are taken in blocks to bound the memory."""
    n = q.shape[0]
    e = np.empty((n, v.shape[1]))
    sig2 = np.empty((n, v.shape[1]))
    av, v2 = np.abs(v), v * v
    for a in range(0, n, row_block):
        rows = np.arange(a, min(n, a + row_block))
        dp, l = weight_error(oracle.scores(q, k, scale, causal, rows))
        e[rows] = (dp @ av) / l[:, None]
        sig2[rows] = ((dp * dp) @ v2) / (3.0 * (l * l)[:, None])
    return e, sig2


def compare_head(o, lse, o_ref, l_ref, e, sig2):
    """Grade one head; returns a dict with 'ok' and the figures."""
    err = np.abs(o - o_ref)
    finite = bool(np.isfinite(o).all() and np.isfinite(lse).all())
    elem_bound = ELEM_FACTOR * e + 2.0 ** -8 * np.abs(o_ref) + 1e-5
    var = sig2 + (2.0 ** -9 * o_ref) ** 2 / 3.0
    rms = float(np.sqrt(np.mean(err * err))) if err.size else 0.0
    rms_pred = float(np.sqrt(np.mean(var))) if err.size else 0.0
    err_l = float(np.abs(lse - l_ref).max()) if lse.size else 0.0
    worst = float((err / elem_bound).max()) if err.size else 0.0
    ok = finite and worst <= 1.0 and rms <= RMS_FACTOR * rms_pred + 1e-7 and err_l <= TOL_L
    return {"ok": ok, "finite": finite, "max_err_O": float(err.max()) if err.size else 0.0,
            "worst_err_over_elem_bound": worst, "rms_err_O": rms, "rms_predicted": rms_pred,
            "rms_ratio": rms / rms_pred if rms_pred > 0 else 0.0, "max_err_L": err_l}


def merge(results):
    """Aggregate per-head results (worst of each figure)."""
    out = {"ok": all(r["ok"] for r in results), "heads": len(results)}
    for key in ("max_err_O", "worst_err_over_elem_bound", "rms_ratio", "max_err_L"):
        out[key] = max(r[key] for r in results) if results else 0.0
    return out
