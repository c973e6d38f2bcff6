"""Backward-pass parity: run the CUDA forward + backward, run the fp64 oracle on
the same rounded inputs, compare element by element against a bound derived
from the arithmetic.

Per output element the bound is

    |g_gpu - g_ref| <= 2^-7 * M + |bf16(g_ref) - g_ref| + 1e-6,

where M is the same product the gradient is, taken over absolute values:

    dV: M = |P|^T |dO|
    dK: M = scale * (|dS|^T |Q| + (P * E)^T |Q|)
    dQ: M = scale * (|dS| |K| + (P * E) |K|),     E_i = sum_c |dO_ic O_ic|.

Each gradient is a sum of products one of whose operands the kernel rounds
to bf16 (P for dV, dS for dK and dQ; relative error <= 2^-9), with fp32
accumulation; D = rowsum(dO * O) is taken from the bf16 O of the forward pass
(error <= 2^-9 E_i per row, entering dS as P * delta D: the second term); the
output is rounded to bf16 once (the second summand).  2^-7 leaves a factor 4
over 2^-9 for fp32 accumulation and the exponential's rounding.  A real error
(a wrong mask, a missing term, a transposed operand) is of the order of M
itself.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle_workers import head_bounds
from tiled_attention_fwd_gb300 import backward, check_status, forward
from tiled_attention_fwd_gb300.inputs import Workload, as_f64_numpy, make_dout, make_qkv

REL = 2.0 ** -7


def bf16_round(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x).to(torch.bfloat16).double().numpy()


def run_cuda_fwd_bwd(q, k, v, do, causal, scale):
    """Forward then backward on cuda:0; returns dict of fp64 numpy arrays (O too)."""
    dev = torch.device("cuda", 0)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = forward(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = backward(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    check_status(dev)
    return {name: as_f64_numpy(t.cpu()) for name, t in (("dq", dq), ("dk", dk), ("dv", dv), ("o", o))}


def compare_head(got, ref, mag):
    """Returns (ok, worst ratio of error to bound) over dQ, dK, dV of one head."""
    worst = 0.0
    ok = True
    for g, r, m in zip(got, ref, mag):
        bound = REL * m + np.abs(bf16_round(r) - r) + 1e-6
        err = np.abs(g - r)
        if not np.isfinite(g).all():
            return False, float("inf")
        ratio = float((err / bound).max()) if err.size else 0.0
        worst = max(worst, ratio)
        ok = ok and bool((err <= bound).all())
    return ok, worst


def check_backward(w: Workload, heads=None):
    """Parity of dQ, dK, dV for workload w (all heads, or the listed (b, h) pairs)."""
    q, k, v = make_qkv(w)
    do = make_dout(w)
    res = run_cuda_fwd_bwd(q, k, v, do, w.causal, w.scale)
    qn, kn, vn, don = (as_f64_numpy(t) for t in (q, k, v, do))
    todo = [(b, h) for b in range(w.B) for h in range(w.H)] if heads is None else heads
    ok_all, worst = True, 0.0
    for b, h in todo:
        ref, mag = head_bounds(qn[b, h], kn[b, h], vn[b, h], don[b, h], res["o"][b, h], w.scale, w.causal)
        got = (res["dq"][b, h], res["dk"][b, h], res["dv"][b, h])
        ok, r = compare_head(got, ref, mag)
        ok_all = ok_all and ok
        worst = max(worst, r)
    return {"ok": ok_all, "worst_error_over_bound": worst,
            "all_finite": bool(all(np.isfinite(res[x]).all() for x in ("dq", "dk", "dv")))}
