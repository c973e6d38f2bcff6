"""Shared helpers of the parity tests: run the CUDA path, run the oracle on the
same seeded inputs, compare element by element with the stated tolerances.

Tolerances (max abs error against the fp64 oracle on the rounded inputs):
  fp32 path: 1e-5 on O and on L.
  bf16 path: 1e-2 on O above the output's own rounding, i.e. per element
             |O_gpu - O_ref| <= 1e-2 + |bf16(O_ref) - O_ref|, and 1e-3 on L.
The rounding term is zero wherever the exact O is representable to 1e-2 in
bf16 (|O| < 4); it only matters for the large-logit head-dim sweep, where a
few hundred exact outputs have |O| in [4, 8) and bf16's half-ulp there is 1/64.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from tiled_attention_fwd_gb300 import check_status, forward
from tiled_attention_fwd_gb300.inputs import Workload, as_f64_numpy, make_qkv

TOL_F32 = 1e-5
TOL_BF16_O = 1e-2
TOL_BF16_L = 1e-3


def run_cuda(q, k, v, causal, scale, poison=True):
    """Copy CPU tensors to cuda:0, run the library, return (O, L) as fp64 numpy."""
    dev = torch.device("cuda", 0)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty_like(qd)
    lse = torch.empty(q.shape[:-1], device=dev, dtype=torch.float32)
    if poison:  # rows the kernel fails to write stay NaN
        o.fill_(float("nan"))
        lse.fill_(float("nan"))
    forward(qd, kd, vd, causal=causal, scale=scale, out=o, lse=lse)
    check_status(dev)  # synchronises; raises if any bounded device wait of this launch expired
    return as_f64_numpy(o.cpu()), lse.cpu().double().numpy()


def bf16_round(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x).to(torch.bfloat16).double().numpy()


def compare(o_gpu, l_gpu, o_ref, l_ref, dtype: str):
    """Returns a dict of error figures and a boolean 'ok'."""
    assert o_gpu.shape == o_ref.shape and l_gpu.shape == l_ref.shape
    finite = bool(np.isfinite(o_gpu).all() and np.isfinite(l_gpu).all())
    err_o = np.abs(o_gpu - o_ref)
    err_l = np.abs(l_gpu - l_ref)
    res = {"finite": finite, "max_err_O": float(np.nanmax(err_o)) if err_o.size else 0.0,
           "max_err_L": float(np.nanmax(err_l)) if err_l.size else 0.0}
    if dtype == "f32":
        res["ok"] = finite and res["max_err_O"] <= TOL_F32 and res["max_err_L"] <= TOL_F32
    else:
        floor = np.abs(bf16_round(o_ref) - o_ref)
        res["rounding_floor"] = float(floor.max()) if floor.size else 0.0
        res["max_err_O_above_floor"] = float((err_o - floor).max()) if err_o.size else 0.0
        res["ok"] = finite and bool((err_o <= TOL_BF16_O + floor).all()) and res["max_err_L"] <= TOL_BF16_L
    return res


def check_full(w: Workload, q=None, k=None, v=None):
    """Whole-tensor parity (the oracle computes every row of every head)."""
    if q is None:
        q, k, v = make_qkv(w)
    o, l = run_cuda(q, k, v, w.causal, w.scale)
    o_ref, l_ref = oracle.attention(as_f64_numpy(q), as_f64_numpy(k), as_f64_numpy(v), w.scale, w.causal)
    return compare(o, l, o_ref, l_ref, w.dtype)


def sample_rows(N: int, seed: int, extra: int = 24):
    """Rows every kernel tiling treats specially (first/last, tile edges) plus random ones."""
    edges = {0, 1, N - 1, N - 2}
    for t in (64, 128, 256):
        for b in range(t, N, t * max(1, N // (8 * t))):
            edges.update({b - 1, b})
    rng = np.random.default_rng(seed)
    rand = rng.choice(N, size=min(extra, N), replace=False)
    rows = sorted(x for x in edges.union(int(r) for r in rand) if 0 <= x < N)
    return rows


def check_sampled(w: Workload, rows=None, heads=None):
    """Parity at full size on sampled rows (and optionally a subset of heads).

    The CUDA path runs the whole workload in the same launch configuration as
    the benchmark; the oracle evaluates the sampled rows one by one.
    """
    q, k, v = make_qkv(w)
    o, l = run_cuda(q, k, v, w.causal, w.scale)
    rows = sample_rows(w.N, w.seed) if rows is None else rows
    if heads is None:
        heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    qn, kn, vn = as_f64_numpy(q), as_f64_numpy(k), as_f64_numpy(v)
    o_ref, l_ref = oracle.attention(qn, kn, vn, w.scale, w.causal, rows=rows, heads=heads)
    bi = np.array([b for b, _ in heads])
    hi = np.array([h for _, h in heads])
    res = compare(o[bi, hi][:, rows], l[bi, hi][:, rows], o_ref[bi, hi], l_ref[bi, hi], w.dtype)
    # Properties over every output (not only the sampled rows).
    res["all_finite"] = bool(np.isfinite(o).all() and np.isfinite(l).all())
    res["ok"] = res["ok"] and res["all_finite"]
    return res
