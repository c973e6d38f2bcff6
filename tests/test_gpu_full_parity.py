"""Whole-tensor parity at full size: every output element of the full-size
workloads (the headline, the 16K-token causal case, the four head-dimension
sweep points) and every gradient element of the backward pass on the
headline shape, against the fp64 oracle.

The CUDA path runs once per workload in the launch configuration of the
benchmark (outputs poisoned with NaN first); the oracle evaluates every head
in a spawn pool of worker processes (one head per task, BLAS single-threaded
in each), and the comparison runs head by head as results arrive.  The figures
printed per workload are the literal max abs error of O and L, the rounding
floor max |bf16(O_ref) - O_ref| and the largest error above that floor.
"""
import multiprocessing as mp
import os

import numpy as np
import pytest
import torch

import bwd_util
import oracle_workers
from parity_util import compare, run_cuda
from tiled_attention_fwd_gb300.inputs import WORKLOADS, as_f64_numpy, make_dout, make_qkv

pytestmark = pytest.mark.gpu

FULL = ["bf16_b4h16n4096d128_causal", "bf16_b1h32n16384d128_causal", "bf16_b2h16n8192d32_qk3",
        "bf16_b2h16n8192d64_qk3", "bf16_b2h16n8192d128_qk3", "bf16_b2h16n8192d256_qk3"]


@pytest.fixture(scope="module")
def pool():
    keys = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")
    saved = {k: os.environ.get(k) for k in keys}
    for k in keys:
        os.environ[k] = "1"  # inherited by the spawned workers
    try:
        p = mp.get_context("spawn").Pool(os.cpu_count() or 1)
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    yield p
    p.close()
    p.join()


@pytest.mark.parametrize("name", FULL)
def test_forward_every_element(name, pool):
    w = WORKLOADS[name]
    q, k, v = make_qkv(w)
    o, lse = run_cuda(q, k, v, w.causal, w.scale)
    qn, kn, vn = as_f64_numpy(q), as_f64_numpy(k), as_f64_numpy(v)
    tasks = ((b, h, qn[b, h], kn[b, h], vn[b, h], w.scale, w.causal) for b in range(w.B) for h in range(w.H))
    agg = {"max_err_O": 0.0, "max_err_L": 0.0, "rounding_floor": 0.0, "max_err_O_above_floor": -np.inf}
    ok, heads = True, 0
    for b, h, o_ref, l_ref in pool.imap_unordered(oracle_workers.forward_head, tasks):
        r = compare(o[b, h], lse[b, h], o_ref, l_ref, "bf16")
        ok = ok and r["ok"]
        heads += 1
        for key in agg:
            agg[key] = max(agg[key], r[key])
    assert heads == w.B * w.H
    print(name, {"heads": heads, "elements_O": o.size, "elements_L": lse.size, **agg})
    assert ok, (name, agg)


def test_backward_headline_every_element(pool):
    """B4 H16 N4096 d128 causal: dQ, dK, dV of all 64 heads within the derived bound."""
    w = WORKLOADS["bf16_b4h16n4096d128_causal"]
    q, k, v = make_qkv(w)
    do = make_dout(w)
    res = bwd_util.run_cuda_fwd_bwd(q, k, v, do, w.causal, w.scale)
    qn, kn, vn, don = (as_f64_numpy(t) for t in (q, k, v, do))
    tasks = ((b, h, qn[b, h], kn[b, h], vn[b, h], don[b, h], res["o"][b, h], w.scale, w.causal)
             for b in range(w.B) for h in range(w.H))
    ok, worst, heads = True, 0.0, 0
    for b, h, ref, mag in pool.imap_unordered(oracle_workers.backward_head, tasks):
        got = (res["dq"][b, h], res["dk"][b, h], res["dv"][b, h])
        hok, r = bwd_util.compare_head(got, ref, mag)
        ok = ok and hok
        worst = max(worst, r)
        heads += 1
    assert heads == w.B * w.H
    print("backward headline", {"heads": heads, "worst_error_over_bound": worst})
    assert ok, worst
