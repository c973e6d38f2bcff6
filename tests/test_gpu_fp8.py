"""GPU parity of the e4m3 (fp8) forward pass (fa_fwd_fp8) against the fp64
oracle on the dequantised inputs, graded with the bound derived in
tests/fp8_util.py (per element, worst case; and each head's RMS error against
the predicted spread of P's e4m3 rounding); L at 1e-3.

Small cases cover ragged N, both masks, d = 64 and 128, the single-tile
kernel (few heads) and the two-tile kernel (160 heads), and large logits; the
full-size workloads (the headline shape and the d = 128 sweep point in e4m3)
are compared element by element with the oracle run head by head in a spawn
pool.
"""
import multiprocessing as mp
import os

import numpy as np
import pytest
import torch

import fp8_util
import oracle_workers
import tiled_attention_fwd_gb300 as fa
from tiled_attention_fwd_gb300.inputs import WORKLOADS, Workload, make_qkv_fp8

pytestmark = pytest.mark.gpu


def _run(w, q8, k8, v8, scales):
    dev = torch.device("cuda", 0)
    o = torch.full(q8.shape, float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full(q8.shape[:-1], float("nan"), dtype=torch.float32, device=dev)
    fa.forward_fp8(q8.to(dev), k8.to(dev), v8.to(dev), scales, causal=w.causal, scale=w.scale, out=o, lse=lse)
    fa.check_status(dev)
    return o.cpu().double().numpy(), lse.cpu().double().numpy()


def _grade_heads(results):
    r = fp8_util.merge(results)
    return r


def _check_small(w):
    (q8, k8, v8), scales = make_qkv_fp8(w)
    o, lse = _run(w, q8, k8, v8, scales)
    qn, kn, vn = (t.double().numpy() for t in (q8, k8, v8))
    res = []
    for b in range(w.B):
        for h in range(w.H):
            _, _, o_ref, l_ref, e, sig2 = oracle_workers.fp8_head(
                (b, h, qn[b, h], kn[b, h], vn[b, h], *scales, w.scale, w.causal))
            res.append(fp8_util.compare_head(o[b, h], lse[b, h], o_ref, l_ref, e, sig2))
    return _grade_heads(res)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 127, 128, 129, 257, 600])
@pytest.mark.parametrize("causal", [False, True])
def test_fp8_ragged_single_tile(d, N, causal):
    w = Workload("fp8_edge", 1, 3, N, d, "fp8", causal, seed=13 * N + d)
    r = _check_small(w)
    assert r["ok"], r


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 257, 600])
@pytest.mark.parametrize("causal", [False, True])
def test_fp8_ragged_two_tile(d, N, causal):
    """Enough heads that the two-tile kernel runs (2 * B * H * ceil(N / 256) > SMs)."""
    w = Workload("fp8_edge_2t", 1, 160, N, d, "fp8", causal, seed=17 * N + d)
    r = _check_small(w)
    assert r["ok"], r


@pytest.mark.parametrize("d", [64, 128])
def test_fp8_large_logits(d):
    for causal in (False, True):
        w = Workload("fp8_qk3", 2, 2, 1100, d, "fp8", causal, seed=19 + d, qk_std=3.0)
        r = _check_small(w)
        assert r["ok"], (causal, r)


def test_fp8_many_units_per_cta():
    w = Workload("fp8_units", 3, 64, 700, 128, "fp8", True, seed=23)
    r = _check_small(w)
    assert r["ok"], r


def test_fp8_non_power_of_two_factors():
    """The entry point takes any finite factors > 0; rescaled factors give the same real inputs."""
    w = Workload("fp8_factors", 1, 4, 300, 128, "fp8", True, seed=29)
    (q8, k8, v8), scales = make_qkv_fp8(w)
    f = (scales[0] * 0.7, scales[1] * 1.3, scales[2] * 0.45)
    o, lse = _run(w, q8, k8, v8, f)
    qn, kn, vn = (t.double().numpy() for t in (q8, k8, v8))
    res = []
    for h in range(w.H):
        _, _, o_ref, l_ref, e, sig2 = oracle_workers.fp8_head((0, h, qn[0, h], kn[0, h], vn[0, h], *f, w.scale, True))
        res.append(fp8_util.compare_head(o[0, h], lse[0, h], o_ref, l_ref, e, sig2))
    r = fp8_util.merge(res)
    assert r["ok"], r


def test_fp8_deterministic():
    w = Workload("fp8_det", 2, 4, 777, 128, "fp8", True, seed=31)
    (q8, k8, v8), scales = make_qkv_fp8(w)
    a = _run(w, q8, k8, v8, scales)
    b = _run(w, q8, k8, v8, scales)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_fp8_argument_errors():
    dev = torch.device("cuda", 0)
    x = torch.zeros(1, 1, 8, 32, dtype=torch.float8_e4m3fn, device=dev)
    with pytest.raises(fa.FAError) as e:
        fa.forward_fp8(x, x, x, (1.0, 1.0, 1.0))
    assert e.value.code == -3  # no e4m3 kernel for d = 32
    x = torch.zeros(1, 1, 8, 64, dtype=torch.float8_e4m3fn, device=dev)
    for bad in ((0.0, 1.0, 1.0), (1.0, float("inf"), 1.0), (1.0, 1.0, -2.0)):
        with pytest.raises(fa.FAError) as e:
            fa.forward_fp8(x, x, x, bad)
        assert e.value.code == -8
    flat = torch.zeros(1 * 1 * 8 * 64 + 8, dtype=torch.float8_e4m3fn, device=dev)
    xs = flat[8:].view(1, 1, 8, 64)  # 8-byte offset: not 16-byte aligned
    with pytest.raises(fa.FAError) as e:
        fa.forward_fp8(xs, xs, xs, (1.0, 1.0, 1.0))
    assert e.value.code == -4


@pytest.fixture(scope="module")
def pool():
    keys = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")
    saved = {k: os.environ.get(k) for k in keys}
    for k in keys:
        os.environ[k] = "1"
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


@pytest.mark.parametrize("name", ["fp8_b4h16n4096d128_causal", "fp8_b2h16n8192d128_qk3"])
def test_fp8_full_size_every_element(name, pool):
    w = WORKLOADS[name]
    (q8, k8, v8), scales = make_qkv_fp8(w)
    o, lse = _run(w, q8, k8, v8, scales)
    qn, kn, vn = (t.double().numpy() for t in (q8, k8, v8))
    tasks = ((b, h, qn[b, h], kn[b, h], vn[b, h], *scales, w.scale, w.causal) for b in range(w.B) for h in range(w.H))
    res = []
    for b, h, o_ref, l_ref, e, sig2 in pool.imap_unordered(oracle_workers.fp8_head, tasks):
        res.append(fp8_util.compare_head(o[b, h], lse[b, h], o_ref, l_ref, e, sig2))
    r = fp8_util.merge(res)
    print(name, r)
    assert r["heads"] == w.B * w.H
    assert r["ok"], r
