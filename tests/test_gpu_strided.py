"""GPU parity of the forward pass with Nq != Nk and non-contiguous layouts
(fa_fwd_strided through forward()) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import compare
from tiled_attention_fwd_gb300 import check_status, fa_fwd, forward
from tiled_attention_fwd_gb300.inputs import as_f64_numpy

pytestmark = pytest.mark.gpu


def _rand(shape, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * std).to(torch.bfloat16)


def _run(q, k, v, causal, scale, out=None):
    dev = torch.device("cuda", 0)
    o, lse = forward(q, k, v, causal=causal, scale=scale, out=out)
    check_status(dev)
    return as_f64_numpy(o.cpu()), lse.cpu().double().numpy()


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("B,H,Nq,Nk,d", [
    (1, 2, 100, 300, 128), (2, 1, 300, 100, 128), (1, 2, 256, 1000, 64), (1, 1, 777, 129, 64),
    (1, 2, 129, 513, 32), (1, 1, 200, 70, 256), (2, 2, 1, 257, 128), (1, 3, 513, 1, 128),
])
def test_rectangular_matches_oracle(B, H, Nq, Nk, d, causal):
    dev = torch.device("cuda", 0)
    q = _rand((B, H, Nq, d), Nq + d)
    k = _rand((B, H, Nk, d), Nk + d + 1, 1.5)
    v = _rand((B, H, Nk, d), Nk + d + 2)
    scale = d ** -0.5
    o, lse = _run(q.to(dev), k.to(dev), v.to(dev), causal, scale)
    o_ref, l_ref = oracle.attention(as_f64_numpy(q), as_f64_numpy(k), as_f64_numpy(v), scale, causal)
    r = compare(o, lse, o_ref, l_ref, "bf16")
    assert r["ok"], r


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("B,H,Nq,Nk,d", [
    (1, 160, 100, 300, 128), (1, 160, 777, 129, 64), (1, 160, 129, 513, 32), (1, 160, 513, 1, 128),
])
def test_rectangular_two_tile_units(B, H, Nq, Nk, d, causal):
    """Enough heads that the two-tile kernel runs (small problems take the single-tile one)."""
    test_rectangular_matches_oracle(B, H, Nq, Nk, d, causal)


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_bshd_layout_matches_oracle(d, causal):
    """Q, K, V and O stored as [B, N, H, d] (rows of one head H*d apart), passed as [B, H, N, d] views."""
    dev = torch.device("cuda", 0)
    B, H, Nq, Nk = 2, 3, 333, 210
    qs = _rand((B, Nq, H, d), 7).to(dev)
    ks = _rand((B, Nk, H, d), 8).to(dev)
    vs = _rand((B, Nk, H, d), 9).to(dev)
    q, k, v = (t.permute(0, 2, 1, 3) for t in (qs, ks, vs))
    out_store = torch.full((B, Nq, H, d), float("nan"), device=dev, dtype=torch.bfloat16)
    out = out_store.permute(0, 2, 1, 3)
    scale = 0.9 * d ** -0.5
    o, lse = _run(q, k, v, causal, scale, out=out)
    o_ref, l_ref = oracle.attention(as_f64_numpy(q.cpu()), as_f64_numpy(k.cpu()), as_f64_numpy(v.cpu()), scale, causal)
    r = compare(as_f64_numpy(out.cpu()), lse, o_ref, l_ref, "bf16")
    assert r["ok"], r


def test_strided_entry_equals_fa_fwd_on_contiguous_inputs():
    """The same contiguous problem through fa_fwd and through fa_fwd_strided gives identical bits."""
    dev = torch.device("cuda", 0)
    B, H, N, d = 2, 4, 700, 128
    q, k, v = (_rand((B, H, N, d), s).to(dev) for s in (1, 2, 3))
    o1 = torch.empty_like(q)
    l1 = torch.empty((B, H, N), device=dev, dtype=torch.float32)
    st = torch.cuda.current_stream().cuda_stream
    assert fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o1.data_ptr(), l1.data_ptr(), B, H, N, d, 0.1, 1, st) == 0
    # A view with a different Nk forces the strided entry: use K/V padded to N+8 rows, first N rows equal.
    kp = torch.zeros((B, H, N + 8, d), device=dev, dtype=torch.bfloat16)
    vp = torch.zeros_like(kp)
    kp[:, :, :N] = k
    vp[:, :, :N] = v
    o2, l2 = forward(q, kp[:, :, :N], vp[:, :, :N], causal=True, scale=0.1)
    check_status(dev)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_rectangular_full_size_sampled():
    """B4 H16 Nq 4096, Nk 8192, d128 causal: sampled rows of two heads against the oracle."""
    dev = torch.device("cuda", 0)
    B, H, Nq, Nk, d = 4, 16, 4096, 8192, 128
    q = _rand((B, H, Nq, d), 31)
    k = _rand((B, H, Nk, d), 32)
    v = _rand((B, H, Nk, d), 33)
    o, lse = _run(q.to(dev), k.to(dev), v.to(dev), True, d ** -0.5)
    rows = [0, 1, 127, 128, 255, 256, 2047, 4095]
    heads = [(0, 0), (3, 15)]
    o_ref, l_ref = oracle.attention(as_f64_numpy(q), as_f64_numpy(k), as_f64_numpy(v), d ** -0.5, True,
                                    rows=rows, heads=heads)
    bi = np.array([b for b, _ in heads])
    hi = np.array([h for _, h in heads])
    r = compare(o[bi, hi][:, rows], lse[bi, hi][:, rows], o_ref[bi, hi], l_ref[bi, hi], "bf16")
    assert r["ok"] and np.isfinite(o).all(), r
