"""GPU parity of the backward pass with Nq != Nk and non-contiguous layouts
(fa_bwd_strided through backward()) against the fp64 oracle, with the bound
of tests/bwd_util.py."""
import numpy as np
import pytest
import torch

import bwd_util
from tiled_attention_fwd_gb300 import backward, check_status, fa_bwd, fa_bwd_workspace_bytes, forward
from tiled_attention_fwd_gb300.inputs import as_f64_numpy

pytestmark = pytest.mark.gpu


def _rand(shape, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * std).to(torch.bfloat16)


def _check_heads(q, k, v, do, res, scale, causal, heads):
    qn, kn, vn, don = (as_f64_numpy(t.cpu()) for t in (q, k, v, do))
    worst, ok_all = 0.0, True
    for b, h in heads:
        ref, mag = bwd_util.head_bounds(qn[b, h], kn[b, h], vn[b, h], don[b, h], res["o"][b, h], scale, causal)
        ok, r = bwd_util.compare_head((res["dq"][b, h], res["dk"][b, h], res["dv"][b, h]), ref, mag)
        ok_all, worst = ok_all and ok, max(worst, r)
    return ok_all, worst


def _fwd_bwd(q, k, v, do, causal, scale, o_out=None, grads_out=None):
    o, lse = forward(q, k, v, causal=causal, scale=scale, out=o_out)
    dq, dk, dv = backward(q, k, v, o, lse, do, causal=causal, scale=scale, out=grads_out)
    check_status(q.device)
    return {n: as_f64_numpy(t.cpu()) for n, t in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv))}


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("B,H,Nq,Nk,d", [
    (1, 2, 100, 300, 128),   # causal: key units past the last query see no query (dK = dV = 0)
    (2, 1, 300, 100, 128),   # causal: queries past the last key see every key
    (1, 2, 256, 1000, 64),
    (1, 1, 777, 129, 64),
    (1, 2, 129, 513, 32),
    (2, 2, 1, 257, 128),
    (1, 3, 513, 1, 128),
    (1, 1, 200, 70, 32),
    (1, 2, 100, 300, 256),   # d = 256: causal key units past the last query, both output halves
    (1, 1, 300, 97, 256),
])
def test_rectangular_matches_oracle(B, H, Nq, Nk, d, causal):
    dev = torch.device("cuda", 0)
    q = _rand((B, H, Nq, d), Nq + d).to(dev)
    k = _rand((B, H, Nk, d), Nk + d + 1, 1.5).to(dev)
    v = _rand((B, H, Nk, d), Nk + d + 2).to(dev)
    do = _rand((B, H, Nq, d), Nq + Nk + 3).to(dev)
    scale = d ** -0.5
    res = _fwd_bwd(q, k, v, do, causal, scale)
    ok, worst = _check_heads(q, k, v, do, res, scale, causal, [(b, h) for b in range(B) for h in range(H)])
    assert ok, worst
    if causal and Nk > Nq:
        assert not res["dk"][:, :, Nq:].any() and not res["dv"][:, :, Nq:].any()


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("d", [32, 64, 128, 256])
def test_bshd_layout_matches_oracle(d, causal):
    """All eight tensors stored as [B, N, H, d] and passed as [B, H, N, d] views."""
    dev = torch.device("cuda", 0)
    B, H, Nq, Nk = 2, 3, 333, 210

    def bshd(n, seed, std=1.0):
        return _rand((B, n, H, d), seed, std).to(dev).permute(0, 2, 1, 3)

    q, k, v, do = bshd(Nq, 7), bshd(Nk, 8, 1.5), bshd(Nk, 9), bshd(Nq, 10)
    nan = lambda n: torch.full((B, n, H, d), float("nan"), device=dev, dtype=torch.bfloat16).permute(0, 2, 1, 3)
    o_out = nan(Nq)
    grads = (nan(Nq), nan(Nk), nan(Nk))
    scale = 0.9 * d ** -0.5
    res = _fwd_bwd(q, k, v, do, causal, scale, o_out=o_out, grads_out=grads)
    for name, t in zip(("dq", "dk", "dv"), grads):
        res[name] = as_f64_numpy(t.cpu())
    ok, worst = _check_heads(q, k, v, do, res, scale, causal, [(b, h) for b in range(B) for h in range(H)])
    assert ok, worst


def test_strided_entry_equals_fa_bwd_on_contiguous_inputs():
    """The same contiguous problem through fa_bwd and through fa_bwd_strided gives identical bits."""
    dev = torch.device("cuda", 0)
    B, H, N, d = 2, 4, 700, 128
    q, k, v, do = (_rand((B, H, N, d), s).to(dev) for s in (1, 2, 3, 4))
    o, lse = forward(q, k, v, causal=True, scale=0.1)
    g1 = [torch.empty_like(q) for _ in range(3)]
    ws = torch.empty(fa_bwd_workspace_bytes(B, H, N, d), device=dev, dtype=torch.uint8)
    st = torch.cuda.current_stream().cuda_stream
    assert fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), do.data_ptr(),
                  *[t.data_ptr() for t in g1], B, H, N, d, 0.1, 1, ws.data_ptr(), ws.numel(), st) == 0
    # dK stored inside a wider buffer makes the layout non-contiguous and forces the strided entry.
    dk_store = torch.zeros((B, H, N + 8, d), device=dev, dtype=torch.bfloat16)
    g2 = (torch.empty_like(q), dk_store[:, :, :N], torch.empty_like(v))
    backward(q, k, v, o, lse, do, causal=True, scale=0.1, out=g2)
    check_status(dev)
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)
    assert not dk_store[:, :, N:].any()  # rows outside the view untouched


def test_rectangular_full_size_sampled():
    """B4 H16 Nq 4096, Nk 8192, d128 causal: two heads checked in full."""
    dev = torch.device("cuda", 0)
    B, H, Nq, Nk, d = 4, 16, 4096, 8192, 128
    q = _rand((B, H, Nq, d), 41).to(dev)
    k = _rand((B, H, Nk, d), 42).to(dev)
    v = _rand((B, H, Nk, d), 43).to(dev)
    do = _rand((B, H, Nq, d), 44).to(dev)
    res = _fwd_bwd(q, k, v, do, True, d ** -0.5)
    for n in ("dq", "dk", "dv"):
        assert np.isfinite(res[n]).all()
    heads = [(0, 0), (3, 15)]
    ok, worst = _check_heads(q, k, v, do, res, d ** -0.5, True, heads)
    assert ok, worst
    assert not res["dk"][:, :, Nq:].any() and not res["dv"][:, :, Nq:].any()
