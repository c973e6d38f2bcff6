"""The kernels write nothing outside their output tensors.

Each output is a view into a larger buffer whose tail (after the tensor's last
element) holds a sentinel pattern; after the call the tail must be unchanged.
Ragged N puts the last query tile partly past the end of the last head, which
is where a store that is not clipped to the tensor would land."""
import pytest
import torch

from tiled_attention_fwd_gb300 import backward, check_status, forward

pytestmark = pytest.mark.gpu

GUARD = 4096  # elements after each tensor


def _rand(shape, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * std).to(torch.bfloat16)


def _guarded(shape, dtype, dev):
    """A contiguous tensor of `shape` at the start of a buffer with GUARD sentinel elements after it."""
    n = 1
    for s in shape:
        n *= s
    buf = torch.empty(n + GUARD, device=dev, dtype=dtype)
    buf.view(torch.int16 if dtype == torch.bfloat16 else torch.int32)[n:] = 0x7A5A
    return buf[:n].view(shape), buf[n:]


def _intact(tail):
    return bool((tail.view(torch.int16 if tail.dtype == torch.bfloat16 else torch.int32) == 0x7A5A).all())


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("d", [32, 64, 128, 256])
@pytest.mark.parametrize("N", [1, 129, 200, 383])
def test_forward_writes_only_its_outputs(N, d, causal):
    dev = torch.device("cuda", 0)
    B, H = 1, 3
    q, k, v = (_rand((B, H, N, d), s).to(dev) for s in (N, N + 1, N + 2))
    o, o_tail = _guarded((B, H, N, d), torch.bfloat16, dev)
    lse, l_tail = _guarded((B, H, N), torch.float32, dev)
    forward(q, k, v, causal=causal, out=o, lse=lse)
    check_status(dev)
    assert _intact(o_tail) and _intact(l_tail)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


@pytest.mark.parametrize("d", [64, 128, 256])
def test_strided_forward_writes_only_its_outputs(d):
    """O as a [B, N, H, d] view: the last row of the last head is the buffer's last row."""
    dev = torch.device("cuda", 0)
    B, H, Nq, Nk = 2, 3, 201, 130
    q = _rand((B, H, Nq, d), 1).to(dev)
    k = _rand((B, H, Nk, d), 2).to(dev)
    v = _rand((B, H, Nk, d), 3).to(dev)
    store, tail = _guarded((B, Nq, H, d), torch.bfloat16, dev)
    lse, l_tail = _guarded((B, H, Nq), torch.float32, dev)
    forward(q, k, v, causal=True, out=store.permute(0, 2, 1, 3), lse=lse)
    check_status(dev)
    assert _intact(tail) and _intact(l_tail)


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("d", [32, 64, 128, 256])
def test_backward_writes_only_its_outputs(d, causal):
    dev = torch.device("cuda", 0)
    B, H, N = 1, 2, 201
    q, k, v, do = (_rand((B, H, N, d), s).to(dev) for s in (5, 6, 7, 8))
    o, lse = forward(q, k, v, causal=causal)
    grads = [_guarded((B, H, N, d), torch.bfloat16, dev) for _ in range(3)]
    backward(q, k, v, o, lse, do, causal=causal, out=tuple(g for g, _ in grads))
    check_status(dev)
    for g, tail in grads:
        assert _intact(tail)
        assert torch.isfinite(g.float()).all()
