"""fa_fwd_noalloc, the entry point for callers that must not allocate device
memory while they run (an operator inside an inference runtime whose enqueue
call may not allocate, a latency-critical serving path that cannot take the
synchronisation of cudaMalloc, a process that reserved all device memory up
front).  Its scratch lives in a static device array shared by every call, so
the GPU test makes two calls in a row and compares each with fa_fwd, the
entry point that allocates its scratch.

This file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

import tiled_attention_fwd_gb300 as fa
from tiled_attention_fwd_gb300.inputs import Workload, as_f64_numpy, make_qkv

FAKE = 1 << 20  # aligned, non-null, never dereferenced by the host-side checks below


def _run(entry, w, q, k, v):
    dev = torch.device("cuda", 0)
    o = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full(q.shape[:-1], float("nan"), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    rc = entry(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), w.B, w.H, w.N, w.d,
               w.scale, w.causal, stream)
    assert rc == 0, fa.fa_strerror(rc)
    torch.cuda.synchronize(dev)
    return as_f64_numpy(o.cpu()), lse.cpu().double().numpy()


@pytest.mark.gpu
def test_noalloc_matches_fa_fwd_on_two_calls_in_a_row():
    """fa_fwd_noalloc launches the same kernel as fa_fwd on the same inputs, so
    each of two calls in a row must give identical bits.  The first two
    workloads are small enough for the single-tile kernel; the third (160
    heads, 480 two-tile work units) takes the two-tile kernel of the headline."""
    dev = torch.device("cuda", 0)
    workloads = [Workload("noalloc_a", 2, 3, 777, 128, "bf16", True, seed=21),
                 Workload("noalloc_b", 1, 4, 300, 64, "bf16", False, seed=22),
                 Workload("noalloc_c", 1, 160, 600, 128, "bf16", True, seed=23)]
    for w in workloads:
        q, k, v = (t.to(dev) for t in make_qkv(w))
        o_ref, l_ref = _run(fa.fa_fwd, w, q, k, v)
        for call in range(2):
            o, lse = _run(fa.fa_fwd_noalloc, w, q, k, v)
            assert np.isfinite(o).all() and np.isfinite(lse).all(), (w.name, call)
            assert np.array_equal(o, o_ref), (w.name, call, float(np.abs(o - o_ref).max()))
            assert np.array_equal(lse, l_ref), (w.name, call, float(np.abs(lse - l_ref).max()))
    # fa_status also reads (and clears) the no-alloc status word: no wait expired.
    assert fa.fa_status(torch.cuda.current_stream(dev).cuda_stream) == 0


def test_noalloc_rejects_bad_arguments_before_touching_a_device():
    assert fa.fa_fwd_noalloc(0, FAKE, FAKE, FAKE, FAKE, 1, 1, 8, 64, 0.125, 0, None) == -1
    assert fa.fa_fwd_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 0, 8, 64, 0.125, 0, None) == -2
    assert fa.fa_fwd_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 8, 48, 0.125, 0, None) == -3
    assert fa.fa_fwd_noalloc(FAKE + 8, FAKE, FAKE, FAKE, FAKE, 1, 1, 8, 64, 0.125, 0, None) == -4
    assert fa.fa_fwd_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 8, 64, -1.0, 0, None) == -8
    assert "scratch" in fa.fa_strerror(-10)
