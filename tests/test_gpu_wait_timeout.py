"""A device-side wait that runs out is reported, bounded, and leaves the device usable.

fa_selftest_wait launches one block whose waits (the attention kernels' own
bounded-wait code) are on barriers that nothing signals, so every wait runs
out after the current limit: no fault, trap or hang is involved.  The status
word must report FA_ERR_TIMEOUT once, the call must return after about the
limit, and a forward pass afterwards must still match the oracle.
"""
import time

import pytest
import torch

import tiled_attention_fwd_gb300 as fa
from tiled_attention_fwd_gb300._lib import FA_ERR_TIMEOUT, FA_OK
from tiled_attention_fwd_gb300.inputs import Workload

from parity_util import check_full

pytestmark = pytest.mark.gpu

LIMIT_MS = 20


def test_expired_wait_is_reported_and_device_stays_usable():
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    assert fa.fa_status(stream) == FA_OK
    old = fa.fa_set_wait_limit_ms(LIMIT_MS)
    try:
        t0 = time.perf_counter()
        assert fa.fa_selftest_wait(stream) == FA_OK
        rc = fa.fa_status(stream)
        elapsed = time.perf_counter() - t0
    finally:
        fa.fa_set_wait_limit_ms(old)
    assert rc == FA_ERR_TIMEOUT
    assert LIMIT_MS * 1e-3 <= elapsed < 2.0, elapsed
    # fa_status cleared the word; nothing else has expired since.
    assert fa.fa_status(stream) == FA_OK
    res = check_full(Workload("after_timeout", 1, 2, 300, 64, "bf16", True, seed=5))
    assert res["ok"], res
