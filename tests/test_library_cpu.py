"""The C-ABI library without a GPU: it builds for sm_103a, loads, exports every
symbol the public header declares, and rejects bad arguments on the host
before touching a device."""
import ctypes
import os
import re
import shutil

import pytest

import tiled_attention_fwd_gb300 as fa
from tiled_attention_fwd_gb300 import _lib, build


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(build.LIB) and shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("neither a built library nor nvcc is available")
    build.build()
    return _lib.load()


def test_every_declared_symbol_is_exported(lib):
    names = _lib.declared_functions()
    assert len(names) >= 8
    raw = ctypes.CDLL(build.LIB)
    for n in names:
        assert hasattr(raw, n), f"{n} declared in include/fa_gb300.h but not exported"
        assert n in _lib._SIGNATURES, f"{n} has no Python binding"


def test_binding_names_match_header(lib):
    assert sorted(_lib._SIGNATURES) == _lib.declared_functions()


def test_strerror_and_version(lib):
    assert fa.fa_abi_version() == 1
    assert fa.fa_strerror(0).startswith("FA_OK")
    assert "TIMEOUT" in fa.fa_strerror(-6)
    assert "unknown" in fa.fa_strerror(12345)


FAKE = 1 << 20  # a 16-byte aligned non-null value; never dereferenced by these calls


@pytest.mark.parametrize("args,code", [
    ((0, FAKE, FAKE, FAKE, FAKE, 1, 1, 8, 64, 0.125, 0), -1),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 0, 1, 8, 64, 0.125, 0), -2),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 0, 64, 0.125, 0), -2),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 8, 48, 0.125, 0), -3),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 8, 16, 0.125, 0), -3),
    ((FAKE + 2, FAKE, FAKE, FAKE, FAKE, 1, 1, 8, 64, 0.125, 0), -4),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 8, 64, 0.0, 0), -8),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 8, 64, float("nan"), 1), -8),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 16, 1 << 16, 8, 64, 0.125, 0), -2),
])
def test_fa_fwd_rejects_bad_arguments_on_host(lib, args, code):
    assert fa.fa_fwd(*args, None) == code


def test_fa_fwd_f32_rejects_bad_arguments_on_host(lib):
    assert fa.fa_fwd_f32(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 8, 257, 0.1, 0, None) == -3
    assert fa.fa_fwd_f32(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 8, 0, 0.1, 0, None) == -3
    assert fa.fa_fwd_f32(FAKE, FAKE, FAKE, FAKE, 0, 1, 1, 8, 16, 0.1, 0, None) == -1
    assert fa.fa_fwd_f32(FAKE + 2, FAKE, FAKE, FAKE, FAKE, 1, 1, 8, 16, 0.1, 0, None) == -4
    assert fa.fa_fwd_f32(FAKE, FAKE, FAKE, FAKE, FAKE, 300, 300, 8, 16, 0.1, 0, None) == -2


def test_host_workspace_size_and_checks(lib):
    n = fa.fa_fwd_host_workspace_bytes(2, 3, 100, 64)
    t = 2 * 3 * 100 * 64 * 2
    r256 = lambda x: (x + 255) // 256 * 256
    assert n == 4 * r256(t) + r256(2 * 3 * 100 * 4)
    assert fa.fa_fwd_host_workspace_bytes(0, 3, 100, 64) == 0
    # too-small workspace is rejected before any copy is enqueued
    assert fa.fa_fwd_host(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE * 16, n - 1, 2, 3, 100, 64, 0.125, 0, None) == -9
    assert fa.fa_fwd_host(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 16, n, 2, 3, 100, 64, 0.125, 0, None) == -4


def test_wait_limit_setting(lib):
    prev = fa.fa_set_wait_limit_ms(1500)
    assert prev >= 1
    assert fa.fa_set_wait_limit_ms(0) == 1500
    assert fa.fa_set_wait_limit_ms(prev) == 1


def test_forward_refuses_cpu_tensors():
    torch = pytest.importorskip("torch")
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.forward(q, q, q)


def test_missing_library_fails_loudly(tmp_path):
    saved = _lib._lib
    _lib._lib = None
    try:
        with pytest.raises(ImportError):
            _lib.load(str(tmp_path / "nope.so"))
    finally:
        _lib._lib = saved


def test_tensor_core_kernels_fit_their_register_split():
    """The two-tile d <= 128 kernels (bf16 and e4m3) launch 512 threads at 128 registers and re-split them
    (184 x 256 softmax + 144 x 128 correction and MMA/TMA, 80/64 = 65536); the
    single-tile d <= 128 kernels launch 384 threads at 168 (208 softmax, 152 correction,
    144 MMA/TMA); any other launch count would stall setmaxnreg, and none of them may spill."""
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    files = {f"fa_tc_d{d}{s}.cu" for d in (32, 64, 128, 256) for s in ("", "_strided")}
    files |= {f"fa_tc_fp8_d{d}.cu" for d in (64, 128)}
    rep = build.ptxas_report(files)
    tc = {k: v for k, v in rep.items() if "fa_fwd_tc_kernel" in k}
    # bf16: 4 head dims x causal / not x contiguous / strided, plus the
    # single-tile kernels of d = 32, 64, 128 (causal / not, contiguous /
    # strided); e4m3: d = 64, 128 x causal / not x two-tile / single-tile.
    assert len(tc) == 36
    # Template parameters <D, CAUSAL, STRIDED, NQ, VAR> in the mangled name.
    pat = re.compile(r"fa_fwd_tc_kernelILi(\d+)ELb([01])ELb([01])ELi([12])ELi([012])E")
    seen = set()
    for name, r in tc.items():
        m = pat.search(name)
        assert m, f"unrecognised kernel name {name}"
        d, causal, strided, nq = int(m.group(1)), m.group(2), m.group(3), int(m.group(4))
        seen.add((d, causal, strided, nq, m.group(5)))
        assert r["spill_stores"] == 0 and r["spill_loads"] == 0, (name, r)
        if d == 256:
            assert nq == 1 and r["registers"] <= 168, (name, r)  # not re-split
        else:
            launch_regs = {2: 128, 1: 168}[nq]  # 65536 / threads, rounded down to a multiple of 8
            assert r["registers"] == launch_regs, (name, r)
    assert len(seen) == 36


def test_backward_workspace_size_and_host_checks(lib):
    r256 = lambda x: (x + 255) // 256 * 256
    n = fa.fa_bwd_workspace_bytes(2, 3, 100, 64)
    assert n == 2 * r256(2 * 3 * 192 * 4)  # N padded to a multiple of 192
    assert fa.fa_bwd_workspace_bytes(2, 3, 0, 64) == 0
    ws = FAKE * 16
    common = (2, 3, 100, 64, 0.125, 0)
    ptrs = [FAKE] * 9
    assert fa.fa_bwd(*ptrs, *common, ws, n - 1, None) == -9            # workspace too small
    assert fa.fa_bwd(*ptrs, *common, FAKE + 16, n, None) == -4         # workspace not 256-byte aligned
    assert fa.fa_bwd(*ptrs, *common, 0, n, None) == -1                 # workspace missing
    assert fa.fa_bwd(*ptrs[:5], 0, *ptrs[6:], *common, ws, n, None) == -1   # dO missing
    assert fa.fa_bwd(*ptrs, 2, 3, 100, 48, 0.125, 0, ws, n, None) == -3     # no d = 48 kernel
    assert fa.fa_bwd(*ptrs, 2, 3, 100, 64, -1.0, 0, ws, n, None) == -8
    bad = list(ptrs)
    bad[6] = FAKE + 8
    assert fa.fa_bwd(*bad, *common, ws, n, None) == -4                 # dq not 16-byte aligned


def test_backward_kernels_do_not_spill():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    rep = build.ptxas_report({f"fa_bwd_d{d}{s}.cu" for d in (32, 64, 128, 256) for s in ("", "_strided")})
    ks = {k: v for k, v in rep.items() if "fa_bwd" in k}
    # per head dimension: 8 tensor-core kernels (dK/dV or dQ x causal or not x contiguous or
    # strided) and 1 preprocessing kernel
    assert len(ks) == 36
    for name, r in ks.items():
        assert r["spill_stores"] == 0 and r["spill_loads"] == 0, (name, r)


def test_strided_forward_rejects_bad_arguments_on_host(lib):
    ok = (1 << 20, 1 << 14, 128)       # {batch, head, row} element strides, multiples of 8
    bad = (1 << 20, 1 << 14, 132)      # row stride not a multiple of 8 elements
    args = [FAKE] * 5 + [2, 3, 100, 70, 128]
    assert fa.fa_fwd_strided(*args, ok, ok, ok, bad, 0.1, 1, None) == -4
    assert fa.fa_fwd_strided(*args, ok, (0, 8, 8), ok, ok, 0.1, 1, None) == -2
    assert fa.fa_fwd_strided(*[FAKE] * 5, 2, 3, 100, 0, 128, ok, ok, ok, ok, 0.1, 1, None) == -2
    assert fa.fa_fwd_strided(*[FAKE] * 5, 2, 3, 100, 70, 48, ok, ok, ok, ok, 0.1, 1, None) == -3
    assert fa.fa_fwd_strided(*[FAKE] * 4, 0, 2, 3, 100, 70, 128, ok, ok, ok, ok, 0.1, 1, None) == -1


def test_strided_backward_rejects_bad_arguments_on_host(lib):
    ok = (1 << 20, 1 << 14, 128)
    st = [ok] * 8
    r256 = lambda x: (x + 255) // 256 * 256
    n = fa.fa_bwd_workspace_bytes(2, 3, 100, 128)       # sized by Nq = 100
    assert n == 2 * r256(2 * 3 * 192 * 4)
    ws = FAKE * 16
    ptrs = [FAKE] * 9

    def call(ptrs=ptrs, Nq=100, Nk=70, d=128, strides=st, scale=0.1, ws=ws, nbytes=n):
        return fa.fa_bwd_strided(*ptrs, 2, 3, Nq, Nk, d, strides, scale, 1, ws, nbytes, None)

    assert call(nbytes=n - 1) == -9                                   # workspace too small for Nq
    assert call(Nq=300) == -9
    assert call(strides=st[:5] + [(1 << 20, 1 << 14, 132)] + st[6:]) == -4   # dq row stride not 16-byte
    assert call(strides=st[:6] + [(0, 8, 8)] + st[7:]) == -2          # dk batch stride 0
    assert call(Nk=0) == -2
    assert call(d=48) == -3
    assert call(scale=float("nan")) == -8
    assert call(ptrs=ptrs[:8] + [0]) == -1                            # dv missing
    assert call(ptrs=ptrs[:2] + [FAKE + 4] + ptrs[3:]) == -4          # v not 16-byte aligned
    with pytest.raises(ValueError):
        fa.fa_bwd_strided(*ptrs, 2, 3, 100, 70, 128, st[:7], 0.1, 1, ws, n, None)
