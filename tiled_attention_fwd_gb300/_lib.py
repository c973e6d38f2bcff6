"""ctypes binding of libfa_gb300.so: the C ABI with the same names, and a
torch-tensor convenience wrappers.  Argument marshalling only: every step of
the forward and backward passes runs in the library's CUDA kernels.  There is no fallback:
if the library is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libfa_gb300.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "fa_gb300.h")

_c_void_p = ctypes.c_void_p
_c_int = ctypes.c_int
_c_float = ctypes.c_float
_c_size_t = ctypes.c_size_t

# (name, restype, argtypes) of every entry point declared in include/fa_gb300.h
_SIGNATURES = {
    "fa_fwd": (_c_int, [_c_void_p] * 5 + [_c_int] * 4 + [_c_float, _c_int, _c_void_p]),
    "fa_fwd_f32": (_c_int, [_c_void_p] * 5 + [_c_int] * 4 + [_c_float, _c_int, _c_void_p]),
    "fa_fwd_fp8": (_c_int, [_c_void_p] * 5 + [_c_int] * 4 + [_c_float] * 4 + [_c_int, _c_void_p]),
    "fa_fwd_strided": (_c_int, [_c_void_p] * 5 + [_c_int] * 5 + [_c_void_p] * 4 + [_c_float, _c_int, _c_void_p]),
    "fa_fwd_host_workspace_bytes": (_c_size_t, [_c_int] * 4),
    "fa_fwd_host": (_c_int, [_c_void_p] * 6 + [_c_size_t] + [_c_int] * 4 + [_c_float, _c_int, _c_void_p]),
    "fa_fwd_noalloc": (_c_int, [_c_void_p] * 5 + [_c_int] * 4 + [_c_float, _c_int, _c_void_p]),
    "fa_bwd_workspace_bytes": (_c_size_t, [_c_int] * 4),
    "fa_bwd": (_c_int, [_c_void_p] * 9 + [_c_int] * 4 + [_c_float, _c_int, _c_void_p, _c_size_t, _c_void_p]),
    "fa_bwd_strided": (_c_int, [_c_void_p] * 9 + [_c_int] * 5 + [_c_void_p, _c_float, _c_int, _c_void_p, _c_size_t,
                                                                  _c_void_p]),
    "fa_status": (_c_int, [_c_void_p]),
    "fa_selftest_wait": (_c_int, [_c_void_p]),
    "fa_set_wait_limit_ms": (_c_int, [_c_int]),
    "fa_strerror": (ctypes.c_char_p, [_c_int]),
    "fa_abi_version": (_c_int, []),
}

FA_OK = 0
FA_ERR_TIMEOUT = -6

_lib = None


class FAError(RuntimeError):
    """A nonzero return code of the C ABI."""

    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {strerror(code)} ({code})")


def declared_functions(header: str = HEADER):
    """Names of the functions declared in the public header."""
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def load(path: str = LIB_PATH):
    """Load the shared library (once) and attach the C signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it with `python -m tiled_attention_fwd_gb300.build` "
            "(or __graft_entry__.build()); there is no fallback implementation")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def strerror(code: int) -> str:
    return load().fa_strerror(code).decode()


def _check(rc: int, where: str):
    if rc != FA_OK:
        raise FAError(rc, where)


# ---------------------------------------------------------------- C ABI, same names
def fa_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, stream) -> int:
    """bf16 tensor-core forward; pointers are integers (device addresses)."""
    return load().fa_fwd(q, k, v, o, lse, B, H, N, d, scale, int(bool(causal)), stream)


def _strides3(st):
    arr = (ctypes.c_longlong * 3)(*[int(x) for x in st])
    return arr


def fa_fwd_strided(q, k, v, o, lse, B, H, Nq, Nk, d, q_stride, k_stride, v_stride, o_stride, scale, causal,
                   stream) -> int:
    """bf16 forward with Nq != Nk allowed and {batch, head, row} element strides per tensor."""
    arrs = [_strides3(x) for x in (q_stride, k_stride, v_stride, o_stride)]
    return load().fa_fwd_strided(q, k, v, o, lse, B, H, Nq, Nk, d, *[ctypes.addressof(a) for a in arrs], scale,
                                 int(bool(causal)), stream)


def fa_fwd_f32(q, k, v, o, lse, B, H, N, d, scale, causal, stream) -> int:
    """fp32 SIMT forward; pointers are integers (device addresses)."""
    return load().fa_fwd_f32(q, k, v, o, lse, B, H, N, d, scale, int(bool(causal)), stream)


def fa_fwd_fp8(q, k, v, o, lse, B, H, N, d, scale, q_descale, k_descale, v_descale, causal, stream) -> int:
    """e4m3 tensor-core forward (bf16 O, fp32 L); pointers are integers (device addresses)."""
    return load().fa_fwd_fp8(q, k, v, o, lse, B, H, N, d, scale, q_descale, k_descale, v_descale, int(bool(causal)),
                             stream)


def fa_fwd_host_workspace_bytes(B, H, N, d) -> int:
    return load().fa_fwd_host_workspace_bytes(B, H, N, d)


def fa_fwd_host(q, k, v, o, lse, workspace, workspace_bytes, B, H, N, d, scale, causal, stream) -> int:
    """bf16 forward on host buffers (copies in, kernel, copies out, all on `stream`)."""
    return load().fa_fwd_host(q, k, v, o, lse, workspace, workspace_bytes, B, H, N, d, scale,
                              int(bool(causal)), stream)


def fa_fwd_noalloc(q, k, v, o, lse, B, H, N, d, scale, causal, stream) -> int:
    """fa_fwd without any device allocation (scratch in a static device array)."""
    return load().fa_fwd_noalloc(q, k, v, o, lse, B, H, N, d, scale, int(bool(causal)), stream)


def fa_bwd_workspace_bytes(B, H, N, d) -> int:
    return load().fa_bwd_workspace_bytes(B, H, N, d)


def fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, scale, causal, workspace, workspace_bytes,
           stream) -> int:
    """bf16 tensor-core backward; pointers are integers (device addresses)."""
    return load().fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, scale, int(bool(causal)), workspace,
                         workspace_bytes, stream)


def fa_bwd_strided(q, k, v, o, lse, dout, dq, dk, dv, B, H, Nq, Nk, d, strides, scale, causal, workspace,
                   workspace_bytes, stream) -> int:
    """fa_bwd with Nq != Nk allowed; `strides` holds 8 {batch, head, row} element-stride triples
    (q, k, v, o, dout, dq, dk, dv)."""
    flat = [int(x) for st in strides for x in st]
    if len(flat) != 24:
        raise ValueError("strides must hold 8 triples")
    arr = (ctypes.c_longlong * 24)(*flat)
    return load().fa_bwd_strided(q, k, v, o, lse, dout, dq, dk, dv, B, H, Nq, Nk, d, ctypes.addressof(arr), scale,
                                 int(bool(causal)), workspace, workspace_bytes, stream)


def fa_status(stream) -> int:
    return load().fa_status(stream)


def fa_selftest_wait(stream) -> int:
    """Enqueue the bounded-wait diagnostic (every wait expires after the current limit)."""
    return load().fa_selftest_wait(stream)


def fa_set_wait_limit_ms(ms: int) -> int:
    return load().fa_set_wait_limit_ms(ms)


def fa_strerror(code: int) -> str:
    return strerror(code)


def fa_abi_version() -> int:
    return load().fa_abi_version()


# ---------------------------------------------------------------- torch convenience
def _stream_handle(torch, device):
    return torch.cuda.current_stream(device).cuda_stream


def forward(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None):
    """O, L = attention forward of CUDA tensors q [B, H, Nq, d], k and v [B, H, Nk, d].

    bf16 inputs run the tensor-core kernel (d in {32, 64, 128, 256}); any
    layout whose last dimension is contiguous is accepted (views of [B, N, H, d]
    storage, for instance), and Nq may differ from Nk (causal: key k visible to
    query i iff k <= i).  fp32 inputs run the SIMT kernel (contiguous, Nq = Nk,
    1 <= d <= 256).  Returns (O, L): O like q ([B, H, Nq, d], contiguous unless
    `out` is given) and L fp32 contiguous [B, H, Nq].  Enqueued on the current stream.
    """
    import torch

    if q.dim() != 4 or k.dim() != 4 or k.shape != v.shape:
        raise ValueError("q must be [B, H, Nq, d] and k, v [B, H, Nk, d]")
    if q.shape[:2] != k.shape[:2] or q.shape[3] != k.shape[3]:
        raise ValueError("q, k, v must share B, H and d")
    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("q, k, v must be CUDA tensors")
    if not (q.dtype == k.dtype == v.dtype) or q.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("q, k, v must all be bf16 or all fp32")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if scale is None:
        scale = d ** -0.5
    o = torch.empty(q.shape, device=q.device, dtype=q.dtype) if out is None else out
    if o.shape != q.shape or o.dtype != q.dtype:
        raise ValueError("out must have q's shape and dtype")
    l = torch.empty((B, H, Nq), device=q.device, dtype=torch.float32) if lse is None else lse
    if l.shape != (B, H, Nq) or l.dtype != torch.float32 or not l.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 tensor [B, H, Nq]")
    plain = Nq == Nk and all(t.is_contiguous() for t in (q, k, v, o))
    with torch.cuda.device(q.device):
        stream = _stream_handle(torch, q.device)
        if plain:
            fn = fa_fwd if q.dtype == torch.bfloat16 else fa_fwd_f32
            rc = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), l.data_ptr(), B, H, Nq, d,
                    float(scale), causal, stream)
            name = fn.__name__
        else:
            if q.dtype != torch.bfloat16:
                raise ValueError("fp32 inputs must be contiguous with Nq == Nk")
            if any(t.stride(3) != 1 for t in (q, k, v, o)):
                raise ValueError("the last dimension of q, k, v and out must be contiguous")
            rc = fa_fwd_strided(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), l.data_ptr(), B, H, Nq, Nk, d,
                                q.stride()[:3], k.stride()[:3], v.stride()[:3], o.stride()[:3], float(scale), causal,
                                stream)
            name = "fa_fwd_strided"
    _check(rc, name)
    return o, l


def forward_fp8(q8, k8, v8, descales, causal: bool = False, scale: float | None = None, out=None, lse=None):
    """O, L = attention forward of e4m3 CUDA tensors q8, k8, v8 [B, H, N, d]
    (torch.float8_e4m3fn, contiguous, d in {64, 128}) whose real values are
    descales[i] * x8 (one factor per tensor, in the order q, k, v).  Returns
    (O, L): O bf16 [B, H, N, d] and L fp32 [B, H, N].  Enqueued on the
    current stream."""
    import torch

    ts = (q8, k8, v8)
    if any(t.dim() != 4 for t in ts) or not (q8.shape == k8.shape == v8.shape):
        raise ValueError("q8, k8, v8 must be [B, H, N, d] of one shape")
    if not all(t.is_cuda and t.dtype == torch.float8_e4m3fn and t.is_contiguous() for t in ts):
        raise ValueError("q8, k8, v8 must be contiguous float8_e4m3fn CUDA tensors")
    B, H, N, d = q8.shape
    if scale is None:
        scale = d ** -0.5
    o = torch.empty(q8.shape, device=q8.device, dtype=torch.bfloat16) if out is None else out
    if o.shape != q8.shape or o.dtype != torch.bfloat16 or not o.is_contiguous():
        raise ValueError("out must be a contiguous bf16 tensor shaped like q8")
    l = torch.empty((B, H, N), device=q8.device, dtype=torch.float32) if lse is None else lse
    if l.shape != (B, H, N) or l.dtype != torch.float32 or not l.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 tensor [B, H, N]")
    qd, kd, vd = (float(x) for x in descales)
    with torch.cuda.device(q8.device):
        rc = fa_fwd_fp8(q8.data_ptr(), k8.data_ptr(), v8.data_ptr(), o.data_ptr(), l.data_ptr(), B, H, N, d,
                        float(scale), qd, kd, vd, causal, _stream_handle(torch, q8.device))
    _check(rc, "fa_fwd_fp8")
    return o, l


def backward(q, k, v, o, lse, dout, causal: bool = False, scale: float | None = None, workspace=None,
             out=None):
    """dQ, dK, dV of the attention forward for bf16 CUDA tensors.

    q, o, dout are [B, H, Nq, d] and k, v [B, H, Nk, d], in any layout whose
    last dimension is contiguous; ``o`` and ``lse`` (fp32 contiguous
    [B, H, Nq]) are the outputs of ``forward`` for the same q, k, v, causal
    and scale; ``dout`` is the upstream gradient.  ``workspace`` (a CUDA uint8
    tensor of at least fa_bwd_workspace_bytes(B, H, Nq, d), 256-byte aligned)
    is allocated here if not given; so are the outputs unless ``out`` =
    (dq, dk, dv) is given (shaped like q, k, v).  Returns (dQ, dK, dV) in
    bf16.  Enqueued on the current stream.
    """
    import torch

    if q.dim() != 4 or k.dim() != 4 or k.shape != v.shape or o.shape != q.shape or dout.shape != q.shape:
        raise ValueError("q, o, dout must be [B, H, Nq, d] and k, v [B, H, Nk, d]")
    if q.shape[:2] != k.shape[:2] or q.shape[3] != k.shape[3]:
        raise ValueError("q, k, v must share B, H and d")
    ts = (q, k, v, o, dout)
    if not all(t.is_cuda and t.dtype == torch.bfloat16 for t in ts):
        raise ValueError("q, k, v, o, dout must be bf16 CUDA tensors")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if lse.shape != (B, H, Nq) or lse.dtype != torch.float32 or not lse.is_cuda or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 CUDA tensor [B, H, Nq]")
    if scale is None:
        scale = d ** -0.5
    need = fa_bwd_workspace_bytes(B, H, Nq, d)
    if workspace is None:
        workspace = torch.empty(need, device=q.device, dtype=torch.uint8)
    if out is None:
        dq, dk, dv = (torch.empty(t.shape, device=t.device, dtype=t.dtype) for t in (q, k, v))
    else:
        dq, dk, dv = out
        if dq.shape != q.shape or dk.shape != k.shape or dv.shape != v.shape or \
                any(t.dtype != torch.bfloat16 or not t.is_cuda for t in out):
            raise ValueError("out must be bf16 CUDA tensors shaped like q, k, v")
    all_t = ts + (dq, dk, dv)
    plain = Nq == Nk and all(t.is_contiguous() for t in all_t)
    ws_bytes = workspace.numel() * workspace.element_size()
    with torch.cuda.device(q.device):
        stream = _stream_handle(torch, q.device)
        if plain:
            rc = fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dout.data_ptr(),
                        dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, Nq, d, float(scale), causal,
                        workspace.data_ptr(), ws_bytes, stream)
            name = "fa_bwd"
        else:
            if any(t.stride(3) != 1 for t in all_t):
                raise ValueError("the last dimension of every tensor must be contiguous")
            rc = fa_bwd_strided(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, Nq, Nk, d,
                                [t.stride()[:3] for t in all_t], float(scale), causal, workspace.data_ptr(),
                                ws_bytes, stream)
            name = "fa_bwd_strided"
    _check(rc, name)
    return dq, dk, dv


def check_status(device=None):
    """Synchronise the current stream and raise FAError if a device wait timed out."""
    import torch

    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        _check(fa_status(_stream_handle(torch, dev)), "fa_status")
