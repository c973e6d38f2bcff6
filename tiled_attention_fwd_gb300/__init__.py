"""FlashAttention-2 forward pass for GB300 (sm_103a).

The compute path is the C-ABI library ``libfa_gb300.so`` (hand-written CUDA:
TMA + tcgen05 tensor-core kernel for bf16, SIMT kernel for fp32); this package
only loads it and marshals arguments.  Build it with
``python -m tiled_attention_fwd_gb300.build``.
"""
from ._lib import (FAError, check_status, declared_functions, fa_abi_version, fa_fwd, fa_fwd_f32,
                   fa_fwd_host, fa_fwd_host_workspace_bytes, fa_fwd_noalloc, fa_set_wait_limit_ms, fa_status, fa_strerror,
                   forward, load)

__all__ = [
    "FAError", "check_status", "declared_functions", "fa_abi_version", "fa_fwd", "fa_fwd_f32", "fa_fwd_host",
    "fa_fwd_host_workspace_bytes", "fa_fwd_noalloc", "fa_set_wait_limit_ms", "fa_status", "fa_strerror", "forward", "load",
]
