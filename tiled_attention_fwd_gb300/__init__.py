"""FlashAttention-2 forward (and backward) pass for GB300 (sm_103a).

The compute path is the C-ABI library ``libfa_gb300.so`` (hand-written CUDA:
TMA + tcgen05 tensor-core kernels for bf16 and e4m3, SIMT kernel for fp32); this package
only loads it and marshals arguments.  Build it with
``python -m tiled_attention_fwd_gb300.build``.
"""
from ._lib import (FAError, backward, check_status, declared_functions, fa_abi_version, fa_bwd, fa_bwd_strided,
                   fa_bwd_workspace_bytes, fa_fwd, fa_fwd_f32, fa_fwd_fp8, fa_fwd_host, fa_fwd_host_workspace_bytes, fa_fwd_noalloc, fa_fwd_strided,
                   fa_selftest_wait, fa_set_wait_limit_ms, fa_status, fa_strerror, forward, forward_fp8, load)

__all__ = [
    "FAError", "backward", "check_status", "declared_functions", "fa_abi_version", "fa_bwd", "fa_bwd_strided",
    "fa_bwd_workspace_bytes",
    "fa_fwd", "fa_fwd_f32", "fa_fwd_fp8", "fa_fwd_host", "fa_fwd_strided",
    "fa_fwd_host_workspace_bytes", "fa_fwd_noalloc", "fa_selftest_wait", "fa_set_wait_limit_ms", "fa_status", "fa_strerror", "forward", "forward_fp8", "load",
]
