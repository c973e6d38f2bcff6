"""fp64 oracle of the fp8 (e4m3) forward pass.

TEST INFRASTRUCTURE ONLY (imported by tests and the benchmark's CPU legs,
never by the product path; shares no code with the CUDA path).

The pages define attention on real-valued inputs and mention low-precision
variants only as context (the closing section of "Case Study:
metal-flash-attention": MFA 2.0's int8 and sparse-indexed attention); they fix
no quantisation.  The reading taken here: each of Q, K, V is given as e4m3
values x8 with one fp32 dequantisation factor per tensor, and the real input
is x = descale * x8.  The method computes standard attention of those real
inputs, so the oracle is the plain definition ("Writing a FlashAttention
kernel in Metal", "Standard attention"; L as in "FlashAttention-2 from
PyTorch to Triton", "What We Are Building") applied to the dequantised
tensors.  How the kernel rounds on the way (P cast to V's dtype before the
P V product, as the Triton kernel of the latter page casts P to V's dtype)
is the kernel's business and enters only the tolerance of the parity tests.
"""
from __future__ import annotations

import numpy as np

from .attention import attention, attention_head


def dequantize(x8, descale: float) -> np.ndarray:
    """Real values of a quantised tensor: its e4m3 values (given widened to
    fp64) times the per-tensor dequantisation factor."""
    return np.asarray(x8, dtype=np.float64) * float(descale)


def attention_fp8_head(q8, k8, v8, q_descale, k_descale, v_descale, scale: float, causal: bool, rows=None):
    """O and L of one head ([N, d] e4m3 values widened to fp64) from the dequantised inputs."""
    return attention_head(dequantize(q8, q_descale), dequantize(k8, k_descale), dequantize(v8, v_descale), scale,
                          causal, rows)


def attention_fp8(q8, k8, v8, q_descale, k_descale, v_descale, scale: float, causal: bool, rows=None, heads=None):
    """O [B, H, R, d] and L [B, H, R] of [B, H, N, d] quantised inputs (see attention())."""
    return attention(dequantize(q8, q_descale), dequantize(k8, k_descale), dequantize(v8, v_descale), scale, causal,
                     rows, heads)
