"""fp64 CPU oracle for the attention forward and backward passes.

TEST INFRASTRUCTURE ONLY: imported by tests, by the smoke check and by the
benchmark's CPU-baseline and reference legs, never by the product path.
"""
from .attention import attention, attention_head, logsumexp_rows, probabilities, scores
from .backward import attention_backward, attention_backward_head
from .fp8 import attention_fp8, attention_fp8_head, dequantize

__all__ = ["attention", "attention_head", "logsumexp_rows", "probabilities", "scores",
           "attention_backward", "attention_backward_head", "attention_fp8", "attention_fp8_head", "dequantize"]
