"""fp64 CPU oracle for the attention forward pass.

TEST INFRASTRUCTURE ONLY: imported by tests, by the smoke check and by the
benchmark's CPU-baseline and reference legs, never by the product path.
"""
from .attention import attention, attention_head, logsumexp_rows, probabilities, scores

__all__ = ["attention", "attention_head", "logsumexp_rows", "probabilities", "scores"]
