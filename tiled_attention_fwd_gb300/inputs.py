"""Seeded synthetic inputs for the attention forward pass.

This module is shared by the oracle-side tests and the CUDA-side tests and
benchmark. It holds no attention arithmetic: it only draws Q, K, V from a
seeded generator with the shapes, dtypes and value distributions of the
workloads below, and rounds them to the compute dtype.

Recipe (identical on every machine): a CPU ``torch.Generator`` seeded with
the workload's seed draws ``randn`` in fp32, in the order Q, K, V, each of
shape [B, H, N, d] (contiguous); Q and K are multiplied by ``qk_std``; the
three tensors are then cast to the workload's dtype (bf16 rounds to nearest
even). The oracle consumes exactly these rounded values, widened to fp64.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    """One attention problem: shapes, dtype, mask and input distribution."""

    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str  # "f32", "bf16" or "fp8" (e4m3 inputs with per-tensor factors, bf16 O)
    causal: bool
    seed: int
    qk_std: float = 1.0

    @property
    def scale(self) -> float:
        """Softmax scale 1/sqrt(d) (the scaled dot product of standard attention)."""
        return 1.0 / math.sqrt(self.d)

    @property
    def flops(self) -> float:
        """Algorithmic FLOPs: 4*B*H*N^2*d for the two matmuls, halved when causal."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2.0 if self.causal else f

    @property
    def torch_dtype(self) -> torch.dtype:
        return {"f32": torch.float32, "bf16": torch.bfloat16, "fp8": torch.float8_e4m3fn}[self.dtype]

    @property
    def elem_bytes(self) -> int:
        return {"f32": 4, "bf16": 2, "fp8": 1}[self.dtype]

    @property
    def io_bytes(self) -> int:
        """Bytes read (Q, K, V once) plus written (O once, L in fp32); O is bf16 for fp8 inputs."""
        n = self.B * self.H * self.N * self.d
        o_bytes = 2 if self.dtype == "fp8" else self.elem_bytes
        return 3 * n * self.elem_bytes + n * o_bytes + self.B * self.H * self.N * 4

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads of the headline measurement plan.  The seed is the
# workload's index; the head-dim sweep reuses seed 4 for every d.
WORKLOADS = {
    "f32_b1h1n128d16": Workload("f32_b1h1n128d16", 1, 1, 128, 16, "f32", False, 0),
    "f32_b1h1n128d16_causal": Workload("f32_b1h1n128d16_causal", 1, 1, 128, 16, "f32", True, 0),
    "bf16_b8h1n1024d64": Workload("bf16_b8h1n1024d64", 8, 1, 1024, 64, "bf16", False, 1),
    "bf16_b8h1n1024d64_causal": Workload("bf16_b8h1n1024d64_causal", 8, 1, 1024, 64, "bf16", True, 1),
    "bf16_b4h16n4096d128_causal": Workload("bf16_b4h16n4096d128_causal", 4, 16, 4096, 128, "bf16", True, 2),
    "bf16_b1h32n16384d128_causal": Workload("bf16_b1h32n16384d128_causal", 1, 32, 16384, 128, "bf16", True, 3),
    "bf16_b2h16n8192d32_qk3": Workload("bf16_b2h16n8192d32_qk3", 2, 16, 8192, 32, "bf16", False, 4, 3.0),
    "bf16_b2h16n8192d64_qk3": Workload("bf16_b2h16n8192d64_qk3", 2, 16, 8192, 64, "bf16", False, 4, 3.0),
    "bf16_b2h16n8192d128_qk3": Workload("bf16_b2h16n8192d128_qk3", 2, 16, 8192, 128, "bf16", False, 4, 3.0),
    "bf16_b2h16n8192d256_qk3": Workload("bf16_b2h16n8192d256_qk3", 2, 16, 8192, 256, "bf16", False, 4, 3.0),
    # The low-precision variant on the headline shape and the d = 128 sweep point (e4m3 inputs).
    "fp8_b4h16n4096d128_causal": Workload("fp8_b4h16n4096d128_causal", 4, 16, 4096, 128, "fp8", True, 2),
    "fp8_b2h16n8192d128_qk3": Workload("fp8_b2h16n8192d128_qk3", 2, 16, 8192, 128, "fp8", False, 4, 3.0),
}

HEADLINE = "bf16_b4h16n4096d128_causal"


def make_qkv(w: Workload):
    """Draw Q, K, V for workload ``w`` on the CPU, already rounded to ``w.dtype``."""
    g = torch.Generator(device="cpu").manual_seed(w.seed)
    shape = (w.B, w.H, w.N, w.d)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.randn(shape, generator=g, dtype=torch.float32)
    if w.qk_std != 1.0:
        q = q * w.qk_std
        k = k * w.qk_std
    dt = w.torch_dtype
    return q.to(dt).contiguous(), k.to(dt).contiguous(), v.to(dt).contiguous()


E4M3_MAX = 448.0  # largest finite e4m3 value


def make_qkv_fp8(w: Workload):
    """Q, K, V of workload ``w`` quantised to e4m3 with one dequantisation
    factor per tensor.

    The same seeded fp32 draws as make_qkv (so the distributions are the
    workload's); each tensor's factor is the power of two 2^ceil(log2(amax /
    448)), which puts the largest magnitude just inside e4m3's range and keeps
    every dequantised value (e4m3 value times factor) exact in fp32; the
    tensor divided by its factor is rounded to e4m3 (nearest even).  Returns
    ((q8, k8, v8) as torch.float8_e4m3fn CPU tensors, (q_descale, k_descale,
    v_descale) as floats).
    """
    g = torch.Generator(device="cpu").manual_seed(w.seed)
    shape = (w.B, w.H, w.N, w.d)
    xs = [torch.randn(shape, generator=g, dtype=torch.float32) for _ in range(3)]
    if w.qk_std != 1.0:
        xs[0] = xs[0] * w.qk_std
        xs[1] = xs[1] * w.qk_std
    out, scales = [], []
    for x in xs:
        amax = float(x.abs().max())
        f = 2.0 ** math.ceil(math.log2(amax / E4M3_MAX)) if amax > 0 else 1.0
        out.append((x / f).to(torch.float8_e4m3fn).contiguous())
        scales.append(f)
    return tuple(out), tuple(scales)


def make_dout(w: Workload):
    """Upstream gradient dO for the backward pass of workload ``w``: N(0, 1) in
    w.dtype, drawn from its own generator (seed w.seed + 1000) so that Q, K, V
    are the same as for the forward pass."""
    g = torch.Generator(device="cpu").manual_seed(w.seed + 1000)
    do = torch.randn((w.B, w.H, w.N, w.d), generator=g, dtype=torch.float32)
    return do.to(w.torch_dtype).contiguous()


def as_f64_numpy(t: torch.Tensor):
    """Widen an (already rounded) CPU tensor to an fp64 numpy array."""
    return t.detach().to("cpu", torch.float64).numpy()
