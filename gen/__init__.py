"""Seeded synthetic inputs for the attention forward pass.

This module is shared by the oracle-side tests, the GPU parity tests and the
benchmark. It holds no attention arithmetic: it only names the workloads and
draws their Q, K, V tensors.

Recipe (the pages benchmark only random-normal inputs, e.g. the CS336
"05_flash_attention.py" demo draws ``torch.randn`` tensors and the
"手写 Flash Attention" page times randn inputs in its measurement section):

* every element of Q, K and V is an independent standard normal draw from
  numpy's PCG64 generator seeded with ``[seed, tensor_id]`` (Q=0, K=1, V=2),
  drawn in float64, multiplied by the workload's ``std`` and then rounded
  round-to-nearest-even to the workload's 16-bit type (fp16 or bf16);
* the 16-bit values are the inputs of BOTH the CUDA path and the oracle (the
  oracle widens them exactly to float64).
* FP8 workloads (dtype "e4m3") draw the same normals and round them to the OCP
  FP8 E4M3 format (torch.float8_e4m3fn, round-to-nearest-even; |x| <= 448 for
  every draw used here); their output O is bf16.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

F16 = "f16"
BF16 = "bf16"
FP8 = "e4m3"

_TORCH_DTYPE = {F16: torch.float16, BF16: torch.bfloat16, FP8: torch.float8_e4m3fn}
_ELEM_BYTES = {F16: 2, BF16: 2, FP8: 1}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Nq: int
    Nk: int
    d: int
    dtype: str
    causal: bool
    std: float = 1.0
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def flops(self) -> float:
        """4*B*H*Nq*Nk*d, halved for the causal mask (two GEMMs, 2 flops per MAC)."""
        f = 4.0 * self.B * self.H * self.Nq * self.Nk * self.d
        return f / 2 if self.causal else f

    @property
    def out_dtype(self) -> str:
        """Type of O: the input type, or bf16 for FP8 inputs."""
        return BF16 if self.dtype == FP8 else self.dtype

    @property
    def io_bytes(self) -> int:
        """Algorithmic HBM bytes: read Q, K, V once; write O (16-bit) and L (fp32)."""
        e = _ELEM_BYTES[self.dtype]
        bh = self.B * self.H
        return bh * (self.Nq * self.d * (e + 2) + self.Nk * self.d * e * 2 + self.Nq * 4)

    def describe(self) -> str:
        return (f"B={self.B},H={self.H},Nq={self.Nq},Nk={self.Nk},d={self.d},"
                f"{self.dtype},{'causal' if self.causal else 'full'},std={self.std:g}")


# The five synthetic workloads (sizes, types and value distributions as the
# project's target configurations state them).
WORKLOADS = {
    "tiny": Workload("tiny", 1, 1, 128, 128, 64, F16, False, 1.0, 1),
    "tiny_causal": Workload("tiny_causal", 1, 1, 128, 128, 64, F16, True, 1.0, 1),
    "b2h8_n4096_d128_full": Workload("b2h8_n4096_d128_full", 2, 8, 4096, 4096, 128, BF16, False, 1.0, 2),
    "b2h8_n8192_d128_causal": Workload("b2h8_n8192_d128_causal", 2, 8, 8192, 8192, 128, BF16, True, 1.0, 3),
    "b1h16_n32768_d128_causal_x2": Workload("b1h16_n32768_d128_causal_x2", 1, 16, 32768, 32768, 128, BF16, True, 2.0, 4),
    "b4h12_q1000_k4097_d64_cross": Workload("b4h12_q1000_k4097_d64_cross", 4, 12, 1000, 4097, 64, F16, False, 1.0, 5),
}

# FP8 (E4M3) versions of the two d=128 benchmark workloads: same sizes, seeds and draws.
FP8_WORKLOADS = {
    "b2h8_n4096_d128_full_fp8": Workload("b2h8_n4096_d128_full_fp8", 2, 8, 4096, 4096, 128, FP8, False, 1.0, 2),
    "b2h8_n8192_d128_causal_fp8": Workload("b2h8_n8192_d128_causal_fp8", 2, 8, 8192, 8192, 128, FP8, True, 1.0, 3),
}


def _draw(seed: int, tensor_id: int, shape, std: float, dtype: str) -> torch.Tensor:
    rng = np.random.default_rng([int(seed), int(tensor_id)])
    x = rng.standard_normal(size=shape, dtype=np.float64)
    if std != 1.0:
        x *= std
    # float64 -> float32 is exact for the subsequent 16-bit rounding except for
    # double rounding at exact ties, which cannot matter for random normals;
    # avoid it anyway by rounding directly from float64 in torch.
    t = torch.from_numpy(x)
    if dtype == FP8:  # torch rounds to E4M3 from float32; a float64 tie is measure-zero
        t = t.to(torch.float32)
    return t.to(_TORCH_DTYPE[dtype])


def make_qkv(w: Workload, seed: int | None = None):
    """Return host (CPU) tensors Q [B,H,Nq,d], K [B,H,Nk,d], V [B,H,Nk,d] of w.dtype."""
    s = w.seed if seed is None else seed
    q = _draw(s, 0, (w.B, w.H, w.Nq, w.d), w.std, w.dtype)
    k = _draw(s, 1, (w.B, w.H, w.Nk, w.d), w.std, w.dtype)
    v = _draw(s, 2, (w.B, w.H, w.Nk, w.d), w.std, w.dtype)
    return q, k, v


def custom(B, H, Nq, Nk, d, dtype=BF16, causal=False, std=1.0, seed=0, name="custom") -> Workload:
    return Workload(name, B, H, Nq, Nk, d, dtype, causal, std, seed)


def torch_dtype(dtype: str) -> torch.dtype:
    return _TORCH_DTYPE[dtype]


def to_f64_numpy(t: torch.Tensor) -> np.ndarray:
    """Exact widening of a 16-bit or FP8 tensor to a float64 numpy array."""
    return t.to(torch.float64).numpy()


def elem_bytes(dtype: str) -> int:
    return _ELEM_BYTES[dtype]
