"""Seeded synthetic inputs for the fused all-reduce epilogue.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic. Both the CUDA path's tests/benchmark and the CPU oracle
take their inputs from here.

Recipe (all draws from one ``torch.Generator`` seeded with ``seed``, in this
order): partials P_0 .. P_{N-1}, then the residual R, then gamma, then (when
outliers are requested) the outlier positions of P_0 .. P_{N-1}.
  * P_r  = bf16(std_p * z), z ~ N(0, 1) drawn in fp32, one RNE rounding
  * R    = bf16(std_r * z)
  * gamma = bf16(1 + 0.1 * z), shape [d]
  * outliers: exactly floor(frac * T * d) distinct positions per partial,
    uniform without replacement (a seeded permutation), whose fp32 draw is
    multiplied by ``outlier_scale`` before the single bf16 rounding.

On ``device='cuda'`` the same recipe runs with a CUDA generator (a different
random stream than on the CPU): large workloads are drawn on the GPU and the
oracle is fed copies of the very same tensors.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    """One shape/distribution of the epilogue, named for what it is."""
    name: str
    n_ranks: int
    T: int
    d: int
    eps: float
    partial_std: float
    residual_std: float = 1.0
    gamma_std: float = 0.1
    outlier_frac: float = 0.0
    outlier_scale: float = 50.0
    nvfp4: bool = False
    seed: int = 0
    note: str = field(default="", compare=False)

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


# The pages' shapes (Llama-3-8B / Llama-3.1-70B decode epilogues, a prefill
# epilogue, an NVFP4-emitting epilogue) and a tiny case the oracle finishes
# instantly.
SMALL = Workload("small N2 T4 d256", 2, 4, 256, 1e-6, 1.0)
DECODE_8B = Workload("decode llama3-8b N8 T8 d4096", 8, 8, 4096, 1e-5, 0.5,
                     note="CUDA-graph captured, 1000 back-to-back calls")
DECODE_70B = Workload("decode llama3.1-70b N8 T8 d8192", 8, 8, 8192, 1e-5, 0.5)
DECODE_70B_TS = (1, 2, 4, 8, 16, 32)
DECODE_70B_NS = (4, 8)
PREFILL = Workload("prefill N8 T4096 d8192", 8, 4096, 8192, 1e-5, 0.5)
NVFP4 = Workload("nvfp4 N4 T16384 d8192 1% x50 outliers", 4, 16384, 8192, 1e-6, 1.0,
                 outlier_frac=0.01, outlier_scale=50.0, nvfp4=True)
NVFP4_TS = tuple(2 ** k for k in range(15))  # 1 .. 16384


def make_inputs(w: Workload, device: str | torch.device = "cpu", T: int | None = None,
                n_ranks: int | None = None, seed: int | None = None, dtype=torch.bfloat16):
    """Draw the inputs of ``w`` (optionally overriding T / N / seed), rounded
    once to ``dtype`` (bf16, or fp16).

    Returns dict(partials=[N x [T, d]], residual=[T, d], gamma=[d]).
    """
    T = w.T if T is None else T
    n = w.n_ranks if n_ranks is None else n_ranks
    seed = w.seed if seed is None else seed
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    d = w.d
    raw = [torch.randn((T, d), generator=g, device=dev, dtype=torch.float32) * w.partial_std
           for _ in range(n)]
    res = torch.randn((T, d), generator=g, device=dev, dtype=torch.float32) * w.residual_std
    gamma = 1.0 + w.gamma_std * torch.randn((d,), generator=g, device=dev, dtype=torch.float32)
    if w.outlier_frac > 0.0 and T * d > 0:
        k = int(math.floor(w.outlier_frac * T * d))
        for p in raw:
            if k:
                idx = torch.randperm(T * d, generator=g, device=dev)[:k]
                flat = p.view(-1)
                flat[idx] = flat[idx] * w.outlier_scale
    return {
        "partials": [p.to(dtype) for p in raw],
        "residual": res.to(dtype),
        "gamma": gamma.to(dtype),
    }


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 or fp16 tensor (any device) -> numpy uint16 bit patterns."""
    if t.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError("expected a bf16 or fp16 tensor")
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def from_bits(a: np.ndarray, device="cpu", dtype=torch.bfloat16) -> torch.Tensor:
    """numpy uint16 bit patterns -> bf16 (or fp16) tensor."""
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16).copy()).view(dtype).to(device)


def random_bf16(shape, std: float, seed: int, device="cpu") -> torch.Tensor:
    """Plain N(0, std^2) bf16 tensor from its own seeded generator."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    return (torch.randn(shape, generator=g, device=dev, dtype=torch.float32) * std).to(torch.bfloat16)
