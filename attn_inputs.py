"""Seeded synthetic inputs for the attention forward pass.

This module is shared by the parity tests, the benchmark and the oracle's
callers.  It holds no attention arithmetic: it only draws random tensors on
the CPU (torch.Generator, so the same seed gives the same bits on any host),
rounds them to the storage dtype and, for e4m3, applies the per-tensor
quantisation that defines the fp8 workload's inputs.

Workloads (shapes and distributions of the pages' benchmarks; the pages name
no public dataset, so these synthetic tensors are the inputs):

  fp32_n128_d64      B=1 H=1 N=128  d=64   fp32, N(0,1)
  bf16_n2048_d128    B=4 H=16 N=2048 d=128 bf16, N(0,1)
  bf16_n8192_d128    B=2 H=16 N=8192 d=128 bf16, N(0,1)   (head dim 128,
                     sequence 8192: the FA3 ablation / pingpong setting)
  outlier_d64        B=8 H=16 N=4096 d=64  fp16|bf16, Q/K N(0,1) with 4
                     seeded channels x20 in both, V U(-1,1)
  outlier_d256       same with d=256
  fp8_n8192_d128     B=2 H=16 N=8192 d=128 e4m3: N(0,1) quantised with a
                     per-tensor fp32 scale amax/448

The seed of workload number c (0-based in the list above, both outlier
workloads share index 3) is 1234 + c; Q is drawn first, then K, then V.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

E4M3_MAX = 448.0

DTYPES = {
    "fp32": torch.float32,
    "fp16": torch.float16,
    "bf16": torch.bfloat16,
    "fp8": torch.float8_e4m3fn,
}


@dataclass
class AttnInputs:
    q: torch.Tensor          # [B, H, N, d] on the CPU, storage dtype
    k: torch.Tensor
    v: torch.Tensor
    scale: float             # softmax scale (1/sqrt(d))
    dtype: str               # "fp32" | "fp16" | "bf16" | "fp8"
    descale: dict = field(default_factory=lambda: {"q": 1.0, "k": 1.0, "v": 1.0})

    @property
    def shape(self):
        return tuple(self.q.shape)

    def as_float64(self):
        """The values the GPU reads, exactly upcast to fp64 (for e4m3: the
        stored code times its per-tensor descale)."""
        out = []
        for name, t in (("q", self.q), ("k", self.k), ("v", self.v)):
            x = t.to(torch.float64)
            if self.dtype == "fp8":
                x = x * float(self.descale[name])
            out.append(x)
        return tuple(out)


def _draw(gen: torch.Generator, shape, dist: str) -> torch.Tensor:
    if dist == "normal":
        return torch.randn(shape, generator=gen, dtype=torch.float32)
    if dist == "uniform":
        return torch.rand(shape, generator=gen, dtype=torch.float32) * 2.0 - 1.0
    raise ValueError(dist)


def _quantise_e4m3(x: torch.Tensor):
    """Per-tensor scale amax/448; codes = RNE(x / scale) in e4m3 (no value
    exceeds 448 after the division, so nothing saturates)."""
    amax = float(x.abs().max())
    scale = amax / E4M3_MAX if amax > 0 else 1.0
    scale = float(torch.tensor(scale, dtype=torch.float32))
    codes = (x / scale).to(torch.float8_e4m3fn)
    return codes, scale


def make_inputs(B: int, H: int, N: int, d: int, dtype: str = "bf16", seed: int = 0,
                outliers: int = 0, outlier_gain: float = 20.0,
                v_dist: str = "normal", scale: Optional[float] = None) -> AttnInputs:
    """Draw Q, K, V of shape [B, H, N, d].

    outliers > 0 picks that many channel indices with the seed and multiplies
    those channels of both Q and K by outlier_gain (stresses the max
    subtraction).  v_dist is "normal" (N(0,1)) or "uniform" (U(-1,1)).
    """
    if dtype not in DTYPES:
        raise ValueError(f"unknown dtype {dtype}")
    gen = torch.Generator(device="cpu")
    gen.manual_seed(int(seed))
    shape = (B, H, N, d)
    q = _draw(gen, shape, "normal")
    k = _draw(gen, shape, "normal")
    v = _draw(gen, shape, v_dist)
    if outliers:
        ch = torch.randperm(d, generator=gen)[:outliers]
        q[..., ch] *= outlier_gain
        k[..., ch] *= outlier_gain
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if dtype == "fp8":
        q8, sq = _quantise_e4m3(q)
        k8, sk = _quantise_e4m3(k)
        v8, sv = _quantise_e4m3(v)
        return AttnInputs(q8, k8, v8, float(scale), dtype, {"q": sq, "k": sk, "v": sv})
    td = DTYPES[dtype]
    return AttnInputs(q.to(td), k.to(td), v.to(td), float(scale), dtype)


# name -> (B, H, N, d, dtype, seed index, extra kwargs)
WORKLOADS = {
    "fp32_n128_d64": (1, 1, 128, 64, "fp32", 0, {}),
    "bf16_n2048_d128": (4, 16, 2048, 128, "bf16", 1, {}),
    "bf16_n8192_d128": (2, 16, 8192, 128, "bf16", 2, {}),
    "outlier_d64": (8, 16, 4096, 64, "bf16", 3, {"outliers": 4, "v_dist": "uniform"}),
    "outlier_d256": (8, 16, 4096, 256, "bf16", 3, {"outliers": 4, "v_dist": "uniform"}),
    "fp8_n8192_d128": (2, 16, 8192, 128, "fp8", 4, {}),
}


def workload(name: str, dtype: Optional[str] = None) -> AttnInputs:
    """Inputs of a named workload; dtype overrides the storage type where the
    workload allows two (the outlier sweeps run in fp16 or bf16)."""
    B, H, N, d, dt, idx, kw = WORKLOADS[name]
    if dtype is not None:
        if name.startswith("outlier") and dtype in ("fp16", "bf16"):
            dt = dtype
        elif dtype != dt:
            raise ValueError(f"{name} is defined for {dt} only")
    return make_inputs(B, H, N, d, dt, seed=1234 + idx, **kw)


def workload_flops(B: int, H: int, N: int, d: int, causal: bool) -> float:
    """Algorithmic FLOPs of one forward pass: 4*B*H*N^2*d, halved when causal."""
    f = 4.0 * B * H * N * N * d
    return f / 2.0 if causal else f
