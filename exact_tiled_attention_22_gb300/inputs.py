"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds no attention arithmetic: it only draws N(0, 1) tensors from
a seeded CPU generator and rounds them (round-to-nearest-even) to fp16 or
bf16.  Both the GPU path and the fp64 oracle consume exactly these rounded
values.

Workloads.  The five shapes below are the attention workloads this library is
measured and checked on: a tiny single-tile case, an encoder-style batch of
short sequences, a GPT training shape, a long-context shape and a very long
small-batch shape.  The very long shape multiplies Q and K by 2 before
rounding (a power of two, so the rounding is unaffected) to sharpen the
softmax.  Seeds: 1000 + workload index; Q, K, V, dO draw from sub-seeds
4*seed + {0, 1, 2, 3}.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str          # "fp16" | "bf16"
    causal: bool
    scale: float
    seed: int
    qk_mult: float = 1.0
    note: str = field(default="", compare=False)

    @property
    def torch_dtype(self):
        return torch_dtype(self.dtype)

    def flops_fwd(self) -> float:
        """4*B*H*N^2*d, halved when causal (the conventional count)."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f

    def flops_bwd(self) -> float:
        return 2.5 * self.flops_fwd()

    def as_dict(self) -> dict:
        return {"workload": self.name, "B": self.B, "H": self.H, "N": self.N,
                "d": self.d, "dtype": self.dtype, "causal": self.causal,
                "scale": self.scale, "seed": self.seed, "qk_mult": self.qk_mult}


WORKLOADS = {
    w.name: w for w in [
        Workload("tiny", 1, 1, 128, 64, "fp16", False, 1 / 8, 1000),
        Workload("encoder", 16, 12, 512, 64, "fp16", False, 1 / 8, 1001),
        Workload("gpt", 4, 16, 2048, 128, "bf16", True, 1 / math.sqrt(128), 1002),
        Workload("long", 2, 16, 8192, 128, "bf16", True, 1 / math.sqrt(128), 1003),
        Workload("very_long", 1, 32, 32768, 128, "bf16", True,
                 1 / math.sqrt(128), 1004, qk_mult=2.0),
    ]
}


def torch_dtype(name: str):
    return {"fp16": torch.float16, "bf16": torch.bfloat16}[name]


def randn(shape, seed: int, dtype, mult: float = 1.0) -> torch.Tensor:
    """N(0,1) in fp32 from a seeded CPU generator, times `mult`, rounded RNE."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if mult != 1.0:
        x = x * mult
    return x.to(dtype)


def make_inputs(B: int, N: int, H: int, d: int, dtype="bf16", seed: int = 0,
                qk_mult: float = 1.0) -> dict:
    """q, k, v, do as contiguous CPU tensors of shape [B, N, H, d]."""
    dt = torch_dtype(dtype) if isinstance(dtype, str) else dtype
    shape = (B, N, H, d)
    return {
        "q": randn(shape, 4 * seed + 0, dt, qk_mult),
        "k": randn(shape, 4 * seed + 1, dt, qk_mult),
        "v": randn(shape, 4 * seed + 2, dt),
        "do": randn(shape, 4 * seed + 3, dt),
    }


def make_block_mask(H: int, N: int, pattern: str = "random", density: float = 0.5,
                    seed: int = 0, width: int = 1) -> torch.Tensor:
    """uint8 [H, nb, nb] mask over 128 x 128 blocks (nb = ceil(N / 128)),
    1 = block kept.  Patterns:
      "random": each block kept independently with probability `density`
                (seeded CPU generator, one draw per head and block);
      "local_global": blocks within `width` of the diagonal, plus the first
                block row and column (a banded mask with global tokens);
      "ones": every block kept."""
    nb = (N + 127) // 128
    if pattern == "random":
        g = torch.Generator(device="cpu")
        g.manual_seed(int(seed))
        m = torch.rand(H, nb, nb, generator=g) < density
    elif pattern == "local_global":
        i = torch.arange(nb)
        band = (i[:, None] - i[None, :]).abs() <= width
        band[0, :] = True
        band[:, 0] = True
        m = band.expand(H, nb, nb)
    elif pattern == "ones":
        m = torch.ones(H, nb, nb, dtype=torch.bool)
    else:
        raise ValueError(pattern)
    return m.to(torch.uint8).contiguous()


def workload_inputs(w: Workload) -> dict:
    return make_inputs(w.B, w.N, w.H, w.d, w.dtype, w.seed, w.qk_mult)


@dataclass(frozen=True)
class DecodeWorkload:
    """Decoding: Nq new query rows (the last Nq positions) against a cache of
    Nk keys and values."""
    name: str
    B: int
    H: int
    Nq: int
    Nk: int
    d: int
    dtype: str
    causal: bool
    scale: float
    seed: int

    def kv_bytes(self) -> int:
        """K and V read once: the dominant, algorithmic HBM traffic."""
        return 2 * self.B * self.Nk * self.H * self.d * 2

    def flops(self) -> float:
        return 4.0 * self.B * self.H * self.Nq * self.Nk * self.d

    def as_dict(self) -> dict:
        return {"workload": self.name, "B": self.B, "H": self.H, "Nq": self.Nq, "Nk": self.Nk,
                "d": self.d, "dtype": self.dtype, "causal": self.causal, "scale": self.scale,
                "seed": self.seed}


# Serving-style decode shapes (seeds 1100 + index): one new token per
# sequence against a 32K cache, 16 draft tokens per sequence (speculative
# decoding) against the same cache, and a smaller cache for profiling.
DECODE_WORKLOADS = {
    w.name: w for w in [
        DecodeWorkload("decode_32k", 8, 32, 1, 32768, 128, "bf16", True, 1 / math.sqrt(128), 1100),
        DecodeWorkload("decode_32k_q16", 8, 32, 16, 32768, 128, "bf16", True, 1 / math.sqrt(128), 1101),
        # a smaller cache (537 MB, still larger than L2) for detailed profiling
        DecodeWorkload("decode_16k_small", 2, 32, 1, 16384, 128, "bf16", True, 1 / math.sqrt(128), 1102),
    ]
}


def make_decode_inputs(w: DecodeWorkload) -> dict:
    """q [B, Nq, H, d] and the cache k, v [B, Nk, H, d] as CPU tensors."""
    dt = torch_dtype(w.dtype)
    return {
        "q": randn((w.B, w.Nq, w.H, w.d), 4 * w.seed + 0, dt),
        "k": randn((w.B, w.Nk, w.H, w.d), 4 * w.seed + 1, dt),
        "v": randn((w.B, w.Nk, w.H, w.d), 4 * w.seed + 2, dt),
    }
