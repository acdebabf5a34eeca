"""Seeded synthetic inputs for the MoE stage1 + combine path.

This module holds no arithmetic of the method itself: it only draws random
tensors with the shapes and distributions of the workloads (token activations,
router logits with an optional Zipf popularity bias, expert weights) and names
the workload configurations.  Both the CUDA path and the CPU oracle are fed from
here; neither side's arithmetic lives here.

Workloads (hidden size H, experts E in G logical groups, top-k, GEMM1 width N):

* ``tiny``: T=128, H=256, E=8, G=2, k=2, N=512, uniform routing.
* ``t2048_uniform``: T=2048, H=7168, E=256, G=8, k=8, N=4096, uniform routing.
* ``t8192_zipf1.2``: as above with T=8192 and Zipf(s=1.2) expert popularity.
* ``bw_t{2048,4096,8192,16384}``: dispatch + combine bandwidth sweep with the
  identity expert (no GEMM), uniform routing.
* ``stage1_t16384_zipf1.0``: fused stage1 workload, T=16384, Zipf(s=1.0).
* ``profile_t8192_e32``: the T=8192 shapes with 32 experts, small enough for
  multi-pass profiler captures.

The shapes (hidden 7168, 256 routed experts, top-8, two 2048-wide projections)
are those of the DeepSeek-V3-class models the mori stage1 page benchmarks
(its "Where we stand" tables name V4.1-Flash and V4-Pro without giving shapes).

Random streams: one base seed; tensor ``i`` (x=0, logits=1, permutation=2,
weights=3) uses ``seed * 16 + i`` so that each tensor is reproducible on its own.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace
from typing import Optional

import torch

STREAM_X, STREAM_LOGITS, STREAM_PERM, STREAM_W = 0, 1, 2, 3


@dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int
    H: int
    E: int
    G: int
    k: int
    N: int
    zipf: Optional[float] = None  # None: uniform logits
    gemm: bool = True             # False: identity expert (bandwidth sweep)
    seed: int = 0

    def with_tokens(self, T: int) -> "MoEConfig":
        return replace(self, T=T, name=f"{self.name}_T{T}")


CONFIGS = {
    "tiny": MoEConfig("tiny", T=128, H=256, E=8, G=2, k=2, N=512),
    "t2048_uniform": MoEConfig("t2048_uniform", T=2048, H=7168, E=256, G=8, k=8, N=4096),
    "t8192_zipf1.2": MoEConfig("t8192_zipf1.2", T=8192, H=7168, E=256, G=8, k=8, N=4096, zipf=1.2),
    "bw_t2048": MoEConfig("bw_t2048", T=2048, H=7168, E=256, G=8, k=8, N=7168, gemm=False),
    "bw_t4096": MoEConfig("bw_t4096", T=4096, H=7168, E=256, G=8, k=8, N=7168, gemm=False),
    "bw_t8192": MoEConfig("bw_t8192", T=8192, H=7168, E=256, G=8, k=8, N=7168, gemm=False),
    "bw_t16384": MoEConfig("bw_t16384", T=16384, H=7168, E=256, G=8, k=8, N=7168, gemm=False),
    "stage1_t16384_zipf1.0": MoEConfig("stage1_t16384_zipf1.0", T=16384, H=7168, E=256, G=8, k=8,
                                       N=4096, zipf=1.0),
    # profiler-sized: the T=8192 shapes with 32 experts (weights 0.5 GB instead of 7.5 GB)
    "profile_t8192_e32": MoEConfig("profile_t8192_e32", T=8192, H=7168, E=32, G=8, k=8, N=4096, zipf=1.2),
}


def _gen(seed: int, stream: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 16 + stream)
    return g


def make_x(T: int, H: int, seed: int = 0, device="cpu") -> torch.Tensor:
    """Token activations x ~ N(0, 1), drawn in fp32 and stored as bf16 [T, H]."""
    g = _gen(seed, STREAM_X, device)
    return torch.randn(T, H, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def zipf_bias(E: int, s: float, seed: int = 0) -> torch.Tensor:
    """Additive logit bias giving expert popularity a Zipf(s) shape over a seeded
    permutation of the experts: the expert of popularity rank r (1-based) gets
    ``-s * ln(r)``, the log of the Zipf pmf with its constant dropped."""
    g = _gen(seed, STREAM_PERM, "cpu")
    perm = torch.randperm(E, generator=g)
    bias = torch.empty(E, dtype=torch.float32)
    ranks = torch.arange(1, E + 1, dtype=torch.float64)
    bias[perm] = (-s * torch.log(ranks)).to(torch.float32)
    return bias


def make_logits(T: int, E: int, zipf: Optional[float] = None, seed: int = 0,
                device="cpu") -> torch.Tensor:
    """Router logits ~ N(0, 1) fp32 [T, E], plus the Zipf bias when ``zipf`` is set."""
    g = _gen(seed, STREAM_LOGITS, device)
    logits = torch.randn(T, E, generator=g, device=device, dtype=torch.float32)
    if zipf is not None:
        logits += zipf_bias(E, zipf, seed).to(device)
    return logits


def make_weights(E: int, N: int, H: int, seed: int = 0, device="cpu") -> torch.Tensor:
    """Expert GEMM1 weights W ~ N(0, 1/H), bf16 [E, N, H] (row n of expert e is
    the K-contiguous column of the projection).  Drawn one expert at a time so
    the fp32 temporary stays one expert large."""
    g = _gen(seed, STREAM_W, device)
    out = torch.empty(E, N, H, device=device, dtype=torch.bfloat16)
    std = 1.0 / math.sqrt(H)
    for e in range(E):
        out[e] = (torch.randn(N, H, generator=g, device=device, dtype=torch.float32) * std).to(
            torch.bfloat16)
    return out


def bf16_bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (for the CPU oracle)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")
