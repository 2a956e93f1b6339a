"""Seeded synthetic inputs for the routed-MoE FFN layer.

This module only draws random tensors.  It holds none of the layer's
arithmetic (no routing, no permutation, no quantisation, no FFN), so both the
CUDA path and the fp64 oracle can consume what it produces without sharing any
of the method with one another.

Shapes and laws follow the workloads of "Systems engineering playbook: Qwen 3.5
MoE on Ironwood TPU" (section "The Architectural Constraints That Break Naive
Sharding": 512 experts of intermediate 1024, top_k=10, one always-on shared
expert, hidden size 4096) at the decode/prefill regimes the roofline section
of that report describes.

Storage convention (identical for both sides):
  x         [T, D]          activations (fp32 for the fp32 layer, else bf16)
  w_router  [E, D]          router weight, one row per expert (K-major)
  b_router  [E]   fp32      router bias (zeros unless the load is Zipf-skewed)
  w_gate    [E+1, I, D]     gate projection, one [I, D] matrix per group
  w_up      [E+1, I, D]     up projection
  w_down    [E+1, D, I]     down projection
Group E (the last) is the always-on shared expert.  Each matrix is stored
[out_features, in_features], i.e. reduction dimension innermost.
For the FP8 layer the expert weights are returned in fp32; turning them into
E4M3 codes with 128x128 block scales is the layer's job (each side does it
itself).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

# Tensor ids feeding each torch.Generator: seed * 1000 + id.
_ID_X, _ID_WR, _ID_BR, _ID_WG, _ID_WU, _ID_WD = 1, 2, 3, 4, 5, 6


@dataclasses.dataclass(frozen=True)
class LayerShape:
    name: str
    T: int          # tokens
    D: int          # hidden size
    E: int          # routed experts
    I: int          # expert (and shared expert) intermediate size
    top_k: int
    dtype: str      # "f32" | "bf16" | "fp8"
    zipf_s: Optional[float] = None   # router-bias skew; None = no bias

    @property
    def has_bias(self) -> bool:
        return self.zipf_s is not None

    def with_tokens(self, T: int) -> "LayerShape":
        return dataclasses.replace(self, T=T)


# The five workloads (tiny fp32, decode, batched decode, prefill, FP8 prefill).
TINY_F32 = LayerShape("tiny_f32_T64_D256_E16_I128_k2", 64, 256, 16, 128, 2, "f32")
DECODE_BF16 = LayerShape("decode_bf16_T128_D4096_E512_I1024_k10", 128, 4096, 512, 1024, 10, "bf16")
BATCHED_DECODE_BF16 = LayerShape("batched_decode_bf16_T1024_zipf1.0", 1024, 4096, 512, 1024, 10, "bf16", 1.0)
PREFILL_BF16 = LayerShape("prefill_bf16_T8192_zipf1.2", 8192, 4096, 512, 1024, 10, "bf16", 1.2)
PREFILL_FP8 = LayerShape("prefill_fp8_T16384_zipf1.2", 16384, 4096, 512, 1024, 10, "fp8", 1.2)

WORKLOADS = {s.name: s for s in (TINY_F32, DECODE_BF16, BATCHED_DECODE_BF16, PREFILL_BF16, PREFILL_FP8)}

# FP8 weights at the decode shapes: the memory-bound regime streams half the
# bytes (E4M3 codes + 128x128 block scales instead of bf16).
DECODE_FP8 = LayerShape("decode_fp8_T128_D4096_E512_I1024_k10", 128, 4096, 512, 1024, 10, "fp8")
BATCHED_DECODE_FP8 = LayerShape("batched_decode_fp8_T1024_zipf1.0", 1024, 4096, 512, 1024, 10, "fp8", 1.0)
EXTRA_WORKLOADS = {s.name: s for s in (DECODE_FP8, BATCHED_DECODE_FP8)}

# Reduced shapes for parity tests: several tiles in every dimension plus a
# ragged tail, small enough for the oracle to finish in seconds.
SMALL_BF16 = LayerShape("small_bf16_T300_D512_E32_I256_k4_zipf1.2", 300, 512, 32, 256, 4, "bf16", 1.2)
SMALL_FP8 = LayerShape("small_fp8_T300_D512_E32_I256_k4_zipf1.2", 300, 512, 32, 256, 4, "fp8", 1.2)
SMALL_F32 = LayerShape("small_f32_T77_D256_E16_I128_k3", 77, 256, 16, 128, 3, "f32")


def _gen(seed: int, tensor_id: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000 + tensor_id)
    return g


def _normal(shape, std: float, g: torch.Generator, device, out_dtype, chunk_dim0: int = 0):
    """N(0, std^2) drawn in fp32, stored as out_dtype; chunked over dim 0."""
    if chunk_dim0 <= 0 or shape[0] <= chunk_dim0:
        t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        t.mul_(std)
        return t.to(out_dtype)
    out = torch.empty(shape, device=device, dtype=out_dtype)
    for s in range(0, shape[0], chunk_dim0):
        e = min(shape[0], s + chunk_dim0)
        t = torch.randn((e - s,) + tuple(shape[1:]), generator=g, device=device, dtype=torch.float32)
        t.mul_(std)
        out[s:e].copy_(t)
        del t
    return out


def zipf_router_bias(E: int, s: float, g: torch.Generator, device) -> torch.Tensor:
    """Router bias b[e] = ln p_{r(e)}, p_i = i^-s / H_{E,s}, r a random ranking.

    This is the input recipe for skewed expert load (a random expert gets rank
    1, the most popular); it shifts the logits, so it also shapes the weights.
    """
    ranks = torch.randperm(E, generator=g, device=device).to(torch.float64) + 1.0
    h = sum(i ** -s for i in range(1, E + 1))
    return (-s * torch.log(ranks) - math.log(h)).to(torch.float32)


def make_inputs(shape: LayerShape, seed: int = 0, device="cpu", T: Optional[int] = None,
                weights: bool = True) -> dict:
    """All tensors of one workload, drawn from one integer seed.

    T overrides the token count (the weights do not depend on it).
    weights=False skips the expert weights (x / router only).
    """
    T = shape.T if T is None else T
    D, E, I = shape.D, shape.E, shape.I
    act_dtype = torch.float32 if shape.dtype == "f32" else torch.bfloat16
    wexp_dtype = {"f32": torch.float32, "bf16": torch.bfloat16, "fp8": torch.float32}[shape.dtype]
    out = {}
    out["x"] = _normal((T, D), 1.0, _gen(seed, _ID_X, device), device, act_dtype)
    out["w_router"] = _normal((E, D), D ** -0.5, _gen(seed, _ID_WR, device), device, act_dtype)
    if shape.has_bias:
        out["b_router"] = zipf_router_bias(E, shape.zipf_s, _gen(seed, _ID_BR, device), device)
    else:
        out["b_router"] = torch.zeros(E, dtype=torch.float32, device=device)
    if weights:
        chunk = max(1, (1 << 27) // (I * D))
        out["w_gate"] = _normal((E + 1, I, D), D ** -0.5, _gen(seed, _ID_WG, device), device, wexp_dtype, chunk)
        out["w_up"] = _normal((E + 1, I, D), D ** -0.5, _gen(seed, _ID_WU, device), device, wexp_dtype, chunk)
        out["w_down"] = _normal((E + 1, D, I), I ** -0.5, _gen(seed, _ID_WD, device), device, wexp_dtype, chunk)
    return out


def tie_logits(T: int, E: int, seed: int = 0, device="cpu", levels: int = 4) -> torch.Tensor:
    """fp32 logits with many exact ties: values drawn from a handful of levels."""
    g = _gen(seed, 7, device)
    lv = torch.randint(0, levels, (T, E), generator=g, device=device).to(torch.float32)
    return lv * 0.25 - 0.5
