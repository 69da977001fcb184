"""Seeded synthetic inputs for the NVFP4 routed-MoE layer.

This module is the ONLY code that both the CUDA path and the CPU oracle consume.  It draws
activations, router logits and fp32 expert weights from seeded torch generators and holds
none of the layer's arithmetic: no quantization, no routing, no GEMM.  Quantizing the fp32
weights to NVFP4 is done independently on each side (the library's load-time quantizer on the
GPU, the oracle's own quantizer on the CPU) and the two results are compared bit for bit.

Workload shapes follow the five benchmark configurations of the layer ("Batched decode",
"Prefill chunk", ... as listed in the package documentation):

  tiny     T=4,     H=256,  E=16,  k=2,  I=128, shared I=128, seed 0
  decode   T in {1,2,4,8}, H=2048, E=512, k=10, I=512 + shared, seeds 1-4 (near-uniform logits)
  batched  T=64,    same shapes, logits N(0,1) + per-expert bias N(0, 1.5^2), seed 5
  prefill  T=4096,  same shapes, 1% of activation rows x30 (outliers), seed 6
  long     4 independent layers, T=32768, Zipf bias -1.2*ln(rank+1) over a seeded expert
           permutation, seed 7 (layer l uses seed 7*1000 + l)

A generator is a `torch.Generator` on the requested device, seeded from (seed, layer, tag,
group) through SplitMix64, so any single expert can be re-drawn on its own.  The same device
always gives the same numbers; CPU and CUDA give different (equally valid) draws, so a parity
test draws once and hands copies of the same tensors to both sides.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

_MASK64 = (1 << 64) - 1


def _splitmix64(z: int) -> int:
    z = (z + 0x9E3779B97F4A7C15) & _MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


_TAGS = {"x": 1, "logits": 2, "bias": 3, "outliers": 4, "perm": 5, "gate_up": 6, "down": 7, "w": 8, "router": 9}


def _generator(device, seed: int, layer: int, tag: str, group: int = 0) -> torch.Generator:
    h = _splitmix64(seed & _MASK64)
    for v in (layer, _TAGS[tag], group):
        h = _splitmix64(h ^ (v & _MASK64))
    g = torch.Generator(device=device)
    g.manual_seed(h & ((1 << 63) - 1))
    return g


@dataclass(frozen=True)
class Shape:
    """Sizes of one MoE layer. E routed experts, the shared expert is group E."""
    T: int
    H: int
    E: int
    k: int
    I: int
    has_shared: int = 1


@dataclass(frozen=True)
class Workload:
    name: str
    H: int
    E: int
    k: int
    I: int
    Ts: tuple
    seeds: tuple
    layers: int = 1
    logit_bias: str = "none"      # none | normal | zipf
    outlier_frac: float = 0.0
    description: str = field(default="", compare=False)

    def shape(self, T: int | None = None) -> Shape:
        return Shape(T=self.Ts[0] if T is None else T, H=self.H, E=self.E, k=self.k, I=self.I)


WORKLOADS = {
    "tiny": Workload("tiny", 256, 16, 2, 128, (4,), (0,),
                     description="tiny correctness case: T=4, H=256, E=16, k=2, I=128"),
    "decode": Workload("decode", 2048, 512, 10, 512, (1, 2, 4, 8), (1, 2, 3, 4),
                       description="decode/verify sweep: T in {1,2,4,8}, H=2048, E=512, k=10, I=512"),
    "batched": Workload("batched", 2048, 512, 10, 512, (64,), (5,), logit_bias="normal",
                        description="batched decode: T=64, skewed logits (bias N(0,1.5^2))"),
    "prefill": Workload("prefill", 2048, 512, 10, 512, (4096,), (6,), outlier_frac=0.01,
                        description="prefill chunk: T=4096, 1% outlier rows x30"),
    "long": Workload("long", 2048, 512, 10, 512, (32768,), (7,), layers=4, logit_bias="zipf",
                     description="long cold prefill: 4 layers, T=32768, Zipf expert popularity"),
}


def layer_seed(w: Workload, seed: int, layer: int) -> int:
    """Seed of layer `layer` of a stacked workload (layer l of the long prefill uses 7*1000+l)."""
    return seed * 1000 + layer if w.layers > 1 else seed


def activations(T: int, H: int, seed: int, layer: int = 0, outlier_frac: float = 0.0,
                device="cpu") -> torch.Tensor:
    """bf16 [T, H] drawn N(0,1).  With outlier_frac > 0, exactly round(outlier_frac*T) rows,
    chosen by a seeded permutation, are multiplied by 30 before the bf16 rounding."""
    g = _generator(device, seed, layer, "x")
    x = torch.randn(T, H, generator=g, device=device, dtype=torch.float32)
    n_out = int(round(outlier_frac * T))
    if n_out > 0:
        go = _generator(device, seed, layer, "outliers")
        rows = torch.randperm(T, generator=go, device=device)[:n_out]
        x[rows] *= 30.0
    return x.to(torch.bfloat16)


def router_logits(T: int, E: int, seed: int, layer: int = 0, bias: str = "none",
                  device="cpu") -> torch.Tensor:
    """fp32 [T, E] router logits: N(0,1) plus an optional per-expert bias.

    bias="normal": each expert gets a bias drawn N(0, 1.5^2) (skewed popularity).
    bias="zipf":   expert e gets -1.2*ln(rank(e)+1), rank from a seeded permutation.
    """
    g = _generator(device, seed, layer, "logits")
    logits = torch.randn(T, E, generator=g, device=device, dtype=torch.float32)
    if bias == "normal":
        gb = _generator(device, seed, layer, "bias")
        logits += 1.5 * torch.randn(E, generator=gb, device=device, dtype=torch.float32)
    elif bias == "zipf":
        gp = _generator(device, seed, layer, "perm")
        rank = torch.randperm(E, generator=gp, device=device).to(torch.float32)
        logits += -1.2 * torch.log(rank + 1.0)
    elif bias != "none":
        raise ValueError(f"unknown logit bias {bias!r}")
    return logits


def expert_weight(N: int, K: int, seed: int, layer: int, group: int, proj: str,
                  device="cpu", std: float = 0.02) -> torch.Tensor:
    """fp32 [N, K] weights of one group (expert index; E = shared) and one projection
    ('gate_up': N = 2I rows, gate rows first; 'down': N = H rows), drawn N(0, std^2)."""
    g = _generator(device, seed, layer, proj, group)
    return std * torch.randn(N, K, generator=g, device=device, dtype=torch.float32)


def projection_weights(shape: Shape, seed: int, layer: int, proj: str, groups=None,
                       device="cpu") -> torch.Tensor:
    """fp32 [len(groups), N, K] for the given groups (default: all E routed + shared)."""
    if groups is None:
        groups = range(shape.E + (1 if shape.has_shared else 0))
    groups = list(groups)
    N, K = (2 * shape.I, shape.H) if proj == "gate_up" else (shape.H, shape.I)
    out = torch.empty(len(groups), N, K, dtype=torch.float32, device=device)
    for i, grp in enumerate(groups):
        out[i] = expert_weight(N, K, seed, layer, grp, proj, device=device)
    return out


def router_weights(shape: Shape, seed: int, layer: int = 0, device="cpu", std: float = 0.02) -> torch.Tensor:
    """fp32 [1, E, H] router weights drawn N(0, std^2) (one projection of E rows; with x ~ N(0,1)
    and H = 2048 the logits come out near N(0, 0.8))."""
    g = _generator(device, seed, layer, "router")
    return std * torch.randn(1, shape.E, shape.H, generator=g, device=device, dtype=torch.float32)


def random_floats(n: int, seed: int, device="cpu", scale: float = 1.0) -> torch.Tensor:
    """n fp32 values N(0, scale^2) for format and encoder sweeps."""
    g = _generator(device, seed, 0, "w", n)
    return scale * torch.randn(n, generator=g, device=device, dtype=torch.float32)


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


__all__ = ["Shape", "Workload", "WORKLOADS", "layer_seed", "activations", "router_logits",
           "expert_weight", "projection_weights", "router_weights", "random_floats", "ceil_div", "math"]
