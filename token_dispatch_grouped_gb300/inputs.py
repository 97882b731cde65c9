"""Seeded synthetic inputs for the dropless MoE layer.

This module only draws random numbers and names the workloads; it holds none of
the layer's arithmetic. Both the CUDA path (tests, bench) and the CPU oracle are
fed from here, so the two sides always see the same bytes.

Workloads (shapes from the layer configurations the method is evaluated on):

    tiny     T=256,    d=128,  E=8,   K=2, h=256
    mixtral  T=4096,   d=4096, E=8,   K=2, h=14336
    fine     T=16384,  d=2048, E=64,  K=6, h=1408
    skew     T=32768,  d=2048, E=128, K=8, h=768   (Zipf(1.2) loads via a logit bias)
    long     T=131072, d=4096, E=16,  K=4, h=2048

Non-gated (SiLU) two-layer experts with h = 4d, T = batch x sequence length,
on the MoEBlaze configurations whose sizes survive in its text:

    moeblaze_conf1  T=65536 (32x2048), d=512,  E=4,  K=1, h=2048
    moeblaze_conf3  T=65536 (32x2048), d=1024, E=16, K=4, h=4096
    moeblaze_conf4  T=32768 (32x1024), d=2048, E=16, K=4, h=8192
    moeblaze_conf7  T=8192  (16x512),  d=2048, E=8,  K=4, h=8192

Recipe: one torch CPU generator per tensor, seeded from (seed, tensor name).
x, dO ~ N(0, 1); W_g, W1, W3 ~ N(0, 1/d); W2 ~ N(0, 1/h). Activations and expert
weights are rounded once to bf16 (round-to-nearest-even); the router weight
W_g stays fp32. The skew workload adds a stored per-expert logit bias.
"""
from __future__ import annotations

import json
import math
import os
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Shape:
    T: int
    d: int
    E: int
    K: int
    h: int
    expert: str = "swiglu"  # or the non-gated "silu" / "relu" (no W3)

    @property
    def gated(self) -> bool:
        return self.expert == "swiglu"

    @property
    def TK(self) -> int:
        return self.T * self.K


WORKLOADS = {
    "tiny": Shape(256, 128, 8, 2, 256),
    "mixtral": Shape(4096, 4096, 8, 2, 14336),
    "fine": Shape(16384, 2048, 64, 6, 1408),
    "skew": Shape(32768, 2048, 128, 8, 768),
    "long": Shape(131072, 4096, 16, 4, 2048),
    # Profiling-size case: the Mixtral-shaped experts (1024 rows each, d=4096,
    # h=14336) with only 2 experts, so an ncu capture holds ~2 GB on the device.
    "mixtral_e2": Shape(1024, 4096, 2, 2, 14336),
    # Profiling-size case for the memory-bound kernels: Mixtral's routing shape
    # (d=4096, E=8, K=2) at T=16384, so x (128 MiB) exceeds L2, with narrow
    # experts (h=1024) to keep the whole step near 1.3 GB on the device.
    "mixtral_t16k_narrow": Shape(16384, 4096, 8, 2, 1024),
    "moeblaze_conf1": Shape(65536, 512, 4, 1, 2048, "silu"),
    "moeblaze_conf3": Shape(65536, 1024, 16, 4, 4096, "silu"),
    "moeblaze_conf4": Shape(32768, 2048, 16, 4, 8192, "silu"),
    "moeblaze_conf7": Shape(8192, 2048, 8, 4, 8192, "silu"),
}

# Fixed per-tensor stream ids, so adding a tensor never shifts another one.
_STREAM = {"x": 1, "Wg": 2, "W1": 3, "W3": 4, "W2": 5, "dO": 6}

_HERE = os.path.dirname(os.path.abspath(__file__))
SKEW_BIAS_FILE = os.path.join(_HERE, "data", "skew_bias_e128.json")


def _gen(seed: int, name: str) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed * 1000003 + _STREAM[name])
    return g


def randn(shape, seed: int, name: str, std: float = 1.0) -> torch.Tensor:
    """fp32 N(0, std^2) draw on the CPU from the tensor's own stream."""
    t = torch.randn(*shape, generator=_gen(seed, name), dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t


def skew_bias(E: int) -> torch.Tensor | None:
    """Stored router logit bias of the skewed workload (fp32 [E]), if present."""
    if not os.path.exists(SKEW_BIAS_FILE):
        return None
    with open(SKEW_BIAS_FILE) as f:
        blob = json.load(f)
    if blob["E"] != E:
        return None
    return torch.tensor(blob["bias"], dtype=torch.float32)


def make_layer_inputs(s: Shape, seed: int = 0, with_bias: bool = False,
                      parts=("x", "Wg", "W1", "W3", "W2", "dO")) -> dict:
    """CPU tensors of one layer step: x, dO bf16 [T,d]; W_g fp32 [E,d];
    W1, W3 bf16 [E,h,d] (W3 None for non-gated experts); W2 bf16 [E,d,h];
    optional bias fp32 [E]."""
    out = {}
    if not s.gated:
        parts = tuple(q for q in parts if q != "W3")
        out["W3"] = None
    if "x" in parts:
        out["x"] = randn((s.T, s.d), seed, "x").to(torch.bfloat16)
    if "Wg" in parts:
        out["Wg"] = randn((s.E, s.d), seed, "Wg", 1.0 / math.sqrt(s.d))
    if "W1" in parts:
        out["W1"] = randn((s.E, s.h, s.d), seed, "W1", 1.0 / math.sqrt(s.d)).to(torch.bfloat16)
    if "W3" in parts:
        out["W3"] = randn((s.E, s.h, s.d), seed, "W3", 1.0 / math.sqrt(s.d)).to(torch.bfloat16)
    if "W2" in parts:
        out["W2"] = randn((s.E, s.d, s.h), seed, "W2", 1.0 / math.sqrt(s.h)).to(torch.bfloat16)
    if "dO" in parts:
        out["dO"] = randn((s.T, s.d), seed, "dO").to(torch.bfloat16)
    out["bias"] = skew_bias(s.E) if with_bias else None
    return out


def random_ids(T: int, E: int, K: int, seed: int, skew: float = 0.0) -> torch.Tensor:
    """Random valid top-K expert ids [T,K] int32 (K distinct experts per token).

    skew > 0 draws experts with probability proportional to (rank+1)^-skew, so
    loads are uneven and high-rank experts can be empty."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    if skew > 0:
        p = torch.arange(1, E + 1, dtype=torch.float64).pow(-skew)
        p = p / p.sum()
        ids = torch.multinomial(p.expand(T, E).float(), K, replacement=False, generator=g)
    else:
        ids = torch.rand(T, E, generator=g).argsort(dim=1)[:, :K]
    return ids.to(torch.int32).contiguous()


def random_ids_gumbel(T: int, E: int, K: int, seed: int, skew: float = 0.0) -> torch.Tensor:
    """Random valid top-K expert ids [T,K] int32 for large T: K distinct experts
    per token drawn without replacement with probability proportional to
    (rank+1)^-skew (uniform for skew = 0), by the Gumbel-top-K construction
    (the K largest of log p_e + Gumbel noise)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    logp = -skew * torch.log(torch.arange(1, E + 1, dtype=torch.float32))
    u = torch.rand(T, E, generator=g).clamp_(min=1e-12)
    keys = logp - torch.log(-torch.log(u))
    return keys.topk(K, dim=1).indices.to(torch.int32).contiguous()


def random_weights(T: int, K: int, seed: int) -> torch.Tensor:
    """Positive routing weights [T,K] fp32, uniform on [0.05, 1.05)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed + 7)
    return (torch.rand(T, K, generator=g) + 0.05).contiguous()
