"""Named workloads for the top-k routed MoE FFN forward pass.

Each workload fixes the layer shape (T tokens, hidden H, N experts, top-k, SwiGLU
width F), the capacity factor (None = no per-expert limit), the storage dtype, the
seed of the synthetic inputs and whether a per-expert router bias is drawn.

The five named workloads follow the shapes the pages discuss: a tiny fp32 layer, a
16-expert bf16 layer, a Mixtral-shaped 8-expert layer, a fine-grained 64-expert layer
with hot experts forced by a router bias (2kiu.com/news/2885792, section 5.2, cools
hot experts with a per-expert logit offset; the same mechanism is used here to make
them hot), and a decode-size 100-expert top-2 layer, i.e. 2% of the experts active
(the devpress.csdn.net MoE page, section 3.2, puts the active share of a large
model's parameters at 2%).

This module holds data only: no part of the layer's arithmetic lives here.
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Optional


@dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int                      # tokens in the batch (batch * seq_len, flattened)
    H: int                      # hidden size
    N: int                      # number of routed experts
    k: int                      # experts per token
    F: int                      # SwiGLU inner width of one expert
    capacity_factor: Optional[float]  # None: no capacity limit
    dtype: str                  # "f32" or "bf16": storage type of x, weights, output
    seed: int = 0
    zipf_bias: bool = False     # draw a per-expert router bias that makes hot experts

    def with_(self, **kw) -> "MoEConfig":
        return replace(self, **kw)

    @property
    def slots(self) -> int:
        return self.T * self.k


TINY_F32 = MoEConfig("tiny_f32_t64_h128_n8_k2_f256", 64, 128, 8, 2, 256, None, "f32")
BF16_T4096 = MoEConfig("bf16_t4096_h1024_n16_k2_f2816_cf1.25", 4096, 1024, 16, 2, 2816,
                       1.25, "bf16")
MIXTRAL_T8192 = MoEConfig("mixtral_t8192_h4096_n8_k2_f14336_cf1.5", 8192, 4096, 8, 2,
                          14336, 1.5, "bf16")
FINEGRAINED_T16384 = MoEConfig("finegrained_t16384_h2048_n64_k2_f1408_cf1.2_zipf", 16384,
                               2048, 64, 2, 1408, 1.2, "bf16", zipf_bias=True)
DECODE_T64 = MoEConfig("decode_t64_h4096_n100_k2_f2048", 64, 4096, 100, 2, 2048, None,
                       "bf16")

NAMED = [TINY_F32, BF16_T4096, MIXTRAL_T8192, FINEGRAINED_T16384, DECODE_T64]

# A profiling case with the Mixtral-shaped layer's per-expert geometry (about 2048 rows
# per expert, H=4096, F=14336) but two experts: 0.7 GB of weights instead of 2.8 GB,
# small enough for multi-pass profiler captures.
MIXTRAL_GEOMETRY_T2048 = MoEConfig("mixtral_geometry_t2048_h4096_n2_k2_f14336_cf1.5", 2048,
                                   4096, 2, 2, 14336, 1.5, "bf16")

BY_NAME = {c.name: c for c in NAMED + [MIXTRAL_GEOMETRY_T2048]}

# Short aliases used on command lines.
ALIASES = {
    "tiny": TINY_F32.name,
    "bf16": BF16_T4096.name,
    "mixtral": MIXTRAL_T8192.name,
    "finegrained": FINEGRAINED_T16384.name,
    "decode": DECODE_T64.name,
    "mixtral_geometry": MIXTRAL_GEOMETRY_T2048.name,
}


def get(name: str) -> MoEConfig:
    return BY_NAME[ALIASES.get(name, name)]
