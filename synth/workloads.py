"""The synthetic workloads of the int4 MoE block.

Each workload fixes the block's sizes, the tokens per step, the number of
stacked layers (each with its own weights) and the optional Zipf skew added
to the router logits.  ``wid`` is the integer that enters the generator's
stream keys, so every workload draws its own weights.
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class Workload:
    wid: int
    name: str
    E: int          # routed experts
    k: int          # experts per token
    H: int          # hidden size
    I: int          # routed-expert intermediate size
    Is: int         # shared-expert intermediate size
    G: int          # quantisation group along the input dimension
    T: int          # tokens per step
    layers: int     # stacked MoE layers, each with its own weights
    zipf_s: float | None = None  # Zipf exponent of the router prior (None: no prior)

    @property
    def shape(self):
        from . import Shape
        return Shape(self.E, self.k, self.H, self.I, self.Is, self.G)

    @property
    def expert_bytes(self) -> int:
        """Bytes of one routed expert: packed int4 codes plus bf16 scale and bias."""
        packed = 3 * self.I * self.H // 2
        sb = 3 * self.I * self.H // self.G * 4
        return packed + sb

    @property
    def shared_bytes(self) -> int:
        return 3 * self.Is * self.H // 2 + 3 * self.Is * self.H // self.G * 4

    @property
    def router_bytes(self) -> int:
        return self.E * self.H * 2 + self.H * 2 + (self.E * 4 if self.zipf_s is not None else 0)


WORKLOADS = {
    0: Workload(0, "tiny-h256-e16-k2", E=16, k=2, H=256, I=64, Is=64, G=32, T=4, layers=1),
    1: Workload(1, "35b-decode-e256-k8-40layers", E=256, k=8, H=2048, I=512, Is=512, G=64,
                T=1, layers=40),
    2: Workload(2, "80b-decode-e512-k10-48layers", E=512, k=10, H=2048, I=512, Is=512, G=64,
                T=1, layers=48),
    3: Workload(3, "80b-batch64-zipf1.1", E=512, k=10, H=2048, I=512, Is=512, G=64, T=64,
                layers=1, zipf_s=1.1),
    4: Workload(4, "80b-prefill4096-zipf0.8", E=512, k=10, H=2048, I=512, Is=512, G=64,
                T=4096, layers=1, zipf_s=0.8),
}
