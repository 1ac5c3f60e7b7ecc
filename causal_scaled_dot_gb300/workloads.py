"""The named attention workloads this library is measured and checked on.

All are causal, bf16 Q/K/V drawn i.i.d. N(0, sigma^2) by ``inputs.qkv_bf16``
with the listed seed, scale = 1/sqrt(D), fp32 LSE output.

* ``small_b1_h2_s256_d64``       -- a small case the CPU oracle finishes in well
  under a second (parity, smoke).
* ``profile_b4_h16_s4096_d128``  -- the profiling shape of the ai-manual.ru
  article (section 1: B=4, H=16, S=4096, D=128).  The headline workload.
* ``llama7b_b1_h32_s2048_d128``  -- one layer of a 7B LLaMA at batch 1 and
  sequence 2048 (the ainews.cool per-operator latency table), values x0.5.
  No weights: random activations of that shape.
* ``long_b2_h32_s8192_d128``     -- a long-context case, S=8192 (the ai-manual.ru
  article's S=8192 memory example, section 1).
* ``gqa_b2_hq32_hkv8_s4096_d128`` -- grouped-query attention, 4 query heads per
  key/value head (the GQA row of the ainews.cool strategy table).
"""
from __future__ import annotations

import math
from dataclasses import dataclass


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    S: int
    D: int
    sigma: float
    seed: int
    causal: bool = True

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def flops(self) -> float:
        """4*B*Hq*S^2*D, halved for causal (exactly S^2/2 key-query pairs)."""
        f = 4.0 * self.B * self.Hq * self.S * self.S * self.D
        return f / 2.0 if self.causal else f

    @property
    def io_bytes(self) -> int:
        """Algorithmic HBM bytes: read Q, K, V once, write O (bf16) and LSE (fp32)."""
        q = self.B * self.Hq * self.S * self.D * 2
        kv = 2 * self.B * self.Hkv * self.S * self.D * 2
        o = q
        lse = self.B * self.Hq * self.S * 4
        return q + kv + o + lse

    @property
    def shape_dict(self) -> dict:
        return {"B": self.B, "Hq": self.Hq, "Hkv": self.Hkv, "S": self.S, "D": self.D}


WORKLOADS = [
    Workload("small_b1_h2_s256_d64", 1, 2, 2, 256, 64, 1.0, 1),
    Workload("profile_b4_h16_s4096_d128", 4, 16, 16, 4096, 128, 1.0, 2),
    Workload("llama7b_b1_h32_s2048_d128", 1, 32, 32, 2048, 128, 0.5, 3),
    Workload("long_b2_h32_s8192_d128", 2, 32, 32, 8192, 128, 1.0, 4),
    Workload("gqa_b2_hq32_hkv8_s4096_d128", 2, 32, 8, 4096, 128, 1.0, 5),
]
BY_NAME = {w.name: w for w in WORKLOADS}
HEADLINE = BY_NAME["profile_b4_h16_s4096_d128"]
SMALL = BY_NAME["small_b1_h2_s256_d64"]
