"""Named synthetic workloads of one sparse-KV decode layer.

Shapes follow the head layouts the pages quote (Llama-3-8B / Qwen3-8B: 32 query
heads, 8 KV heads, head dim 128; a 32B-class GQA model: 64 / 8 / 128) with
context lengths from 4K to 512K tokens and sparse budgets of 256 to 2048
tokens per KV head.  The pages measure on long-context benchmarks with real
models; these seeded synthetic tensors stand in for them.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    L: int
    cs: int
    k: int
    n_q: int
    spec_scale: tuple = ()          # fp32 scale of the noise added to query j (index 0 unused)
    key_bias: str = "none"          # "none" | "hot" | "zipf"
    hot_frac: float = 0.0
    zipf_alpha: float = 0.0
    bias_sigma: float = 3.0
    residency: str = "none"         # "none" | "carry" | "uniform"
    resident_frac: float = 0.0
    seed: int = 1000

    @property
    def C(self) -> int:
        return self.L // self.cs

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def units(self) -> int:
        return self.B * self.Hkv

    @property
    def max_union(self) -> int:
        return min(self.C, self.n_q * self.k)

    @property
    def max_misses(self) -> int:
        return self.units * self.max_union

    def chunk_bytes(self) -> int:
        """Bytes of one chunk of one head, K or V (bf16)."""
        return self.cs * self.d * 2

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


def _spec(n_q: int, per_j) -> tuple:
    return tuple([0.0] + [per_j(j) for j in range(1, n_q)])


TINY = Workload("tiny_b1_ctx4k", B=1, Hq=32, Hkv=8, d=128, L=4096, cs=16, k=16, n_q=2,
                spec_scale=_spec(2, lambda j: 0.3), seed=1001)
LLAMA8B_32K = Workload("llama3_8b_layer_b16_ctx32k", B=16, Hq=32, Hkv=8, d=128, L=32768, cs=16, k=64,
                       n_q=2, spec_scale=_spec(2, lambda j: 0.3), key_bias="hot", hot_frac=0.01,
                       seed=1002)
QWEN8B_128K = Workload("qwen3_8b_layer_b8_ctx128k", B=8, Hq=32, Hkv=8, d=128, L=131072, cs=32, k=64,
                       n_q=2, spec_scale=_spec(2, lambda j: 0.3), residency="carry",
                       resident_frac=0.9, seed=1003)
GQA32B_5Q = Workload("gqa32b_layer_b32_ctx32k_5q", B=32, Hq=64, Hkv=8, d=128, L=32768, cs=16, k=128,
                     n_q=5, spec_scale=_spec(5, lambda j: 0.2 * j), seed=1004)
STRESS_512K = Workload("stress_layer_b4_ctx512k", B=4, Hq=32, Hkv=8, d=128, L=524288, cs=64, k=32,
                       n_q=2, spec_scale=_spec(2, lambda j: 0.3), key_bias="zipf", zipf_alpha=1.1,
                       residency="uniform", resident_frac=0.5, seed=1005)

ALL = (TINY, LLAMA8B_32K, QWEN8B_128K, GQA32B_5Q, STRESS_512K)
BY_NAME = {w.name: w for w in ALL}
