"""Seeded synthetic inputs for the MoE routing path.

This module is the only code shared by the CUDA path's tests/benchmarks and the
CPU oracle. It draws random numbers and nothing else: no scoring, selection,
normalisation or sorting happens here.

Every generator uses a CPU ``torch.Generator`` with a fixed seed, so the same
bytes reach the GPU and the oracle. Seeds: logits 0, gradients 1, bias 2,
expert offsets / permutation 3.

The shapes and value distributions follow the workloads the router pages
measure on (TransformerEngine PR 3012, "Performance": T=8192, E in {512, 2304},
fp32; FlyDSL PR 582, "Test Result": DeepSeek-R1 E=256 topk=8 bf16 decode;
aiter PR 3828, "Results": Kimi-K2.5 NE=385 TOPK=9). No public dataset is
involved; these stand in for real router logits.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import torch

SEED_LOGITS = 0
SEED_GRAD = 1
SEED_BIAS = 2
SEED_OFFSETS = 3

SOFTMAX = 0
SIGMOID = 1
F32 = 0
BF16 = 1


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def normal(shape, sigma: float = 1.0, seed: int = SEED_LOGITS) -> torch.Tensor:
    """fp32 N(0, sigma^2) samples."""
    x = torch.randn(*shape, generator=_gen(seed), dtype=torch.float32)
    if sigma != 1.0:
        x = x * sigma
    return x


def uniform(n: int, lo: float, hi: float, seed: int = SEED_BIAS) -> torch.Tensor:
    """fp32 U(lo, hi) samples."""
    u = torch.rand(n, generator=_gen(seed), dtype=torch.float32)
    return lo + (hi - lo) * u


def zipf_offsets(E: int, s: float = 1.1, seed: int = SEED_OFFSETS) -> torch.Tensor:
    """Per-expert logit offsets giving Zipf(s)-skewed expert load.

    Expert e gets rank r[e] from a seeded random permutation of 1..E and the
    offset -s*ln(r[e]); exp(offset) is then proportional to r^-s.
    """
    rank = torch.randperm(E, generator=_gen(seed)) + 1
    return (-s * torch.log(rank.to(torch.float64))).to(torch.float32)


def as_dtype(x: torch.Tensor, in_dtype: int) -> torch.Tensor:
    """Round fp32 samples to the logits storage dtype (bf16: round to nearest even)."""
    return x.to(torch.bfloat16) if in_dtype == BF16 else x.contiguous()


def logits(T: int, E: int, sigma: float = 1.0, in_dtype: int = F32,
           zipf_s: Optional[float] = None, seed: int = SEED_LOGITS) -> torch.Tensor:
    x = normal((T, E), sigma, seed)
    if zipf_s is not None:
        x = x + zipf_offsets(E, zipf_s)[None, :]
    return as_dtype(x, in_dtype)


def grad(T: int, E: int, seed: int = SEED_GRAD) -> torch.Tensor:
    return normal((T, E), 1.0, seed)


def random_topk_idx(T: int, topk: int, E_tot: int, skew: Optional[float] = None,
                    seed: int = SEED_OFFSETS) -> tuple[torch.Tensor, torch.Tensor]:
    """Random (token, slot) -> expert assignments for exercising the sort alone.

    Each token gets ``topk`` distinct experts; with ``skew`` set, expert e is
    drawn with probability proportional to (rank of e)^-skew.
    """
    g = _gen(seed)
    if skew is None:
        w = torch.ones(E_tot, dtype=torch.float64)
    else:
        rank = torch.randperm(E_tot, generator=g) + 1
        w = rank.to(torch.float64) ** (-skew)
    idx = torch.multinomial(w.expand(T, E_tot), topk, replacement=False, generator=g)
    wt = torch.rand(T, topk, generator=g, dtype=torch.float32)
    return idx.to(torch.int32).contiguous(), wt.contiguous()


@dataclass
class Workload:
    """One router workload: sizes, options and the seeded inputs that go with them."""
    name: str
    T: int
    E: int
    topk: int
    score_fn: int = SOFTMAX
    in_dtype: int = F32
    renorm: int = 0
    scaling: float = 1.0
    n_group: int = 0
    topk_group: int = 0
    n_shared: int = 0
    shared_weight: float = 1.0
    sigma: float = 1.0
    bias_range: Optional[float] = None
    zipf_s: Optional[float] = None
    block_m: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def E_tot(self) -> int:
        return self.E + self.n_shared

    def make_logits(self) -> torch.Tensor:
        return logits(self.T, self.E, self.sigma, self.in_dtype, self.zipf_s)

    def make_bias(self) -> Optional[torch.Tensor]:
        if self.bias_range is None:
            return None
        return uniform(self.E, -self.bias_range, self.bias_range)

    def make_grad(self) -> torch.Tensor:
        return grad(self.T, self.E)


def tiny() -> Workload:
    """T=16, E=8, topk=2, fp32 N(0,1), softmax + renorm, scaling 1, block_m=4."""
    return Workload("tiny_T16_E8_k2", 16, 8, 2, SOFTMAX, F32, renorm=1, block_m=4)


def decode(T: int) -> Workload:
    """DeepSeek-R1-shaped decode: E=256, topk=8, bf16 N(0,1), softmax + renorm, block_m=32."""
    return Workload(f"decode_T{T}_E256_k8_bf16", T, 256, 8, SOFTMAX, BF16, renorm=1, block_m=32)


def decode_gpt_oss(T: int) -> Workload:
    """GPT-OSS-shaped decode: E=128, topk=4, bf16 N(0,1), softmax + renorm, block_m=32."""
    return Workload(f"decode_T{T}_E128_k4_bf16", T, 128, 4, SOFTMAX, BF16, renorm=1, block_m=32)


DECODE_TS = (1, 2, 4, 8, 12, 16, 24, 32, 48, 64)
# decode and small-batch sizes of the benchmark's latency tables (to 256 tokens)
DECODE_BENCH_TS = DECODE_TS + (96, 128, 192, 256)


def large_softmax(topk: int) -> Workload:
    """T=8192, E=512, fp32 N(0, 2^2), softmax, no renorm."""
    return Workload(f"softmax_T8192_E512_k{topk}", 8192, 512, topk, SOFTMAX, F32, sigma=2.0)


LARGE_TOPKS = (4, 8, 22, 36)


def large_e_softmax() -> Workload:
    """T=8192, E=2304, topk=36, fp32 N(0,1), softmax, no renorm."""
    return Workload("softmax_T8192_E2304_k36", 8192, 2304, 36, SOFTMAX, F32)


def large_e_sigmoid() -> Workload:
    """T=8192, E=2304, topk=36, fp32 N(0,1), sigmoid + bias U(-0.1,0.1), renorm, scaling 2.5."""
    return Workload("sigmoid_bias_T8192_E2304_k36", 8192, 2304, 36, SIGMOID, F32, renorm=1,
                    scaling=2.5, bias_range=0.1)


def widest_softmax() -> Workload:
    """T=8192, E=8160 (the widest row the pages' radix path takes), topk=36, fp32 N(0,1), softmax."""
    return Workload("softmax_T8192_E8160_k36", 8192, 8160, 36, SOFTMAX, F32)


def prefill_grouped() -> Workload:
    """T=16384, E=384 (+1 shared), topk=9, bf16 N(0,1)+Zipf(1.1) offsets, sigmoid + bias
    U(-0.05,0.05), 8 groups of 48 keep 4, renorm, scaling 2.827, block_m=64."""
    return Workload("prefill_T16384_E384+1_k9_grouped", 16384, 384, 9, SIGMOID, BF16, renorm=1,
                    scaling=2.827, n_group=8, topk_group=4, n_shared=1, shared_weight=1.0,
                    bias_range=0.05, zipf_s=1.1, block_m=64)


__all__ = [n for n in dir() if not n.startswith("_") and n not in ("torch",)]
