"""Seeded synthetic inputs for the MoE routing path.

This module only draws random numbers and names workloads; it holds none of
the routing arithmetic.  Both the CPU oracle (``oracle/``) and the CUDA
library's tests and benchmark take their inputs from here, so the two sides
see the same bf16 bits.

Workload recipe (shapes from the routing throughput table and the text of the
moe-engine page, "moe-engine：面向万卡集群的稀疏MoE训练基础设施", section
实验结果与性能数据; value distributions chosen so that logits have unit scale):

* ``X``  [N, H]  bf16, entries N(0, 1) drawn in fp32 and rounded to bf16;
* ``W``  [H, E]  bf16, entries N(0, 1/H) (std 1/sqrt(H)) drawn after X from
  the same generator;
* ``bias`` [E] fp32, only for the skewed workload:
  ``bias[e] = 2.0 * ln(1 / (e + 1))`` (a Zipf-like preference for low expert
  ids), added to the logits by the router.

All draws use a CPU ``torch.Generator`` seeded with ``seed``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    N: int
    H: int
    E: int
    K: int
    renorm: bool = True
    fp8: bool = False
    skew: bool = False
    seeds: tuple = (0,)
    note: str = ""

    def as_dict(self):
        return dict(workload=self.name, N=self.N, H=self.H, E=self.E, K=self.K,
                    renorm=self.renorm, fp8=self.fp8, skew=self.skew)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_n512_h256_e16_k2", 512, 256, 16, 2,
                 note="tiny router+dispatch case"),
        Workload("n2048_h1024_e64_k2", 2048, 1024, 64, 2,
                 note="dispatch + combine over bf16 rows of width H"),
        Workload("n4096_h2048_e64_k4", 4096, 2048, 64, 4, seeds=tuple(range(20)),
                 note="full route->dispatch->combine, 20 seeds"),
        Workload("moe_layer_n16384_h2048_e128_k8_fp8", 16384, 2048, 128, 8, fp8=True,
                 note="4 sequences x 4096 tokens, dispatch also emits E4M3 + fp32 1x128 scales"),
        Workload("skewed_zipf_n65536_h4096_e64_k2", 65536, 4096, 64, 2, skew=True,
                 note="per-expert logit bias 2*ln(1/rank)"),
    ]
}

# The workload the benchmark times by default: the largest of the five, the one
# that fits a single GPU and where the copy and router kernels run at HBM speed.
BENCH_WORKLOAD = "skewed_zipf_n65536_h4096_e64_k2"


def zipf_bias(E: int) -> torch.Tensor:
    """bias[e] = 2.0 * ln(1/(e+1)) in fp32 (rank = e + 1)."""
    r = torch.arange(1, E + 1, dtype=torch.float64)
    return (2.0 * torch.log(1.0 / r)).to(torch.float32)


def make_route_inputs(N: int, H: int, E: int, seed: int = 0, skew: bool = False):
    """Returns (X bf16 [N,H], W bf16 [H,E], bias fp32 [E] or None) as CPU tensors."""
    g = torch.Generator().manual_seed(seed)
    X = torch.randn(N, H, generator=g, dtype=torch.float32).to(torch.bfloat16)
    W = (torch.randn(H, E, generator=g, dtype=torch.float32) * (1.0 / math.sqrt(H))).to(torch.bfloat16)
    bias = zipf_bias(E) if skew else None
    return X, W, bias


def make_workload_inputs(w: Workload, seed: int | None = None):
    return make_route_inputs(w.N, w.H, w.E, w.seeds[0] if seed is None else seed, w.skew)


def make_replica_inputs(w: Workload, rank: int):
    """Inputs of one data-parallel replica: rank r routes its own tokens (the X
    drawn from a generator seeded with seed0 + r) against the gate every rank
    shares (the W drawn from the seed0 generator, after its X).  Rank 0's inputs
    are the workload's own."""
    seed0 = w.seeds[0]
    X0, W, bias = make_route_inputs(w.N, w.H, w.E, seed0, w.skew)
    if rank == 0:
        return X0, W, bias
    del X0
    X, _, _ = make_route_inputs(w.N, w.H, w.E, seed0 + rank, w.skew)
    return X, W, bias


def random_topk_idx(N: int, E: int, K: int, seed: int = 0) -> torch.Tensor:
    """K distinct experts per token, uniformly at random (int32 [N,K], CPU)."""
    g = torch.Generator().manual_seed(seed)
    keys = torch.rand(N, E, generator=g)
    return keys.argsort(dim=1)[:, :K].to(torch.int32).contiguous()


def random_bf16(shape, seed: int = 0, scale: float = 1.0) -> torch.Tensor:
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g, dtype=torch.float32) * scale).to(torch.bfloat16)


def random_weights(N: int, K: int, seed: int = 0) -> torch.Tensor:
    """Positive fp32 weights [N,K] (uniform in (0,1]); not normalised."""
    g = torch.Generator().manual_seed(seed)
    return (1.0 - torch.rand(N, K, generator=g, dtype=torch.float32)).contiguous()


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The raw uint16 bits of a CPU bf16 tensor as numpy."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def bits_to_bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)
