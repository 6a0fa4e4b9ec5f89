"""Synthetic workloads: shapes, value distributions and seeded generators.

This module holds no arithmetic of the method itself.  It only says how large
each workload is and draws its seeded random inputs.  The GPU path and the
CPU oracle are both fed from here, and from nothing else they share.

The shapes follow the training runs on the pages:
  * "Merge LoCo with Zero++" (DeepSpeed PR #6730), Experimental Results:
    Llama-2-architecture pretraining at 0.8B and 8B parameters.  The gradient
    of one transformer layer is 4*d^2 (attention) + 3*d*ffn (gated MLP):
    d=2048, ffn=5504 gives 50,593,792 elements; d=4096, ffn=11008 gives
    202,375,168.
  * "Zero 2 #593" (llm.c): GPT-2 small gradient shards, 124,475,904 elements.
The pages' dataset (RedPajama-V2) is not used.  Seeded normal gradients with
a sparse fraction of outliers stand in for it.

Seeds: 1000 * workload_index + 100 * step + rank, one torch.Generator per
(rank, step) on the device the tensor is made on.  Values are drawn in fp32,
the outliers are multiplied in fp32, and the result is rounded to bf16 by
torch's conversion.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


def llama_layer_numel(d: int, ffn: int) -> int:
    """Weights of one Llama-2 layer: q, k, v, o (4 d^2) + gate, up, down (3 d ffn)."""
    return 4 * d * d + 3 * d * ffn


@dataclass(frozen=True)
class QgzWorkload:
    """Quantized-gradient reduce over R simulated ranks of N elements each."""
    index: int          # seed namespace
    name: str
    R: int              # simulated ranks
    N: int              # gradient elements per rank
    G: int              # rank groups (1 = flat reduce, >1 = two hops)
    B: int              # quantization block (elements)
    err_scale: float    # LoCo error scale s
    err_beta: float     # LoCo moving-average factor beta
    steps: int
    sigma: float        # std of the gradient values
    outlier_frac: float
    outlier_mult: float
    out_bf16: bool      # reduced shards stored as bf16 (else fp32)

    @property
    def S(self) -> int:
        return self.N // self.R

    @property
    def L(self) -> int:
        return self.R // self.G

    def scaled(self, N: int, name: str | None = None) -> "QgzWorkload":
        """Same workload with a different per-rank size (tests, samples)."""
        return QgzWorkload(self.index, name or f"{self.name}@N={N}", self.R, N, self.G,
                           self.B, self.err_scale, self.err_beta, self.steps,
                           self.sigma, self.outlier_frac, self.outlier_mult,
                           self.out_bf16)


@dataclass(frozen=True)
class QwzWorkload:
    index: int
    name: str
    n: int
    B: int
    sigma: float


@dataclass(frozen=True)
class SrWorkload:
    index: int
    name: str
    n: int
    micro_steps: int
    sigma: float
    seed: int


# Four ranks of 1M elements, pure error feedback (s=1, beta=0), 3 steps.
QGZ_TINY = QgzWorkload(1, "qgz_tiny R=4 N=1048576 B=256", R=4, N=1_048_576, G=1,
                       B=256, err_scale=1.0, err_beta=0.0, steps=3, sigma=1e-3,
                       outlier_frac=1e-3, outlier_mult=100.0, out_bf16=False)

# One d=2048, ffn=5504 layer on 8 ranks, LoCo (s=1, beta=0.5), 10 steps.
QGZ_SINGLE_HOP = QgzWorkload(2, "qgz_single_hop R=8 N=50593792 B=256", R=8,
                             N=llama_layer_numel(2048, 5504), G=1, B=256,
                             err_scale=1.0, err_beta=0.5, steps=10, sigma=1e-3,
                             outlier_frac=1e-4, outlier_mult=50.0, out_bf16=False)

# One d=4096, ffn=11008 layer on 16 ranks in 2 groups of 8, two hops, bf16 out.
QGZ_HIERARCHICAL = QgzWorkload(3, "qgz_hierarchical R=16 G=2 N=202375168 B=512",
                               R=16, N=llama_layer_numel(4096, 11008), G=2, B=512,
                               err_scale=1.0, err_beta=0.5, steps=5, sigma=1e-3,
                               outlier_frac=1e-4, outlier_mult=50.0, out_bf16=True)

# 16 d=2048 layers plus a tied 32000 x 2048 embedding: ~0.875B weights.
QWZ_WEIGHTS = QwzWorkload(4, "qwz n=875036672 B=2048",
                          n=16 * llama_layer_numel(2048, 5504) + 32000 * 2048,
                          B=2048, sigma=0.02)

# GPT-2 small gradient shard, 8 micro-steps.
SR_ACCUMULATE = SrWorkload(5, "sr_accumulate n=124475904 x8", n=124_475_904,
                           micro_steps=8, sigma=1e-4, seed=5)

QGZ_WORKLOADS = {"qgz_tiny": QGZ_TINY, "qgz_single_hop": QGZ_SINGLE_HOP,
                 "qgz_hierarchical": QGZ_HIERARCHICAL}


def seed_of(index: int, step: int, rank: int) -> int:
    return 1000 * index + 100 * step + rank


def draw_bf16(n: int, sigma: float, seed: int, device="cpu",
              outlier_frac: float = 0.0, outlier_mult: float = 1.0,
              out: torch.Tensor | None = None) -> torch.Tensor:
    """n bf16 values: N(0, sigma^2) in fp32, an independent Bernoulli(frac)
    subset multiplied by outlier_mult, then rounded to bf16."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    x = torch.randn(n, generator=gen, device=device, dtype=torch.float32)
    x.mul_(sigma)
    if outlier_frac > 0.0:
        u = torch.rand(n, generator=gen, device=device, dtype=torch.float32)
        x = torch.where(u < outlier_frac, x * outlier_mult, x)
    if out is None:
        return x.to(torch.bfloat16)
    out.copy_(x)
    return out


def qgz_gradients(w: QgzWorkload, step: int, device="cpu",
                  out: torch.Tensor | None = None) -> torch.Tensor:
    """[R, N] bf16 gradients of every simulated rank at one step."""
    if out is None:
        out = torch.empty((w.R, w.N), dtype=torch.bfloat16, device=device)
    for r in range(w.R):
        draw_bf16(w.N, w.sigma, seed_of(w.index, step, r), device,
                  w.outlier_frac, w.outlier_mult, out=out[r])
    return out


def qwz_weights(w: QwzWorkload, device="cpu") -> torch.Tensor:
    return draw_bf16(w.n, w.sigma, seed_of(w.index, 0, 0), device)


def sr_micro_gradient(w: SrWorkload, step: int, device="cpu",
                      out: torch.Tensor | None = None) -> torch.Tensor:
    return draw_bf16(w.n, w.sigma, seed_of(w.index, step, 0), device, out=out)


def as_u16(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view("uint16")


def from_u16(a, device="cpu") -> torch.Tensor:
    """numpy uint16 bit patterns -> bf16 tensor."""
    import numpy as np
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
