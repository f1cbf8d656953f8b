"""Seeded synthetic inputs for the NVFP4 linear layer.

This module draws random tensors and nothing else: it holds none of the
quantization or GEMM arithmetic, so the CUDA path and the CPU oracle can both
be fed from it without sharing any of the method.

The pages' workloads (Gemma-4 31B projections on the "nvfp4-gemma4" page,
the Flux2 / Wan 2.1 diffusion-transformer qkv and feed-forward linears on the
"nvfp4-difusion" page, section 1) need trained weights that are not
available, so seeded synthetic tensors with the shapes below stand in:

* activations X ~ N(0, 1) in bfloat16; for the LLM shapes, round(0.001 K)
  input channels (picked without replacement) are multiplied by 50 -- the
  ~0.1 % outlier dimensions that the LLM.int8 discussion on the
  "cuantizacion e inferencia local" page describes; for the DiT shapes each
  token (row) is multiplied by its own U(0.5, 4) factor;
* weights W ~ N(0, 0.02) in bfloat16, quantized offline before use.

Values are drawn in float32 by a CPU ``torch.Generator`` and rounded to
bfloat16 (round to nearest even), so the same seed gives the same bytes on
every machine.
"""
from __future__ import annotations

import dataclasses

import torch

__all__ = ["Workload", "WORKLOADS", "make_x", "make_w", "x_seed", "w_seed"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    index: int
    M: tuple
    K: int
    N: tuple
    x_kind: str          # "normal" | "outlier" | "token_scaled"
    description: str


WORKLOADS = {
    w.name: w for w in (
        Workload("tiny", 0, (64,), 256, (128,), "normal",
                 "tiny NVFP4 linear 64x256 -> 128"),
        Workload("prefill", 1, (4096,), 5120, (5120,), "outlier",
                 "LLM prefill projection 4096 tokens, 5120 -> 5120"),
        Workload("decode", 2, (1, 8, 32), 5120, (27648,), "outlier",
                 "LLM decode FFN-up, M in {1,8,32}, 5120 -> 27648"),
        Workload("dit", 3, (4096,), 3072, (9216, 12288), "token_scaled",
                 "DiT block, 4096 image tokens, 3072 -> 9216 (qkv) and 12288 (FFN)"),
        Workload("square", 4, (16384,), 16384, (16384,), "outlier",
                 "square 16384^3 GEMM and 16384x16384 activation quantize"),
    )
}


def x_seed(w: Workload) -> int:
    return 1234 + w.index


def w_seed(w: Workload) -> int:
    return 4321 + w.index


def make_x(kind: str, M: int, K: int, seed: int, device: str = "cpu") -> torch.Tensor:
    """Activation tensor (M, K) bfloat16. The CPU generator (the default) is
    what parity tests use; ``device="cuda"`` draws the same distribution
    with the device generator (different values), for large benchmark
    inputs."""
    g = torch.Generator(device=device).manual_seed(seed)
    x = torch.randn((M, K), generator=g, dtype=torch.float32, device=device)
    if kind == "outlier":
        n_out = int(round(0.001 * K))
        if n_out:
            cols = torch.randperm(K, generator=g, device=device)[:n_out]
            x[:, cols] *= 50.0
    elif kind == "token_scaled":
        scale = torch.rand((M, 1), generator=g, dtype=torch.float32, device=device) * 3.5 + 0.5
        x *= scale
    elif kind != "normal":
        raise ValueError("unknown activation kind %r" % kind)
    return x.to(torch.bfloat16)


def make_w(N: int, K: int, seed: int, std: float = 0.02, device: str = "cpu") -> torch.Tensor:
    """Weight tensor (N, K) bfloat16 (CPU generator by default)."""
    g = torch.Generator(device=device).manual_seed(seed)
    w = torch.randn((N, K), generator=g, dtype=torch.float32, device=device) * std
    return w.to(torch.bfloat16)


def make_bias(N: int, seed: int, std: float = 0.5, device: str = "cpu") -> torch.Tensor:
    """Bias vector (N,) bfloat16 (CPU generator by default), on the scale of
    the linear layers' outputs (unit-variance activations against 0.02-std
    weights over thousands of inputs give outputs of order 1)."""
    g = torch.Generator(device=device).manual_seed(seed)
    b = torch.randn((N,), generator=g, dtype=torch.float32, device=device) * std
    return b.to(torch.bfloat16)


def make_lora(r: int, K: int, N: int, seed: int, std: float = 0.02, device: str = "cpu"):
    """LoRA factors (A: (r, K) down projection, B: (N, r) up projection),
    bfloat16, both ~N(0, std^2) (CPU generator by default); with unit-variance
    activations the correction is about a tenth of the layer's output."""
    g = torch.Generator(device=device).manual_seed(seed)
    a = torch.randn((r, K), generator=g, dtype=torch.float32, device=device) * std
    b = torch.randn((N, r), generator=g, dtype=torch.float32, device=device) * std
    return a.to(torch.bfloat16), b.to(torch.bfloat16)
