"""Seeded synthetic inputs for the BitLinear forward.

This module holds no arithmetic of the method: it only draws latent weights
and activations with fixed seeds, in the shapes and value distributions of the
workloads below, so that the CUDA library and the CPU oracle see identical
inputs.  Both the tests and ``bench.py`` import it; neither side of the parity
check depends on the other through it.

Workloads (shapes are [M tokens, K in-features] -> N out-features):

* ``tiny``     M=8, K=512, N=256; W ~ N(0, 0.02), X fp32 ~ N(0, 1), seed 0.
* ``decode``   M=1; (K=2560 -> N=6912) and (K=6912 -> N=2560); W ~ N(0, 0.02);
               X bf16 ~ N(0, 1).  A 2B-class FFN pair at one token.
* ``skinny``   M in {1, 16, 64}; (K=3200 -> N=8640) and (K=8640 -> N=3200);
               W ~ N(0, 0.02); X bf16 ~ N(0, 1) with 1% of entries times 20.
* ``prefill``  M=2048, K=2560 -> N=6912; W ~ N(0, 0.02); X bf16 ~ N(0, 1).
* ``llama70b`` M in {1, 16, 176}; (K=8192 -> N=28672) and (K=28672 -> N=8192);
               W ~ N(0, 0.01); X bf16 ~ N(0, 1).

The 2B/3B/70B labels follow the model sizes the BitNet b1.58 pages discuss
(2B4T on the yousumm.com transcript; 3B and 70B in the cost paragraph of
anthology note-168, "Where the claim is strong, and where it stops"; batch 176
is the 70B maximum batch quoted there).  No dataset is involved: every value
is drawn here.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Layer:
    """One BitLinear problem: y[M, N] = BitLinear(W[N, K]) (X[M, K])."""

    M: int
    K: int
    N: int
    w_sigma: float
    x_dtype: str  # "f32" or "bf16"
    outlier_frac: float = 0.0
    outlier_scale: float = 20.0


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    layers: tuple
    eps: float = 1e-5
    source_index: tuple = ()  # layer indices in the full workload (set by select_layers)


WORKLOADS = {
    "tiny": Workload("tiny", 0, (Layer(8, 512, 256, 0.02, "f32"),)),
    "decode": Workload("decode", 2, (Layer(1, 2560, 6912, 0.02, "bf16"), Layer(1, 6912, 2560, 0.02, "bf16"))),
    "skinny": Workload(
        "skinny",
        3,
        tuple(
            Layer(m, k, n, 0.02, "bf16", outlier_frac=0.01)
            for m in (1, 16, 64)
            for (k, n) in ((3200, 8640), (8640, 3200))
        ),
    ),
    "prefill": Workload("prefill", 4, (Layer(2048, 2560, 6912, 0.02, "bf16"),)),
    "llama70b": Workload(
        "llama70b",
        5,
        tuple(Layer(m, k, n, 0.01, "bf16") for m in (1, 16, 176) for (k, n) in ((8192, 28672), (28672, 8192))),
    ),
}


def select_layers(wl: Workload, indices) -> Workload:
    """The workload restricted to some of its layers, each keeping the seeds it
    has in the full workload (so its inputs are unchanged)."""
    return Workload(wl.name, wl.seed, tuple(wl.layers[i] for i in indices), wl.eps,
                    tuple(_layer_index(wl, i) for i in indices))


def _layer_index(wl: Workload, i: int) -> int:
    return wl.source_index[i] if wl.source_index else i


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def latent_weights(N: int, K: int, sigma: float, seed: int) -> torch.Tensor:
    """fp32 [N, K] ~ N(0, sigma), CPU tensor."""
    return torch.randn((N, K), generator=_gen(seed), dtype=torch.float32) * float(sigma)


def activations(M: int, K: int, dtype: str, seed: int, outlier_frac: float = 0.0,
                outlier_scale: float = 20.0) -> torch.Tensor:
    """[M, K] ~ N(0, 1) in fp32 or bf16 (CPU tensor).  With outlier_frac > 0 a
    Bernoulli(outlier_frac) mask from the same generator multiplies the chosen
    entries by outlier_scale (before the cast to bf16)."""
    g = _gen(seed)
    x = torch.randn((M, K), generator=g, dtype=torch.float32)
    if outlier_frac > 0:
        mask = torch.rand((M, K), generator=g) < outlier_frac
        x = torch.where(mask, x * float(outlier_scale), x)
    if dtype == "bf16":
        return x.to(torch.bfloat16)
    if dtype == "f32":
        return x
    raise ValueError(dtype)


def weight_seed(wl: Workload, index: int) -> int:
    """Layers of a workload that differ only in M are one weight matrix seen at
    several batch sizes: the weight seed depends on the (K, N) shape only."""
    full = WORKLOADS[wl.name]
    shapes = []
    for L in full.layers:
        if (L.K, L.N) not in shapes:
            shapes.append((L.K, L.N))
    L = wl.layers[index]
    return 1000 * wl.seed + shapes.index((L.K, L.N))


def activation_seed(wl: Workload, index: int) -> int:
    return 1000 * wl.seed + 500 + _layer_index(wl, index)


def layer_weights(wl: Workload, index: int) -> torch.Tensor:
    L = wl.layers[index]
    return latent_weights(L.N, L.K, L.w_sigma, seed=weight_seed(wl, index))


def layer_activations(wl: Workload, index: int) -> torch.Tensor:
    L = wl.layers[index]
    return activations(L.M, L.K, L.x_dtype, seed=activation_seed(wl, index), outlier_frac=L.outlier_frac,
                       outlier_scale=L.outlier_scale)


def layer_inputs(wl: Workload, index: int) -> tuple[torch.Tensor, torch.Tensor]:
    """(W fp32 [N,K], X [M,K]) for layer ``index`` of workload ``wl``."""
    return layer_weights(wl, index), layer_activations(wl, index)


def x_as_f32_numpy(X: torch.Tensor) -> np.ndarray:
    """Exact fp32 numpy copy of X (bf16 -> fp32 widening is exact)."""
    return X.to(torch.float32).numpy()


def x_bits_numpy(X: torch.Tensor) -> np.ndarray:
    """Raw bit patterns of a bf16 tensor as uint16 numpy."""
    assert X.dtype == torch.bfloat16
    return X.view(torch.int16).numpy().view(np.uint16)
