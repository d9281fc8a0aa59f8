"""Seeded synthetic inputs for the quantized linear layers.

Shared by the tests (both the CUDA parity tests and the oracle's own tests)
and by the benchmark. It holds none of the method's arithmetic: it only draws
fp16 activations and fp16 weights. Everything is drawn on the CPU with a
torch CPU generator, so the same seed gives the same bits on every machine.

Recipe (the workload shapes of the Cider operator-latency tables, README
"Performance (Apple M5 Pro)", "Individual Operator Latency", with the value
distributions of the linear layers they time):
  1. x = randn(M, K) in fp32;
  2. idx = randperm(K)[:n_out]; x[:, idx] *= 20 (a few outlier channels, as
     LLM activations have);
  3. x = x.half();
  4. W = (randn(N, K) * 0.02).half()  (weights stored [out, in]).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

# Decoder-layer prefill (8B-class model, 2048 tokens): the seven linears in
# order, (name, K = in_features, N = out_features).
DECODER_LAYER = (
    ("q", 4096, 4096),
    ("k", 4096, 1024),
    ("v", 4096, 1024),
    ("o", 4096, 4096),
    ("gate", 4096, 12288),
    ("up", 4096, 12288),
    ("down", 12288, 4096),
)


def generator(seed: int = 0) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def activations(M: int, K: int, n_out: int, gen: torch.Generator) -> torch.Tensor:
    """fp16 [M, K]: N(0,1) with ``n_out`` random channels scaled by 20."""
    x = torch.randn(M, K, generator=gen, dtype=torch.float32)
    if n_out > 0:
        idx = torch.randperm(K, generator=gen)[:n_out]
        x[:, idx] *= 20.0
    return x.half()


def weights(N: int, K: int, gen: torch.Generator) -> torch.Tensor:
    """fp16 [N, K]: N(0, 0.02)."""
    return (torch.randn(N, K, generator=gen, dtype=torch.float32) * 0.02).half()


@dataclass
class LinearInputs:
    x: torch.Tensor  # fp16 [M, K], CPU
    w: torch.Tensor  # fp16 [N, K], CPU


def linear_inputs(M: int, N: int, K: int, n_out: int = 4, seed: int = 0) -> LinearInputs:
    """Draw order: x, outlier indices, W (one generator, seeded once)."""
    g = generator(seed)
    x = activations(M, K, n_out, g)
    w = weights(N, K, g)
    return LinearInputs(x, w)


def decoder_layer_inputs(M: int = 2048, seed: int = 0):
    """One independent (x, W) per linear of DECODER_LAYER, drawn in order from
    one generator; 1% of the input channels are outliers."""
    g = generator(seed)
    out = []
    for name, K, N in DECODER_LAYER:
        x = activations(M, K, max(1, round(K * 0.01)), g)
        w = weights(N, K, g)
        out.append((name, LinearInputs(x, w)))
    return out
