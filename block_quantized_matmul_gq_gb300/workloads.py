"""Seeded synthetic inputs and the workload shapes -- shared by the tests, the oracle
checks and the benchmark. This module holds none of the method's arithmetic: it draws
random fp32 tensors and lists matrix shapes, nothing else.

Shapes are those of the models the pages build or name:
  - TinyLLaMA-1.1B ("Development Guide for Small AI Models (TinyLLaMA, etc.) Using C++",
    sections 4.3 and 4.4 for GQA and SwiGLU): hidden 2048, 22 layers, 32 query heads and
    4 key/value heads of 64, FFN 5632, vocabulary 32000.
  - LLaMA-7B ("No Python! Building an AI Inference Engine Exclusively in C++", section 9):
    hidden 4096, FFN 11008, vocabulary 32000.
No real weights exist here: weights are N(0, 0.02) and activations N(0, 1), both fp32.

Seeds: weight matrix j of workload c uses seed 1000*c + j; the activations of N tokens
for matrix j use 1000*c + 500 + N + 7919*j (7919 keeps matrices of one step apart).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

W_STD = 0.02
X_STD = 1.0


@dataclass(frozen=True)
class MatShape:
    name: str
    M: int          # output features (rows of W)
    K: int          # input features (contiguous in W and X)
    layer: int = -1


def tinyllama_layer() -> list[MatShape]:
    h, kv, ffn = 2048, 4 * 64, 5632
    return [
        MatShape("q_proj", h, h), MatShape("k_proj", kv, h), MatShape("v_proj", kv, h),
        MatShape("o_proj", h, h), MatShape("gate_proj", ffn, h), MatShape("up_proj", ffn, h),
        MatShape("down_proj", h, ffn),
    ]


def tinyllama_decode_set() -> list[MatShape]:
    """All matmuls of one TinyLLaMA decode step: 7 per layer x 22 layers + lm_head."""
    out = []
    for layer in range(22):
        for s in tinyllama_layer():
            out.append(MatShape(s.name, s.M, s.K, layer))
    out.append(MatShape("lm_head", 32000, 2048))
    return out


def tinyllama_prefill_set() -> list[MatShape]:
    return [MatShape("gate_proj", 5632, 2048), MatShape("down_proj", 2048, 5632),
            MatShape("lm_head", 32000, 2048)]


def llama7b_set() -> list[MatShape]:
    return [MatShape("attn_proj", 4096, 4096), MatShape("gate_up_proj", 11008, 4096),
            MatShape("down_proj", 4096, 11008), MatShape("lm_head", 32000, 4096)]


WORKLOADS = {
    # id: (description, block type, token counts N, shapes)
    1: ("single Q4_0 GEMV 2048x2048, N=1", "q4_0", (1,), [MatShape("proj", 2048, 2048)]),
    2: ("TinyLLaMA-1.1B decode step, Q4_0, N=1", "q4_0", (1,), tinyllama_decode_set()),
    3: ("TinyLLaMA-1.1B decode step, Q8_0, N in 1..16", "q8_0", (1, 2, 4, 8, 16),
        tinyllama_decode_set()),
    4: ("TinyLLaMA-1.1B prefill, Q4_0, N=512", "q4_0", (512,), tinyllama_prefill_set()),
    5: ("LLaMA-7B shapes, Q4_0, N in {1,16,2048}", "q4_0", (1, 16, 2048), llama7b_set()),
}


def weight_seed(workload: int, j: int) -> int:
    return 1000 * workload + j


def act_seed(workload: int, N: int, j: int = 0) -> int:
    return 1000 * workload + 500 + N + 7919 * j


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def weights(M: int, K: int, seed: int, device="cpu") -> torch.Tensor:
    """fp32 M x K, N(0, 0.02), row-major."""
    g = _gen(seed, device)
    w = torch.randn((M, K), generator=g, dtype=torch.float32, device=device)
    return w.mul_(W_STD)


def activations(N: int, K: int, seed: int, device="cpu") -> torch.Tensor:
    """fp32 N x K, N(0, 1), row-major (token n is row n)."""
    g = _gen(seed, device)
    return torch.randn((N, K), generator=g, dtype=torch.float32, device=device).mul_(X_STD)
