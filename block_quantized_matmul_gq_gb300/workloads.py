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


def q4k_superblocks(M: int, K: int, seed: int):
    """Hand-made Q4_K super-block bytes (numpy uint8, M x K/256 super-blocks of 144 bytes,
    the published GGUF Q4_K layout: fp16 d, fp16 dmin, 12 scale bytes, 128 code bytes).
    Row m has kind m % 8:
      0  random scale and code bytes, d and dmin N(0, 0.01) of either sign
      1  every scale and min at 63 (all twelve scale bytes 0xFF), codes 0 and 15 only,
         d and dmin +-65504 (the largest finite fp16)
      2  random bytes, d and dmin fp16 subnormals of either sign
      3  random bytes, d and dmin +0 or -0 (the row's weights are exactly zero)
      4  random bytes, d and dmin both negative
      5-7 random bytes, each super-block's d and dmin drawn from all of the above
    Only bytes are drawn here; nothing of the method is computed."""
    import numpy as np
    if K % 256:
        raise ValueError("K must be a multiple of 256")
    rng = np.random.default_rng(seed)
    nsb = K // 256
    blocks = rng.integers(0, 256, size=(M, nsb, 144), dtype=np.uint8)

    def normal(shape):
        return (rng.standard_normal(shape) * 0.01).astype(np.float16).view(np.uint16)

    def subnormal(shape):
        return (rng.integers(1, 1024, shape) | (rng.integers(0, 2, shape) << 15)).astype(np.uint16)

    def huge(shape):
        return (np.uint16(_F16_MAX) | (rng.integers(0, 2, shape) << 15)).astype(np.uint16)

    def zero(shape):
        return (rng.integers(0, 2, shape) << 15).astype(np.uint16)

    heads = np.empty((M, nsb, 2), np.uint16)
    for m in range(M):
        kind = m % 8
        if kind == 0:
            heads[m] = normal((nsb, 2))
        elif kind == 1:
            heads[m] = huge((nsb, 2))
            blocks[m, :, 4:16] = 0xFF
            blocks[m, :, 16:] = np.where(rng.random((nsb, 128)) < 0.5, 0x00, 0xFF)
        elif kind == 2:
            heads[m] = subnormal((nsb, 2))
        elif kind == 3:
            heads[m] = zero((nsb, 2))
        elif kind == 4:
            heads[m] = normal((nsb, 2)) | np.uint16(_F16_SIGN)
        else:
            pick = rng.integers(0, 4, (nsb, 2))
            heads[m] = np.choose(pick, [normal((nsb, 2)), subnormal((nsb, 2)), huge((nsb, 2)),
                                        zero((nsb, 2))]).astype(np.uint16)
    blocks[:, :, 0:4] = heads.view(np.uint8).reshape(M, nsb, 4)
    return blocks.reshape(M, nsb * 144)


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


# fp16 bit patterns of the hand-made blocks' scales
_F16_MAX = 0x7BFF            # 65504, the largest finite fp16
_F16_SIGN = 0x8000


def edge_blocks(t: str, M: int, K: int, seed: int):
    """Hand-made block bytes (numpy uint8, M x K/32 blocks, the public layout) that the
    quantizer never writes but the layout allows. Row m has kind m % 8, so every kind
    lands at every position of a tile:
      0  every code at its minimum (Q4_0 code 0, i.e. -8; Q8_0 code -128), normal scales
      1  every code at its minimum, every scale +-65504 (the largest finite fp16)
      2  random codes, every scale an fp16 subnormal (magnitude 2^-24 .. 1023 * 2^-24)
      3  random codes, every scale +0 or -0 (the row's outputs are exactly zero)
      4  only the extreme codes (0 / 15, or -128 / 127), every scale negative
      5-7 random codes, each block's scale drawn from a mixture of all the above and
         ordinary N(0, 0.01) scales of either sign
    Random codes are uniform over every byte value, so Q4_0 code 0 and Q8_0 code -128
    occur throughout. Only bytes are drawn here; nothing of the method is computed."""
    import numpy as np
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    rng = np.random.default_rng(seed)
    nb = K // 32
    bb = 18 if t == "q4_0" else 34
    blocks = rng.integers(0, 256, size=(M, nb, bb), dtype=np.uint8)
    codes = blocks[:, :, 2:]
    low = 0x00 if t == "q4_0" else 0x80           # Q4_0: both nibbles 0; Q8_0: int8 -128
    high = 0xFF if t == "q4_0" else 0x7F          # Q4_0: both nibbles 15; Q8_0: 127

    def normal(shape):
        return (rng.standard_normal(shape) * 0.01).astype(np.float16).view(np.uint16)

    def subnormal(shape):
        return (rng.integers(1, 1024, shape) | (rng.integers(0, 2, shape) << 15)).astype(np.uint16)

    def huge(shape):
        mag = rng.uniform(3.0e4, 65504.0, shape).astype(np.float16).view(np.uint16)
        mag = np.where(rng.random(shape) < 0.5, np.uint16(_F16_MAX), mag)
        return (mag | (rng.integers(0, 2, shape) << 15)).astype(np.uint16)

    def zero(shape):
        return (rng.integers(0, 2, shape) << 15).astype(np.uint16)

    scales = np.empty((M, nb), np.uint16)
    for m in range(M):
        kind = m % 8
        if kind == 0:
            codes[m] = low
            scales[m] = normal(nb)
        elif kind == 1:
            codes[m] = low
            scales[m] = huge(nb)
        elif kind == 2:
            scales[m] = subnormal(nb)
        elif kind == 3:
            scales[m] = zero(nb)
        elif kind == 4:
            codes[m] = np.where(rng.random(codes[m].shape) < 0.5, low, high).astype(np.uint8)
            scales[m] = normal(nb) | np.uint16(_F16_SIGN)
        else:
            pick = rng.integers(0, 6, nb)
            cand = np.stack([normal(nb), normal(nb) | np.uint16(_F16_SIGN), subnormal(nb),
                             zero(nb), huge(nb), normal(nb)])
            scales[m] = cand[pick, np.arange(nb)]
    blocks[:, :, 0] = (scales & 0xFF).astype(np.uint8)
    blocks[:, :, 1] = (scales >> 8).astype(np.uint8)
    return np.ascontiguousarray(blocks.reshape(M, nb * bb))
