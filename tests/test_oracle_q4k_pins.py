"""Pins for the oracle's Q4_K super-blocks: a hand-worked golden super-block, closed-form
super-blocks the quantizer must recover exactly, exact-rational mul_mat and one-hot rows.

The pages name Q4_K ("Development Guide for Small AI Models (TinyLLaMA, etc.) Using C++",
section 6; "A Complete Guide to llama.cpp and Customization with C++", section 2.2)
without a layout; the oracle follows the published GGUF Q4_K block format: 256 weights in
8 sub-blocks of 32, 144 bytes (fp16 d, fp16 dmin, 12 bytes of packed 6-bit sub-block
scales and mins, 128 bytes of 4-bit codes), What = d sc_j q - dmin m_j.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

from block_quantized_matmul_gq_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "q4k_superblock.json")


def _code_bytes(codes):
    """The 128 code bytes as the format places them: byte 32 g + l holds weight 64 g + l
    in its low nibble and weight 64 g + 32 + l in its high nibble."""
    return bytes(codes[64 * g + l] | (codes[64 * g + 32 + l] << 4)
                 for g in range(4) for l in range(32))


def _fp16_bits(v: float) -> int:
    return int(np.array([v], np.float16).view(np.uint16)[0])


def test_golden_superblock_dequantizes_to_hand_worked_values(oracle_mod):
    g = json.load(open(GOLDEN))
    head = bytes([g["d_fp16_bits"] & 0xFF, g["d_fp16_bits"] >> 8,
                  g["dmin_fp16_bits"] & 0xFF, g["dmin_fp16_bits"] >> 8])
    blk = head + bytes(g["scale_bytes"]) + _code_bytes([k % 16 for k in range(256)])
    assert len(blk) == 144 == oracle_mod.block_bytes("q4_k")
    w = oracle_mod.dequantize("q4_k", np.frombuffer(blk, np.uint8), 1, 256)[0]
    for k, v in g["values"].items():
        assert w[int(k)] == np.float32(v), k


def _closed_form(rng, d_exp, dmin_exp, positive_subblocks=()):
    """A super-block whose exact values the quantizer must reproduce: d = 2^d_exp and
    dmin = 2^dmin_exp; sub-block 7 has sc = 63 and sub-block 0 has m = 63, so that
    d = max step / 63 and dmin = max min / 63 come out exact; every sub-block holds codes
    0 and 15 (min = -M_j, max = 15 D_j - M_j) except `positive_subblocks`, which have
    m = 0 and codes 1..15 only (all weights > 0: the range must still start at 0)."""
    d, dmin = 2.0 ** d_exp, 2.0 ** dmin_exp
    sc = rng.integers(1, 64, 8)
    sc[7] = 63
    m = rng.integers(0, 64, 8)
    m[0] = 63
    codes = rng.integers(0, 16, 256)
    for j in range(8):
        if j in positive_subblocks:
            m[j] = 0
            codes[32 * j: 32 * j + 32] = rng.integers(1, 16, 32)
            codes[32 * j + 3] = 15
        else:
            codes[32 * j + 1], codes[32 * j + 30] = 0, 15
    W = np.array([d * sc[k // 32] * codes[k] - dmin * m[k // 32] for k in range(256)],
                 np.float64)
    assert np.array_equal(W.astype(np.float32).astype(np.float64), W)   # exact in fp32
    return W.astype(np.float32), d, dmin, sc, m, codes


@pytest.mark.parametrize("d_exp,dmin_exp", [(-8, -9), (-12, -7), (-3, -5), (-14, -14)])
def test_closed_form_superblocks(oracle_mod, d_exp, dmin_exp):
    rng = np.random.default_rng(100 + d_exp - 3 * dmin_exp)
    W, d, dmin, sc, m, codes = _closed_form(rng, d_exp, dmin_exp, positive_subblocks=(2, 5))
    q = oracle_mod.quantize("q4_k", W.reshape(1, 256))[0]
    assert int(q[0]) | int(q[1]) << 8 == _fp16_bits(d)
    assert int(q[2]) | int(q[3]) << 8 == _fp16_bits(dmin)
    assert bytes(q[16:]) == _code_bytes(list(codes))
    # the recovered scales and mins reproduce every weight exactly
    assert np.array_equal(oracle_mod.dequantize("q4_k", q, 1, 256)[0], W)


def test_zero_and_constant_subblocks(oracle_mod):
    W = np.zeros((1, 256), np.float32)
    assert not oracle_mod.quantize("q4_k", W).any()                   # d = dmin = 0, codes 0
    W[0, 64:96] = -63 * 2.0 ** -8          # constant, negative: step 0, dmin = 2^-8, m = 63
    q = oracle_mod.quantize("q4_k", W)
    wh = oracle_mod.dequantize("q4_k", q, 1, 256)[0]
    assert np.array_equal(wh[64:96], W[0, 64:96])                     # What = -dmin m exactly
    assert not wh[:64].any() and not wh[96:].any()


def test_roundtrip_idempotence_and_error_bound(oracle_mod):
    """quant(dequant(quant(w))) keeps every weight: the second pass sees a super-block that
    the first pass's parameters represent, and reproduces its values. Per element the
    first pass errs by at most half a code step plus what the 6-bit scales cost."""
    W = workloads.weights(16, 1024, seed=33).numpy()
    q1 = oracle_mod.quantize("q4_k", W)
    w1 = oracle_mod.dequantize("q4_k", q1, 16, 1024)
    w2 = oracle_mod.dequantize("q4_k", oracle_mod.quantize("q4_k", w1), 16, 1024)
    assert np.array_equal(w1, w2)
    sub = W.reshape(16, -1, 32).astype(np.float64)
    rng_ = sub.max(axis=2) - np.minimum(sub.min(axis=2), 0.0)
    # step D_j deviates from (hi - lo) / 15 by at most d/2 (6-bit rounding) + fp16 error
    bound = (rng_ / 15.0)[..., None] * 1.2 + np.abs(sub).max(axis=2, keepdims=True) * 0.1
    assert np.all(np.abs(sub - w1.reshape(sub.shape)) <= bound)


def _ulp32(v: float) -> Fraction:
    a = abs(np.float32(v))
    if a == 0:
        return Fraction(2) ** -149
    return Fraction(float(np.nextafter(np.float32(a), np.float32(np.inf)))) - Fraction(float(a))


@pytest.mark.parametrize("M,N,K", [(1, 1, 256), (3, 2, 512), (2, 3, 256)])
def test_mul_mat_exact_rational(oracle_mod, M, N, K):
    W = workloads.weights(M, K, seed=M * 10 + K).numpy()
    X = workloads.activations(N, K, seed=N * 10 + K).numpy()
    q = oracle_mod.quantize("q4_k", W)
    wh = oracle_mod.dequantize("q4_k", q, M, K)
    Y = oracle_mod.mul_mat("q4_k", q, M, K, X)
    for n in range(N):
        for m in range(M):
            terms = [Fraction(float(wh[m, k])) * Fraction(float(X[n, k])) for k in range(K)]
            exact = sum(terms, Fraction(0))
            slack = _ulp32(Y[n, m]) / 2 + K * Fraction(2) ** -53 * sum(abs(x) for x in terms)
            assert abs(Fraction(float(Y[n, m])) - exact) <= slack, (n, m)


def test_mul_mat_one_hot_returns_dequantized_rows(oracle_mod):
    M, K = 5, 512
    q = oracle_mod.quantize("q4_k", workloads.weights(M, K, seed=7).numpy())
    wh = oracle_mod.dequantize("q4_k", q, M, K)
    ks = [0, 31, 32, 63, 64, 255, 256, 300, 511]
    X = np.zeros((len(ks), K), np.float32)
    for n, k in enumerate(ks):
        X[n, k] = 1.0
    Y = oracle_mod.mul_mat("q4_k", q, M, K, X)
    for n, k in enumerate(ks):
        assert np.array_equal(Y[n], wh[:, k]), k


def test_rows_must_hold_whole_superblocks(oracle_mod):
    with pytest.raises(ValueError):
        oracle_mod.quantize("q4_k", np.zeros((1, 288), np.float32))
    assert oracle_mod.row_bytes("q4_k", 2048) == 8 * 144


def test_codes_follow_the_rounded_subblock_scale(oracle_mod):
    """Worked by hand. Sub-block 7 spans [0, 945 * 2^-6]: step 63 * 2^-6, so d = 2^-6
    exactly and sc_7 = 63. Sub-block 0 spans [0, 157.5 * 2^-6]: step 10.5 * 2^-6, so
    sc_0 = round(10.5) = 11 (halves away from zero) and D_0 = 11 * 2^-6. Its largest
    weight then gets code round(157.5 / 11) = 14 (What = 154 * 2^-6), not 15: codes follow
    the dequantization's own D_j, not the unrounded step. No weight is negative, so
    dmin = 0 and every M_j = 0."""
    W = np.zeros((1, 256), np.float32)
    W[0, 224], W[0, 255] = 0.0, 945 * 2.0 ** -6
    W[0, 0], W[0, 17] = 0.0, 157.5 * 2.0 ** -6
    q = oracle_mod.quantize("q4_k", W)[0]
    assert int(q[0]) | int(q[1]) << 8 == _fp16_bits(2.0 ** -6)
    assert int(q[2]) == 0 and int(q[3]) == 0
    wh = oracle_mod.dequantize("q4_k", q, 1, 256)[0]
    assert wh[17] == np.float32(154 * 2.0 ** -6)
    assert wh[255] == np.float32(945 * 2.0 ** -6)
    assert int(q[16 + 17]) & 15 == 14
