"""Pins for the CPU oracle: each test checks it against something other than itself --
an IEEE conversion in numpy / torch, a closed-form block, exact rational arithmetic, a
one-hot activation or a figure the pages print (tests/golden/page_facts.json).

Pages cited: "A Complete Guide to llama.cpp and Customization with C++" (section 2.2,
block quantization), "Development Guide for Small AI Models (TinyLLaMA, etc.) Using C++"
(sections 6, 6.1, 6.2: sizes, Q4_0 layout, dequantize-then-FMA), "No Python! Building an
AI Inference Engine Exclusively in C++" (sections 6, 7.2, 9: the product, its layout and
the size ratios).
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

from block_quantized_matmul_gq_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")


def _pow2_fp16_bits(e: int) -> int:
    """binary16 bit pattern of 2^e for a normal exponent (-14 <= e <= 15)."""
    return (e + 15) << 10


def _block_bytes_q4(dh_bits: int, codes) -> bytes:
    """Q4_0 block as the layout defines it: fp16 scale little-endian, then byte j =
    code[j] | code[j+16] << 4."""
    out = bytes([dh_bits & 0xFF, dh_bits >> 8])
    return out + bytes(codes[j] | (codes[j + 16] << 4) for j in range(16))


def _block_bytes_q8(dh_bits: int, codes) -> bytes:
    return bytes([dh_bits & 0xFF, dh_bits >> 8]) + bytes((c & 0xFF) for c in codes)


# ------------------------------------------------------------------------------------
# fp32 -> fp16 (IEEE 754 binary16, round to nearest even)
# ------------------------------------------------------------------------------------
_LOW_PATTERNS = np.array(
    [0x0000, 0x0001, 0x0002, 0x0FFF, 0x1000, 0x1001, 0x1FFF, 0x2000, 0x2001, 0x3000,
     0x3FFF, 0x4000, 0x4001, 0x5FFF, 0x6000, 0x6001, 0x7FFF, 0x8000, 0x8001, 0x9000,
     0xBFFF, 0xC000, 0xC001, 0xDFFF, 0xE000, 0xEFFF, 0xF000, 0xF001, 0xFFFE, 0xFFFF],
    dtype=np.uint32)


def _check_fp16(oracle_mod, bits: np.ndarray):
    f = bits.view(np.float32)
    ours = oracle_mod.fp16_from_f32(f)
    with np.errstate(over="ignore"):
        ref = f.astype(np.float16).view(np.uint16)
    nan = np.isnan(f)
    bad = np.nonzero((ours != ref) & ~nan)[0]
    assert bad.size == 0, f"{bad.size} mismatches, first input bits {bits[bad[0]]:#010x}"
    # NaN stays NaN (payload is not specified by IEEE)
    assert np.all((ours[nan] & 0x7C00) == 0x7C00) and np.all((ours[nan] & 0x3FF) != 0)


def test_fp16_structured_sweep(oracle_mod):
    """Every sign / exponent / top-7-fraction pattern (upper 16 bits) crossed with the
    lower-16-bit patterns where round-to-nearest-even changes its mind."""
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    bits = (hi[:, None] | _LOW_PATTERNS[None, :]).reshape(-1)
    _check_fp16(oracle_mod, bits)


def test_fp16_random_patterns(oracle_mod):
    rng = np.random.default_rng(12345)
    bits = rng.integers(0, 1 << 32, size=1 << 22, dtype=np.uint64).astype(np.uint32)
    _check_fp16(oracle_mod, bits)


def test_fp16_matches_torch(oracle_mod):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 1 << 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    f = f[~np.isnan(f)]
    ref = torch.from_numpy(f.copy()).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle_mod.fp16_from_f32(f), ref)


@pytest.mark.slow
@pytest.mark.skipif(os.environ.get("GQ_EXHAUSTIVE_FP16") != "1",
                    reason="set GQ_EXHAUSTIVE_FP16=1 for all 2^32 inputs (about 10 minutes)")
def test_fp16_exhaustive(oracle_mod):
    for c in range(256):
        bits = np.arange(c << 24, (c + 1) << 24, dtype=np.uint64).astype(np.uint32)
        _check_fp16(oracle_mod, bits)


def test_fp16_spot_values(oracle_mod):
    cases = {
        65504.0: 0x7BFF,                 # largest finite half
        65519.99: 0x7BFF,                # just below the rounding boundary
        65520.0: 0x7C00,                 # halfway to 2^16: ties to even -> infinity
        2.0 ** -24: 0x0001,              # smallest subnormal
        2.0 ** -25: 0x0000,              # exactly half of it: ties to even -> 0
        1.5 * 2.0 ** -25: 0x0001,
        2.0 ** -14: 0x0400,              # smallest normal
        1.0 + 2.0 ** -11: 0x3C00,        # tie between 1 and 1+2^-10: even is 1
        1.0 + 3 * 2.0 ** -11: 0x3C02,    # tie between 1+2^-10 and 1+2^-9: even is the latter
        -2.0: 0xC000,
        0.1: 0x2E66,
    }
    for x, want in cases.items():
        got = int(oracle_mod.fp16_from_f32(np.array([x], np.float32))[0])
        assert got == want, (x, hex(got), hex(want))


def test_f32_from_fp16_all_patterns(oracle_mod):
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = oracle_mod.f32_from_fp16(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


# ------------------------------------------------------------------------------------
# Quantizer: closed-form blocks, ties, zero blocks, layout
# ------------------------------------------------------------------------------------
@pytest.mark.parametrize("e", [-14, -9, -6, 0, 5, 12])
def test_q4_0_closed_form_blocks(oracle_mod, e):
    """w = (c - 8) * s with s = 2^e and one element at +-7s: then max|w| = 7s, Delta =
    7s / 7 = s exactly, fp16(Delta) = 2^e and every code comes back as c."""
    rng = np.random.default_rng(100 + e)
    s = 2.0 ** e
    for trial in range(20):
        codes = rng.integers(1, 16, size=32)
        codes[rng.integers(32)] = 15 if trial % 2 == 0 else 1   # pin amax = 7s (either sign)
        w = ((codes - 8) * s).astype(np.float32)[None, :]
        got = oracle_mod.quantize("q4_0", w).tobytes()
        assert got == _block_bytes_q4(_pow2_fp16_bits(e), list(codes)), (e, trial)


def test_q4_0_ties_round_away_from_zero(oracle_mod):
    """w / Delta landing exactly on k + 1/2 rounds away from zero (C roundf)."""
    s = 0.25
    ratios = [7.0, 2.5, -2.5, 0.5, -0.5, 1.5, -1.5, 6.5, -6.5, 3.5, -3.5, 0.0]
    w = np.zeros(32, np.float32)
    w[: len(ratios)] = np.array(ratios) * s
    want_int = [7, 3, -3, 1, -1, 2, -2, 7, -7, 4, -4, 0] + [0] * 20
    codes = [v + 8 for v in want_int]
    got = oracle_mod.quantize("q4_0", w[None, :]).tobytes()
    assert got == _block_bytes_q4(_pow2_fp16_bits(-2), codes)


def test_q4_0_nibble_order(oracle_mod):
    """Byte j carries element j in its low nibble and element j+16 in its high nibble."""
    w = np.zeros(32, np.float32)
    w[0], w[16], w[31] = -7.0, 6.0, 7.0      # Delta = 1: codes 1, 14, 15
    blk = oracle_mod.quantize("q4_0", w[None, :])[0]
    assert blk[2] == 0xE1          # element 0 -> low nibble 1, element 16 -> high nibble 14
    assert blk[2 + 15] == 0xF8     # element 15 -> 8 (zero), element 31 -> 15


def test_zero_blocks(oracle_mod):
    z = np.zeros((3, 64), np.float32)
    q4 = oracle_mod.quantize("q4_0", z)
    q8 = oracle_mod.quantize("q8_0", z)
    assert q4.tobytes() == (bytes([0, 0]) + bytes([0x88] * 16)) * 6
    assert q8.tobytes() == bytes(34) * 6
    assert not np.any(oracle_mod.dequantize("q4_0", q4, 3, 64))


@pytest.mark.parametrize("e", [-14, -10, -3, 4])
def test_q8_0_closed_form_blocks(oracle_mod, e):
    rng = np.random.default_rng(200 + e)
    s = 2.0 ** e
    for trial in range(20):
        codes = rng.integers(-127, 128, size=32)
        codes[rng.integers(32)] = 127 if trial % 2 == 0 else -127
        w = (codes * s).astype(np.float32)[None, :]
        got = oracle_mod.quantize("q8_0", w).tobytes()
        assert got == _block_bytes_q8(_pow2_fp16_bits(e), list(codes)), (e, trial)


def test_q8_0_ties(oracle_mod):
    s = 2.0 ** -5
    ratios = [127.0, 2.5, -2.5, 100.5, -100.5, 0.5]
    w = np.zeros(32, np.float32)
    w[: len(ratios)] = np.array(ratios) * s
    codes = [127, 3, -3, 101, -101, 1] + [0] * 26
    got = oracle_mod.quantize("q8_0", w[None, :]).tobytes()
    assert got == _block_bytes_q8(_pow2_fp16_bits(-5), codes)


# ------------------------------------------------------------------------------------
# Dequantize and round trip
# ------------------------------------------------------------------------------------
def test_dequantize_hand_made_blocks(oracle_mod):
    """Codes the quantizer never emits (0, i.e. -8) still dequantize as (c - 8) * d."""
    d_bits = 0x3555   # 0.333251953125, a normal fp16 with a full fraction
    d = float(np.array([d_bits], np.uint16).view(np.float16)[0])
    codes = list(range(16)) + list(range(15, -1, -1))
    blk = np.frombuffer(_block_bytes_q4(d_bits, codes), np.uint8)
    got = oracle_mod.dequantize("q4_0", blk, 1, 32)[0]
    assert np.array_equal(got, np.array([(c - 8) * d for c in codes], np.float32))
    q8codes = [-128, 127, -1, 0, 1, 64, -64] + [5] * 25
    blk8 = np.frombuffer(_block_bytes_q8(d_bits, q8codes), np.uint8)
    got8 = oracle_mod.dequantize("q8_0", blk8, 1, 32)[0]
    assert np.array_equal(got8, np.array([c * d for c in q8codes], np.float32))


@pytest.mark.parametrize("t", ["q4_0", "q8_0"])
def test_roundtrip_idempotence(oracle_mod, t):
    """quant(dequant(quant(w))) == quant(w): max|What| = 7*dh (127*dh) exactly, so the
    second pass recovers the same scale and the same codes (blocks with a normal dh)."""
    W = workloads.weights(64, 512, seed=31).numpy()
    q1 = oracle_mod.quantize(t, W)
    wh = oracle_mod.dequantize(t, q1, 64, 512)
    q2 = oracle_mod.quantize(t, wh)
    assert np.array_equal(q1, q2)


@pytest.mark.parametrize("t,div", [("q4_0", 7.0), ("q8_0", 127.0)])
def test_quantization_error_bound(oracle_mod, t, div):
    """|w - What| <= Delta/2 + |code| * |Delta - fp16(Delta)|, per element."""
    W = workloads.weights(32, 1024, seed=41).numpy().astype(np.float64)
    q = oracle_mod.quantize(t, W.astype(np.float32))
    wh = oracle_mod.dequantize(t, q, 32, 1024).astype(np.float64)
    blocks = W.reshape(32, -1, 32)
    d = (np.abs(blocks).max(axis=2, keepdims=True) / div).astype(np.float32).astype(np.float64)
    dh = d.astype(np.float16).astype(np.float64)
    code_mag = np.abs(wh.reshape(blocks.shape)) / np.where(dh == 0, 1, dh)
    bound = d / 2 + code_mag * np.abs(d - dh) + 1e-12
    assert np.all(np.abs(blocks - wh.reshape(blocks.shape)) <= bound)


# ------------------------------------------------------------------------------------
# mul_mat: exact rational brute force, one-hot rows, block sums
# ------------------------------------------------------------------------------------
def _ulp32(v: float) -> Fraction:
    a = abs(np.float32(v))
    if a == 0:
        return Fraction(2) ** -149
    nxt = np.nextafter(np.float32(a), np.float32(np.inf))
    return Fraction(float(nxt)) - Fraction(float(a))


@pytest.mark.parametrize("t", ["q4_0", "q8_0"])
@pytest.mark.parametrize("M,N,K", [(1, 1, 32), (3, 5, 64), (8, 2, 96), (5, 7, 32), (2, 8, 96)])
def test_mul_mat_exact_rational(oracle_mod, t, M, N, K):
    """Y equals the exact sum of What * X, rounded to fp32, within half an fp32 ulp plus
    the fp64 summation bound K * 2^-53 * sum|terms|."""
    W = workloads.weights(M, K, seed=M * 100 + K).numpy()
    X = workloads.activations(N, K, seed=N * 100 + K).numpy()
    q = oracle_mod.quantize(t, W)
    wh = oracle_mod.dequantize(t, q, M, K)
    Y = oracle_mod.mul_mat(t, q, M, K, X)
    assert Y.shape == (N, M)
    for n in range(N):
        for m in range(M):
            terms = [Fraction(float(wh[m, k])) * Fraction(float(X[n, k])) for k in range(K)]
            exact = sum(terms, Fraction(0))
            slack = _ulp32(Y[n, m]) / 2 + K * Fraction(2) ** -53 * sum(abs(x) for x in terms)
            assert abs(Fraction(float(Y[n, m])) - exact) <= slack, (n, m)


@pytest.mark.parametrize("t", ["q4_0", "q8_0"])
def test_mul_mat_one_hot_returns_dequantized_rows(oracle_mod, t):
    """X = e_k picks column k of What exactly: Y[n][m] == What[m][k] bit for bit."""
    M, K = 7, 96
    W = workloads.weights(M, K, seed=5).numpy()
    q = oracle_mod.quantize(t, W)
    wh = oracle_mod.dequantize(t, q, M, K)
    ks = [0, 1, 15, 16, 31, 32, 50, 95]
    X = np.zeros((len(ks), K), np.float32)
    for n, k in enumerate(ks):
        X[n, k] = 1.0
    Y = oracle_mod.mul_mat(t, q, M, K, X)
    for n, k in enumerate(ks):
        assert np.array_equal(Y[n], wh[:, k]), k


def test_mul_mat_block_of_ones(oracle_mod):
    """X = 1 over block b only: Y[m] = dh * sum_i (code_i - 8), an exact small multiple."""
    M, K = 4, 128
    W = workloads.weights(M, K, seed=9).numpy()
    q = oracle_mod.quantize("q4_0", W)
    for b in range(K // 32):
        X = np.zeros((1, K), np.float32)
        X[0, 32 * b: 32 * b + 32] = 1.0
        Y = oracle_mod.mul_mat("q4_0", q, M, K, X)[0]
        for m in range(M):
            blk = q[m, 18 * b: 18 * b + 18]
            dh = float(blk[:2].view(np.float16)[0])
            codes = [int(v) & 0xF for v in blk[2:]] + [int(v) >> 4 for v in blk[2:]]
            assert Y[m] == np.float32(dh * sum(c - 8 for c in codes))


def test_mul_mat_matches_fp64_matmul(oracle_mod):
    """Context check at a mid size: the oracle agrees with numpy's fp64 matmul of the
    dequantized weights to within fp32 rounding."""
    M, N, K = 96, 6, 1024
    W = workloads.weights(M, K, seed=77).numpy()
    X = workloads.activations(N, K, seed=78).numpy()
    q = oracle_mod.quantize("q4_0", W)
    wh = oracle_mod.dequantize("q4_0", q, M, K).astype(np.float64)
    ref = X.astype(np.float64) @ wh.T
    Y = oracle_mod.mul_mat("q4_0", q, M, K, X)
    assert np.all(np.abs(Y - ref) <= np.abs(ref) * 2.0 ** -23 + 1e-12)


def test_mul_mat_rows_subset(oracle_mod):
    M, N, K = 40, 3, 256
    W = workloads.weights(M, K, seed=3).numpy()
    X = workloads.activations(N, K, seed=4).numpy()
    q = oracle_mod.quantize("q8_0", W)
    full = oracle_mod.mul_mat("q8_0", q, M, K, X)
    rows = [0, 7, 39, 12]
    assert np.array_equal(oracle_mod.mul_mat_rows("q8_0", q, M, K, X, rows), full[:, rows])


# ------------------------------------------------------------------------------------
# mul_mat with quantized activations (integer block sums)
# ------------------------------------------------------------------------------------
@pytest.mark.parametrize("t", ["q4_0", "q8_0"])
@pytest.mark.parametrize("M,N,K", [(1, 1, 32), (3, 4, 64), (6, 2, 96)])
def test_mul_mat_q8x_exact_rational(oracle_mod, t, M, N, K):
    """Y equals the exact sum over blocks of Delta_w * Delta_x * sum q_i q_x,i, written
    out here from the block bytes (codes, scales) with rational arithmetic."""
    W = workloads.weights(M, K, seed=7 * M + K).numpy()
    X = workloads.activations(N, K, seed=11 * N + K).numpy()
    q = oracle_mod.quantize(t, W)
    xq = oracle_mod.quantize("q8_0", X)
    Y = oracle_mod.mul_mat_q8x(t, q, M, K, X)
    bb = 18 if t == "q4_0" else 34
    for n in range(N):
        for m in range(M):
            exact = Fraction(0)
            terms = []
            for b in range(K // 32):
                wb = q[m, bb * b: bb * b + bb]
                xb = xq[n, 34 * b: 34 * b + 34]
                if t == "q4_0":
                    codes = [(int(wb[2 + (i & 15)]) >> (4 if i >= 16 else 0) & 0xF) - 8
                             for i in range(32)]
                else:
                    codes = [int(v) - 256 if v > 127 else int(v) for v in wb[2:]]
                xc = [int(v) - 256 if v > 127 else int(v) for v in xb[2:]]
                s_b = sum(a * c for a, c in zip(codes, xc))
                term = (Fraction(float(wb[:2].view(np.float16)[0])) *
                        Fraction(float(xb[:2].view(np.float16)[0])) * s_b)
                terms.append(term)
                exact += term
            slack = _ulp32(Y[n, m]) / 2 + (K // 32) * Fraction(2) ** -53 * sum(abs(x) for x in terms)
            assert abs(Fraction(float(Y[n, m])) - exact) <= slack, (n, m)


@pytest.mark.parametrize("t", ["q4_0", "q8_0"])
def test_mul_mat_q8x_equals_mul_mat_of_dequantized_x(oracle_mod, t):
    """Delta_w Delta_x sum q q_x = sum What * Xhat with Xhat the Q8_0-dequantized X, every
    product exact: the two oracle paths agree to fp32 rounding."""
    M, N, K = 24, 3, 512
    W = workloads.weights(M, K, seed=12).numpy()
    X = workloads.activations(N, K, seed=13).numpy()
    q = oracle_mod.quantize(t, W)
    xhat = oracle_mod.dequantize("q8_0", oracle_mod.quantize("q8_0", X), N, K)
    a = oracle_mod.mul_mat_q8x(t, q, M, K, X).astype(np.float64)
    b = oracle_mod.mul_mat(t, q, M, K, xhat).astype(np.float64)
    assert np.all(np.abs(a - b) <= np.abs(b) * 2.0 ** -23 + 1e-30)


def test_mul_mat_q8x_exact_when_x_is_representable(oracle_mod):
    """X whose blocks are integers times a power of two with max |code| = 127 quantizes
    without error, so the quantized-activation product equals the plain one."""
    M, N, K = 9, 2, 256
    rng = np.random.default_rng(5)
    codes = rng.integers(-127, 128, size=(N, K))
    codes[:, ::32] = 127                                   # every block reaches 127
    X = (codes * 2.0 ** -7).astype(np.float32)
    W = workloads.weights(M, K, seed=14).numpy()
    for t in ("q4_0", "q8_0"):
        q = oracle_mod.quantize(t, W)
        a = oracle_mod.mul_mat_q8x(t, q, M, K, X).astype(np.float64)
        b = oracle_mod.mul_mat(t, q, M, K, X).astype(np.float64)
        assert np.all(np.abs(a - b) <= np.abs(b) * 2.0 ** -23 + 1e-30), t


# ------------------------------------------------------------------------------------
# Figures the pages print
# ------------------------------------------------------------------------------------
# ------------------------------------------------------------------------------------
# Fused adjacent steps: RMSNorm ahead of the product, SwiGLU after it
# ("Development Guide for Small AI Models (TinyLLaMA, etc.) Using C++", sections 4.1, 4.4)
# ------------------------------------------------------------------------------------
@pytest.mark.parametrize("t", ["q4_0", "q8_0"])
def test_rmsnorm_one_hot_closed_form(oracle_mod, t):
    """eps = 0, gamma = 1, x = a e_k: mean(x^2) = a^2 / K, so RMSNorm(x) = sign(a) sqrt(K) e_k
    and Y[m] = sign(a) sqrt(K) What[m][k], within an fp32 rounding."""
    M, K = 6, 96
    W = workloads.weights(M, K, seed=81).numpy()
    q = oracle_mod.quantize(t, W)
    wh = oracle_mod.dequantize(t, q, M, K).astype(np.float64)
    gamma = np.ones(K, np.float32)
    for k, a in [(0, 1.0), (17, -3.5), (95, 0.002)]:
        X = np.zeros((1, K), np.float32)
        X[0, k] = a
        Y = oracle_mod.mul_mat_rmsnorm(t, q, M, K, X, gamma, 0.0)[0].astype(np.float64)
        ref = np.sign(a) * np.sqrt(K) * wh[:, k]
        assert np.all(np.abs(Y - ref) <= np.abs(ref) * 2.0 ** -23), (k, a)


def test_rmsnorm_scale_invariant_and_gamma_linear(oracle_mod):
    """eps = 0: scaling X by a power of two leaves Y unchanged bit for bit; scaling gamma by
    a power of two scales Y by it exactly."""
    M, N, K = 9, 3, 256
    W = workloads.weights(M, K, seed=82).numpy()
    X = workloads.activations(N, K, seed=83).numpy()
    q = oracle_mod.quantize("q4_0", W)
    gamma = (1.0 + 0.1 * np.random.default_rng(84).standard_normal(K)).astype(np.float32)
    Y = oracle_mod.mul_mat_rmsnorm("q4_0", q, M, K, X, gamma, 0.0)
    for s in (8.0, 1.0 / 16.0):
        assert np.array_equal(oracle_mod.mul_mat_rmsnorm("q4_0", q, M, K, X * np.float32(s), gamma, 0.0), Y)
    assert np.array_equal(oracle_mod.mul_mat_rmsnorm("q4_0", q, M, K, X, gamma * np.float32(2.0), 0.0),
                          Y * np.float32(2.0))


def test_rmsnorm_eps_dominates(oracle_mod):
    """eps far above mean(x^2): RMSNorm(x) -> x * gamma / sqrt(eps), so Y equals the pinned
    mul_mat of X * gamma divided by sqrt(eps) to within the neglected mean(x^2) / eps."""
    M, N, K = 5, 2, 128
    W = workloads.weights(M, K, seed=85).numpy()
    X = workloads.activations(N, K, seed=86).numpy()
    q = oracle_mod.quantize("q8_0", W)
    gamma = np.linspace(0.5, 1.5, K, dtype=np.float32)
    eps = 1.0e12
    Y = oracle_mod.mul_mat_rmsnorm("q8_0", q, M, K, X, gamma, eps).astype(np.float64)
    ref = oracle_mod.mul_mat("q8_0", q, M, K, X * gamma).astype(np.float64) / np.sqrt(eps)
    assert np.all(np.abs(Y - ref) <= np.abs(ref) * 1e-6 + 1e-30)


@pytest.mark.parametrize("t", ["q4_0", "q8_0"])
def test_swiglu_one_hot_closed_form(oracle_mod, t):
    """x = a e_k: g = What_gate[m][k] a and u = What_up[m][k] a exactly, so
    H[m] = g / (1 + e^-g) * u (computed here with Python's math, in fp64)."""
    import math
    M, K = 7, 64
    qg = oracle_mod.quantize(t, workloads.weights(M, K, seed=87).numpy())
    qu = oracle_mod.quantize(t, workloads.weights(M, K, seed=88).numpy())
    wg = oracle_mod.dequantize(t, qg, M, K).astype(np.float64)
    wu = oracle_mod.dequantize(t, qu, M, K).astype(np.float64)
    for k, a in [(3, 1.0), (40, -250.0), (63, 900.0)]:
        X = np.zeros((1, K), np.float32)
        X[0, k] = a
        H = oracle_mod.mul_mat_swiglu(t, qg, qu, M, K, X)[0].astype(np.float64)
        for m in range(M):
            g, u = wg[m, k] * a, wu[m, k] * a
            ref = g / (1.0 + math.exp(-g)) * u
            assert abs(H[m] - ref) <= abs(ref) * 2.0 ** -23 + 1e-45, (k, a, m)


def test_swiglu_zero_input_and_roles(oracle_mod):
    """X = 0 gives H = 0; with the same matrix as gate and up, H = Swish(g) g against the
    pinned mul_mat, and exchanging gate and up changes the result."""
    M, N, K = 6, 2, 96
    qg = oracle_mod.quantize("q4_0", workloads.weights(M, K, seed=89).numpy())
    qu = oracle_mod.quantize("q4_0", workloads.weights(M, K, seed=90).numpy())
    assert not oracle_mod.mul_mat_swiglu("q4_0", qg, qu, M, K, np.zeros((N, K), np.float32)).any()
    X = workloads.activations(N, K, seed=91).numpy() * np.float32(10.0)
    g = oracle_mod.mul_mat("q4_0", qg, M, K, X).astype(np.float64)
    H = oracle_mod.mul_mat_swiglu("q4_0", qg, qg, M, K, X).astype(np.float64)
    ref = g / (1.0 + np.exp(-g)) * g
    assert np.all(np.abs(H - ref) <= np.abs(ref) * 1e-6 + 1e-30)
    assert not np.array_equal(oracle_mod.mul_mat_swiglu("q4_0", qg, qu, M, K, X),
                              oracle_mod.mul_mat_swiglu("q4_0", qu, qg, M, K, X))


def test_fused_rows_subsets(oracle_mod):
    M, N, K = 20, 2, 128
    qg = oracle_mod.quantize("q4_0", workloads.weights(M, K, seed=92).numpy())
    qu = oracle_mod.quantize("q4_0", workloads.weights(M, K, seed=93).numpy())
    X = workloads.activations(N, K, seed=94).numpy()
    gamma = np.ones(K, np.float32)
    rows = [0, 19, 7]
    assert np.array_equal(oracle_mod.mul_mat_rmsnorm_rows("q4_0", qg, M, K, X, gamma, 1e-5, rows),
                          oracle_mod.mul_mat_rmsnorm("q4_0", qg, M, K, X, gamma, 1e-5)[:, rows])
    assert np.array_equal(oracle_mod.mul_mat_swiglu_rows("q4_0", qg, qu, M, K, X, rows),
                          oracle_mod.mul_mat_swiglu("q4_0", qg, qu, M, K, X)[:, rows])


def test_page_facts():
    import oracle
    facts = json.load(open(GOLDEN))
    blk = facts["q4_0_block"]
    assert oracle.block_bytes("q4_0") == blk["scale_bytes"] + blk["code_bytes"] == 18
    assert blk["weights_per_block"] == 32
    # 4.5 bits per weight; the TinyLLaMA decode set (every matmul of one step) at Q4_0
    # is "about 600 MB" as the pages say of 4-bit TinyLLaMA.
    n_weights = sum(s.M * s.K for s in workloads.tinyllama_decode_set())
    q4_bytes = n_weights // 32 * oracle.block_bytes("q4_0")
    assert q4_bytes == 581_861_376
    approx = facts["tinyllama_4bit_bytes"]["approx_bytes"]
    assert abs(q4_bytes - approx) / approx < 0.1
    # fp16 of the same set plus the 32000 x 2048 embedding table is the "2.2 GB"
    fp16 = (n_weights + 32000 * 2048) * 2
    assert abs(fp16 - facts["tinyllama_4bit_bytes"]["fp16_bytes"]) / 2.2e9 < 0.05
    # INT4 is 1/8 of FP32 before the per-block scale; with it Q4_0 is 18/128 of FP32.
    assert facts["size_ratios_vs_fp32"]["int4"] == 16 / 128
    assert oracle.block_bytes("q8_0") / 128 == pytest.approx(0.25 + 2 / 128)
