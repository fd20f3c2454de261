"""Q4_K super-blocks on the GPU, through the C ABI, against the CPU oracle.

The layout is the published GGUF Q4_K block (the pages name the format without one:
"Development Guide for Small AI Models (TinyLLaMA, etc.) Using C++", section 6; "A Complete
Guide to llama.cpp and Customization with C++", section 2.2): 256 weights in eight
sub-blocks of 32, What = d sc_j q - dmin m_j.

Bars:
  - gq_quantize_q4_k and gq_dequantize: bit-exact;
  - mul_mat on quantizer output: |Y - Y_oracle| <= 1e-3 ||X[n]||_2 ||What[m]||_2;
  - mul_mat on arbitrary super-block bytes: the same plus the fp32 rounding of the
    format's two partial sums, (K / 256 + 32) 2^-23 sum_k (|D_j q_k| + |M_j|) |x_k|
    (where d sc q and dmin m cancel, What can be far smaller than either term);
  - one-hot X returns What exactly on the CUDA-core decode kernels (and bf16(What) on the
    tensor-core decode and the prefill GEMM, which tests/test_gpu_parity.py covers for all
    three types).
Token counts route as for the other types: N <= 2 (and shapes the tensor-core paths do
not take) on the CUDA-core kernels, 3..64 on the tensor-core decode, >= 65 on the GEMM.
"""
import numpy as np
import pytest
import torch

from block_quantized_matmul_gq_gb300 import workloads

pytestmark = pytest.mark.gpu

TOL = 1e-3
T = "q4_k"


def _tol(X, What, extra=None):
    xn = np.linalg.norm(np.asarray(X, np.float64), axis=1)
    wn = np.linalg.norm(np.asarray(What, np.float64), axis=1)
    tol = TOL * xn[:, None] * wn[None, :]
    return tol if extra is None else tol + extra


def _check(Y, Y_ref, tol, where):
    Y = np.asarray(Y, np.float64)
    assert np.isfinite(Y).all(), f"{where}: non-finite output"
    err = np.abs(Y - np.asarray(Y_ref, np.float64))
    bad = err > tol
    if bad.any():
        n, m = np.argwhere(bad)[0]
        raise AssertionError(f"{where}: {bad.sum()} out of tolerance, first (n={n}, m={m}) "
                             f"err={err[n, m]:.3e} tol={tol[n, m]:.3e}")


def _rounding_slack(oracle_mod, q, M, K, X):
    """(K / 256 + 32) 2^-23 sum_k (|D_j q_k| + |M_j|) |x_k|, with D_j q_k and M_j read from
    the oracle's own dequantization of the blocks with dmin (resp. d) set to zero."""
    blk = q.reshape(M, K // 256, 144)
    no_min = blk.copy()
    no_min[:, :, 2:4] = 0
    no_scale = blk.copy()
    no_scale[:, :, 0:2] = 0
    Dq = np.abs(oracle_mod.dequantize(T, no_min.reshape(M, -1), M, K).astype(np.float64))
    Mj = np.abs(oracle_mod.dequantize(T, no_scale.reshape(M, -1), M, K).astype(np.float64))
    ax = np.abs(np.asarray(X, np.float64))
    return (K / 256 + 32) * 2.0 ** -23 * (ax @ (Dq + Mj).T)


# ------------------------------------------------------------------------------------
# quantize / dequantize: bit-exact
# ------------------------------------------------------------------------------------
@pytest.mark.parametrize("M,K", [(1, 256), (3, 512), (37, 2304), (64, 2048), (129, 5632),
                                 (5, 11008)])
def test_quantize_bit_exact(gq_lib, oracle_mod, cuda_dev, M, K):
    W = workloads.weights(M, K, seed=M * 7 + K).numpy()
    got = gq_lib.quantize(torch.from_numpy(W).to(cuda_dev), T).cpu().numpy()
    assert got.shape == (M, K // 256 * 144)
    assert np.array_equal(got, oracle_mod.quantize(T, W))


def test_quantize_special_rows(gq_lib, oracle_mod, cuda_dev):
    """Zeros (+0 and -0), a negative constant, all-positive and all-negative sub-blocks,
    exact ties of step / d and of (w + M) / D, fp16-subnormal d, fp32-subnormal weights,
    large magnitudes."""
    rng = np.random.default_rng(41)
    rows = [np.zeros(256, np.float32), np.full(256, -0.0, np.float32),
            np.full(256, -3.0, np.float32)]
    r = np.zeros(256, np.float32)                 # ties (hand-worked in the oracle pins)
    r[224], r[255] = 0.0, 945 * 2.0 ** -6
    r[0], r[17] = 0.0, 157.5 * 2.0 ** -6
    rows.append(r)
    r = (rng.integers(0, 16, 256) * 2.0 ** -7).astype(np.float32)       # codes on the grid
    r[32:64] = -r[32:64]
    rows.append(r)
    rows.append(np.abs(rng.standard_normal(256)).astype(np.float32))      # all positive
    rows.append(-np.abs(rng.standard_normal(256)).astype(np.float32))     # all negative
    rows.append((rng.standard_normal(256) * 1e-6).astype(np.float32))     # subnormal fp16 d
    rows.append((rng.standard_normal(256) * 1e-41).astype(np.float32))    # subnormal fp32 w
    rows.append((rng.standard_normal(256) * 1e4).astype(np.float32))
    mixed = rng.standard_normal(256).astype(np.float32)
    mixed[::2] = 0.0
    mixed[1::4] = -0.0
    rows.append(mixed)
    W = np.stack(rows)
    got = gq_lib.quantize(torch.from_numpy(W).to(cuda_dev), T).cpu().numpy()
    assert np.array_equal(got, oracle_mod.quantize(T, W))


def test_dequantize_bit_exact_on_arbitrary_bytes(gq_lib, oracle_mod, cuda_dev):
    M, K = 48, 2304
    q = workloads.q4k_superblocks(M, K, seed=9)
    got = gq_lib.dequantize(torch.from_numpy(q).to(cuda_dev), T, M, K).cpu().numpy()
    ref = oracle_mod.dequantize(T, q, M, K)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


# ------------------------------------------------------------------------------------
# mul_mat
# ------------------------------------------------------------------------------------
# N <= 2: the streaming kernel (M leaves ragged 4-row tiles; K = 11008 is 43 super-blocks,
# a partial last column group; K = 256 one super-block; small M splits columns between
# warps). N = 3..64: the tensor-core decode; N = 70: the prefill GEMM.
STREAM = [(1, 256, 1), (7, 2048, 1), (300, 2048, 1), (1000, 2048, 2), (129, 5632, 3),
          (64, 11008, 4), (33, 4096, 5), (257, 1024, 9), (2048, 2048, 1), (200, 11008, 1),
          (65, 4096, 2), (96, 2048, 16), (50, 2048, 70)]
# Generic kernel: K too large for the activation records in shared memory.
GENERIC = [(8, 65536, 1), (3, 40960, 2)]


def _run(gq_lib, oracle_mod, dev, M, K, N, seed, q=None, X=None, offset=0):
    if q is None:
        q = oracle_mod.quantize(T, workloads.weights(M, K, seed=seed).numpy())
    if X is None:
        X = workloads.activations(N, K, seed=seed + 1).numpy()
    if offset:   # X starts `offset` floats into its buffer: not 16-byte aligned
        buf = torch.zeros(N * K + offset, device=dev)
        buf[offset:] = torch.from_numpy(X).reshape(-1).to(dev)
        Xd = buf[offset:].view(N, K)
    else:
        Xd = torch.from_numpy(X).to(dev)
    Y = gq_lib.mul_mat(torch.from_numpy(q).to(dev), T, M, K, Xd).cpu().numpy()
    assert gq_lib.get_last_error() == 0
    return q, X, Y


@pytest.mark.parametrize("M,K,N", STREAM + GENERIC)
def test_mul_mat_matches_oracle(gq_lib, oracle_mod, cuda_dev, M, K, N):
    q, X, Y = _run(gq_lib, oracle_mod, cuda_dev, M, K, N, seed=M + K + N)
    assert Y.shape == (N, M)
    _check(Y, oracle_mod.mul_mat(T, q, M, K, X), _tol(X, oracle_mod.dequantize(T, q, M, K)),
           f"M={M} K={K} N={N}")


@pytest.mark.parametrize("N", [1, 2])
def test_mul_mat_misaligned_x_takes_the_generic_kernel(gq_lib, oracle_mod, cuda_dev, N):
    M, K = 70, 2048
    q, X, Y = _run(gq_lib, oracle_mod, cuda_dev, M, K, N, seed=5, offset=1)
    _check(Y, oracle_mod.mul_mat(T, q, M, K, X), _tol(X, oracle_mod.dequantize(T, q, M, K)),
           f"misaligned N={N}")


@pytest.mark.parametrize("N,offset", [(2, 0), (2, 1)])
def test_mul_mat_one_hot_is_exact(gq_lib, oracle_mod, cuda_dev, N, offset):
    """X = e_k returns column k of What bit for bit on the CUDA-core kernels: the streaming
    kernel with two tokens and with one, the generic kernel (offset X)."""
    M, K = 77, 2048
    q = oracle_mod.quantize(T, workloads.weights(M, K, seed=6).numpy())
    What = oracle_mod.dequantize(T, q, M, K)
    ks = [0, 1, 31, 32, 63, 64, 127, 128, 255, 256, 1000, 1791, 2047, 17, 200, 1500]
    for i in range(0, len(ks), N):
        group = ks[i:i + N]
        X = np.zeros((len(group), K), np.float32)
        for n, k in enumerate(group):
            X[n, k] = 1.0
        _, _, Y = _run(gq_lib, oracle_mod, cuda_dev, M, K, len(group), 0, q=q, X=X, offset=offset)
        for n, k in enumerate(group):
            assert np.array_equal(Y[n], What[:, k]), k
    # one token alone
    X = np.zeros((1, K), np.float32)
    X[0, 700] = 1.0
    _, _, Y = _run(gq_lib, oracle_mod, cuda_dev, M, K, 1, 0, q=q, X=X, offset=offset)
    assert np.array_equal(Y[0], What[:, 700])


@pytest.mark.parametrize("M,K,N,offset", [(64, 2048, 1, 0), (200, 2048, 3, 0),
                                          (40, 5632, 5, 0), (48, 2304, 2, 1)])
def test_mul_mat_arbitrary_superblocks(gq_lib, oracle_mod, cuda_dev, M, K, N, offset):
    """Super-block bytes the quantizer never writes (extreme, subnormal, zero and negative
    d / dmin, every scale and min at 63), every row kind at every tile position."""
    q = workloads.q4k_superblocks(M, K, seed=M + N)
    X = workloads.activations(N, K, seed=K + N).numpy()
    _, _, Y = _run(gq_lib, oracle_mod, cuda_dev, M, K, N, 0, q=q, X=X, offset=offset)
    What = oracle_mod.dequantize(T, q, M, K)
    _check(Y, oracle_mod.mul_mat(T, q, M, K, X),
           _tol(X, What, _rounding_slack(oracle_mod, q, M, K, X)), f"arbitrary M={M} N={N}")
    zero_rows = [m for m in range(M) if m % 8 == 3]
    assert not Y[:, zero_rows].any()          # d = dmin = +-0: exactly zero


def test_mul_mat_scaled_activations(gq_lib, oracle_mod, cuda_dev):
    M, K = 50, 2048
    rng = np.random.default_rng(3)
    X = rng.standard_normal((4, K)).astype(np.float32)
    X[0] *= 3e4
    X[1] *= 1e-30
    X[2, ::64] *= 1e3
    X[3, :256] = 0.0
    q, X, Y = _run(gq_lib, oracle_mod, cuda_dev, M, K, 4, seed=12, X=X)
    _check(Y, oracle_mod.mul_mat(T, q, M, K, X), _tol(X, oracle_mod.dequantize(T, q, M, K)),
           "scaled")


@pytest.mark.parametrize("N", [1, 5])
def test_batched_mixed_shapes(gq_lib, oracle_mod, cuda_dev, N):
    """One batched call over problems of different shapes, one of them with X that only the
    generic kernel takes (not 16-byte aligned)."""
    shapes = [(2048, 2048), (256, 2048), (5632, 2048), (2048, 5632), (3, 256), (100, 4096)]
    items, refs = [], []
    for j, (M, K) in enumerate(shapes):
        q = oracle_mod.quantize(T, workloads.weights(M, K, seed=300 + j).numpy())
        X = workloads.activations(N, K, seed=400 + j).numpy()
        if j == 4:
            buf = torch.zeros(N * K + 1, device=cuda_dev)
            buf[1:] = torch.from_numpy(X).reshape(-1).to(cuda_dev)
            Xd = buf[1:].view(N, K)
        else:
            Xd = torch.from_numpy(X).to(cuda_dev)
        Y = torch.full((N, M), float("nan"), device=cuda_dev)
        items.append((torch.from_numpy(q).to(cuda_dev), M, K, Xd, Y))
        refs.append((q, M, K, X, Y))
    gq_lib.mul_mat_batched(gq_lib.make_problems(items), T, N)
    assert gq_lib.get_last_error() == 0
    for q, M, K, X, Y in refs:
        _check(Y.cpu().numpy(), oracle_mod.mul_mat(T, q, M, K, X),
               _tol(X, oracle_mod.dequantize(T, q, M, K)), f"batched {M}x{K}")


def test_deterministic(gq_lib, cuda_dev):
    M, K = 3000, 5632
    q = gq_lib.quantize(workloads.weights(M, K, 1, device=cuda_dev), T)
    for N in (1, 3):
        X = workloads.activations(N, K, 2, device=cuda_dev)
        a = gq_lib.mul_mat(q, T, M, K, X)
        b = gq_lib.mul_mat(q, T, M, K, X)
        assert torch.equal(a, b)


def test_tinyllama_decode_step_q4_k_full_size(gq_lib, oracle_mod, cuda_dev):
    """All 155 matmuls of the TinyLLaMA decode step in Q4_K at N = 1, batched as the
    benchmark times them; sampled rows against the oracle, their blocks bit-exact."""
    from test_gpu_parity import _sampled_step_check
    _sampled_step_check(gq_lib, oracle_mod, cuda_dev, 2, T, 1, workloads.tinyllama_decode_set(),
                        rows_per_mat=4)


def test_tinyllama_prefill_q4_k_full_size(gq_lib, oracle_mod, cuda_dev):
    """gate / down / lm_head at N = 512 tokens in Q4_K on the tensor-core GEMM."""
    from test_gpu_parity import _sampled_step_check
    _sampled_step_check(gq_lib, oracle_mod, cuda_dev, 4, T, 512, workloads.tinyllama_prefill_set(),
                        rows_per_mat=3)


@pytest.mark.parametrize("M,K,N", [(200, 2048, 70), (64, 1024, 300), (1000, 2304, 512)])
def test_gemm_arbitrary_superblocks(gq_lib, oracle_mod, cuda_dev, M, K, N):
    """Hand-made super-blocks through the prefill GEMM (in its split-K and plain forms).
    The GEMM forms What exactly as gq_dequantize does and rounds it to bf16, so the
    plain tolerance applies."""
    q = workloads.q4k_superblocks(M, K, seed=M + K + N)
    X = workloads.activations(N, K, seed=N + 3).numpy()
    _, _, Y = _run(gq_lib, oracle_mod, cuda_dev, M, K, N, 0, q=q, X=X)
    _check(Y, oracle_mod.mul_mat(T, q, M, K, X), _tol(X, oracle_mod.dequantize(T, q, M, K)),
           f"gemm arbitrary M={M} K={K} N={N}")
    zero_rows = [m for m in range(M) if m % 8 == 3]
    assert not Y[:, zero_rows].any()


@pytest.mark.parametrize("M,K,N", [(300, 2048, 1), (64, 5632, 3), (40, 2048, 70)])
def test_rmsnorm_and_swiglu_composites(gq_lib, oracle_mod, cuda_dev, M, K, N):
    from test_gpu_parity import _check_swiglu, _gamma, check_tolerance
    q = oracle_mod.quantize(T, workloads.weights(M, K, seed=M + K).numpy())
    X = workloads.activations(N, K, seed=N + 7).numpy() * np.float32(3.0)
    gamma, eps = _gamma(K, K), 1e-5
    Y = gq_lib.mul_mat_rmsnorm(torch.from_numpy(q).to(cuda_dev), T, M, K,
                               torch.from_numpy(X).to(cuda_dev),
                               torch.from_numpy(gamma).to(cuda_dev), eps).cpu().numpy()
    x64 = X.astype(np.float64)
    xhat = x64 / np.sqrt((x64 ** 2).mean(axis=1, keepdims=True) + eps) * gamma
    check_tolerance(Y, oracle_mod.mul_mat_rmsnorm(T, q, M, K, X, gamma, eps),
                    oracle_mod.dequantize(T, q, M, K), xhat, f"rmsnorm q4_k {M} {K} {N}")
    qu = oracle_mod.quantize(T, workloads.weights(M, K, seed=M + 3 * K).numpy())
    H = gq_lib.mul_mat_swiglu(torch.from_numpy(q).to(cuda_dev), torch.from_numpy(qu).to(cuda_dev),
                              T, M, K, torch.from_numpy(X).to(cuda_dev)).cpu().numpy()
    assert gq_lib.get_last_error() == 0
    _check_swiglu(oracle_mod, T, q, qu, M, K, X, H, f"swiglu q4_k {M} {K} {N}")


def test_rejections(gq_lib, cuda_dev):
    q = torch.zeros((4, 144), dtype=torch.uint8, device=cuda_dev)
    X = torch.zeros((1, 256), device=cuda_dev)
    with pytest.raises(gq_lib.GQError) as e:
        gq_lib.mul_mat_q8x(q, T, 4, 256, X)
    assert e.value.status == -3
    with pytest.raises(gq_lib.GQError) as e:
        gq_lib.mul_mat(torch.zeros((4, 162), dtype=torch.uint8, device=cuda_dev), T, 4, 288,
                       torch.zeros((1, 288), device=cuda_dev))
    assert e.value.status == -2
    with pytest.raises(gq_lib.GQError) as e:
        gq_lib.quantize(torch.zeros((2, 288), device=cuda_dev), T)
    assert e.value.status == -2
