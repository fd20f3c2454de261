"""Hand-made blocks through every mul_mat path, against the oracle.

The quantizer never writes some blocks that the public layout allows, and every kernel
must still accept them ("A Complete Guide to llama.cpp and Customization with C++",
section 2.2 gives the 4-bit codes the range [-8, 7], which includes -8 = code 0 although
Delta = max|w| / 7 never produces it):
  - Q4_0 code 0 (What = -8 d) and Q8_0 code -128;
  - fp16 scales that are negative, +-0, subnormal, or as large as 65504;
  - rows in which every block is such a block.
workloads.edge_blocks draws these bytes directly. Each path is reached by a shape that
routes to it (the routing rules are in include/gq.h): the streaming CUDA-core decode
(N = 1, 2), the generic kernel (K % 256 != 0), the tensor-core decode in its scaled form
(Q4_0, N <= 16) and its bf16 form (N = 17..64, and Q8_0), the prefill GEMM in 256-token
tiles, in 512-token tiles and split along K in clusters, the quantized-activation entry
point and both fused entry points.

Bar: per element |Y - Y_oracle| <= 1e-3 ||X[n]||_2 ||What[m]||_2 (the mul_mat tolerance),
the fp32 accumulation bound for gq_mul_mat_q8x against its own definition, and exact
equality where a path promises it (one-hot X).
"""
import numpy as np
import pytest
import torch

from block_quantized_matmul_gq_gb300 import workloads

pytestmark = pytest.mark.gpu

TOL = 1e-3


def _tol_check(Y, Y_ref, What, X, where):
    Y = np.asarray(Y, np.float64)
    xn = np.linalg.norm(np.asarray(X, np.float64), axis=1)
    wn = np.linalg.norm(np.asarray(What, np.float64), axis=1)
    tol = TOL * xn[:, None] * wn[None, :]
    err = np.abs(Y - np.asarray(Y_ref, np.float64))
    assert np.isfinite(Y).all(), f"{where}: non-finite output"
    bad = err > tol
    if bad.any():
        n, m = np.argwhere(bad)[0]
        raise AssertionError(f"{where}: {bad.sum()} out of tolerance, first (n={n}, m={m}, "
                             f"row kind {m % 8}) err={err[n, m]:.3e} tol={tol[n, m]:.3e}")


def _rows(M):
    """All rows of small problems; for large ones the first and last 24 rows (every row
    kind at both ends, the ragged last tile) and rows around tile boundaries."""
    if M <= 1200:
        return np.arange(M)
    edges = [np.arange(24), np.arange(M - 24, M)]
    for b in (128, 256, 1024, M // 2 // 128 * 128):
        edges.append(np.arange(b - 8, b + 8))
    return np.unique(np.concatenate(edges))


def _run(gq_lib, oracle_mod, dev, t, M, K, N, seed, X=None):
    q = workloads.edge_blocks(t, M, K, seed)
    if X is None:
        X = workloads.activations(N, K, seed=seed + 1).numpy()
    Y = gq_lib.mul_mat(torch.from_numpy(q).to(dev), t, M, K,
                       torch.from_numpy(X).to(dev)).cpu().numpy()
    assert gq_lib.get_last_error() == 0
    rows = _rows(M)
    Y_ref = oracle_mod.mul_mat_rows(t, q, M, K, X, rows)
    What = oracle_mod.dequantize(t, q[rows], len(rows), K)
    return Y[:, rows], Y_ref, What, X, q


# (M, K, N, path). Routing: N <= 2 and K % 256 == 0 streaming; K % 256 != 0 generic;
# 3..64 tensor-core decode (scaled form for Q4_0 up to 16 tokens); N >= 65 the GEMM:
# 256-token tiles when they fill the SMs, 512-token tiles when those need no more waves
# than half as many 256-token waves, split-K clusters when the tiles fill under half the SMs.
PATHS = [
    (300, 2048, 1, "streaming"), (129, 5632, 2, "streaming"), (64, 11008, 1, "streaming"),
    (37, 288, 3, "generic"), (9, 160, 1, "generic"), (40, 800, 2, "generic"),
    (300, 2048, 3, "tc-decode"), (1000, 2048, 16, "tc-decode"), (200, 11008, 8, "tc-decode"),
    (129, 5632, 17, "tc-decode bf16"), (300, 2048, 40, "tc-decode bf16"),
    (128, 512, 64, "tc-decode bf16"),
    (10236, 256, 200, "gemm 256"), (10239, 256, 130, "gemm 256"),
    (10240, 512, 300, "gemm 512"), (9728, 768, 777, "gemm 512"),
    (300, 512, 100, "gemm split 2"), (1000, 2048, 257, "gemm split 4"),
    (1001, 1280, 70, "gemm split 4"),
]


@pytest.mark.parametrize("t", ["q4_0", "q8_0"])
@pytest.mark.parametrize("M,K,N,path", PATHS)
def test_edge_blocks_match_oracle(gq_lib, oracle_mod, cuda_dev, t, M, K, N, path):
    Y, Y_ref, What, X, _ = _run(gq_lib, oracle_mod, cuda_dev, t, M, K, N, seed=M + 7 * K + N)
    _tol_check(Y, Y_ref, What, X, f"{path} {t} M={M} K={K} N={N}")
    # rows whose every scale is +-0 (kind 3) give exactly zero
    zero_rows = np.nonzero(_rows(M) % 8 == 3)[0]
    assert not Y[:, zero_rows].any()


@pytest.mark.parametrize("t", ["q4_0", "q8_0"])
def test_edge_blocks_small_activations(gq_lib, oracle_mod, cuda_dev, t):
    """Scales up to 65504 with activations of 1e-6 and 1e-20: nothing flushes to zero or
    loses its scale on any path."""
    M, K = 200, 2048
    for N in (1, 2, 4, 16, 40, 100):
        X = workloads.activations(N, K, seed=N).numpy()
        X[0::2] *= np.float32(1e-6)
        X[1::2] *= np.float32(1e-20)
        Y, Y_ref, What, X, _ = _run(gq_lib, oracle_mod, cuda_dev, t, M, K, N, seed=5, X=X)
        _tol_check(Y, Y_ref, What, X, f"small x {t} N={N}")


def _one_hot(K, N, shift):
    ks = [(shift + 37 * n) % K for n in range(N)]
    X = np.zeros((N, K), np.float32)
    for n, k in enumerate(ks):
        X[n, k] = 1.0
    return X, ks


# (K, N, exact): "exact" paths return What itself for X = e_k (the CUDA-core kernels: exact
# integer block products; the scaled tensor-core form for Q4_0 up to 16 tokens: exact codes
# times the fp32 scale); the others return bf16(What), the operand the MMA multiplied.
ONE_HOT = [(2048, 1, "exact"), (2048, 2, "exact"), (96, 2, "exact"),
           (1024, 4, "scaled"), (1024, 16, "scaled"), (1024, 40, "bf16"), (512, 100, "bf16")]


@pytest.mark.parametrize("t", ["q4_0", "q8_0"])
@pytest.mark.parametrize("K,N,form", ONE_HOT)
def test_edge_blocks_one_hot(gq_lib, oracle_mod, cuda_dev, t, K, N, form):
    M = 203
    X, ks = _one_hot(K, N, shift=11)
    Y, _, What, _, _ = _run(gq_lib, oracle_mod, cuda_dev, t, M, K, N, seed=17, X=X)
    if form == "exact" or (form == "scaled" and t == "q4_0"):
        expect = What
    else:
        expect = torch.from_numpy(What).to(torch.bfloat16).float().numpy()
    for n, k in enumerate(ks):
        got, want = Y[n], expect[:, k]
        assert np.array_equal(got, want), (n, k, np.nonzero(got != want)[0][:8])


def _q8x_bound(oracle_mod, t, q, M, K, X):
    """fp32 accumulation bound of the block sums: (blocks + 8) 2^-24 sum |What| |Xhat|."""
    wa = np.abs(oracle_mod.dequantize(t, q, M, K).astype(np.float64))
    N = X.shape[0]
    xa = np.abs(oracle_mod.dequantize("q8_0", oracle_mod.quantize("q8_0", X), N, K)
                .astype(np.float64))
    return (K // 32 + 8) * 2.0 ** -24 * (xa @ wa.T) + 1e-30


@pytest.mark.parametrize("t", ["q4_0", "q8_0"])
@pytest.mark.parametrize("M,K,N", [(300, 2048, 1), (129, 5632, 2), (64, 11008, 5),
                                   (1000, 2048, 16)])
def test_edge_blocks_q8x(gq_lib, oracle_mod, cuda_dev, t, M, K, N):
    """gq_mul_mat_q8x: Q4_0 subtracts 8 sum q_x from unsigned-nibble sums and Q8_0 feeds
    -128 to the signed byte products; both against the oracle's own definition."""
    q = workloads.edge_blocks(t, M, K, seed=M + K)
    X = workloads.activations(N, K, seed=N + 3).numpy()
    Y = gq_lib.mul_mat_q8x(torch.from_numpy(q).to(cuda_dev), t, M, K,
                           torch.from_numpy(X).to(cuda_dev)).cpu().numpy()
    assert gq_lib.get_last_error() == 0
    Y_ref = oracle_mod.mul_mat_q8x(t, q, M, K, X).astype(np.float64)
    err = np.abs(Y.astype(np.float64) - Y_ref)
    bound = _q8x_bound(oracle_mod, t, q, M, K, X)
    assert np.all(err <= bound), f"q8x {t} M={M} K={K} N={N}: {(err > bound).sum()} out"
    zero_rows = np.arange(M) % 8 == 3
    assert not Y[:, zero_rows].any()


# N <= 2 runs fused in the decode kernel; N = 8 and 100 compose plain kernels.
FUSED = [(300, 2048, 1), (129, 5632, 2), (200, 2048, 8), (300, 512, 100)]


@pytest.mark.parametrize("t", ["q4_0", "q8_0"])
@pytest.mark.parametrize("M,K,N", FUSED)
def test_edge_blocks_rmsnorm(gq_lib, oracle_mod, cuda_dev, t, M, K, N):
    q = workloads.edge_blocks(t, M, K, seed=M + 2 * K)
    X = workloads.activations(N, K, seed=N + 5).numpy()
    gamma = (1.0 + 0.1 * np.random.default_rng(K).standard_normal(K)).astype(np.float32)
    Y = gq_lib.mul_mat_rmsnorm(torch.from_numpy(q).to(cuda_dev), t, M, K,
                               torch.from_numpy(X).to(cuda_dev),
                               torch.from_numpy(gamma).to(cuda_dev), 1e-5).cpu().numpy()
    assert gq_lib.get_last_error() == 0
    Y_ref = oracle_mod.mul_mat_rmsnorm(t, q, M, K, X, gamma, 1e-5)
    x64 = X.astype(np.float64)
    xhat = x64 / np.sqrt((x64 ** 2).mean(axis=1, keepdims=True) + 1e-5) * gamma
    _tol_check(Y, Y_ref, oracle_mod.dequantize(t, q, M, K), xhat, f"rmsnorm {t} {M} {K} {N}")


@pytest.mark.parametrize("t", ["q4_0", "q8_0"])
@pytest.mark.parametrize("M,K,N", FUSED)
def test_edge_blocks_swiglu(gq_lib, oracle_mod, cuda_dev, t, M, K, N):
    """H = Swish(G) U. Swish is 1.1-Lipschitz, so with the products' bounds e_G, e_U:
    |H - H_ref| <= 1.1 e_G (|U| + e_U) + |Swish(G)| e_U. The e_G e_U term matters here:
    scales of 65504 make both bounds large at once."""
    qg = workloads.edge_blocks(t, M, K, seed=M + 3 * K)
    qu = workloads.edge_blocks(t, M, K, seed=M + 4 * K)
    X = workloads.activations(N, K, seed=N + 9).numpy()
    H = gq_lib.mul_mat_swiglu(torch.from_numpy(qg).to(cuda_dev), torch.from_numpy(qu).to(cuda_dev),
                              t, M, K, torch.from_numpy(X).to(cuda_dev)).cpu().numpy()
    assert gq_lib.get_last_error() == 0
    assert np.isfinite(H).all()
    H_ref = oracle_mod.mul_mat_swiglu(t, qg, qu, M, K, X).astype(np.float64)
    G = oracle_mod.mul_mat(t, qg, M, K, X).astype(np.float64)
    U = oracle_mod.mul_mat(t, qu, M, K, X).astype(np.float64)
    xn = np.linalg.norm(X.astype(np.float64), axis=1)[:, None]
    eg = TOL * xn * np.linalg.norm(oracle_mod.dequantize(t, qg, M, K).astype(np.float64), axis=1)
    eu = TOL * xn * np.linalg.norm(oracle_mod.dequantize(t, qu, M, K).astype(np.float64), axis=1)
    with np.errstate(over="ignore"):
        swish = G / (1.0 + np.exp(-G))
    tol = 1.1 * eg * (np.abs(U) + eu) + np.abs(swish) * eu + 1e-6 * np.abs(H_ref)
    bad = np.abs(H - H_ref) > tol
    assert not bad.any(), f"swiglu {t} {M} {K} {N}: {bad.sum()} out, first {np.argwhere(bad)[0]}"


@pytest.mark.parametrize("t", ["q4_0", "q8_0"])
def test_edge_blocks_batched_step(gq_lib, oracle_mod, cuda_dev, t):
    """The batched launch the decode benchmark times, with hand-made blocks in every
    problem: N = 1 (streaming) and N = 8 (tensor-core decode)."""
    shapes = [(256, 2048), (2048, 2048), (300, 5632), (64, 11008), (33, 96)]
    for N in (1, 8):
        items, refs = [], []
        for i, (M, K) in enumerate(shapes):
            q = workloads.edge_blocks(t, M, K, seed=400 + i)
            X = workloads.activations(N, K, seed=410 + i).numpy()
            items.append((torch.from_numpy(q).to(cuda_dev), M, K,
                          torch.from_numpy(X).to(cuda_dev),
                          torch.full((N, M), float("nan"), device=cuda_dev)))
            refs.append((q, X))
        gq_lib.mul_mat_batched(items, t, N)
        assert gq_lib.get_last_error() == 0
        for (M, K), (q, X), it in zip(shapes, refs, items):
            _tol_check(it[4].cpu().numpy(), oracle_mod.mul_mat(t, q, M, K, X),
                       oracle_mod.dequantize(t, q, M, K), X, f"batched {t} N={N} M={M} K={K}")
