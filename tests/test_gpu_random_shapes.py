"""A seeded sweep of random problems through the C ABI against the oracle: block type,
M, K, N, the entry point (gq_mul_mat, _ws, _batched), X's alignment and the token count
(CUDA-core decode, generic kernel, tensor-core decode, prefill GEMM) all drawn at random,
so that shapes nobody picked by hand reach every path. Bar: |Y - Y_oracle| <= 1e-3
||X[n]|| ||What[m]|| per element, on quantizer output."""
import numpy as np
import pytest
import torch

from block_quantized_matmul_gq_gb300 import workloads

pytestmark = pytest.mark.gpu

CASES = 48


def _draw(rng):
    t = ["q4_0", "q8_0", "q4_k"][rng.integers(0, 3)]
    blk = 256 if t == "q4_k" else 32
    # K: mostly multiples of 256 (every path), sometimes only of 32 (CUDA-core kernels)
    K = int(rng.integers(1, 17)) * 256 if (t == "q4_k" or rng.random() < 0.75) \
        else int(rng.integers(1, 80)) * 32
    M = int(rng.integers(1, 700))
    N = int(rng.choice([1, 2, int(rng.integers(3, 17)), int(rng.integers(17, 65)),
                        int(rng.integers(65, 200))]))
    entry = ["mul_mat", "ws", "batched"][rng.integers(0, 3)]
    offset = int(rng.random() < 0.2)   # X one float into its buffer: not 16-byte aligned
    return t, M, K - K % blk, N, entry, offset


@pytest.mark.parametrize("case", range(CASES))
def test_random_problem_matches_oracle(gq_lib, oracle_mod, cuda_dev, case):
    rng = np.random.default_rng(7000 + case)
    t, M, K, N, entry, offset = _draw(rng)
    q = oracle_mod.quantize(t, workloads.weights(M, K, seed=case).numpy())
    X = workloads.activations(N, K, seed=100 + case).numpy()
    qd = torch.from_numpy(q).to(cuda_dev)
    buf = torch.zeros(N * K + offset, device=cuda_dev)
    buf[offset:] = torch.from_numpy(X).reshape(-1).to(cuda_dev)
    Xd = buf[offset:].view(N, K)
    Y = torch.full((N, M), float("nan"), device=cuda_dev)
    if entry == "mul_mat":
        gq_lib.mul_mat(qd, t, M, K, Xd, out=Y)
    elif entry == "ws":
        need = gq_lib.workspace_size(t, M, K, N)
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=cuda_dev) if need else None
        gq_lib.mul_mat_ws(qd, t, M, K, Xd, ws, out=Y)
    else:
        gq_lib.mul_mat_batched(gq_lib.make_problems([(qd, M, K, Xd, Y)]), t, N)
    Y = Y.cpu().numpy()
    assert gq_lib.get_last_error() == 0
    What = oracle_mod.dequantize(t, q, M, K).astype(np.float64)
    tol = 1e-3 * np.linalg.norm(X.astype(np.float64), axis=1)[:, None] * \
        np.linalg.norm(What, axis=1)[None, :]
    err = np.abs(Y.astype(np.float64) - oracle_mod.mul_mat(t, q, M, K, X))
    where = f"{t} M={M} K={K} N={N} {entry} offset={offset}"
    assert np.isfinite(Y).all(), where
    assert (err <= tol).all(), f"{where}: max err/tol {(err / np.where(tol > 0, tol, 1)).max():.3f}"
