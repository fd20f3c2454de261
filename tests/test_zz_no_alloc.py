"""gq_mul_mat_noalloc -- the entry point for callers that cannot allocate device memory
(engines whose arena owns all device memory, real-time loops that must not stall on an
allocation) -- must give what gq_mul_mat gives. Collected
last on purpose: a failure here comes after every other test has run.

Calls go through the C ABI (the ctypes binding). Each result is checked against the CPU
oracle within the suite's tolerance, |dY| <= 1e-3 * ||x|| * ||What_row||, and against
gq_mul_mat on the same inputs, on two calls in a row (the second call finds the fixed
array holding the first call's contents).
"""
import numpy as np
import pytest
import torch

from block_quantized_matmul_gq_gb300 import workloads

pytestmark = pytest.mark.gpu

TOL = 1e-3


def _check_close(Y, Y_ref, What, X, where):
    Y = np.asarray(Y, np.float64)
    Y_ref = np.asarray(Y_ref, np.float64)
    xn = np.linalg.norm(np.asarray(X, np.float64), axis=1)
    wn = np.linalg.norm(np.asarray(What, np.float64), axis=1)
    bad = np.abs(Y - Y_ref) > TOL * xn[:, None] * wn[None, :]
    assert not bad.any(), f"{where}: {bad.sum()} elements out of tolerance"


# N = 300 / 512: prefill GEMM (workspace in the fixed array); N = 3 and 16: tensor-core
# decode (X tiles, partial sums and counters in the fixed array); N = 2: CUDA-core decode.
# Q4_K takes the same paths: N = 1 CUDA-core, 5 and 40 tensor-core decode, 300 prefill.
@pytest.mark.parametrize("t,M,K,N", [(t, *s) for t in ("q4_0", "q8_0") for s in
                                     [(1000, 2048, 300), (256, 5632, 512), (300, 2048, 3),
                                      (129, 5632, 16), (77, 2048, 2)]] +
                         [("q4_k", 300, 2048, 1), ("q4_k", 129, 5632, 5),
                          ("q4_k", 77, 2048, 40), ("q4_k", 300, 2048, 300)])
def test_noalloc_matches_oracle_on_two_calls(gq_lib, oracle_mod, cuda_dev, t, M, K, N):
    q = oracle_mod.quantize(t, workloads.weights(M, K, seed=71).numpy())
    What = oracle_mod.dequantize(t, q, M, K)
    qd = torch.from_numpy(q).to(cuda_dev)
    for call in range(2):
        X = workloads.activations(N, K, seed=80 + call).numpy()
        Xd = torch.from_numpy(X).to(cuda_dev)
        Y = torch.full((N, M), float("nan"), device=cuda_dev)
        gq_lib.mul_mat_noalloc(qd, t, M, K, Xd, out=Y)
        ref = gq_lib.mul_mat(qd, t, M, K, Xd)
        torch.cuda.synchronize()
        Y = Y.cpu().numpy()
        assert not np.isnan(Y).any()
        _check_close(Y, oracle_mod.mul_mat(t, q, M, K, X), What, X, f"oracle, call {call}")
        _check_close(Y, ref.cpu().numpy(), What, X, f"gq_mul_mat, call {call}")
    assert gq_lib.get_last_error() == 0


def test_noalloc_workspace_at_the_exact_limit(gq_lib, oracle_mod, cuda_dev):
    """N * K * 2 == 64 MiB: the bf16 copy of X fills the array to its last byte and is
    accepted. Sampled tokens from both ends (the last ones live in the array's last bytes)
    are checked against the oracle."""
    M, K, N = 128, 2048, 16384
    assert N * K * 2 == 64 << 20
    q = oracle_mod.quantize("q4_0", workloads.weights(M, K, seed=72).numpy())
    X = workloads.activations(N, K, seed=73, device=cuda_dev)
    Y = torch.full((N, M), float("nan"), device=cuda_dev)
    gq_lib.mul_mat_noalloc(torch.from_numpy(q).to(cuda_dev), "q4_0", M, K, X, out=Y)
    assert gq_lib.get_last_error() == 0
    tokens = np.concatenate([np.arange(8), np.arange(N // 2 - 4, N // 2 + 4), np.arange(N - 24, N)])
    Xs = X[torch.from_numpy(tokens).to(cuda_dev)].cpu().numpy()
    Ys = Y[torch.from_numpy(tokens).to(cuda_dev)].cpu().numpy()
    _check_close(Ys, oracle_mod.mul_mat("q4_0", q, M, K, Xs), oracle_mod.dequantize("q4_0", q, M, K),
                 Xs, "exact limit")


def test_noalloc_rejects_workspace_beyond_the_fixed_array(gq_lib, cuda_dev):
    # N * K * 2 = 64 MiB + 512 KiB > 64 MiB: refused before anything is launched.
    M, K, N = 128, 2048, 16400
    q = torch.zeros((M, K // 32 * 18), dtype=torch.uint8, device=cuda_dev)
    X = torch.zeros((N, K), device=cuda_dev)
    with pytest.raises(gq_lib.GQError) as e:
        gq_lib.mul_mat_noalloc(q, "q4_0", M, K, X)
    assert e.value.status == -2
