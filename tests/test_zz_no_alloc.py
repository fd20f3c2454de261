"""gq_mul_mat_noalloc -- the entry point for callers that cannot allocate device memory
(graph capture, arena-owned memory, fixed real-time budgets) -- must give what gq_mul_mat
gives. Collected last on purpose: a failure here comes after every other test has run.

Calls go through the C ABI (the ctypes binding) and are compared with gq_mul_mat within
the suite's tolerance, |dY| <= 1e-3 * ||x|| * ||What_row||, on two calls in a row.
"""
import numpy as np
import pytest
import torch

from block_quantized_matmul_gq_gb300 import workloads

pytestmark = pytest.mark.gpu

TOL = 1e-3


def _check_close(Y, Y_ref, What, X):
    Y = Y.double().cpu().numpy()
    Y_ref = Y_ref.double().cpu().numpy()
    xn = np.linalg.norm(X.double().cpu().numpy(), axis=1)
    wn = np.linalg.norm(What.double().cpu().numpy(), axis=1)
    assert np.all(np.abs(Y - Y_ref) <= TOL * xn[:, None] * wn[None, :])


@pytest.mark.parametrize("t", ["q4_0", "q8_0"])
@pytest.mark.parametrize("M,K,N", [(1000, 2048, 300), (256, 5632, 512), (300, 2048, 3)])
def test_noalloc_matches_mul_mat_on_two_calls(gq_lib, cuda_dev, t, M, K, N):
    W = workloads.weights(M, K, seed=71, device=cuda_dev)
    q = gq_lib.quantize(W, t)
    What = gq_lib.dequantize(q, t, M, K)
    for call in range(2):
        X = workloads.activations(N, K, seed=80 + call, device=cuda_dev)
        ref = gq_lib.mul_mat(q, t, M, K, X)
        Y = torch.full_like(ref, float("nan"))
        gq_lib.mul_mat_noalloc(q, t, M, K, X, out=Y)
        torch.cuda.synchronize()
        assert not torch.isnan(Y).any()
        _check_close(Y, ref, What, X)
    assert gq_lib.get_last_error() == 0


def test_noalloc_rejects_workspace_beyond_the_fixed_array(gq_lib, cuda_dev):
    # N * K * 2 = 64 MiB + 512 KiB > 64 MiB: refused before anything is launched.
    M, K, N = 128, 2048, 16400
    q = torch.zeros((M, K // 32 * 18), dtype=torch.uint8, device=cuda_dev)
    X = torch.zeros((N, K), device=cuda_dev)
    with pytest.raises(gq_lib.GQError) as e:
        gq_lib.mul_mat_noalloc(q, "q4_0", M, K, X)
    assert e.value.status == -2
