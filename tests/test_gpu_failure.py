"""Failure detection on the GPU without a fault: a device-side wait that can only run out
must end in GQ_ERR_TIMEOUT on the host, and the context must stay usable afterwards."""
import pytest
import torch

from block_quantized_matmul_gq_gb300 import workloads

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_cleared(gq_lib, cuda_dev):
    assert gq_lib.get_last_error() == 0
    gq_lib.selftest_wait_timeout(20000)             # 20 ms limit on a barrier nobody completes
    assert gq_lib.get_last_error() == -6             # GQ_ERR_TIMEOUT
    assert gq_lib.get_last_error() == 0              # read clears it
    # the context still works: a normal mul_mat right after
    M, K = 64, 256
    q = gq_lib.quantize(workloads.weights(M, K, 1, device=cuda_dev), "q4_0")
    y = gq_lib.mul_mat(q, "q4_0", M, K, workloads.activations(1, K, 2, device=cuda_dev))
    assert torch.isfinite(y).all()
    assert gq_lib.get_last_error() == 0


def test_selftest_rejects_bad_limit(gq_lib):
    with pytest.raises(gq_lib.GQError):
        gq_lib.selftest_wait_timeout(0)
