"""X and Y in pinned host memory, passed straight to the C ABI (include/gq.h: the kernels
read X and write Y over the host link). Every path gives the same bits as with device
buffers, and stays within the mul_mat tolerance of the oracle."""
import numpy as np
import pytest
import torch

from block_quantized_matmul_gq_gb300 import workloads

pytestmark = pytest.mark.gpu

# (type, M, K, N): streaming decode (N = 1, 2), generic kernel (K % 256 != 0), tensor-core
# decode (N = 5, 40), prefill GEMM (N = 80, 300)
CASES = [("q4_0", 300, 2048, 1), ("q8_0", 129, 5632, 2), ("q4_0", 37, 96, 3),
         ("q4_k", 200, 2048, 1), ("q4_0", 1000, 2048, 5), ("q8_0", 300, 2048, 40),
         ("q4_k", 129, 2048, 16), ("q4_0", 520, 1792, 80), ("q4_k", 256, 1024, 300)]


def _pinned(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(a).pin_memory()


@pytest.mark.parametrize("t,M,K,N", CASES)
def test_host_x_and_y_match_device_buffers_and_the_oracle(gq_lib, oracle_mod, cuda_dev, t, M, K,
                                                         N):
    q = oracle_mod.quantize(t, workloads.weights(M, K, seed=M + K).numpy())
    X = workloads.activations(N, K, seed=N + K).numpy()
    qd = torch.from_numpy(q).to(cuda_dev)
    Xh = _pinned(X)
    Yh = torch.full((N, M), float("nan")).pin_memory()
    gq_lib.mul_mat(qd, t, M, K, Xh, out=Yh)
    torch.cuda.synchronize()
    Yd = gq_lib.mul_mat(qd, t, M, K, torch.from_numpy(X).to(cuda_dev)).cpu()
    assert torch.equal(Yh.view(torch.int32), Yd.view(torch.int32))
    What = oracle_mod.dequantize(t, q, M, K).astype(np.float64)
    tol = 1e-3 * np.linalg.norm(X.astype(np.float64), axis=1)[:, None] * \
        np.linalg.norm(What, axis=1)[None, :]
    assert (np.abs(Yh.numpy().astype(np.float64) - oracle_mod.mul_mat(t, q, M, K, X)) <= tol).all()
    assert gq_lib.get_last_error() == 0


@pytest.mark.parametrize("N", [1, 16])
def test_batched_step_with_host_buffers(gq_lib, cuda_dev, N):
    """The benchmark's end-to-end form: one flat pinned X and one flat pinned Y for a whole
    TinyLLaMA decode step, one batched call, bit-equal to the same call on device buffers."""
    from block_quantized_matmul_gq_gb300.weightset import QuantizedWeightSet
    shapes = workloads.tinyllama_decode_set()
    ws = QuantizedWeightSet.synthetic(2, shapes, "q4_0", cuda_dev)
    xt, yt = sum(N * s.K for s in shapes), sum(N * s.M for s in shapes)
    Xd = torch.empty(xt, device=cuda_dev)
    o = 0
    for j, s in enumerate(shapes):
        Xd[o:o + N * s.K].copy_(workloads.activations(N, s.K, j, device=cuda_dev).reshape(-1))
        o += N * s.K
    Xh = Xd.cpu().pin_memory()
    Yd = torch.empty(yt, device=cuda_dev)
    Yh = torch.full((yt,), float("nan")).pin_memory()

    def items(X, Y):
        out, xo, yo = [], 0, 0
        for m, s in zip(ws.mats, shapes):
            out.append((m.blocks, s.M, s.K, X[xo:xo + N * s.K].view(N, s.K),
                        Y[yo:yo + N * s.M].view(N, s.M)))
            xo += N * s.K
            yo += N * s.M
        return out
    gq_lib.mul_mat_batched(gq_lib.make_problems(items(Xd, Yd)), "q4_0", N)
    gq_lib.mul_mat_batched(gq_lib.make_problems(items(Xh, Yh)), "q4_0", N)
    torch.cuda.synchronize()
    assert torch.equal(Yh.view(torch.int32), Yd.cpu().view(torch.int32))
    assert gq_lib.get_last_error() == 0


def test_fused_forms_with_host_buffers(gq_lib, cuda_dev):
    M, K, N = 256, 2048, 1
    W = workloads.weights(M, K, 3, device=cuda_dev)
    q = gq_lib.quantize(W, "q4_0")
    qu = gq_lib.quantize(workloads.weights(M, K, 4, device=cuda_dev), "q4_0")
    Xd = workloads.activations(N, K, 5, device=cuda_dev)
    g = (1.0 + 0.1 * workloads.activations(1, K, 6)).reshape(-1)
    Xh, gh = Xd.cpu().pin_memory(), g.pin_memory()
    a = gq_lib.mul_mat_rmsnorm(q, "q4_0", M, K, Xh, gh, 1e-5)
    b = gq_lib.mul_mat_rmsnorm(q, "q4_0", M, K, Xd, g.to(cuda_dev), 1e-5)
    c = gq_lib.mul_mat_swiglu(q, qu, "q4_0", M, K, Xh)
    d = gq_lib.mul_mat_swiglu(q, qu, "q4_0", M, K, Xd)
    torch.cuda.synchronize()
    assert not a.is_cuda and a.is_pinned()
    assert torch.equal(a.view(torch.int32), b.cpu().view(torch.int32))
    assert torch.equal(c.view(torch.int32), d.cpu().view(torch.int32))


def test_plain_host_tensors_are_refused(gq_lib, cuda_dev):
    q = torch.zeros((4, 36), dtype=torch.uint8, device=cuda_dev)
    with pytest.raises(ValueError, match="pinned"):
        gq_lib.mul_mat(q, "q4_0", 4, 64, torch.zeros(1, 64))
