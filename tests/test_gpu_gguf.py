"""GGUF tensors to the GPU and through mul_mat: a file holding Q4_0, Q8_0 and Q4_K weight
matrices (quantized by the oracle, written by tests/gguf_writer.py) is opened by libgq's
reader, each matrix uploaded with gq_gguf_upload, and the products checked against the
oracle on the same bytes (|dY| <= 1e-3 ||x|| ||What_row||)."""
import numpy as np
import pytest
import torch

import gguf_writer as gw
from block_quantized_matmul_gq_gb300 import workloads

pytestmark = pytest.mark.gpu

GGML = {"q4_0": 2, "q8_0": 8, "q4_k": 12}


def _model(oracle_mod, tmp_path, alignment=32):
    mats = [("blk.0.attn_q.weight", "q4_0", 256, 2048), ("blk.0.attn_k.weight", "q8_0", 64, 2048),
            ("blk.0.ffn_down.weight", "q4_k", 300, 5632), ("output.weight", "q4_k", 1000, 2048),
            ("blk.0.ffn_gate.weight", "q4_0", 129, 768)]
    tensors, blocks = [], {}
    for j, (name, t, M, K) in enumerate(mats):
        q = oracle_mod.quantize(t, workloads.weights(M, K, seed=500 + j).numpy())
        blocks[name] = (t, M, K, q)
        tensors.append((name, [K, M], GGML[t], q.tobytes()))
    norm = np.linspace(0.5, 1.5, 2048).astype("<f4")
    tensors.append(("output_norm.weight", [2048], 0, norm.tobytes()))
    data, _ = gw.build([("general.architecture", gw.STRING, "llama")], tensors,
                       alignment=alignment)
    p = tmp_path / "model.gguf"
    p.write_bytes(data)
    return p, blocks, norm


@pytest.mark.parametrize("alignment", [32, 64])
@pytest.mark.parametrize("N", [1, 5, 80])
def test_uploaded_matrices_multiply_like_the_oracle(gq_lib, oracle_mod, cuda_dev, tmp_path,
                                                    alignment, N):
    from block_quantized_matmul_gq_gb300.gguf import GGUFFile
    path, blocks, norm = _model(oracle_mod, tmp_path, alignment)
    with GGUFFile(path) as f:
        for name, (t, M, K, q) in blocks.items():
            assert f.matrix(name) == (t, M, K)
            W = f.upload(name, cuda_dev)
            assert W.shape == (M, gq_lib.row_bytes(t, K))
            assert np.array_equal(W.cpu().numpy(), q)            # one copy, no conversion
            X = workloads.activations(N, K, seed=M + N).numpy()
            Y = gq_lib.mul_mat(W, t, M, K, torch.from_numpy(X).to(cuda_dev)).cpu().numpy()
            Y_ref = oracle_mod.mul_mat(t, q, M, K, X)
            xn = np.linalg.norm(X.astype(np.float64), axis=1)[:, None]
            wn = np.linalg.norm(oracle_mod.dequantize(t, q, M, K).astype(np.float64), axis=1)
            err = np.abs(Y.astype(np.float64) - Y_ref)
            assert (err <= 1e-3 * xn * wn[None, :]).all(), name
        g = f.upload("output_norm.weight", cuda_dev)              # a plain F32 tensor
        assert g.shape == (2048 * 4,)
        assert np.array_equal(g.cpu().numpy().view("<f4"), norm)
    assert gq_lib.get_last_error() == 0


def test_upload_on_a_stream_then_a_batched_step(gq_lib, oracle_mod, cuda_dev, tmp_path):
    """Uploads on a side stream, then all matrices of one type in one batched call on it."""
    from block_quantized_matmul_gq_gb300.gguf import GGUFFile
    path, blocks, _ = _model(oracle_mod, tmp_path)
    s = torch.cuda.Stream()
    with GGUFFile(path) as f, torch.cuda.stream(s):
        items, refs = [], []
        for name, (t, M, K, q) in blocks.items():
            if t != "q4_k":
                continue
            W = f.upload(name, cuda_dev, stream=s)
            X = workloads.activations(1, K, seed=K).to(cuda_dev)
            Y = torch.empty((1, M), device=cuda_dev)
            items.append((W, M, K, X, Y))
            refs.append((q, M, K, X.cpu().numpy(), Y))
        gq_lib.mul_mat_batched(gq_lib.make_problems(items), "q4_k", 1, stream=s)
    s.synchronize()
    for q, M, K, X, Y in refs:
        Y_ref = oracle_mod.mul_mat("q4_k", q, M, K, X)
        wn = np.linalg.norm(oracle_mod.dequantize("q4_k", q, M, K).astype(np.float64), axis=1)
        tol = 1e-3 * np.linalg.norm(X.astype(np.float64)) * wn
        assert (np.abs(Y.cpu().numpy()[0] - Y_ref[0]) <= tol).all()
