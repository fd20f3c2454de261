"""Parity of the CUDA path (through the C ABI) with the CPU oracle, element by element.

Quantize and dequantize must be bit-exact. mul_mat must satisfy, per element,
    |Y - Y_oracle| <= 1e-3 * ||X[n]||_2 * ||What[m]||_2
where What is the oracle's own dequantization of the oracle's own blocks. Inputs are
seeded synthetic tensors drawn on the CPU; no oracle input comes from the CUDA path.
"""
import numpy as np
import pytest
import torch

from block_quantized_matmul_gq_gb300 import workloads

pytestmark = pytest.mark.gpu

TOL = 1e-3


def _np_weights(M, K, seed, scale=None):
    W = workloads.weights(M, K, seed).numpy()
    return W if scale is None else (W * scale).astype(np.float32)


def check_tolerance(Y, Y_ref, What, X, where=""):
    Y = np.asarray(Y, np.float64)
    xn = np.linalg.norm(np.asarray(X, np.float64), axis=1)
    wn = np.linalg.norm(np.asarray(What, np.float64), axis=1)
    tol = TOL * xn[:, None] * wn[None, :]
    err = np.abs(Y - np.asarray(Y_ref, np.float64))
    bad = err > tol
    if bad.any():
        n, m = np.argwhere(bad)[0]
        raise AssertionError(f"{where}: {bad.sum()} elements out of tolerance, first (n={n}, "
                             f"m={m}) err={err[n, m]:.3e} tol={tol[n, m]:.3e}")
    return float((err / np.where(tol > 0, tol, 1)).max()) if err.size else 0.0


def gpu_quantize(gq_lib, W, t, dev):
    return gq_lib.quantize(torch.from_numpy(W).to(dev), t).cpu().numpy()


# ------------------------------------------------------------------------------------
# quantize / dequantize: bit-exact
# ------------------------------------------------------------------------------------
QUANT_SHAPES = [(1, 32), (3, 96), (37, 288), (64, 2048), (129, 5632), (5, 11008)]


@pytest.mark.parametrize("t", ["q4_0", "q8_0"])
@pytest.mark.parametrize("M,K", QUANT_SHAPES)
def test_quantize_bit_exact(gq_lib, oracle_mod, cuda_dev, t, M, K):
    W = _np_weights(M, K, seed=M * 7 + K)
    assert np.array_equal(gpu_quantize(gq_lib, W, t, cuda_dev), oracle_mod.quantize(t, W))


@pytest.mark.parametrize("t", ["q4_0", "q8_0"])
def test_quantize_special_blocks(gq_lib, oracle_mod, cuda_dev, t):
    """Zero blocks, exact ties of w/d, powers of two, subnormal and huge magnitudes."""
    rng = np.random.default_rng(99)
    rows = []
    rows.append(np.zeros(64, np.float32))
    s = 0.25
    tie = np.zeros(32, np.float32)
    tie[:8] = np.array([7, 2.5, -2.5, 0.5, -0.5, 6.5, -6.5, 1.5]) * s
    rows.append(np.concatenate([tie, tie * 4]))
    rows.append((rng.integers(-8, 8, 64) * 2.0 ** -10).astype(np.float32))
    rows.append((rng.standard_normal(64) * 1e-7).astype(np.float32))     # fp16 subnormal d
    rows.append((rng.standard_normal(64) * 1e-41).astype(np.float32))    # fp32 subnormal w
    rows.append((rng.standard_normal(64) * 1e4).astype(np.float32))
    rows.append(np.full(64, -3.0, np.float32))
    W = np.stack(rows)
    assert np.array_equal(gpu_quantize(gq_lib, W, t, cuda_dev), oracle_mod.quantize(t, W))


@pytest.mark.parametrize("t", ["q4_0", "q8_0"])
def test_dequantize_bit_exact(gq_lib, oracle_mod, cuda_dev, t):
    """Arbitrary block bytes (random codes, any finite fp16 scale, code 0 included)."""
    rng = np.random.default_rng(5)
    M, K = 41, 288
    bb = oracle_mod.block_bytes(t)
    blocks = rng.integers(0, 256, size=(M, K // 32, bb), dtype=np.uint8)
    scales = rng.standard_normal((M, K // 32)).astype(np.float16)
    scales[0, 0] = np.float16(6e-8)          # subnormal scale
    blocks[..., :2] = scales.view(np.uint8).reshape(M, K // 32, 2)
    blocks = blocks.reshape(M, -1)
    got = gq_lib.dequantize(torch.from_numpy(blocks).to(cuda_dev), t, M, K).cpu().numpy()
    ref = oracle_mod.dequantize(t, blocks, M, K)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


# ------------------------------------------------------------------------------------
# mul_mat
# ------------------------------------------------------------------------------------
def run_mul_mat(gq_lib, oracle_mod, dev, t, M, K, N, seed=0, X=None):
    W = _np_weights(M, K, seed=seed + 11)
    q = oracle_mod.quantize(t, W)
    if X is None:
        X = workloads.activations(N, K, seed=seed + 12).numpy()
    Y = gq_lib.mul_mat(torch.from_numpy(q).to(dev), t, M, K, torch.from_numpy(X).to(dev))
    Y = Y.cpu().numpy()
    Y_ref = oracle_mod.mul_mat(t, q, M, K, X)
    What = oracle_mod.dequantize(t, q, M, K)
    return Y, Y_ref, What, X


# Fast streaming kernel: K % 256 == 0. Rows of K = 11008 (Q4_0: 43 chunks) straddle the
# 256-chunk stages, M values leave ragged tails, N covers 1..4 and token groups 4+4+1.
FAST = [(1, 256, 1), (7, 2048, 1), (300, 2048, 1), (1000, 2048, 2), (129, 5632, 3),
        (64, 11008, 4), (33, 4096, 5), (257, 1024, 9), (2048, 2048, 1), (200, 11008, 1),
        (65, 4096, 2)]
# Generic kernel: K % 256 != 0.
GENERIC = [(1, 32, 1), (5, 96, 2), (37, 288, 3), (64, 800, 4), (9, 160, 7)]


@pytest.mark.parametrize("t", ["q4_0", "q8_0"])
@pytest.mark.parametrize("M,K,N", FAST + GENERIC)
def test_mul_mat_matches_oracle(gq_lib, oracle_mod, cuda_dev, t, M, K, N):
    Y, Y_ref, What, X = run_mul_mat(gq_lib, oracle_mod, cuda_dev, t, M, K, N, seed=M + K + N)
    assert Y.shape == (N, M)
    check_tolerance(Y, Y_ref, What, X, f"{t} M={M} K={K} N={N}")


@pytest.mark.parametrize("t", ["q4_0", "q8_0"])
@pytest.mark.parametrize("K", [2048, 96])
def test_mul_mat_one_hot_is_exact(gq_lib, oracle_mod, cuda_dev, t, K):
    """X = e_k returns column k of What bit for bit on the CUDA-core decode kernels (the
    streaming one for K = 2048, the generic one for K = 96), called with <= 2 tokens."""
    M = 77
    ks = [0, 1, 15, 16, 31, 32, K - 1] + ([255, 256, 1000] if K > 1000 else [])
    W = _np_weights(M, K, seed=5)
    q = oracle_mod.quantize(t, W)
    What = oracle_mod.dequantize(t, q, M, K)
    qd = torch.from_numpy(q).to(cuda_dev)
    for i in range(0, len(ks), 2):
        group = ks[i:i + 2]
        X = np.zeros((len(group), K), np.float32)
        for n, k in enumerate(group):
            X[n, k] = 1.0
        Y = gq_lib.mul_mat(qd, t, M, K, torch.from_numpy(X).to(cuda_dev)).cpu().numpy()
        for n, k in enumerate(group):
            assert np.array_equal(Y[n], What[:, k]), k


@pytest.mark.parametrize("t", ["q4_0", "q8_0"])
def test_mul_mat_scaled_inputs(gq_lib, oracle_mod, cuda_dev, t):
    """Activations far from N(0,1): huge, tiny and mixed magnitudes per block."""
    M, K = 50, 2048
    rng = np.random.default_rng(3)
    X = rng.standard_normal((4, K)).astype(np.float32)
    X[0] *= 3e4
    X[1] *= 1e-30
    X[2, ::64] *= 1e3
    X[3, :256] = 0.0
    Y, Y_ref, What, _ = run_mul_mat(gq_lib, oracle_mod, cuda_dev, t, M, K, 4, X=X)
    check_tolerance(Y, Y_ref, What, X, t)


def test_mul_mat_deterministic(gq_lib, cuda_dev):
    M, K, N = 3000, 5632, 2
    W = workloads.weights(M, K, 1, device=cuda_dev)
    q = gq_lib.quantize(W, "q4_0")
    X = workloads.activations(N, K, 2, device=cuda_dev)
    y1 = gq_lib.mul_mat(q, "q4_0", M, K, X)
    y2 = gq_lib.mul_mat(q, "q4_0", M, K, X)
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32))


@pytest.mark.parametrize("N", [1, 2, 8, 40, 96])
def test_back_to_back_calls_see_previous_results(gq_lib, cuda_dev, N):
    """Calls launched back to back on one stream, each call's X being the previous call's Y
    (read after write) and each call's Y overwriting the X of the call before (write after
    read), give bitwise the results of the same chain with a synchronize after every call.
    A decode call may start streaming its weights while the previous one finishes; this
    pins that it touches X, Y and its workspace (N = 8, 40: the tensor-core path's X tiles,
    partial sums and counters, reused by every call) only after that call is complete.
    N = 96 runs the prefill GEMM, which starts while its own X conversion runs and must
    read the converted X only after it is complete."""
    D = 2048
    qs = [gq_lib.quantize(workloads.weights(D, D, 40 + i, device=cuda_dev), "q4_0")
          for i in range(4)]
    x0 = workloads.activations(N, D, 50, device=cuda_dev)

    def chain(sync):
        bufs = [x0.clone(), torch.empty_like(x0)]   # ping-pong: call i + 1 writes what call i read
        for i in range(24):
            src, dst = bufs[i % 2], bufs[(i + 1) % 2]
            gq_lib.mul_mat(qs[i % 4], "q4_0", D, D, src, out=dst)
            # keep the values in range: scale by a power of two with a separate kernel
            # every few calls (exact, and a different kernel between two mul_mats)
            if i % 6 == 5:
                dst.mul_(2.0 ** -4)
            if sync:
                torch.cuda.synchronize(cuda_dev)
        torch.cuda.synchronize(cuda_dev)
        return bufs[24 % 2]

    ref = chain(True)
    assert torch.isfinite(ref).all()
    for _ in range(3):
        out = chain(False)
        assert torch.equal(out.view(torch.int32), ref.view(torch.int32))
    assert gq_lib.get_last_error() == 0


@pytest.mark.parametrize("N", [1, 8, 96])
def test_decode_after_quantize_into_the_same_blocks(gq_lib, cuda_dev, N):
    """A decode call may load its weights before the kernel ahead of it on the stream has
    completed, but only when that kernel lets it start early, which only libgq's decode
    kernels do; the prefill GEMM (N = 96) loads its weights early only behind its own X
    conversion, an ordinary launch. Quantizing a different matrix into the same block
    buffer right before each call, with no synchronize, must give bitwise the results of
    the same sequence with a synchronize after every launch."""
    M = K = 2048
    Ws = [workloads.weights(M, K, 70 + i, device=cuda_dev) for i in range(3)]
    X = workloads.activations(N, K, 73, device=cuda_dev)
    q = torch.empty((M, gq_lib.row_bytes("q4_0", K)), dtype=torch.uint8, device=cuda_dev)

    def run(sync):
        outs = []
        for i in range(12):
            gq_lib.quantize(Ws[i % 3], "q4_0", out=q)
            if sync:
                torch.cuda.synchronize(cuda_dev)
            outs.append(gq_lib.mul_mat(q, "q4_0", M, K, X))
            if sync:
                torch.cuda.synchronize(cuda_dev)
        torch.cuda.synchronize(cuda_dev)
        return torch.stack(outs)

    ref = run(True)
    assert not torch.equal(ref[0], ref[1])   # the matrices differ, so stale blocks would show
    for _ in range(3):
        assert torch.equal(run(False).view(torch.int32), ref.view(torch.int32))
    assert gq_lib.get_last_error() == 0


def test_mul_mat_misaligned_x(gq_lib, oracle_mod, cuda_dev):
    """X 4-byte but not 16-byte aligned: correct through the generic kernel."""
    M, K = 40, 2048
    W = _np_weights(M, K, seed=8)
    q = oracle_mod.quantize("q4_0", W)
    X = workloads.activations(1, K, seed=9).numpy()
    buf = torch.zeros(K + 1, dtype=torch.float32, device=cuda_dev)
    buf[1:] = torch.from_numpy(X[0]).to(cuda_dev)
    xv = buf[1:].view(1, K)
    assert xv.data_ptr() % 16 == 4
    Y = gq_lib.mul_mat(torch.from_numpy(q).to(cuda_dev), "q4_0", M, K, xv).cpu().numpy()
    check_tolerance(Y, oracle_mod.mul_mat("q4_0", q, M, K, X),
                    oracle_mod.dequantize("q4_0", q, M, K), X)


def test_empty_and_zero_k(gq_lib, cuda_dev):
    q = torch.zeros(16, dtype=torch.uint8, device=cuda_dev)
    X = torch.zeros((3, 0), device=cuda_dev)
    Y = torch.full((3, 5), 7.0, device=cuda_dev)
    gq_lib.mul_mat(q, "q4_0", 5, 0, X, out=Y)          # empty sum
    assert torch.count_nonzero(Y) == 0
    Y2 = torch.full((0, 5), 7.0, device=cuda_dev)
    gq_lib.mul_mat(q, "q4_0", 5, 64, torch.zeros((0, 64), device=cuda_dev), out=Y2)
    Y3 = torch.full((2, 0), 7.0, device=cuda_dev)
    gq_lib.mul_mat(q, "q8_0", 0, 64, torch.zeros((2, 64), device=cuda_dev), out=Y3)
    assert gq_lib.get_last_error() == 0


@pytest.mark.parametrize("t", ["q4_0", "q8_0"])
def test_batched_mixed_shapes(gq_lib, oracle_mod, cuda_dev, t):
    """Problems of different M and K (fast and generic mixed) in one batched call."""
    shapes = [(256, 2048), (2048, 2048), (7, 96), (300, 5632), (1, 256), (64, 11008),
              (0, 512), (5, 0)]
    N = 3
    items, refs = [], []
    for i, (M, K) in enumerate(shapes):
        W = _np_weights(M, K, seed=50 + i) if M * K else np.zeros((M, K), np.float32)
        q = oracle_mod.quantize(t, W) if M * K else np.zeros((M, 0), np.uint8)
        X = workloads.activations(N, K, seed=60 + i).numpy()
        Yd = torch.full((N, M), 9.0, device=cuda_dev)
        items.append((torch.from_numpy(q).contiguous().to(cuda_dev), M, K,
                      torch.from_numpy(X).to(cuda_dev), Yd))
        refs.append((q, X))
    gq_lib.mul_mat_batched(items, t, N)
    for (M, K), (q, X), it in zip(shapes, refs, items):
        Y = it[4].cpu().numpy()
        if M == 0:
            continue
        if K == 0:
            assert not Y.any()
            continue
        check_tolerance(Y, oracle_mod.mul_mat(t, q, M, K, X),
                        oracle_mod.dequantize(t, q, M, K), X, f"M={M} K={K}")
    assert gq_lib.get_last_error() == 0


# ------------------------------------------------------------------------------------
# Full-size workloads, in the launch configuration the benchmark times, on sampled rows
# ------------------------------------------------------------------------------------
def _sampled_step_check(gq_lib, oracle_mod, dev, workload, t, N, shapes, rows_per_mat=6):
    from block_quantized_matmul_gq_gb300.weightset import QuantizedWeightSet
    rng = np.random.default_rng(workload * 10 + N)
    keep = {j: np.unique(np.concatenate([[0, s.M - 1], rng.integers(0, s.M, rows_per_mat)]))
            for j, s in enumerate(shapes)}
    ws = QuantizedWeightSet.synthetic(workload, shapes, t, dev, keep_rows=keep)
    xs, ys = ws.make_io(N, workload, dev)
    ws.run(ws.problem_arrays(xs, ys), N)
    assert gq_lib.get_last_error() == 0
    worst = 0.0
    for j, s in enumerate(shapes):
        rows = keep[j]
        W_rows = ws.kept[j].numpy()
        q_rows = oracle_mod.quantize(t, W_rows)
        got_blocks = ws.mats[j].blocks[torch.as_tensor(rows, device=dev)].cpu().numpy()
        assert np.array_equal(got_blocks, q_rows), (j, s)
        X = xs[j].cpu().numpy()
        Y_ref = oracle_mod.mul_mat(t, q_rows, len(rows), s.K, X)
        Y = ys[j].cpu().numpy()[:, rows]
        worst = max(worst, check_tolerance(Y, Y_ref, oracle_mod.dequantize(t, q_rows, len(rows), s.K),
                                           X, f"{s.name}[{j}]"))
    return worst


def test_tinyllama_decode_step_q4_0_full_size(gq_lib, oracle_mod, cuda_dev):
    """All 155 matmuls of the TinyLLaMA decode step, Q4_0, N = 1, batched as timed."""
    _sampled_step_check(gq_lib, oracle_mod, cuda_dev, 2, "q4_0", 1,
                        workloads.tinyllama_decode_set())


@pytest.mark.parametrize("N", [1, 16])
def test_tinyllama_decode_step_q8_0_full_size(gq_lib, oracle_mod, cuda_dev, N):
    _sampled_step_check(gq_lib, oracle_mod, cuda_dev, 3, "q8_0", N,
                        workloads.tinyllama_decode_set(), rows_per_mat=3)


@pytest.mark.parametrize("N", [1, 16])
def test_llama7b_shapes_full_size(gq_lib, oracle_mod, cuda_dev, N):
    _sampled_step_check(gq_lib, oracle_mod, cuda_dev, 5, "q4_0", N, workloads.llama7b_set())


# ------------------------------------------------------------------------------------
# Tensor-core paths (N >= 3, K % 256 == 0): bf16 operands, fp32 accumulation
# ------------------------------------------------------------------------------------
# Few-tile shapes also run the cluster split-K form: (300, 512, 100) and (129, 768, 300) split
# K two ways (the latter unevenly, ragged M), (1000, 2048, 257), (520, 1792, 130) and
# (1001, 1280, 70) four ways (7 and 5 super-steps: uneven shares; M % 4 != 0 in the last);
# (128, 256, 65) has one super-step and does not split.
GEMM = [(128, 256, 64), (7, 256, 64), (300, 512, 100), (129, 768, 300), (1000, 2048, 257),
        (256, 5632, 64), (128, 256, 65), (520, 1792, 130), (1001, 1280, 70)]


@pytest.mark.parametrize("t", ["q4_0", "q8_0", "q4_k"])
@pytest.mark.parametrize("M,K,N", GEMM)
def test_gemm_matches_oracle(gq_lib, oracle_mod, cuda_dev, t, M, K, N):
    assert gq_lib.workspace_size(t, M, K, N) >= N * K * 2
    Y, Y_ref, What, X = run_mul_mat(gq_lib, oracle_mod, cuda_dev, t, M, K, N, seed=M + K + N)
    check_tolerance(Y, Y_ref, What, X, f"gemm {t} M={M} K={K} N={N}")


@pytest.mark.parametrize("t", ["q4_0", "q8_0", "q4_k"])
def test_gemm_one_hot_returns_bf16_weights(gq_lib, oracle_mod, cuda_dev, t):
    """X = e_k: Y[n][m] is bf16(What[m][k]) exactly (one nonzero product, fp32 sum). This
    pins the in-kernel dequantization, the swizzled operand layouts and the descriptors."""
    M, K = 200, 512
    ks = list(range(0, K, 7))[:64] + [K - 1]
    X = np.zeros((len(ks), K), np.float32)
    for n, k in enumerate(ks):
        X[n, k] = 1.0
    Y, _, What, _ = run_mul_mat(gq_lib, oracle_mod, cuda_dev, t, M, K, len(ks), X=X)
    wb = torch.from_numpy(What).to(torch.bfloat16).float().numpy()
    for n, k in enumerate(ks):
        assert np.array_equal(Y[n], wb[:, k]), k


def test_gemm_workspace_entry_point(gq_lib, oracle_mod, cuda_dev):
    M, K, N = 256, 1024, 128
    W = _np_weights(M, K, seed=21)
    q = torch.from_numpy(oracle_mod.quantize("q4_0", W)).to(cuda_dev)
    X = workloads.activations(N, K, seed=22).to(cuda_dev)
    need = gq_lib.workspace_size("q4_0", M, K, N)
    assert need == N * K * 2
    assert gq_lib.workspace_size("q4_0", M, K, 2) == 0          # CUDA-core decode: none
    # tensor-core decode: 16-token X tiles, two 128 x 16 partial tiles per CTA (<= 256) and
    # 4 KB of split-tile counters
    assert gq_lib.workspace_size("q4_0", M, K, 8) == 16 * K * 2 + 2 * 256 * 128 * 16 * 4 + 4096
    ws = torch.empty(need, dtype=torch.uint8, device=cuda_dev)
    y1 = gq_lib.mul_mat_ws(q, "q4_0", M, K, X, ws)
    y2 = gq_lib.mul_mat(q, "q4_0", M, K, X)
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32))
    with pytest.raises(gq_lib.GQError) as e:
        gq_lib.mul_mat_ws(q, "q4_0", M, K, X, None)
    assert e.value.status == -1
    with pytest.raises(gq_lib.GQError) as e:
        gq_lib.mul_mat_ws(q, "q4_0", M, K, X, ws[: need - 256])
    assert e.value.status == -2
    assert gq_lib.get_last_error() == 0


def test_gemm_deterministic(gq_lib, cuda_dev):
    M, K, N = 1024, 2048, 320
    W = workloads.weights(M, K, 31, device=cuda_dev)
    q = gq_lib.quantize(W, "q4_0")
    X = workloads.activations(N, K, 32, device=cuda_dev)
    y1 = gq_lib.mul_mat(q, "q4_0", M, K, X)
    y2 = gq_lib.mul_mat(q, "q4_0", M, K, X)
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32))


def test_tinyllama_prefill_full_size(gq_lib, oracle_mod, cuda_dev):
    """gate / down / lm_head at N = 512 tokens, Q4_0, one call per matrix."""
    _sampled_step_check(gq_lib, oracle_mod, cuda_dev, 4, "q4_0", 512,
                        workloads.tinyllama_prefill_set(), rows_per_mat=3)


def test_llama7b_prefill_full_size(gq_lib, oracle_mod, cuda_dev):
    _sampled_step_check(gq_lib, oracle_mod, cuda_dev, 5, "q4_0", 2048, workloads.llama7b_set(),
                        rows_per_mat=2)


# Shapes whose 256-token tiles fill two or more waves take 512-token tiles (two N = 256
# MMAs per dequantized A stage): N = 300 leaves the second half mostly empty, N = 777 a
# 9-token second half in the last tile.
GEMM_WIDE = [(10240, 512, 300), (9728, 768, 777)]


@pytest.mark.parametrize("t", ["q4_0", "q8_0", "q4_k"])
@pytest.mark.parametrize("M,K,N", GEMM_WIDE)
def test_gemm_wide_tiles_sampled(gq_lib, oracle_mod, cuda_dev, t, M, K, N):
    _sampled_step_check(gq_lib, oracle_mod, cuda_dev, 7, t, N, [workloads.MatShape("wide", M, K)],
                        rows_per_mat=24)


# Enough 256-token tiles to fill the SMs, too few tokens for 512-token tiles: the plain
# tile kernel, with a last tile of 124 (M % 4 == 0) or 127 rows and a 200-token tail.
GEMM_UNSPLIT = [(10236, 256, 200), (10239, 256, 200)]


@pytest.mark.parametrize("t", ["q4_0", "q8_0", "q4_k"])
@pytest.mark.parametrize("M,K,N", GEMM_UNSPLIT)
def test_gemm_unsplit_tiles_sampled(gq_lib, oracle_mod, cuda_dev, t, M, K, N):
    _sampled_step_check(gq_lib, oracle_mod, cuda_dev, 8, t, N, [workloads.MatShape("tile", M, K)],
                        rows_per_mat=24)


# Several waves of 256-token tiles with ragged edges: 471 tiles (3.1 waves) with a 31-row
# last row block and an 8-token tail; 400 tiles (2.6 waves) with a 4-token tail.
GEMM_MULTIWAVE = [(19999, 256, 520), (25600, 512, 260)]


@pytest.mark.parametrize("t", ["q4_0", "q8_0", "q4_k"])
@pytest.mark.parametrize("M,K,N", GEMM_MULTIWAVE)
def test_gemm_multiwave_tiles_sampled(gq_lib, oracle_mod, cuda_dev, t, M, K, N):
    _sampled_step_check(gq_lib, oracle_mod, cuda_dev, 9, t, N, [workloads.MatShape("tiles", M, K)],
                        rows_per_mat=24)


@pytest.mark.parametrize("t", ["q4_0", "q8_0", "q4_k"])
def test_gemm_multiwave_tiles_deterministic(gq_lib, cuda_dev, t):
    M, K, N = GEMM_MULTIWAVE[0]
    q = gq_lib.quantize(workloads.weights(M, K, 10, device=cuda_dev), t)
    X = workloads.activations(N, K, 11, device=cuda_dev)
    y1 = gq_lib.mul_mat(q, t, M, K, X)
    y2 = gq_lib.mul_mat(q, t, M, K, X)
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32))
    assert gq_lib.get_last_error() == 0


@pytest.mark.parametrize("t", ["q4_0", "q8_0", "q4_k"])
def test_gemm_wide_tiles_deterministic(gq_lib, cuda_dev, t):
    M, K, N = GEMM_WIDE[1]
    q = gq_lib.quantize(workloads.weights(M, K, 8, device=cuda_dev), t)
    X = workloads.activations(N, K, 9, device=cuda_dev)
    y1 = gq_lib.mul_mat(q, t, M, K, X)
    y2 = gq_lib.mul_mat(q, t, M, K, X)
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32))
    assert gq_lib.get_last_error() == 0


# ------------------------------------------------------------------------------------
# Tensor-core decode (3 <= N <= 64, K % 256 == 0): grouped, bf16 operands
# ------------------------------------------------------------------------------------
DECODE_TC = [(1, 256, 5), (7, 2048, 8), (129, 2048, 16), (1000, 2048, 17), (300, 5632, 32),
             (200, 11008, 33), (128, 512, 64), (2048, 4096, 16)]


@pytest.mark.parametrize("t", ["q4_0", "q8_0", "q4_k"])
@pytest.mark.parametrize("M,K,N", DECODE_TC)
def test_decode_tc_matches_oracle(gq_lib, oracle_mod, cuda_dev, t, M, K, N):
    Y, Y_ref, What, X = run_mul_mat(gq_lib, oracle_mod, cuda_dev, t, M, K, N, seed=3 * M + K + N)
    check_tolerance(Y, Y_ref, What, X, f"decode-tc {t} M={M} K={K} N={N}")


@pytest.mark.parametrize("t", ["q4_0", "q8_0", "q4_k"])
@pytest.mark.parametrize("N", [4, 16, 40])
def test_decode_tc_one_hot_returns_operand_weights(gq_lib, oracle_mod, cuda_dev, t, N):
    """X = e_k returns column k of the weights exactly as the MMA saw them. Q4_0 and Q4_K
    with up to 16 tokens multiply the exact codes (c - 8, q) and apply the scales (Q4_K: and
    the mins, against the block sums of X) in fp32, so they return What itself; the other
    forms (Q4_K: What as gq_dequantize writes it) dequantize to bf16 and return bf16(What).
    This pins the operand layout, the per-block accumulators and the scale of each block."""
    M, K = 300, 1024
    ks = [(37 * n) % K for n in range(N)]
    X = np.zeros((N, K), np.float32)
    for n, k in enumerate(ks):
        X[n, k] = 1.0
    Y, _, What, _ = run_mul_mat(gq_lib, oracle_mod, cuda_dev, t, M, K, N, X=X)
    if t in ("q4_0", "q4_k") and N <= 16:
        expect = What
    else:
        expect = torch.from_numpy(What).to(torch.bfloat16).float().numpy()
    for n, k in enumerate(ks):
        assert np.array_equal(Y[n], expect[:, k]), (n, k)


@pytest.mark.parametrize("t", ["q4_0", "q8_0", "q4_k"])
def test_decode_tc_batched_mixed_shapes(gq_lib, oracle_mod, cuda_dev, t):
    """One grouped tensor-core launch over problems of different M and K, with a
    CUDA-core-only shape (K % 256 != 0) mixed in."""
    shapes = [(256, 2048), (2048, 2048), (7, 256), (300, 5632), (1, 1024), (64, 11008),
              (33, 96)]
    if t == "q4_k":   # whole super-blocks only
        shapes = [s for s in shapes if s[1] % 256 == 0]
    N = 16
    items, refs = [], []
    for i, (M, K) in enumerate(shapes):
        q = oracle_mod.quantize(t, _np_weights(M, K, seed=90 + i))
        X = workloads.activations(N, K, seed=95 + i).numpy()
        items.append((torch.from_numpy(q).to(cuda_dev), M, K, torch.from_numpy(X).to(cuda_dev),
                      torch.full((N, M), 9.0, device=cuda_dev)))
        refs.append((q, X))
    gq_lib.mul_mat_batched(items, t, N)
    for (M, K), (q, X), it in zip(shapes, refs, items):
        check_tolerance(it[4].cpu().numpy(), oracle_mod.mul_mat(t, q, M, K, X),
                        oracle_mod.dequantize(t, q, M, K), X, f"M={M} K={K}")
    assert gq_lib.get_last_error() == 0


def test_decode_tc_deterministic(gq_lib, cuda_dev):
    M, K, N = 3000, 5632, 16
    q = gq_lib.quantize(workloads.weights(M, K, 41, device=cuda_dev), "q8_0")
    X = workloads.activations(N, K, 42, device=cuda_dev)
    y1 = gq_lib.mul_mat(q, "q8_0", M, K, X)
    y2 = gq_lib.mul_mat(q, "q8_0", M, K, X)
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32))


@pytest.mark.parametrize("N", [16, 96])
def test_batched_ws_records_into_a_graph(gq_lib, cuda_dev, N):
    """The caller-owned-workspace batched call allocates nothing, so it can be captured into
    a CUDA graph on any stream; replays give the same bits as a direct call."""
    shapes = [(256, 2048), (640, 5632), (33, 96)]
    items = []
    for i, (M, K) in enumerate(shapes):
        q = gq_lib.quantize(workloads.weights(M, K, 60 + i, device=cuda_dev), "q4_0")
        items.append((q, M, K, workloads.activations(N, K, 70 + i, device=cuda_dev),
                      torch.empty((N, M), device=cuda_dev)))
    arr = gq_lib.make_problems(items)
    need = gq_lib.batched_workspace_size(arr, "q4_0", N)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device=cuda_dev)
    gq_lib.mul_mat_batched_ws(arr, "q4_0", N, ws)
    torch.cuda.synchronize()
    direct = [it[4].clone() for it in items]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        gq_lib.mul_mat_batched_ws(arr, "q4_0", N, ws)
    for it in items:
        it[4].zero_()
    g.replay()
    torch.cuda.synchronize()
    for d, it in zip(direct, items):
        assert torch.equal(d.view(torch.int32), it[4].view(torch.int32))
    with pytest.raises(gq_lib.GQError):
        gq_lib.mul_mat_batched_ws(arr, "q4_0", N, None)
    assert gq_lib.get_last_error() == 0


# ------------------------------------------------------------------------------------
# Quantized activations (gq_mul_mat_q8x): X quantized per 32-block like Q8_0, integer
# block sums ("A Complete Guide to llama.cpp ...", section 2.2)
# ------------------------------------------------------------------------------------
Q8X = [(7, 256, 1), (300, 2048, 3), (129, 5632, 8), (64, 11008, 5), (1000, 2048, 16),
       (33, 4096, 9), (257, 1024, 2)]


def _q8x_bound(oracle_mod, t, q, M, K, X):
    """Worst-case fp32 accumulation bound of the block sums: (blocks + 8) * 2^-24 times
    sum |What| |Xhat| (Xhat the Q8_0-dequantized X), per element."""
    wa = np.abs(oracle_mod.dequantize(t, q, M, K).astype(np.float64))
    N = X.shape[0]
    xa = np.abs(oracle_mod.dequantize("q8_0", oracle_mod.quantize("q8_0", X), N, K)
                .astype(np.float64))
    return (K // 32 + 8) * 2.0 ** -24 * (xa @ wa.T) + 1e-30


@pytest.mark.parametrize("t", ["q4_0", "q8_0"])
@pytest.mark.parametrize("M,K,N", Q8X)
def test_q8x_matches_oracle(gq_lib, oracle_mod, cuda_dev, t, M, K, N):
    W = _np_weights(M, K, seed=M + 3 * K)
    q = oracle_mod.quantize(t, W)
    X = workloads.activations(N, K, seed=N + 5 * K).numpy()
    Y = gq_lib.mul_mat_q8x(torch.from_numpy(q).to(cuda_dev), t, M, K,
                           torch.from_numpy(X).to(cuda_dev)).cpu().numpy()
    Y_ref = oracle_mod.mul_mat_q8x(t, q, M, K, X)
    err = np.abs(Y.astype(np.float64) - Y_ref.astype(np.float64))
    assert np.all(err <= _q8x_bound(oracle_mod, t, q, M, K, X)), f"q8x {t} M={M} K={K} N={N}"
    assert gq_lib.get_last_error() == 0


@pytest.mark.parametrize("t", ["q4_0", "q8_0"])
def test_q8x_accuracy_against_exact_product(gq_lib, oracle_mod, cuda_dev, t):
    """Quantizing X moves the result by far less than the mul_mat tolerance on the
    seeded N(0, 1) activations (the method's own error, measured)."""
    M, K, N = 512, 2048, 4
    W = _np_weights(M, K, seed=91)
    q = oracle_mod.quantize(t, W)
    X = workloads.activations(N, K, seed=92).numpy()
    Y = gq_lib.mul_mat_q8x(torch.from_numpy(q).to(cuda_dev), t, M, K,
                           torch.from_numpy(X).to(cuda_dev)).cpu().numpy()
    check_tolerance(Y, oracle_mod.mul_mat(t, q, M, K, X), oracle_mod.dequantize(t, q, M, K), X,
                    f"q8x vs exact {t}")


@pytest.mark.parametrize("t", ["q4_0", "q8_0"])
def test_q8x_batched_matches_oracle(gq_lib, oracle_mod, cuda_dev, t):
    shapes = [(256, 2048), (1000, 5632), (33, 256), (2048, 11008)]
    N = 6
    items, refs = [], []
    for i, (M, K) in enumerate(shapes):
        q = oracle_mod.quantize(t, _np_weights(M, K, seed=200 + i))
        X = workloads.activations(N, K, seed=300 + i).numpy()
        items.append((torch.from_numpy(q).to(cuda_dev), M, K, torch.from_numpy(X).to(cuda_dev),
                      torch.full((N, M), float("nan"), device=cuda_dev)))
        refs.append((q, X))
    gq_lib.mul_mat_q8x_batched(items, t, N)
    torch.cuda.synchronize()
    for (qd, M, K, Xd, Y), (q, X) in zip(items, refs):
        rows = np.arange(M) if M <= 1000 else np.array([0, 1, 127, 128, 1000, M - 1])
        Y_ref = oracle_mod.mul_mat_q8x_rows(t, q, M, K, X, rows)
        got = Y.cpu().numpy()[:, rows].astype(np.float64)
        bound = _q8x_bound(oracle_mod, t, q.reshape(M, -1)[rows].copy(), len(rows), K, X)
        assert np.all(np.abs(got - Y_ref) <= bound), f"batched q8x {t} M={M} K={K}"
    assert gq_lib.get_last_error() == 0


def test_q8x_rejects_unsupported_shapes(gq_lib, cuda_dev):
    q = torch.zeros((4, 96 // 32 * 18), dtype=torch.uint8, device=cuda_dev)
    X = torch.zeros((1, 96), device=cuda_dev)
    with pytest.raises(gq_lib.GQError) as e:
        gq_lib.mul_mat_q8x(q, "q4_0", 4, 96, X)
    assert e.value.status == -2
    q = torch.zeros((4, 256 // 32 * 18), dtype=torch.uint8, device=cuda_dev)
    Xb = torch.zeros(257 * 2, device=cuda_dev)
    with pytest.raises(gq_lib.GQError) as e:
        gq_lib.mul_mat_q8x(q, "q4_0", 4, 256, Xb[1:257].view(1, 256))
    assert e.value.status == -4


# ------------------------------------------------------------------------------------
# Fused adjacent steps ("Development Guide for Small AI Models (TinyLLaMA, etc.) Using
# C++", sections 4.1 and 4.4): RMSNorm ahead of the product, SwiGLU of gate/up after it
# ------------------------------------------------------------------------------------
# (M, K, N): N <= 2 with K % 256 == 0 runs fused in the decode kernel (K = 1024: whole-row
# stages; M = 20: few rows, so tiles split K between warps); the rest composes plain kernels
# (N = 8 tensor-core decode, N = 100 GEMM, K = 96 the generic kernel).
FUSED = [(300, 2048, 1), (129, 5632, 2), (129, 1024, 1), (20, 2048, 1), (7, 256, 2),
         (200, 2048, 8), (300, 512, 100), (40, 96, 2)]


def _gamma(K, seed):
    return (1.0 + 0.1 * np.random.default_rng(seed).standard_normal(K)).astype(np.float32)


@pytest.mark.parametrize("t", ["q4_0", "q8_0"])
@pytest.mark.parametrize("M,K,N", FUSED)
def test_mul_mat_rmsnorm_matches_oracle(gq_lib, oracle_mod, cuda_dev, t, M, K, N):
    """Y = RMSNorm(X) . What^T within 1e-3 ||RMSNorm(X)[n]|| ||What[m]||: the gq_mul_mat bound
    on the normalized activations (their norm from the page formula in fp64)."""
    W = _np_weights(M, K, seed=M + K)
    q = oracle_mod.quantize(t, W)
    X = workloads.activations(N, K, seed=N + 7).numpy() * np.float32(3.0)
    gamma, eps = _gamma(K, K), 1e-5
    Y = gq_lib.mul_mat_rmsnorm(torch.from_numpy(q).to(cuda_dev), t, M, K,
                               torch.from_numpy(X).to(cuda_dev),
                               torch.from_numpy(gamma).to(cuda_dev), eps).cpu().numpy()
    assert gq_lib.get_last_error() == 0
    Y_ref = oracle_mod.mul_mat_rmsnorm(t, q, M, K, X, gamma, eps)
    x64 = X.astype(np.float64)
    xhat = x64 / np.sqrt((x64 ** 2).mean(axis=1, keepdims=True) + eps) * gamma
    check_tolerance(Y, Y_ref, oracle_mod.dequantize(t, q, M, K), xhat, f"rmsnorm {t} {M} {K} {N}")


def _check_swiglu(oracle_mod, t, qg, qu, M, K, X, H, where):
    """|H - H_ref| <= 1.1 |U| e_G + |Swish(G)| e_U + 1e-6 |H_ref|: first-order propagation of
    the mul_mat bounds e = 1e-3 ||x|| ||w_m|| of both products (|Swish'| <= 1.1)."""
    H_ref = oracle_mod.mul_mat_swiglu(t, qg, qu, M, K, X).astype(np.float64)
    G = oracle_mod.mul_mat(t, qg, M, K, X).astype(np.float64)
    U = oracle_mod.mul_mat(t, qu, M, K, X).astype(np.float64)
    xn = np.linalg.norm(X.astype(np.float64), axis=1)[:, None]
    eg = TOL * xn * np.linalg.norm(oracle_mod.dequantize(t, qg, M, K).astype(np.float64), axis=1)[None, :]
    eu = TOL * xn * np.linalg.norm(oracle_mod.dequantize(t, qu, M, K).astype(np.float64), axis=1)[None, :]
    tol = 1.1 * np.abs(U) * eg + np.abs(G / (1.0 + np.exp(-G))) * eu + 1e-6 * np.abs(H_ref)
    err = np.abs(np.asarray(H, np.float64) - H_ref)
    bad = err > tol
    assert not bad.any(), f"{where}: {bad.sum()} out of tolerance, first {np.argwhere(bad)[0]}"


@pytest.mark.parametrize("t", ["q4_0", "q8_0"])
@pytest.mark.parametrize("M,K,N", FUSED)
def test_mul_mat_swiglu_matches_oracle(gq_lib, oracle_mod, cuda_dev, t, M, K, N):
    qg = oracle_mod.quantize(t, _np_weights(M, K, seed=M + 2 * K))
    qu = oracle_mod.quantize(t, _np_weights(M, K, seed=M + 3 * K))
    X = workloads.activations(N, K, seed=N + 11).numpy() * np.float32(4.0)
    H = gq_lib.mul_mat_swiglu(torch.from_numpy(qg).to(cuda_dev), torch.from_numpy(qu).to(cuda_dev),
                              t, M, K, torch.from_numpy(X).to(cuda_dev)).cpu().numpy()
    assert gq_lib.get_last_error() == 0
    _check_swiglu(oracle_mod, t, qg, qu, M, K, X, H, f"swiglu {t} {M} {K} {N}")


def test_fused_decode_full_size_and_deterministic(gq_lib, oracle_mod, cuda_dev):
    """TinyLLaMA at N = 1: the FFN gate/up pair (5632 x 2048) through the fused SwiGLU, and
    the final RMSNorm into the LM head (32000 x 2048); all outputs against the oracle, and
    bitwise-equal reruns."""
    M, K = 5632, 2048
    qg = gq_lib.quantize(workloads.weights(M, K, 95, device=cuda_dev), "q4_0")
    qu = gq_lib.quantize(workloads.weights(M, K, 96, device=cuda_dev), "q4_0")
    X = workloads.activations(1, K, 97)
    Xd = X.to(cuda_dev)
    H = gq_lib.mul_mat_swiglu(qg, qu, "q4_0", M, K, Xd)
    assert torch.equal(H.view(torch.int32), gq_lib.mul_mat_swiglu(qg, qu, "q4_0", M, K, Xd).view(torch.int32))
    _check_swiglu(oracle_mod, "q4_0", qg.cpu().numpy(), qu.cpu().numpy(), M, K, X.numpy(),
                  H.cpu().numpy(), "tinyllama ffn")
    Ml = 32000
    ql = gq_lib.quantize(workloads.weights(Ml, K, 98, device=cuda_dev), "q4_0")
    gamma = torch.from_numpy(_gamma(K, 99))
    Y = gq_lib.mul_mat_rmsnorm(ql, "q4_0", Ml, K, Xd, gamma.to(cuda_dev), 1e-5)
    assert torch.equal(Y.view(torch.int32),
                       gq_lib.mul_mat_rmsnorm(ql, "q4_0", Ml, K, Xd, gamma.to(cuda_dev), 1e-5).view(torch.int32))
    q_np = ql.cpu().numpy()
    Y_ref = oracle_mod.mul_mat_rmsnorm("q4_0", q_np, Ml, K, X.numpy(), gamma.numpy(), 1e-5)
    x64 = X.numpy().astype(np.float64)
    xhat = x64 / np.sqrt((x64 ** 2).mean(axis=1, keepdims=True) + 1e-5) * gamma.numpy()
    check_tolerance(Y.cpu().numpy(), Y_ref, oracle_mod.dequantize("q4_0", q_np, Ml, K), xhat, "lm_head")
    assert gq_lib.get_last_error() == 0


@pytest.mark.parametrize("t", ["q4_0", "q8_0"])
def test_fused_misaligned_inputs_take_the_composite_path(gq_lib, oracle_mod, cuda_dev, t):
    """gamma and X only 4-byte aligned: the decode kernel's 16-byte loads cannot take them,
    so both entry points compose plain kernels at N = 1 and must still match the oracle."""
    M, K, N = 96, 512, 1
    q = oracle_mod.quantize(t, _np_weights(M, K, seed=101))
    qu = oracle_mod.quantize(t, _np_weights(M, K, seed=102))
    X = workloads.activations(N, K, seed=103).numpy()
    gamma = _gamma(K, 104)
    xbuf = torch.zeros(N * K + 1, dtype=torch.float32, device=cuda_dev)
    xbuf[1:] = torch.from_numpy(X.reshape(-1)).to(cuda_dev)
    Xm = xbuf[1:].view(N, K)                      # 4-byte aligned, not 16
    gbuf = torch.zeros(K + 1, dtype=torch.float32, device=cuda_dev)
    gbuf[1:] = torch.from_numpy(gamma).to(cuda_dev)
    qd = torch.from_numpy(q).to(cuda_dev)
    Y = gq_lib.mul_mat_rmsnorm(qd, t, M, K, torch.from_numpy(X).to(cuda_dev), gbuf[1:], 1e-5)
    x64 = X.astype(np.float64)
    xhat = x64 / np.sqrt((x64 ** 2).mean(axis=1, keepdims=True) + 1e-5) * gamma
    check_tolerance(Y.cpu().numpy(), oracle_mod.mul_mat_rmsnorm(t, q, M, K, X, gamma, 1e-5),
                    oracle_mod.dequantize(t, q, M, K), xhat, "rmsnorm, gamma misaligned")
    H = gq_lib.mul_mat_swiglu(qd, torch.from_numpy(qu).to(cuda_dev), t, M, K, Xm)
    _check_swiglu(oracle_mod, t, q, qu, M, K, X, H.cpu().numpy(), "swiglu, X misaligned")
    assert gq_lib.get_last_error() == 0


# GEMM forms under back-to-back replay: 256-token tiles (80 tiles, unsplit), cluster split-K
# (4 and 2 ways), 512-token tiles (two MMA issuers for Q4_0 / Q4_K). Each call's stage rings run many phases and the next
# call starts right after the last; every replayed result must equal a single call's bits.
GEMM_REPLAY = [(10236, 256, 200), (1000, 2048, 257), (300, 512, 100), (10240, 512, 300)]


@pytest.mark.parametrize("t", ["q4_0", "q8_0", "q4_k"])
@pytest.mark.parametrize("M,K,N", GEMM_REPLAY)
def test_gemm_graph_replays_match_a_single_call(gq_lib, cuda_dev, t, M, K, N):
    q = gq_lib.quantize(workloads.weights(M, K, 61, device=cuda_dev), t)
    X = workloads.activations(N, K, 62, device=cuda_dev)
    ref = gq_lib.mul_mat(q, t, M, K, X)
    ws = torch.empty(gq_lib.workspace_size(t, M, K, N), dtype=torch.uint8, device=cuda_dev)
    outs = [torch.empty((N, M), device=cuda_dev) for _ in range(4)]
    gq_lib.mul_mat_ws(q, t, M, K, X, ws, out=outs[0])
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(12):
            gq_lib.mul_mat_ws(q, t, M, K, X, ws, out=outs[i % 4])
    for _ in range(5):
        g.replay()
    torch.cuda.synchronize()
    assert gq_lib.get_last_error() == 0
    for o in outs:
        assert torch.equal(o.view(torch.int32), ref.view(torch.int32))
