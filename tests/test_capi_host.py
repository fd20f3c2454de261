"""C ABI checks that need no GPU: the library loads, exports every function that
include/gq.h declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in ("gq.h", "gq_gguf.h")]


def declared_functions():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b(gq_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("gq_quantize_q4_0", "gq_quantize_q8_0", "gq_dequantize", "gq_mul_mat",
                 "gq_mul_mat_batched", "gq_get_last_error", "gq_block_bytes", "gq_row_bytes",
                 "gq_status_string", "gq_abi_version"):
        assert want in names


def test_library_exports_every_declared_symbol(gq_lib):
    lib = ctypes.CDLL(gq_lib.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in gq.h but not exported"
    assert set(declared_functions()) == set(gq_lib.EXPORTS)


def test_sizes(gq_lib):
    lib = gq_lib.lib
    assert lib.gq_abi_version() == 1
    assert lib.gq_block_bytes(2) == 18 and lib.gq_block_bytes(8) == 34
    assert lib.gq_block_bytes(5) == 0
    assert lib.gq_row_bytes(2, 2048) == 1152 and lib.gq_row_bytes(8, 5632) == 5984
    assert lib.gq_row_bytes(2, 33) == 0 and lib.gq_row_bytes(2, -32) == 0
    assert lib.gq_row_bytes(2, 0) == 0


def test_status_strings(gq_lib):
    for code in range(-8, 1):
        assert gq_lib.lib.gq_status_string(code)
    assert b"unknown" in gq_lib.lib.gq_status_string(-99)


# Fake device addresses: the library must reject these before dereferencing anything.
A16 = 0x7000_0000_0000
A4 = A16 + 4
A2 = A16 + 2


def test_mul_mat_argument_checks(gq_lib):
    mm = gq_lib.lib.gq_mul_mat
    assert mm(A16, 7, 4, 64, A16, 1, A16, None) == -3              # unknown type
    assert mm(A16, 2, 4, 48, A16, 1, A16, None) == -2              # K % 32
    assert mm(A16, 2, -1, 64, A16, 1, A16, None) == -2             # negative M
    assert mm(A16, 2, 4, 64, A16, -1, A16, None) == -2             # negative N
    assert mm(A16, 2, 1 << 31, 64, A16, 1, A16, None) == -2        # dimension too large
    assert mm(None, 2, 4, 64, A16, 1, A16, None) == -1             # NULL weights
    assert mm(A16, 2, 4, 64, None, 1, A16, None) == -1             # NULL X
    assert mm(A16, 2, 4, 64, A16, 1, None, None) == -1             # NULL Y
    assert mm(A4, 2, 4, 64, A16, 1, A16, None) == -4               # blocks not 16B aligned
    assert mm(A16, 2, 4, 64, A2, 1, A16, None) == -4               # X not 4B aligned
    assert mm(A16, 2, 4, 64, A16, 1, A2, None) == -4               # Y not 4B aligned
    assert mm(None, 2, 0, 64, None, 1, None, None) == 0            # M = 0: no-op
    assert mm(None, 2, 4, 64, None, 0, None, None) == 0            # N = 0: no-op


def test_batched_argument_checks(gq_lib):
    P = gq_lib.Problem
    arr = (P * 2)(P(A16, A16, A16, 4, 64), P(A16, A16, A16, 4, 48))
    bm = gq_lib.lib.gq_mul_mat_batched
    assert bm(arr, 2, 2, 1, None) == -2                            # second problem: K % 32
    assert bm(arr, 257, 2, 1, None) == -2                          # count > GQ_MAX_BATCH
    assert bm(arr, -1, 2, 1, None) == -2
    assert bm(arr, 1, 9, 1, None) == -3
    assert bm(None, 1, 2, 1, None) == -1
    assert bm(arr, 0, 2, 1, None) == 0
    arr2 = (P * 1)(P(A16, A16, A16, 0, 64))
    assert bm(arr2, 1, 2, 1, None) == 0                            # only empty problems


def test_quantize_dequantize_argument_checks(gq_lib):
    lib = gq_lib.lib
    for q in (lib.gq_quantize_q4_0, lib.gq_quantize_q8_0):
        assert q(A16, 4, 40, A16, None) == -2
        assert q(None, 4, 64, A16, None) == -1
        assert q(A2, 4, 64, A16, None) == -4
        assert q(A16, 4, 64, A4, None) == -4
        assert q(None, 0, 64, None, None) == 0
    dq = lib.gq_dequantize
    assert dq(A16, 3, 4, 64, A16, None) == -3
    assert dq(A4, 2, 4, 64, A16, None) == -4
    assert dq(A16, 2, 4, 64, None, None) == -1
    assert dq(None, 8, 0, 64, None, None) == 0


def test_binding_refuses_cpu_tensors(gq_lib):
    torch = pytest.importorskip("torch")
    with pytest.raises(ValueError, match="CUDA"):
        gq_lib.quantize(torch.zeros(4, 64), "q4_0", out=torch.zeros(4, 36, dtype=torch.uint8))


def test_selftest_limit_checked_on_host(gq_lib):
    assert gq_lib.lib.gq_selftest_wait_timeout(0, None) == -2
    assert gq_lib.lib.gq_selftest_wait_timeout(20_000_000, None) == -2


def test_mul_mat_q8x_argument_checks(gq_lib):
    f = gq_lib.lib.gq_mul_mat_q8x
    assert f(A16, 7, 4, 256, A16, 1, A16, None) == -3              # unknown type
    assert f(A16, 2, 4, 96, A16, 1, A16, None) == -2               # K % 256 (needs whole chunks)
    assert f(A16, 2, 4, 48, A16, 1, A16, None) == -2               # K % 32
    assert f(A16, 2, 4, 256, A4, 1, A16, None) == -4               # X not 16-byte aligned
    assert f(A4, 2, 4, 256, A16, 1, A16, None) == -4               # W not 16-byte aligned
    assert f(None, 2, 4, 256, A16, 1, A16, None) == -1             # NULL W
    assert f(A16, 2, 0, 256, A16, 1, A16, None) == 0               # empty: nothing to do
    fb = gq_lib.lib.gq_mul_mat_q8x_batched
    assert fb(None, 0, 2, 1, None) == 0
    assert fb(None, 1, 2, 1, None) == -1
    assert fb(None, 300, 2, 1, None) == -2
    arr = gq_lib.make_problems([])
    assert fb(arr, 1, 7, 1, None) == -3


def test_fused_entry_points_argument_checks(gq_lib):
    rn = gq_lib.lib.gq_mul_mat_rmsnorm
    assert rn(A16, 7, 4, 64, A16, A16, 1e-5, 1, A16, None) == -3     # unknown type
    assert rn(A16, 2, 4, 48, A16, A16, 1e-5, 1, A16, None) == -2     # K % 32
    assert rn(A16, 2, 4, 64, A16, A16, -1.0, 1, A16, None) == -2     # eps < 0
    assert rn(A16, 2, 4, 64, A16, A16, float("nan"), 1, A16, None) == -2
    assert rn(A16, 2, 4, 64, A16, A16, float("inf"), 1, A16, None) == -2
    assert rn(A16, 2, 4, 0, A16, A16, 1e-5, 1, A16, None) == -2      # mean of nothing
    assert rn(A16, 2, 4, 64, A16, None, 1e-5, 1, A16, None) == -1    # gamma missing
    assert rn(A16, 2, 4, 64, A16, A2, 1e-5, 1, A16, None) == -4      # gamma misaligned
    assert rn(A4, 2, 4, 64, A16, A16, 1e-5, 1, A16, None) == -4      # W misaligned
    assert rn(A16, 2, 0, 64, A16, A16, 1e-5, 1, A16, None) == 0      # M == 0: nothing to do
    sw = gq_lib.lib.gq_mul_mat_swiglu
    assert sw(A16, A16, 7, 4, 64, A16, 1, A16, None) == -3
    assert sw(A16, A16, 2, 4, 48, A16, 1, A16, None) == -2
    assert sw(A16, None, 2, 4, 64, A16, 1, A16, None) == -1          # up missing
    assert sw(A16, A4, 2, 4, 64, A16, 1, A16, None) == -4            # up misaligned
    assert sw(None, A16, 2, 4, 64, A16, 1, A16, None) == -1          # gate missing
    assert sw(A16, A16, 2, 4, 64, A16, 0, A16, None) == 0            # N == 0


def test_q4_k_sizes_and_host_checks(gq_lib):
    """Q4_K super-blocks: 144 bytes per 256 weights; K must hold whole super-blocks, and the
    entry points that take only 32-weight blocks refuse the type before any CUDA call."""
    lib = gq_lib.lib
    assert gq_lib.Q4_K == 12 and gq_lib.TYPES["q4_k"] == 12
    assert lib.gq_block_bytes(12) == 144
    assert lib.gq_row_bytes(12, 2048) == 8 * 144 and lib.gq_row_bytes(12, 5632) == 22 * 144
    assert lib.gq_row_bytes(12, 288) == 0 and lib.gq_row_bytes(12, 0) == 0
    q = lib.gq_quantize_q4_k
    assert q(A16, 4, 288, A16, None) == -2                          # K % 256
    assert q(A16, 4, 32, A16, None) == -2
    assert q(None, 4, 256, A16, None) == -1
    assert q(A2, 4, 256, A16, None) == -4
    assert q(A16, 4, 256, A4, None) == -4
    assert q(None, 0, 256, None, None) == 0
    assert lib.gq_dequantize(A16, 12, 4, 288, A16, None) == -2
    mm = lib.gq_mul_mat
    assert mm(A16, 12, 4, 288, A16, 1, A16, None) == -2             # K % 256
    assert mm(A4, 12, 4, 256, A16, 1, A16, None) == -4
    assert mm(None, 12, 0, 256, None, 1, None, None) == 0
    assert lib.gq_mul_mat_noalloc(A16, 12, 4, 288, A16, 1, A16, None) == -2
    # the workspace of Q4_0 on every path (none for N <= 2, X tiles and partial sums for the
    # tensor-core decode, the bf16 copy of X for prefill), plus at 3..16 tokens the X block
    # sums of the scaled form: 1 KB per 256 k
    for N in (1, 2, 40, 64, 512):
        assert lib.gq_mul_mat_workspace_size(12, 64, 2048, N) == \
            lib.gq_mul_mat_workspace_size(2, 64, 2048, N)
    for N in (3, 4, 16):
        assert lib.gq_mul_mat_workspace_size(12, 64, 2048, N) == \
            lib.gq_mul_mat_workspace_size(2, 64, 2048, N) + 2048 // 256 * 1024
    assert lib.gq_mul_mat_workspace_size(12, 64, 2048, 2) == 0
    assert lib.gq_mul_mat_workspace_size(12, 64, 2048, 512) == 512 * 2048 * 2
    # quantized activations pair with 32-weight blocks only
    assert lib.gq_mul_mat_q8x(A16, 12, 4, 256, A16, 1, A16, None) == -3
    P = gq_lib.Problem
    arr = (P * 1)(P(A16, A16, A16, 4, 256))
    assert lib.gq_mul_mat_q8x_batched(arr, 1, 12, 1, None) == -3
    arr_bad = (P * 1)(P(A16, A16, A16, 4, 288))
    assert lib.gq_mul_mat_batched(arr_bad, 1, 12, 1, None) == -2
    assert lib.gq_mul_mat_rmsnorm(A16, 12, 4, 288, A16, A16, 1e-5, 1, A16, None) == -2
    assert lib.gq_mul_mat_swiglu(A16, A16, 12, 4, 288, A16, 1, A16, None) == -2
