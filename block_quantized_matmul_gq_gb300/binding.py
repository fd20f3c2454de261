"""Python face of libgq (include/gq.h): argument marshalling only.

Every call passes device pointers and sizes straight to the C ABI on torch's current
CUDA stream; all arithmetic runs in the library's sm_103a kernels. There is no CPU path:
importing this module fails loudly if libgq.so has not been built, and the calls refuse
CPU tensors, except pinned (page-locked) host tensors for activations and outputs, which
the kernels read and write in place (include/gq.h).
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgq.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"libgq.so not found at {LIB_PATH}: build it first "
        "(python -m block_quantized_matmul_gq_gb300.build); there is no fallback path")

lib = None

Q4_0 = 2
Q8_0 = 8
Q4_K = 12
TYPES = {"q4_0": Q4_0, "q8_0": Q8_0, "q4_k": Q4_K, Q4_0: Q4_0, Q8_0: Q8_0, Q4_K: Q4_K}
MAX_BATCH = 256

STATUS = {0: "GQ_OK", -1: "GQ_ERR_NULL", -2: "GQ_ERR_SHAPE", -3: "GQ_ERR_TYPE",
          -4: "GQ_ERR_ALIGN", -5: "GQ_ERR_CUDA", -6: "GQ_ERR_TIMEOUT", -7: "GQ_ERR_FORMAT",
          -8: "GQ_ERR_IO"}

# Every symbol declared in include/gq.h.
EXPORTS = ("gq_abi_version", "gq_block_bytes", "gq_row_bytes", "gq_quantize_q4_0",
           "gq_quantize_q8_0", "gq_quantize_q4_k", "gq_dequantize", "gq_mul_mat", "gq_mul_mat_workspace_size",
           "gq_mul_mat_ws", "gq_mul_mat_noalloc", "gq_mul_mat_batched",
           "gq_mul_mat_batched_workspace_size", "gq_mul_mat_batched_ws", "gq_mul_mat_q8x",
           "gq_mul_mat_q8x_batched", "gq_mul_mat_rmsnorm", "gq_mul_mat_swiglu",
           "gq_get_last_error",
           "gq_selftest_wait_timeout", "gq_status_string",
           # include/gq_gguf.h
           "gq_gguf_open", "gq_gguf_close", "gq_gguf_version", "gq_gguf_tensor_count",
           "gq_gguf_kv_count", "gq_gguf_alignment", "gq_gguf_tensor_info",
           "gq_gguf_find_tensor", "gq_gguf_tensor_data", "gq_gguf_tensor_matrix",
           "gq_gguf_upload", "gq_gguf_find_key", "gq_gguf_kv_key", "gq_gguf_kv_type",
           "gq_gguf_kv_int", "gq_gguf_kv_float", "gq_gguf_kv_string", "gq_gguf_kv_array")


class Problem(ctypes.Structure):
    """gq_mul_mat_problem."""
    _fields_ = [("W_blocks", ctypes.c_void_p), ("X", ctypes.c_void_p), ("Y", ctypes.c_void_p),
                ("M", ctypes.c_int64), ("K", ctypes.c_int64)]


class GgufTensor(ctypes.Structure):
    """gq_gguf_tensor."""
    _fields_ = [("name", ctypes.c_char_p), ("n_dims", ctypes.c_uint32),
                ("type", ctypes.c_uint32), ("ne", ctypes.c_int64 * 4),
                ("offset", ctypes.c_uint64), ("nbytes", ctypes.c_uint64)]


def load(path: str = LIB_PATH):
    """(Re)binds this module to the libgq shared library at `path` (default: the in-tree
    build) and declares the C signatures of include/gq.h."""
    global lib
    L = ctypes.CDLL(path)
    i64, i32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
    L.gq_abi_version.argtypes, L.gq_abi_version.restype = [], i32
    L.gq_block_bytes.argtypes, L.gq_block_bytes.restype = [ctypes.c_int], ctypes.c_size_t
    L.gq_row_bytes.argtypes, L.gq_row_bytes.restype = [ctypes.c_int, i64], ctypes.c_size_t
    for q in (L.gq_quantize_q4_0, L.gq_quantize_q8_0, L.gq_quantize_q4_k):
        q.argtypes, q.restype = [vp, i64, i64, vp, vp], ctypes.c_int
    L.gq_dequantize.argtypes = [vp, ctypes.c_int, i64, i64, vp, vp]
    L.gq_dequantize.restype = ctypes.c_int
    L.gq_mul_mat.argtypes = [vp, ctypes.c_int, i64, i64, vp, i64, vp, vp]
    L.gq_mul_mat.restype = ctypes.c_int
    L.gq_mul_mat_workspace_size.argtypes = [ctypes.c_int, i64, i64, i64]
    L.gq_mul_mat_workspace_size.restype = ctypes.c_size_t
    L.gq_mul_mat_ws.argtypes = [vp, ctypes.c_int, i64, i64, vp, i64, vp, vp, ctypes.c_size_t, vp]
    L.gq_mul_mat_ws.restype = ctypes.c_int
    L.gq_mul_mat_noalloc.argtypes = [vp, ctypes.c_int, i64, i64, vp, i64, vp, vp]
    L.gq_mul_mat_noalloc.restype = ctypes.c_int
    L.gq_mul_mat_batched.argtypes = [ctypes.POINTER(Problem), i32, ctypes.c_int, i64, vp]
    L.gq_mul_mat_batched.restype = ctypes.c_int
    L.gq_mul_mat_batched_workspace_size.argtypes = [ctypes.POINTER(Problem), i32, ctypes.c_int, i64]
    L.gq_mul_mat_batched_workspace_size.restype = ctypes.c_size_t
    L.gq_mul_mat_batched_ws.argtypes = [ctypes.POINTER(Problem), i32, ctypes.c_int, i64, vp,
                                        ctypes.c_size_t, vp]
    L.gq_mul_mat_batched_ws.restype = ctypes.c_int
    L.gq_mul_mat_q8x.argtypes = [vp, ctypes.c_int, i64, i64, vp, i64, vp, vp]
    L.gq_mul_mat_q8x.restype = ctypes.c_int
    L.gq_mul_mat_rmsnorm.argtypes = [vp, ctypes.c_int, i64, i64, vp, vp, ctypes.c_float, i64,
                                     vp, vp]
    L.gq_mul_mat_rmsnorm.restype = ctypes.c_int
    L.gq_mul_mat_swiglu.argtypes = [vp, vp, ctypes.c_int, i64, i64, vp, i64, vp, vp]
    L.gq_mul_mat_swiglu.restype = ctypes.c_int
    L.gq_mul_mat_q8x_batched.argtypes = [ctypes.POINTER(Problem), i32, ctypes.c_int, i64, vp]
    L.gq_mul_mat_q8x_batched.restype = ctypes.c_int
    L.gq_get_last_error.argtypes, L.gq_get_last_error.restype = [vp], ctypes.c_int
    L.gq_selftest_wait_timeout.argtypes = [i64, vp]
    L.gq_selftest_wait_timeout.restype = ctypes.c_int
    L.gq_status_string.argtypes, L.gq_status_string.restype = [ctypes.c_int], ctypes.c_char_p
    u32, u64, c = ctypes.c_uint32, ctypes.c_uint64, ctypes.c_char_p
    L.gq_gguf_open.argtypes, L.gq_gguf_open.restype = [c, ctypes.POINTER(vp)], ctypes.c_int
    L.gq_gguf_close.argtypes, L.gq_gguf_close.restype = [vp], None
    L.gq_gguf_version.argtypes, L.gq_gguf_version.restype = [vp], u32
    L.gq_gguf_tensor_count.argtypes, L.gq_gguf_tensor_count.restype = [vp], i64
    L.gq_gguf_kv_count.argtypes, L.gq_gguf_kv_count.restype = [vp], i64
    L.gq_gguf_alignment.argtypes, L.gq_gguf_alignment.restype = [vp], u64
    L.gq_gguf_tensor_info.argtypes = [vp, i64, ctypes.POINTER(GgufTensor)]
    L.gq_gguf_tensor_info.restype = ctypes.c_int
    L.gq_gguf_find_tensor.argtypes, L.gq_gguf_find_tensor.restype = [vp, c], i64
    L.gq_gguf_tensor_data.argtypes, L.gq_gguf_tensor_data.restype = [vp, i64], vp
    L.gq_gguf_tensor_matrix.argtypes = [vp, i64, ctypes.POINTER(ctypes.c_int),
                                        ctypes.POINTER(i64), ctypes.POINTER(i64)]
    L.gq_gguf_tensor_matrix.restype = ctypes.c_int
    L.gq_gguf_upload.argtypes, L.gq_gguf_upload.restype = [vp, i64, vp, ctypes.c_size_t, vp], ctypes.c_int
    L.gq_gguf_find_key.argtypes, L.gq_gguf_find_key.restype = [vp, c], i64
    L.gq_gguf_kv_key.argtypes, L.gq_gguf_kv_key.restype = [vp, i64], c
    L.gq_gguf_kv_type.argtypes, L.gq_gguf_kv_type.restype = [vp, i64], i32
    L.gq_gguf_kv_int.argtypes = [vp, i64, ctypes.POINTER(i64)]
    L.gq_gguf_kv_float.argtypes = [vp, i64, ctypes.POINTER(ctypes.c_double)]
    L.gq_gguf_kv_string.argtypes = [vp, i64, ctypes.POINTER(vp), ctypes.POINTER(u64)]
    L.gq_gguf_kv_array.argtypes = [vp, i64, ctypes.POINTER(u32), ctypes.POINTER(u64),
                                   ctypes.POINTER(vp)]
    for fn in (L.gq_gguf_kv_int, L.gq_gguf_kv_float, L.gq_gguf_kv_string, L.gq_gguf_kv_array):
        fn.restype = ctypes.c_int
    lib = L
    return L


load()


class GQError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = lib.gq_status_string(status).decode()
        super().__init__(f"{what}: {STATUS.get(status, status)} ({msg})")


def _check(status: int, what: str) -> None:
    if status != 0:
        raise GQError(status, what)


def _type(t) -> int:
    try:
        return TYPES[t]
    except KeyError:
        raise ValueError(f"unknown block type {t!r}") from None


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _dev(t: torch.Tensor, dtype, name: str) -> int:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (libgq has no CPU path)")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _act(t: torch.Tensor, dtype, name: str) -> int:
    """X, Y, gamma: a CUDA tensor, or a pinned (page-locked) host tensor, which the device
    addresses directly (include/gq.h: the kernels read and write it over the host link)."""
    if not (t.is_cuda or t.is_pinned()):
        raise ValueError(f"{name} must be a CUDA tensor or pinned host memory "
                         "(libgq has no CPU path)")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _out_like(X: torch.Tensor, shape) -> torch.Tensor:
    """Y where X lives: on X's device, or pinned host memory for a pinned host X."""
    if X.is_cuda:
        return torch.empty(shape, dtype=torch.float32, device=X.device)
    return torch.empty(shape, dtype=torch.float32, pin_memory=True)


def block_bytes(t) -> int:
    return int(lib.gq_block_bytes(_type(t)))


def row_bytes(t, K: int) -> int:
    return int(lib.gq_row_bytes(_type(t), K))


def quantize(W: torch.Tensor, t, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """fp32 (M, K) CUDA tensor -> uint8 (M, row_bytes) blocks."""
    M, K = W.shape
    if out is None:
        out = torch.empty((M, row_bytes(t, K)), dtype=torch.uint8, device=W.device)
    fn = {Q4_0: lib.gq_quantize_q4_0, Q8_0: lib.gq_quantize_q8_0,
          Q4_K: lib.gq_quantize_q4_k}[_type(t)]
    _check(fn(_dev(W, torch.float32, "W"), M, K, _dev(out, torch.uint8, "W_blocks"),
              _stream(stream)), "gq_quantize")
    return out


def dequantize(blocks: torch.Tensor, t, M: int, K: int, out: torch.Tensor | None = None,
               stream=None) -> torch.Tensor:
    if out is None:
        out = torch.empty((M, K), dtype=torch.float32, device=blocks.device)
    _check(lib.gq_dequantize(_dev(blocks, torch.uint8, "W_blocks"), _type(t), M, K,
                             _dev(out, torch.float32, "W_out"), _stream(stream)),
           "gq_dequantize")
    return out


def mul_mat(blocks: torch.Tensor, t, M: int, K: int, X: torch.Tensor,
            out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Y (N, M) = X (N, K) . What^T."""
    if X.dim() == 1:
        X = X.view(1, -1)
    N = X.shape[0]
    if X.shape[1] != K:
        raise ValueError("X must be (N, K)")
    if out is None:
        out = _out_like(X, (N, M))
    _check(lib.gq_mul_mat(_dev(blocks, torch.uint8, "W_blocks"), _type(t), M, K,
                          _act(X, torch.float32, "X"), N, _act(out, torch.float32, "Y"),
                          _stream(stream)), "gq_mul_mat")
    return out


def workspace_size(t, M: int, K: int, N: int) -> int:
    return int(lib.gq_mul_mat_workspace_size(_type(t), M, K, N))


def mul_mat_ws(blocks: torch.Tensor, t, M: int, K: int, X: torch.Tensor,
               workspace: torch.Tensor | None, out: torch.Tensor | None = None,
               stream=None) -> torch.Tensor:
    """mul_mat with a caller-owned workspace (uint8 CUDA tensor of workspace_size bytes)."""
    if X.dim() == 1:
        X = X.view(1, -1)
    N = X.shape[0]
    if out is None:
        out = _out_like(X, (N, M))
    wp = _dev(workspace, torch.uint8, "workspace") if workspace is not None else None
    wn = workspace.numel() if workspace is not None else 0
    _check(lib.gq_mul_mat_ws(_dev(blocks, torch.uint8, "W_blocks"), _type(t), M, K,
                             _act(X, torch.float32, "X"), N, _act(out, torch.float32, "Y"),
                             wp, wn, _stream(stream)), "gq_mul_mat_ws")
    return out


def mul_mat_noalloc(blocks: torch.Tensor, t, M: int, K: int, X: torch.Tensor,
                    out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """mul_mat through gq_mul_mat_noalloc: the library allocates nothing (its tensor-core
    path uses a fixed 64 MiB device array). `out` lets the caller own Y as well."""
    if X.dim() == 1:
        X = X.view(1, -1)
    N = X.shape[0]
    if out is None:
        out = _out_like(X, (N, M))
    _check(lib.gq_mul_mat_noalloc(_dev(blocks, torch.uint8, "W_blocks"), _type(t), M, K,
                                  _act(X, torch.float32, "X"), N,
                                  _act(out, torch.float32, "Y"), _stream(stream)),
           "gq_mul_mat_noalloc")
    return out


def make_problems(items) -> ctypes.Array:
    """items: iterable of (blocks, M, K, X, Y) tensors (blocks on the device; X and Y on the
    device or in pinned host memory) -> a gq_mul_mat_problem array that can be handed to
    mul_mat_batched repeatedly (e.g. while capturing a graph)."""
    items = list(items)
    arr = (Problem * max(1, len(items)))()
    for i, (blocks, M, K, X, Y) in enumerate(items):
        arr[i] = Problem(_dev(blocks, torch.uint8, "W_blocks"), _act(X, torch.float32, "X"),
                         _act(Y, torch.float32, "Y"), M, K)
    arr._count = len(items)
    # The array holds raw device pointers: keep the tensors alive as long as it lives.
    arr._tensors = [(blocks, X, Y) for blocks, _, _, X, Y in items]
    return arr


def mul_mat_batched(problems, t, N: int, stream=None) -> None:
    """Independent problems sharing type and N, in one launch. `problems` is the result
    of make_problems() or an iterable of (blocks, M, K, X, Y)."""
    if not isinstance(problems, ctypes.Array):
        problems = make_problems(problems)
    _check(lib.gq_mul_mat_batched(problems, problems._count, _type(t), N, _stream(stream)),
           "gq_mul_mat_batched")


def selftest_wait_timeout(limit_us: int = 20000, stream=None) -> None:
    """Launches the bounded-wait self-test (a wait that can only run out)."""
    _check(lib.gq_selftest_wait_timeout(limit_us, _stream(stream)), "gq_selftest_wait_timeout")


def batched_workspace_size(problems, t, N: int) -> int:
    if not isinstance(problems, ctypes.Array):
        problems = make_problems(problems)
    return int(lib.gq_mul_mat_batched_workspace_size(problems, problems._count, _type(t), N))


def mul_mat_batched_ws(problems, t, N: int, workspace: torch.Tensor | None, stream=None) -> None:
    """mul_mat_batched with a caller-owned workspace (uint8 CUDA tensor)."""
    if not isinstance(problems, ctypes.Array):
        problems = make_problems(problems)
    wp = _dev(workspace, torch.uint8, "workspace") if workspace is not None else None
    wn = workspace.numel() if workspace is not None else 0
    _check(lib.gq_mul_mat_batched_ws(problems, problems._count, _type(t), N, wp, wn,
                                     _stream(stream)), "gq_mul_mat_batched_ws")


def mul_mat_q8x(blocks: torch.Tensor, t, M: int, K: int, X: torch.Tensor,
                out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Y (N, M) with X quantized per 32-block like Q8_0 and integer block sums."""
    if X.dim() == 1:
        X = X.view(1, -1)
    N = X.shape[0]
    if X.shape[1] != K:
        raise ValueError("X must be (N, K)")
    if out is None:
        out = _out_like(X, (N, M))
    _check(lib.gq_mul_mat_q8x(_dev(blocks, torch.uint8, "W_blocks"), _type(t), M, K,
                              _act(X, torch.float32, "X"), N, _act(out, torch.float32, "Y"),
                              _stream(stream)), "gq_mul_mat_q8x")
    return out


def mul_mat_rmsnorm(blocks: torch.Tensor, t, M: int, K: int, X: torch.Tensor,
                    gamma: torch.Tensor, eps: float, out: torch.Tensor | None = None,
                    stream=None) -> torch.Tensor:
    """Y (N, M) = RMSNorm(X) . What^T, RMSNorm(x) = x / sqrt(mean(x^2) + eps) * gamma."""
    if X.dim() == 1:
        X = X.view(1, -1)
    N = X.shape[0]
    if X.shape[1] != K or gamma.numel() != K:
        raise ValueError("X must be (N, K) and gamma (K,)")
    if out is None:
        out = _out_like(X, (N, M))
    _check(lib.gq_mul_mat_rmsnorm(_dev(blocks, torch.uint8, "W_blocks"), _type(t), M, K,
                                  _act(X, torch.float32, "X"), _act(gamma, torch.float32, "gamma"),
                                  float(eps), N, _act(out, torch.float32, "Y"), _stream(stream)),
           "gq_mul_mat_rmsnorm")
    return out


def mul_mat_swiglu(gate: torch.Tensor, up: torch.Tensor, t, M: int, K: int, X: torch.Tensor,
                   out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """H (N, M) = Swish(X . Wgate_hat^T) * (X . Wup_hat^T), Swish(z) = z / (1 + e^-z)."""
    if X.dim() == 1:
        X = X.view(1, -1)
    N = X.shape[0]
    if X.shape[1] != K:
        raise ValueError("X must be (N, K)")
    if out is None:
        out = _out_like(X, (N, M))
    _check(lib.gq_mul_mat_swiglu(_dev(gate, torch.uint8, "W_gate"), _dev(up, torch.uint8, "W_up"),
                                 _type(t), M, K, _act(X, torch.float32, "X"), N,
                                 _act(out, torch.float32, "H"), _stream(stream)),
           "gq_mul_mat_swiglu")
    return out


def mul_mat_q8x_batched(problems, t, N: int, stream=None) -> None:
    if not isinstance(problems, ctypes.Array):
        problems = make_problems(problems)
    _check(lib.gq_mul_mat_q8x_batched(problems, problems._count, _type(t), N, _stream(stream)),
           "gq_mul_mat_q8x_batched")


def get_last_error(stream=None) -> int:
    """Synchronizes the stream; returns the device-side status (0, or -6 for a timeout)."""
    return int(lib.gq_get_last_error(_stream(stream)))
