"""GGUF files through libgq's reader (include/gq_gguf.h): argument marshalling only.

The file is memory-mapped and parsed by the library; this module turns its answers into
Python values and copies tensors to the device with gq_gguf_upload. A Q4_0 / Q8_0 / Q4_K
weight matrix arrives as an (M, row_bytes) uint8 CUDA tensor that binding.mul_mat takes
as it is.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import numpy as np
import torch

from . import binding

# GGUF metadata value types (gq_gguf.h)
UINT8, INT8, UINT16, INT16, UINT32, INT32, FLOAT32, BOOL, STRING, ARRAY, UINT64, INT64, \
    FLOAT64 = range(13)
_NUMPY = {UINT8: "<u1", INT8: "<i1", UINT16: "<u2", INT16: "<i2", UINT32: "<u4", INT32: "<i4",
          FLOAT32: "<f4", BOOL: "<u1", UINT64: "<u8", INT64: "<i8", FLOAT64: "<f8"}
_BLOCK_TYPES = {binding.Q4_0: "q4_0", binding.Q8_0: "q8_0", binding.Q4_K: "q4_k"}


@dataclass(frozen=True)
class TensorInfo:
    index: int
    name: str
    type: int              # ggml type id
    shape: tuple           # (ne[0], ..., ne[n_dims - 1]); ne[0] is contiguous
    offset: int            # from the start of the file
    nbytes: int            # 0 for a type of unknown size


class GGUFFile:
    """An open GGUF file. Use as a context manager, or call close()."""

    def __init__(self, path: str):
        h = ctypes.c_void_p()
        binding._check(binding.lib.gq_gguf_open(str(path).encode(), ctypes.byref(h)),
                       f"gq_gguf_open({path})")
        self._h = h

    def close(self) -> None:
        if getattr(self, "_h", None):
            binding.lib.gq_gguf_close(self._h)
            self._h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        self.close()

    @property
    def version(self) -> int:
        return int(binding.lib.gq_gguf_version(self._h))

    @property
    def alignment(self) -> int:
        return int(binding.lib.gq_gguf_alignment(self._h))

    # ---- tensors ------------------------------------------------------------------
    def tensor(self, i: int) -> TensorInfo:
        t = binding.GgufTensor()
        binding._check(binding.lib.gq_gguf_tensor_info(self._h, i, ctypes.byref(t)),
                       "gq_gguf_tensor_info")
        return TensorInfo(i, t.name.decode(), int(t.type), tuple(t.ne[:t.n_dims]),
                          int(t.offset), int(t.nbytes))

    def tensors(self) -> list:
        return [self.tensor(i) for i in range(binding.lib.gq_gguf_tensor_count(self._h))]

    def find(self, name: str) -> int:
        return int(binding.lib.gq_gguf_find_tensor(self._h, name.encode()))

    def _index(self, name_or_index) -> int:
        i = self.find(name_or_index) if isinstance(name_or_index, str) else int(name_or_index)
        if i < 0:
            raise KeyError(name_or_index)
        return i

    def host_bytes(self, name_or_index) -> np.ndarray:
        """The tensor's bytes inside the mapping, as a read-only uint8 array (a copy)."""
        i = self._index(name_or_index)
        info = self.tensor(i)
        ptr = binding.lib.gq_gguf_tensor_data(self._h, i)
        return np.ctypeslib.as_array(ctypes.cast(ptr, ctypes.POINTER(ctypes.c_uint8)),
                                     shape=(info.nbytes,)).copy()

    def matrix(self, name_or_index):
        """(block type name, M, K) of a 2-D Q4_0 / Q8_0 / Q4_K tensor."""
        i = self._index(name_or_index)
        t, M, K = ctypes.c_int(), ctypes.c_int64(), ctypes.c_int64()
        binding._check(binding.lib.gq_gguf_tensor_matrix(self._h, i, ctypes.byref(t),
                                                         ctypes.byref(M), ctypes.byref(K)),
                       "gq_gguf_tensor_matrix")
        return _BLOCK_TYPES[t.value], int(M.value), int(K.value)

    def upload(self, name_or_index, device, stream=None) -> torch.Tensor:
        """Copies the tensor to `device`: an (M, row_bytes) uint8 tensor for a block-type
        matrix (W_blocks of binding.mul_mat), else a flat uint8 tensor of its bytes."""
        i = self._index(name_or_index)
        info = self.tensor(i)
        try:
            btype, M, K = self.matrix(i)
            out = torch.empty((M, binding.row_bytes(btype, K)), dtype=torch.uint8, device=device)
        except binding.GQError:
            out = torch.empty((info.nbytes,), dtype=torch.uint8, device=device)
        binding._check(binding.lib.gq_gguf_upload(self._h, i, out.data_ptr(), out.numel(),
                                                  binding._stream(stream)),
                       "gq_gguf_upload")
        return out

    # ---- metadata -----------------------------------------------------------------
    def keys(self) -> list:
        return [binding.lib.gq_gguf_kv_key(self._h, i).decode()
                for i in range(binding.lib.gq_gguf_kv_count(self._h))]

    def value_type(self, key: str) -> int:
        return int(binding.lib.gq_gguf_kv_type(self._h, self._key(key)))

    def _key(self, key: str) -> int:
        i = int(binding.lib.gq_gguf_find_key(self._h, key.encode()))
        if i < 0:
            raise KeyError(key)
        return i

    def value(self, key: str):
        """A metadata value: int, bool, float, str, or for an array a numpy array (numeric
        elements) or a list (string and array elements)."""
        i = self._key(key)
        t = binding.lib.gq_gguf_kv_type(self._h, i)
        L = binding.lib
        if t in (FLOAT32, FLOAT64):
            v = ctypes.c_double()
            binding._check(L.gq_gguf_kv_float(self._h, i, ctypes.byref(v)), key)
            return v.value
        if t == STRING:
            p, n = ctypes.c_void_p(), ctypes.c_uint64()
            binding._check(L.gq_gguf_kv_string(self._h, i, ctypes.byref(p), ctypes.byref(n)), key)
            return ctypes.string_at(p.value, n.value).decode("utf-8", "replace") if n.value else ""
        if t == ARRAY:
            et, n, p = ctypes.c_uint32(), ctypes.c_uint64(), ctypes.c_void_p()
            binding._check(L.gq_gguf_kv_array(self._h, i, ctypes.byref(et), ctypes.byref(n),
                                              ctypes.byref(p)), key)
            return _array(et.value, n.value, p.value)
        v = ctypes.c_int64()
        binding._check(L.gq_gguf_kv_int(self._h, i, ctypes.byref(v)), key)
        return bool(v.value) if t == BOOL else int(v.value)


def _array(et: int, n: int, addr: int):
    """Decodes n array elements of type et starting at host address addr (inside the
    mapping, already bounds-checked by the library's parser)."""
    if et in _NUMPY:
        dt = np.dtype(_NUMPY[et])
        raw = ctypes.string_at(addr, n * dt.itemsize) if n else b""
        a = np.frombuffer(raw, dtype=dt).copy()
        return a.astype(bool) if et == BOOL else a
    out, pos = [], addr
    for _ in range(n):
        if et == STRING:
            ln = int.from_bytes(ctypes.string_at(pos, 8), "little")
            out.append(ctypes.string_at(pos + 8, ln).decode("utf-8", "replace") if ln else "")
            pos += 8 + ln
        else:   # nested array: element type, count, elements
            sub_t = int.from_bytes(ctypes.string_at(pos, 4), "little")
            sub_n = int.from_bytes(ctypes.string_at(pos + 4, 8), "little")
            out.append(_array(sub_t, sub_n, pos + 12))
            pos += 12 + _encoded_size(sub_t, sub_n, pos + 12)
    return out


def _encoded_size(et: int, n: int, addr: int) -> int:
    if et in _NUMPY:
        return n * np.dtype(_NUMPY[et]).itemsize
    size, pos = 0, addr
    for _ in range(n):
        if et == STRING:
            ln = int.from_bytes(ctypes.string_at(pos, 8), "little")
            size += 8 + ln
            pos += 8 + ln
        else:
            sub_t = int.from_bytes(ctypes.string_at(pos, 4), "little")
            sub_n = int.from_bytes(ctypes.string_at(pos + 4, 8), "little")
            inner = 12 + _encoded_size(sub_t, sub_n, pos + 12)
            size += inner
            pos += inner
    return size
