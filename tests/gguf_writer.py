"""A small GGUF writer for the tests: builds files in the published GGUF layout (the
structure "Development Guide for Small AI Models (TinyLLaMA, etc.) Using C++", section 3.2
lists; field widths from the GGUF specification) so that the library's reader can be
checked on files with known contents. Test infrastructure only; it shares nothing with the
reader in libgq.
"""
from __future__ import annotations

import struct

MAGIC = b"GGUF"
UINT8, INT8, UINT16, INT16, UINT32, INT32, FLOAT32, BOOL, STRING, ARRAY, UINT64, INT64, \
    FLOAT64 = range(13)
_FMT = {UINT8: "<B", INT8: "<b", UINT16: "<H", INT16: "<h", UINT32: "<I", INT32: "<i",
        FLOAT32: "<f", BOOL: "<?", UINT64: "<Q", INT64: "<q", FLOAT64: "<d"}


def gstr(s) -> bytes:
    b = s.encode() if isinstance(s, str) else bytes(s)
    return struct.pack("<Q", len(b)) + b


def value(t: int, v) -> bytes:
    """Encoding of one value of type t. An array value is (element type, list)."""
    if t in _FMT:
        return struct.pack(_FMT[t], v)
    if t == STRING:
        return gstr(v)
    if t == ARRAY:
        et, items = v
        return struct.pack("<IQ", et, len(items)) + b"".join(value(et, x) for x in items)
    raise ValueError(t)


def header(version: int, n_tensors: int, n_kv: int) -> bytes:
    return MAGIC + struct.pack("<IQQ", version, n_tensors, n_kv)


def kv_entry(key: str, t: int, v) -> bytes:
    return gstr(key) + struct.pack("<I", t) + value(t, v)


def tensor_info(name: str, ne, ggml_type: int, rel_offset: int) -> bytes:
    return (gstr(name) + struct.pack("<I", len(ne)) + b"".join(struct.pack("<Q", e) for e in ne)
            + struct.pack("<IQ", ggml_type, rel_offset))


def build(kv, tensors, version: int = 3, alignment: int | None = None) -> tuple[bytes, list]:
    """kv: [(key, type, value)], tensors: [(name, ne, ggml_type, data bytes)].
    Returns (file bytes, [(data offset in the file, nbytes)] per tensor). With `alignment`,
    a uint32 general.alignment entry is appended to kv; tensor data are padded to it."""
    a = 32 if alignment is None else alignment
    kv = list(kv) + ([("general.alignment", UINT32, alignment)] if alignment is not None else [])
    rel, offs = 0, []
    infos = b""
    for name, ne, gt, data in tensors:
        infos += tensor_info(name, ne, gt, rel)
        offs.append(rel)
        rel += (len(data) + a - 1) // a * a
    head = header(version, len(tensors), len(kv)) + b"".join(kv_entry(*e) for e in kv) + infos
    data_start = (len(head) + a - 1) // a * a
    out = bytearray(head + b"\0" * (data_start - len(head)))
    placed = []
    for (name, ne, gt, data), r in zip(tensors, offs):
        assert len(out) == data_start + r
        out += data + b"\0" * ((len(data) + a - 1) // a * a - len(data))
        placed.append((data_start + r, len(data)))
    return bytes(out), placed
