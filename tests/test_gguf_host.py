"""The GGUF reader of include/gq_gguf.h on the host (no GPU): files written by
tests/gguf_writer.py, with known contents, read back through the C ABI; malformed and
truncated files refused with GQ_ERR_FORMAT; missing files with GQ_ERR_IO."""
import ctypes
import struct

import numpy as np
import pytest

import gguf_writer as gw

Q4_0, Q8_0, Q4_K, F32, F16 = 2, 8, 12, 0, 1


def _blocks(rng, n):
    return rng.integers(0, 256, n, dtype=np.uint8).tobytes()


def _sample_file(tmp_path, alignment=64, version=3):
    rng = np.random.default_rng(1)
    kv = [("general.architecture", gw.STRING, "llama"),
          ("general.name", gw.STRING, "synthetic tiny"),
          ("llama.block_count", gw.UINT32, 22),
          ("llama.rope.freq_base", gw.FLOAT32, 10000.0),
          ("u8", gw.UINT8, 250), ("i8", gw.INT8, -5), ("u16", gw.UINT16, 65000),
          ("i16", gw.INT16, -30000), ("i32", gw.INT32, -2_000_000_000),
          ("u64", gw.UINT64, 2 ** 40 + 3), ("i64", gw.INT64, -(2 ** 50)),
          ("f64", gw.FLOAT64, -1.5e-300), ("flag", gw.BOOL, True),
          ("empty", gw.STRING, ""),
          ("ints", gw.ARRAY, (gw.INT32, [1, -2, 3, 2 ** 31 - 1])),
          ("floats", gw.ARRAY, (gw.FLOAT32, [0.5, -0.25])),
          ("tokens", gw.ARRAY, (gw.STRING, ["<s>", "", "hello"])),
          ("nested", gw.ARRAY, (gw.ARRAY, [(gw.UINT8, [1, 2]), (gw.STRING, ["x"])])),
          ("no_items", gw.ARRAY, (gw.UINT64, []))]
    tensors = [("blk.0.attn_q.weight", [64, 5], Q4_0, _blocks(rng, 5 * 2 * 18)),
               ("blk.0.ffn_up.weight", [96, 3], Q8_0, _blocks(rng, 3 * 3 * 34)),
               ("output.weight", [512, 4], Q4_K, _blocks(rng, 4 * 2 * 144)),
               ("output_norm.weight", [7], F32, np.arange(7, dtype="<f4").tobytes()),
               ("rope_freqs", [4, 2], F16, _blocks(rng, 16)),
               ("stack", [64, 2, 3], Q4_0, _blocks(rng, 6 * 2 * 18)),
               ("mystery", [3], 99, b"abc")]
    data, placed = gw.build(kv, tensors, version=version, alignment=alignment)
    path = tmp_path / "model.gguf"
    path.write_bytes(data)
    return path, kv, tensors, placed, data


def test_reads_back_every_field(gq_lib, tmp_path):
    from block_quantized_matmul_gq_gb300.gguf import GGUFFile
    path, kv, tensors, placed, data = _sample_file(tmp_path)
    with GGUFFile(path) as f:
        assert f.version == 3 and f.alignment == 64
        assert f.keys() == [k for k, _, _ in kv] + ["general.alignment"]
        v = {k: f.value(k) for k in f.keys()}
        assert v["general.architecture"] == "llama" and v["general.name"] == "synthetic tiny"
        assert v["llama.block_count"] == 22 and v["llama.rope.freq_base"] == 10000.0
        assert (v["u8"], v["i8"], v["u16"], v["i16"], v["i32"]) == (250, -5, 65000, -30000,
                                                                   -2_000_000_000)
        assert v["u64"] == 2 ** 40 + 3 and v["i64"] == -(2 ** 50) and v["f64"] == -1.5e-300
        assert v["flag"] is True and v["empty"] == ""
        assert v["ints"].tolist() == [1, -2, 3, 2 ** 31 - 1]
        assert v["floats"].tolist() == [0.5, -0.25]
        assert v["tokens"] == ["<s>", "", "hello"]
        assert v["nested"][0].tolist() == [1, 2] and v["nested"][1] == ["x"]
        assert v["no_items"].size == 0 and v["general.alignment"] == 64
        infos = f.tensors()
        assert [t.name for t in infos] == [t[0] for t in tensors]
        for t, (name, ne, gt, raw), (off, n) in zip(infos, tensors, placed):
            assert t.type == gt and t.shape == tuple(ne) and t.offset == off
            assert t.offset % 64 == 0
            if gt == 99:
                assert t.nbytes == 0          # a type this library cannot size
            else:
                assert t.nbytes == n == len(raw)
                assert f.host_bytes(name).tobytes() == raw
        assert f.matrix("blk.0.attn_q.weight") == ("q4_0", 5, 64)
        assert f.matrix("blk.0.ffn_up.weight") == ("q8_0", 3, 96)
        assert f.matrix("output.weight") == ("q4_k", 4, 512)
        assert f.find("missing") == -1
        with pytest.raises(gq_lib.GQError) as e:
            f.matrix("output_norm.weight")               # F32 is not a block type
        assert e.value.status == -3
        with pytest.raises(gq_lib.GQError) as e:
            f.matrix("stack")                             # three non-unit dimensions
        assert e.value.status == -2


def test_version_2_and_default_alignment(gq_lib, tmp_path):
    from block_quantized_matmul_gq_gb300.gguf import GGUFFile
    path, _, tensors, placed, _ = _sample_file(tmp_path, alignment=None, version=2)
    with GGUFFile(path) as f:
        assert f.version == 2 and f.alignment == 32
        assert [t.offset for t in f.tensors()] == [o for o, _ in placed]
        assert all(t.offset % 32 == 0 for t in f.tensors())


def test_empty_file_of_metadata_only(gq_lib, tmp_path):
    from block_quantized_matmul_gq_gb300.gguf import GGUFFile
    p = tmp_path / "meta.gguf"
    p.write_bytes(gw.header(3, 0, 1) + gw.kv_entry("k", gw.UINT32, 7))
    with GGUFFile(p) as f:
        assert f.tensors() == [] and f.value("k") == 7


def _open_status(gq_lib, path):
    h = ctypes.c_void_p()
    st = gq_lib.lib.gq_gguf_open(str(path).encode(), ctypes.byref(h))
    if st == 0:
        gq_lib.lib.gq_gguf_close(h)
    else:
        assert not h.value                              # nothing handed out on failure
    return st


def test_every_truncation_is_refused(gq_lib, tmp_path):
    """Every prefix that ends before the last byte of sized tensor data, or before the
    offset of the last tensor (a type of unknown size), is refused; the file cut right at
    that offset is whole enough to open."""
    _, _, tensors, placed, data = _sample_file(tmp_path)
    assert tensors[-1][2] == 99
    end = placed[-1][0]
    assert end >= max(off + n for off, n in placed[:-1])
    p = tmp_path / "cut.gguf"
    for n in list(range(0, min(end, 1500))) + [end - 100, end - 1]:
        p.write_bytes(data[:n])
        assert _open_status(gq_lib, p) == -7, n
    p.write_bytes(data[:end])
    assert _open_status(gq_lib, p) == 0


def _minimal(version=3, ne=(32, 1), gt=Q4_0, rel=0, n_dims=None, alignment=None, kv=()):
    t = gw.tensor_info("w", ne, gt, rel)
    if n_dims is not None:   # overwrite the n_dims field after the name
        t = t[:8 + 1] + struct.pack("<I", n_dims) + t[8 + 1 + 4:]
    kv = list(kv) + ([("general.alignment", gw.UINT32, alignment)] if alignment is not None
                     else [])
    head = gw.header(version, 1, len(kv)) + b"".join(gw.kv_entry(*e) for e in kv) + t
    a = alignment or 32
    pad = (-len(head)) % a
    return head + b"\0" * pad + b"\x11" * (rel + 18 * ((ne[0] // 32) if ne[0] % 32 == 0 else 1))


@pytest.mark.parametrize("what,blob", [
    ("magic", b"GGUG" + _minimal()[4:]),
    ("version 1", _minimal(version=1)),
    ("version 4", _minimal(version=4)),
    ("big-endian version", _minimal()[:4] + struct.pack(">I", 3) + _minimal()[8:]),
    ("n_dims 0", _minimal(n_dims=0)),
    ("n_dims 5", _minimal(n_dims=5)),
    ("Q4_0 row of 48", _minimal(ne=(48, 1))),
    ("extent >= 2^63", _minimal(ne=(32, 2 ** 63))),
    ("offset not aligned", _minimal(rel=16)),
    ("data past the end", _minimal(ne=(32 * 64, 1))[:-100]),
    ("alignment 0", _minimal(alignment=0)),
    ("alignment 48", _minimal(alignment=48)),
    ("alignment as uint64", _minimal(kv=[("general.alignment", gw.UINT64, 64)])),
    ("unknown value type", gw.header(3, 0, 1) + gw.gstr("k") + struct.pack("<I", 13) +
        b"\0" * 16),
    ("string length past the end", gw.header(3, 0, 1) + gw.gstr("k") +
        struct.pack("<IQ", gw.STRING, 2 ** 62) + b"xy"),
    ("array count past the end", gw.header(3, 0, 1) + gw.gstr("k") +
        struct.pack("<IIQ", gw.ARRAY, gw.UINT32, 2 ** 61) + b"\0" * 16),
    ("string array count past the end", gw.header(3, 0, 1) + gw.gstr("k") +
        struct.pack("<IIQ", gw.ARRAY, gw.STRING, 2 ** 40) + gw.gstr("a")),
    ("arrays nested 9 deep", gw.header(3, 0, 1) + gw.gstr("k") + struct.pack("<I", gw.ARRAY) +
        struct.pack("<IQ", gw.ARRAY, 1) * 8 + struct.pack("<IQ", gw.UINT8, 1) + b"\1"),
    ("kv count too large", gw.header(3, 0, 2 ** 60) + b"\0" * 64),
    ("tensor count too large", gw.header(3, 2 ** 60, 0) + b"\0" * 64),
])
def test_malformed_files_are_refused(gq_lib, tmp_path, what, blob):
    p = tmp_path / "bad.gguf"
    p.write_bytes(blob)
    assert _open_status(gq_lib, p) == -7, what


def test_the_minimal_file_itself_is_valid(gq_lib, tmp_path):
    p = tmp_path / "ok.gguf"
    p.write_bytes(_minimal())
    assert _open_status(gq_lib, p) == 0
    p.write_bytes(_minimal(alignment=64, kv=[("a", gw.STRING, "b")]))
    assert _open_status(gq_lib, p) == 0
    nested8 = (gw.header(3, 0, 1) + gw.gstr("k") + struct.pack("<I", gw.ARRAY) +
               struct.pack("<IQ", gw.ARRAY, 1) * 7 + struct.pack("<IQ", gw.UINT8, 1) + b"\1")
    p.write_bytes(nested8)
    assert _open_status(gq_lib, p) == 0


def test_io_errors_and_null_arguments(gq_lib, tmp_path):
    lib = gq_lib.lib
    assert _open_status(gq_lib, tmp_path / "does_not_exist.gguf") == -8
    assert _open_status(gq_lib, tmp_path) == -8                  # a directory
    h = ctypes.c_void_p()
    assert lib.gq_gguf_open(None, ctypes.byref(h)) == -1
    assert lib.gq_gguf_tensor_count(None) == 0 and lib.gq_gguf_kv_key(None, 0) is None
    assert lib.gq_gguf_find_tensor(None, b"x") == -1
    t = gq_lib.GgufTensor()
    assert lib.gq_gguf_tensor_info(None, 0, ctypes.byref(t)) == -1
    lib.gq_gguf_close(None)


def test_query_errors(gq_lib, tmp_path):
    path, *_ = _sample_file(tmp_path)
    lib = gq_lib.lib
    h = ctypes.c_void_p()
    assert lib.gq_gguf_open(str(path).encode(), ctypes.byref(h)) == 0
    try:
        t = gq_lib.GgufTensor()
        assert lib.gq_gguf_tensor_info(h, 99, ctypes.byref(t)) == -2
        assert lib.gq_gguf_tensor_data(h, -1) is None
        i = lib.gq_gguf_find_key(h, b"general.name")
        v = ctypes.c_int64()
        assert lib.gq_gguf_kv_int(h, i, ctypes.byref(v)) == -3        # a string
        d = ctypes.c_double()
        assert lib.gq_gguf_kv_float(h, lib.gq_gguf_find_key(h, b"u8"), ctypes.byref(d)) == -3
        assert lib.gq_gguf_kv_type(h, 10 ** 6) == -1
        # a uint64 beyond int64 does not fit the int64 accessor
        big = tmp_path / "big.gguf"
        big.write_bytes(gw.header(3, 0, 1) + gw.kv_entry("big", gw.UINT64, 2 ** 64 - 1))
        h2 = ctypes.c_void_p()
        assert lib.gq_gguf_open(str(big).encode(), ctypes.byref(h2)) == 0
        assert lib.gq_gguf_kv_int(h2, 0, ctypes.byref(v)) == -2
        lib.gq_gguf_close(h2)
        # upload refuses a type of unknown size and a too-small or misaligned destination
        # before any CUDA call
        A16 = 0x7000_0000_0000
        assert lib.gq_gguf_upload(h, lib.gq_gguf_find_tensor(h, b"mystery"), A16, 1 << 20,
                                  None) == -2
        q = lib.gq_gguf_find_tensor(h, b"blk.0.attn_q.weight")
        assert lib.gq_gguf_upload(h, q, A16, 5 * 2 * 18 - 1, None) == -2
        assert lib.gq_gguf_upload(h, q, A16 + 4, 1 << 20, None) == -4
        assert lib.gq_gguf_upload(h, q, None, 1 << 20, None) == -1
    finally:
        lib.gq_gguf_close(h)
