"""GGUF reader (host only): the page's type-10 fixture, a richer file with every
metadata value type and a custom alignment, and malformed files.

The writer below is this test's own, from the container layout: "GGUF",
version u32, tensor count u64, metadata count u64, metadata (key string, type
u32, value), tensor entries (name string, n_dims u32, extents u64 innermost
first, type u32, offset u64 from the data section), zero padding to the
alignment, then the data.  Strings are a u64 length and the bytes.
"""

import os
import struct

import numpy as np
import pytest

import q2k_workloads as wl
import ggml_q2_quantized_gb300 as q2k
from ggml_q2_quantized_gb300 import build as q2k_build


@pytest.fixture(scope="module", autouse=True)
def lib():
    q2k_build.build()
    return q2k.load()


def gstr(s: bytes) -> bytes:
    return struct.pack("<Q", len(s)) + s


def kv(key: str, vtype: int, payload: bytes) -> bytes:
    return gstr(key.encode()) + struct.pack("<I", vtype) + payload


def tensor_entry(name: str, dims, ggml_type: int, offset: int) -> bytes:
    return (gstr(name.encode()) + struct.pack("<I", len(dims)) +
            b"".join(struct.pack("<Q", d) for d in dims) + struct.pack("<IQ", ggml_type, offset))


def gguf_bytes(tensors, kvs=(), version=3, alignment=32, data_pad=True):
    """tensors: (name, dims, type, data bytes); offsets laid out at `alignment`."""
    offsets, off = [], 0
    for _, _, _, data in tensors:
        off = (off + alignment - 1) // alignment * alignment
        offsets.append(off)
        off += len(data)
    head = b"GGUF" + struct.pack("<IQQ", version, len(tensors), len(kvs)) + b"".join(kvs)
    head += b"".join(tensor_entry(n, d, t, o) for (n, d, t, _), o in zip(tensors, offsets))
    head += b"\0" * ((-len(head)) % alignment)
    body = bytearray()
    for (_, _, _, data), o in zip(tensors, offsets):
        body += b"\0" * (o - len(body))
        body += data
    return head + bytes(body)


def write(tmp_path, name, data: bytes) -> str:
    p = tmp_path / name
    p.write_bytes(data)
    return str(p)


def test_page_type_10_fixture(tmp_path):
    """Page test q2_k_gguf_type_10_parses_with_exact_block_size: one tensor
    "q2.weight" of 256 elements, type 10, no metadata, data block(3) at 32."""
    block = wl.page_block(3).tobytes()
    data = gguf_bytes([("q2.weight", [256], 10, block)])
    assert len(data) == 96 + 84     # header of 65 bytes padded to 96
    with q2k.GgufFile(write(tmp_path, "page.gguf", data)) as g:
        assert g.names == ["q2.weight"]
        info = g.info("q2.weight")
        assert info.ggml_type == 10
        assert info.byte_len == 84
        assert info.n_dims == 1 and info.dims[0] == 256 and info.n_elements == 256
        assert info.offset == 96
        assert g.read("q2.weight").tobytes() == block


def test_metadata_of_every_type_and_custom_alignment(tmp_path):
    rng = np.random.default_rng(3)
    q2 = wl.random_blocks(rng, 3 * 2).tobytes()              # [k = 512, n = 3]
    f32 = rng.standard_normal(7).astype("<f4").tobytes()
    f16 = rng.standard_normal(10).astype("<f2").tobytes()
    kvs = [
        kv("general.architecture", 8, gstr(b"llama")),
        kv("a.u8", 0, b"\x07"), kv("a.i8", 1, b"\xf9"), kv("a.u16", 2, struct.pack("<H", 7)),
        kv("a.i16", 3, struct.pack("<h", -7)), kv("a.u32", 4, struct.pack("<I", 7)),
        kv("a.i32", 5, struct.pack("<i", -7)), kv("a.f32", 6, struct.pack("<f", 0.5)),
        kv("a.bool", 7, b"\x01"), kv("a.u64", 10, struct.pack("<Q", 7)),
        kv("a.i64", 11, struct.pack("<q", -7)), kv("a.f64", 12, struct.pack("<d", 0.25)),
        kv("a.arr_u32", 9, struct.pack("<IQ", 4, 3) + struct.pack("<3I", 1, 2, 3)),
        kv("a.arr_str", 9, struct.pack("<IQ", 8, 2) + gstr(b"x") + gstr(b"yz")),
        kv("general.alignment", 4, struct.pack("<I", 64)),
    ]
    tensors = [("blk.0.ffn_up.weight", [512, 3], 10, q2), ("norm", [7], 0, f32),
               ("emb", [5, 2], 1, f16)]
    data = gguf_bytes(tensors, kvs, alignment=64)
    with q2k.GgufFile(write(tmp_path, "rich.gguf", data)) as g:
        assert g.names == [t[0] for t in tensors]
        base = None
        for name, dims, t, payload in tensors:
            info = g.info(name)
            assert info.ggml_type == t and info.n_dims == len(dims)
            assert list(info.dims[:len(dims)]) == dims and all(d == 1 for d in info.dims[len(dims):])
            assert info.n_elements == int(np.prod(dims))
            assert info.byte_len == len(payload)
            assert info.offset % 64 == 0
            base = info.offset if base is None else base
            assert g.read(name).tobytes() == payload
        assert g.info("blk.0.ffn_up.weight").byte_len == 3 * 2 * 84


def test_version_2_and_unknown_type(tmp_path):
    data = gguf_bytes([("w", [256, 2], 10, wl.page_block(1).tobytes() * 2),
                       ("odd", [4], 99, b"\0" * 16)], version=2)
    with q2k.GgufFile(write(tmp_path, "v2.gguf", data)) as g:
        assert g.info("w").byte_len == 168
        assert g.info("odd").ggml_type == 99 and g.info("odd").byte_len == 0
        with pytest.raises(q2k.InvalidArgument, match="does not know"):
            g.read("odd")
        with pytest.raises(q2k.InvalidArgument, match="no tensor"):
            g.info("missing")


def _malformed_cases():
    block = wl.page_block(3).tobytes()
    good = gguf_bytes([("q2.weight", [256], 10, block)])
    yield "magic", b"GGUF"[::-1] + good[4:], "magic"
    yield "version1", good[:4] + struct.pack("<I", 1) + good[8:], "version"
    yield "truncated_header", good[:40], "truncated"
    yield "data_past_eof", good[:-1], "past the end"
    yield "five_dims", gguf_bytes([("t", [256, 1, 1, 1, 1], 10, block)]), "dimensions"
    yield "not_whole_blocks", gguf_bytes([("t", [300], 10, b"\0" * 84)]), "multiple of 256"
    yield "duplicate", gguf_bytes([("t", [256], 10, block), ("t", [256], 10, block)]), "twice"
    yield "zero_extent", gguf_bytes([("t", [0], 0, b"")]), "extent"
    yield ("bad_alignment", gguf_bytes([("t", [256], 10, block)],
                                       [kv("general.alignment", 4, struct.pack("<I", 48))]),
           "power of two")
    yield ("alignment_type", gguf_bytes([("t", [256], 10, block)],
                                        [kv("general.alignment", 10, struct.pack("<Q", 32))]),
           "u32")
    yield ("unknown_kv_type", gguf_bytes([("t", [256], 10, block)], [kv("x", 13, b"")]),
           "unknown value type")
    yield ("nested_array", gguf_bytes([("t", [256], 10, block)],
                                      [kv("x", 9, struct.pack("<IQ", 9, 1) + struct.pack("<IQ", 4, 0))]),
           "array")
    # an offset off the 32-byte alignment
    head = b"GGUF" + struct.pack("<IQQ", 3, 1, 0) + tensor_entry("t", [256], 10, 4)
    head += b"\0" * ((-len(head)) % 32)
    yield "offset_unaligned", head + b"\0" * 4 + block, "alignment"
    yield "huge_count", b"GGUF" + struct.pack("<IQQ", 3, 1 << 40, 0), "count"


@pytest.mark.parametrize("name,data,fragment", list(_malformed_cases()),
                         ids=[c[0] for c in _malformed_cases()])
def test_malformed_files_are_rejected(tmp_path, name, data, fragment):
    with pytest.raises(q2k.InvalidArgument) as e:
        q2k.GgufFile(write(tmp_path, name + ".gguf", data))
    assert fragment in str(e.value)


def test_missing_file_is_an_io_error(tmp_path):
    with pytest.raises(q2k.Q2KError) as e:
        q2k.GgufFile(str(tmp_path / "absent.gguf"))
    assert e.value.status == 6


def test_read_needs_exact_destination(lib, tmp_path):
    import ctypes
    data = gguf_bytes([("q2.weight", [256], 10, wl.page_block(3).tobytes())])
    with q2k.GgufFile(write(tmp_path, "page.gguf", data)) as g:
        buf = (ctypes.c_uint8 * 100)()
        assert lib.q2k_gguf_read_tensor(g._h, b"q2.weight", buf, 83) == 1
        assert "84 bytes" in lib.q2k_last_error().decode()


@pytest.mark.gpu
def test_gguf_weights_into_matmul(tmp_path):
    """A Q2_K matrix stored in a GGUF file, loaded to the device, multiplied."""
    torch = pytest.importorskip("torch")
    import oracle
    n, k = 96, 1024
    x, w = wl.make_matmul_inputs(41, 2, n, k)
    data = gguf_bytes([("blk.0.attn_q.weight", [k, n], 10, w.tobytes())])
    with q2k.GgufFile(write(tmp_path, "w.gguf", data)) as g:
        info = g.info("blk.0.attn_q.weight")
        assert (info.dims[0], info.dims[1]) == (k, n)
        wd = g.to_device("blk.0.attn_q.weight")
    y = q2k.matmul(torch.from_numpy(x).cuda(), wd, n, path="gemv")
    torch.cuda.synchronize()
    yref, s = oracle.matmul(x, w, n)
    assert (np.abs(y.cpu().numpy().astype(np.float64) - yref) <= 1e-5 * s).all()
