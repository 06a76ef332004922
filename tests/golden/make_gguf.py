"""Builds a small GGUF checkpoint for the container tests of kq_gguf_index.

The container follows the public GGUF description (version 3,
little-endian): "GGUF", u32 version, u64 tensor count, u64 key/value count;
the key/value pairs (u64-length string key, u32 value type, value); the
tensor infos (string name, u32 n_dims, u64 dims -- dims[0] the row length --,
u32 tensor type, u64 offset from the start of the data section); padding to
the alignment (the key "general.alignment", here 64 instead of the default
32); the data.  Value types: 0 u8, 1 i8, 2 u16, 3 i16, 4 u32, 5 i32, 6 f32,
7 bool, 8 string, 9 array, 10 u64, 11 i64, 12 f64.  Tensor types used: 0
F32, 12 Q4_K, 13 Q5_K, 14 Q6_K.

The K-quant tensors hold blocks from the oracle's quantiser on seeded
weights; nothing here comes from the library under test.
"""
from __future__ import annotations

import struct

import numpy as np

import workloads as wl

ALIGN = 64
# (name, ggml type, dims (row length first), kq format or None)
TENSORS = [
    ("blk.0.attn_q.weight", 12, (512, 40), 0),
    ("blk.0.ffn_down.weight", 14, (768, 24), 2),
    ("blk.0.ffn_up.weight", 13, (256, 3), 1),
    ("token_embd.weight", 0, (64, 4), None),
    ("blk.0.attn_norm.weight", 0, (64,), None),
    ("blk.1.attn_k.weight", 12, (256, 2, 3), 0),   # 3-D: 6 rows of 256
]


def _str(s: str) -> bytes:
    b = s.encode()
    return struct.pack("<Q", len(b)) + b


def _kv(key: str, vtype: int, payload: bytes) -> bytes:
    return _str(key) + struct.pack("<I", vtype) + payload


def metadata() -> list[bytes]:
    strings = [_str(s) for s in ("alpha", "", "gamma")]
    nested = struct.pack("<IQ", 2, 3) + b"".join(struct.pack("<H", v) for v in (1, 2, 3))
    return [
        _kv("general.architecture", 8, _str("test-decoder")),
        _kv("general.alignment", 4, struct.pack("<I", ALIGN)),
        _kv("test.u8", 0, struct.pack("<B", 7)),
        _kv("test.i8", 1, struct.pack("<b", -7)),
        _kv("test.u16", 2, struct.pack("<H", 700)),
        _kv("test.i16", 3, struct.pack("<h", -700)),
        _kv("test.i32", 5, struct.pack("<i", -70000)),
        _kv("test.f32", 6, struct.pack("<f", 1.5)),
        _kv("test.bool", 7, struct.pack("<B", 1)),
        _kv("test.u64", 10, struct.pack("<Q", 1 << 40)),
        _kv("test.i64", 11, struct.pack("<q", -(1 << 40))),
        _kv("test.f64", 12, struct.pack("<d", 2.25)),
        _kv("test.strings", 9, struct.pack("<IQ", 8, 3) + b"".join(strings)),
        _kv("test.nested", 9, struct.pack("<IQ", 9, 2) + nested + nested),
    ]


def tensor_data(oracle, i: int):
    """The bytes of tensor i (K-quant: oracle-quantised seeded weights)."""
    name, gtype, dims, fmt = TENSORS[i]
    K = dims[0]
    N = int(np.prod(dims[1:])) if len(dims) > 1 else 1
    w = wl.weights_f32(wl.derive_seed(600, i), N, K)
    if fmt is None:
        return w.astype("<f4").tobytes()
    return oracle.quantize(fmt, w, N, K).tobytes()


def build(oracle) -> tuple[bytes, list[dict]]:
    """(file bytes, per-tensor manifest with the expected index entries)."""
    kvs = metadata()
    datas = [tensor_data(oracle, i) for i in range(len(TENSORS))]
    infos, manifest, off = [], [], 0
    for (name, gtype, dims, fmt), d in zip(TENSORS, datas):
        infos.append(_str(name) + struct.pack("<I", len(dims)) + b"".join(struct.pack("<Q", x) for x in dims)
                     + struct.pack("<IQ", gtype, off))
        manifest.append({"name": name, "ggml_type": gtype, "dims": dims, "format": fmt, "offset": off,
                         "bytes": len(d)})
        off += (len(d) + ALIGN - 1) // ALIGN * ALIGN
    head = b"GGUF" + struct.pack("<IQQ", 3, len(TENSORS), len(kvs)) + b"".join(kvs) + b"".join(infos)
    data_start = (len(head) + ALIGN - 1) // ALIGN * ALIGN
    body = bytearray(head + b"\0" * (data_start - len(head)))
    for m, d in zip(manifest, datas):
        pad = data_start + m["offset"] - len(body)
        body += b"\0" * pad + d
        m["data_offset"] = data_start + m["offset"]
    return bytes(body), manifest


if __name__ == "__main__":
    import sys
    import os
    sys.path.insert(0, os.path.join(os.path.dirname(os.path.abspath(__file__)), "..", ".."))
    import oracle
    data, man = build(oracle)
    out = sys.argv[1] if len(sys.argv) > 1 else "test.gguf"
    with open(out, "wb") as fh:
        fh.write(data)
    print(out, len(data), "bytes")
