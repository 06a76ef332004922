"""kq_gguf_index: the GGUF container reader.

A checkpoint built by tests/golden/make_gguf.py from the public container
description (every metadata value type, nested arrays, a non-default
alignment, K-quant and F32 tensors, a 3-D tensor) is indexed: names, types,
dims, the kq_format of each K-quant type, data offsets on the alignment and
the exact byte ranges of the oracle-quantised blocks.  Malformed files --
every truncation, a wrong magic, an unknown version, an unaligned offset, a
row length off the 256 grid, an absurd tensor count, deep nesting -- return
an error without reading outside the buffer.  On the GPU the indexed bytes go
straight into kq_gemv and match the oracle.

Parity unpinned: agreement of the record bit placement with real GGUF
checkpoint files (none are available here); the container itself is pinned
by the description.
"""
import os
import struct
import sys

import numpy as np
import pytest

import workloads as wl

sys.path.insert(0, os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden"))
import make_gguf  # noqa: E402

KQ_OK, KQ_ERR_ARG, KQ_ERR_SHAPE, KQ_ERR_UNSUPPORTED = 0, 1, 2, 7


@pytest.fixture(scope="module")
def kq():
    from quant_weight_gemv_dequant_b300 import build
    build.build()
    import quant_weight_gemv_dequant_b300 as k
    k.lib()
    return k


@pytest.fixture(scope="module")
def gguf(oracle):
    return make_gguf.build(oracle)


def test_index_matches_the_container(kq, gguf):
    data, man = gguf
    st, ts, align = kq.kq_gguf_index(data)
    assert st == KQ_OK and align == make_gguf.ALIGN and len(ts) == len(man)
    for t, m in zip(ts, man):
        assert t.name.decode() == m["name"]
        assert t.ggml_type == m["ggml_type"]
        assert t.n_dims == len(m["dims"])
        assert list(t.dims[:t.n_dims]) == list(m["dims"])
        assert t.data_offset == m["data_offset"] and t.data_offset % make_gguf.ALIGN == 0
        assert t.format == (m["format"] if m["format"] is not None else -1)
        if m["format"] is not None:
            assert t.K == m["dims"][0] and t.N_out == int(np.prod(m["dims"][1:]))
            assert t.bytes == m["bytes"] == kq.kq_matrix_bytes(t.format, t.N_out, t.K)
        else:
            assert t.bytes == 0


def test_indexed_bytes_are_the_oracle_blocks(kq, oracle, gguf):
    data, man = gguf
    _, ts, _ = kq.kq_gguf_index(data)
    for i, t in enumerate(ts):
        ref = make_gguf.tensor_data(oracle, i)
        n = len(ref)
        assert data[t.data_offset:t.data_offset + n] == ref


def test_fewer_entries_than_tensors(kq, gguf):
    data, man = gguf
    st, ts, _ = kq.kq_gguf_index(data, max_tensors=2)
    assert st == KQ_OK and len(ts) == 2 and ts[1].name.decode() == man[1]["name"]


def test_every_truncation_is_an_error(kq, gguf):
    # the index succeeds exactly when the data section starts inside the
    # buffer, every tensor's offset lies inside it and every K-quant tensor's
    # records fit (F32 data are not the index's concern); every other cut
    # returns an error
    data, man = gguf
    start = man[0]["data_offset"]
    end = man[-1]["data_offset"] + man[-1]["bytes"]

    def expect_ok(n):
        return n >= start and all(m["data_offset"] <= n and
                                  (m["format"] is None or m["data_offset"] + m["bytes"] <= n) for m in man)

    cuts = set(range(0, start + 1)) | {m["data_offset"] + m["bytes"] + d for m in man for d in (-1, 0)}
    for n in sorted(c for c in cuts if 0 <= c <= end):
        st = kq.kq_gguf_index(data[:n])[0]
        assert (st == KQ_OK) == expect_ok(n), (n, st)
        assert st in (KQ_OK, KQ_ERR_ARG), (n, st)


def _patch(data, off, fmt, value):
    b = bytearray(data)
    struct.pack_into(fmt, b, off, value)
    return bytes(b)


def test_malformed_headers(kq, gguf):
    data, man = gguf
    assert kq.kq_gguf_index(b"GGUX" + data[4:])[0] == KQ_ERR_ARG
    assert kq.kq_gguf_index(_patch(data, 4, "<I", 1))[0] == KQ_ERR_UNSUPPORTED
    assert kq.kq_gguf_index(_patch(data, 8, "<Q", 1 << 40))[0] == KQ_ERR_ARG    # tensor count
    assert kq.kq_gguf_index(_patch(data, 16, "<Q", 1 << 40))[0] == KQ_ERR_ARG   # kv count
    # the first tensor info: its name, then n_dims, dims, type, offset
    pos = data.index(make_gguf.TENSORS[0][0].encode()) + len(make_gguf.TENSORS[0][0])
    nd = make_gguf.TENSORS[0][2]
    off_at = pos + 4 + 8 * len(nd) + 4
    assert kq.kq_gguf_index(_patch(data, off_at, "<Q", 8))[0] == KQ_ERR_ARG      # unaligned offset
    assert kq.kq_gguf_index(_patch(data, pos + 4, "<Q", 500))[0] == KQ_ERR_SHAPE  # row length
    assert kq.kq_gguf_index(_patch(data, pos, "<I", 9))[0] == KQ_ERR_ARG          # n_dims


def test_deep_nesting_is_rejected(kq):
    # an array of arrays nested five deep
    v = struct.pack("<IQ", 4, 1) + struct.pack("<I", 1)   # innermost: one u32
    for _ in range(5):
        v = struct.pack("<IQ", 9, 1) + v
    f = b"GGUF" + struct.pack("<IQQ", 3, 0, 1) + make_gguf._kv("deep", 9, v)
    assert kq.kq_gguf_index(f)[0] == KQ_ERR_ARG


@pytest.mark.gpu
def test_indexed_tensors_run_on_the_gpu(kq, oracle, gguf):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    data, _ = gguf
    _, ts, _ = kq.kq_gguf_index(data)
    for t in ts:
        if t.format < 0:
            continue
        W = np.frombuffer(data, dtype=np.uint8, count=t.bytes, offset=t.data_offset)
        x = wl.activations_bf16(wl.derive_seed(601, t.K), 2, t.K)
        y_ref, A = oracle.gemv(t.format, W, t.N_out, t.K, x)
        y = torch.empty((2, t.N_out), dtype=torch.float32, device="cuda")
        kq.kq_gemv(t.format, torch.from_numpy(W.copy()).cuda(),
                   torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16), y, t.N_out, t.K, 2)
        torch.cuda.synchronize()
        assert np.all(np.abs(y.cpu().numpy() - y_ref) <= 1e-3 * A + 1e-5), t.name
