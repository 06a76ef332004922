"""C-ABI checks that need no GPU: the library loads, exports every function
include/kq.h declares, its host-side quantiser and merge agree bit for bit
with the oracle's, and invalid arguments are rejected before any launch."""
import ctypes
import os
import re

import numpy as np
import pytest

import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kq():
    from quant_weight_gemv_dequant_b300 import build
    build.build()
    import quant_weight_gemv_dequant_b300 as k
    k.lib()
    return k


def _declared_functions():
    names = set()
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*[A-Za-z_][\w\s\*]*?\b(kq_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("kq_gemv", "kq_layer_step", "kq_dequantize", "kq_quantize",
                     "kq_merge_g128", "kq_block_bytes", "kq_matrix_bytes", "kq_status_str"):
        assert required in names


def test_every_declaration_states_its_source():
    # the comment right above each function declaration carries a "Source:"
    # line: the page passage that defines it, or that the pages define none
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        for m in re.finditer(r"^\s*[A-Za-z_][\w\s\*]*?\b(kq_\w+)\s*\(", text, flags=re.M):
            before = text[:m.start()]
            c0, c1 = before.rfind("/*"), before.rfind("*/")
            assert c0 >= 0 and c1 > c0, m.group(1)
            assert not before[c1 + 2:].strip(), f"{m.group(1)}: no comment right above"
            assert "Source:" in before[c0:c1], f"{m.group(1)}: comment has no Source: line"


def test_library_exports_every_declared_symbol(kq):
    L = ctypes.CDLL(kq.LIB_PATH)
    for name in _declared_functions():
        assert hasattr(L, name), name


def test_sizes_and_status_strings(kq):
    assert [kq.kq_block_bytes(f) for f in range(4)] == [144, 176, 210, 136]
    assert kq.kq_block_bytes(9) == 0
    assert kq.kq_matrix_bytes(kq.Q4_K, 4096, 4096) == 9437184
    assert kq.kq_matrix_bytes(kq.Q6_K, 200000, 5120) == 200000 * 20 * 210
    assert kq.kq_matrix_bytes(kq.Q4_G128, 4096, 5120) == 11141120
    assert kq.kq_matrix_bytes(kq.Q4_K, 4, 300) == 0
    for s in range(10):
        assert kq.kq_status_str(s)


@pytest.mark.parametrize("fmt", [0, 1, 2, 3])
def test_host_quantiser_matches_oracle_bytes(kq, oracle, fmt):
    # Same rule written twice (library C++ and oracle C) must give the same
    # bytes: normal, heavy-tailed, constant, zero and tiny-magnitude data.
    N, K = 24, 768
    w = wl.weights_f32(wl.derive_seed(30, fmt), N, K)
    u = wl.uniform01(wl.derive_seed(31), 0, N * K).reshape(N, K)
    w[4:8] = np.where(u[4:8] < 0.05, w[4:8] * 20, w[4:8])
    w[8] = 0.0
    w[9] = -0.125
    w[10] *= 1e-6
    w[11] = np.abs(w[11]) + 0.3
    a = kq.kq_quantize(fmt, w, N, K)
    b = oracle.quantize(fmt, w, N, K)
    assert np.array_equal(a, b)


def test_host_quantiser_pool_matches_oracle(kq, oracle):
    pw = wl.pool_weights(wl.derive_seed(32), 2048)
    for fmt in (0, 1, 2, 3):
        assert np.array_equal(kq.kq_quantize(fmt, pw, 2048, 256), oracle.quantize(fmt, pw, 2048, 256))


def test_host_quantiser_range_error(kq):
    w = np.zeros((1, 256), np.float32)
    w[0, 5] = -4e9
    for fmt in range(4):
        with pytest.raises(kq.KqError) as e:
            kq.kq_quantize(fmt, w, 1, 256)
        assert e.value.status == 5


def test_host_merge_matches_oracle(kq, oracle):
    N, K = 10, 1280
    w = wl.weights_f32(wl.derive_seed(33), N, K)
    q4g = oracle.quantize_q4k_group128(w, N, K)
    st, g = kq.kq_merge_g128(q4g, N, K)
    st_o, g_o = oracle.merge_g128(q4g, N, K)
    assert st == 0 and st_o == 0 and np.array_equal(g, g_o)
    q4 = oracle.quantize(oracle.Q4_K, w, N, K)
    assert kq.kq_merge_g128(q4, N, K)[0] == 4


def test_validation_rejects_before_launch(kq):
    # None of these reaches a CUDA call: statuses come from host validation.
    A16 = 1 << 20          # a 16-byte aligned (never dereferenced) address
    cases = [
        (dict(fmt=7), 1), (dict(W=0), 1), (dict(x=0), 1), (dict(y=0), 1),
        (dict(n_tok=0), 1), (dict(n_tok=17), 1), (dict(K=300), 2), (dict(K=0), 2),
        (dict(N_out=0), 2), (dict(N_out=-4), 2), (dict(W=A16 + 8), 3), (dict(x=A16 + 2), 3),
        (dict(y=A16 + 2), 3),
    ]
    for over, want in cases:
        a = dict(fmt=0, W=A16, x=A16, y=A16, N_out=16, K=256, n_tok=1)
        a.update(over)
        st = kq.kq_gemv(a["fmt"], a["W"], a["x"], a["y"], a["N_out"], a["K"], a["n_tok"],
                        stream=0, check=False)
        assert st == want, (over, st)
    assert kq.kq_dequantize(0, A16, 0, 4, 256, stream=0, check=False) == 1
    assert kq.kq_dequantize(0, A16 + 4, A16, 4, 256, stream=0, check=False) == 3
    # layer step: mismatched K between q and k
    m = kq.make_matrix(0, A16, 256, 512)
    bad = kq.make_matrix(0, A16, 256, 768)
    layer = kq.kq_layer(m, bad, m, m, m, m, m)
    io = kq.kq_layer_io(*([A16] * 11))
    assert kq.kq_layer_step(layer, io, 1, stream=0, check=False) == 2
    layer = kq.kq_layer(m, m, m, m, m, m, m)
    io.y_v = 0
    assert kq.kq_layer_step(layer, io, 1, stream=0, check=False) == 1


def test_binding_raises_without_library(monkeypatch, tmp_path):
    import quant_weight_gemv_dequant_b300 as k
    monkeypatch.setattr(k, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(k, "_lib", None)
    with pytest.raises(k.KqError):
        k.lib()
