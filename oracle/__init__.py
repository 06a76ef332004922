"""CPU oracle for K-quant GEMV -- TEST INFRASTRUCTURE ONLY.

This package is the plain fp64 reference that the GPU library is checked
against.  Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` may import it; the library never does, and it never imports
the library.  The arithmetic lives in ``kq_oracle.c`` (single-threaded,
fp64, built with ``-O2 -ffp-contract=off``); this module only builds it with
gcc and marshals numpy arrays.

Sources (see the header of ``kq_oracle.c`` for the per-function passages):
the daily.dev summary "Fast on-device agentic AI with Muse Glimmer on
ExecuTorch" (answer on exporting GGUF checkpoints: Q4_K/Q5_K/Q6_K GEMV and the
lossless merge into groups of up to 128) and the SGLang day-0 post (GGUF
paragraph: a Q4_K_M checkpoint with 128-weight groups).

Parity unpinned: GGUF bit-placement compatibility with real checkpoint files.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

Q4_K, Q5_K, Q6_K, Q4_G128 = 0, 1, 2, 3
FORMATS = (Q4_K, Q5_K, Q6_K, Q4_G128)
NAMES = {Q4_K: "Q4_K", Q5_K: "Q5_K", Q6_K: "Q6_K", Q4_G128: "Q4_G128"}
BLOCK_BYTES = {Q4_K: 144, Q5_K: 176, Q6_K: 210, Q4_G128: 136}

OK, BAD_ARG, BAD_SHAPE, NOT_MERGEABLE, RANGE = 0, 1, 2, 4, 5

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kq_oracle.c")
_LIB = os.path.join(_HERE, "libkqoracle.so")
_lib = None


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile kq_oracle.c into libkqoracle.so next to it (gcc, fp64, no
    contraction) and return the path."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-o", _LIB + ".tmp", _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I = ctypes.c_int
        lib.kqo_block_bytes.argtypes = [I]
        lib.kqo_half_to_double.argtypes = [ctypes.c_uint16]
        lib.kqo_half_to_double.restype = ctypes.c_double
        lib.kqo_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.kqo_bf16_to_double.restype = ctypes.c_double
        lib.kqo_half_round_up.argtypes = [ctypes.c_double, P, P]
        lib.kqo_dequantize.argtypes = [I, P, I64, I64, P]
        lib.kqo_gemv.argtypes = [I, P, I64, I64, P, I, P, P]
        lib.kqo_gemv_rows.argtypes = [I, P, I64, I64, P, I64, P, I, P, P]
        lib.kqo_quantize.argtypes = [I, P, I64, I64, P]
        lib.kqo_quantize_q4k_group128.argtypes = [P, I64, I64, P]
        lib.kqo_merge_g128.argtypes = [P, I64, I64, P]
        lib.kqo_silu.argtypes = [ctypes.c_double]
        lib.kqo_silu.restype = ctypes.c_double
        lib.kqo_bf16_from_double.argtypes = [ctypes.c_double]
        lib.kqo_bf16_from_double.restype = ctypes.c_uint16
        lib.kqo_swiglu.argtypes = [P, P, I64, P, P]
        lib.kqo_swiglu.restype = None
        lib.kqo_gemv_absw.argtypes = [I, P, I64, I64, P, P]
        lib.kqo_quantize_x_q8.argtypes = [P, I, I64, P, P]
        lib.kqo_gemv_q8.argtypes = [I, P, I64, I64, P, P, I, P, P]
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _check(st: int, what: str):
    if st != OK:
        raise OracleError(f"{what} failed with status {st}")


def matrix_bytes(fmt: int, N: int, K: int) -> int:
    return N * (K // 256) * BLOCK_BYTES[fmt]


def half_to_double(h: int) -> float:
    return _load().kqo_half_to_double(h)


def bf16_to_double(b: int) -> float:
    return _load().kqo_bf16_to_double(b)


def half_round_up(v: float):
    """(value, bits) of the smallest fp16 >= v, or None above 65504."""
    val = ctypes.c_double()
    bits = ctypes.c_uint16()
    ok = _load().kqo_half_round_up(v, ctypes.byref(val), ctypes.byref(bits))
    return (val.value, bits.value) if ok else None


def dequantize(fmt: int, W: np.ndarray, N: int, K: int) -> np.ndarray:
    """w^ as fp64 [N][K]."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    assert W.size >= matrix_bytes(fmt, N, K)
    out = np.empty((N, K), dtype=np.float64)
    _check(_load().kqo_dequantize(fmt, _ptr(W), N, K, _ptr(out)), "dequantize")
    return out


def gemv(fmt: int, W: np.ndarray, N: int, K: int, x_bf16: np.ndarray):
    """(y, A), each fp64 [n_tok][N]: y = sum_k w^ x in k order, A = sum |w^ x|."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16).reshape(-1, K)
    n_tok = x.shape[0]
    y = np.empty((n_tok, N), dtype=np.float64)
    A = np.empty((n_tok, N), dtype=np.float64)
    _check(_load().kqo_gemv(fmt, _ptr(W), N, K, _ptr(x), n_tok, _ptr(y), _ptr(A)), "gemv")
    return y, A


def gemv_rows(fmt: int, W: np.ndarray, N: int, K: int, rows, x_bf16: np.ndarray):
    """(y, A), each fp64 [n_tok][len(rows)], for the listed output rows only."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16).reshape(-1, K)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    n_tok = x.shape[0]
    y = np.empty((n_tok, rows.size), dtype=np.float64)
    A = np.empty((n_tok, rows.size), dtype=np.float64)
    _check(_load().kqo_gemv_rows(fmt, _ptr(W), N, K, _ptr(rows), rows.size, _ptr(x),
                                 n_tok, _ptr(y), _ptr(A)), "gemv_rows")
    return y, A


def quantize(fmt: int, W_f32: np.ndarray, N: int, K: int) -> np.ndarray:
    W = np.ascontiguousarray(W_f32, dtype=np.float32).reshape(N, K)
    out = np.zeros(matrix_bytes(fmt, N, K), dtype=np.uint8)
    _check(_load().kqo_quantize(fmt, _ptr(W), N, K, _ptr(out)), "quantize")
    return out


def quantize_q4k_group128(W_f32: np.ndarray, N: int, K: int) -> np.ndarray:
    """Q4_K blocks whose (sc, m) are taken over 128-weight groups (mergeable)."""
    W = np.ascontiguousarray(W_f32, dtype=np.float32).reshape(N, K)
    out = np.zeros(matrix_bytes(Q4_K, N, K), dtype=np.uint8)
    _check(_load().kqo_quantize_q4k_group128(_ptr(W), N, K, _ptr(out)), "quantize_q4k_group128")
    return out


def merge_g128(q4k: np.ndarray, N: int, K: int):
    """(status, G128 bytes).  status is OK or NOT_MERGEABLE."""
    q4k = np.ascontiguousarray(q4k, dtype=np.uint8)
    out = np.zeros(matrix_bytes(Q4_G128, N, K), dtype=np.uint8)
    st = _load().kqo_merge_g128(_ptr(q4k), N, K, _ptr(out))
    return st, out


def silu(v: float) -> float:
    """silu(v) = v / (1 + e^-v) in fp64."""
    return _load().kqo_silu(float(v))


def bf16_from_double(v: float) -> int:
    """bf16 bits of v rounded to nearest, ties to even (from the double)."""
    return _load().kqo_bf16_from_double(float(v))


def swiglu(g: np.ndarray, u: np.ndarray):
    """(h_exact fp64, h_bf16 uint16 bits) with h = silu(g) * u elementwise."""
    g = np.ascontiguousarray(g, dtype=np.float64)
    u = np.ascontiguousarray(u, dtype=np.float64)
    assert g.shape == u.shape
    h = np.empty(g.shape, dtype=np.float64)
    hb = np.empty(g.shape, dtype=np.uint16)
    _load().kqo_swiglu(_ptr(g), _ptr(u), g.size, _ptr(h), _ptr(hb))
    return h, hb


def gemv_absw(fmt: int, W: np.ndarray, N: int, K: int, e: np.ndarray) -> np.ndarray:
    """sum_k |w^[n][k]| e[k] for every row n (fp64 [N]); e >= 0, length K."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    e = np.ascontiguousarray(e, dtype=np.float64).reshape(K)
    out = np.empty(N, dtype=np.float64)
    _check(_load().kqo_gemv_absw(fmt, _ptr(W), N, K, _ptr(e), _ptr(out)), "gemv_absw")
    return out


def quantize_x_q8(x_bf16: np.ndarray, K: int):
    """int8 activations of the dp4a path: (xq int8 [n_tok][K], dx fp32
    [n_tok][K/32]) with dx = amax/127 per 32-block, xq = rint(x / dx)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16).reshape(-1, K)
    n_tok = x.shape[0]
    xq = np.empty((n_tok, K), dtype=np.int8)
    dx = np.empty((n_tok, K // 32), dtype=np.float32)
    _check(_load().kqo_quantize_x_q8(_ptr(x), n_tok, K, _ptr(xq), _ptr(dx)), "quantize_x_q8")
    return xq, dx


def gemv_q8(fmt: int, W: np.ndarray, N: int, K: int, xq: np.ndarray, dx: np.ndarray):
    """(y, A) fp64 [n_tok][N] of the int8-activation GEMV: sum_k w^ * dx * xq."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.int8).reshape(-1, K)
    dx = np.ascontiguousarray(dx, dtype=np.float32).reshape(xq.shape[0], K // 32)
    n_tok = xq.shape[0]
    y = np.empty((n_tok, N), dtype=np.float64)
    A = np.empty((n_tok, N), dtype=np.float64)
    _check(_load().kqo_gemv_q8(fmt, _ptr(W), N, K, _ptr(xq), _ptr(dx), n_tok, _ptr(y), _ptr(A)),
           "gemv_q8")
    return y, A


def tolerance(A: np.ndarray) -> np.ndarray:
    """Per-element bound on |y - y_ref|: 1e-3 * sum|w^ x| + 1e-5."""
    return 1e-3 * A + 1e-5
