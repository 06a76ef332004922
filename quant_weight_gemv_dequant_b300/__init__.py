"""Python binding of libkq (include/kq.h): K-quant GEMV on one B300.

Argument marshalling only: every computation runs in libkq.so (CUDA kernels
for sm_103a, plus the host-side quantiser and merge).  There is no fallback:
if the library is missing, every call raises ``KqError``.

Functions keep the C names (``kq_gemv``, ``kq_layer_step``, ``kq_dequantize``,
``kq_quantize``, ``kq_merge_g128``, ``kq_block_bytes``, ``kq_matrix_bytes``,
``kq_status_str``).  Device arguments are torch CUDA tensors (or raw device
addresses as ints); streams default to torch's current stream.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

Q4_K, Q5_K, Q6_K, Q4_G128 = 0, 1, 2, 3
FORMATS = {"Q4_K": Q4_K, "Q5_K": Q5_K, "Q6_K": Q6_K, "Q4_G128": Q4_G128}
KQ_OK = 0
STATUS_NAMES = {0: "KQ_OK", 1: "KQ_ERR_ARG", 2: "KQ_ERR_SHAPE", 3: "KQ_ERR_ALIGN",
                4: "KQ_ERR_NOT_MERGEABLE", 5: "KQ_ERR_RANGE", 6: "KQ_ERR_CUDA",
                7: "KQ_ERR_UNSUPPORTED", 8: "KQ_ERR_TIMEOUT", 9: "KQ_ERR_TOO_LARGE"}

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkq.so")
_lib = None


class KqError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")


class kq_matrix(ctypes.Structure):
    _fields_ = [("format", ctypes.c_int), ("W", ctypes.c_void_p),
                ("N_out", ctypes.c_int64), ("K", ctypes.c_int64)]


class kq_gguf_tensor(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 128), ("ggml_type", ctypes.c_int32),
                ("format", ctypes.c_int32), ("n_dims", ctypes.c_int32),
                ("dims", ctypes.c_int64 * 4), ("N_out", ctypes.c_int64), ("K", ctypes.c_int64),
                ("data_offset", ctypes.c_uint64), ("bytes", ctypes.c_uint64)]


class kq_layer(ctypes.Structure):
    _fields_ = [(n, kq_matrix) for n in ("q", "k", "v", "o", "gate", "up", "down")]


class kq_layer_io(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("x_attn", "x_o", "x_ffn", "x_down",
                                                "y_q", "y_k", "y_v", "y_o", "y_gate",
                                                "y_up", "y_down")]


def lib() -> ctypes.CDLL:
    """The loaded libkq.so; raises KqError if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise KqError(7, f"libkq.so not found at {LIB_PATH}; build it with "
                             "python -m quant_weight_gemv_dequant_b300.build")
        L = ctypes.CDLL(LIB_PATH)
        P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.kq_block_bytes.argtypes = [I]
        L.kq_block_bytes.restype = ctypes.c_size_t
        L.kq_matrix_bytes.argtypes = [I, I64, I64]
        L.kq_matrix_bytes.restype = ctypes.c_size_t
        L.kq_gemv.argtypes = [I, P, P, P, I64, I64, I, P]
        L.kq_gemv_multi.argtypes = [I, I, P, P, P, P, I64, I, P]
        L.kq_gemv_noalloc.argtypes = [I, P, P, P, I64, I64, I, P]
        L.kq_layer_step.argtypes = [ctypes.POINTER(kq_layer), ctypes.POINTER(kq_layer_io), I, P]
        L.kq_gemv_swiglu.argtypes = [I, P, P, P, P, P, P, I64, I64, I, P]
        L.kq_gemv_q8.argtypes = [I, P, P, P, I64, I64, I, P]
        L.kq_gguf_index.argtypes = [P, ctypes.c_size_t, ctypes.POINTER(kq_gguf_tensor), I,
                                    ctypes.POINTER(I), ctypes.POINTER(ctypes.c_uint32)]
        L.kq_gguf_index.restype = I
        L.kq_quantize_x_q8.argtypes = [P, I64, I, P, P, P]
        L.kq_ffn_swiglu.argtypes = [ctypes.POINTER(kq_matrix)] * 3 + [P, P, P, P, P, I, P]
        L.kq_dequantize.argtypes = [I, P, P, I64, I64, P]
        L.kq_quantize.argtypes = [I, P, I64, I64, P]
        L.kq_merge_g128.argtypes = [P, I64, I64, P]
        L.kq_device_status.argtypes = [P]
        L.kq_device_status.restype = I
        L.kq_test_wait_timeout.argtypes = [ctypes.c_uint, P]
        L.kq_test_wait_timeout.restype = I
        L.kq_status_str.argtypes = [I]
        L.kq_status_str.restype = ctypes.c_char_p
        for name in ("kq_gemv", "kq_gemv_multi", "kq_gemv_noalloc", "kq_layer_step", "kq_dequantize",
                     "kq_quantize", "kq_merge_g128", "kq_gemv_swiglu", "kq_ffn_swiglu",
                     "kq_gemv_q8", "kq_quantize_x_q8"):
            getattr(L, name).restype = I
        _lib = L
    return _lib


def _addr(t) -> int:
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(st: int, where: str) -> int:
    if st != KQ_OK:
        raise KqError(st, where)
    return st


def kq_status_str(status: int) -> str:
    try:
        return lib().kq_status_str(status).decode()
    except KqError:
        return STATUS_NAMES.get(status, "unknown")


def kq_device_status(stream=None, check=True) -> int:
    """Synchronise the stream and report whether any bounded wait timed out."""
    st = lib().kq_device_status(_stream(stream))
    return _check(st, "kq_device_status") if check else st


def kq_test_wait_timeout(wait_us: int, stream=None, check=True) -> int:
    """Launch one warp whose bounded wait (about wait_us) runs out; the next
    kq_device_status reports KQ_ERR_TIMEOUT.  For testing the failure path."""
    st = lib().kq_test_wait_timeout(wait_us, _stream(stream))
    return _check(st, "kq_test_wait_timeout") if check else st


def kq_block_bytes(fmt: int) -> int:
    return lib().kq_block_bytes(fmt)


def kq_matrix_bytes(fmt: int, N_out: int, K: int) -> int:
    return lib().kq_matrix_bytes(fmt, N_out, K)


def kq_gemv(fmt, W, x, y, N_out, K, n_tok, stream=None, check=True) -> int:
    """y[t][n] = sum_k w^[n][k] x[t][k] (device tensors; y overwritten)."""
    st = lib().kq_gemv(fmt, _addr(W), _addr(x), _addr(y), N_out, K, n_tok, _stream(stream))
    return _check(st, "kq_gemv") if check else st


def kq_gemv_noalloc(fmt, W, x, y, N_out, K, n_tok, stream=None, check=True) -> int:
    """kq_gemv that never allocates device memory (fixed 4 MiB scratch);
    KQ_ERR_TOO_LARGE for requests beyond that array."""
    st = lib().kq_gemv_noalloc(fmt, _addr(W), _addr(x), _addr(y), N_out, K, n_tok,
                               _stream(stream))
    return _check(st, "kq_gemv_noalloc") if check else st


def kq_gemv_multi(fmt, Ws, ys, N_outs, x, K, n_tok, stream=None, check=True) -> int:
    """y_i = w^_i x for up to four matrices sharing x, in one launch."""
    n = len(Ws)
    Wa = (ctypes.c_void_p * n)(*[_addr(w) for w in Ws])
    ya = (ctypes.c_void_p * n)(*[_addr(v) for v in ys])
    Na = (ctypes.c_int64 * n)(*N_outs)
    st = lib().kq_gemv_multi(fmt, n, Wa, ya, Na, _addr(x), K, n_tok, _stream(stream))
    return _check(st, "kq_gemv_multi") if check else st


def kq_gemv_q8(fmt, W, x, y, N_out, K, n_tok, stream=None, check=True) -> int:
    """The int8-activation (dp4a) GEMV: y = w^ x~, x~ = x quantised per 32."""
    st = lib().kq_gemv_q8(fmt, _addr(W), _addr(x), _addr(y), N_out, K, n_tok, _stream(stream))
    return _check(st, "kq_gemv_q8") if check else st


def kq_quantize_x_q8(x, K, n_tok, xq, dx, stream=None, check=True) -> int:
    """The activation codes (int8 [n_tok][K]) and steps (fp32 [n_tok][K/32]) of kq_gemv_q8."""
    st = lib().kq_quantize_x_q8(_addr(x), K, n_tok, _addr(xq), _addr(dx), _stream(stream))
    return _check(st, "kq_quantize_x_q8") if check else st


def kq_gemv_swiglu(fmt, W_gate, W_up, x, y_gate, y_up, h, N_out, K, n_tok, stream=None,
                   check=True) -> int:
    """y_gate, y_up = w^ x for the pair; h = bf16(silu(y_gate) * y_up) (bf16 tensor)."""
    st = lib().kq_gemv_swiglu(fmt, _addr(W_gate), _addr(W_up), _addr(x), _addr(y_gate), _addr(y_up),
                              _addr(h), N_out, K, n_tok, _stream(stream))
    return _check(st, "kq_gemv_swiglu") if check else st


def kq_ffn_swiglu(gate: kq_matrix, up: kq_matrix, down: kq_matrix, x, y_gate, y_up, h, y_down,
                  n_tok: int, stream=None, check=True) -> int:
    """kq_gemv_swiglu(gate, up) into h, then y_down = w^_down h."""
    st = lib().kq_ffn_swiglu(ctypes.byref(gate), ctypes.byref(up), ctypes.byref(down), _addr(x),
                             _addr(y_gate), _addr(y_up), _addr(h), _addr(y_down), n_tok,
                             _stream(stream))
    return _check(st, "kq_ffn_swiglu") if check else st


def kq_layer_step(layer: kq_layer, io: kq_layer_io, n_tok: int, stream=None, check=True) -> int:
    st = lib().kq_layer_step(ctypes.byref(layer), ctypes.byref(io), n_tok, _stream(stream))
    return _check(st, "kq_layer_step") if check else st


def kq_dequantize(fmt, W, W_out, N_out, K, stream=None, check=True) -> int:
    st = lib().kq_dequantize(fmt, _addr(W), _addr(W_out), N_out, K, _stream(stream))
    return _check(st, "kq_dequantize") if check else st


def kq_quantize(fmt: int, W_host: np.ndarray, N_out: int, K: int) -> np.ndarray:
    """Host quantiser: fp32 [N_out][K] -> uint8 blocks."""
    W = np.ascontiguousarray(W_host, dtype=np.float32)
    out = np.zeros(max(1, kq_matrix_bytes(fmt, N_out, K)), dtype=np.uint8)
    _check(lib().kq_quantize(fmt, W.ctypes.data, N_out, K, out.ctypes.data), "kq_quantize")
    return out


def kq_gguf_index(data, max_tensors: int = 4096):
    """Index a GGUF checkpoint held in host memory (bytes or a uint8 array):
    (status, [kq_gguf_tensor], alignment)."""
    buf = np.frombuffer(data, dtype=np.uint8) if isinstance(data, (bytes, bytearray)) else \
        np.ascontiguousarray(data, dtype=np.uint8)
    out = (kq_gguf_tensor * max_tensors)()
    n = ctypes.c_int(0)
    al = ctypes.c_uint32(0)
    st = lib().kq_gguf_index(buf.ctypes.data, buf.size, out, max_tensors, ctypes.byref(n),
                             ctypes.byref(al))
    if st != KQ_OK:
        return st, [], 0
    return st, [out[i] for i in range(min(n.value, max_tensors))], al.value


def kq_merge_g128(q4k_host: np.ndarray, N_out: int, K: int):
    """Host merge Q4_K -> Q4_G128; returns (status, bytes)."""
    src = np.ascontiguousarray(q4k_host, dtype=np.uint8)
    out = np.zeros(max(1, kq_matrix_bytes(Q4_G128, N_out, K)), dtype=np.uint8)
    st = lib().kq_merge_g128(src.ctypes.data, N_out, K, out.ctypes.data)
    return st, out


# ------------------------------------------------------------ conveniences

def gemv(fmt: int, W, x, N_out: int, K: int, stream=None):
    """Allocate y (fp32 [n_tok][N_out]) and run kq_gemv."""
    import torch
    n_tok = x.numel() // K
    y = torch.empty((n_tok, N_out), dtype=torch.float32, device=x.device)
    kq_gemv(fmt, W, x, y, N_out, K, n_tok, stream)
    return y


def make_matrix(fmt: int, W, N_out: int, K: int) -> kq_matrix:
    return kq_matrix(fmt, _addr(W), N_out, K)
