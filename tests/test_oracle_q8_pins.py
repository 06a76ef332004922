"""Pins of the oracle's int8-activation pieces (the dp4a path).

The quantiser (per 32 activations of a token: dx = amax/127, xq =
rint(x/dx) in fp32) is pinned by what the definition forces, not by
retyping it: the largest |x| of a block maps to +-127; every value lies
within half a step of its code; all-zero blocks give zeros; negating x
negates the codes; codes are monotone in x within a block; exact multiples
of the step give their multiple, and exact half-steps round to even.  The
GEMV of the path is pinned against numpy on the dequantised matrix and the
dequantised activations.
"""
import numpy as np
import pytest

import workloads as wl


def _bf16(v):
    return wl.bf16_bits(np.asarray(v, dtype=np.float32))


def _x_f64(x_bits):
    return (x_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_quantiser_extremes_and_half_step(oracle):
    x = np.concatenate([wl.activations_bf16(wl.derive_seed(570), 3, 1024),
                        wl.activations_bf16(wl.derive_seed(571), 1, 1024, heavy=True)])
    xq, dx = oracle.quantize_x_q8(x, 1024)
    xv = _x_f64(x).reshape(4, 32, 32)
    q = xq.reshape(4, 32, 32).astype(np.int64)
    assert np.all(np.abs(q) <= 127)
    # the block's largest |x| takes the extreme code
    i = np.argmax(np.abs(xv), axis=2)
    ext = np.take_along_axis(q, i[..., None], axis=2)[..., 0]
    sgn = np.sign(np.take_along_axis(xv, i[..., None], axis=2)[..., 0])
    assert np.all(ext == 127 * sgn)
    # every value within half a step of its code, plus the rounding of the
    # fp32 quotient x / dx (|x / dx| <= 127: at most 127 2^-24 of a step),
    # which can turn a value just inside a half step into a tie
    d = dx.astype(np.float64)[..., None]
    assert np.all(np.abs(xv - d * q) <= d * (0.5 + 128 * 2.0 ** -24))


def test_quantiser_zero_sign_and_order(oracle):
    x = wl.activations_bf16(wl.derive_seed(572), 2, 256)
    x[0, 32:64] = 0                                   # one all-zero block
    xq, dx = oracle.quantize_x_q8(x, 256)
    assert np.all(xq[0, 32:64] == 0) and dx[0, 1] == 0.0
    xn = x ^ np.uint16(0x8000)                        # -x (sign bit)
    xqn, dxn = oracle.quantize_x_q8(xn, 256)
    assert np.array_equal(dxn, dx)
    assert np.array_equal(xqn.astype(np.int64), -xq.astype(np.int64))
    xv = _x_f64(x).reshape(-1, 32)
    q = xq.reshape(-1, 32)
    for b in range(xv.shape[0]):
        o = np.argsort(xv[b], kind="stable")
        assert np.all(np.diff(q[b][o].astype(np.int64)) >= 0)


def test_quantiser_exact_multiples_and_ties(oracle):
    # block max 127 * 2^-7: dx = 2^-7 exactly; x = k 2^-7 -> k; x = (k + 1/2)
    # 2^-7 -> the even neighbour
    k = np.arange(-127, 128)
    x = np.zeros(512, dtype=np.float64)
    x[:32] = np.concatenate([[127.0], k[::8][:31]]) * 2.0 ** -7
    halves = np.array([0.5, 1.5, 2.5, -0.5, -1.5, 3.5, 6.5, -6.5, 100.5, -100.5])
    x[32:64] = np.concatenate([[127.0], halves, np.zeros(21)]) * 2.0 ** -7
    xb = _bf16(x).reshape(1, 512)
    assert np.array_equal(_x_f64(xb[0]), x)           # all exact in bf16
    xq, dx = oracle.quantize_x_q8(xb, 512)
    assert dx[0, 0] == np.float32(2.0 ** -7) and dx[0, 1] == np.float32(2.0 ** -7)
    assert np.array_equal(xq[0, :32].astype(np.int64), np.round(x[:32] * 128).astype(np.int64))
    assert list(xq[0, 33:43]) == [0, 2, 2, 0, -2, 4, 6, -6, 100, -100]


@pytest.mark.parametrize("fmt", [0, 1, 2, 3])
def test_gemv_q8_matches_numpy(oracle, fmt):
    N, K, T = 11, 1024, 3
    Wb = oracle.quantize(fmt, wl.weights_f32(wl.derive_seed(573, fmt), N, K), N, K)
    x = wl.activations_bf16(wl.derive_seed(574), T, K, heavy=True)
    xq, dx = oracle.quantize_x_q8(x, K)
    y, A = oracle.gemv_q8(fmt, Wb, N, K, xq, dx)
    w = oracle.dequantize(fmt, Wb, N, K)
    xt = xq.astype(np.float64) * np.repeat(dx.astype(np.float64), 32, axis=1)
    assert np.allclose(y, xt @ w.T, rtol=1e-12, atol=1e-12)
    assert np.allclose(A, np.abs(xt) @ np.abs(w).T, rtol=1e-12, atol=0)
