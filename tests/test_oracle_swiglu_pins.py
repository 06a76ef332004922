"""Pins of the oracle's SwiGLU pieces against things other than themselves.

silu(v) = v * s(v), s the logistic function (the standard reading of the
SwiGLU block named in the Core AI card's architecture section):
  * closed forms: silu(0) = 0; s(ln 3) = 3/4, so silu(ln 3) = 0.75 ln 3;
    silu(v) - silu(-v) = v for every v; silu(v) -> v and silu(-v) -> -0 for
    large v;
  * the library routine: v * scipy.special.expit(v) within 2 ulp.
bf16 rounding from fp64 (ties to even): torch's fp32 -> bf16 conversion on
values that fp32 holds exactly (then there is no double rounding), hand-made
ties, overflow to infinity, subnormals.
sum_k |w^| e: numpy on the dequantised matrix, and the oracle's own A (the
tolerance sum) when e = |x|.
"""
import math

import numpy as np
import pytest

import workloads as wl


def test_silu_closed_forms(oracle):
    assert oracle.silu(0.0) == 0.0
    assert math.isclose(oracle.silu(math.log(3.0)), 0.75 * math.log(3.0), rel_tol=4e-16)
    for v in (1e-300, 1e-8, 0.3, 1.0, 2.5, 17.0, 300.0):
        assert math.isclose(oracle.silu(v) - oracle.silu(-v), v, rel_tol=4e-16, abs_tol=1e-300)
    assert oracle.silu(800.0) == 800.0
    s = oracle.silu(-800.0)
    assert s == 0.0 and math.copysign(1.0, s) == -1.0
    # silu(-40) = -40 e^-40 / (1 + e^-40)
    assert math.isclose(oracle.silu(-40.0), -40.0 * math.exp(-40.0) / (1 + math.exp(-40.0)), rel_tol=1e-15)


def test_silu_matches_scipy_expit():
    from scipy.special import expit
    import oracle as o
    v = np.concatenate([np.linspace(-60, 60, 4001), wl.normal_f32(wl.derive_seed(510), 2000, 3.0)
                        .astype(np.float64)])
    ref = v * expit(v)
    got = np.array([o.silu(float(a)) for a in v])
    ulp = np.spacing(np.maximum(np.abs(ref), 1e-300))
    assert np.all(np.abs(got - ref) <= 2 * ulp)


def test_bf16_from_double_matches_torch_on_fp32_values(oracle):
    torch = pytest.importorskip("torch")
    f32 = np.concatenate([wl.normal_f32(wl.derive_seed(511), 20000, 1.0),
                          wl.normal_f32(wl.derive_seed(512), 2000, 1e-38),
                          wl.normal_f32(wl.derive_seed(513), 2000, 1e37),
                          np.array([0.0, -0.0, 1.0, -1.0, 3.3895314e38, 1e-45], np.float32)])
    # fp32 values whose low 16 bits make exact ties between two bf16 values
    ties = (wl.splitmix64(514, np.arange(2000, dtype=np.uint64)).astype(np.uint32) & 0x7F7F0000) | 0x8000
    f32 = np.concatenate([f32, ties.view(np.float32)])
    ref = torch.from_numpy(f32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_from_double(float(v)) for v in f32], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_from_double_hand_cases(oracle):
    assert oracle.bf16_from_double(1.0) == 0x3F80
    assert oracle.bf16_from_double(1 + 2 ** -8) == 0x3F80          # tie -> even (1.0)
    assert oracle.bf16_from_double(1 + 3 * 2 ** -8) == 0x3F82      # tie -> even (1 + 2^-6)
    assert oracle.bf16_from_double(1 + 2 ** -8 + 2 ** -40) == 0x3F81   # above the tie: no double rounding
    assert oracle.bf16_from_double(-2.5) == 0xC020
    assert oracle.bf16_from_double(3.5e38) == 0x7F80               # overflow -> +inf
    assert oracle.bf16_from_double(-3.5e38) == 0xFF80
    assert oracle.bf16_from_double(2.0 ** -133) == 0x0001          # smallest subnormal
    assert oracle.bf16_from_double(2.0 ** -135) == 0x0000          # below half of it: +0
    assert oracle.bf16_from_double(-0.0) == 0x8000


def test_swiglu_elementwise(oracle):
    g = np.array([0.0, math.log(3.0), 2.0, -3.0, 40.0])
    u = np.array([5.0, 4.0, -0.5, 2.0, 0.25])
    h, hb = oracle.swiglu(g, u)
    assert h[0] == 0.0
    assert math.isclose(h[1], 3.0 * math.log(3.0), rel_tol=1e-15)
    assert math.isclose(h[2], -0.5 * 2.0 / (1 + math.exp(-2.0)), rel_tol=1e-15)
    assert math.isclose(h[4], 10.0, rel_tol=1e-15)
    assert all(hb[i] == oracle.bf16_from_double(h[i]) for i in range(5))


@pytest.mark.parametrize("fmt", [0, 2])
def test_gemv_absw_matches_numpy_and_A(oracle, fmt):
    N, K = 9, 768
    Wb = oracle.quantize(fmt, wl.weights_f32(wl.derive_seed(515, fmt), N, K), N, K)
    w = oracle.dequantize(fmt, Wb, N, K)
    e = np.abs(wl.normal_f32(wl.derive_seed(516), K, 1.0).astype(np.float64))
    got = oracle.gemv_absw(fmt, Wb, N, K, e)
    assert np.allclose(got, np.abs(w) @ e, rtol=1e-13, atol=0)
    # with e = |x| it is the tolerance sum A of the product
    x = wl.activations_bf16(wl.derive_seed(517), 1, K)
    xd = np.array([oracle.bf16_to_double(int(b)) for b in x[0]])
    _, A = oracle.gemv(fmt, Wb, N, K, x)
    assert np.allclose(oracle.gemv_absw(fmt, Wb, N, K, np.abs(xd)), A[0], rtol=1e-13, atol=0)
