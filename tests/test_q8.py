"""GPU parity of the int8-activation (dp4a) GEMV, kq_gemv_q8.

  * The activation codes and steps (kq_quantize_x_q8, the kernel's own
    steps) are bit-exact against the oracle's: both take the same binary32
    decisions.  Hand-made blocks cover exact multiples, exact half steps
    (ties to even), zero blocks and the block maximum.
  * y matches the oracle's product of the same path, sum w^ dx xq in fp64,
    at the bar |y - y_ref| <= 1e-3 A + 1e-5 (A = sum |w^ x~|), for every
    format at 1..16 tokens, on quantised, random-byte and zero-weight
    records (tests/test_exact_edges.py's types), long rows split over K
    and grouped launches.
  * Against the bf16-activation product (the oracle's y for x itself) it
    stays within the activation rounding: sum_k |w^| dx(k) / 2, plus the
    bar.
"""
import numpy as np
import pytest

import workloads as wl
from test_exact_edges import degenerate_matrix

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
FMTS = [0, 1, 2, 3]
FMT_IDS = ["Q4_K", "Q5_K", "Q6_K", "G128"]


@pytest.fixture(scope="module")
def kq():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from quant_weight_gemv_dequant_b300 import build
    build.build()
    import quant_weight_gemv_dequant_b300 as k
    k.lib()
    return k


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _dev_x(x):
    return _dev(x.view(np.int16)).view(torch.bfloat16)


def test_codes_bit_exact(kq, oracle):
    K, T = 5120, 16
    x = wl.activations_bf16(wl.derive_seed(580), T, K, heavy=True)
    x[3, 64:96] = 0                                       # a zero block
    # exact multiples of 2^-7 and exact half steps in a block whose max is 127 2^-7
    vals = np.array([127.0, 0.5, 1.5, 2.5, -0.5, -1.5, 3.5, 6.5, -6.5, 100.5, -100.5, 64, -1, 0]
                    + [0.0] * 18) * 2.0 ** -7
    x[4, :32] = wl.bf16_bits(vals.astype(np.float32))
    xq_ref, dx_ref = oracle.quantize_x_q8(x, K)
    xq = torch.empty((T, K), dtype=torch.int8, device="cuda")
    dx = torch.empty((T, K // 32), dtype=torch.float32, device="cuda")
    kq.kq_quantize_x_q8(_dev_x(x), K, T, xq, dx)
    torch.cuda.synchronize()
    assert np.array_equal(xq.cpu().numpy(), xq_ref)
    assert np.array_equal(dx.cpu().numpy().view(np.uint32), dx_ref.view(np.uint32))


def _check(y, y_ref, A, what):
    err = np.abs(y.astype(np.float64) - y_ref)
    tol = 1e-3 * A + 1e-5
    bad = ~(err <= tol)
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err / tol, 0)), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside; worst {i}: "
                             f"y={y[i]!r} ref={y_ref[i]!r} tol={tol[i]!r}")


def _q8(kq, fmt, W, x, N, K):
    T = x.shape[0]
    y = torch.full((T, N), 1234.5, dtype=torch.float32, device="cuda")
    kq.kq_gemv_q8(fmt, _dev(W), _dev_x(x), y, N, K, T)
    assert kq.kq_device_status() == 0
    return y.cpu().numpy()


@pytest.mark.parametrize("fmt", FMTS, ids=FMT_IDS)
@pytest.mark.parametrize("shape", [(8300, 4352), (1100, 32768), (300, 2048), (7, 256)],
                         ids=lambda s: f"{s[0]}x{s[1]}")
def test_q8_matches_oracle(kq, oracle, fmt, shape):
    N, K = shape
    Wb = oracle.quantize(fmt, wl.weights_f32(wl.derive_seed(581, fmt, N), N, K), N, K)
    x = wl.activations_bf16(wl.derive_seed(582, N, K), 16, K, heavy=True)
    xq, dx = oracle.quantize_x_q8(x, K)
    y_ref, A = oracle.gemv_q8(fmt, Wb, N, K, xq, dx)
    for T in (1, 2, 3, 4, 5, 8, 16):
        _check(_q8(kq, fmt, Wb, x[:T], N, K), y_ref[:T], A[:T], f"fmt={fmt} {N}x{K} n_tok={T}")


@pytest.mark.parametrize("fmt", FMTS, ids=FMT_IDS)
def test_q8_random_and_zero_weight_records(kq, oracle, fmt):
    N, K = 1000, 4096
    W = degenerate_matrix(oracle, fmt, N, K, 590 + fmt)
    x = wl.activations_bf16(wl.derive_seed(591, fmt), 4, K, heavy=True)
    xq, dx = oracle.quantize_x_q8(x, K)
    y_ref, A = oracle.gemv_q8(fmt, W, N, K, xq, dx)
    for T in (1, 4):
        y = _q8(kq, fmt, W, x[:T], N, K)
        _check(y, y_ref[:T], A[:T], f"fmt={fmt} n_tok={T}")
        zero_rows = [r for r in range(N) if r % 37 in (0, 1, 4)]
        assert np.all(y[:, zero_rows] == 0.0)


@pytest.mark.parametrize("fmt", [0, 2], ids=["Q4_K", "Q6_K"])
def test_q8_within_activation_rounding_of_bf16_product(kq, oracle, fmt):
    N, K, T = 2000, 5120, 2
    Wb = oracle.quantize(fmt, wl.weights_f32(wl.derive_seed(592, fmt), N, K), N, K)
    x = wl.activations_bf16(wl.derive_seed(593), T, K, heavy=True)
    xq, dx = oracle.quantize_x_q8(x, K)
    y_bf16, A = oracle.gemv(fmt, Wb, N, K, x)
    y = _q8(kq, fmt, Wb, x, N, K)
    for t in range(T):
        bound = oracle.gemv_absw(fmt, Wb, N, K, np.repeat(dx[t].astype(np.float64), 32) / 2)
        tol = 1e-3 * (A[t] + bound) + 1e-5 + bound
        assert np.all(np.abs(y[t] - y_bf16[t]) <= tol), f"token {t}"
        # and the int8 path really differs from the bf16 one (it is a different product)
        assert np.any(y[t] != np.float32(y_bf16[t]))
