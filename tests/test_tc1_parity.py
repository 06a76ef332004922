"""GPU parity of launches on large matrices (at least 32 M weights) at one
token and at the verify widths.  At n_tok = 1, Q4_K and Q4_G128 run on the
tensor cores with the sub-blocks of the one token as the columns of the mma's
n8 operand (gemv_tc1); Q5_K and Q6_K on the streaming CUDA-core kernel.  At
n_tok 2..16, Q4_K and Q4_G128 run on the one-CTA-per-SM tensor-core kernel
with tokens as columns (gemv_tcv); Q5_K and Q6_K on gemv_mma.  n_tok 3 on the
1100 x 32768 shape is a full-size split-K launch at an odd width.

Every row is checked against the fp64 oracle (|y - y_ref| <= 1e-3 sum|w^ x| +
1e-5).  The shapes cover: ragged last tiles; an odd super-block count; Q6_K
and Q4_G128 rows whose stride is off the 16-byte grid (per-row bulk copies;
the tensor-core kernel declines those and the streaming kernel serves them);
long rows split into many K segments (split-K at verify widths; the
single-token kernel takes whole rows); K / 256 = 20 (its five-column
stages) with a ragged last tile;
rows on the 16-byte grid (2-D tensor copies); random block bytes (every scale
and field value); a grouped launch whose tiles straddle the two matrices; and
repeated launches (tiles are claimed at run time, the result must not vary).
"""
import numpy as np
import pytest

import workloads as wl

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
CANARY = 1234.5678
FMTS = [0, 1, 2, 3]
FMT_IDS = ["Q4_K", "Q5_K", "Q6_K", "G128"]

# (N, K): ragged tiles + odd K/256 (per-row copies for Q6_K and G128);
# long rows with few tiles (many K segments); rows on the 16-byte grid;
# K / 256 = 20 (the single-token kernel's five-column stages) with a ragged
# last 64-row tile
CASES = [(8300, 4352), (1100, 32768), (20000, 2048), (6600, 5120)]


@pytest.fixture(scope="module")
def kq():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from quant_weight_gemv_dequant_b300 import build
    build.build()
    import quant_weight_gemv_dequant_b300 as k
    k.lib()
    return k


_W = {}


def _weights_f32(N, K):
    if (N, K) not in _W:
        _W[(N, K)] = wl.weights_f32(wl.derive_seed(700, N, K), N, K)
    return _W[(N, K)]


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _dev_x(x_u16):
    return _dev(x_u16.view(np.int16)).view(torch.bfloat16)


def _gemv(kq, fmt, Wb, x, N, K):
    pad = 64
    ybuf = torch.full((N + 2 * pad,), CANARY, dtype=torch.float32, device="cuda")
    kq.kq_gemv(fmt, _dev(Wb), _dev_x(x), ybuf[pad:pad + N], N, K, 1)
    kq.kq_device_status()
    out = ybuf.cpu().numpy()
    assert np.all(out[:pad] == np.float32(CANARY)) and np.all(out[pad + N:] == np.float32(CANARY))
    return out[pad:pad + N].reshape(1, N)


def _gemv_t(kq, fmt, Wb, x, N, K):
    T = x.shape[0]
    pad = 64
    ybuf = torch.full((T * N + 2 * pad,), CANARY, dtype=torch.float32, device="cuda")
    kq.kq_gemv(fmt, _dev(Wb), _dev_x(x), ybuf[pad:pad + T * N], N, K, T)
    kq.kq_device_status()
    out = ybuf.cpu().numpy()
    assert np.all(out[:pad] == np.float32(CANARY)) and np.all(out[pad + T * N:] == np.float32(CANARY))
    return out[pad:pad + T * N].reshape(T, N)


def _assert_parity(y, yref, A, what):
    tol = 1e-3 * A + 1e-5
    err = np.abs(y.astype(np.float64) - yref)
    bad = ~(err <= tol)
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err / tol, 0)), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst at {i}: "
                             f"y={y[i]!r} ref={yref[i]!r} tol={tol[i]!r}")


@pytest.mark.parametrize("fmt", FMTS, ids=FMT_IDS)
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}x{c[1]}")
def test_single_token_large_matches_oracle(kq, oracle, fmt, case):
    N, K = case
    Wb = oracle.quantize(fmt, _weights_f32(N, K), N, K)
    x = wl.activations_bf16(wl.derive_seed(701, fmt, N), 1, K, heavy=True)
    yref, A = oracle.gemv(fmt, Wb, N, K, x)
    _assert_parity(_gemv(kq, fmt, Wb, x, N, K), yref, A, f"fmt={fmt} {N}x{K}")


@pytest.mark.parametrize("fmt", FMTS, ids=FMT_IDS)
def test_single_token_large_random_blocks(kq, oracle, fmt):
    N, K = 8300, 4352
    Wb = wl.random_block_bytes(wl.derive_seed(702, fmt), fmt, N * K // 256)
    x = wl.activations_bf16(wl.derive_seed(703, fmt), 1, K)
    yref, A = oracle.gemv(fmt, Wb, N, K, x)
    _assert_parity(_gemv(kq, fmt, Wb, x, N, K), yref, A, f"random fmt={fmt}")


@pytest.mark.parametrize("fmt", [0, 2], ids=["Q4_K", "Q6_K"])
def test_single_token_grouped_launch(kq, oracle, fmt):
    # two matrices in one launch (gate / up style); 9000 and 7001 rows: the
    # tiles of the first end mid-tile, the second has a ragged tail
    K = 2304
    Ns = [9000, 7001]
    x = wl.activations_bf16(wl.derive_seed(704, fmt), 1, K, heavy=True)
    Ws, ys, refs = [], [], []
    for j, N in enumerate(Ns):
        Wb = oracle.quantize(fmt, wl.weights_f32(wl.derive_seed(705, fmt, j), N, K), N, K)
        refs.append(oracle.gemv(fmt, Wb, N, K, x))
        Ws.append(_dev(Wb))
        ys.append(torch.full((1, N), CANARY, dtype=torch.float32, device="cuda"))
    kq.kq_gemv_multi(fmt, Ws, ys, Ns, _dev_x(x), K, 1)
    kq.kq_device_status()
    for j, (yref, A) in enumerate(refs):
        _assert_parity(ys[j].cpu().numpy(), yref, A, f"matrix {j}")


@pytest.mark.parametrize("fmt", [0, 2], ids=["Q4_K", "Q6_K"])
def test_single_token_repeated_launches_agree(kq, oracle, fmt):
    # the tile order differs run to run (tiles are claimed at run time); the
    # result must not: every tile's sum is formed in a fixed order
    N, K = 1100, 32768
    Wb = oracle.quantize(fmt, _weights_f32(N, K), N, K)
    x = wl.activations_bf16(wl.derive_seed(706), 1, K, heavy=True)
    W, xd = _dev(Wb), _dev_x(x)
    y0 = torch.empty((1, N), dtype=torch.float32, device="cuda")
    kq.kq_gemv(fmt, W, xd, y0, N, K, 1)
    for _ in range(5):
        y = torch.empty((1, N), dtype=torch.float32, device="cuda")
        kq.kq_gemv(fmt, W, xd, y, N, K, 1)
        assert torch.equal(y, y0)
    kq.kq_device_status()


@pytest.mark.parametrize("fmt", FMTS, ids=FMT_IDS)
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}x{c[1]}")
def test_verify_widths_large_match_oracle(kq, oracle, fmt, case):
    N, K = case
    Wb = oracle.quantize(fmt, _weights_f32(N, K), N, K)
    x = wl.activations_bf16(wl.derive_seed(707, fmt, N), 16, K, heavy=True)
    yref, A = oracle.gemv(fmt, Wb, N, K, x)
    for T in (2, 3, 4, 5, 8, 11, 16):
        _assert_parity(_gemv_t(kq, fmt, Wb, x[:T], N, K), yref[:T], A[:T], f"fmt={fmt} {N}x{K} n_tok={T}")


@pytest.mark.parametrize("fmt", [0, 3], ids=["Q4_K", "G128"])
def test_verify_width_random_blocks(kq, oracle, fmt):
    N, K = 20000, 2048
    Wb = wl.random_block_bytes(wl.derive_seed(708, fmt), fmt, N * K // 256)
    x = wl.activations_bf16(wl.derive_seed(709, fmt), 8, K)
    yref, A = oracle.gemv(fmt, Wb, N, K, x)
    _assert_parity(_gemv_t(kq, fmt, Wb, x, N, K), yref, A, f"random fmt={fmt}")


def test_verify_width_grouped_launch(kq, oracle):
    K, T = 2304, 8
    Ns = [9000, 7001]
    x = wl.activations_bf16(wl.derive_seed(710), T, K, heavy=True)
    Ws, ys, refs = [], [], []
    for j, N in enumerate(Ns):
        Wb = oracle.quantize(0, wl.weights_f32(wl.derive_seed(711, j), N, K), N, K)
        refs.append(oracle.gemv(0, Wb, N, K, x))
        Ws.append(_dev(Wb))
        ys.append(torch.full((T, N), CANARY, dtype=torch.float32, device="cuda"))
    kq.kq_gemv_multi(0, Ws, ys, Ns, _dev_x(x), K, T)
    kq.kq_device_status()
    for j, (yref, A) in enumerate(refs):
        _assert_parity(ys[j].cpu().numpy(), yref, A, f"matrix {j}")


@pytest.mark.parametrize("fmt", [0, 3], ids=["Q4_K", "G128"])
def test_single_token_five_columns_zero_weight_records(kq, oracle, fmt):
    # the five-column stages (K / 256 = 20), a ragged last tile, and records
    # of zero weights with nonzero scales, which must give exactly zero
    from test_exact_edges import PERIOD, ZERO_TYPES, degenerate_matrix
    N, K = 6600, 5120
    W = degenerate_matrix(oracle, fmt, N, K, 4400 + fmt)
    x = wl.activations_bf16(wl.derive_seed(4401, fmt), 1, K, heavy=True)
    yref, A = oracle.gemv(fmt, W, N, K, x)
    y = _gemv(kq, fmt, W, x, N, K)
    _assert_parity(y, yref, A, f"fmt={fmt} five columns")
    zero_rows = [r for r in range(N) if r % PERIOD in ZERO_TYPES]
    assert np.all(yref[0, zero_rows] == 0.0) and np.all(y[0, zero_rows] == 0.0)
