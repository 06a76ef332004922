"""GPU parity of the SwiGLU chain: gate/up launch with the activation fused
into its epilogue (h = bf16(silu(gate) * up)), then the down projection on h.

References come from the oracle only: y_gate, y_up = the fp64 products,
h_exact = silu(y_gate) * y_up in fp64, h_or its bf16 rounding, y_down_ref =
the fp64 product of down with h_or.

Bounds (derived from the GEMV bar |y - y_ref| <= 1e-3 A + 1e-5 =: tol):
  * y_gate, y_up: tol each;
  * h: silu' lies in [-0.1, 1.1], so
      |h_gpu - h_exact| <= 1.1 tol_g (|u| + tol_u) + |silu(g)| tol_u + 2^-8 |h_exact| =: E
    (the last term: bf16 rounding, 2^-9 relative, plus the fp32 evaluation);
  * y_down: the GEMV bar on the GPU's own h, plus how far h_gpu may lie from
    h_or: with D = sum_k |w^_down| (E + |h_exact - h_or|),
      |y_down - y_down_ref| <= 1e-3 (A + D) + 1e-5 + D.
Shapes: the fused single-token tensor-core path (Q4_K 32768 x 5120 with K
split, the full-size feed-forward of the decode step; Q4_G128 8192 x 4096;
a ragged 8300-feature launch without the chain) and launches that run the
grouped GEMV plus the elementwise kernel (small, 3 tokens, Q5_K).
"""
import numpy as np
import pytest

import workloads as wl

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
CANARY = 1234.5


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


def _bf16_to_f64(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _silu(v):
    return v / (1.0 + np.exp(-v))


def _h_bound(g, u, Ag, Au, h_exact):
    tg, tu = 1e-3 * Ag + 1e-5, 1e-3 * Au + 1e-5
    return 1.1 * tg * (np.abs(u) + tu) + np.abs(_silu(g)) * tu + 2.0 ** -8 * np.abs(h_exact)


def _weights(oracle, fmt, N, K, seed, pools=None):
    if fmt == 3:
        w = wl.weights_f32(wl.derive_seed(seed), N, K)
        return oracle.quantize(3, w, N, K)
    if pools is not None and N * K >= (1 << 26):
        return wl.tiled_rows(pools[fmt], fmt, wl.derive_seed(seed), N, K, np.arange(N))
    return oracle.quantize(fmt, wl.weights_f32(wl.derive_seed(seed), N, K), N, K)


@pytest.fixture(scope="module")
def pools(oracle):
    pw = wl.pool_weights(wl.derive_seed(900), wl.POOL_BLOCKS)
    return {f: oracle.quantize(f, pw, wl.POOL_BLOCKS, 256) for f in (0, 1, 2)}


# (format, N (features), K, n_tok, with the down projection)
CASES = [(0, 32768, 5120, 1, True), (3, 8192, 4096, 1, True), (0, 8300, 2048, 1, False),
         (0, 1024, 1024, 1, True), (0, 8192, 4096, 3, True), (1, 4096, 2048, 1, True)]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"f{c[0]}_{c[1]}x{c[2]}_t{c[3]}")
def test_swiglu_chain_matches_oracle(kq, oracle, pools, case):
    fmt, N, K, T, chain = case
    Wg = _weights(oracle, fmt, N, K, 530 + fmt, pools)
    Wu = _weights(oracle, fmt, N, K, 540 + fmt, pools)
    x = wl.activations_bf16(wl.derive_seed(550, N, K), T, K, heavy=True)
    g_ref, Ag = oracle.gemv(fmt, Wg, N, K, x)
    u_ref, Au = oracle.gemv(fmt, Wu, N, K, x)
    h_exact, h_or = oracle.swiglu(g_ref, u_ref)
    xd = _dev(x.view(np.int16)).view(torch.bfloat16)
    yg = torch.full((T, N), CANARY, dtype=torch.float32, device="cuda")
    yu = torch.full((T, N), CANARY, dtype=torch.float32, device="cuda")
    h = torch.full((T, N), 7, dtype=torch.int16, device="cuda")
    if chain:
        Kd, Nd = N, 5120
        Wd = _weights(oracle, 2, Nd, Kd, 560, pools)
        yd = torch.full((T, Nd), CANARY, dtype=torch.float32, device="cuda")
        Wgd, Wud, Wdd = _dev(Wg), _dev(Wu), _dev(Wd)   # kq_matrix holds only their addresses
        gate = kq.make_matrix(fmt, Wgd, N, K)
        up = kq.make_matrix(fmt, Wud, N, K)
        down = kq.make_matrix(2, Wdd, Nd, Kd)
        kq.kq_ffn_swiglu(gate, up, down, xd, yg, yu, h, yd, T)
    else:
        Wgd, Wud = _dev(Wg), _dev(Wu)
        kq.kq_gemv_swiglu(fmt, Wgd, Wud, xd, yg, yu, h, N, K, T)
    assert kq.kq_device_status() == 0
    got_g = yg.cpu().numpy().astype(np.float64)
    got_u = yu.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got_g - g_ref) <= 1e-3 * Ag + 1e-5), "y_gate"
    assert np.all(np.abs(got_u - u_ref) <= 1e-3 * Au + 1e-5), "y_up"
    got_h = _bf16_to_f64(h.cpu().numpy().view(np.uint16))
    E = _h_bound(g_ref, u_ref, Ag, Au, h_exact)
    bad = ~(np.abs(got_h - h_exact) <= E)
    assert not bad.any(), (f"h: {bad.sum()} outside; worst {np.max(np.abs(got_h - h_exact) / E)} of the bound")
    if chain:
        rows = np.unique(np.concatenate([[0, Nd - 1], (wl.splitmix64(561, np.arange(64, dtype=np.uint64))
                                                      % np.uint64(Nd)).astype(np.int64)]))
        yd_ref, Ad = oracle.gemv_rows(2, Wd, Nd, Kd, rows, h_or.reshape(T, Kd))
        got_d = yd.cpu().numpy()[:, rows].astype(np.float64)
        for t in range(T):
            D = oracle.gemv_absw(2, Wd, Nd, Kd, E[t] + np.abs(h_exact[t] - _bf16_to_f64(h_or[t])))[rows]
            tol = 1e-3 * (Ad[t] + D) + 1e-5 + D
            assert np.all(np.abs(got_d[t] - yd_ref[t]) <= tol), f"y_down token {t}"


def test_swiglu_rejects_bad_arguments(kq):
    W = torch.zeros(64 * 4 * 144, dtype=torch.uint8, device="cuda")
    x = torch.zeros((1, 1024), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((1, 64), dtype=torch.float32, device="cuda")
    hbuf = torch.zeros(80, dtype=torch.int16, device="cuda")
    assert kq.kq_gemv_swiglu(0, W, W, x, y, y, 0, 64, 1024, 1, check=False) == 1       # null h
    assert kq.kq_gemv_swiglu(0, W, W, x, y, y, hbuf.data_ptr() + 2, 64, 1024, 1, check=False) == 3
    assert kq.kq_gemv_swiglu(0, W, W, x, y, y, hbuf, 64, 1000, 1, check=False) == 2    # K % 256
