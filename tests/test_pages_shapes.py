"""GPU parity of the pages' own model shapes: the 52-layer decode step at
hidden 6656, SwiGLU intermediate 19968 and vocab 202048, with q, k, v and the
attention's sigmoid output gate (all reading the pre-attention hidden state)
in one launch of four matrices -- the qkvg fold of the Core AI card's
architecture section.  Q4_K attention and gate/up, Q6_K down and LM head, as
in the benchmark step; K = 6656 and 19968 are not powers of two, and the
Q6_K rows (5460 and 16380 bytes) are off the 16-byte grid.

The step runs as the CUDA graph the benchmark times, at one token and at
eight.  Layer 0 is checked on every row at one token, layers 1, 25 and 51 and
the LM head on sampled rows, against the oracle (|y - y_ref| <= 1e-3 A +
1e-5).  The fused SwiGLU chain runs on the same weights at one token.
"""
import numpy as np
import pytest

import workloads as wl

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
CANARY = 1234.5678


@pytest.fixture(scope="module")
def kq():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from quant_weight_gemv_dequant_b300 import build
    build.build()
    import quant_weight_gemv_dequant_b300 as k
    k.lib()
    return k


@pytest.fixture(scope="module")
def pools(oracle):
    pw = wl.pool_weights(wl.derive_seed(900), wl.POOL_BLOCKS)
    return {f: oracle.quantize(f, pw, wl.POOL_BLOCKS, 256) for f in (0, 2)}


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _sample_rows(N, n, seed):
    r = wl.splitmix64(seed, np.arange(n, dtype=np.uint64)) % np.uint64(N)
    return np.unique(np.concatenate([[0, N - 1], r.astype(np.int64)]))


def _assert_parity(y, yref, A, what):
    tol = 1e-3 * A + 1e-5
    err = np.abs(y.astype(np.float64) - yref)
    bad = ~(err <= tol)
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err / tol, 0)), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside; worst {i}: "
                             f"y={y[i]!r} ref={yref[i]!r} tol={tol[i]!r}")


@pytest.fixture(scope="module")
def weights(pools):
    pdev = {f: _dev(p) for f, p in pools.items()}
    layers = []
    for l in range(wl.LAYERS):
        L = {}
        for i, m in enumerate(wl.GLIMMER_LAYER):
            L[m.name] = (m.fmt, wl.tile_matrix_device(pdev[m.fmt], m.fmt, wl.derive_seed(8, l, i), m.N, m.K),
                         m.N, m.K)
        layers.append(L)
    h = wl.GLIMMER_HEAD
    head = (h.fmt, wl.tile_matrix_device(pdev[h.fmt], h.fmt, wl.derive_seed(8, 999), h.N, h.K), h.N, h.K)
    return layers, head


@pytest.mark.parametrize("n_tok", [1, 8])
def test_pages_shape_step_graph(kq, oracle, pools, weights, n_tok):
    from quant_weight_gemv_dequant_b300.decode_step import DecodeStep, X_OF
    layers, head = weights
    step = DecodeStep(layers, head, n_tok)
    assert step.launches() == wl.LAYERS * 4 + 1          # q/k/v/attn_gate, o, gate/up, down; head
    xs = []
    for l in range(wl.LAYERS):
        d = {}
        for j, key in enumerate(("x_attn", "x_o", "x_ffn", "x_down")):
            d[key] = wl.activations_bf16(wl.derive_seed(8, l, 100 + j), n_tok, step.x[l][key].shape[1])
            step.x[l][key].copy_(_dev(d[key].view(np.int16)).view(torch.bfloat16))
        xs.append(d)
    h = wl.GLIMMER_HEAD
    xh = wl.activations_bf16(wl.derive_seed(8, 998), n_tok, h.K)
    step.x_head.copy_(_dev(xh.view(np.int16)).view(torch.bfloat16))
    step.capture()
    for y in [step.y_head] + [t for ys in step.y for t in ys.values()]:
        y.fill_(CANARY)
    step.replay()
    torch.cuda.synchronize()
    assert kq.kq_device_status() == 0
    for l in (0, 1, 25, 51):
        for i, m in enumerate(wl.GLIMMER_LAYER):
            seed = wl.derive_seed(8, l, i)
            full = l == 0 and n_tok == 1
            rows = np.arange(m.N) if full else _sample_rows(m.N, 48, seed)
            sub = wl.tiled_rows(pools[m.fmt], m.fmt, seed, m.N, m.K, rows)
            yref, A = oracle.gemv(m.fmt, sub, len(rows), m.K, xs[l][X_OF[m.name]])
            _assert_parity(step.y[l][m.name].cpu().numpy()[:, rows], yref, A, f"layer {l} {m.name}")
    rows = _sample_rows(h.N, 400 if n_tok == 1 else 64, 8)
    sub = wl.tiled_rows(pools[h.fmt], h.fmt, wl.derive_seed(8, 999), h.N, h.K, rows)
    yref, A = oracle.gemv(h.fmt, sub, len(rows), h.K, xh)
    _assert_parity(step.y_head.cpu().numpy()[:, rows], yref, A, "lm_head")


def test_pages_shape_fused_ffn_layer(kq, oracle, pools, weights):
    # the fused SwiGLU chain on layer 0's feed-forward weights at one token:
    # y_gate / y_up at the bar, and down's output against the oracle's chain
    # (bound derived in test_swiglu.py)
    from quant_weight_gemv_dequant_b300.decode_step import DecodeStep
    layers, _ = weights
    step = DecodeStep(layers[:1], None, 1, fused_ffn=True)
    x = {}
    for j, key in enumerate(("x_attn", "x_o", "x_ffn", "x_down")):
        x[key] = wl.activations_bf16(wl.derive_seed(8, 0, 100 + j), 1, step.x[0][key].shape[1])
        step.x[0][key].copy_(_dev(x[key].view(np.int16)).view(torch.bfloat16))
    step.run()
    torch.cuda.synchronize()
    assert kq.kq_device_status() == 0
    by = {m.name: (i, m) for i, m in enumerate(wl.GLIMMER_LAYER)}
    host = {}
    for n in ("gate", "up", "down"):
        i, m = by[n]
        host[n] = wl.tiled_rows(pools[m.fmt], m.fmt, wl.derive_seed(8, 0, i), m.N, m.K, np.arange(m.N))
    G, U, D = by["gate"][1], by["up"][1], by["down"][1]
    g_ref, Ag = oracle.gemv(G.fmt, host["gate"], G.N, G.K, x["x_ffn"])
    u_ref, Au = oracle.gemv(U.fmt, host["up"], U.N, U.K, x["x_ffn"])
    _assert_parity(step.y[0]["gate"].cpu().numpy(), g_ref, Ag, "gate")
    _assert_parity(step.y[0]["up"].cpu().numpy(), u_ref, Au, "up")
    h_exact, h_or = oracle.swiglu(g_ref, u_ref)
    tg, tu = 1e-3 * Ag + 1e-5, 1e-3 * Au + 1e-5
    E = 1.1 * tg * (np.abs(u_ref) + tu) + np.abs(g_ref / (1 + np.exp(-g_ref))) * tu + 2.0 ** -8 * np.abs(h_exact)
    got_h = (step.h[0].view(torch.int16).cpu().numpy().view(np.uint16).astype(np.uint32) << 16) \
        .view(np.float32).astype(np.float64)
    assert np.all(np.abs(got_h - h_exact) <= E), "h"
    rows = _sample_rows(D.N, 64, 9)
    yd_ref, Ad = oracle.gemv_rows(D.fmt, host["down"], D.N, D.K, rows, h_or)
    h_or_f = (h_or.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    Dn = oracle.gemv_absw(D.fmt, host["down"], D.N, D.K, E[0] + np.abs(h_exact[0] - h_or_f[0]))[rows]
    tol = 1e-3 * (Ad[0] + Dn) + 1e-5 + Dn
    got_d = step.y[0]["down"].cpu().numpy()[0, rows].astype(np.float64)
    assert np.all(np.abs(got_d - yd_ref[0]) <= tol), "down after the fused activation"
