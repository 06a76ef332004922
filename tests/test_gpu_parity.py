"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Bar: |y - y_ref| <= 1e-3 * sum_k |w^ x| + 1e-5 per element (y_ref and the
sum from the oracle); kq_dequantize bit-exact against the oracle's exact
value rounded to fp32.  Inputs come from the seeded generators and the
oracle's quantiser only.
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


def dev(a: np.ndarray):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def dev_x(x_u16: np.ndarray):
    return dev(x_u16.view(np.int16)).view(torch.bfloat16)


def gpu_gemv(kq, fmt, Wb, x_u16, N, K):
    """Run kq_gemv with canaries around y; return y as numpy [T][N]."""
    T = x_u16.shape[0]
    pad = 64
    ybuf = torch.full((T * N + 2 * pad,), CANARY, dtype=torch.float32, device="cuda")
    y = ybuf[pad:pad + T * N]
    kq.kq_gemv(fmt, dev(Wb), dev_x(x_u16), y, N, K, T)
    kq.kq_device_status()
    out = ybuf.cpu().numpy()
    assert np.all(out[:pad] == np.float32(CANARY)) and np.all(out[pad + T * N:] == np.float32(CANARY))
    return out[pad:pad + T * N].reshape(T, N)


def assert_parity(y, yref, A, what=""):
    tol = 1e-3 * A + 1e-5
    err = np.abs(y.astype(np.float64) - yref)
    bad = ~(err <= tol)
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err / tol, 0)), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst at {i}: "
                             f"y={y[i]!r} ref={yref[i]!r} tol={tol[i]!r}")


def weights(oracle, fmt, N, K, seed, kind="quant"):
    if kind == "random":
        return wl.random_block_bytes(seed, fmt, N * K // 256)
    return oracle.quantize(fmt, wl.weights_f32(seed, N, K), N, K)


SHAPES = [(1, 256), (3, 256), (8, 512), (37, 768), (130, 2304), (64, 5120), (9, 4096)]
NTOKS = [1, 2, 3, 4, 5, 8, 11, 16]


@pytest.mark.parametrize("fmt", [0, 1, 2, 3], ids=["Q4_K", "Q5_K", "Q6_K", "G128"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s[0]}x{s[1]}")
def test_gemv_small_shapes_all_ntok(kq, oracle, fmt, shape):
    N, K = shape
    for kind in ("quant", "random"):
        Wb = weights(oracle, fmt, N, K, wl.derive_seed(100, fmt, N, K), kind)
        x = wl.activations_bf16(wl.derive_seed(101, N, K), 16, K, heavy=(kind == "quant"))
        yref, A = oracle.gemv(fmt, Wb, N, K, x)
        for T in NTOKS:
            y = gpu_gemv(kq, fmt, Wb, x[:T], N, K)
            assert_parity(y, yref[:T], A[:T], f"{kind} fmt={fmt} {N}x{K} n_tok={T}")


@pytest.mark.parametrize("fmt", [0, 1, 2, 3], ids=["Q4_K", "Q5_K", "Q6_K", "G128"])
def test_gemv_many_tiles_ragged_tail(kq, oracle, fmt):
    N, K = 1003, 4352          # several row tiles + ragged tail; K/256 = 17 (odd)
    Wb = weights(oracle, fmt, N, K, wl.derive_seed(102, fmt))
    x = wl.activations_bf16(wl.derive_seed(103), 16, K)
    yref, A = oracle.gemv(fmt, Wb, N, K, x)
    for T in (1, 2, 4, 8, 16):
        assert_parity(gpu_gemv(kq, fmt, Wb, x[:T], N, K), yref[:T], A[:T], f"n_tok={T}")


def test_gemv_long_rows(kq, oracle):
    # the largest K on the path (down projection) and beyond; at K = 98304 a
    # one-token small launch's warp slice (16 super-blocks) is wider than one
    # tensor copy's box, so its rows are copied one by one;
    # K = 31744 (31 slabs of four super-blocks: no even split) takes K
    # segments whose last one is shorter
    for fmt, K in ((2, 32768), (0, 65536), (0, 98304), (2, 31744), (1, 31744)):
        N = 5
        Wb = weights(oracle, fmt, N, K, wl.derive_seed(104, fmt))
        x = wl.activations_bf16(wl.derive_seed(105), 4, K, heavy=True)
        yref, A = oracle.gemv(fmt, Wb, N, K, x)
        for T in (1, 2, 4):
            assert_parity(gpu_gemv(kq, fmt, Wb, x[:T], N, K), yref[:T], A[:T],
                          f"fmt={fmt} K={K} n_tok={T}")


@pytest.mark.parametrize("fmt", [0, 1, 2, 3], ids=["Q4_K", "Q5_K", "Q6_K", "G128"])
def test_dequantize_bit_exact(kq, oracle, fmt):
    for kind, N, K in (("random", 7, 768), ("quant", 33, 1024), ("random", 1, 256)):
        Wb = weights(oracle, fmt, N, K, wl.derive_seed(106, fmt, N), kind)
        ref = oracle.dequantize(fmt, Wb, N, K).astype(np.float32)
        pad = 32
        buf = torch.full((N * K + 2 * pad,), CANARY, dtype=torch.float32, device="cuda")
        kq.kq_dequantize(fmt, dev(Wb), buf[pad:pad + N * K], N, K)
        torch.cuda.synchronize()
        out = buf.cpu().numpy()
        assert np.all(out[:pad] == np.float32(CANARY)) and np.all(out[-pad:] == np.float32(CANARY))
        got = out[pad:pad + N * K].reshape(N, K)
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), f"{kind} {N}x{K}"


def test_merged_g128_matches_q4k_on_gpu(kq, oracle):
    N, K = 96, 1536
    w = wl.weights_f32(wl.derive_seed(107), N, K)
    q4 = oracle.quantize_q4k_group128(w, N, K)
    st, g = kq.kq_merge_g128(q4, N, K)
    assert st == 0
    x = wl.activations_bf16(wl.derive_seed(108), 4, K)
    yref, A = oracle.gemv(oracle.Q4_K, q4, N, K, x)
    yq = gpu_gemv(kq, 0, q4, x, N, K)
    yg = gpu_gemv(kq, 3, g, x, N, K)
    assert_parity(yq, yref, A, "Q4_K")
    assert_parity(yg, yref, A, "G128")


def _small_layer(oracle, seed, fmts):
    # k and v have 130 rows (not a multiple of any tile) and share a launch
    # with q when their formats agree.
    shapes = {"q": (256, 512), "k": (130, 512), "v": (130, 512), "o": (512, 256),
              "gate": (776, 512), "up": (776, 512), "down": (512, 768)}
    return {n: (fmts[n], weights(oracle, fmts[n], N, K, wl.derive_seed(seed, i)), N, K)
            for i, (n, (N, K)) in enumerate(shapes.items())}


@pytest.mark.parametrize("mix", ["uniform", "mixed"])
def test_layer_step_parity(kq, oracle, mix):
    from quant_weight_gemv_dequant_b300.decode_step import DecodeStep, LAYER_NAMES, X_OF
    if mix == "uniform":
        fmts = dict(q=0, k=0, v=0, o=0, gate=0, up=0, down=2)
    else:
        fmts = dict(q=0, k=1, v=0, o=3, gate=1, up=2, down=2)
    host = _small_layer(oracle, 110 + (mix == "mixed"), fmts)
    T = 5
    layers = [{n: (f, dev(W), N, K) for n, (f, W, N, K) in host.items()}]
    step = DecodeStep(layers, None, T)
    xs = {}
    for i, key in enumerate(("x_attn", "x_o", "x_ffn", "x_down")):
        K = {"x_attn": host["q"][3], "x_o": host["o"][3], "x_ffn": host["gate"][3],
             "x_down": host["down"][3]}[key]
        xs[key] = wl.activations_bf16(wl.derive_seed(112, i), T, K)
        step.x[0][key].copy_(dev_x(xs[key]))
    step.run()
    torch.cuda.synchronize()
    for n in LAYER_NAMES:
        f, W, N, K = host[n]
        yref, A = oracle.gemv(f, W, N, K, xs[X_OF[n]])
        assert_parity(step.y[0][n].cpu().numpy(), yref, A, f"{mix} {n}")


def test_graph_capture_replay(kq, oracle):
    N, K, T = 300, 2048, 3
    Wb = weights(oracle, 0, N, K, wl.derive_seed(113))
    x = wl.activations_bf16(wl.derive_seed(114), T, K)
    W, xd = dev(Wb), dev_x(x)
    y = torch.empty((T, N), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    kq.kq_gemv(0, W, xd, y, N, K, T, s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        kq.kq_gemv(0, W, xd, y, N, K, T, s)
    y.fill_(CANARY)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    yref, A = oracle.gemv(0, Wb, N, K, x)
    assert_parity(y.cpu().numpy(), yref, A, "graph replay")


# ------------------------------------------------------- full-size workloads

@pytest.fixture(scope="module")
def pools(oracle):
    """Oracle-quantised pools of N(0, 0.02) super-blocks, per format."""
    pw = wl.pool_weights(wl.derive_seed(900), wl.POOL_BLOCKS)
    return {f: oracle.quantize(f, pw, wl.POOL_BLOCKS, 256) for f in (0, 1, 2)}


def test_single_q4k_4096(kq, oracle):
    m = wl.SINGLE_Q4K[0]
    Wb = weights(oracle, m.fmt, m.N, m.K, wl.derive_seed(1, 0))
    x = wl.activations_bf16(wl.derive_seed(1, 100), 8, m.K)
    yref, A = oracle.gemv(m.fmt, Wb, m.N, m.K, x)
    for T in (1, 8):
        assert_parity(gpu_gemv(kq, m.fmt, Wb, x[:T], m.N, m.K), yref[:T], A[:T], f"n_tok={T}")


def test_attention_projections_and_g128(kq, oracle):
    x = wl.activations_bf16(wl.derive_seed(2, 100), 1, wl.HIDDEN)
    xo = wl.activations_bf16(wl.derive_seed(2, 101), 1, 4096)
    for i, m in enumerate(wl.ATTN_Q4K[:4]):
        w = wl.weights_f32(wl.derive_seed(2, i), m.N, m.K)
        Wb = oracle.quantize_q4k_group128(w, m.N, m.K) if m.name == "q" else oracle.quantize(m.fmt, w, m.N, m.K)
        xi = xo if m.name == "o" else x
        yref, A = oracle.gemv(m.fmt, Wb, m.N, m.K, xi)
        y = gpu_gemv(kq, m.fmt, Wb, xi, m.N, m.K)
        assert_parity(y, yref, A, m.name)
        if m.name == "q":                      # the same q weights, merged
            st, g = kq.kq_merge_g128(Wb, m.N, m.K)
            assert st == 0
            assert_parity(gpu_gemv(kq, 3, g, xi, m.N, m.K), yref, A, "q_g128")


def _sample_rows(N, n, seed):
    r = wl.splitmix64(seed, np.arange(n, dtype=np.uint64)) % np.uint64(N)
    return np.unique(np.concatenate([[0, N - 1], r.astype(np.int64)]))


def test_ffn_layer_heavy_tailed(kq, oracle, pools):
    x = wl.activations_bf16(wl.derive_seed(3, 100), 1, wl.HIDDEN, heavy=True)
    xd = wl.activations_bf16(wl.derive_seed(3, 101), 1, wl.INTER, heavy=True)
    P = torch.device("cuda")
    for i, m in enumerate(wl.FFN_Q4K_Q6K):
        seed = wl.derive_seed(3, i)
        W = wl.tile_matrix_device(dev(pools[m.fmt]), m.fmt, seed, m.N, m.K)
        xi = xd if m.name == "down" else x
        y = torch.empty((1, m.N), dtype=torch.float32, device=P)
        kq.kq_gemv(m.fmt, W, dev_x(xi), y, m.N, m.K, 1)
        rows = _sample_rows(m.N, 256, seed)
        sub = wl.tiled_rows(pools[m.fmt], m.fmt, seed, m.N, m.K, rows)
        yref, A = oracle.gemv(m.fmt, sub, len(rows), m.K, xi)
        assert_parity(y.cpu().numpy()[:, rows], yref, A, m.name)


def test_q5k_layer_verify_sweep(kq, oracle, pools):
    P = torch.device("cuda")
    for i, m in enumerate(wl.LAYER_Q5K):
        seed = wl.derive_seed(4, i)
        W = wl.tile_matrix_device(dev(pools[m.fmt]), m.fmt, seed, m.N, m.K)
        x = wl.activations_bf16(wl.derive_seed(4, 100 + i), 16, m.K)
        rows = _sample_rows(m.N, 64, seed)
        sub = wl.tiled_rows(pools[m.fmt], m.fmt, seed, m.N, m.K, rows)
        yref, A = oracle.gemv(m.fmt, sub, len(rows), m.K, x)
        for T in (1, 2, 4, 8, 16):
            y = torch.empty((T, m.N), dtype=torch.float32, device=P)
            kq.kq_gemv(m.fmt, W, dev_x(x[:T]), y, m.N, m.K, T)
            assert_parity(y.cpu().numpy()[:, rows], yref[:T], A[:T], f"{m.name} n_tok={T}")


@pytest.mark.parametrize("n_tok", [1, 8])
def test_whole_decode_step_graph(kq, oracle, pools, n_tok):
    """The 52-layer step + LM head, in the CUDA-graph launch the benchmark
    times; layer 0 and the LM head checked on every row (n_tok = 1) or on
    sampled rows, every other matrix on sampled rows."""
    from quant_weight_gemv_dequant_b300.decode_step import DecodeStep, LAYER_NAMES, X_OF
    pdev = {f: dev(p) for f, p in pools.items()}
    layers, seeds = [], []
    for l in range(wl.LAYERS):
        L = {}
        for i, m in enumerate(wl.DECODE_LAYER):
            seed = wl.derive_seed(5, l, i)
            L[m.name] = (m.fmt, wl.tile_matrix_device(pdev[m.fmt], m.fmt, seed, m.N, m.K), m.N, m.K)
        layers.append(L)
    hs = wl.derive_seed(5, 999)
    h = wl.LM_HEAD
    head = (h.fmt, wl.tile_matrix_device(pdev[h.fmt], h.fmt, hs, h.N, h.K), h.N, h.K)
    step = DecodeStep(layers, head, n_tok)
    xs = []
    for l in range(wl.LAYERS):
        d = {}
        for j, key in enumerate(("x_attn", "x_o", "x_ffn", "x_down")):
            K = step.x[l][key].shape[1]
            d[key] = wl.activations_bf16(wl.derive_seed(5, l, 100 + j), n_tok, K)
            step.x[l][key].copy_(dev_x(d[key]))
        xs.append(d)
    xh = wl.activations_bf16(wl.derive_seed(5, 998), n_tok, h.K)
    step.x_head.copy_(dev_x(xh))
    step.capture()
    for y in [step.y_head] + [t for ys in step.y for t in ys.values()]:
        y.fill_(CANARY)
    step.replay()
    torch.cuda.synchronize()
    for l in (0, 1, 25, 51):
        for i, m in enumerate(wl.DECODE_LAYER):
            seed = wl.derive_seed(5, l, i)
            nrow = m.N if (l == 0 and n_tok == 1) else 48
            rows = np.arange(m.N) if nrow == m.N else _sample_rows(m.N, nrow, seed)
            sub = wl.tiled_rows(pools[m.fmt], m.fmt, seed, m.N, m.K, rows)
            yref, A = oracle.gemv(m.fmt, sub, len(rows), m.K, xs[l][X_OF[m.name]])
            assert_parity(step.y[l][m.name].cpu().numpy()[:, rows], yref, A, f"layer {l} {m.name}")
    rows = np.arange(0, h.N, 1 if n_tok == 1 else 97)
    sub = wl.tiled_rows(pools[h.fmt], h.fmt, hs, h.N, h.K, rows)
    yref, A = oracle.gemv(h.fmt, sub, len(rows), h.K, xh)
    assert_parity(step.y_head.cpu().numpy()[:, rows], yref, A, "lm_head")


def test_graph_survives_scratch_growth(kq, oracle, pools):
    """A captured launch that splits K keeps its split-K scratch: after a
    later, larger split-K request makes the library allocate a bigger
    buffer, replaying the earlier graph still gives the right result."""
    fmt, N, K, T = 2, 600, 32768, 1
    Wb = weights(oracle, fmt, N, K, wl.derive_seed(131))
    x = wl.activations_bf16(wl.derive_seed(132), T, K)
    W, xd = dev(Wb), dev_x(x)
    y = torch.empty((T, N), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    kq.kq_gemv(fmt, W, xd, y, N, K, T, s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        kq.kq_gemv(fmt, W, xd, y, N, K, T, s)
    # 20000 x 32768 Q6_K at 16 tokens: about 20 MB of partial sums, more than
    # the scratch held so far
    Nb, Tb, sb = 20000, 16, wl.derive_seed(133)
    big = wl.tile_matrix_device(dev(pools[fmt]), fmt, sb, Nb, K)
    xb = wl.activations_bf16(wl.derive_seed(134), Tb, K)
    yb = torch.full((Tb, Nb), CANARY, dtype=torch.float32, device="cuda")
    kq.kq_gemv(fmt, big, dev_x(xb), yb, Nb, K, Tb, s)
    torch.cuda.synchronize()
    y.fill_(CANARY)
    g.replay()
    torch.cuda.synchronize()
    assert kq.kq_device_status() == 0
    yref, A = oracle.gemv(fmt, Wb, N, K, x)
    assert_parity(y.cpu().numpy(), yref, A, "graph replay after scratch growth")
    rows = _sample_rows(Nb, 16, sb)
    sub = wl.tiled_rows(pools[fmt], fmt, sb, Nb, K, rows)
    yref, A = oracle.gemv(fmt, sub, len(rows), K, xb)
    assert_parity(yb.cpu().numpy()[:, rows], yref, A, "large split-K request")


@pytest.mark.parametrize("fmt", [0, 1, 2, 3], ids=["Q4_K", "Q5_K", "Q6_K", "G128"])
def test_degenerate_rows_and_tokens(kq, oracle, fmt):
    """Degenerate cases of the method through every kernel: rows that are all
    zero (d = dmin = 0), constant (one sub-block value, the scale term zero),
    a million times smaller than the rest, a single spike, and rows whose
    sub-blocks alternate between zero and constant; a token of all-zero x
    among heavy-tailed ones.  8300 x 4352 (36 M weights) takes the
    tensor-core kernels for Q4_K / Q4_G128 at n_tok 1 and 8, the streaming
    kernel at 2, gemv_mma for Q5_K / Q6_K at 8."""
    N, K = 8300, 4352
    w = wl.weights_f32(wl.derive_seed(120, fmt), N, K)
    w[0] = 0.0
    w[1] = 0.5
    w[2] = -0.125
    w[3] *= 1e-6
    w[4] = 0.0
    w[4, 1234] = 3.0
    for j in range(0, K, 64):
        w[5, j:j + 32] = 0.0
        w[5, j + 32:j + 64] = 0.03
    w[N - 1] = 0.0
    Wb = oracle.quantize(fmt, w, N, K)
    x = wl.activations_bf16(wl.derive_seed(121, fmt), 8, K, heavy=True)
    x[1] = 0
    yref, A = oracle.gemv(fmt, Wb, N, K, x)
    for T in (1, 2, 8):
        y = gpu_gemv(kq, fmt, Wb, x[:T], N, K)
        assert_parity(y, yref[:T], A[:T], f"fmt={fmt} n_tok={T}")
        assert np.all(y[:, 0] == 0.0) and np.all(y[:, N - 1] == 0.0)   # zero rows give exact zeros
        if T > 1:
            assert np.all(y[1] == 0.0)                                  # so does a zero token


def test_decode_step_graph_copies_host_inputs(kq, oracle, pools):
    """DecodeStep.capture(host_x=...): the graph copies the step's inputs
    from pinned host memory, layer by layer on a second stream, and each
    layer waits for its own inputs.  Three layers and the LM head; the host
    inputs change between replays, and each replay's outputs match the
    oracle on that replay's inputs (a layer that ran before its copy landed
    would use the previous inputs)."""
    from quant_weight_gemv_dequant_b300.decode_step import DecodeStep, X_OF
    nl = 3
    pdev = {f: dev(p) for f, p in pools.items()}
    layers = []
    for l in range(nl):
        L = {}
        for i, m in enumerate(wl.DECODE_LAYER):
            seed = wl.derive_seed(6, l, i)
            L[m.name] = (m.fmt, wl.tile_matrix_device(pdev[m.fmt], m.fmt, seed, m.N, m.K), m.N, m.K)
        layers.append(L)
    h = wl.LM_HEAD
    hs = wl.derive_seed(6, 999)
    head = (h.fmt, wl.tile_matrix_device(pdev[h.fmt], h.fmt, hs, h.N, h.K), h.N, h.K)
    step = DecodeStep(layers, head, 1)
    host_x = torch.empty(step.x_all.shape, dtype=torch.bfloat16).pin_memory()
    step.capture(host_x=host_x)
    for r in range(2):
        parts, xs = [], []
        for l in range(nl):
            d = {}
            for j, key in enumerate(("x_attn", "x_o", "x_ffn", "x_down")):
                d[key] = wl.activations_bf16(wl.derive_seed(6, r, l, j), 1, step.x[l][key].shape[1])
                parts.append(d[key].reshape(-1))
            xs.append(d)
        xh = wl.activations_bf16(wl.derive_seed(6, r, 998), 1, h.K)
        parts.append(xh.reshape(-1))
        host_x.copy_(torch.from_numpy(np.concatenate(parts).view(np.int16)).view(torch.bfloat16))
        for y in [step.y_head] + [t for ys in step.y for t in ys.values()]:
            y.fill_(CANARY)
        step.replay()
        torch.cuda.synchronize()
        for l in range(nl):
            for i, m in enumerate(wl.DECODE_LAYER):
                seed = wl.derive_seed(6, l, i)
                rows = _sample_rows(m.N, 32, seed)
                sub = wl.tiled_rows(pools[m.fmt], m.fmt, seed, m.N, m.K, rows)
                yref, A = oracle.gemv(m.fmt, sub, len(rows), m.K, xs[l][X_OF[m.name]])
                assert_parity(step.y[l][m.name].cpu().numpy()[:, rows], yref, A,
                              f"replay {r} layer {l} {m.name}")
        rows = _sample_rows(h.N, 64, hs)
        sub = wl.tiled_rows(pools[h.fmt], h.fmt, hs, h.N, h.K, rows)
        yref, A = oracle.gemv(h.fmt, sub, len(rows), h.K, xh)
        assert_parity(step.y_head.cpu().numpy()[:, rows], yref, A, f"replay {r} lm_head")
