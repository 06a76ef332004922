"""The split-K exchange across launches and graph replays.

One CUDA graph holds a launch of every kernel that splits K (the
single-token tensor-core kernel, the streaming kernel, the multi-token
tensor-core kernel, the verify kernel).  Its inputs change between replays
and plain launches of the same shapes run in between, so a reader that took
a stale partial sum -- one left in the scratch by the previous replay or
launch (the streaming kernel's tagged partials: a graph replays its tag, the
reader clears every slot it reads) -- would return the previous input's
sums: every replay is checked against the oracle on its own input.  Two
replays of the same input give bit-identical outputs (the segments are added
in a fixed order, whichever arrives last).
"""
import numpy as np
import pytest

import workloads as wl
from test_gpu_parity import CANARY, assert_parity, dev, dev_x, weights

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

# (format, N, K, n_tok): the kernels that split K at these shapes
CASES = [(0, 8192, 4096, 1),     # single-token tensor-core kernel (Q4_K, >= 32 M weights)
         (2, 600, 32768, 1),     # streaming kernel, long rows
         (0, 8192, 4096, 8),     # multi-token tensor-core kernel
         (2, 1100, 32768, 8)]    # verify kernel (Q6_K)


@pytest.fixture(scope="module")
def kq():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from quant_weight_gemv_dequant_b300 import build
    build.build()
    import quant_weight_gemv_dequant_b300 as k
    k.lib()
    return k


def test_replays_with_changing_inputs(kq, oracle):
    mats = []
    for i, (fmt, N, K, T) in enumerate(CASES):
        Wb = weights(oracle, fmt, N, K, wl.derive_seed(700, i))
        xs = [wl.activations_bf16(wl.derive_seed(701, i, r), T, K) for r in range(3)]
        xd = dev_x(xs[0])
        y = torch.full((T, N), CANARY, dtype=torch.float32, device="cuda")
        mats.append((fmt, N, K, T, Wb, dev(Wb), xs, xd, y))
    s = torch.cuda.Stream()

    def launch_all(stream):
        for fmt, N, K, T, _, W, _, xd, y in mats:
            kq.kq_gemv(fmt, W, xd, y, N, K, T, stream)

    launch_all(s)   # first launches outside the capture (scratch sized)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        launch_all(s)
    first = None
    for r in range(3):
        for m in mats:
            m[7].copy_(dev_x(m[6][r]))
            m[8].fill_(CANARY)
        g.replay()
        torch.cuda.synchronize()
        assert kq.kq_device_status() == 0
        ys = [m[8].cpu().numpy().copy() for m in mats]
        for (fmt, N, K, T, Wb, _, xs, _, _), y in zip(mats, ys):
            yref, A = oracle.gemv(fmt, Wb, N, K, xs[r])
            assert_parity(y, yref, A, f"fmt {fmt} {N}x{K} n_tok {T}, replay {r}")
        if r == 0:
            first = ys
        # plain launches of the same shapes (their own tags) between replays
        launch_all(s)
        torch.cuda.synchronize()
        for m, y0 in zip(mats, first):
            if r == 0:
                assert np.array_equal(m[8].cpu().numpy(), y0), "plain launch differs from the replay"
    # the first input again: bit-identical to the first replay
    for m in mats:
        m[7].copy_(dev_x(m[6][0]))
    g.replay()
    torch.cuda.synchronize()
    for m, y0 in zip(mats, first):
        assert np.array_equal(m[8].cpu().numpy(), y0), "replay of the same input differs"
