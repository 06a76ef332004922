"""kq_gemv_noalloc: the GEMV entry point that never allocates device memory.

Some callers cannot call cudaMalloc when they run the GEMV: code inside a
CUDA-graph stream capture, engines that own all device memory through their
own pool, latency-critical loops that cannot take an allocation's implicit
synchronisation.  For them kq_gemv_noalloc keeps the split-K scratch in a
fixed array inside the library.  These tests call it through the C ABI and
check it against kq_gemv (and the oracle's tolerance) on two calls in a row,
plus the rejection of a request beyond the fixed scratch.  This file is
collected last so that, if it fails, a run stopping at the first failure has
already run every other test; it also passes when run alone.
"""
import numpy as np
import pytest

import workloads as wl

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


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


# (format, N_out, K, n_tok): split-K cases (long rows, several K segments),
# an unsplit case and an n_tok > 4 case (served without scratch)
CASES = [(2, 600, 32768, 1), (0, 300, 32768, 2), (1, 96, 5120, 3), (0, 4096, 4096, 1), (0, 1100, 32768, 1),
         (3, 64, 1024, 8)]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"f{c[0]}_{c[1]}x{c[2]}_t{c[3]}")
def test_noalloc_matches_gemv_on_two_calls(kq, oracle, case):
    fmt, N, K, T = case
    Wb = oracle.quantize(fmt, wl.weights_f32(wl.derive_seed(300, fmt, N), N, K), N, K)
    x = wl.activations_bf16(wl.derive_seed(301, N, K), T, K, heavy=True)
    _, A = oracle.gemv(fmt, Wb, N, K, x)
    tol = 1e-3 * A + 1e-5
    W, xd = _dev(Wb), _dev(x.view(np.int16)).view(torch.bfloat16)
    y_ref = torch.empty((T, N), dtype=torch.float32, device="cuda")
    kq.kq_gemv(fmt, W, xd, y_ref, N, K, T)
    torch.cuda.synchronize()
    ref = y_ref.cpu().numpy().astype(np.float64)
    for call in range(2):
        y = torch.full((T, N), 1234.5, dtype=torch.float32, device="cuda")
        assert kq.kq_gemv_noalloc(fmt, W, xd, y, N, K, T) == 0
        assert kq.kq_device_status() == 0
        got = y.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(got - ref) <= tol), f"call {call}"


def test_noalloc_rejects_beyond_its_scratch(kq):
    # 10000 rows x K 32768 x 4 tokens needs ~2.6 MB of split-K partial sums,
    # more than the fixed array holds: rejected before anything is launched
    # (the buffers are full-size, so nothing could read out of bounds).
    fmt, N, K, T = 0, 10000, 32768, 4
    W = torch.zeros(N * (K // 256) * 144, dtype=torch.uint8, device="cuda")
    x = torch.zeros((T, K), dtype=torch.bfloat16, device="cuda")
    y = torch.full((T, N), 7.0, dtype=torch.float32, device="cuda")
    st = kq.kq_gemv_noalloc(fmt, W, x, y, N, K, T, check=False)
    assert st == 9                                  # KQ_ERR_TOO_LARGE
    assert kq.kq_status_str(st)
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())                   # y untouched
