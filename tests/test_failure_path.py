"""The failure path of the kernels' bounded waits, exercised without a fault.

Every spin-wait in the kernels (a warp waiting on a shared-memory barrier
for a copy or for another warp) gives up after a bounded number of cycles,
counts the event in a device word and lets the kernel return; the host reads
the count with kq_device_status, which then reports KQ_ERR_TIMEOUT and
re-arms the split-K and tile-claiming counters a stopped kernel may leave
behind.  kq_test_wait_timeout launches one warp whose wait on a barrier that
nothing completes is shortened to a few milliseconds, so the wait runs out
for real.  Nothing faults and nothing hangs: the context stays usable, which
the normal launches after it show.
"""
import numpy as np
import pytest

import workloads as wl

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
KQ_OK, KQ_ERR_ARG, KQ_ERR_TIMEOUT = 0, 1, 8


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


def test_bounded_wait_runs_out_and_is_reported(kq, oracle):
    assert kq.kq_device_status() == KQ_OK
    assert kq.kq_test_wait_timeout(3000) == KQ_OK          # ~3 ms wait on a barrier nobody completes
    assert kq.kq_device_status(check=False) == KQ_ERR_TIMEOUT
    assert kq.kq_device_status(check=False) == KQ_OK       # the count was cleared
    # two in a row are both counted, and reported once
    kq.kq_test_wait_timeout(1000)
    kq.kq_test_wait_timeout(1000)
    assert kq.kq_device_status(check=False) == KQ_ERR_TIMEOUT
    assert kq.kq_device_status(check=False) == KQ_OK
    # the next normal launches are correct: split-K long rows (arrival
    # counters) and many tiles (tile-claiming counters), at 1 and 3 tokens
    for fmt, N, K, T in ((2, 1100, 32768, 1), (0, 9000, 4096, 1), (1, 700, 32768, 3)):
        Wb = oracle.quantize(fmt, wl.weights_f32(wl.derive_seed(320, fmt), N, K), N, K)
        x = wl.activations_bf16(wl.derive_seed(321, fmt), T, K, heavy=True)
        y_ref, A = oracle.gemv(fmt, Wb, N, K, x)
        y = torch.full((T, N), 1234.5, dtype=torch.float32, device="cuda")
        kq.kq_gemv(fmt, _dev(Wb), _dev(x.view(np.int16)).view(torch.bfloat16), y, N, K, T)
        assert kq.kq_device_status(check=False) == KQ_OK
        err = np.abs(y.cpu().numpy().astype(np.float64) - y_ref)
        assert np.all(err <= 1e-3 * A + 1e-5), (fmt, N, K, T)


def test_wait_timeout_hook_rejects_bad_limits(kq):
    assert kq.kq_test_wait_timeout(0, check=False) == KQ_ERR_ARG
    assert kq.kq_test_wait_timeout(2_000_000, check=False) == KQ_ERR_ARG
    assert kq.kq_device_status(check=False) == KQ_OK
