"""kq_gemv_noalloc: the GEMV entry point that never allocates device memory.

Some callers cannot call cudaMalloc when they run the GEMV: code inside a
CUDA-graph stream capture, engines that own all device memory through their
own pool, latency-critical loops that cannot take an allocation's implicit
synchronisation.  For them kq_gemv_noalloc keeps the split-K scratch in a
fixed array inside the library.  These tests call it through the C ABI and
check:
  * its output against the fp64 oracle (|y - y_ref| <= 1e-3 sum|w^ x| +
    1e-5) and against kq_gemv's, on two calls in a row, for split-K long
    rows at 1..16 tokens, grouped-format and small shapes;
  * in a fresh process, that none of those calls allocates: after them the
    library's own split-K buffer still does not exist (the first kq_gemv
    that needs it then allocates it, which the device's free memory shows);
  * the rejection of a request that needs more scratch than the array holds.
This file is collected last so that, if it fails, a run stopping at the
first failure has already run every other test; it also passes when run
alone.
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import workloads as wl

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


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


# (format, N_out, K, n_tok): split-K long rows at 1, 2, 3, 8 and 16 tokens
# (CUDA-core, single-token and multi-token tensor-core kernels), an unsplit
# case, a 33.5 M-weight Q4_K verify case and a small G128 case
CASES = [(2, 600, 32768, 1), (0, 300, 32768, 2), (1, 96, 5120, 3), (0, 4096, 4096, 1),
         (0, 1100, 32768, 1), (3, 64, 1024, 8), (2, 1100, 32768, 8), (1, 600, 32768, 16),
         (0, 8192, 4096, 16)]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"f{c[0]}_{c[1]}x{c[2]}_t{c[3]}")
def test_noalloc_matches_oracle_on_two_calls(kq, oracle, case):
    fmt, N, K, T = case
    Wb = oracle.quantize(fmt, wl.weights_f32(wl.derive_seed(300, fmt, N), N, K), N, K)
    x = wl.activations_bf16(wl.derive_seed(301, N, K), T, K, heavy=True)
    y_ref, A = oracle.gemv(fmt, Wb, N, K, x)
    tol = 1e-3 * A + 1e-5
    W, xd = _dev(Wb), _dev(x.view(np.int16)).view(torch.bfloat16)
    for call in range(2):
        y = torch.full((T, N), 1234.5, dtype=torch.float32, device="cuda")
        assert kq.kq_gemv_noalloc(fmt, W, xd, y, N, K, T) == 0
        assert kq.kq_device_status() == 0
        got = y.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(got - y_ref) <= tol), f"call {call}: outside the oracle's tolerance"
    y_gemv = torch.empty((T, N), dtype=torch.float32, device="cuda")
    kq.kq_gemv(fmt, W, xd, y_gemv, N, K, T)
    torch.cuda.synchronize()
    assert np.all(np.abs(y_gemv.cpu().numpy().astype(np.float64) - got) <= 2 * tol)


_CHILD = r"""
import json, os, sys
import numpy as np
import torch
sys.path.insert(0, os.environ["KQ_ROOT"])
import quant_weight_gemv_dequant_b300 as kq
import workloads as wl
kq.lib()
cases = json.loads(os.environ["KQ_CASES"])
dev = torch.device("cuda", 0)
bufs = []
for fmt, N, K, T in cases:
    W = torch.from_numpy(wl.random_block_bytes(wl.derive_seed(310, fmt, N), fmt, N * K // 256)).to(dev)
    x = torch.from_numpy(wl.activations_bf16(wl.derive_seed(311, N), T, K).view(np.int16)).to(dev)
    bufs.append((W, x.view(torch.bfloat16), torch.empty((T, N), dtype=torch.float32, device=dev)))
torch.cuda.synchronize()
status = []
free = []
for rnd in range(2):
    for (fmt, N, K, T), (W, x, y) in zip(cases, bufs):
        status.append(kq.kq_gemv_noalloc(fmt, W, x, y, N, K, T, check=False))
    torch.cuda.synchronize()
    free.append(torch.cuda.mem_get_info(dev)[0])
y_na = bufs[0][2].clone()
fmt, N, K, T = cases[0]
W, x, _ = bufs[0]
y_g = torch.empty((T, N), dtype=torch.float32, device=dev)
torch.cuda.synchronize()
free.append(torch.cuda.mem_get_info(dev)[0])
status.append(kq.kq_gemv(fmt, W, x, y_g, N, K, T, check=False))
torch.cuda.synchronize()
free.append(torch.cuda.mem_get_info(dev)[0])
status.append(kq.kq_device_status(check=False))
rel = float(((y_na - y_g).abs().max() / y_g.abs().max().clamp_min(1e-30)).item())
print(json.dumps({"status": status, "free": free, "rel": rel}))
"""


def test_noalloc_allocates_nothing_in_a_fresh_process(kq):
    # A fresh process runs kq_gemv_noalloc on split-K long rows (the first
    # request of its shape), at 1, 8 and 16 tokens, twice, before any kq_gemv.
    # Had any of these calls reached the library's growing split-K buffer,
    # that buffer (at least 16 MiB) would exist afterwards and the first
    # kq_gemv that needs it would allocate nothing; instead that kq_gemv
    # allocates it, which the device's free memory shows.  The second round
    # of no-alloc calls changes free memory by less than 2 MiB.
    cases = [(2, 600, 32768, 1), (0, 1100, 32768, 1), (2, 1100, 32768, 8), (1, 600, 32768, 16),
             (0, 300, 32768, 2)]
    env = dict(os.environ, KQ_ROOT=ROOT, KQ_CASES=json.dumps(cases))
    out = subprocess.run([sys.executable, "-c", _CHILD], env=env, capture_output=True, text=True,
                         timeout=600)
    assert out.returncode == 0, out.stderr[-3000:]
    r = json.loads(out.stdout.strip().splitlines()[-1])
    assert all(s == 0 for s in r["status"]), r["status"]
    f_first, f_second, f_before_gemv, f_after_gemv = r["free"]
    assert abs(f_second - f_first) < 2 << 20, "a second round of no-alloc calls changed free device memory"
    assert f_before_gemv - f_after_gemv >= 16 << 20, (
        "kq_gemv allocated no split-K buffer, so an earlier no-alloc call must have")
    assert r["rel"] <= 1e-4


def test_noalloc_rejects_beyond_its_scratch(kq):
    # 200000 rows of 32768 weights at 4 tokens: every kernel that serves this
    # shape splits K (x does not fit shared memory whole), and even two K
    # segments need 6.4 MB of partial sums, more than the fixed array holds:
    # rejected before anything is launched (the buffers are full-size, so
    # nothing could read out of bounds).
    fmt, N, K, T = 0, 200000, 32768, 4
    W = torch.zeros(N * (K // 256) * 144, dtype=torch.uint8, device="cuda")
    x = torch.zeros((T, K), dtype=torch.bfloat16, device="cuda")
    y = torch.full((T, N), 7.0, dtype=torch.float32, device="cuda")
    st = kq.kq_gemv_noalloc(fmt, W, x, y, N, K, T, check=False)
    assert st == 9                                  # KQ_ERR_TOO_LARGE
    assert kq.kq_status_str(st)
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())                   # y untouched
    del W
    torch.cuda.empty_cache()
