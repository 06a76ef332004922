"""GPU parity on legal records whose dequantised weights are zero (or nearly
all zero) while their scales are not: the encodings where an offset form of
the product (computing sum (c + q) x and subtracting c sum x afterwards)
would lose the result in the rounding of the two large terms.

Record types, spread over the rows of each matrix (row r is of type r % 37
for r % 37 < 6, an ordinary quantised row otherwise):
  0  q = 0 everywhere, every sub-block scale nonzero (1..63), m = 0, d*sc
     around 0.06                                       -> w^ = 0, y = 0 exactly
  1  the same with d = 1000, sc = 63 (d*sc = 63000)    -> y = 0 exactly
  2  q = 0 except one q = 1 per sub-block, d = 1000, sc = 63, m = 0
  3  q = 0 except one q = 15 per sub-block, small scales, m = 0
  4  q = 0 everywhere, nonzero scales, nonzero dmin but m = 0 -> y = 0 exactly
  5  every field random (legal fp16 scales), the tail of the distribution
Q6_K has no min term; its zero weight is q = 32, so types 0, 1 and 4 store q =
32 everywhere and types 2, 3 store q = 33 or q = 63 at one position per
sub-block.  Q5_K's fifth bits are zero in types 0..4.

The record layouts are those of include/kq.h (the daily.dev ExecuTorch
summary, answer on exporting GGUF checkpoints, names the formats; the bit
placement is GGUF's public layout).  Each matrix runs through every kernel
the dispatch takes for its size at n_tok 1, 2, 3, 4, 5, 8 and 16: the
single-token and verify-width tensor-core kernels (33.5 M and 36 M weight
Q4_K / Q4_G128 launches), the streaming CUDA-core kernel, the mma verify
kernel (Q5_K, Q6_K and small launches) and the small-launch kernel.  Bar:
the oracle's |y - y_ref| <= 1e-3 sum|w^ x| + 1e-5, and exact zeros for the
zero-weight rows.
"""
import numpy as np
import pytest

import workloads as wl

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

FMTS = [0, 1, 2, 3]
FMT_IDS = ["Q4_K", "Q5_K", "Q6_K", "G128"]
ZERO_TYPES = (0, 1, 4)
PERIOD = 37
NTOKS = (1, 2, 3, 4, 5, 8, 16)
# (N, K): 33.5 M weights on the 16-byte grid (tensor-core kernels for the Q4
# family at every width); 36 M weights with K = 32768 (split K); a small
# launch (a few rows per SM)
SHAPES = [(8192, 4096), (1100, 32768), (300, 2048)]


@pytest.fixture(scope="module")
def kq():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from quant_weight_gemv_dequant_b300 import build
    build.build()
    import quant_weight_gemv_dequant_b300 as k
    k.lib()
    return k


def _h(v):
    """fp16 bits of v (exactly representable values only)."""
    b = int(np.array(v, dtype=np.float16).view(np.uint16))
    assert float(np.array(b, dtype=np.uint16).view(np.float16)) == v
    return b


def _pack_scales(sc, m):
    """The 12-byte 6-bit (sc, m) field of Q4_K / Q5_K (layout in kq.h)."""
    s = bytearray(12)
    for j in range(4):
        s[j] = (sc[j] & 63) | ((sc[j + 4] >> 4) << 6)
        s[j + 4] = (m[j] & 63) | ((m[j + 4] >> 4) << 6)
        s[j + 8] = (sc[j + 4] & 15) | ((m[j + 4] & 15) << 4)
    return bytes(s)


def _qs_from_q(q):
    """Q4_K qs[128] from 256 4-bit values: weight 64c + r (r < 32) is the low
    nibble of qs[32c + r], weight 64c + 32 + r its high nibble."""
    qs = bytearray(128)
    for c in range(4):
        for r in range(32):
            qs[32 * c + r] = (q[64 * c + r] & 15) | ((q[64 * c + 32 + r] & 15) << 4)
    return bytes(qs)


def _q6_bytes(q):
    """Q6_K ql[128], qh[64] from 256 6-bit values (layout in kq.h)."""
    ql, qh = bytearray(128), bytearray(64)
    for i in range(256):
        h, t, l = i // 128, (i % 128) // 32, i % 32
        p = 64 * h + l + 32 * (t & 1)
        ql[p] |= (q[i] & 15) << (4 * (t >= 2))
        qh[32 * h + l] |= ((q[i] >> 4) & 3) << (2 * t)
    return bytes(ql), bytes(qh)


def _special_q(typ, fmt, rng):
    """The 256 q values of one super-block of record type typ."""
    zero = 32 if fmt == 2 else 0
    q = np.full(256, zero, dtype=np.int64)
    sub = 16 if fmt == 2 else 32
    if typ in (2, 3):
        for j in range(256 // sub):
            pos = j * sub + int(rng.integers(sub))
            q[pos] = (zero + 1) if typ == 2 else (63 if fmt == 2 else 15)
    return q


def _special_record(typ, fmt, rng):
    """(record bytes, params) of one super-block of type typ (0..5)."""
    if typ == 5:
        return None
    q = _special_q(typ, fmt, rng)
    if typ == 1 or typ == 2:
        d = 1000.0
    else:
        d = float(rng.choice([0.0009765625, 0.001953125, 0.0029296875]))
    dmin = 0.0 if typ != 4 else 0.5
    nsub = 16 if fmt == 2 else 8
    if typ in (1, 2):
        sc = [63] * nsub if fmt != 2 else [127 if j % 2 else -127 for j in range(nsub)]
    else:
        sc = [int(v) for v in rng.integers(1, 64, nsub)]
        if fmt == 2:
            sc = [v if j % 3 else -v for j, v in enumerate(sc)]
    m = [0] * 8
    if fmt == 2:
        ql, qh = _q6_bytes(q)
        return ql + qh + bytes(s & 255 for s in sc) + _h(d).to_bytes(2, "little")
    hdr = _h(d).to_bytes(2, "little") + _h(dmin).to_bytes(2, "little")
    if fmt == 0:
        return hdr + _pack_scales(sc, m) + _qs_from_q(q)
    if fmt == 1:
        qh = bytes(32)   # fifth bits zero
        return hdr + _pack_scales(sc, m) + qh + _qs_from_q(q)
    # G128: (q plane bytes, 8 param bytes); groups take sub-blocks 0 and 4
    par = hdr + bytes([sc[0], sc[4], 0, 0])
    return _qs_from_q(q), par


def degenerate_matrix(oracle, fmt, N, K, seed):
    """Oracle-quantised N x K matrix with the special record types written
    into the rows r % PERIOD < 6 (type r % PERIOD; type 5 = random bytes)."""
    rng = np.random.default_rng(seed)
    base = oracle.quantize(fmt, wl.weights_f32(wl.derive_seed(seed), N, K), N, K)
    nsb = K // 256
    rnd = wl.random_block_bytes(wl.derive_seed(seed, 1), fmt, N * nsb)
    W = base.copy()
    if fmt == 3:
        qp = W[: N * nsb * 128].reshape(N, nsb, 128)
        pp = W[N * nsb * 128:].reshape(N, nsb, 8)
        rq = rnd[: N * nsb * 128].reshape(N, nsb, 128)
        rp = rnd[N * nsb * 128:].reshape(N, nsb, 8)
    else:
        bb = oracle.BLOCK_BYTES[fmt]
        Wv = W.reshape(N, nsb, bb)
        Rv = rnd.reshape(N, nsb, bb)
    for r in range(N):
        typ = r % PERIOD
        if typ > 5:
            continue
        for s in range(nsb):
            rec = _special_record(typ, fmt, rng)
            if fmt == 3:
                if rec is None:
                    qp[r, s], pp[r, s] = rq[r, s], rp[r, s]
                else:
                    qp[r, s] = np.frombuffer(rec[0], np.uint8)
                    pp[r, s] = np.frombuffer(rec[1], np.uint8)
            else:
                Wv[r, s] = Rv[r, s] if rec is None else np.frombuffer(rec, np.uint8)
    return W


def _checked_rows(N):
    special = [r for r in range(N) if r % PERIOD < 6]
    rest = wl.splitmix64(77, np.arange(96, dtype=np.uint64)) % np.uint64(N)
    return np.unique(np.concatenate([special, rest.astype(np.int64), [N - 1]]))


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("fmt", FMTS, ids=FMT_IDS)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s[0]}x{s[1]}")
def test_zero_weight_records_with_nonzero_scales(kq, oracle, fmt, shape):
    N, K = shape
    W = degenerate_matrix(oracle, fmt, N, K, 4100 + 10 * fmt + SHAPES.index(shape))
    x = wl.activations_bf16(wl.derive_seed(4200, fmt, N), 16, K, heavy=True)
    rows = _checked_rows(N)
    yref, A = oracle.gemv_rows(fmt, W, N, K, rows, x)
    # the zero-weight rows really dequantise to zero (the oracle's values)
    zrows = [i for i, r in enumerate(rows) if r % PERIOD in ZERO_TYPES]
    assert np.all(yref[:, zrows] == 0.0) and np.all(A[:, zrows] == 0.0)
    Wd = _dev(W)
    xd = _dev(x.view(np.int16)).view(torch.bfloat16)
    for T in NTOKS:
        y = torch.full((T, N), 1234.5, dtype=torch.float32, device="cuda")
        kq.kq_gemv(fmt, Wd, xd[:T], y, N, K, T)
        assert kq.kq_device_status() == 0
        got = y.cpu().numpy()[:, rows].astype(np.float64)
        err = np.abs(got - yref[:T])
        tol = 1e-3 * A[:T] + 1e-5
        bad = ~(err <= tol)
        if bad.any():
            t, i = np.unravel_index(np.argmax(np.where(bad, err / tol, 0)), err.shape)
            raise AssertionError(
                f"n_tok={T}: {bad.sum()} of {bad.size} outside tolerance; worst row {rows[i]} "
                f"(type {rows[i] % PERIOD}) token {t}: y={got[t, i]!r} ref={yref[t, i]!r} "
                f"tol={tol[t, i]!r}")
        assert np.all(got[:, zrows] == 0.0), f"n_tok={T}: zero-weight rows not exactly zero"
