"""Pins of the CPU oracle against things other than itself.

Each test checks the oracle against a library routine (numpy float16, torch
bfloat16, numpy matmul), a closed form, a hand-derived value from
tests/golden/, an invariant or a bound -- chosen so that a dropped term, a
wrong sign, a wrong index or a transposed operand fails at least one.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------- scalars

def test_half_decode_matches_numpy_exhaustive(oracle):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    finite = np.isfinite(ref)
    got = np.array([oracle.half_to_double(int(b)) for b in bits[finite][::7]])
    assert np.array_equal(got, ref[finite][::7])
    # signed zeros keep their sign
    assert np.signbit(oracle.half_to_double(0x8000))


def test_bf16_decode_matches_torch_exhaustive(oracle):
    import torch
    bits = np.arange(0, 65536, 5, dtype=np.int64)
    t = torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    finite = np.isfinite(t)
    got = np.array([oracle.bf16_to_double(int(b)) for b in bits[finite]])
    assert np.array_equal(got, t[finite])


def test_half_round_up_is_smallest_fp16_above(oracle):
    rng = np.random.default_rng(5)
    vals = np.concatenate([rng.uniform(0, 1, 400) * 10.0 ** rng.integers(-9, 5, 400),
                           [2.0 ** -24, 2.0 ** -14, 1.0, 65504.0, 3e-8, 1e-12]])
    for v in vals:
        r = oracle.half_round_up(float(v))
        assert r is not None
        val, b = r
        h = np.uint16(b).view(np.float16)
        assert float(h) == val                     # encoding matches value
        assert val >= v
        below = np.nextafter(h, np.float16(0))     # previous fp16 value
        assert float(below) < v
    assert oracle.half_round_up(70000.0) is None
    assert oracle.half_round_up(0.0) == (0.0, 0)


# ------------------------------------------------------- decoder closed forms

def _q4k_const_block(d_bits, dmin_bits, sc, m, qbyte):
    """One Q4_K block with every sub-block's (sc, m) equal; sc, m < 16 so the
    high two bits stored for sub-blocks 4..7 are zero (hand-encoded)."""
    b = bytearray(144)
    b[0:2] = d_bits.to_bytes(2, "little")
    b[2:4] = dmin_bits.to_bytes(2, "little")
    for j in range(4):
        b[4 + j] = sc
        b[8 + j] = m
        b[12 + j] = (sc & 15) | ((m & 15) << 4)
    b[16:144] = bytes([qbyte]) * 128
    return np.frombuffer(bytes(b), dtype=np.uint8)


def test_q4k_constant_block_closed_form(oracle):
    # d = 0.5 (0x3800), dmin = 0.25 (0x3400), sc = 10, m = 3, q = 7 everywhere:
    # w^ = 0.5*10*7 - 0.25*3 = 34.25 for all 256 weights.
    blk = _q4k_const_block(0x3800, 0x3400, 10, 3, 0x77)
    w = oracle.dequantize(oracle.Q4_K, blk, 1, 256)
    assert np.all(w == 34.25)
    # y = 34.25 * sum(x) exactly for small-integer x
    x = wl.bf16_bits(np.arange(-128, 128, dtype=np.float32) % 7 - 3).reshape(1, 256)
    xs = float(np.sum(np.arange(-128, 128) % 7 - 3))
    y, A = oracle.gemv(oracle.Q4_K, blk, 1, 256, x)
    assert y[0, 0] == 34.25 * xs
    assert A[0, 0] == 34.25 * float(np.sum(np.abs(np.arange(-128, 128) % 7 - 3)))


def test_q4k_min_term_sign_and_high_nibble(oracle):
    # q byte 0xf0: low nibble 0 (sub-blocks 0,2,4,6), high nibble 15
    # (sub-blocks 1,3,5,7).  d = 1, dmin = 2, sc = 1, m = 5:
    # low: 1*1*0 - 2*5 = -10 ; high: 1*1*15 - 10 = 5.
    blk = _q4k_const_block(0x3C00, 0x4000, 1, 5, 0xF0)
    w = oracle.dequantize(oracle.Q4_K, blk, 1, 256)[0]
    for c in range(4):
        assert np.all(w[64 * c: 64 * c + 32] == -10.0)
        assert np.all(w[64 * c + 32: 64 * c + 64] == 5.0)


def test_q4k_scale_field_bit_placement(oracle):
    # Hand-placed bits in the 12-byte field (d = 1, dmin = 1, q = 1):
    #  scales[0] = 0xC5: sc0 = 5, top bits 3 -> sc4 high bits = 3
    #  scales[5] = 0x82: m1 = 2, top bits 2 -> m5 high bits = 2
    #  scales[8] = 0x97: sc4 low = 7, m4 low = 9 -> sc4 = 7 | 3<<4 = 55, m4 = 9
    #  scales[9] = 0x04: sc5 = 4, m5 low = 0 -> m5 = 0 | 2<<4 = 32
    b = bytearray(144)
    b[0:2] = (0x3C00).to_bytes(2, "little")
    b[2:4] = (0x3C00).to_bytes(2, "little")
    b[4 + 0] = 0xC5
    b[4 + 5] = 0x82
    b[4 + 8] = 0x97
    b[4 + 9] = 0x04
    b[16:144] = bytes([0x11]) * 128
    w = oracle.dequantize(oracle.Q4_K, np.frombuffer(bytes(b), np.uint8), 1, 256)[0]
    expect_sc = [5, 0, 0, 0, 55, 4, 0, 0]
    expect_m = [0, 2, 0, 0, 9, 32, 0, 0]
    for j in range(8):
        seg = w[32 * j: 32 * j + 32]
        assert np.all(seg == expect_sc[j] * 1 - expect_m[j]), j


def test_q4k_nibble_index_map(oracle):
    # d = 1, dmin = 0, all sc = 1; one qs byte p = 0x21 at a time: the low
    # nibble (1) lands on weight 64*(p//32) + p%32, the high nibble (2) on the
    # same index + 32.
    for p in range(0, 128, 5):
        blk = bytearray(_q4k_const_block(0x3C00, 0x0000, 1, 0, 0x00).tobytes())
        blk[16 + p] = 0x21
        w = oracle.dequantize(oracle.Q4_K, np.frombuffer(bytes(blk), np.uint8), 1, 256)[0]
        lo = 64 * (p // 32) + p % 32
        nz = np.nonzero(w)[0]
        assert list(nz) == [lo, lo + 32]
        assert w[lo] == 1.0 and w[lo + 32] == 2.0


def test_q5k_fifth_bit(oracle):
    # d = 1, dmin = 0, sc = 1; qs = 0 and a single qh bit set: the bit k of
    # qh[l] adds 16 to weight 64*(k//2) + 32*(k%2) + l.
    for l in (0, 7, 31):
        for k in range(8):
            b = bytearray(176)
            b[0:2] = (0x3C00).to_bytes(2, "little")
            for j in range(4):
                b[4 + j] = 1
                b[12 + j] = 1
            b[16 + l] = 1 << k
            w = oracle.dequantize(oracle.Q5_K, np.frombuffer(bytes(b), np.uint8), 1, 256)[0]
            idx = 64 * (k // 2) + 32 * (k % 2) + l
            assert list(np.nonzero(w)[0]) == [idx]
            assert w[idx] == 16.0
    # all bits set: q = 31 everywhere -> w = 31 with qs = 0xff
    b = bytearray(176)
    b[0:2] = (0x3C00).to_bytes(2, "little")
    for j in range(4):
        b[4 + j] = 1
        b[12 + j] = 1
    b[16:48] = b"\xff" * 32
    b[48:176] = b"\xff" * 128
    w = oracle.dequantize(oracle.Q5_K, np.frombuffer(bytes(b), np.uint8), 1, 256)[0]
    assert np.all(w == 31.0)


def test_q6k_closed_forms_and_signed_scales(oracle):
    def blk(ql, qh, scales, d_bits):
        b = bytearray(210)
        b[0:128] = bytes([ql]) * 128
        b[128:192] = bytes([qh]) * 64
        b[192:208] = bytes(s & 255 for s in scales)
        b[208:210] = d_bits.to_bytes(2, "little")
        return np.frombuffer(bytes(b), np.uint8)
    one = [1] * 16
    assert np.all(oracle.dequantize(oracle.Q6_K, blk(0, 0, one, 0x3C00), 1, 256) == -32.0)
    assert np.all(oracle.dequantize(oracle.Q6_K, blk(0xFF, 0xFF, one, 0x3C00), 1, 256) == 31.0)
    # negative int8 scale -1 flips the sign: q = 63 -> -31
    assert np.all(oracle.dequantize(oracle.Q6_K, blk(0xFF, 0xFF, [-1] * 16, 0x3C00), 1, 256) == -31.0)
    # scale j = 2 doubles exactly weights 16j..16j+15 (d = 0.5)
    for j in (0, 5, 15):
        sc = [1] * 16
        sc[j] = 2
        w = oracle.dequantize(oracle.Q6_K, blk(0xFF, 0xFF, sc, 0x3800), 1, 256)[0]
        assert np.all(w[16 * j: 16 * j + 16] == 31.0)
        rest = np.delete(w, np.arange(16 * j, 16 * j + 16))
        assert np.all(rest == 15.5)


def test_q6k_bit_index_map(oracle):
    # ql byte p: low nibble -> weight 128h + l + 32*(p%64 >= 32), high nibble
    # -> +64.  qh byte (h, l) bit pair t -> weight 128h + 32t + l.
    base = bytearray(210)
    base[192:208] = bytes([1] * 16)
    base[208:210] = (0x3C00).to_bytes(2, "little")
    for p in (0, 17, 40, 63, 64, 100, 127):
        b = bytearray(base)
        b[p] = 0x21
        w = oracle.dequantize(oracle.Q6_K, np.frombuffer(bytes(b), np.uint8), 1, 256)[0] + 32.0
        h, r = divmod(p, 64)
        lo = 128 * h + (r % 32) + 32 * (r // 32)
        nz = np.nonzero(w)[0]
        assert list(nz) == [lo, lo + 64] and w[lo] == 1.0 and w[lo + 64] == 2.0
    for hl in (0, 9, 31, 32, 50, 63):
        for t in range(4):
            b = bytearray(base)
            b[128 + hl] = 1 << (2 * t)
            w = oracle.dequantize(oracle.Q6_K, np.frombuffer(bytes(b), np.uint8), 1, 256)[0] + 32.0
            h, l = divmod(hl, 32)
            assert list(np.nonzero(w)[0]) == [128 * h + 32 * t + l]
            assert w[128 * h + 32 * t + l] == 16.0


def test_g128_param_record(oracle):
    # one super-block: q plane all 0x31 (low 1, high 3); params d = 1,
    # dmin = 0.5, sc = (2, 7), m = (4, 6):
    # group 0: low 1*2*1 - 0.5*4 = 0, high 1*2*3 - 2 = 4
    # group 1: low 7 - 3 = 4, high 21 - 3 = 18
    W = np.frombuffer(bytes([0x31]) * 128 + (0x3C00).to_bytes(2, "little")
                      + (0x3800).to_bytes(2, "little") + bytes([2, 7, 4, 6]), np.uint8)
    w = oracle.dequantize(oracle.Q4_G128, W, 1, 256)[0]
    for c in range(4):
        g = c // 2
        lo, hi = (0.0, 4.0) if g == 0 else (4.0, 18.0)
        assert np.all(w[64 * c: 64 * c + 32] == lo)
        assert np.all(w[64 * c + 32: 64 * c + 64] == hi)


# ------------------------------------------------------------------ product

@pytest.mark.parametrize("fmt", [0, 1, 2, 3])
def test_gemv_matches_numpy_on_dequantised(oracle, fmt):
    N, K, T = 5, 768, 3
    Wb = wl.random_block_bytes(wl.derive_seed(1, fmt), fmt, N * K // 256)
    x = wl.activations_bf16(wl.derive_seed(2, fmt), T, K)
    Wd = oracle.dequantize(fmt, Wb, N, K)
    xd = x.astype(np.uint32).__lshift__(16).view(np.float32).astype(np.float64)
    y, A = oracle.gemv(fmt, Wb, N, K, x)
    ref = xd @ Wd.T
    refA = np.abs(xd) @ np.abs(Wd).T
    scale = refA + 1e-300
    assert np.all(np.abs(y - ref) <= 1e-12 * scale)
    assert np.all(np.abs(A - refA) <= 1e-12 * scale)
    # one-hot x picks a column exactly
    for k in (0, 255, 256, 767):
        e = np.zeros((1, K), np.float32)
        e[0, k] = 1.0
        ye, _ = oracle.gemv(fmt, Wb, N, K, wl.bf16_bits(e))
        assert np.array_equal(ye[0], Wd[:, k])


def test_gemv_brute_force_exact_rational(oracle):
    # N = 2, K = 256: the fp64 sum in k order stays within the classical
    # recursive-summation bound of the exact rational sum of w^ x.
    for fmt in (0, 1, 2, 3):
        Wb = wl.random_block_bytes(wl.derive_seed(3, fmt), fmt, 2)
        x = wl.activations_bf16(wl.derive_seed(4, fmt), 1, 256, heavy=True)
        Wd = oracle.dequantize(fmt, Wb, 2, 256)
        xd = x.astype(np.uint32).__lshift__(16).view(np.float32).astype(np.float64)[0]
        y, A = oracle.gemv(fmt, Wb, 2, 256, x)
        for n in range(2):
            exact = sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(Wd[n], xd))
            bound = 256 * 2.0 ** -53 * A[0, n] * 1.01
            assert abs(float(Fraction(y[0, n]) - exact)) <= bound


def test_gemv_rows_and_token_consistency(oracle):
    fmt, N, K = 0, 7, 512
    Wb = wl.random_block_bytes(wl.derive_seed(5), fmt, N * K // 256)
    x = wl.activations_bf16(wl.derive_seed(6), 16, K)
    y, A = oracle.gemv(fmt, Wb, N, K, x)
    for t in (0, 5, 15):
        yt, At = oracle.gemv(fmt, Wb, N, K, x[t:t + 1])
        assert np.array_equal(yt[0], y[t]) and np.array_equal(At[0], A[t])
    rows = [6, 0, 3]
    yr, Ar = oracle.gemv_rows(fmt, Wb, N, K, rows, x)
    assert np.array_equal(yr, y[:, rows]) and np.array_equal(Ar, A[:, rows])


def test_gemv_linearity(oracle):
    fmt, N, K = 2, 4, 512
    Wb = wl.random_block_bytes(wl.derive_seed(8), fmt, N * K // 256)
    x1 = np.rint(np.random.default_rng(0).normal(0, 8, (1, K))).astype(np.float32)
    x2 = np.rint(np.random.default_rng(1).normal(0, 8, (1, K))).astype(np.float32)
    y1, A1 = oracle.gemv(fmt, Wb, N, K, wl.bf16_bits(x1))
    y2, A2 = oracle.gemv(fmt, Wb, N, K, wl.bf16_bits(x2))
    y3, _ = oracle.gemv(fmt, Wb, N, K, wl.bf16_bits(x1 + x2))
    assert np.all(np.abs(y3 - (y1 + y2)) <= 1e-12 * (A1 + A2))


# --------------------------------------------------------------- quantiser

def _golden_cases():
    cases, cur = [], None
    for line in open(os.path.join(GOLDEN, "quantiser_hand_cases.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        tok = line.split()
        if tok[0] == "case":
            cur = {"name": tok[1], "fmt": {"Q4_K": 0, "Q5_K": 1, "Q6_K": 2}[tok[2]],
                   "w": {}, "expect": {}}
            cases.append(cur)
        elif tok[0] == "w":
            cur["w"][int(tok[1])] = float(tok[2])
        elif tok[0] == "expect":
            off = int(tok[1])
            for i, h in enumerate(tok[2:]):
                cur["expect"][off + i] = int(h, 16)
    return cases


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_quantiser_hand_derived_bytes(oracle, case):
    w = np.zeros(256, np.float32)
    for i, v in case["w"].items():
        w[i] = v
    got = oracle.quantize(case["fmt"], w, 1, 256)
    want = np.zeros_like(got)
    for off, v in case["expect"].items():
        want[off] = v
    assert got.tobytes().hex() == want.tobytes().hex()


def _steps(oracle, fmt, Wb, N, K):
    """Quantisation step d*sc per weight, from the hand-read record fields."""
    nsb = K // 256
    steps = np.zeros((N, K))
    nb = oracle.BLOCK_BYTES[fmt]
    for n in range(N):
        for b in range(nsb):
            if fmt == 3:
                p = Wb[N * nsb * 128 + (n * nsb + b) * 8:][:8]
                d = oracle.half_to_double(int(p[0]) | int(p[1]) << 8)
                st = np.repeat([d * p[4], d * p[5]], 128)
            else:
                r = Wb[(n * nsb + b) * nb:][:nb]
                if fmt == 2:
                    d = oracle.half_to_double(int(r[208]) | int(r[209]) << 8)
                    st = np.repeat(d * np.abs(r[192:208].view(np.int8).astype(float)), 16)
                else:
                    d = oracle.half_to_double(int(r[0]) | int(r[1]) << 8)
                    s = r[4:16]
                    sc = [s[j] & 63 if j < 4 else (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4)
                          for j in range(8)]
                    st = np.repeat(d * np.array(sc, float), 32)
            steps[n, 256 * b: 256 * b + 256] = st
    return steps


@pytest.mark.parametrize("fmt", [0, 1, 2, 3])
@pytest.mark.parametrize("kind", ["normal", "heavy", "shifted", "negative", "outlier"])
def test_quantiser_round_trip_half_step(oracle, fmt, kind):
    N, K = 6, 512
    w = wl.weights_f32(wl.derive_seed(10, fmt), N, K).astype(np.float64)
    if kind == "heavy":
        u = wl.uniform01(wl.derive_seed(11), 0, N * K).reshape(N, K)
        w = np.where(u < 0.05, w * 20, w)
    elif kind == "shifted":
        w = w + 0.05
    elif kind == "negative":
        w = -np.abs(w) - 0.01
    elif kind == "outlier":
        w[:, 3] = 5.0
        w[:, 300] = -7.0
    w = w.astype(np.float32)
    Wb = oracle.quantize(fmt, w, N, K)
    wd = oracle.dequantize(fmt, Wb, N, K)
    step = _steps(oracle, fmt, Wb, N, K)
    err = np.abs(w.astype(np.float64) - wd)
    assert np.all(err <= 0.5 * step * (1 + 1e-12) + 1e-300)
    # field ranges
    if fmt in (0, 1):
        for n in range(N):
            for b in range(K // 256):
                s = Wb[(n * (K // 256) + b) * (144 if fmt == 0 else 176) + 4:][:12]
                for j in range(8):
                    sc = s[j] & 63 if j < 4 else (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4)
                    assert 0 <= sc <= 63


def test_quantiser_zero_and_constant_blocks(oracle):
    for fmt in (0, 1, 2, 3):
        Wb = oracle.quantize(fmt, np.zeros((2, 256), np.float32), 2, 256)
        assert not Wb.any()
        assert np.all(oracle.dequantize(fmt, Wb, 2, 256) == 0.0)
    # a constant block at -63*2^-10 sits on the min grid: dmin = 2^-10,
    # m = 63, r = 0 so d = sc = q = 0, and w^ = -dmin*m reproduces it exactly
    c = -63.0 * 2.0 ** -10
    for fmt in (0, 1, 3):
        Wb = oracle.quantize(fmt, np.full((1, 256), c, np.float32), 1, 256)
        assert np.all(oracle.dequantize(fmt, Wb, 1, 256) == c)


def test_quantiser_range_error(oracle):
    w = np.zeros((1, 256), np.float32)
    w[0, 0] = 3.0e9
    for fmt in (0, 1, 2, 3):
        with pytest.raises(oracle.OracleError):
            oracle.quantize(fmt, w, 1, 256)


# -------------------------------------------------------------------- merge

def test_merge_lossless_invariant(oracle):
    N, K = 9, 1024
    w = wl.weights_f32(wl.derive_seed(20), N, K)
    q4 = oracle.quantize_q4k_group128(w, N, K)
    st, g = oracle.merge_g128(q4, N, K)
    assert st == oracle.OK
    # the direct G128 quantiser lands on the same bytes
    assert np.array_equal(g, oracle.quantize(oracle.Q4_G128, w, N, K))
    wq = oracle.dequantize(oracle.Q4_K, q4, N, K)
    wg = oracle.dequantize(oracle.Q4_G128, g, N, K)
    assert np.array_equal(wq.view(np.uint64), wg.view(np.uint64))
    x = wl.activations_bf16(wl.derive_seed(21), 4, K)
    yq, Aq = oracle.gemv(oracle.Q4_K, q4, N, K, x)
    yg, Ag = oracle.gemv(oracle.Q4_G128, g, N, K, x)
    assert np.array_equal(yq, yg) and np.array_equal(Aq, Ag)
    # group statistics keep the half-step bound over the 128-weight groups
    step = _steps(oracle, oracle.Q4_G128, g, N, K)
    assert np.all(np.abs(w - wg) <= 0.5 * step * (1 + 1e-12) + 1e-300)


def test_merge_rejects_unmergeable(oracle):
    N, K = 3, 512
    w = wl.weights_f32(wl.derive_seed(22), N, K)
    q4 = oracle.quantize(oracle.Q4_K, w, N, K)
    assert oracle.merge_g128(q4, N, K)[0] == oracle.NOT_MERGEABLE
    # a single differing min in an otherwise mergeable matrix is rejected
    q4g = oracle.quantize_q4k_group128(w, N, K)
    assert oracle.merge_g128(q4g, N, K)[0] == oracle.OK
    bad = q4g.copy()
    blk = 144 * 4 + 4            # super-block 4, scale field
    bad[blk + 5] ^= 1            # m1 changes, m0 does not
    assert oracle.merge_g128(bad, N, K)[0] == oracle.NOT_MERGEABLE


# ------------------------------------------------------- pages' bookkeeping

def _pages():
    vals = {}
    for line in open(os.path.join(GOLDEN, "pages_numbers.txt")):
        line = line.split("#")[0].strip()
        if line:
            k, v = line.split()
            vals[k] = float(v)
    return vals


def test_pages_bandwidth_arithmetic():
    p = _pages()
    gbs = wl.weight_gb_per_s(p["weight_gb"] * 1e9, 1.0 / p["decode_tok_s"])
    assert round(gbs) == p["traffic_gb_s"]
    assert gbs < p["bin_gb_s"]


def test_pages_parameter_count():
    p = _pages()
    L = wl.layer_matrices(0, 0, 0, hidden=int(p["hidden"]), inter=int(p["intermediate"]),
                          nq=int(p["q_heads"]), nkv=int(p["kv_heads"]), hd=int(p["head_dim"]))
    q_width = int(p["q_heads"] * p["head_dim"])
    per_layer = sum(m.N * m.K for m in L) + q_width * int(p["hidden"])   # + attention gate
    total = int(p["layers"]) * per_layer + 2 * int(p["vocab"]) * int(p["hidden"])
    assert abs(total / 1e9 - p["text_params_b"]) / p["text_params_b"] < 1e-4


def test_pages_shape_workload_is_the_cards_model():
    # the second workload (the card's own shapes, q/k/v and the attention
    # gate in one launch) has exactly the card's text-tower parameters
    p = _pages()
    assert (wl.GLIMMER_HIDDEN, wl.GLIMMER_INTER, wl.GLIMMER_VOCAB) == \
        (int(p["hidden"]), int(p["intermediate"]), int(p["vocab"]))
    per_layer = sum(m.N * m.K for m in wl.GLIMMER_LAYER)
    total = int(p["layers"]) * per_layer + 2 * wl.GLIMMER_HEAD.N * wl.GLIMMER_HEAD.K   # + embedding
    assert abs(total / 1e9 - p["text_params_b"]) / p["text_params_b"] < 1e-4
    assert [m.name for m in wl.GLIMMER_LAYER[:4]] == ["q", "k", "v", "attn_gate"]
    assert all(m.K == wl.GLIMMER_HIDDEN for m in wl.GLIMMER_LAYER[:4])
