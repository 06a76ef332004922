"""Seeded synthetic workloads for K-quant GEMV: shapes and random inputs.

This module is shared by the tests, the benchmark and the smoke check.  It
holds no arithmetic of the method itself (no dequantisation, no dot
products, no quantiser): only counter-based random numbers, bf16 rounding of
activations, the workload shapes and a block-tiling index map.

Generators (published definitions, written out here):
  * splitmix64 (S. Vigna): state += 0x9E3779B97F4A7C15; z = state;
    z = (z ^ z>>30) * 0xBF58476D1CE4E5B9; z = (z ^ z>>27) * 0x94D049BB133111EB;
    z ^ z>>31.  Used counter-style: value(i) = mix(seed + (i+1)*golden).
  * Box-Muller: n = sqrt(-2 ln u1) cos(2 pi u2) with u1, u2 in (0, 1] built
    from the top 53 bits of two splitmix64 outputs.  Computed in fp64, scaled
    by sigma, rounded to fp32.
  * bf16 activations: N(0,1) in fp32, rounded to bf16 (nearest, ties to
    even).  Heavy-tailed rows multiply a Bernoulli(0.05) subset by 20 in fp32
    before the rounding.

Workload shapes.  The pages (Muse-Glimmer-30B: 52 layers, GQA 32 q / 2 kv
heads of dim 128, SwiGLU; Core AI card architecture section and SGLang day-0
post) fix the layer structure; the hidden size 5120 and intermediate size
32768 used for the benchmark shapes are assumptions, with the Core AI card's
6656 / 19968 / vocab 202048 kept as a second shape set (``GLIMMER_LAYER``,
with the attention's sigmoid gate as a fourth matrix of the q/k/v launch).

Large workloads (the FFN layer, the Q5_K layer sweep and the whole decode
step) are tiled from a pool of quantised super-blocks: super-block i of a
matrix is pool block (a*i + c) mod P, with (a odd, c) drawn from the matrix's
seed.  Every pool block is an independent N(0, 0.02) super-block quantised by
the rounding quantiser, so each matrix has the intended per-block statistics
without quantising 29.5 G weights on the host.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

BASE_SEED = 20260
GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

Q4_K, Q5_K, Q6_K, Q4_G128 = 0, 1, 2, 3
BLOCK_BYTES = {Q4_K: 144, Q5_K: 176, Q6_K: 210, Q4_G128: 136}
FORMAT_NAMES = {Q4_K: "Q4_K", Q5_K: "Q5_K", Q6_K: "Q6_K", Q4_G128: "Q4_G128"}


# --------------------------------------------------------------- generators

def _mix(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def splitmix64(seed: int, counters: np.ndarray) -> np.ndarray:
    """uint64 outputs for the given counters (0-based) of stream `seed`."""
    c = np.asarray(counters, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + (c + np.uint64(1)) * GOLDEN
    return _mix(z)


def derive_seed(*parts: int) -> int:
    """A 64-bit seed from a tuple of small integers (config, layer, matrix)."""
    s = BASE_SEED
    for p in parts:
        s = int(splitmix64(s, np.array([p], dtype=np.uint64))[0])
    return s


def uniform01(seed: int, start: int, n: int) -> np.ndarray:
    """n doubles in (0, 1] from counters start .. start+n-1."""
    z = splitmix64(seed, np.arange(start, start + n, dtype=np.uint64))
    return ((z >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)


def normal_f32(seed: int, n: int, sigma: float, start: int = 0) -> np.ndarray:
    """n fp32 draws of N(0, sigma^2): Box-Muller on counters 2i, 2i+1."""
    out = np.empty(n, dtype=np.float32)
    chunk = 1 << 22
    for s in range(0, n, chunk):
        m = min(chunk, n - s)
        u = uniform01(seed, 2 * (start + s), 2 * m)
        u1, u2 = u[0::2], u[1::2]
        out[s:s + m] = (np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2) * sigma).astype(np.float32)
    return out


def bf16_bits(a_f32: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns the uint16 bits."""
    u = np.ascontiguousarray(a_f32, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def weights_f32(seed: int, N: int, K: int, sigma: float = 0.02) -> np.ndarray:
    return normal_f32(seed, N * K, sigma).reshape(N, K)


def activations_bf16(seed: int, n_tok: int, K: int, heavy: bool = False) -> np.ndarray:
    """bf16 bits [n_tok][K] of N(0,1); heavy=True scales a Bernoulli(0.05)
    subset of entries by 20 (in fp32, before rounding)."""
    x = normal_f32(seed, n_tok * K, 1.0)
    if heavy:
        u = uniform01(derive_seed(seed, 7), 0, n_tok * K)
        x = np.where(u < 0.05, x * np.float32(20.0), x).astype(np.float32)
    return bf16_bits(x).reshape(n_tok, K)


def random_block_bytes(seed: int, fmt: int, n_blocks: int) -> np.ndarray:
    """Uniformly random bytes for n_blocks super-blocks, except that every
    fp16 field gets a finite value (exponent field != 31).  Exercises every
    bit of every field, negative Q6_K scales and extreme q included."""
    nb = BLOCK_BYTES[fmt]
    z = splitmix64(seed, np.arange((n_blocks * nb + 7) // 8, dtype=np.uint64))
    raw = z.view(np.uint8)[: n_blocks * nb].copy()
    if fmt == Q4_G128:
        q = raw[: n_blocks * 128]
        p = raw[n_blocks * 128:].reshape(n_blocks, 8)
        for off in (0, 2):          # d, dmin: clear one exponent bit if all set
            hi = p[:, off + 1]
            p[:, off + 1] = np.where((hi & 0x7C) == 0x7C, hi & 0xFB, hi)
        return np.concatenate([q, p.reshape(-1)])
    b = raw.reshape(n_blocks, nb)
    offs = {Q4_K: (0, 2), Q5_K: (0, 2), Q6_K: (208,)}[fmt]
    for off in offs:
        hi = b[:, off + 1]
        b[:, off + 1] = np.where((hi & 0x7C) == 0x7C, hi & 0xFB, hi)
    return b.reshape(-1)


# ----------------------------------------------------------- block tiling

def tile_params(seed: int, pool_blocks: int):
    """(a, c) of the tiling map i -> (a*i + c) mod pool_blocks (a odd)."""
    z = splitmix64(seed, np.array([0, 1], dtype=np.uint64))
    a = int(z[0] % np.uint64(1 << 30)) | 1
    c = int(z[1] % np.uint64(pool_blocks))
    return a, c


def tile_indices(seed: int, n_blocks: int, pool_blocks: int, start: int = 0) -> np.ndarray:
    assert pool_blocks & (pool_blocks - 1) == 0
    a, c = tile_params(seed, pool_blocks)
    i = np.arange(start, start + n_blocks, dtype=np.int64)
    return (i * a + c) & (pool_blocks - 1)


def tiled_rows(pool: np.ndarray, fmt: int, seed: int, N: int, K: int, rows) -> np.ndarray:
    """Host bytes of a tiled N x K matrix restricted to `rows` (returned as a
    len(rows) x K matrix in the same format)."""
    assert fmt != Q4_G128
    nb = BLOCK_BYTES[fmt]
    P = pool.size // nb
    nsb = K // 256
    pb = pool.reshape(P, nb)
    a, c = tile_params(seed, P)
    i = np.asarray(rows, dtype=np.int64)[:, None] * nsb + np.arange(nsb, dtype=np.int64)[None, :]
    return pb[(i * a + c) & (P - 1)].reshape(-1)


def pool_weights(seed: int, pool_blocks: int) -> np.ndarray:
    """fp32 [pool_blocks][256] of N(0, 0.02): the super-blocks of a pool."""
    return normal_f32(seed, pool_blocks * 256, 0.02).reshape(pool_blocks, 256)


# --------------------------------------------------------------- workloads

@dataclass(frozen=True)
class Matrix:
    name: str
    fmt: int
    N: int
    K: int

    @property
    def nbytes(self) -> int:
        return self.N * (self.K // 256) * BLOCK_BYTES[self.fmt]


HIDDEN, INTER, NQ, NKV, HEAD_DIM = 5120, 32768, 32, 2, 128
LAYERS, VOCAB = 52, 200000


def layer_matrices(fmt_attn: int, fmt_ffn: int, fmt_down: int, hidden: int = HIDDEN,
                   inter: int = INTER, nq: int = NQ, nkv: int = NKV, hd: int = HEAD_DIM):
    qd, kvd = nq * hd, nkv * hd
    return [Matrix("q", fmt_attn, qd, hidden), Matrix("k", fmt_attn, kvd, hidden),
            Matrix("v", fmt_attn, kvd, hidden), Matrix("o", fmt_attn, hidden, qd),
            Matrix("gate", fmt_ffn, inter, hidden), Matrix("up", fmt_ffn, inter, hidden),
            Matrix("down", fmt_down, hidden, inter)]


# C1..C5: the five benchmark shapes.
SINGLE_Q4K = [Matrix("w", Q4_K, 4096, 4096)]
ATTN_Q4K = layer_matrices(Q4_K, Q4_K, Q6_K)[:4] + [Matrix("q_g128", Q4_G128, 4096, HIDDEN)]
FFN_Q4K_Q6K = layer_matrices(Q4_K, Q4_K, Q6_K)[4:]
LAYER_Q5K = layer_matrices(Q5_K, Q5_K, Q5_K)
DECODE_LAYER = layer_matrices(Q4_K, Q4_K, Q6_K)
LM_HEAD = Matrix("lm_head", Q6_K, VOCAB, HIDDEN)


# The pages' own shapes (Core AI card, "The architecture, and what the port
# had to do about it"): hidden 6656, SwiGLU intermediate 19968, vocab 202048,
# 32 q / 2 kv heads of 128, and a sigmoid output gate of the attention read
# from the pre-attention hidden state, which the card folds with q, k and v
# into one qkvg projection (one launch of four matrices here).
GLIMMER_HIDDEN, GLIMMER_INTER, GLIMMER_VOCAB = 6656, 19968, 202048


def glimmer_layer(fmt_attn: int = Q4_K, fmt_ffn: int = Q4_K, fmt_down: int = Q6_K):
    L = layer_matrices(fmt_attn, fmt_ffn, fmt_down, hidden=GLIMMER_HIDDEN, inter=GLIMMER_INTER)
    q = L[0]
    return L[:3] + [Matrix("attn_gate", fmt_attn, q.N, q.K)] + L[3:]


GLIMMER_LAYER = glimmer_layer()
GLIMMER_HEAD = Matrix("lm_head", Q6_K, GLIMMER_VOCAB, GLIMMER_HIDDEN)


def glimmer_step_bytes(layers: int = LAYERS) -> int:
    return layers * sum(m.nbytes for m in GLIMMER_LAYER) + GLIMMER_HEAD.nbytes


def decode_step_bytes(layers: int = LAYERS) -> int:
    return layers * sum(m.nbytes for m in DECODE_LAYER) + LM_HEAD.nbytes


def decode_step_weights(layers: int = LAYERS) -> int:
    return layers * sum(m.N * m.K for m in DECODE_LAYER) + LM_HEAD.N * LM_HEAD.K


def weight_gb_per_s(weight_bytes: float, seconds: float) -> float:
    """Weight traffic in GB/s (1 GB = 1e9 bytes) for bytes streamed per step."""
    return weight_bytes / seconds / 1e9


# ------------------------------------------------------ device-side tiling

POOL_BLOCKS = 1 << 17


def tile_matrix_device(pool_dev, fmt: int, seed: int, N: int, K: int, out=None):
    """Device bytes of a tiled N x K matrix: super-block i is pool block
    (a*i + c) mod P (torch gather on the GPU; same map as tiled_rows)."""
    import torch
    assert fmt != Q4_G128
    nb = BLOCK_BYTES[fmt]
    P = pool_dev.numel() // nb
    nblk = N * (K // 256)
    a, c = tile_params(seed, P)
    pb = pool_dev.view(P, nb)
    if out is None:
        out = torch.empty(nblk * nb, dtype=torch.uint8, device=pool_dev.device)
    ov = out.view(nblk, nb)
    step = 1 << 22
    for s in range(0, nblk, step):
        m = min(step, nblk - s)
        i = torch.arange(s, s + m, dtype=torch.int64, device=pool_dev.device)
        idx = (i * a + c) & (P - 1)
        torch.index_select(pb, 0, idx, out=ov[s:s + m])
    return out
