// kq_gemv.cu -- K-quant GEMV and dequantisation kernels for sm_103a.
//
// y[t][n] = sum_k w^[n][k] x[t][k], fp32 accumulation (daily.dev ExecuTorch
// summary, answer on exporting GGUF checkpoints; record layouts in kq.h).
//
// Per sub-block the product is factored:  sum_i (a q_i - b) x_i
//   = a * sum_i q_i x_i - b * sum_i x_i,  with a = d*sc, b = dmin*m
// (Q6_K: a = d*sc applied to the signed q - 32, b = 0), so the per-weight work
// is one nibble decode and one FMA.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kq_decode.cuh"
#include "kq_kernels.cuh"

namespace kq {
namespace {

constexpr int kWarps = 8;   // rows per CTA: one warp per output row

// One 64-weight chunk decoded into segments that share (a, b).
template <int F>
struct Chunk {
  static constexpr int kSeg = (F == kQ6K) ? 4 : 2;      // segments per chunk
  static constexpr int kLen = 64 / kSeg;                // weights per segment
  float a[kSeg], b[kSeg];
  int k0[kSeg];                                         // k of segment start
  int q[64];                                            // signed q per weight
};

template <int F>
__device__ __forceinline__ void load_chunk(const uint8_t* W, int64_t qplane_bytes, int nsb,
                                           int64_t row, int sb, int c, Chunk<F>& ch) {
  const int64_t idx = row * nsb + sb;
  if constexpr (F == kQ4K || F == kQ5K) {
    const uint8_t* blk = W + idx * block_bytes(F);
    const uint4 hdr = ldg_stream16(blk);
    const float d = half_bits_to_float(hdr.x & 0xFFFF);
    const float dmin = half_bits_to_float(hdr.x >> 16);
    const int qoff = (F == kQ4K) ? 16 : 48;
    const uint4 q0 = ldg_stream16(blk + qoff + 32 * c);
    const uint4 q1 = ldg_stream16(blk + qoff + 32 * c + 16);
    const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    uint32_t hw[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if constexpr (F == kQ5K) {
      const uint4 h0 = ldg_stream16(blk + 16);
      const uint4 h1 = ldg_stream16(blk + 32);
      hw[0] = h0.x; hw[1] = h0.y; hw[2] = h0.z; hw[3] = h0.w;
      hw[4] = h1.x; hw[5] = h1.y; hw[6] = h1.z; hw[7] = h1.w;
    }
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      int sc, m;
      scale_min_6bit(hdr.y, hdr.z, hdr.w, 2 * c + s, sc, m);
      ch.a[s] = d * static_cast<float>(sc);
      ch.b[s] = dmin * static_cast<float>(m);
      ch.k0[s] = sb * 256 + 64 * c + 32 * s;
    }
#pragma unroll
    for (int r = 0; r < 32; ++r) {
      const uint32_t byte = (qw[r >> 2] >> (8 * (r & 3))) & 0xFF;
      int lo = byte & 15, hi = byte >> 4;
      if constexpr (F == kQ5K) {
        const uint32_t hb = (hw[r >> 2] >> (8 * (r & 3))) & 0xFF;
        lo |= ((hb >> (2 * c)) & 1) << 4;
        hi |= ((hb >> (2 * c + 1)) & 1) << 4;
      }
      ch.q[r] = lo;
      ch.q[32 + r] = hi;
    }
  } else if constexpr (F == kG128) {
    const uint8_t* qs = W + idx * 128 + 32 * c;
    const uint8_t* par = W + qplane_bytes + idx * 8;
    const uint32_t p0 = ldg_u16(par) | (ldg_u16(par + 2) << 16);
    const uint32_t p1 = ldg_u16(par + 4) | (ldg_u16(par + 6) << 16);
    const float d = half_bits_to_float(p0 & 0xFFFF);
    const float dmin = half_bits_to_float(p0 >> 16);
    const int g = c >> 1;
    const int sc = (p1 >> (8 * g)) & 0xFF;
    const int m = (p1 >> (16 + 8 * g)) & 0xFF;
    const uint4 q0 = ldg_stream16(qs);
    const uint4 q1 = ldg_stream16(qs + 16);
    const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      ch.a[s] = d * static_cast<float>(sc);
      ch.b[s] = dmin * static_cast<float>(m);
      ch.k0[s] = sb * 256 + 64 * c + 32 * s;
    }
#pragma unroll
    for (int r = 0; r < 32; ++r) {
      const uint32_t byte = (qw[r >> 2] >> (8 * (r & 3))) & 0xFF;
      ch.q[r] = byte & 15;
      ch.q[32 + r] = byte >> 4;
    }
  } else {  // Q6_K
    const uint8_t* blk = W + idx * 210;
    const int h = c >> 1, u = c & 1;
    uint32_t A[4], B[4], H[4];
    ldg16_align2(blk + 64 * h + 16 * u, A);
    ldg16_align2(blk + 64 * h + 32 + 16 * u, B);
    ldg16_align2(blk + 128 + 32 * h + 16 * u, H);
    const float d = half_bits_to_float(ldg_u16(blk + 208));
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int sidx = 8 * h + 2 * t + u;
      const int8_t sc = static_cast<int8_t>(ldg_u16(blk + 192 + (sidx & ~1)) >> (8 * (sidx & 1)));
      ch.a[t] = d * static_cast<float>(sc);
      ch.b[t] = 0.0f;
      ch.k0[t] = sb * 256 + 128 * h + 32 * t + 16 * u;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int sh = 8 * (i & 3);
      const uint32_t a = (A[i >> 2] >> sh) & 0xFF, b = (B[i >> 2] >> sh) & 0xFF;
      const uint32_t hb = (H[i >> 2] >> sh) & 0xFF;
      ch.q[i] = static_cast<int>((a & 15) | ((hb & 3) << 4)) - 32;
      ch.q[16 + i] = static_cast<int>((b & 15) | (((hb >> 2) & 3) << 4)) - 32;
      ch.q[32 + i] = static_cast<int>((a >> 4) | (((hb >> 4) & 3) << 4)) - 32;
      ch.q[48 + i] = static_cast<int>((b >> 4) | (((hb >> 6) & 3) << 4)) - 32;
    }
  }
}

__device__ __forceinline__ float bf16_to_float(uint16_t v) {
  return __uint_as_float(static_cast<uint32_t>(v) << 16);
}

template <int F, int NT>
__global__ void __launch_bounds__(kWarps * 32)
gemv_warp_row(GemvGroup g, const uint16_t* __restrict__ x, int K, int nt) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int64_t row = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
  int mi = 0;
  while (mi < g.count - 1 && row >= g.N[mi]) {
    row -= g.N[mi];
    ++mi;
  }
  if (row >= g.N[mi]) return;
  const uint8_t* W = g.W[mi];
  const int N = g.N[mi];
  const int nsb = K >> 8;
  const int64_t qplane = static_cast<int64_t>(N) * nsb * 128;
  float acc[NT];
#pragma unroll
  for (int t = 0; t < NT; ++t) acc[t] = 0.0f;
  for (int p = lane; p < 4 * nsb; p += 32) {
    Chunk<F> ch;
    load_chunk<F>(W, qplane, nsb, row, p >> 2, p & 3, ch);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      if (t < nt) {
        const uint16_t* xt = x + static_cast<int64_t>(t) * K;
#pragma unroll
        for (int s = 0; s < Chunk<F>::kSeg; ++s) {
          float dot = 0.0f, sx = 0.0f;
#pragma unroll
          for (int i = 0; i < Chunk<F>::kLen; ++i) {
            const float xv = bf16_to_float(xt[ch.k0[s] + i]);
            dot = fmaf(static_cast<float>(ch.q[s * Chunk<F>::kLen + i]), xv, dot);
            sx += xv;
          }
          acc[t] = fmaf(ch.a[s], dot, acc[t]);
          acc[t] = fmaf(-ch.b[s], sx, acc[t]);
        }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    float v = acc[t];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    if (lane == 0 && t < nt) g.y[mi][static_cast<int64_t>(t) * N + row] = v;
  }
}

// Dequantisation: one thread per chunk.  Q4_K / Q5_K / Q4_G128 compute
// fmaf(d*sc, q, -(dmin*m)): d*sc and dmin*m are exact in fp32, so the single
// rounding of the fma is the round-to-nearest of the exact value.  Q6_K
// computes (d*sc)*(q-32), which is exact.
template <int F>
__global__ void dequant_chunks(const uint8_t* __restrict__ W, float* __restrict__ out, int N,
                               int K) {
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int nsb = K >> 8;
  const int64_t total = static_cast<int64_t>(N) * nsb * 4;
  if (gid >= total) return;
  const int64_t row = gid / (4 * nsb);
  const int p = static_cast<int>(gid % (4 * nsb));
  const int64_t qplane = static_cast<int64_t>(N) * nsb * 128;
  Chunk<F> ch;
  load_chunk<F>(W, qplane, nsb, row, p >> 2, p & 3, ch);
  float* o = out + row * K;
#pragma unroll
  for (int s = 0; s < Chunk<F>::kSeg; ++s)
#pragma unroll
    for (int i = 0; i < Chunk<F>::kLen; ++i) {
      const float q = static_cast<float>(ch.q[s * Chunk<F>::kLen + i]);
      o[ch.k0[s] + i] = (F == kQ6K) ? ch.a[s] * q : fmaf(ch.a[s], q, -ch.b[s]);
    }
}

template <int F, int NT>
void launch_t(const GemvGroup& g, const uint16_t* x, int K, int n_tok, cudaStream_t s) {
  int64_t rows = 0;
  for (int i = 0; i < g.count; ++i) rows += g.N[i];
  const int64_t blocks = (rows + kWarps - 1) / kWarps;
  // Row tiles must not straddle matrices: pad each matrix to a multiple of
  // kWarps rows by launching per-matrix when N is not a multiple.
  bool aligned = true;
  for (int i = 0; i + 1 < g.count; ++i) aligned &= (g.N[i] % kWarps) == 0;
  if (aligned) {
    gemv_warp_row<F, NT><<<static_cast<unsigned>(blocks), kWarps * 32, 0, s>>>(g, x, K, n_tok);
  } else {
    for (int i = 0; i < g.count; ++i) {
      GemvGroup one{};
      one.count = 1;
      one.W[0] = g.W[i];
      one.y[0] = g.y[i];
      one.N[0] = g.N[i];
      const int64_t b = (g.N[i] + kWarps - 1) / kWarps;
      gemv_warp_row<F, NT><<<static_cast<unsigned>(b), kWarps * 32, 0, s>>>(one, x, K, n_tok);
    }
  }
}

template <int F>
void launch_f(const GemvGroup& g, const uint16_t* x, int K, int n_tok, cudaStream_t s) {
  if (n_tok <= 1) launch_t<F, 1>(g, x, K, n_tok, s);
  else if (n_tok <= 2) launch_t<F, 2>(g, x, K, n_tok, s);
  else if (n_tok <= 4) launch_t<F, 4>(g, x, K, n_tok, s);
  else if (n_tok <= 8) launch_t<F, 8>(g, x, K, n_tok, s);
  else launch_t<F, 16>(g, x, K, n_tok, s);
}

}  // namespace

StreamResult launch_gemv(int fmt, const GemvGroup& g, const uint16_t* x, int K, int n_tok,
                         cudaStream_t s, bool noalloc) {
  const StreamResult r = launch_stream(fmt, g, x, K, n_tok, s, noalloc);
  if (r != StreamResult::kNotServed) return r;
  // a shape the streaming kernels decline (x too large for shared memory
  // even in bf16): the warp-per-row kernel, which overwrites every output
  switch (fmt) {
    case kQ4K: launch_f<kQ4K>(g, x, K, n_tok, s); break;
    case kQ5K: launch_f<kQ5K>(g, x, K, n_tok, s); break;
    case kQ6K: launch_f<kQ6K>(g, x, K, n_tok, s); break;
    case kG128: launch_f<kG128>(g, x, K, n_tok, s); break;
    default: return StreamResult::kNotServed;
  }
  return StreamResult::kLaunched;
}

void launch_dequant(int fmt, const uint8_t* W, float* out, int N, int K, cudaStream_t s) {
  const int64_t total = static_cast<int64_t>(N) * (K / 256) * 4;
  const unsigned blocks = static_cast<unsigned>((total + 255) / 256);
  switch (fmt) {
    case kQ4K: dequant_chunks<kQ4K><<<blocks, 256, 0, s>>>(W, out, N, K); break;
    case kQ5K: dequant_chunks<kQ5K><<<blocks, 256, 0, s>>>(W, out, N, K); break;
    case kQ6K: dequant_chunks<kQ6K><<<blocks, 256, 0, s>>>(W, out, N, K); break;
    default: dequant_chunks<kG128><<<blocks, 256, 0, s>>>(W, out, N, K); break;
  }
}

}  // namespace kq
