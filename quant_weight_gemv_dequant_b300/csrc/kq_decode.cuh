// kq_decode.cuh -- device-side field decoding shared by the GEMV and the
// dequantisation kernels of libkq.
//
// The record layouts are the GGUF K-quant super-blocks named by the daily.dev
// ExecuTorch summary (answer on exporting GGUF checkpoints), with the byte
// placement written out in include/kq.h, plus this library's planar
// group-128 layout.  Every format is processed in "chunks" of 64 weights, four
// per 256-weight super-block:
//   Q4_K / Q5_K / Q4_G128 chunk c: weights 64c + r (r < 64); the low nibble
//     of byte 32c + r' is weight 64c + r', the high nibble weight 64c+32+r'.
//   Q6_K chunk c = 2h + u: weights 128h + 32t + l for t < 4, 16u <= l < 16u+16.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>

namespace kq {

constexpr int kQ4K = 0, kQ5K = 1, kQ6K = 2, kG128 = 3;

__host__ __device__ constexpr int block_bytes(int f) {
  return f == kQ4K ? 144 : f == kQ5K ? 176 : f == kQ6K ? 210 : 136;
}

__device__ __forceinline__ float half_bits_to_float(uint32_t bits16) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16)));
}

// 6-bit (scale, min) of sub-block j from the 12-byte field of Q4_K / Q5_K,
// given as three little-endian words s0 = bytes 0..3, s1 = 4..7, s2 = 8..11.
__device__ __forceinline__ void scale_min_6bit(uint32_t s0, uint32_t s1, uint32_t s2, int j,
                                               int& sc, int& m) {
  if (j < 4) {
    sc = (s0 >> (8 * j)) & 63;
    m = (s1 >> (8 * j)) & 63;
  } else {
    const int k = j - 4;
    const uint32_t lo = (s2 >> (8 * k)) & 0xFF;
    sc = (lo & 15) | (((s0 >> (8 * k + 6)) & 3) << 4);
    m = (lo >> 4) | (((s1 >> (8 * k + 6)) & 3) << 4);
  }
}

// Read-only 16-byte load that bypasses L1 allocation (streamed weights).
__device__ __forceinline__ uint4 ldg_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ldg_u16(const void* p) {
  unsigned short v;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

// 16 bytes from a 2-byte aligned address, as four little-endian words.
__device__ __forceinline__ void ldg16_align2(const uint8_t* p, uint32_t w[4]) {
  if ((reinterpret_cast<uintptr_t>(p) & 15) == 0) {
    const uint4 v = ldg_stream16(p);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = ldg_u16(p + 4 * i) | (ldg_u16(p + 4 * i + 2) << 16);
  }
}

}  // namespace kq
