// kq_stream.cu -- the streaming K-quant GEMV kernel for sm_103a
// (n_tok = 1, 2, 4 on CUDA cores).
//
// y[t][n] = sum_k w^[n][k] x[t][k]  (daily.dev ExecuTorch summary, answer on
// exporting GGUF checkpoints; the Core AI card's 424 GB/s arithmetic shows the
// product is bound by streaming the packed weights once).
//
// Structure.  The rows of the (grouped) matrices are cut into tiles of
// 2 * kWC * RT rows; a tile is streamed in slabs of 16 "units" (a unit = kCW
// weights of one row, kCW = 64 / NT).  One CTA = kWC consumer warps + 1
// producer warp, persistent over its tiles:
//   * at start, all warps convert x (bf16) once into shared memory (fp32, or
//     bf16 when fp32 would not fit) together with the sum of x over every
//     sub-block part (for the min term), while the first stages' weights are
//     already in flight;
//   * the producer warp copies every row segment of a (tile, slab) stage into
//     a ring of shared-memory slots with cp.async.bulk (16-byte aligned spans;
//     a record that does not start on 16 bytes is copied with its aligned
//     halo);
//   * each consumer half-warp owns RT rows of the tile, each lane one unit
//     position of the slab, so the lane's x values stay in registers across
//     its rows.  Per row: decode the unit's scales, turn every q into an
//     exact fp32 value with the 2^23 magic number and one packed
//     fma.rn.f32x2 (scale 2^-s, offset), and accumulate with packed fmas;
//   * after the tile's last slab, the 16 lanes of a half-warp reduce with
//     shuffles and write y.
// Stages are handed over with mbarriers (full: producer -> consumers with the
// bulk-copy byte count; empty: consumers -> producer).  Every wait is bounded
// and records a timeout in a device word that kq_device_status reads.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kq_decode.cuh"
#include "kq_kernels.cuh"

namespace kq {

__device__ unsigned int g_wait_timeouts = 0;

namespace {

constexpr int kWC = 4;                  // consumer warps per CTA
constexpr int kThreads = (kWC + 1) * 32;
constexpr long long kWaitCycles = 4000000000LL;   // ~2 s at 2 GHz

// ------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2; "
      "selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded, warp-uniform wait (every lane of the warp calls it): true once
// the phase with this parity has completed for all lanes; false, with a
// recorded timeout, if that takes longer than kWaitCycles.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity) {
  long long t0 = 0;
  for (int i = 0;; ++i) {
    const bool done = mbar_try(bar, parity);
    if (__all_sync(0xFFFFFFFFu, done)) return true;
    if (i == 0) {
      t0 = clock64();
    } else if (__shfl_sync(0xFFFFFFFFu, (clock64() - t0 > kWaitCycles) ? 1 : 0, 0)) {
      if ((threadIdx.x & 31) == 0) atomicAdd(&g_wait_timeouts, 1u);
      return false;
    }
  }
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ float4 lds_f4(uint32_t a) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(a));
  return v;
}
__device__ __forceinline__ float2 lds_f2(uint32_t a) {
  float2 v;
  asm volatile("ld.shared.v2.f32 {%0,%1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a));
  return v;
}

// n consecutive 32-bit words from a 2-byte aligned shared address.
template <int N>
__device__ __forceinline__ void lds_words_a2(uint32_t a, uint32_t (&w)[N]) {
  const uint32_t base = a & ~3u, sh = (a & 3u) * 8u;
  uint32_t raw[N + 1];
#pragma unroll
  for (int i = 0; i <= N; ++i) raw[i] = lds32(base + 4 * i);
#pragma unroll
  for (int i = 0; i < N; ++i) w[i] = __funnelshift_r(raw[i], raw[i + 1], sh);
}

// One LOP3 each.  Written as PTX with every operand in a register: with two
// immediate operands the compiler splits (w & mask) | magic into two
// instructions, which doubles the integer work per weight.
__device__ __forceinline__ uint32_t lop_mask_or(uint32_t w, uint32_t mask, uint32_t magic) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(w), "r"(mask), "r"(magic));
  return d;   // (w & mask) | magic
}
__device__ __forceinline__ uint32_t bitsel(uint32_t a, uint32_t b, uint32_t m) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xE4;" : "=r"(d) : "r"(a), "r"(b), "r"(m));
  return d;   // (a & m) | (b & ~m)
}

__device__ __forceinline__ float2 f2(uint32_t a, uint32_t b) {
  return make_float2(__uint_as_float(a), __uint_as_float(b));
}

// 2^23 magic: as_float(0x4B000000 | (q << s)) = 2^23 + q 2^s (q 2^s < 2^23),
// and subtracting 2^23 leaves q 2^s exactly.
constexpr uint32_t kMagic = 0x4B000000u;
__host__ __device__ constexpr float pow2(int e) {
  return e >= 0 ? static_cast<float>(1ull << e) : 1.0f / static_cast<float>(1ull << (-e));
}

// -------------------------------------------------------------- geometry

template <int F, int NT, int RT>
struct Geo {
  static constexpr int kRows = 2 * kWC * RT;             // rows per tile
  static constexpr int kCW = 64 / NT;                    // weights per unit
  // x positions per part sum: one sub-block part of a unit (Q4 family:
  // kCW/2 low or high nibbles; Q6_K: the kCW/4 weights of one t-run)
  static constexpr int kPart = (F == kQ6K) ? kCW / 4 : kCW / 2;
  static constexpr int kUnitsPerSB = 256 / kCW;          // 4, 8, 16
  static constexpr int kSlabSB = 16 / kUnitsPerSB;       // super-blocks per slab: 4, 2, 1
  static constexpr int kSlabK = 256 * kSlabSB;           // 1024, 512, 256
  static constexpr int kBB = block_bytes(F);
  // per-row shared slot (16-byte aligned): records (+ halo for unaligned
  // starts); G128 keeps the q plane and the param plane in separate parts.
  static constexpr int kQBytes = (F == kG128) ? 128 * kSlabSB : kBB * kSlabSB;
  static constexpr int kSlot = ((kQBytes + 16 + 15) / 16) * 16;
  static constexpr int kPSlot = (F == kG128) ? ((8 * kSlabSB + 16 + 15) / 16) * 16 : 0;
  static constexpr int kStage = kRows * (kSlot + kPSlot);
};

struct Tile {
  int mi;      // matrix of the group
  int row0;    // first row in that matrix
  int rcnt;    // rows in this tile
};

// Select element i (< kMaxGroup) of a small parameter array without
// dynamic indexing (which would force the array into local memory).
template <typename T>
__device__ __forceinline__ T pick(const T (&a)[kMaxGroup], int i) {
  return i == 0 ? a[0] : i == 1 ? a[1] : i == 2 ? a[2] : a[3];
}

struct Params {
  GemvGroup g;
  const uint16_t* x;         // bf16 [nt][K]
  int K, nsb, nt;
  int slabs;                 // slabs of one K segment
  int kpad;                  // staged x positions per token (one K segment)
  int ksplit;                // K segments (CTA c works on segment c % ksplit)
  int tiles;
  int tile_rows;             // rows per tile (<= the CTA's 2 * kWC * RT)
  int tile_end[kMaxGroup];   // cumulative tile counts per matrix
  uint32_t x_bytes;          // shared bytes of the staged x (+ part sums), 16-aligned
  float* part;               // split-K partial sums [ksplit][tiles][tile_rows][NT]
  unsigned int* arrivals;    // split-K per-tile arrival counters (left at zero)
};

__device__ __forceinline__ Tile tile_of(const Params& p, int t) {
  int mi = 0, base = 0;
#pragma unroll
  for (int i = 0; i < kMaxGroup - 1; ++i)
    if (i < p.g.count - 1 && t >= p.tile_end[i]) {
      mi = i + 1;
      base = p.tile_end[i];
    }
  Tile r;
  r.mi = mi;
  r.row0 = (t - base) * p.tile_rows;
  r.rcnt = min(p.tile_rows, pick(p.g.N, mi) - r.row0);
  return r;
}

// ----------------------------------------------------------- x staging

// Bit position s at which the consumers extract the q that multiplies x at
// byte b (= position % 4) of a word, in the low (lo) or high half of a Q4
// family chunk.  Q4_K / G128 low nibbles come from w (b0 s=0, b1 s=8, b2
// s=16) and w >> 12 (b3 s=12); high nibbles from w (b0 s=4, b1 s=12) and
// w >> 12 (b2 s=8, b3 s=16).  Q5_K and Q6_K extract whole bytes (b3 from
// w >> 8).  x is staged pre-scaled by 2^-s, so (2^23 + q 2^s) - 2^23 = q 2^s
// times the staged x is exactly q x.
template <int F>
__host__ __device__ constexpr int field_shift(bool lo, int b) {
  if (F == kQ5K || F == kQ6K) return b == 0 ? 0 : b == 1 ? 8 : 16;
  if (lo) return b == 0 ? 0 : b == 1 ? 8 : b == 2 ? 16 : 12;
  return b == 0 ? 4 : b == 1 ? 12 : b == 2 ? 8 : 16;
}

// Shared-memory layout of the staged activations.  Value i (= token * kpad
// + position) sits at byte i * kE + kPad * (i / kPer): the padding staggers
// the 16 units of a half-warp over all bank groups, so every x load of the
// consumers is conflict-free (Q4 family: 16 B per 64 values, Q6_K: 16 B per
// 128 values; half of that for bf16).  When kInterleave, each aligned group
// of 8 positions is stored as x0 x4 x1 x5 x2 x6 x3 x7, so one 16-byte load
// yields the two (word j, word j+1) pairs that the packed fmas consume.
template <int F, int NT, bool XBF>
struct XLayout {
  static constexpr int kE = XBF ? 2 : 4;
  static constexpr int kPer = (F == kQ6K) ? 128 : 64;
  static constexpr int kPad = XBF ? 8 : 16;
  static constexpr bool kInterleave = (F == kQ6K) ? (NT <= 2) : true;
  __host__ __device__ static constexpr size_t bytes(size_t n) { return n * kE + kPad * (n / kPer); }
  __device__ static uint32_t addr(int i) {
    return static_cast<uint32_t>(i * kE + kPad * (i / kPer));
  }
};

// X (layout above) followed by SX: [NT][kpad/kPart] fp32 part sums.
// Entries beyond K or for tokens >= nt are zero.
template <int F, int NT, int RT, bool XBF>
__device__ void stage_x(const Params& p, uint8_t* smem, int kbase) {
  using G = Geo<F, NT, RT>;
  using L = XLayout<F, NT, XBF>;
  constexpr int P = G::kPart;                 // positions per part sum (>= 4)
  constexpr int CH = P > 8 ? P : 8;           // positions per work item
  constexpr int NS = CH / P;                  // part sums per work item
  const int parts_per_tok = p.kpad / P;
  const int items_per_tok = p.kpad / CH;
  float* sx = reinterpret_cast<float*>(smem + L::bytes(static_cast<size_t>(NT) * p.kpad));
  for (int q = threadIdx.x; q < NT * items_per_tok; q += blockDim.x) {
    const int tk = q / items_per_tok, k0 = (q % items_per_tok) * CH;
    const uint16_t* xt = p.x + static_cast<int64_t>(tk) * p.K + kbase + k0;
    const bool live = tk < p.nt && kbase + k0 < p.K;
    float sums[NS];
#pragma unroll
    for (int n = 0; n < NS; ++n) sums[n] = 0.0f;
#pragma unroll
    for (int i = 0; i < CH; i += 8) {
      uint4 raw = make_uint4(0, 0, 0, 0);
      if (live) raw = *reinterpret_cast<const uint4*>(xt + i);
      uint32_t r[4] = {raw.x, raw.y, raw.z, raw.w};
      float v[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[2 * j] = __uint_as_float(r[j] << 16);
        v[2 * j + 1] = __uint_as_float(r[j] & 0xFFFF0000u);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) sums[(i + j) / P] += v[j];
      // pre-scale by 2^-s, s = bit position at which the consumers extract
      // the q of this x (exact: a power of two)
      const bool lo = ((k0 + i) & 63) < 32;
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] *= pow2(-field_shift<F>(lo, j & 3));
      const int idx = tk * p.kpad + k0 + i;   // first of an aligned group of 8
      uint8_t* d = smem + L::addr(idx);
      if constexpr (XBF) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          r[j] = (__float_as_uint(v[2 * j]) >> 16) | (__float_as_uint(v[2 * j + 1]) & 0xFFFF0000u);
        uint4 o = make_uint4(r[0], r[1], r[2], r[3]);
        if (L::kInterleave)   // bf16 pairs (x0,x4) (x1,x5) (x2,x6) (x3,x7)
          o = make_uint4(__byte_perm(r[0], r[2], 0x5410), __byte_perm(r[0], r[2], 0x7632),
                         __byte_perm(r[1], r[3], 0x5410), __byte_perm(r[1], r[3], 0x7632));
        // the bf16 layout pads by 8 bytes: a group start is 8-byte aligned
        uint2* d2 = reinterpret_cast<uint2*>(d);
        d2[0] = make_uint2(o.x, o.y);
        d2[1] = make_uint2(o.z, o.w);
      } else {
        float4* d4 = reinterpret_cast<float4*>(d);
        if (L::kInterleave) {
          d4[0] = make_float4(v[0], v[4], v[1], v[5]);
          d4[1] = make_float4(v[2], v[6], v[3], v[7]);
        } else {
          d4[0] = make_float4(v[0], v[1], v[2], v[3]);
          d4[1] = make_float4(v[4], v[5], v[6], v[7]);
        }
      }
    }
#pragma unroll
    for (int n = 0; n < NS; ++n) sx[tk * parts_per_tok + k0 / P + n] = sums[n];
  }
}

// The four values stored at slots idx .. idx+3 (idx a multiple of 4) as two
// float2 pairs.
template <int F, int NT, bool XBF>
__device__ __forceinline__ void x_quad(uint32_t xs, int idx, float2& a, float2& b) {
  using L = XLayout<F, NT, XBF>;
  if constexpr (XBF) {
    const uint2 r = lds64(xs + L::addr(idx));
    a = make_float2(__uint_as_float(r.x << 16), __uint_as_float(r.x & 0xFFFF0000u));
    b = make_float2(__uint_as_float(r.y << 16), __uint_as_float(r.y & 0xFFFF0000u));
  } else {
    const float4 v = lds_f4(xs + L::addr(idx));
    a = make_float2(v.x, v.y);
    b = make_float2(v.z, v.w);
  }
}

// ------------------------------------------------------------- producer

template <int F, int NT, int RT>
__device__ __forceinline__ void issue_stage(const Params& p, uint8_t* smem, uint32_t st_a,
                                            uint32_t full, const Tile& tl, int sl) {
  using G = Geo<F, NT, RT>;
  const int lane = threadIdx.x & 31;
  const uint8_t* W = pick(p.g.W, tl.mi);
  const int64_t N = pick(p.g.N, tl.mi);
  const int sb0 = sl * G::kSlabSB;
  const int nsb_here = min(G::kSlabSB, p.nsb - sb0);
  uint32_t tx = 0;
  if (lane < tl.rcnt) {   // lane r copies row r of the tile
    const int64_t idx = (tl.row0 + lane) * static_cast<int64_t>(p.nsb) + sb0;
    auto copy_span = [&](const uint8_t* plane, int64_t plane_bytes, int64_t off, int len,
                         uint32_t dst) {
      const int64_t lo_off = off & ~int64_t{15};
      const int64_t end = off + len;
      int64_t hi = (end + 15) & ~int64_t{15};
      const int64_t cap = plane_bytes & ~int64_t{15};
      if (hi > cap) hi = cap;
      if (hi > lo_off) {
        const uint32_t n = static_cast<uint32_t>(hi - lo_off);
        bulk_g2s(dst, plane + lo_off, n, full);
        tx += n;
      }
      // bytes past the plane's last 16-byte boundary: plain loads
      for (int64_t b = (hi > lo_off ? hi : lo_off); b < end; ++b)
        smem[(dst - smem_addr(smem)) + (b - lo_off)] = __ldg(plane + b);
    };
    if constexpr (F == kG128) {
      const int64_t total = N * p.nsb;
      copy_span(W, total * 128, idx * 128, nsb_here * 128, st_a + lane * G::kSlot);
      copy_span(W + total * 128, total * 8, idx * 8, nsb_here * 8,
                st_a + G::kRows * G::kSlot + lane * G::kPSlot);
    } else {
      copy_span(W, N * p.nsb * G::kBB, idx * G::kBB, nsb_here * G::kBB, st_a + lane * G::kSlot);
    }
  }
  mbar_arrive_tx(full, tx);   // every producer lane arrives (count 32)
}

// ------------------------------------------------------------- consumers

// 6-bit (sc, m) of sub-blocks 2c and 2c+1 from the 12-byte field words s0,
// s1, s2 (bytes 0-3, 4-7, 8-11), two bytes each in the low 16 bits.
__device__ __forceinline__ void scale_pairs(uint32_t s0, uint32_t s1, uint32_t s2, int c,
                                            uint32_t& sc, uint32_t& mn) {
  const int sh = 16 * (c & 1);
  const uint32_t a0 = s0 >> sh, a1 = s1 >> sh, a2 = s2 >> sh;
  if (c < 2) {
    sc = a0 & 0x3F3Fu;
    mn = a1 & 0x3F3Fu;
  } else {
    sc = (a2 & 0x0F0Fu) | ((a0 >> 2) & 0x3030u);
    mn = ((a2 >> 4) & 0x0F0Fu) | ((a1 >> 2) & 0x3030u);
  }
}

template <int NW>
__device__ __forceinline__ void lds_words(uint32_t a, uint32_t (&w)[NW]) {
  if constexpr (NW == 8) {
    const uint4 v0 = lds128(a), v1 = lds128(a + 16);
    w[0] = v0.x; w[1] = v0.y; w[2] = v0.z; w[3] = v0.w;
    w[4] = v1.x; w[5] = v1.y; w[6] = v1.z; w[7] = v1.w;
  } else if constexpr (NW == 4) {
    const uint4 v0 = lds128(a);
    w[0] = v0.x; w[1] = v0.y; w[2] = v0.z; w[3] = v0.w;
  } else {
    const uint2 v0 = lds64(a);
    w[0] = v0.x; w[1] = v0.y;
  }
}

__device__ __forceinline__ uint64_t u64(uint32_t lo, uint32_t hi) {
  return (static_cast<uint64_t>(hi) << 32) | lo;
}
__device__ __forceinline__ float2 as_f2(uint64_t v) {
  return make_float2(__uint_as_float(static_cast<uint32_t>(v)),
                     __uint_as_float(static_cast<uint32_t>(v >> 32)));
}
__device__ __forceinline__ uint64_t bitsel64(uint64_t a, uint64_t b, uint32_t m) {
  return u64(bitsel(static_cast<uint32_t>(a), static_cast<uint32_t>(b), m),
             bitsel(static_cast<uint32_t>(a >> 32), static_cast<uint32_t>(b >> 32), m));
}
// exact q 2^s for the field at bit s of both halves of v (width mask m):
// one LOP3 per half builds 2^23 + q 2^s in a register pair, one packed add
// of (-2^23, -2^23) removes the offset; the same constant pair serves every
// field position.
__device__ __forceinline__ float2 conv64(uint64_t v, uint32_t m) {
  float2 r;
  asm("{\n\t.reg .b32 t0, t1;\n\t.reg .b64 p, q;\n\t"
      "lop3.b32 t0, %2, %4, %5, 0xEA;\n\t"
      "lop3.b32 t1, %3, %4, %5, 0xEA;\n\t"
      "mov.b64 p, {t0, t1};\n\t"
      "add.rn.f32x2 q, p, %6;\n\t"
      "mov.b64 {%0, %1}, q;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "r"(static_cast<uint32_t>(v)), "r"(static_cast<uint32_t>(v >> 32)), "r"(m),
        "r"(kMagic), "l"(0xCB000000CB000000ull));
  return r;
}

// Q4_K / Q5_K / Q4_G128 unit: kCW/2 bytes of the qs (chunk c, byte offset
// off): low nibbles -> sub-block 2c (weights 64c + off + i), high nibbles ->
// sub-block 2c+1 (weights 64c + 32 + off + i).  Words are taken in pairs
// (2i, 2i+1) as 64-bit values, so each conversion and each accumulation is
// one packed fma on a register pair.  xl[t][i][b] / xh[t][i][b] are the x
// pairs of nibble position b of that word pair; alo/ahi hold two partial
// sums per sub-block (word pairs alternate between them).
template <int F, int NT, int NW>
__device__ __forceinline__ void unit_q4(const uint32_t (&w)[NW], const uint32_t (&h)[NW], int c,
                                        const float2 (&xl)[NT][NW / 2][4],
                                        const float2 (&xh)[NT][NW / 2][4], float2 (&alo)[2][NT],
                                        float2 (&ahi)[2][NT]) {
#pragma unroll
  for (int i = 0; i < NW / 2; ++i) {
    const uint64_t W = u64(w[2 * i], w[2 * i + 1]);
    float2 ql[4], qh[4];
    if constexpr (F == kQ5K) {
      // byte b of lo5 / hi5 = nibble | fifth bit << 4 (bits 5..7 are masked
      // off by the 5-bit extraction masks below)
      const int rlo = (2 * c + 28) & 31, rhi = (2 * c + 29) & 31;   // rotate bit 2c(+1) to 4
      const uint64_t RL = u64(__funnelshift_r(h[2 * i], h[2 * i], rlo),
                              __funnelshift_r(h[2 * i + 1], h[2 * i + 1], rlo));
      const uint64_t RH = u64(__funnelshift_r(h[2 * i], h[2 * i], rhi),
                              __funnelshift_r(h[2 * i + 1], h[2 * i + 1], rhi));
      const uint32_t M = 0x0F0F0F0Fu;
      const uint64_t L5 = bitsel64(W, RL, M), H5 = bitsel64(W >> 4, RH, M);
      const uint64_t L5s = L5 >> 8, H5s = H5 >> 8;
      ql[0] = conv64(L5, 0x1Fu);
      ql[1] = conv64(L5, 0x1F00u);
      ql[2] = conv64(L5, 0x1F0000u);
      ql[3] = conv64(L5s, 0x1F0000u);
      qh[0] = conv64(H5, 0x1Fu);
      qh[1] = conv64(H5, 0x1F00u);
      qh[2] = conv64(H5, 0x1F0000u);
      qh[3] = conv64(H5s, 0x1F0000u);
    } else {
      // in W: lo b0 s=0, lo b1 s=8, lo b2 s=16, hi b0 s=4, hi b1 s=12;
      // in W >> 12 (bits crossing the halves land above bit 19 and are
      // masked off): lo b3 s=12, hi b2 s=8, hi b3 s=16
      const uint64_t B = W >> 12;
      ql[0] = conv64(W, 0xFu);
      ql[1] = conv64(W, 0xF00u);
      ql[2] = conv64(W, 0xF0000u);
      ql[3] = conv64(B, 0xF000u);
      qh[0] = conv64(W, 0xF0u);
      qh[1] = conv64(W, 0xF000u);
      qh[2] = conv64(B, 0xF00u);
      qh[3] = conv64(B, 0xF0000u);
    }
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        alo[i & 1][t] = __ffma2_rn(ql[b], xl[t][i][b], alo[i & 1][t]);
        ahi[i & 1][t] = __ffma2_rn(qh[b], xh[t][i][b], ahi[i & 1][t]);
      }
  }
}

// One stage of a Q4_K / Q5_K / Q4_G128 tile for this thread's rows.
template <int F, int NT, int RT, bool XBF>
__device__ __forceinline__ void stage_q4(const Params& p, const Tile& tl, int sl, int xsl,
                                         uint32_t st, uint32_t xs, int hw, int sbl, int c,
                                         int off, float (&acc)[RT][NT]) {
  using G = Geo<F, NT, RT>;
  using L = XLayout<F, NT, XBF>;
  constexpr int kCW = G::kCW, NW = kCW / 8;
  float2 xl[NT][NW / 2][4], xh[NT][NW / 2][4];
  float sxlo[NT], sxhi[NT];
  const int k0 = xsl * G::kSlabK + sbl * 256 + 64 * c + off;   // first lo position (staged x)
  const uint32_t sxa = xs + static_cast<uint32_t>(L::bytes(static_cast<size_t>(NT) * p.kpad));
  const int parts = p.kpad / G::kPart;
#pragma unroll
  for (int k = 0; k < NT; ++k) {
#pragma unroll
    for (int i = 0; i < NW / 2; ++i) {
      const int g = k * p.kpad + k0 + 8 * i;   // aligned group of 8 (interleaved)
      x_quad<F, NT, XBF>(xs, g, xl[k][i][0], xl[k][i][1]);
      x_quad<F, NT, XBF>(xs, g + 4, xl[k][i][2], xl[k][i][3]);
      x_quad<F, NT, XBF>(xs, g + 32, xh[k][i][0], xh[k][i][1]);
      x_quad<F, NT, XBF>(xs, g + 36, xh[k][i][2], xh[k][i][3]);
    }
    sxlo[k] = __uint_as_float(lds32(sxa + 4 * (k * parts + k0 / G::kPart)));
    sxhi[k] = __uint_as_float(lds32(sxa + 4 * (k * parts + (k0 + 32) / G::kPart)));
  }
#pragma unroll
  for (int r = 0; r < RT; ++r) {
    const int row = hw + 2 * kWC * r;
    if (row < tl.rcnt) {
      const uint32_t rs = st + row * G::kSlot;
      uint32_t w[NW], hq[NW];
      float2 dsc, dmn;
#pragma unroll
      for (int j = 0; j < NW; ++j) hq[j] = 0;
      if constexpr (F == kG128) {
        lds_words<NW>(rs + 128 * sbl + 32 * c + off, w);
        const int64_t pstart =
            ((tl.row0 + row) * static_cast<int64_t>(p.nsb) + sl * G::kSlabSB) * 8;
        const uint32_t pa = st + G::kRows * G::kSlot + row * G::kPSlot +
                            static_cast<uint32_t>(pstart & 15) + 8 * sbl;
        const uint2 pr = lds64(pa);
        const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&pr.x));
        const int g = c >> 1;
        const float sc = static_cast<float>((pr.y >> (8 * g)) & 0xFF);
        const float mn = static_cast<float>((pr.y >> (16 + 8 * g)) & 0xFF);
        dsc = make_float2(dd.x * sc, dd.x * sc);
        dmn = make_float2(dd.y * mn, dd.y * mn);
      } else {
        const uint32_t rec = rs + G::kBB * sbl;
        const uint4 hdr = lds128(rec);
        lds_words<NW>(rec + (F == kQ4K ? 16 : 48) + 32 * c + off, w);
        if constexpr (F == kQ5K) lds_words<NW>(rec + 16 + off, hq);
        const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&hdr.x));
        uint32_t scp, mnp;
        scale_pairs(hdr.y, hdr.z, hdr.w, c, scp, mnp);
        dsc = make_float2(dd.x * static_cast<float>(scp & 0xFF),
                          dd.x * static_cast<float>(scp >> 8));
        dmn = make_float2(dd.y * static_cast<float>(mnp & 0xFF),
                          dd.y * static_cast<float>(mnp >> 8));
      }
      float2 alo[2][NT], ahi[2][NT];
#pragma unroll
      for (int k = 0; k < NT; ++k) {
        alo[0][k] = alo[1][k] = make_float2(0.0f, 0.0f);
        ahi[0][k] = ahi[1][k] = make_float2(0.0f, 0.0f);
      }
      unit_q4<F, NT, NW>(w, hq, c, xl, xh, alo, ahi);
#pragma unroll
      for (int k = 0; k < NT; ++k) {
        const float slo = (alo[0][k].x + alo[1][k].x) + (alo[0][k].y + alo[1][k].y);
        const float shi = (ahi[0][k].x + ahi[1][k].x) + (ahi[0][k].y + ahi[1][k].y);
        float v = acc[r][k];
        v = fmaf(dsc.x, slo, v);
        v = fmaf(dsc.y, shi, v);
        v = fmaf(-dmn.x, sxlo[k], v);
        v = fmaf(-dmn.y, sxhi[k], v);
        acc[r][k] = v;
      }
    }
  }
}

// One stage of a Q6_K tile.  Unit (h, u2): weights 128h + 32t + l0 + i for
// t < 4, i < kCW/4 (l0 = u2 kCW/4); sub-block of (t, l) = 8h + 2t + l/16.
// Records start on 2-byte boundaries: words are read aligned and shifted.
// With at least two words per t-run the words are paired (64-bit), as in
// unit_q4; with one word (n_tok 4) each word is used alone.
template <int NT, int RT, bool XBF>
__device__ __forceinline__ void stage_q6(const Params& p, const Tile& tl, int sl, int xsl,
                                         uint32_t st, uint32_t xs, int hw, int sbl, int un,
                                         float (&acc)[RT][NT]) {
  using G = Geo<kQ6K, NT, RT>;
  using L = XLayout<kQ6K, NT, XBF>;
  constexpr int kCW = G::kCW, QW = kCW / 16;
  constexpr bool kPaired = L::kInterleave;
  constexpr int NX = kPaired ? QW / 2 : QW;   // x groups per t-run
  const int h = un / (G::kUnitsPerSB / 2);
  const int u2 = un % (G::kUnitsPerSB / 2);
  const int l0 = u2 * (kCW / 4);
  const int su = l0 >> 4;
  // xv[t-run tt][group][b]: paired -> pairs of nibble position b (b < 4);
  // single -> (x0,x1), (x2,x3) in [0], [1]
  float2 xv[NT][4][NX][4];
  float sxt[NT][4];   // sum of x over each t-run (for the -32 of q - 32)
  const int kb = xsl * G::kSlabK + sbl * 256 + 128 * h + l0;
  const uint32_t sxa = xs + static_cast<uint32_t>(L::bytes(static_cast<size_t>(NT) * p.kpad));
  const int parts = p.kpad / G::kPart;
#pragma unroll
  for (int k = 0; k < NT; ++k)
#pragma unroll
    for (int tt = 0; tt < 4; ++tt)
      sxt[k][tt] = __uint_as_float(lds32(sxa + 4 * (k * parts + (kb + 32 * tt) / G::kPart)));
#pragma unroll
  for (int k = 0; k < NT; ++k)
#pragma unroll
    for (int tt = 0; tt < 4; ++tt)
#pragma unroll
      for (int j = 0; j < NX; ++j) {
        const int g = k * p.kpad + kb + 32 * tt + (kPaired ? 8 : 4) * j;
        x_quad<kQ6K, NT, XBF>(xs, g, xv[k][tt][j][0], xv[k][tt][j][1]);
        if (kPaired) x_quad<kQ6K, NT, XBF>(xs, g + 4, xv[k][tt][j][2], xv[k][tt][j][3]);
      }
#pragma unroll
  for (int r = 0; r < RT; ++r) {
    const int row = hw + 2 * kWC * r;
    if (row < tl.rcnt) {
      const int64_t start =
          ((tl.row0 + row) * static_cast<int64_t>(p.nsb) + sl * G::kSlabSB) * 210;
      const uint32_t rec = st + row * G::kSlot + static_cast<uint32_t>(start & 15) + 210 * sbl;
      uint32_t A[QW], B[QW], H[QW], S[2], D[1];
      lds_words_a2<QW>(rec + 64 * h + l0, A);
      lds_words_a2<QW>(rec + 64 * h + 32 + l0, B);
      lds_words_a2<QW>(rec + 128 + 32 * h + l0, H);
      lds_words_a2<2>(rec + 192 + 8 * h, S);
      lds_words_a2<1>(rec + 208, D);
      float2 at[NT][4];
#pragma unroll
      for (int k = 0; k < NT; ++k)
#pragma unroll
        for (int tt = 0; tt < 4; ++tt) at[k][tt] = make_float2(0.0f, 0.0f);
      if constexpr (kPaired) {
        const uint32_t M = 0x0F0F0F0Fu;
#pragma unroll
        for (int j = 0; j < NX; ++j) {
          const uint64_t A64 = u64(A[2 * j], A[2 * j + 1]), B64 = u64(B[2 * j], B[2 * j + 1]);
          const uint64_t H64 = u64(H[2 * j], H[2 * j + 1]);
          // 6-bit q per byte (bits that cross the 32-bit halves in the
          // 64-bit shifts land in bits the masks discard)
          uint64_t q6[4];
          q6[0] = bitsel64(A64, H64 << 4, M);
          q6[1] = bitsel64(B64, H64 << 2, M);
          q6[2] = bitsel64(A64 >> 4, H64, M);
          q6[3] = bitsel64(B64 >> 4, H64 >> 2, M);
#pragma unroll
          for (int tt = 0; tt < 4; ++tt) {
            const uint64_t v = q6[tt], vs = v >> 8;
            float2 q[4];
            q[0] = conv64(v, 0x3Fu);
            q[1] = conv64(v, 0x3F00u);
            q[2] = conv64(v, 0x3F0000u);
            q[3] = conv64(vs, 0x3F0000u);
#pragma unroll
            for (int k = 0; k < NT; ++k)
#pragma unroll
              for (int b = 0; b < 4; ++b) at[k][tt] = __ffma2_rn(q[b], xv[k][tt][j][b], at[k][tt]);
          }
        }
      } else {
        const float2 nm = make_float2(-8388608.0f, -8388608.0f);
#pragma unroll
        for (int j = 0; j < QW; ++j) {
          uint32_t q6[4];
          q6[0] = bitsel(A[j], H[j] << 4, 0x0F0F0F0Fu);
          q6[1] = bitsel(B[j], H[j] << 2, 0x0F0F0F0Fu);
          q6[2] = bitsel(A[j] >> 4, H[j], 0x0F0F0F0Fu);
          q6[3] = bitsel(B[j] >> 4, H[j] >> 2, 0x0F0F0F0Fu);
#pragma unroll
          for (int tt = 0; tt < 4; ++tt) {
            const uint32_t v = q6[tt], vs = v >> 8;
            const float2 q0 = __fadd2_rn(f2(lop_mask_or(v, 0x3Fu, kMagic), lop_mask_or(v, 0x3F00u, kMagic)), nm);
            const float2 q1 = __fadd2_rn(f2(lop_mask_or(v, 0x3F0000u, kMagic), lop_mask_or(vs, 0x3F0000u, kMagic)), nm);
#pragma unroll
            for (int k = 0; k < NT; ++k) {
              at[k][tt] = __ffma2_rn(q0, xv[k][tt][j][0], at[k][tt]);
              at[k][tt] = __ffma2_rn(q1, xv[k][tt][j][1], at[k][tt]);
            }
          }
        }
      }
      const float d = half_bits_to_float(D[0] & 0xFFFFu);
#pragma unroll
      for (int tt = 0; tt < 4; ++tt) {
        const int bi = su + 2 * tt;   // byte of the 8 scales of half h
        const int8_t sc = static_cast<int8_t>((S[bi >> 2] >> (8 * (bi & 3))) & 0xFF);
        const float ds = d * static_cast<float>(sc);
#pragma unroll
        for (int k = 0; k < NT; ++k)
          acc[r][k] = fmaf(ds, fmaf(-32.0f, sxt[k][tt], at[k][tt].x + at[k][tt].y), acc[r][k]);
      }
    }
  }
}

constexpr int kMaxStages = 8;

template <int F, int NT, int RT, bool XBF>
__global__ void __launch_bounds__(kThreads) gemv_stream(const Params p, int stages) {
  using G = Geo<F, NT, RT>;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[2 * kMaxStages];
  __shared__ int last_flag;
  const uint32_t bar_full = smem_addr(&bars[0]);
  const uint32_t bar_empty = smem_addr(&bars[kMaxStages]);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t xs = smem_addr(smem);
  uint8_t* ring = smem + p.x_bytes;
  const uint32_t ring_a = xs + p.x_bytes;
  // CTA c works on K segment c % ksplit and on tiles c / ksplit + i * cps
  const int kseg = static_cast<int>(blockIdx.x) % p.ksplit;
  const int cta = static_cast<int>(blockIdx.x) / p.ksplit;
  const int cps = static_cast<int>(gridDim.x) / p.ksplit;   // CTAs per segment
  const int my_tiles = (p.tiles - cta + cps - 1) / cps;
  const int total = my_tiles * p.slabs;   // stages of this CTA
  const int sl0 = kseg * p.slabs;         // first slab (of the row) of the segment
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(bar_full + 8 * s, 32);      // every producer lane arrives
      mbar_init(bar_empty + 8 * s, kWC);    // one arrival per consumer warp
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const bool producer = warp == kWC;
  const int first = total < stages ? total : stages;
  // Programmatic dependent launch: the next kernel on the stream may start
  // its CTAs as SMs free up; it reads its activations and touches the
  // split-K scratch only after its own griddepcontrol.wait, i.e. after this
  // grid has completed.
  asm volatile("griddepcontrol.launch_dependents;");
  if (producer) {
    // weights do not depend on the previous kernel: the first ring of stages
    // (no empty wait needed) streams while that kernel may still be running
    for (int it = 0; it < first; ++it) {
      const Tile tl = tile_of(p, cta + (it / p.slabs) * cps);
      issue_stage<F, NT, RT>(p, smem, ring_a + it * G::kStage, bar_full + 8 * it, tl,
                             sl0 + it % p.slabs);
    }
  }
  // x may be produced by the previous kernel: wait for it to complete
  asm volatile("griddepcontrol.wait;" ::: "memory");
  stage_x<F, NT, RT, XBF>(p, smem, kseg * p.kpad);
  __syncthreads();
  if (producer) {
    for (int it = first; it < total; ++it) {
      const int slot = it % stages;
      const uint32_t use = static_cast<uint32_t>(it / stages);
      if (!mbar_wait_warp(bar_empty + 8 * slot, (use - 1) & 1)) return;
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      const Tile tl = tile_of(p, cta + (it / p.slabs) * cps);
      issue_stage<F, NT, RT>(p, smem, ring_a + slot * G::kStage, bar_full + 8 * slot, tl,
                             sl0 + it % p.slabs);
    }
    return;
  }
  // consumers
  constexpr int kCW = G::kCW;
  const int hw = 2 * warp + (lane >> 4);   // half-warp: rows hw + 8 r of a tile
  const int ul = lane & 15;                // unit position in the slab
  const int sbl = ul / G::kUnitsPerSB;     // super-block in the slab
  const int un = ul % G::kUnitsPerSB;      // unit in the super-block
  const int c = un / (64 / kCW);           // Q4 family: chunk
  const int off = (un % (64 / kCW)) * (kCW / 2);
  float acc[RT][NT];
  Tile tl{};
  int t = 0;
  for (int it = 0; it < total; ++it) {
    const int xsl = it % p.slabs;   // slab within the segment
    const int sl = sl0 + xsl;       // slab within the row
    if (xsl == 0) {
      t = cta + (it / p.slabs) * cps;
      tl = tile_of(p, t);
#pragma unroll
      for (int r = 0; r < RT; ++r)
#pragma unroll
        for (int k = 0; k < NT; ++k) acc[r][k] = 0.0f;
    }
    const int slot = it % stages;
    const uint32_t use = static_cast<uint32_t>(it / stages);
    if (!mbar_wait_warp(bar_full + 8 * slot, use & 1)) return;
    const uint32_t st = ring_a + slot * G::kStage;
    if (sl * G::kSlabSB + sbl < p.nsb) {
      if constexpr (F == kQ6K)
        stage_q6<NT, RT, XBF>(p, tl, sl, xsl, st, xs, hw, sbl, un, acc);
      else
        stage_q4<F, NT, RT, XBF>(p, tl, sl, xsl, st, xs, hw, sbl, c, off, acc);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * slot);
    if (xsl == p.slabs - 1) {
#pragma unroll
      for (int r = 0; r < RT; ++r)
#pragma unroll
        for (int k = 0; k < NT; ++k) {
          float v = acc[r][k];
          v += __shfl_xor_sync(0xFFFFFFFFu, v, 8);
          v += __shfl_xor_sync(0xFFFFFFFFu, v, 4);
          v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
          v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
          acc[r][k] = v;
        }
      float* y = pick(p.g.y, tl.mi);
      const int64_t N = pick(p.g.N, tl.mi);
      if (p.ksplit == 1) {
        if (ul == 0) {
#pragma unroll
          for (int r = 0; r < RT; ++r) {
            const int row = hw + 2 * kWC * r;
            if (row < tl.rcnt) {
#pragma unroll
              for (int k = 0; k < NT; ++k)
                if (k < p.nt) y[static_cast<int64_t>(k) * N + tl.row0 + row] = acc[r][k];
            }
          }
        }
      } else {
        // split-K: publish this segment's partial sums; the last CTA of the
        // tile to arrive adds the segments in order 0..ksplit-1 (the result
        // does not depend on arrival order) and re-arms the counter
        float* part = p.part + static_cast<int64_t>(t) * p.tile_rows * NT;
        const int64_t seg_stride = static_cast<int64_t>(p.tiles) * p.tile_rows * NT;
        if (ul == 0) {
#pragma unroll
          for (int r = 0; r < RT; ++r) {
            const int row = hw + 2 * kWC * r;
            if (row < tl.rcnt) {
#pragma unroll
              for (int k = 0; k < NT; ++k) __stcg(part + kseg * seg_stride + row * NT + k, acc[r][k]);
            }
          }
          __threadfence();
        }
        asm volatile("bar.sync 1, %0;" ::"r"(kWC * 32) : "memory");
        if (threadIdx.x == 0) last_flag = atomicAdd(p.arrivals + t, 1u) == static_cast<unsigned>(p.ksplit - 1);
        asm volatile("bar.sync 1, %0;" ::"r"(kWC * 32) : "memory");
        if (last_flag) {
          __threadfence();
          if (ul == 0) {
#pragma unroll
            for (int r = 0; r < RT; ++r) {
              const int row = hw + 2 * kWC * r;
              if (row < tl.rcnt) {
#pragma unroll
                for (int k = 0; k < NT; ++k) {
                  float v = 0.0f;
                  for (int j = 0; j < p.ksplit; ++j) v += __ldcg(part + j * seg_stride + row * NT + k);
                  if (k < p.nt) y[static_cast<int64_t>(k) * N + tl.row0 + row] = v;
                }
              }
            }
          }
          if (threadIdx.x == 0) p.arrivals[t] = 0u;
        }
      }
    }
  }
}

struct DevInfo {
  int sms = 0;
  size_t smem_optin = 0;
};

DevInfo& dev_info() {
  static DevInfo info[64];
  int d = 0;
  cudaGetDevice(&d);
  DevInfo& i = info[d & 63];
  if (i.sms == 0) {
    cudaDeviceGetAttribute(&i.sms, cudaDevAttrMultiProcessorCount, d);
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, d);
    i.smem_optin = static_cast<size_t>(v);
  }
  return i;
}

constexpr size_t kSmemPerSM = 228 * 1024;   // usable shared memory per SM (B300)

// Split-K scratch of the current device: a fixed region of kMaxTiles arrival
// counters, then the partial sums.  The counter region never moves or
// shrinks, so counters stay zero across launches of any shape (partial sums
// of one launch never land on another launch's counters).  Grown on demand
// (never while the stream is being captured), zero-filled when allocated;
// kernels leave every counter they use at zero when they finish.
constexpr int kMaxTiles = 1 << 16;
constexpr size_t kCounterBytes = size_t{kMaxTiles} * sizeof(unsigned int);
struct Scratch {
  void* base = nullptr;
  size_t bytes = 0;
};
Scratch& scratch_of_device() {
  static Scratch sc[64];
  int d = 0;
  cudaGetDevice(&d);
  return sc[d & 63];
}
void* scratch_get(size_t bytes, cudaStream_t s) {
  Scratch& sc = scratch_of_device();
  if (sc.bytes >= bytes) return sc.base;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
    (void)cudaGetLastError();
    return nullptr;
  }
  size_t want = bytes < (size_t{1} << 20) ? (size_t{1} << 20) : bytes;
  void* p = nullptr;
  if (sc.base != nullptr) cudaFree(sc.base);   // synchronises with work using it
  sc.base = nullptr;
  sc.bytes = 0;
  if (cudaMalloc(&p, want) != cudaSuccess || cudaMemset(p, 0, want) != cudaSuccess) {
    (void)cudaGetLastError();
    if (p != nullptr) cudaFree(p);
    return nullptr;
  }
  sc.base = p;
  sc.bytes = want;
  return p;
}

// Shared-memory plan of one configuration: staged x bytes, CTAs per SM (as
// many as fit with at least two ring stages, up to three) and ring stages.
struct Plan {
  uint32_t x_bytes = 0;
  int per_sm = 0;
  int stages = 0;
  size_t smem = 0;
};

template <int F, int NT, int RT, bool XBF>
Plan make_plan(int K, int ksplit) {
  using G = Geo<F, NT, RT>;
  Plan pl;
  const int slabs_row = (K / 256 + G::kSlabSB - 1) / G::kSlabSB;
  if (slabs_row % ksplit != 0) return pl;
  const int kpad = slabs_row / ksplit * G::kSlabK;
  const size_t xb = XLayout<F, NT, XBF>::bytes(static_cast<size_t>(NT) * kpad) +
                    static_cast<size_t>(NT) * (kpad / G::kPart) * 4;
  pl.x_bytes = static_cast<uint32_t>((xb + 127) & ~size_t{127});
  const size_t optin = dev_info().smem_optin;
  for (int per_sm = 3; per_sm >= 1; --per_sm) {
    size_t budget = (per_sm == 1 ? optin : kSmemPerSM / per_sm) - 2048;
    if (budget > optin - 1024) budget = optin - 1024;
    if (pl.x_bytes + 2 * static_cast<size_t>(G::kStage) > budget) continue;
    int stages = static_cast<int>((budget - pl.x_bytes) / G::kStage);
    if (stages > kMaxStages) stages = kMaxStages;
    pl.per_sm = per_sm;
    pl.stages = stages;
    pl.smem = pl.x_bytes + static_cast<size_t>(stages) * G::kStage;
    return pl;
  }
  return pl;
}

// Where split-K partial sums live.  kDevice: the per-device buffer above
// (grown with cudaMalloc).  kStatic: the fixed array of kq_gemv_noalloc below
// (never allocates; too_large reports a request beyond its capacity).
enum class ScratchSrc { kDevice, kStatic };
struct StaticScratch {
  uint8_t* base;
  bool too_large;
};
constexpr int kNoAllocMaxTiles = 1 << 14;
constexpr size_t kNoAllocCounterBytes = size_t{kNoAllocMaxTiles} * sizeof(unsigned int);
constexpr size_t kNoAllocScratchBytes = size_t{2} << 20;   // 2 MiB per device

template <int F, int NT, int RT, bool XBF>
bool launch_cfg(const GemvGroup& g, const uint16_t* x, int K, int n_tok, cudaStream_t s,
                int ksplit, ScratchSrc src = ScratchSrc::kDevice,
                StaticScratch* st = nullptr) {
  using G = Geo<F, NT, RT>;
  const DevInfo& di = dev_info();
  Params p;
  p.g = g;
  p.x = x;
  p.K = K;
  p.nsb = K / 256;
  const int slabs_row = (p.nsb + G::kSlabSB - 1) / G::kSlabSB;
  if (slabs_row % ksplit != 0) return false;
  p.ksplit = ksplit;
  p.slabs = slabs_row / ksplit;
  p.kpad = p.slabs * G::kSlabK;
  p.nt = n_tok;
  p.part = nullptr;
  p.arrivals = nullptr;
  const Plan pl = make_plan<F, NT, RT, XBF>(K, ksplit);
  if (pl.per_sm == 0) return false;
  p.x_bytes = pl.x_bytes;
  int per_sm = pl.per_sm;
  const int stages = pl.stages;
  const size_t smem = pl.smem;
  static size_t configured = 0;   // dynamic shared memory above 48 KB is opt-in
  if (smem > configured) {
    if (cudaFuncSetAttribute(gemv_stream<F, NT, RT, XBF>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess) {
      (void)cudaGetLastError();
      return false;
    }
    configured = smem;
  }
  int occ = 0;   // registers may allow fewer CTAs than shared memory does
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, gemv_stream<F, NT, RT, XBF>, kThreads,
                                                    smem) == cudaSuccess &&
      occ >= 1 && occ < per_sm)
    per_sm = occ;
  // CTAs per K segment, all resident at once
  int cps = per_sm * di.sms / ksplit;
  if (cps < 1) cps = 1;
  // Balanced tiling: every CTA of a segment streams (about) the same number
  // of equal tiles.  k = tiles per CTA, rows per tile = ceil(rows / (cps k)).
  int64_t rows = 0;
  for (int i = 0; i < g.count; ++i) rows += g.N[i];
  const int64_t k = (rows + static_cast<int64_t>(cps) * G::kRows - 1) /
                    (static_cast<int64_t>(cps) * G::kRows);
  int tr = static_cast<int>((rows + cps * k - 1) / (cps * k));
  if (tr > G::kRows) tr = G::kRows;
  if (tr < 1) tr = 1;
  p.tile_rows = tr;
  p.tiles = 0;
  for (int i = 0; i < kMaxGroup; ++i) {
    if (i < g.count) p.tiles += (g.N[i] + tr - 1) / tr;
    p.tile_end[i] = p.tiles;
  }
  if (cps > p.tiles) cps = p.tiles;
  if (ksplit > 1) {
    const size_t part_bytes =
        static_cast<size_t>(ksplit) * p.tiles * p.tile_rows * NT * sizeof(float);
    if (src == ScratchSrc::kDevice) {
      if (p.tiles > kMaxTiles) return false;
      uint8_t* base = static_cast<uint8_t*>(scratch_get(kCounterBytes + part_bytes, s));
      if (base == nullptr) return false;
      p.arrivals = reinterpret_cast<unsigned int*>(base);
      p.part = reinterpret_cast<float*>(base + kCounterBytes);
    } else {
      if (p.tiles > kNoAllocMaxTiles ||
          kNoAllocCounterBytes + part_bytes > kNoAllocScratchBytes) {
        st->too_large = true;
        return false;
      }
      // the array keeps the previous call's contents: clear the counters
      // this launch uses (a stream-ordered memset, not an allocation)
      if (cudaMemsetAsync(st->base, 0, static_cast<size_t>(p.tiles) * sizeof(unsigned int), s) !=
          cudaSuccess)
        return false;
      p.arrivals = reinterpret_cast<unsigned int*>(st->base);
      p.part = reinterpret_cast<float*>(st->base + kNoAllocCounterBytes);
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(cps * ksplit));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemv_stream<F, NT, RT, XBF>, p, stages) == cudaSuccess;
}

template <int F, int NT, int RT>
bool launch_rt(const GemvGroup& g, const uint16_t* x, int K, int n_tok, cudaStream_t s,
               ScratchSrc src = ScratchSrc::kDevice, StaticScratch* st = nullptr) {
  using G = Geo<F, NT, RT>;
  // K segments: the fewest (a power of two dividing the slabs of a row, at
  // most 16) that reach three CTAs per SM, else the fewest that reach the
  // most CTAs per SM.  x is staged as bf16 only when its fp32 copy would not
  // fit at all.
  const int slabs_row = (K / 256 + G::kSlabSB - 1) / G::kSlabSB;
  int best_ks = 0, best_sm = 0;
  bool best_bf = false;
  for (int ks = 1; ks <= 16 && slabs_row % ks == 0; ks *= 2) {
    Plan pl = make_plan<F, NT, RT, false>(K, ks);
    bool bf = false;
    if (pl.per_sm == 0) {
      pl = make_plan<F, NT, RT, true>(K, ks);
      bf = true;
    }
    if (pl.per_sm > best_sm) {
      best_sm = pl.per_sm;
      best_ks = ks;
      best_bf = bf;
    }
    if (best_sm == 3) break;
  }
  if (best_ks == 0) return false;
  for (int ks = best_ks;; ks = 1) {
    const bool ok = best_bf ? launch_cfg<F, NT, RT, true>(g, x, K, n_tok, s, ks, src, st)
                            : launch_cfg<F, NT, RT, false>(g, x, K, n_tok, s, ks, src, st);
    if (ok || ks == 1) return ok;   // no scratch (e.g. during capture): unsplit
    if (st != nullptr && st->too_large) return false;
    best_bf = static_cast<size_t>(NT) * K * 4 > 96 * 1024;
  }
}

template <int F, int NT>
bool launch_nt(const GemvGroup& g, const uint16_t* x, int K, int n_tok, cudaStream_t s,
               ScratchSrc src = ScratchSrc::kDevice, StaticScratch* st = nullptr) {
  const DevInfo& di = dev_info();
  // rows per thread: 4, or 2 for small matrices (fewer than 16 rows per SM)
  int64_t rows = 0;
  for (int i = 0; i < g.count; ++i) rows += g.N[i];
  if (rows < 16LL * di.sms) return launch_rt<F, NT, 2>(g, x, K, n_tok, s, src, st);
  return launch_rt<F, NT, 4>(g, x, K, n_tok, s, src, st);
}

}  // namespace

bool launch_stream(int fmt, const GemvGroup& g, const uint16_t* x, int K, int n_tok,
                   cudaStream_t s) {
  if (n_tok > 4) return false;
  const int nt = n_tok <= 1 ? 1 : (n_tok <= 2 ? 2 : 4);
#define KQ_CASE(F)                                                  \
  case F:                                                           \
    if (nt == 1) return launch_nt<F, 1>(g, x, K, n_tok, s);         \
    if (nt == 2) return launch_nt<F, 2>(g, x, K, n_tok, s);         \
    return launch_nt<F, 4>(g, x, K, n_tok, s);
  switch (fmt) {
    KQ_CASE(kQ4K)
    KQ_CASE(kQ5K)
    KQ_CASE(kQ6K)
    KQ_CASE(kG128)
  }
#undef KQ_CASE
  return false;
}

// ------------------------------------------------------- no-allocation path
//
// Scratch of kq_gemv_noalloc: a fixed 2 MiB array in every device that loads
// this library (held until the process exits).  The first 64 KiB hold the
// split-K arrival counters of at most kNoAllocMaxTiles tiles, the rest the
// partial sums.  All calls share it; calls that overlap on the GPU race on it.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
// Device address of g_noalloc_scratch on the current device.  In host code
// the array's name is only a host-side stand-in, never a device address: the
// address is looked up once per device (with that device current) and
// cached.  nullptr if the lookup fails.
void* noalloc_scratch_address() {
  static void* addr[64] = {};
  static bool looked_up[64] = {};
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) return nullptr;
  d &= 63;
  if (!looked_up[d]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) {
      (void)cudaGetLastError();
      return nullptr;
    }
    addr[d] = ptr;
    looked_up[d] = true;
  }
  return addr[d];
}
}  // namespace

NoAllocResult launch_stream_noalloc(int fmt, const GemvGroup& g, const uint16_t* x, int K,
                                    int n_tok, cudaStream_t s) {
  if (n_tok > 4) return NoAllocResult::kNotServed;
  StaticScratch st{static_cast<uint8_t*>(noalloc_scratch_address()), false};
  if (st.base == nullptr) return NoAllocResult::kFailed;
  const int nt = n_tok <= 1 ? 1 : (n_tok <= 2 ? 2 : 4);
  bool ok = false;
#define KQ_CASE(F)                                                                          \
  case F:                                                                                   \
    ok = nt == 1   ? launch_nt<F, 1>(g, x, K, n_tok, s, ScratchSrc::kStatic, &st)           \
         : nt == 2 ? launch_nt<F, 2>(g, x, K, n_tok, s, ScratchSrc::kStatic, &st)           \
                   : launch_nt<F, 4>(g, x, K, n_tok, s, ScratchSrc::kStatic, &st);          \
    break;
  switch (fmt) {
    KQ_CASE(kQ4K)
    KQ_CASE(kQ5K)
    KQ_CASE(kQ6K)
    KQ_CASE(kG128)
    default:
      return NoAllocResult::kFailed;
  }
#undef KQ_CASE
  if (st.too_large) return NoAllocResult::kTooLarge;
  return ok ? NoAllocResult::kLaunched : NoAllocResult::kNotServed;
}

bool read_wait_timeouts(unsigned int* count, cudaStream_t s) {
  unsigned int zero = 0;
  if (cudaMemcpyFromSymbolAsync(count, g_wait_timeouts, sizeof(unsigned int), 0,
                                cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return false;
  if (cudaStreamSynchronize(s) != cudaSuccess) return false;
  if (*count != 0) {
    // a kernel stopped early: clear the count and re-arm the split-K
    // arrival counters it may have left behind
    if (cudaMemcpyToSymbolAsync(g_wait_timeouts, &zero, sizeof(unsigned int), 0,
                                cudaMemcpyHostToDevice, s) != cudaSuccess)
      return false;
    Scratch& sc = scratch_of_device();
    if (sc.base != nullptr && cudaMemsetAsync(sc.base, 0, sc.bytes, s) != cudaSuccess) return false;
  }
  return cudaStreamSynchronize(s) == cudaSuccess;
}

}  // namespace kq
