// kq_stream.cu -- the streaming K-quant GEMV kernels for sm_103a: n_tok 1..4
// on the CUDA cores (gemv_stream), n_tok 5..16 on the tensor cores
// (gemv_mma, the speculative-verify widths).
//
// y[t][n] = sum_k w^[n][k] x[t][k]  (daily.dev ExecuTorch summary, answer on
// exporting GGUF checkpoints; the Core AI card's 424 GB/s arithmetic shows the
// product is bound by streaming the packed weights once).
//
// Structure.  The rows of the (grouped) matrices are cut into tiles of
// 2 * kWC * RT rows; a tile is streamed in slabs of 16 "units" (a unit = kCW
// weights of one row, kCW = 64 / NT).  One CTA = kWC consumer warps + 1
// producer warp, persistent over its tiles (a first fixed tile, then tiles
// claimed from a per-K-segment counter, so CTAs that get more of the SM and
// of the memory system take more tiles):
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
#include <cuda.h>   // CUtensorMap and its enums (the encoder is fetched at run time)
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>
#include <type_traits>

#include "kq_decode.cuh"
#include "kq_kernels.cuh"

namespace kq {

__device__ unsigned int g_wait_timeouts = 0;

// Dynamic tile scheduling of the streaming kernels.  Per K segment j:
// g_sched[j] counts the tiles claimed past the fixed ones, g_sched[kMaxSegs
// + j] the producers that found none left; the last of those re-arms both, so
// they are zero between launches.  Launches touch them only after
// griddepcontrol.wait, i.e. after the previous kernel on the stream is done.
constexpr int kMaxSegs = 32;
__device__ unsigned int g_sched[2 * kMaxSegs];

namespace {

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
// recorded timeout, if that takes longer than `limit` cycles.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity,
                                               long long limit = kWaitCycles) {
  long long t0 = 0;
  for (int i = 0;; ++i) {
    const bool done = mbar_try(bar, parity);
    if (__all_sync(0xFFFFFFFFu, done)) return true;
    if (i == 0) {
      t0 = clock64();
    } else if (__shfl_sync(0xFFFFFFFFu, (clock64() - t0 > limit) ? 1 : 0, 0)) {
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
__device__ __forceinline__ void sts128u(uint32_t a, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void sts128(uint32_t a, float4 v) {
  asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(a), "f"(v.x), "f"(v.y), "f"(v.z),
               "f"(v.w)
               : "memory");
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

// n consecutive 32-bit words at byte offset off (a multiple of 4) of a
// record that starts on a 2-byte boundary: base = record & ~3, sh = 8 *
// (record & 3), both computed once per record.
template <int N>
__device__ __forceinline__ void lds_words_rec(uint32_t base, uint32_t sh, uint32_t off,
                                              uint32_t (&w)[N]) {
  uint32_t raw[N + 1];
#pragma unroll
  for (int i = 0; i <= N; ++i) raw[i] = lds32(base + off + 4 * i);
#pragma unroll
  for (int i = 0; i < N; ++i) w[i] = __funnelshift_r(raw[i], raw[i + 1], sh);
}

// (a - b) on two bf16 halves.  Used as bf16(c + q) - bf16(c) = bf16(q): both
// operands and the difference are small integers, so the result is exact.
__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
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

template <int F, int NT, int RT, int WC>
struct Geo {
  static constexpr int kF = F;
  static constexpr int kWC = WC;                         // consumer warps per CTA
  static constexpr int kThreads = (WC + 1) * 32;         // + one producer warp
  static constexpr int kRows = 2 * WC * RT;              // rows per tile
  static constexpr int kCW = 64 / NT;                    // weights per unit
  // x positions per part sum: one sub-block part of a unit (Q4 family:
  // kCW/2 low or high nibbles; Q6_K: the kCW/4 weights of one t-run)
  static constexpr int kPart = (F == kQ6K) ? kCW / 4 : kCW / 2;
  static constexpr int kUnitsPerSB = 256 / kCW;          // 4, 8, 16
  static constexpr int kSlabSB = 16 / kUnitsPerSB;       // super-blocks per slab: 4, 2, 1
  static constexpr int kSlabK = 256 * kSlabSB;           // 1024, 512, 256
  static constexpr int kBB = block_bytes(F);
  // Bytes of one row's slab: records (G128: the q plane; its param plane
  // holds kPBytes more).
  static constexpr int kQBytes = (F == kG128) ? 128 * kSlabSB : kBB * kSlabSB;
  static constexpr int kPBytes = (F == kG128) ? 8 * kSlabSB : 0;
  // Per-row shared slot.  Tensor copies: the slab rounded out to the 16-byte
  // grid (a slab that does not start on 16 bytes starts up to 15 bytes into
  // its slot).  Per-row bulk copies: one more 16 bytes of halo.
  static constexpr int round16(int b) { return (b + 15) / 16 * 16; }
  static constexpr int kSlotTma = round16(kQBytes + (kQBytes % 16 ? 15 : 0));
  static constexpr int kPSlotTma = (F == kG128) ? round16(kPBytes + (kPBytes % 16 ? 15 : 0)) : 0;
  static constexpr int kSlotBulk = round16(kQBytes + 16);
  static constexpr int kPSlotBulk = (F == kG128) ? round16(kPBytes + 16) : 0;
};

// Shared-memory shape of one ring stage: rows x slot bytes of records (q
// plane), then (G128) rows x pslot bytes of params at offset pbase.
struct StageShape {
  uint32_t slot, pslot, pbase, bytes;
};
template <class G>
StageShape stage_shape(bool tma, int rows = G::kRows) {
  auto r128 = [](uint32_t b) { return (b + 127u) / 128u * 128u; };
  StageShape s;
  s.slot = tma ? G::kSlotTma : G::kSlotBulk;
  s.pslot = tma ? G::kPSlotTma : G::kPSlotBulk;
  s.pbase = r128(rows * s.slot);
  s.bytes = s.pbase + r128(rows * s.pslot);
  return s;
}

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
  int tile_rows;             // rows per tile (<= the CTA's 2 * WC * RT)
  int tile_end[kMaxGroup];   // cumulative tile counts per matrix
  uint32_t x_bytes;          // shared bytes of the staged x (+ part sums), 16-aligned
  void* part;                // split-K partial sums [ksplit][tiles][tile_rows][NT]: float,
                             // or tagged 64-bit words (gemv_stream, put_partial)
  unsigned int* arrivals;    // split-K per-tile arrival counters (left at zero)
  uint32_t tag;              // this launch's partial-sum tag (nonzero; gemv_stream)
  int static_tiles;          // tiles a CTA takes without claiming: cta + i * cps, i < this
  int tma;                   // 1: a stage arrives as one tensor copy per plane
  uint32_t slot, pslot, pbase, stage;   // StageShape of the ring
  uint32_t tx;               // bytes the tensor copies of one stage deliver
  // SwiGLU mode of the single-token tensor-core kernel: g holds (gate, up)
  // of the same shape; a tile is tile_rows / 2 output features, staged as
  // their gate rows then their up rows, and the kernel also writes
  // h = bf16(silu(gate) * up) (bf16 [N]).
  int swiglu = 0;
  uint16_t* h = nullptr;
  // per matrix: 2-D tensor maps (8-byte elements x rows) of the records / the
  // G128 q plane [0] and the G128 param plane [1]; box = slot bytes x tile_rows
  // (SwiGLU mode: x tile_rows / 2)
  CUtensorMap tm[kMaxGroup][2];
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
  const int feat = p.swiglu ? p.tile_rows / 2 : p.tile_rows;   // output features per tile
  r.row0 = (t - base) * feat;
  r.rcnt = min(feat, pick(p.g.N, mi) - r.row0);
  return r;
}

// ----------------------------------------------------------- x staging

// Bit position s at which the consumers extract the q that multiplies x at
// byte b (= position % 4) of a word, in the low (lo) or high half of a Q4
// family chunk.  Q4_K / G128 low nibbles come from w (b0 s=0, b1 s=8, b2
// s=16) and w >> 12 (b3 s=12); high nibbles from w (b0 s=4, b1 s=12) and
// w >> 12 (b2 s=8, b3 s=16).  Q5_K and Q6_K extract 5- or 6-bit fields from
// two assembled words (Q5_K: low / high nibble with its fifth bit; Q6_K:
// the t0 / t2 or t1 / t3 values of a byte column): b0..b2 at s = 0, 8, 16 of
// each, b3 from one byte-permuted word that holds the first word's b3 at
// s=0 and the second's at s=16 ("lo" = the first word).  x is staged
// pre-scaled by 2^-s, so (2^23 + q 2^s) - 2^23 = q 2^s times the staged x is
// exactly q x.
template <int F>
__host__ __device__ constexpr int field_shift(bool lo, int b) {
  if (F == kQ5K || F == kQ6K) return b == 0 ? 0 : b == 1 ? 8 : b == 2 ? 16 : (lo ? 0 : 16);
  if (lo) return b == 0 ? 0 : b == 1 ? 8 : b == 2 ? 16 : 12;
  return b == 0 ? 4 : b == 1 ? 12 : b == 2 ? 8 : 16;
}

// Shared-memory layout of the staged activations.  Slot i (= token * kpad +
// staged index) sits at byte i * kE + kPad * (i / kPer): the padding
// staggers the 16 units of a half-warp over all bank groups (each unit's x
// is a contiguous run of staged slots), so every x load of the consumers is
// conflict-free (16 B per 64 slots; 8 B for bf16).
//   Q4 family: within each aligned block of 64 positions, position
//     32h + 4i + b (h < 2, i < 8, b < 4) has staged index 8i + 2b + h, so the
//     two positions one byte of a chunk multiplies (its low nibble: h = 0,
//     its high nibble: h = 1) form one fp32 pair for the packed fmas.
//   Q6_K: see stage_x_q6.
template <int F, int NT, bool XBF>
struct XLayout {
  static constexpr int kE = XBF ? 2 : 4;
  static constexpr int kPer = 64;
  static constexpr int kPad = XBF ? 8 : 16;
  __host__ __device__ static constexpr size_t bytes(size_t n) { return n * kE + kPad * (n / kPer); }
  __device__ static uint32_t addr(int i) {
    return static_cast<uint32_t>(i * kE + kPad * (i / kPer));
  }
};

// X (layout above) followed by SX: [NT][kpad/kPart] fp32 part sums.
// Entries beyond K or for tokens >= nt are zero.  Q6_K: part sums in
// position order.  Q4 family: within a 64-block, the sum over positions
// [32h + j kPart, 32h + (j+1) kPart) sits at index 2j + h, so the (low, high)
// sums of one unit form a pair.
template <int F, int NT, bool XBF>
__device__ void stage_x_q4(const Params& p, uint8_t* smem, int kbase) {
  using G = Geo<F, NT, 1, 1>;
  using L = XLayout<F, NT, XBF>;
  constexpr int P = G::kPart;        // 32, 16, 8 positions per part sum
  constexpr int GP = P / 4;          // 4-position groups per part: 8, 4, 2
  const int groups_per_tok = p.kpad / 4 / 2;   // one group = 4 low + 4 high positions
  const int total = NT * groups_per_tok;
  const int parts_per_tok = p.kpad / P;
  float* sx = reinterpret_cast<float*>(smem + L::bytes(static_cast<size_t>(NT) * p.kpad));
  const int lane = threadIdx.x & 31;
  // trip count uniform per warp (the part sums are reduced with shuffles over
  // GP consecutive lanes; total and groups_per_tok are multiples of 8); the
  // loads of four items are in flight together
  constexpr int U = 4;
  for (int base0 = static_cast<int>(threadIdx.x) & ~31; base0 < total;
       base0 += U * static_cast<int>(blockDim.x)) {
    uint2 rlu[U], rhu[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int q = base0 + u * static_cast<int>(blockDim.x) + lane;
      const int tk = q / groups_per_tok, gi = q % groups_per_tok;
      const int k = (gi >> 3) * 64 + 4 * (gi & 7);
      rlu[u] = rhu[u] = make_uint2(0, 0);
      if (q < total && tk < p.nt && kbase + k < p.K) {
        const uint16_t* xt = p.x + static_cast<int64_t>(tk) * p.K + kbase + k;
        rlu[u] = *reinterpret_cast<const uint2*>(xt);
        rhu[u] = *reinterpret_cast<const uint2*>(xt + 32);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
    const int q = base0 + u * static_cast<int>(blockDim.x) + lane;
    const bool in = q < total;
    const int tk = q / groups_per_tok, gi = q % groups_per_tok;
    const int blk = gi >> 3, i = gi & 7;
    const uint2 rl = rlu[u], rh = rhu[u];
    float v[8];   // staged order: (lo b, hi b) for b = 0..3
    v[0] = __uint_as_float(rl.x << 16);
    v[2] = __uint_as_float(rl.x & 0xFFFF0000u);
    v[4] = __uint_as_float(rl.y << 16);
    v[6] = __uint_as_float(rl.y & 0xFFFF0000u);
    v[1] = __uint_as_float(rh.x << 16);
    v[3] = __uint_as_float(rh.x & 0xFFFF0000u);
    v[5] = __uint_as_float(rh.y << 16);
    v[7] = __uint_as_float(rh.y & 0xFFFF0000u);
    float slo = (v[0] + v[2]) + (v[4] + v[6]);
    float shi = (v[1] + v[3]) + (v[5] + v[7]);
#pragma unroll
    for (int m = 1; m < GP; m <<= 1) {
      slo += __shfl_xor_sync(0xFFFFFFFFu, slo, m);
      shi += __shfl_xor_sync(0xFFFFFFFFu, shi, m);
    }
    if (!in) continue;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      v[2 * b] *= pow2(-field_shift<F>(true, b));
      v[2 * b + 1] *= pow2(-field_shift<F>(false, b));
    }
    uint8_t* d = smem + L::addr(tk * p.kpad + blk * 64 + 8 * i);
    if constexpr (XBF) {
      uint32_t r[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        r[j] = (__float_as_uint(v[2 * j]) >> 16) | (__float_as_uint(v[2 * j + 1]) & 0xFFFF0000u);
      // the bf16 layout pads by 8 bytes: a group start is 8-byte aligned
      uint2* d2 = reinterpret_cast<uint2*>(d);
      d2[0] = make_uint2(r[0], r[1]);
      d2[1] = make_uint2(r[2], r[3]);
    } else {
      float4* d4 = reinterpret_cast<float4*>(d);
      d4[0] = make_float4(v[0], v[1], v[2], v[3]);
      d4[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
    if (i % GP == 0) {
      float* o = sx + tk * parts_per_tok + blk * (64 / P) + 2 * (i / GP);
      o[0] = slo;
      o[1] = shi;
    }
    }
  }
}

// Q6_K: within each aligned block of 128 positions (one half h of a
// super-block), position 32t + 4j + b (t, b < 4, j < 8) has staged index
// 16j + 4b + (0, 2, 1, 3)[t]: the four positions one byte column of the unit
// multiplies sit together as the pairs (t0, t2), (t1, t3) -- t0 and t2 come
// from the low and high nibble of one ql byte, t1 and t3 from another.  Part
// sums: over positions 32t + [q kPart, (q+1) kPart) at index 4q + (0, 2, 1,
// 3)[t] of the block, so one unit's four sums load as one float4.
template <int F, int NT, bool XBF>
__device__ void stage_x_q6(const Params& p, uint8_t* smem, int kbase) {
  using G = Geo<F, NT, 1, 1>;
  using L = XLayout<F, NT, XBF>;
  constexpr int P = G::kPart;        // 16, 8, 4 positions per part sum
  constexpr int GP = P / 4;          // 4-position groups per part: 4, 2, 1
  const int groups_per_tok = p.kpad / 16;   // one group = 4 positions of each t-run
  const int total = NT * groups_per_tok;
  const int parts_per_tok = p.kpad / P;
  float* sx = reinterpret_cast<float*>(smem + L::bytes(static_cast<size_t>(NT) * p.kpad));
  const int lane = threadIdx.x & 31;
  // trip count uniform per warp (part sums are reduced with shuffles over GP
  // consecutive lanes; total and groups_per_tok are multiples of 8); the
  // loads of two items are in flight together
  constexpr int U = 2;
  for (int base0 = static_cast<int>(threadIdx.x) & ~31; base0 < total;
       base0 += U * static_cast<int>(blockDim.x)) {
    uint2 ru[U][4];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int q = base0 + u * static_cast<int>(blockDim.x) + lane;
      const int tk = q / groups_per_tok, gi = q % groups_per_tok;
      const int k = (gi >> 3) * 128 + 4 * (gi & 7);
#pragma unroll
      for (int t = 0; t < 4; ++t) ru[u][t] = make_uint2(0, 0);
      if (q < total && tk < p.nt && kbase + k < p.K) {
        const uint16_t* xt = p.x + static_cast<int64_t>(tk) * p.K + kbase + k;
#pragma unroll
        for (int t = 0; t < 4; ++t) ru[u][t] = *reinterpret_cast<const uint2*>(xt + 32 * t);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
    const int q = base0 + u * static_cast<int>(blockDim.x) + lane;
    const bool in = q < total;
    const int tk = q / groups_per_tok, gi = q % groups_per_tok;
    const int blk = gi >> 3, j = gi & 7;
    const uint2 (&r)[4] = ru[u];
    float v[4][4];   // [t][b]
    float sum[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      v[t][0] = __uint_as_float(r[t].x << 16);
      v[t][1] = __uint_as_float(r[t].x & 0xFFFF0000u);
      v[t][2] = __uint_as_float(r[t].y << 16);
      v[t][3] = __uint_as_float(r[t].y & 0xFFFF0000u);
      sum[t] = (v[t][0] + v[t][1]) + (v[t][2] + v[t][3]);
    }
#pragma unroll
    for (int m = 1; m < GP; m <<= 1)
#pragma unroll
      for (int t = 0; t < 4; ++t) sum[t] += __shfl_xor_sync(0xFFFFFFFFu, sum[t], m);
    if (!in) continue;
    // pre-scale: t0 / t1 fields sit at s = 0, 8, 16, 0 of their word, t2 /
    // t3 fields at s = 0, 8, 16, 16 (byte 3 comes from a byte-permuted word)
    float o[16];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      o[4 * b + 0] = v[0][b] * pow2(-field_shift<F>(true, b));
      o[4 * b + 1] = v[2][b] * pow2(-field_shift<F>(false, b));
      o[4 * b + 2] = v[1][b] * pow2(-field_shift<F>(true, b));
      o[4 * b + 3] = v[3][b] * pow2(-field_shift<F>(false, b));
    }
    uint8_t* d = smem + L::addr(tk * p.kpad + blk * 128 + 16 * j);
    if constexpr (XBF) {
      uint32_t w[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        w[i] = (__float_as_uint(o[2 * i]) >> 16) | (__float_as_uint(o[2 * i + 1]) & 0xFFFF0000u);
      // the bf16 layout pads by 8 bytes: a group start is 8-byte aligned
      uint2* d2 = reinterpret_cast<uint2*>(d);
#pragma unroll
      for (int i = 0; i < 4; ++i) d2[i] = make_uint2(w[2 * i], w[2 * i + 1]);
    } else {
      float4* d4 = reinterpret_cast<float4*>(d);
#pragma unroll
      for (int i = 0; i < 4; ++i) d4[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
    }
    if (j % GP == 0) {
      float* sp = sx + tk * parts_per_tok + blk * (128 / P) + 4 * (j / GP);
      *reinterpret_cast<float4*>(sp) = make_float4(sum[0], sum[2], sum[1], sum[3]);
    }
    }
  }
}

template <int F, int NT, bool XBF>
__device__ __forceinline__ void stage_x(const Params& p, uint8_t* smem, int kbase) {
  if constexpr (F == kQ6K)
    stage_x_q6<F, NT, XBF>(p, smem, kbase);
  else
    stage_x_q4<F, NT, XBF>(p, smem, kbase);
}

// The four values stored at the shared address addr (slots idx .. idx+3,
// idx a multiple of 4) as two float2 pairs.  A unit's x is a run of staged
// slots inside one 64-slot block, so the addresses of a run are its first
// slot's address plus slot * kE.
template <int F, int NT, bool XBF>
__device__ __forceinline__ void x_quad(uint32_t addr, float2& a, float2& b) {
  if constexpr (XBF) {
    const uint2 r = lds64(addr);
    a = make_float2(__uint_as_float(r.x << 16), __uint_as_float(r.x & 0xFFFF0000u));
    b = make_float2(__uint_as_float(r.y << 16), __uint_as_float(r.y & 0xFFFF0000u));
  } else {
    const float4 v = lds_f4(addr);
    a = make_float2(v.x, v.y);
    b = make_float2(v.z, v.w);
  }
}

// ------------------------------------------------------------- producer

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

template <class G>
__device__ __forceinline__ void issue_stage(const Params& p, uint8_t* smem, uint32_t st_a,
                                            uint32_t full, const Tile& tl, int sl) {
  constexpr int F = G::kF;
  if (p.tma) {
    // one copy per plane: the slab of tile_rows rows, from the 16-byte
    // boundary at or below the slab's first byte (x in 8-byte elements);
    // rows past the matrix and bytes past a row are zero-filled and counted
    if ((threadIdx.x & 31) == 0) {
      mbar_arrive_tx(full, p.tx);
      const int xq = ((sl * G::kQBytes) & ~15) / 8, xp = ((sl * G::kPBytes) & ~15) / 8;
      if (p.swiglu) {
        // the tile's gate rows, then the same rows of up
        const uint32_t half = static_cast<uint32_t>(p.tile_rows / 2);
        tma_load_2d(st_a, &p.tm[0][0], xq, tl.row0, full);
        tma_load_2d(st_a + half * p.slot, &p.tm[1][0], xq, tl.row0, full);
        if constexpr (F == kG128) {
          tma_load_2d(st_a + p.pbase, &p.tm[0][1], xp, tl.row0, full);
          tma_load_2d(st_a + p.pbase + half * p.pslot, &p.tm[1][1], xp, tl.row0, full);
        }
      } else {
        tma_load_2d(st_a, &p.tm[tl.mi][0], xq, tl.row0, full);
        if constexpr (F == kG128) tma_load_2d(st_a + p.pbase, &p.tm[tl.mi][1], xp, tl.row0, full);
      }
    }
    return;
  }
  const int lane = threadIdx.x & 31;
  const uint8_t* W = pick(p.g.W, tl.mi);
  const int64_t N = pick(p.g.N, tl.mi);
  const int sb0 = sl * G::kSlabSB;
  const int nsb_here = min(G::kSlabSB, p.nsb - sb0);
  uint32_t tx = 0;
  for (int r = lane; r < tl.rcnt; r += 32) {   // lane l copies rows l, l + 32, ...
    const int64_t idx = (tl.row0 + r) * static_cast<int64_t>(p.nsb) + sb0;
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
      copy_span(W, total * 128, idx * 128, nsb_here * 128, st_a + r * p.slot);
      copy_span(W + total * 128, total * 8, idx * 8, nsb_here * 8, st_a + p.pbase + r * p.pslot);
    } else {
      copy_span(W, N * p.nsb * G::kBB, idx * G::kBB, nsb_here * G::kBB, st_a + r * p.slot);
    }
  }
  mbar_arrive_tx(full, tx);   // every producer lane arrives (count 32)
}

// ------------------------------------------------------------- producer
//
// The producer warp's stage sequence: the slabs of the CTA's tiles in order.
// Its tiles are the fixed ones cta + i * cps (i < static_tiles), then tiles
// claimed from the K segment's counter (one claim ahead, sent with the
// current tile's last stage so its latency hides behind the next empty
// wait).  stage_tile[slot] tells the consumers the tile of a slot; -1 ends
// their loop.  Claims are made only after griddepcontrol.wait (the previous
// kernel may still be using the counters before it).
struct Ring {
  int pt = 0;        // tile of the stage being issued
  int taken = 0;     // tiles taken so far
  int xsl = 0;       // slab within the segment
  int slot = 0;      // ring slot
  int issued = 0;    // stages issued
  uint32_t epar = 1u;   // parity of the empty wait (waited from the second lap on)
  unsigned int claim = 0u;
  bool pending = false;
  __device__ __forceinline__ void advance(int slabs, int stages) {
    if (++xsl == slabs) xsl = 0;
    if (++slot == stages) {
      slot = 0;
      epar ^= 1u;
    }
    ++issued;
  }
};

// Before griddepcontrol.wait: the stages of the fixed tiles that fit the ring.
template <class G>
__device__ __forceinline__ void produce_prefill(const Params& p, uint8_t* smem, uint32_t ring_a,
                                                uint32_t bar_full, int* stage_tile, int stages,
                                                int cta, int cps, int sl0, Ring& r) {
  const int lane = threadIdx.x & 31;
  while (r.issued < stages) {
    if (r.xsl == 0) {
      const int t = cta + r.taken * cps;
      if (r.taken >= p.static_tiles || t >= p.tiles) break;
      r.pt = t;
      ++r.taken;
    }
    if (lane == 0) stage_tile[r.slot] = r.pt;
    issue_stage<G>(p, smem, ring_a + r.slot * p.stage, bar_full + 8 * r.slot, tile_of(p, r.pt),
                   sl0 + r.xsl);
    r.advance(p.slabs, stages);
  }
}

// After griddepcontrol.wait: every further stage, then the end marker.
template <class G>
__device__ __forceinline__ void produce_rest(const Params& p, uint8_t* smem, uint32_t ring_a,
                                             uint32_t bar_full, uint32_t bar_empty,
                                             int* stage_tile, int stages, int cta, int cps,
                                             int kseg, int sl0, Ring& r) {
  const int lane = threadIdx.x & 31;
  const int dyn0 = p.static_tiles * cps;   // first claimed tile index
  for (;;) {
    if (r.xsl == 0) {
      int t = cta + r.taken * cps;
      if (r.taken >= p.static_tiles || t >= p.tiles) {
        if (!r.pending && lane == 0) r.claim = atomicAdd(&g_sched[kseg], 1u);
        t = dyn0 + static_cast<int>(__shfl_sync(0xFFFFFFFFu, r.claim, 0));
        r.pending = false;
      }
      ++r.taken;
      if (t >= p.tiles) {
        // nothing left: tell the consumers through the next slot, and let
        // the segment's last producer re-arm its counters
        if (r.issued >= stages && !mbar_wait_warp(bar_empty + 8 * r.slot, r.epar)) return;
        if (lane == 0) {
          stage_tile[r.slot] = -1;
          if (atomicAdd(&g_sched[kMaxSegs + kseg], 1u) == static_cast<unsigned>(cps - 1)) {
            g_sched[kseg] = 0u;
            g_sched[kMaxSegs + kseg] = 0u;
          }
        }
        if (!p.tma || lane == 0) mbar_arrive(bar_full + 8 * r.slot);
        return;
      }
      r.pt = t;
    }
    if (r.xsl == p.slabs - 1 && !r.pending &&
        (r.taken >= p.static_tiles || cta + r.taken * cps >= p.tiles)) {
      if (lane == 0) r.claim = atomicAdd(&g_sched[kseg], 1u);
      r.pending = true;
    }
    if (r.issued >= stages && !mbar_wait_warp(bar_empty + 8 * r.slot, r.epar)) return;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (lane == 0) stage_tile[r.slot] = r.pt;
    issue_stage<G>(p, smem, ring_a + r.slot * p.stage, bar_full + 8 * r.slot, tile_of(p, r.pt),
                   sl0 + r.xsl);
    r.advance(p.slabs, stages);
  }
}

// Split-K partial sums.  A partial sum travels in one 64-bit word with a
// nonzero tag in its high half, written and read with relaxed device-scope
// accesses: a reader that sees the tag sees the value, so no fence has to
// order a value before a separate flag (a device-scope fence stalls for
// microseconds while the SM has its ring of copies in flight).  The tile's
// last segment to arrive (a relaxed counter) adds a value's segments in
// segment order 0..ksplit-1, so the result does not depend on arrival order;
// a partial not yet visible is waited for (bounded).  The reader clears
// every slot it read, so all slots are zero between launches; the tag
// changes from launch to launch (a graph replays its own), so slots left
// behind by a launch that stopped early are not taken for this launch's.
__device__ __forceinline__ void put_partial(uint64_t* slot, float v, uint32_t tag) {
  const uint64_t w = (static_cast<uint64_t>(tag) << 32) | __float_as_uint(v);
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(slot), "l"(w) : "memory");
}
__device__ __forceinline__ uint64_t load_partial(const uint64_t* slot) {
  uint64_t w;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(w) : "l"(slot) : "memory");
  return w;
}
__device__ __forceinline__ void clear_partial(uint64_t* slot) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(slot), "l"(uint64_t{0}) : "memory");
}
// The word at `slot` once it carries `tag` (bounded wait; a timeout is
// counted and the value read last is returned).
__device__ __noinline__ uint64_t wait_partial(const uint64_t* slot, uint32_t tag) {
  const long long t0 = clock64();
  for (;;) {
    const uint64_t w = load_partial(slot);
    if (static_cast<uint32_t>(w >> 32) == tag) return w;
    if (clock64() - t0 > kWaitCycles) {
      atomicAdd(&g_wait_timeouts, 1u);
      return w;
    }
  }
}
__device__ __forceinline__ float partial_value(uint64_t w) {
  return __uint_as_float(static_cast<uint32_t>(w));
}
// One value's partial sums (ksplit <= 16 segments, seg_stride slots apart)
// added in segment order; every slot is cleared.  The loads of eight
// segments are issued together rather than one L2 round trip after another.
__device__ __forceinline__ float take_partials(uint64_t* part, int64_t seg_stride, int ksplit,
                                               uint32_t tag) {
  constexpr int kJ = 8;
  float v = 0.0f;
  for (int j0 = 0; j0 < ksplit; j0 += kJ) {
    uint64_t w[kJ];
#pragma unroll
    for (int j = 0; j < kJ; ++j)
      w[j] = j0 + j < ksplit ? load_partial(part + (j0 + j) * seg_stride) : 0;
#pragma unroll
    for (int j = 0; j < kJ; ++j)
      if (j0 + j < ksplit) {
        if (static_cast<uint32_t>(w[j] >> 32) != tag)
          w[j] = wait_partial(part + (j0 + j) * seg_stride, tag);
        v += partial_value(w[j]);
      }
  }
  for (int j = 0; j < ksplit; ++j) clear_partial(part + j * seg_stride);
  return v;
}

// The sum of a value's split-K partial sums (ksplit <= 16 segments, seg_stride
// floats apart), added in segment order 0..ksplit-1; the loads are issued
// together rather than one L2 round trip after another.
constexpr int kMaxSplitSum = 16;
__device__ __forceinline__ float sum_segments(const float* part, int64_t seg_stride, int ksplit) {
  float pv[kMaxSplitSum];
#pragma unroll
  for (int j = 0; j < kMaxSplitSum; ++j) pv[j] = j < ksplit ? __ldcg(part + j * seg_stride) : 0.0f;
  float v = 0.0f;
#pragma unroll
  for (int j = 0; j < kMaxSplitSum; ++j)
    if (j < ksplit) v += pv[j];
  return v;
}

// ------------------------------------------------------------- consumers

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

// prmt.b32 in its default mode: selector nibble n picks byte n of the result
// from the eight bytes of (b:a); with its bit 3 set, the picked byte's sign
// bit fills the result byte instead.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Exact (q_a 2^sa, q_b 2^sb) for the field under mask MA of a and under mask
// MB of b: one LOP3 each builds 2^23 + q 2^s (the mask an immediate, the
// magic exponent word a register), one packed add of (-2^23, -2^23) removes
// the offset.
template <uint32_t MA, uint32_t MB>
__device__ __forceinline__ float2 cvt_pair(uint32_t a, uint32_t b, uint32_t magic, uint64_t neg) {
  float2 r;
  asm("{\n\t.reg .b32 t0, t1;\n\t.reg .b64 p, q;\n\t"
      "lop3.b32 t0, %2, %4, %6, 0xEA;\n\t"
      "lop3.b32 t1, %3, %5, %6, 0xEA;\n\t"
      "mov.b64 p, {t0, t1};\n\t"
      "add.rn.f32x2 q, p, %7;\n\t"
      "mov.b64 {%0, %1}, q;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "r"(a), "r"(b), "n"(MA), "n"(MB), "r"(magic), "l"(neg));
  return r;
}
constexpr uint64_t kNegMagic2 = 0xCB000000CB000000ull;   // (-2^23, -2^23)
// Q6_K: -(2^23 + 32 2^s) for the field shifts s = 0, 8, 16, so that
// (2^23 + q 2^s) - (2^23 + 32 2^s) = (q - 32) 2^s exactly (both terms are
// integers in [2^23, 2^24)): the signed weight without a separate -32 sum x
// correction.  Halves: (s, s) for 0, 8, 16, and (0, 16) for the permuted byte.
constexpr uint64_t kNegQ6s0 = 0xCB000020CB000020ull;
constexpr uint64_t kNegQ6s8 = 0xCB002000CB002000ull;
constexpr uint64_t kNegQ6s16 = 0xCB200000CB200000ull;
constexpr uint64_t kNegQ6s0s16 = 0xCB200000CB000020ull;

// The same on 64-bit register pairs: a .b64 operand of the packed f32x2
// instructions is one aligned register pair by construction, so the hot loop
// never needs moves to form pairs.
template <uint32_t MA, uint32_t MB>
__device__ __forceinline__ uint64_t cvt_pair64(uint32_t a, uint32_t b, uint32_t magic,
                                               uint64_t neg) {
  uint64_t r;
  asm("{\n\t.reg .b32 t0, t1;\n\t.reg .b64 p;\n\t"
      "lop3.b32 t0, %1, %3, %5, 0xEA;\n\t"
      "lop3.b32 t1, %2, %4, %5, 0xEA;\n\t"
      "mov.b64 p, {t0, t1};\n\t"
      "add.rn.f32x2 %0, p, %6;\n\t}"
      : "=l"(r)
      : "r"(a), "r"(b), "n"(MA), "n"(MB), "r"(magic), "l"(neg));
  return r;
}
__device__ __forceinline__ void fma2u(uint64_t& d, uint64_t a, uint64_t b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
}
__device__ __forceinline__ uint64_t mul2u(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t add2u(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float2 u2f2(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ uint64_t pack2u(uint32_t lo, uint32_t hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}

// x_quad on 64-bit register pairs
template <bool XBF>
__device__ __forceinline__ void x_quad64(uint32_t addr, uint64_t& a, uint64_t& b) {
  if constexpr (XBF) {
    const uint2 r = lds64(addr);
    a = pack2u(r.x << 16, r.x & 0xFFFF0000u);
    b = pack2u(r.y << 16, r.y & 0xFFFF0000u);
  } else {
    asm volatile("ld.shared.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "r"(addr));
  }
}

// Per-lane constants of the 6-bit (sc, m) decode of Q4_K / Q5_K for the two
// sub-blocks 2c and 2c+1 of the lane's chunk c (bytes j = 2c, 2c+1 of the
// 12-byte field, words s0 = bytes 0-3, s1 = 4-7, s2 = 8-11 of the field).
// j < 4: sc = s0[j] & 63, m = s1[j] & 63; j >= 4: sc = (s2[j-4] & 15) |
// (s0[j-4] >> 6) << 4, m = (s2[j-4] >> 4) | (s1[j-4] >> 6) << 4.  Both cases
// are (A & 0x0F0F) | (B & 0x3030) of the byte pair at 16 (c & 1) in suitably
// shifted words, so every lane runs the same instructions.
struct ScaleSel {
  bool hi;        // c >= 2
  uint32_t sh;    // 16 (c & 1)
  uint32_t shb;   // shift of the word giving bits 4-5: sh (+2 when hi)
  uint32_t shm;   // shift of the word giving m's bits 0-3: sh (+4 when hi)
};
__device__ __forceinline__ ScaleSel scale_sel(int c) {
  ScaleSel r;
  r.hi = c >= 2;
  r.sh = 16u * static_cast<uint32_t>(c & 1);
  r.shb = r.sh + (r.hi ? 2u : 0u);
  r.shm = r.sh + (r.hi ? 4u : 0u);
  return r;
}
// (float(byte 0), float(byte 1)) of v, exact: each byte goes into the
// mantissa of 2^23 with a byte permute and 2^23 is subtracted (no integer
// to float conversion, which runs at a fraction of the FMA rate)
__device__ __forceinline__ float2 bytes01_f2(uint32_t v) {
  const float a = __uint_as_float(__byte_perm(v, 0x4B000000u, 0x7440u));
  const float b = __uint_as_float(__byte_perm(v, 0x4B000000u, 0x7441u));
  return __fadd2_rn(make_float2(a, b), make_float2(-8388608.0f, -8388608.0f));
}

// float(byte i) of v, exact, the same way
__device__ __forceinline__ float byte_f(uint32_t v, int i) {
  return __uint_as_float(__byte_perm(v, 0x4B000000u, 0x7440u | static_cast<uint32_t>(i))) - 8388608.0f;
}

// (sc, m) byte pairs (sub-block 2c in byte 0, 2c+1 in byte 1), 6 bits each
__device__ __forceinline__ void scale_pair6(const ScaleSel& q, uint32_t s0, uint32_t s1,
                                            uint32_t s2, uint32_t& sc, uint32_t& mn) {
  const uint32_t a_sc = (q.hi ? s2 : s0) >> q.sh;
  const uint32_t a_m = (q.hi ? s2 : s1) >> q.shm;
  sc = (a_sc & 0x0F0Fu) | ((s0 >> q.shb) & 0x3030u);
  mn = (a_m & 0x0F0Fu) | ((s1 >> q.shb) & 0x3030u);
}

// One stage of a Q4_K / Q5_K / Q4_G128 tile for the NR live rows of this
// thread.  The lane's unit is bytes off .. off + kCW/2 of chunk c of
// super-block sbl of the slab: the low nibbles belong to sub-block 2c
// (weights 64c + off + r), the high nibbles to 2c+1 (weights 64c + 32 + off +
// r).  Every byte gives one (low, high) pair: converted with one cvt_pair and
// accumulated with one packed fma against the staged (x_lo, x_hi) pair, so
// the accumulators hold (sub-block 2c, sub-block 2c+1) sums and the scales
// apply as pairs too:
//   acc += (d sc_lo, d sc_hi) * S + (-dmin m_lo, -dmin m_hi) * (sx_lo, sx_hi)
// acc[r][k] is a pair whose two halves are added at the end of the tile.
// Word-outer order: the x pairs of one word are loaded once and used for
// every row, so only one word's x is live at a time; the scales are decoded
// after the products.
template <int F, int NT, int RT, int WC, int NR, bool XBF>
__device__ __forceinline__ void stage_q4(const Params& p, const Tile& tl, int sl, int xsl,
                                         uint32_t st, uint32_t xs, int hw, int sbl, int c,
                                         int off, const ScaleSel& ss, float2 (&acc)[RT][NT]) {
  using G = Geo<F, NT, RT, WC>;
  using L = XLayout<F, NT, XBF>;
  constexpr int kCW = G::kCW, NW = kCW / 8;
  constexpr int CH = NT == 1 ? 2 : 1;   // accumulator chains per (row, token)
  const uint32_t magic = kMagic;
  const uint64_t neg = kNegMagic2;
  const int kb = xsl * G::kSlabK + sbl * 256 + 64 * c;   // the chunk's 64-block
  // first staged slot of the unit's x run (token 0), and the token stride
  const uint32_t xrun = xs + L::addr(kb + 2 * off);
  const uint32_t xtok = static_cast<uint32_t>(L::bytes(static_cast<size_t>(p.kpad)));
  // the rows' weight words
  uint32_t w[NR][NW], hq[NR][NW];
  uint32_t rec[NR];
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    const int row = hw + 2 * WC * r;
    const uint32_t rs = st + row * p.slot;
#pragma unroll
    for (int j = 0; j < NW; ++j) hq[r][j] = 0;
    if constexpr (F == kG128) {
      rec[r] = rs;
      lds_words<NW>(rs + 128 * sbl + 32 * c + off, w[r]);
    } else {
      rec[r] = rs + G::kBB * sbl;
      lds_words<NW>(rec[r] + (F == kQ4K ? 16 : 48) + 32 * c + off, w[r]);
      if constexpr (F == kQ5K) lds_words<NW>(rec[r] + 16 + off, hq[r]);
    }
  }
  uint64_t A[NR][NT][CH];   // (lo, hi) pairs, set by the first word's products
  const int rlo = (2 * c + 28) & 31, rhi = (2 * c + 29) & 31;   // Q5_K: bit 2c(+1) -> bit 4
#pragma unroll
  for (int i = 0; i < NW; ++i) {
    // x pairs of word i: xq[k][b] = (x_lo, x_hi) of byte b
    uint64_t xq[NT][4];
#pragma unroll
    for (int k = 0; k < NT; ++k) {
      const uint32_t a = xrun + k * xtok + 8 * i * L::kE;
      x_quad64<XBF>(a, xq[k][0], xq[k][1]);
      x_quad64<XBF>(a + 4 * L::kE, xq[k][2], xq[k][3]);
    }
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      const uint32_t v = w[r][i];
      uint64_t q[4];
      if constexpr (F == kQ5K) {
        const uint32_t h = hq[r][i];
        // byte b of lo5 / hi5 = nibble | fifth bit << 4 (bits 5..7 are
        // masked off by the 5-bit extraction masks)
        const uint32_t lo5 = bitsel(v, __funnelshift_r(h, h, rlo), 0x0F0F0F0Fu);
        const uint32_t hi5 = bitsel(v >> 4, __funnelshift_r(h, h, rhi), 0x0F0F0F0Fu);
        const uint32_t b3 = prmt(lo5, hi5, 0x0703u);   // lo5 byte 3 -> byte 0, hi5 byte 3 -> byte 2
        q[0] = cvt_pair64<0x1Fu, 0x1Fu>(lo5, hi5, magic, neg);
        q[1] = cvt_pair64<0x1F00u, 0x1F00u>(lo5, hi5, magic, neg);
        q[2] = cvt_pair64<0x1F0000u, 0x1F0000u>(lo5, hi5, magic, neg);
        q[3] = cvt_pair64<0x1Fu, 0x1F0000u>(b3, b3, magic, neg);
      } else {
        // lo b0 s0, hi b0 s4, lo b1 s8, hi b1 s12, lo b2 s16 from v; from
        // v >> 12: hi b2 s8, lo b3 s12, hi b3 s16
        const uint32_t u = v >> 12;
        q[0] = cvt_pair64<0xFu, 0xF0u>(v, v, magic, neg);
        q[1] = cvt_pair64<0xF00u, 0xF000u>(v, v, magic, neg);
        q[2] = cvt_pair64<0xF0000u, 0xF00u>(v, u, magic, neg);
        q[3] = cvt_pair64<0xF000u, 0xF0000u>(u, u, magic, neg);
      }
#pragma unroll
      for (int k = 0; k < NT; ++k)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          if (i == 0 && b < CH)
            A[r][k][b % CH] = mul2u(q[b], xq[k][b]);
          else
            fma2u(A[r][k][b % CH], q[b], xq[k][b]);
        }
    }
  }
  // scales, then the stage's contribution
  const uint32_t sxa = xs + static_cast<uint32_t>(L::bytes(static_cast<size_t>(NT) * p.kpad));
  const int parts = p.kpad / G::kPart;
  float2 sxp[NT];
#pragma unroll
  for (int k = 0; k < NT; ++k)
    sxp[k] = lds_f2(sxa + 4 * (k * parts + (kb / 64) * (64 / G::kPart) + 2 * (off / G::kPart)));
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    float2 dsc, ndm;
    if constexpr (F == kG128) {
      const int row = hw + 2 * WC * r;
      // byte offset of the slab's params in its 16-byte aligned copy: (row
      // start + slab start) mod 16, from the row stride mod 16
      const uint32_t po =
          (static_cast<uint32_t>(tl.row0 + row) * ((8u * p.nsb) & 15u) + sl * G::kPBytes) & 15u;
      const uint32_t pa = st + p.pbase + row * p.pslot + po + 8 * sbl;
      const uint2 pr = lds64(pa);
      const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&pr.x));
      const int g = c >> 1;
      const float sc = byte_f(pr.y, g);
      const float mn = byte_f(pr.y, 2 + g);
      dsc = make_float2(dd.x * sc, dd.x * sc);
      ndm = make_float2(-dd.y * mn, -dd.y * mn);
    } else {
      const uint4 hdr = lds128(rec[r]);
      const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&hdr.x));
      uint32_t scp, mnp;
      scale_pair6(ss, hdr.y, hdr.z, hdr.w, scp, mnp);
      dsc = __fmul2_rn(make_float2(dd.x, dd.x), bytes01_f2(scp));
      ndm = __fmul2_rn(make_float2(-dd.y, -dd.y), bytes01_f2(mnp));
    }
#pragma unroll
    for (int k = 0; k < NT; ++k) {
      const float2 S = u2f2(CH == 2 ? add2u(A[r][k][0], A[r][k][CH - 1]) : A[r][k][0]);
      acc[r][k] = __ffma2_rn(dsc, S, acc[r][k]);
      acc[r][k] = __ffma2_rn(ndm, sxp[k], acc[r][k]);
    }
  }
}

// One stage of a Q6_K tile for the NR live rows of this thread.  Unit (h,
// u2): weights 128h + 32t + l0 + l for t < 4, l < kCW/4 (l0 = u2 kCW/4), in
// sub-block 8h + 2t + l0/16.  Byte column l of the unit: ql[64h + l0 + l]
// holds t0 (low nibble) and t2 (high), ql[64h + 32 + l0 + l] holds t1 and t3,
// qh[32h + l0 + l] the two high bits of each.  Each byte column gives the
// pairs (t0, t2), (t1, t3), accumulated with packed fmas against the staged x
// pairs; every 6-bit field converts straight to the signed (q - 32) 2^s (no
// offset to remove afterwards), and the scales apply as the pairs (d sc_t0,
// d sc_t2), (d sc_t1, d sc_t3).  Records start on 2-byte boundaries: words
// are read aligned and shifted.  Word-outer order, as in stage_q4: one
// word's x is live at a time and the scales are decoded after the products.
template <int NT, int RT, int WC, int NR, bool XBF>
__device__ __forceinline__ void stage_q6(const Params& p, const Tile& tl, int sl, int xsl,
                                         uint32_t st, uint32_t xs, int hw, int sbl, int un,
                                         float2 (&acc)[RT][NT]) {
  using G = Geo<kQ6K, NT, RT, WC>;
  using L = XLayout<kQ6K, NT, XBF>;
  constexpr int kCW = G::kCW, QW = kCW / 16;   // words per t-run of the unit: 4, 2, 1
  const uint32_t magic = kMagic;
  const int h = un / (G::kUnitsPerSB / 2);
  const int u2 = un % (G::kUnitsPerSB / 2);
  const int l0 = u2 * (kCW / 4);
  const int su = l0 >> 4;   // sub-block of the unit within each t-run
  const int kb = xsl * G::kSlabK + sbl * 256 + 128 * h;   // the unit's 128-block
  const uint32_t xrun = xs + L::addr(kb + 4 * l0);   // the unit's x run (token 0)
  const uint32_t xtok = static_cast<uint32_t>(L::bytes(static_cast<size_t>(p.kpad)));
  // the rows' words: record base (4-byte aligned) and shift of each row
  uint32_t rb[NR], rsh[NR];
  uint32_t A[NR][QW], B[NR][QW], H[NR][QW];
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    const int row = hw + 2 * WC * r;
    const uint32_t ro =
        (static_cast<uint32_t>(tl.row0 + row) * ((210u * p.nsb) & 15u) + sl * G::kQBytes) & 15u;
    const uint32_t rec = st + row * p.slot + ro + 210 * sbl;
    rb[r] = rec & ~3u;
    rsh[r] = (rec & 3u) * 8u;
    lds_words_rec<QW>(rb[r], rsh[r], 64 * h + l0, A[r]);
    lds_words_rec<QW>(rb[r], rsh[r], 64 * h + 32 + l0, B[r]);
    lds_words_rec<QW>(rb[r], rsh[r], 128 + 32 * h + l0, H[r]);
  }
  float2 a02[NR][NT], a13[NR][NT];
#pragma unroll
  for (int r = 0; r < NR; ++r)
#pragma unroll
    for (int k = 0; k < NT; ++k) a02[r][k] = a13[r][k] = make_float2(0.0f, 0.0f);
  const uint32_t M = 0x0F0F0F0Fu;
#pragma unroll
  for (int j = 0; j < QW; ++j) {
    // x pairs of word j: xq[k][b][0] = (x_t0, x_t2), [1] = (x_t1, x_t3) of column 4j + b
    float2 xq[NT][4][2];
#pragma unroll
    for (int k = 0; k < NT; ++k)
#pragma unroll
      for (int b = 0; b < 4; ++b)
        x_quad<kQ6K, NT, XBF>(xrun + k * xtok + (16 * j + 4 * b) * L::kE, xq[k][b][0], xq[k][b][1]);
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      // 6-bit values of the four t-runs, one per byte (bits 6-7 are masked
      // off by the extraction masks)
      const uint32_t q0 = bitsel(A[r][j], H[r][j] << 4, M);
      const uint32_t q2 = bitsel(A[r][j] >> 4, H[r][j], M);
      const uint32_t q1 = bitsel(B[r][j], H[r][j] << 2, M);
      const uint32_t q3 = bitsel(B[r][j] >> 4, H[r][j] >> 2, M);
      const uint32_t p02 = prmt(q0, q2, 0x0703u);   // byte 3 of q0 -> byte 0, of q2 -> byte 2
      const uint32_t p13 = prmt(q1, q3, 0x0703u);
      // signed (q - 32) 2^s, exact (kNegQ6*)
      float2 c02[4], c13[4];
      c02[0] = cvt_pair<0x3Fu, 0x3Fu>(q0, q2, magic, kNegQ6s0);
      c02[1] = cvt_pair<0x3F00u, 0x3F00u>(q0, q2, magic, kNegQ6s8);
      c02[2] = cvt_pair<0x3F0000u, 0x3F0000u>(q0, q2, magic, kNegQ6s16);
      c02[3] = cvt_pair<0x3Fu, 0x3F0000u>(p02, p02, magic, kNegQ6s0s16);
      c13[0] = cvt_pair<0x3Fu, 0x3Fu>(q1, q3, magic, kNegQ6s0);
      c13[1] = cvt_pair<0x3F00u, 0x3F00u>(q1, q3, magic, kNegQ6s8);
      c13[2] = cvt_pair<0x3F0000u, 0x3F0000u>(q1, q3, magic, kNegQ6s16);
      c13[3] = cvt_pair<0x3Fu, 0x3F0000u>(p13, p13, magic, kNegQ6s0s16);
#pragma unroll
      for (int k = 0; k < NT; ++k)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          a02[r][k] = __ffma2_rn(c02[b], xq[k][b][0], a02[r][k]);
          a13[r][k] = __ffma2_rn(c13[b], xq[k][b][1], a13[r][k]);
        }
    }
  }
  // scales of the unit's sub-blocks: t0 byte su, t1 su+2 (of S[0]), t2 su,
  // t3 su+2 (of S[1]); sign-extended with a byte permute
  const uint32_t sel0 = su | ((8 | su) << 4) | ((8 | su) << 8) | ((8 | su) << 12);
  const uint32_t sel2 = (su + 2) | ((10 + su) << 4) | ((10 + su) << 8) | ((10 + su) << 12);
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    uint32_t S[2], D[1];
    lds_words_rec<2>(rb[r], rsh[r], 192 + 8 * h, S);
    lds_words_rec<1>(rb[r], rsh[r], 208, D);
    const float d = half_bits_to_float(D[0] & 0xFFFFu);
    const float2 ds02 = make_float2(d * static_cast<float>(static_cast<int>(prmt(S[0], 0, sel0))),
                                    d * static_cast<float>(static_cast<int>(prmt(S[1], 0, sel0))));
    const float2 ds13 = make_float2(d * static_cast<float>(static_cast<int>(prmt(S[0], 0, sel2))),
                                    d * static_cast<float>(static_cast<int>(prmt(S[1], 0, sel2))));
#pragma unroll
    for (int k = 0; k < NT; ++k) {
      acc[r][k] = __ffma2_rn(ds02, a02[r][k], acc[r][k]);
      acc[r][k] = __ffma2_rn(ds13, a13[r][k], acc[r][k]);
    }
  }
}

// ------------------------------------------- int8 activations (dp4a)
//
// The x mode XM == kXQ8 of gemv_stream: the activations are quantised to
// int8 per 32 positions of a token, dx = amax / 127 and xq = rint(x / dx),
// both in binary32 (the daily.dev summary says the CUDA backend runs the
// K-quant weights as integer GEMV with dp4a; block size and rounding are
// this library's reading), and every sub-block's dot product is an exact
// integer sum built with dp4a (four int8 products per instruction):
//   y += dx (d sc sum q xq - dmin m sum xq)        (Q4_K, Q5_K, Q4_G128)
//   y += dx  d sc (sum q xq - 32 sum xq)            (Q6_K)
// The staged segment holds the codes in position order (16 bytes of padding
// per 64 positions, so a half-warp's 16-byte loads of different units hit
// different banks), then dx per 32 positions, then the code sum of every
// part (kPart positions: the run of one unit within one sub-block).
constexpr int kXF32 = 0, kXBF16 = 1, kXQ8 = 2;

__host__ __device__ constexpr uint32_t q8_row_bytes(int kpad) {
  return static_cast<uint32_t>(kpad + 16 * (kpad / 64));
}
__host__ __device__ constexpr uint32_t q8_x_bytes(int nt, int kpad, int part) {
  return (static_cast<uint32_t>(nt) * q8_row_bytes(kpad) + 4u * nt * (kpad / 32) +
          4u * nt * (kpad / part) + 127u) & ~127u;
}
__device__ __forceinline__ uint32_t q8_pos(int pos) { return static_cast<uint32_t>(pos + 16 * (pos / 64)); }

// The int8 code of x (binary32) for the block step d: rint(x / d) with the
// division rounded to nearest, 0 when d == 0.
__device__ __forceinline__ int q8_code(float v, float d) {
  if (!(d > 0.0f)) return 0;
  int q = __float2int_rn(__fdiv_rn(v, d));
  return q > 127 ? 127 : (q < -127 ? -127 : q);
}

template <int F, int NT>
__device__ void stage_x_q8(const Params& p, uint8_t* smem, int kbase) {
  using G = Geo<F, NT, 1, 1>;
  constexpr int P = G::kPart;              // positions per part sum: 32..4
  const uint32_t rowb = q8_row_bytes(p.kpad);
  float* dxs = reinterpret_cast<float*>(smem + NT * rowb);
  int* ps = reinterpret_cast<int*>(dxs + NT * (p.kpad / 32));
  const int per_tok = p.kpad / 8;          // items of 8 positions (a multiple of 32)
  const int lane = threadIdx.x & 31;
  for (int base = static_cast<int>(threadIdx.x) & ~31; base < NT * per_tok;
       base += static_cast<int>(blockDim.x)) {
    const int q = base + lane;
    const int tk = q / per_tok, c = q % per_tok;
    const int k = kbase + 8 * c;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (tk < p.nt && k < p.K) v = *reinterpret_cast<const uint4*>(p.x + static_cast<int64_t>(tk) * p.K + k);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float f[8];
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      f[2 * j] = __uint_as_float(w[j] << 16);
      f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
      amax = fmaxf(amax, fmaxf(fabsf(f[2 * j]), fabsf(f[2 * j + 1])));
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
    const float d = __fdiv_rn(amax, 127.0f);
    int qs[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) qs[j] = q8_code(f[j], d);
    uint32_t b0 = 0, b1 = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      b0 |= (static_cast<uint32_t>(qs[j]) & 0xFFu) << (8 * j);
      b1 |= (static_cast<uint32_t>(qs[4 + j]) & 0xFFu) << (8 * j);
    }
    *reinterpret_cast<uint2*>(smem + tk * rowb + q8_pos(8 * c)) = make_uint2(b0, b1);
    if ((c & 3) == 0) dxs[tk * (p.kpad / 32) + c / 4] = d;
    // code sums per part
    int s0 = qs[0] + qs[1] + qs[2] + qs[3], s1 = qs[4] + qs[5] + qs[6] + qs[7];
    if constexpr (P == 4) {
      ps[tk * (p.kpad / 4) + 2 * c] = s0;
      ps[tk * (p.kpad / 4) + 2 * c + 1] = s1;
    } else {
      int sp = s0 + s1;
      if constexpr (P >= 16) sp += __shfl_xor_sync(0xFFFFFFFFu, sp, 1);
      if constexpr (P >= 32) sp += __shfl_xor_sync(0xFFFFFFFFu, sp, 2);
      if ((c & (P / 8 - 1)) == 0) ps[tk * (p.kpad / P) + c / (P / 8)] = sp;
    }
  }
}

// NW consecutive 32-bit words of the staged codes from shared address a
// (16-byte aligned for NW >= 4, 8-byte aligned for NW == 2)
template <int NW>
__device__ __forceinline__ void lds_codes(uint32_t a, uint32_t (&w)[NW]) {
#pragma unroll
  for (int i = 0; i < NW; i += 4) {
    if constexpr (NW >= 4) {
      const uint4 v = lds128(a + 4 * i);
      w[i] = v.x; w[i + 1] = v.y; w[i + 2] = v.z; w[i + 3] = v.w;
    } else {
      const uint2 v = lds64(a);
      w[0] = v.x; w[1] = v.y;
    }
  }
}

// One stage of a Q4_K / Q5_K / Q4_G128 tile on int8 activations, for the NR
// live rows of this thread (unit and accumulators as in stage_q4).
template <int F, int NT, int RT, int WC, int NR>
__device__ __forceinline__ void stage_q4_q8(const Params& p, const Tile& tl, int sl, int xsl,
                                            uint32_t st, uint32_t xs, int hw, int sbl, int c,
                                            int off, const ScaleSel& ss, float2 (&acc)[RT][NT]) {
  using G = Geo<F, NT, RT, WC>;
  constexpr int kCW = G::kCW, NW = kCW / 8, P = G::kPart;
  const int kb = xsl * G::kSlabK + sbl * 256 + 64 * c;   // the chunk's 64-block
  const uint32_t rowb = q8_row_bytes(p.kpad);
  const uint32_t dxa = xs + NT * rowb;
  const uint32_t psa = dxa + 4u * NT * (p.kpad / 32);
  uint32_t w[NR][NW], hq[NR][NW];
  uint32_t rec[NR];
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    const uint32_t rs = st + (hw + 2 * WC * r) * p.slot;
#pragma unroll
    for (int j = 0; j < NW; ++j) hq[r][j] = 0;
    if constexpr (F == kG128) {
      rec[r] = rs;
      lds_words<NW>(rs + 128 * sbl + 32 * c + off, w[r]);
    } else {
      rec[r] = rs + G::kBB * sbl;
      lds_words<NW>(rec[r] + (F == kQ4K ? 16 : 48) + 32 * c + off, w[r]);
      if constexpr (F == kQ5K) lds_words<NW>(rec[r] + 16 + off, hq[r]);
    }
  }
  const int rlo = (2 * c + 28) & 31, rhi = (2 * c + 29) & 31;   // Q5_K: bit 2c(+1) -> bit 4
  int il[NR][NT], ih[NR][NT];
#pragma unroll
  for (int r = 0; r < NR; ++r)
#pragma unroll
    for (int k = 0; k < NT; ++k) il[r][k] = ih[r][k] = 0;
#pragma unroll
  for (int k = 0; k < NT; ++k) {
    uint32_t xl[NW], xh[NW];
    lds_codes<NW>(xs + k * rowb + q8_pos(kb + off), xl);
    lds_codes<NW>(xs + k * rowb + q8_pos(kb + 32 + off), xh);
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
      for (int i = 0; i < NW; ++i) {
        uint32_t lo = w[r][i] & 0x0F0F0F0Fu, hi = (w[r][i] >> 4) & 0x0F0F0F0Fu;
        if constexpr (F == kQ5K) {
          lo |= __funnelshift_r(hq[r][i], hq[r][i], rlo) & 0x10101010u;
          hi |= __funnelshift_r(hq[r][i], hq[r][i], rhi) & 0x10101010u;
        }
        il[r][k] = __dp4a(static_cast<int>(lo), static_cast<int>(xl[i]), il[r][k]);
        ih[r][k] = __dp4a(static_cast<int>(hi), static_cast<int>(xh[i]), ih[r][k]);
      }
  }
  // scales: acc += (dx_lo, dx_hi) * (d sc * sum q xq - dmin m * sum xq)
  float2 dxp[NT], sxp[NT];
#pragma unroll
  for (int k = 0; k < NT; ++k) {
    dxp[k] = lds_f2(dxa + 4u * (k * (p.kpad / 32) + kb / 32));
    int slo, shi;
    asm volatile("ld.shared.s32 %0, [%1];" : "=r"(slo) : "r"(psa + 4u * (k * (p.kpad / P) + (kb + off) / P)));
    asm volatile("ld.shared.s32 %0, [%1];" : "=r"(shi) : "r"(psa + 4u * (k * (p.kpad / P) + (kb + 32 + off) / P)));
    sxp[k] = make_float2(static_cast<float>(slo), static_cast<float>(shi));
  }
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    float2 dsc, ndm;
    if constexpr (F == kG128) {
      const int row = hw + 2 * WC * r;
      const uint32_t po =
          (static_cast<uint32_t>(tl.row0 + row) * ((8u * p.nsb) & 15u) + sl * G::kPBytes) & 15u;
      const uint2 pr = lds64(st + p.pbase + row * p.pslot + po + 8 * sbl);
      const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&pr.x));
      const int g = c >> 1;
      const float sc = byte_f(pr.y, g);
      const float mn = byte_f(pr.y, 2 + g);
      dsc = make_float2(dd.x * sc, dd.x * sc);
      ndm = make_float2(-dd.y * mn, -dd.y * mn);
    } else {
      const uint4 hdr = lds128(rec[r]);
      const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&hdr.x));
      uint32_t scp, mnp;
      scale_pair6(ss, hdr.y, hdr.z, hdr.w, scp, mnp);
      dsc = __fmul2_rn(make_float2(dd.x, dd.x), bytes01_f2(scp));
      ndm = __fmul2_rn(make_float2(-dd.y, -dd.y), bytes01_f2(mnp));
    }
#pragma unroll
    for (int k = 0; k < NT; ++k) {
      const float2 t = __ffma2_rn(dsc, make_float2(static_cast<float>(il[r][k]), static_cast<float>(ih[r][k])),
                                  __fmul2_rn(ndm, sxp[k]));
      acc[r][k] = __ffma2_rn(dxp[k], t, acc[r][k]);
    }
  }
}

// One stage of a Q6_K tile on int8 activations (unit as in stage_q6: four
// t-runs of kCW/4 positions; each 6-bit field is assembled into a byte and
// multiplied with dp4a, and q - 32 becomes sum q xq - 32 sum xq, exactly).
template <int NT, int RT, int WC, int NR>
__device__ __forceinline__ void stage_q6_q8(const Params& p, const Tile& tl, int sl, int xsl,
                                            uint32_t st, uint32_t xs, int hw, int sbl, int un,
                                            float2 (&acc)[RT][NT]) {
  using G = Geo<kQ6K, NT, RT, WC>;
  constexpr int kCW = G::kCW, QW = kCW / 16, P = G::kPart;
  const int h = un / (G::kUnitsPerSB / 2);
  const int u2 = un % (G::kUnitsPerSB / 2);
  const int l0 = u2 * (kCW / 4);
  const int su = l0 >> 4;
  const int kb = xsl * G::kSlabK + sbl * 256 + 128 * h;   // the unit's 128-block
  const uint32_t rowb = q8_row_bytes(p.kpad);
  const uint32_t dxa = xs + NT * rowb;
  const uint32_t psa = dxa + 4u * NT * (p.kpad / 32);
  uint32_t rb[NR], rsh[NR];
  uint32_t A[NR][QW], B[NR][QW], H[NR][QW];
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    const int row = hw + 2 * WC * r;
    const uint32_t ro =
        (static_cast<uint32_t>(tl.row0 + row) * ((210u * p.nsb) & 15u) + sl * G::kQBytes) & 15u;
    const uint32_t rec = st + row * p.slot + ro + 210 * sbl;
    rb[r] = rec & ~3u;
    rsh[r] = (rec & 3u) * 8u;
    lds_words_rec<QW>(rb[r], rsh[r], 64 * h + l0, A[r]);
    lds_words_rec<QW>(rb[r], rsh[r], 64 * h + 32 + l0, B[r]);
    lds_words_rec<QW>(rb[r], rsh[r], 128 + 32 * h + l0, H[r]);
  }
  int it[NR][NT][4];
#pragma unroll
  for (int r = 0; r < NR; ++r)
#pragma unroll
    for (int k = 0; k < NT; ++k)
#pragma unroll
      for (int t = 0; t < 4; ++t) it[r][k][t] = 0;
  const uint32_t M = 0x0F0F0F0Fu, M6 = 0x3F3F3F3Fu;
#pragma unroll
  for (int k = 0; k < NT; ++k) {
    uint32_t xt[4][QW];   // codes of t-run t, positions l0 .. l0 + kCW/4
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      if constexpr (QW >= 4) {
        lds_codes<QW>(xs + k * rowb + q8_pos(kb + 32 * t + l0), xt[t]);
      } else if constexpr (QW == 2) {
        lds_codes<2>(xs + k * rowb + q8_pos(kb + 32 * t + l0), xt[t]);
      } else {
        xt[t][0] = lds32(xs + k * rowb + q8_pos(kb + 32 * t + l0));
      }
    }
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
      for (int j = 0; j < QW; ++j) {
        const uint32_t q0 = bitsel(A[r][j], H[r][j] << 4, M) & M6;
        const uint32_t q2 = bitsel(A[r][j] >> 4, H[r][j], M) & M6;
        const uint32_t q1 = bitsel(B[r][j], H[r][j] << 2, M) & M6;
        const uint32_t q3 = bitsel(B[r][j] >> 4, H[r][j] >> 2, M) & M6;
        it[r][k][0] = __dp4a(static_cast<int>(q0), static_cast<int>(xt[0][j]), it[r][k][0]);
        it[r][k][1] = __dp4a(static_cast<int>(q1), static_cast<int>(xt[1][j]), it[r][k][1]);
        it[r][k][2] = __dp4a(static_cast<int>(q2), static_cast<int>(xt[2][j]), it[r][k][2]);
        it[r][k][3] = __dp4a(static_cast<int>(q3), static_cast<int>(xt[3][j]), it[r][k][3]);
      }
  }
  // per t-run: the code sum of its part and dx of its 32 positions
  float2 dx02[NT], dx13[NT];
  int s[NT][4];
#pragma unroll
  for (int k = 0; k < NT; ++k) {
    const float4 d4 = lds_f4(dxa + 4u * (k * (p.kpad / 32) + kb / 32));   // t-runs 0..3
    dx02[k] = make_float2(d4.x, d4.z);
    dx13[k] = make_float2(d4.y, d4.w);
#pragma unroll
    for (int t = 0; t < 4; ++t)
      asm volatile("ld.shared.s32 %0, [%1];"
                   : "=r"(s[k][t])
                   : "r"(psa + 4u * (k * (p.kpad / P) + (kb + 32 * t + l0) / P)));
  }
  const uint32_t sel0 = su | ((8 | su) << 4) | ((8 | su) << 8) | ((8 | su) << 12);
  const uint32_t sel2 = (su + 2) | ((10 + su) << 4) | ((10 + su) << 8) | ((10 + su) << 12);
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    uint32_t S[2], D[1];
    lds_words_rec<2>(rb[r], rsh[r], 192 + 8 * h, S);
    lds_words_rec<1>(rb[r], rsh[r], 208, D);
    const float d = half_bits_to_float(D[0] & 0xFFFFu);
    const float2 ds02 = make_float2(d * static_cast<float>(static_cast<int>(prmt(S[0], 0, sel0))),
                                    d * static_cast<float>(static_cast<int>(prmt(S[1], 0, sel0))));
    const float2 ds13 = make_float2(d * static_cast<float>(static_cast<int>(prmt(S[0], 0, sel2))),
                                    d * static_cast<float>(static_cast<int>(prmt(S[1], 0, sel2))));
#pragma unroll
    for (int k = 0; k < NT; ++k) {
      const float2 i02 = make_float2(static_cast<float>(it[r][k][0] - 32 * s[k][0]),
                                     static_cast<float>(it[r][k][2] - 32 * s[k][2]));
      const float2 i13 = make_float2(static_cast<float>(it[r][k][1] - 32 * s[k][1]),
                                     static_cast<float>(it[r][k][3] - 32 * s[k][3]));
      acc[r][k] = __ffma2_rn(__fmul2_rn(dx02[k], ds02), i02, acc[r][k]);
      acc[r][k] = __ffma2_rn(__fmul2_rn(dx13[k], ds13), i13, acc[r][k]);
    }
  }
}

constexpr int kMaxStages = 8;

// Registers capped so that three CTAs (two with eight consumer warps) fit an SM.
// XM: how x is staged -- kXF32 (fp32, pre-scaled), kXBF16 (bf16, when fp32
// would not fit) or kXQ8 (int8 codes: the dp4a path).
template <int F, int NT, int RT, int WC, int XM>
__global__ void __launch_bounds__((WC + 1) * 32, WC == 8 ? 2 : 3)
    gemv_stream(const __grid_constant__ Params p, int stages) {
  constexpr bool XBF = XM == kXBF16;
  using G = Geo<F, NT, RT, WC>;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[2 * kMaxStages];
  __shared__ int last_flag;
  __shared__ int stage_tile[kMaxStages];   // tile of each ring slot; -1: no more tiles
  const uint32_t bar_full = smem_addr(&bars[0]);
  const uint32_t bar_empty = smem_addr(&bars[kMaxStages]);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t xs = smem_addr(smem);
  const uint32_t ring_a = xs + p.x_bytes;
  // CTA c works on K segment c % ksplit: first on its fixed tiles
  // c / ksplit + i * cps (i < static_tiles), then on tiles it claims from
  // the segment's counter until none is left, so that CTAs which stream
  // faster take more tiles
  const int kseg = static_cast<int>(blockIdx.x) % p.ksplit;
  const int cta = static_cast<int>(blockIdx.x) / p.ksplit;
  const int cps = static_cast<int>(gridDim.x) / p.ksplit;   // CTAs per segment
  const int sl0 = kseg * p.slabs;         // first slab (of the row) of the segment
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(bar_full + 8 * s, p.tma ? 1 : 32);   // the issuing lane / every producer lane
      mbar_init(bar_empty + 8 * s, WC);     // one arrival per consumer warp
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const bool producer = warp == WC;
  // Programmatic dependent launch: the next kernel on the stream may start
  // its CTAs as SMs free up; it reads its activations, the scheduler counters
  // and the split-K scratch only after its own griddepcontrol.wait, i.e.
  // after this grid has completed.
  asm volatile("griddepcontrol.launch_dependents;");
  Ring ring;
  if (producer) produce_prefill<G>(p, smem, ring_a, bar_full, stage_tile, stages, cta, cps, sl0, ring);
  // x may be produced by the previous kernel: wait for it to complete
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if constexpr (XM == kXQ8)
    stage_x_q8<F, NT>(p, smem, kseg * p.kpad);
  else
    stage_x<F, NT, XBF>(p, smem, kseg * p.kpad);
  __syncthreads();
  if (producer) {
    produce_rest<G>(p, smem, ring_a, bar_full, bar_empty, stage_tile, stages, cta, cps, kseg, sl0,
                    ring);
    return;
  }
  // consumers
  constexpr int kCW = G::kCW;
  const int hw = 2 * warp + (lane >> 4);   // half-warp: rows hw + 2 WC r of a tile
  const int ul = lane & 15;                // unit position in the slab
  const int sbl = ul / G::kUnitsPerSB;     // super-block in the slab
  const int un = ul % G::kUnitsPerSB;      // unit in the super-block
  const int c = un / (64 / kCW);           // Q4 family: chunk
  const int off = (un % (64 / kCW)) * (kCW / 2);
  const ScaleSel ss = scale_sel(c);
  float2 acc[RT][NT];
  Tile tl{};
  int t = 0;
  // slab within the segment, ring slot and full-barrier parity, advanced by
  // counting (no division per stage)
  int xsl = 0, slot = 0;
  uint32_t parity = 0;
  for (;;) {
    const int sl = sl0 + xsl;       // slab within the row
    if (!mbar_wait_warp(bar_full + 8 * slot, parity)) return;
    if (xsl == 0) {
      t = stage_tile[slot];
      if (t < 0) return;
      tl = tile_of(p, t);
#pragma unroll
      for (int r = 0; r < RT; ++r)
#pragma unroll
        for (int k = 0; k < NT; ++k) acc[r][k] = make_float2(0.0f, 0.0f);
    }
    const uint32_t st = ring_a + slot * p.stage;
    if (sl * G::kSlabSB + sbl < p.nsb) {
      // rows of this half-warp inside the tile (the same for all its lanes)
      const int nr = tl.rcnt > hw ? min(RT, (tl.rcnt - hw + 2 * WC - 1) / (2 * WC)) : 0;
      auto run = [&](auto nrc) {
        constexpr int NR = decltype(nrc)::value;
        if constexpr (XM == kXQ8) {
          if constexpr (F == kQ6K)
            stage_q6_q8<NT, RT, WC, NR>(p, tl, sl, xsl, st, xs, hw, sbl, un, acc);
          else
            stage_q4_q8<F, NT, RT, WC, NR>(p, tl, sl, xsl, st, xs, hw, sbl, c, off, ss, acc);
        } else if constexpr (F == kQ6K) {
          stage_q6<NT, RT, WC, NR, XBF>(p, tl, sl, xsl, st, xs, hw, sbl, un, acc);
        } else {
          stage_q4<F, NT, RT, WC, NR, XBF>(p, tl, sl, xsl, st, xs, hw, sbl, c, off, ss, acc);
        }
      };
      if (nr == RT) {
        run(std::integral_constant<int, RT>{});
      } else if constexpr (RT >= 2) {
        if (nr == 1) run(std::integral_constant<int, 1>{});
        if constexpr (RT == 4) {
          if (nr == 2)
            run(std::integral_constant<int, 2>{});
          else if (nr == 3)
            run(std::integral_constant<int, 3>{});
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * slot);
    if (xsl == p.slabs - 1) {
      float red[RT][NT];
#pragma unroll
      for (int r = 0; r < RT; ++r)
#pragma unroll
        for (int k = 0; k < NT; ++k) {
          float v = acc[r][k].x + acc[r][k].y;
          v += __shfl_xor_sync(0xFFFFFFFFu, v, 8);
          v += __shfl_xor_sync(0xFFFFFFFFu, v, 4);
          v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
          v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
          red[r][k] = v;
        }
      float* y = pick(p.g.y, tl.mi);
      const int64_t N = pick(p.g.N, tl.mi);
      if (p.ksplit == 1) {
        if (ul == 0) {
#pragma unroll
          for (int r = 0; r < RT; ++r) {
            const int row = hw + 2 * WC * r;
            if (row < tl.rcnt) {
#pragma unroll
              for (int k = 0; k < NT; ++k)
                if (k < p.nt) y[static_cast<int64_t>(k) * N + tl.row0 + row] = red[r][k];
            }
          }
        }
      } else {
        // split-K: publish this segment's partial sums (tagged); the last
        // CTA of the tile to arrive adds the segments in order
        // 0..ksplit-1 and re-arms the counter
        uint64_t* part = static_cast<uint64_t*>(p.part) + static_cast<int64_t>(t) * p.tile_rows * NT;
        const int64_t seg_stride = static_cast<int64_t>(p.tiles) * p.tile_rows * NT;
        if (ul == 0) {
#pragma unroll
          for (int r = 0; r < RT; ++r) {
            const int row = hw + 2 * WC * r;
            if (row < tl.rcnt) {
#pragma unroll
              for (int k = 0; k < NT; ++k)
                put_partial(part + kseg * seg_stride + row * NT + k, red[r][k], p.tag);
            }
          }
        }
        // one arrival per CTA, after every warp has published
        asm volatile("bar.sync 1, %0;" ::"r"(WC * 32) : "memory");
        if (threadIdx.x == 0)
          last_flag = atomicAdd(p.arrivals + t, 1u) == static_cast<unsigned>(p.ksplit - 1);
        asm volatile("bar.sync 1, %0;" ::"r"(WC * 32) : "memory");
        if (last_flag) {
          // every consumer thread takes (row, token) values of the tile
          for (int e = static_cast<int>(threadIdx.x); e < tl.rcnt * NT; e += WC * 32) {
            const int row = e / NT, k = e % NT;
            const float v = take_partials(part + e, seg_stride, p.ksplit, p.tag);
            if (k < p.nt) y[static_cast<int64_t>(k) * N + tl.row0 + row] = v;
          }
          if (threadIdx.x == 0) p.arrivals[t] = 0u;
        }
      }
    }
    if (++xsl == p.slabs) xsl = 0;
    if (++slot == stages) {
      slot = 0;
      parity ^= 1u;
    }
  }
}

// ============================================================ verify kernel
//
// n_tok 5..16 (speculative verify): the products run on the tensor cores as
// mma.sync m16n8k16 (bf16 operands, fp32 accumulators).  A = weights: a warp
// owns 16 rows of a tile; each qs byte's nibble becomes the exact bf16 value
// q (one LOP3 builds two bf16 128 + q: (w & 0x000F000F) | 0x43004300, and one
// bf16 subtraction of (128, 128) leaves (q, q); Q6_K subtracts 160 and gets
// q - 32).  No offset is left in the products, so a record whose weights are
// zero contributes exactly zero whatever its scales.  B = x,
// eight tokens per mma (two mmas per A fragment for 9..16 tokens): the CTA's
// K segment of x is staged once as bf16 in shared memory, one row per token
// padded by 64 bytes so that the eight tokens of a fragment load hit
// different banks.  Per sub-block the accumulator holds D = sum q x, and (Q4
// family) a second mma against an all-ones A gives Sx for the min term, so
//   y += s1 D + s2 Sx,  s1 = d sc,  s2 = -dmin m                  (Q4 family)
//   y += s1 D,          s1 = d sc,  D = sum (q - 32) x            (Q6_K)
// s1, s2 per (row, sub-block) are decoded once per stage into a per-warp
// shared table.  The weight ring, tiling, split-K and bounded waits are those
// of gemv_stream.

template <int F, int WC_>
struct MGeo {
  static constexpr int kF = F;
  static constexpr int kWC = WC_;
  static constexpr int kThreads = (WC_ + 1) * 32;
  static constexpr int kRows = 16 * WC_;     // a warp owns 16 rows of a tile
  static constexpr int kSlabSB = 2;
  static constexpr int kSlabK = 512;
  static constexpr int kBB = block_bytes(F);
  static constexpr int kQBytes = (F == kG128) ? 128 * kSlabSB : kBB * kSlabSB;
  static constexpr int kPBytes = (F == kG128) ? 8 * kSlabSB : 0;
  static constexpr int round16(int b) { return (b + 15) / 16 * 16; }
  // row pitch an odd multiple of 16 bytes: the 8 rows a warp reads at once
  // start in 8 different 16-byte bank groups (a tensor copy's box then reads
  // up to 16 bytes of the next slab, or zeros past the row)
  static constexpr int odd16(int b) { return (b / 16) % 2 ? b : b + 16; }
  static constexpr int kSlotTma = odd16(round16(kQBytes + (kQBytes % 16 ? 15 : 0)));
  static constexpr int kPSlotTma = (F == kG128) ? round16(kPBytes + (kPBytes % 16 ? 15 : 0)) : 0;
  static constexpr int kSlotBulk = odd16(round16(kQBytes + 16));
  static constexpr int kPSlotBulk = (F == kG128) ? round16(kPBytes + 16) : 0;
  // per-warp scale table, one row of float4 per weight row (+1 float4 of
  // padding against bank conflicts):
  //   Q4 family: (row, s, c) -> (s1, s1, s2, s2) of sub-block 2c, then of 2c+1
  //   Q6_K:      (row, s, j) -> (s1, s1) of sub-block j (two per float4)
  static constexpr int kTabRow = (F == kQ6K) ? kSlabSB * 8 + 1 : kSlabSB * 8 + 1;
  static constexpr int kTabBytes = 16 * kTabRow * 16;
  // bytes of padding per staged token row of x: the B loads of the eight
  // tokens of a fragment (16-byte loads in 8-lane phases for the Q4 family,
  // 8-byte loads in 16-lane phases for Q6_K) fall in distinct banks
  static constexpr int kXPad = (F == kQ6K) ? 32 : 64;
};

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// (w & mask) | magic as one LOP3 (mask an immediate)
template <uint32_t M>
__device__ __forceinline__ uint32_t lop_or(uint32_t w, uint32_t magic) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(w), "n"(M), "r"(magic));
  return d;
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint2 ldg_nc_v2(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

constexpr uint32_t kBf16Magic2 = 0x43004300u;   // bf16 (128, 128)

// prmt selector: byte b of the source, sign-extended to 32 bits
__device__ __forceinline__ uint32_t sext_sel(uint32_t b) { return b | ((8u | b) * 0x1110u); }
constexpr uint32_t kBf16One2 = 0x3F803F80u;     // bf16 (1, 1)

constexpr uint32_t kBf16Q6Zero2 = 0x43204320u;  // bf16 (160, 160) = 128 + the Q6_K zero point 32

// Exact bf16 pairs of the fields under mask M in bytes (0, 1) and in bytes
// (2, 3) of v: the two bytes of a pair are moved to the two halves with a
// byte permute (a pair is two consecutive positions), one LOP3 makes the
// bf16 (128 + field), and one bf16 subtraction of `off` leaves field + 128 -
// off exactly: the field itself (off = 128) or Q6_K's q - 32 (off = 160).
template <uint32_t M>
__device__ __forceinline__ void bf16_pairs(uint32_t v, uint32_t off, uint32_t& p01, uint32_t& p23) {
  p01 = bf16x2_sub(lop_or<M>(prmt(v, 0, 0x4140u), kBf16Magic2), off);
  p23 = bf16x2_sub(lop_or<M>(prmt(v, 0, 0x4342u), kBf16Magic2), off);
}

// The per-warp scale table of one stage: lane -> (row = lane & 15, super-block
// s = lane >> 4) of the warp's 16 rows.
template <class G>
__device__ __forceinline__ void build_scale_table(const Params& p, const Tile& tl, int sl,
                                                  uint32_t st, int rbase, uint32_t tab) {
  constexpr int F = G::kF;
  const int lane = threadIdx.x & 31;
  const int row = rbase + (lane & 15), s = lane >> 4;
  const uint32_t trow = tab + static_cast<uint32_t>((lane & 15) * G::kTabRow * 16);
  if constexpr (F == kQ6K) {
    const uint32_t ro =
        (static_cast<uint32_t>(tl.row0 + row) * ((210u * p.nsb) & 15u) + sl * G::kQBytes) & 15u;
    const uint32_t rec = st + row * p.slot + ro + 210 * s;
    uint32_t S[4], D[1];
    lds_words_a2<4>(rec + 192, S);
    lds_words_a2<1>(rec + 208, D);
    const float d = half_bits_to_float(D[0] & 0xFFFFu);
#pragma unroll
    for (int j = 0; j < 16; j += 2) {
      const uint32_t w = S[j >> 2];
      const uint32_t sh = 8 * (j & 3);
      const float a = d * static_cast<float>(static_cast<int>(prmt(w, 0, sext_sel(sh / 8))));
      const float b = d * static_cast<float>(static_cast<int>(prmt(w, 0, sext_sel(sh / 8 + 1))));
      sts128(trow + (s * 8 + j / 2) * 16, make_float4(a, a, b, b));
    }
  } else if constexpr (F == kG128) {
    const uint32_t po =
        (static_cast<uint32_t>(tl.row0 + row) * ((8u * p.nsb) & 15u) + sl * G::kPBytes) & 15u;
    const uint2 pr = lds64(st + p.pbase + row * p.pslot + po + 8 * s);
    const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&pr.x));
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      const float s1 = dd.x * byte_f(pr.y, g);
      const float s2 = -(dd.y * byte_f(pr.y, 2 + g));
      const float4 e = make_float4(s1, s1, s2, s2);
#pragma unroll
      for (int c = 2 * g; c < 2 * g + 2; ++c) {
        sts128(trow + ((s * 4 + c) * 2) * 16, e);
        sts128(trow + ((s * 4 + c) * 2 + 1) * 16, e);
      }
    }
  } else {
    const uint4 hdr = lds128(st + row * p.slot + G::kBB * s);
    const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&hdr.x));
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t scp, mnp;
      scale_pair6(scale_sel(c), hdr.y, hdr.z, hdr.w, scp, mnp);
      const float s1l = dd.x * bytes01_f2(scp).x;
      const float s1h = dd.x * bytes01_f2(scp).y;
      const float s2l = -(dd.y * bytes01_f2(mnp).x);
      const float s2h = -(dd.y * bytes01_f2(mnp).y);
      sts128(trow + ((s * 4 + c) * 2) * 16, make_float4(s1l, s1l, s2l, s2l));
      sts128(trow + ((s * 4 + c) * 2 + 1) * 16, make_float4(s1h, s1h, s2h, s2h));
    }
  }
}

// y += s1 D + s2 Sx for the two rows (g, g+8) of this thread and tokens
// (2t, 2t+1) of one n8 block; e = the rows' (s1, s1, s2, s2)
__device__ __forceinline__ void mma_epilogue(float2 (&acc)[2], const float (&d)[4],
                                             const float (&sx)[4], float4 eg, float4 eg8) {
  const float2 x01 = make_float2(sx[0], sx[1]);
  acc[0] = __ffma2_rn(make_float2(eg.x, eg.y), make_float2(d[0], d[1]), acc[0]);
  acc[0] = __ffma2_rn(make_float2(eg.z, eg.w), x01, acc[0]);
  acc[1] = __ffma2_rn(make_float2(eg8.x, eg8.y), make_float2(d[2], d[3]), acc[1]);
  acc[1] = __ffma2_rn(make_float2(eg8.z, eg8.w), x01, acc[1]);
}

// One stage of the verify kernel for this warp's 16 rows (Q4 family).
template <class G, int NB>
__device__ __forceinline__ void mma_stage_q4(const Params& p, const Tile& tl, int sl, int kx,
                                             uint32_t st, int rbase, uint32_t tab, uint32_t xsh,
                                             uint32_t xstride, float2 (&acc)[NB][2]) {
  constexpr int F = G::kF;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const uint32_t ones = kBf16One2;
#pragma unroll
  for (int s = 0; s < G::kSlabSB; ++s) {
    if (sl * G::kSlabSB + s >= p.nsb) break;
    // this thread's rows g and g+8: qs bytes 8t .. 8t+7 of every chunk
    uint32_t rq[2], rh[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = rbase + g + 8 * h;
      if constexpr (F == kG128) {
        rq[h] = st + row * p.slot + 128 * s + 8 * t;
      } else {
        const uint32_t rec = st + row * p.slot + G::kBB * s;
        rq[h] = rec + (F == kQ4K ? 16 : 48) + 8 * t;
        rh[h] = rec + 16 + 8 * t;
      }
    }
    uint2 qh[2] = {};
    if constexpr (F == kQ5K) {
      qh[0] = lds64(rh[0]);
      qh[1] = lds64(rh[1]);
    }
    // staged x of this super-block: tokens g (+8), positions kx + 256 s + 64 c
    // + [8t, 8t+8) of the segment
    const uint32_t xb = xsh + g * xstride + 2 * (kx + 256 * s + 8 * t);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      // A fragments: [h][word][lo01, lo23, hi01, hi23]
      uint32_t a[2][2][4];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint2 wv = lds64(rq[h] + 32 * c);
        const uint32_t wd[2] = {wv.x, wv.y};
        const uint32_t hq[2] = {qh[h].x, qh[h].y};
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          if constexpr (F == kQ5K) {
            const int rlo = (2 * c + 28) & 31, rhi = (2 * c + 29) & 31;
            const uint32_t lo5 = bitsel(wd[i], __funnelshift_r(hq[i], hq[i], rlo), 0x0F0F0F0Fu);
            const uint32_t hi5 = bitsel(wd[i] >> 4, __funnelshift_r(hq[i], hq[i], rhi), 0x0F0F0F0Fu);
            bf16_pairs<0x001F001Fu>(lo5, kBf16Magic2, a[h][i][0], a[h][i][1]);
            bf16_pairs<0x001F001Fu>(hi5, kBf16Magic2, a[h][i][2], a[h][i][3]);
          } else {
            bf16_pairs<0x000F000Fu>(wd[i], kBf16Magic2, a[h][i][0], a[h][i][1]);
            bf16_pairs<0x000F000Fu>(wd[i] >> 4, kBf16Magic2, a[h][i][2], a[h][i][3]);
          }
        }
      }
      const float4 elo = lds_f4(tab + (g * G::kTabRow + (s * 4 + c) * 2) * 16);
      const float4 ehi = lds_f4(tab + (g * G::kTabRow + (s * 4 + c) * 2 + 1) * 16);
      const float4 elo8 = lds_f4(tab + ((g + 8) * G::kTabRow + (s * 4 + c) * 2) * 16);
      const float4 ehi8 = lds_f4(tab + ((g + 8) * G::kTabRow + (s * 4 + c) * 2 + 1) * 16);
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        const uint4 blo = lds128(xb + nb * 8 * xstride + 128 * c);
        const uint4 bhi = lds128(xb + nb * 8 * xstride + 128 * c + 64);
        float dlo[4] = {0.f, 0.f, 0.f, 0.f}, dhi[4] = {0.f, 0.f, 0.f, 0.f};
        float slo[4] = {0.f, 0.f, 0.f, 0.f}, shi[4] = {0.f, 0.f, 0.f, 0.f};
        // k-slots (2t, 2t+1) <- positions 8t + (0,1) of a word, (2t+8, 2t+9)
        // <- 8t + (2,3); word 1 is positions 8t + 4 .. 8t + 7
        mma_bf16(dlo, a[0][0][0], a[1][0][0], a[0][0][1], a[1][0][1], blo.x, blo.y);
        mma_bf16(dlo, a[0][1][0], a[1][1][0], a[0][1][1], a[1][1][1], blo.z, blo.w);
        mma_bf16(dhi, a[0][0][2], a[1][0][2], a[0][0][3], a[1][0][3], bhi.x, bhi.y);
        mma_bf16(dhi, a[0][1][2], a[1][1][2], a[0][1][3], a[1][1][3], bhi.z, bhi.w);
        mma_bf16(slo, ones, ones, ones, ones, blo.x, blo.y);
        mma_bf16(slo, ones, ones, ones, ones, blo.z, blo.w);
        mma_bf16(shi, ones, ones, ones, ones, bhi.x, bhi.y);
        mma_bf16(shi, ones, ones, ones, ones, bhi.z, bhi.w);
        mma_epilogue(acc[nb], dlo, slo, elo, elo8);
        mma_epilogue(acc[nb], dhi, shi, ehi, ehi8);
      }
    }
  }
}

// One stage of the verify kernel for this warp's 16 rows (Q6_K).  Unit of
// an mma: sub-block j = 8h + 2tr + u (positions 128h + 32tr + 16u + [0,16));
// thread t takes positions 4t .. 4t+3 of it: ql word A (t-runs 0 / 2), ql
// word B (t-runs 1 / 3) and qh word H.
template <class G, int NB>
__device__ __forceinline__ void mma_stage_q6(const Params& p, const Tile& tl, int sl, int kx,
                                             uint32_t st, int rbase, uint32_t tab, uint32_t xsh,
                                             uint32_t xstride, float2 (&acc)[NB][2]) {
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  uint32_t rec[2];
#pragma unroll
  for (int s = 0; s < G::kSlabSB; ++s) {
    if (sl * G::kSlabSB + s >= p.nsb) break;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = rbase + g + 8 * h;
      const uint32_t ro =
          (static_cast<uint32_t>(tl.row0 + row) * ((210u * p.nsb) & 15u) + sl * G::kQBytes) & 15u;
      rec[h] = st + row * p.slot + ro + 210 * s;
    }
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        // A fragments [row h][t-run][01, 23]
        uint32_t a[2][4][2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t A[1], B[1], H[1];
          const uint32_t rb = rec[h] & ~3u, rsh = (rec[h] & 3u) * 8u;
          lds_words_rec<1>(rb, rsh, 64 * hf + 16 * u + 4 * t, A);
          lds_words_rec<1>(rb, rsh, 64 * hf + 32 + 16 * u + 4 * t, B);
          lds_words_rec<1>(rb, rsh, 128 + 32 * hf + 16 * u + 4 * t, H);
          const uint32_t M4 = 0x0F0F0F0Fu;
          const uint32_t q0 = bitsel(A[0], H[0] << 4, M4);
          const uint32_t q2 = bitsel(A[0] >> 4, H[0], M4);
          const uint32_t q1 = bitsel(B[0], H[0] << 2, M4);
          const uint32_t q3 = bitsel(B[0] >> 4, H[0] >> 2, M4);
          bf16_pairs<0x003F003Fu>(q0, kBf16Q6Zero2, a[h][0][0], a[h][0][1]);
          bf16_pairs<0x003F003Fu>(q1, kBf16Q6Zero2, a[h][1][0], a[h][1][1]);
          bf16_pairs<0x003F003Fu>(q2, kBf16Q6Zero2, a[h][2][0], a[h][2][1]);
          bf16_pairs<0x003F003Fu>(q3, kBf16Q6Zero2, a[h][3][0], a[h][3][1]);
        }
#pragma unroll
        for (int tr = 0; tr < 4; ++tr) {
          const int j = 8 * hf + 2 * tr + u;   // sub-block
          const float4 eg = lds_f4(tab + (g * G::kTabRow + s * 8 + j / 2) * 16);
          const float4 eg8 = lds_f4(tab + ((g + 8) * G::kTabRow + s * 8 + j / 2) * 16);
          const float2 s1 = (j & 1) ? make_float2(eg.z, eg.w) : make_float2(eg.x, eg.y);
          const float2 s18 = (j & 1) ? make_float2(eg8.z, eg8.w) : make_float2(eg8.x, eg8.y);
          const uint32_t xb =
              xsh + g * xstride + 2 * (kx + 256 * s + 128 * hf + 32 * tr + 16 * u + 4 * t);
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) {
            const uint2 b = lds64(xb + nb * 8 * xstride);
            float d[4] = {0.f, 0.f, 0.f, 0.f};
            mma_bf16(d, a[0][tr][0], a[1][tr][0], a[0][tr][1], a[1][tr][1], b.x, b.y);
            acc[nb][0] = __ffma2_rn(s1, make_float2(d[0], d[1]), acc[nb][0]);
            acc[nb][1] = __ffma2_rn(s18, make_float2(d[2], d[3]), acc[nb][1]);
          }
        }
      }
    }
  }
}

template <int F, int NB, int WC>
__global__ void __launch_bounds__((WC + 1) * 32, WC <= 4 ? 2 : 1)
    gemv_mma(const __grid_constant__ Params p, int stages) {
  using G = MGeo<F, WC>;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[2 * kMaxStages];
  __shared__ int last_flag;
  const uint32_t bar_full = smem_addr(&bars[0]);
  const uint32_t bar_empty = smem_addr(&bars[kMaxStages]);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int NTP = 8 * NB;   // staged token rows
  const uint32_t tab0 = smem_addr(smem);                            // WC scale tables
  const uint32_t xsh = tab0 + static_cast<uint32_t>(WC * G::kTabBytes);   // x segment
  const uint32_t xstride = static_cast<uint32_t>(p.kpad * 2 + G::kXPad);
  const uint32_t ring_a = tab0 + p.x_bytes;
  const int kseg = static_cast<int>(blockIdx.x) % p.ksplit;
  const int cta = static_cast<int>(blockIdx.x) / p.ksplit;
  const int cps = static_cast<int>(gridDim.x) / p.ksplit;
  const int my_tiles = (p.tiles - cta + cps - 1) / cps;
  const int total = my_tiles * p.slabs;
  const int sl0 = kseg * p.slabs;
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(bar_full + 8 * s, p.tma ? 1 : 32);
      mbar_init(bar_empty + 8 * s, WC);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const int first = total < stages ? total : stages;
  asm volatile("griddepcontrol.launch_dependents;");
  if (warp == WC) {
    for (int it = 0; it < first; ++it) {
      const Tile tl = tile_of(p, cta + (it / p.slabs) * cps);
      issue_stage<G>(p, smem, ring_a + it * p.stage, bar_full + 8 * it, tl, sl0 + it % p.slabs);
    }
  }
  // x may be produced by the previous kernel: wait for it, then stage the
  // segment (bf16, zeros past K and for tokens >= n_tok), four 16-byte
  // chunks per thread in flight
  asm volatile("griddepcontrol.wait;" ::: "memory");
  {
    const int kbase = kseg * p.kpad;
    const int per_tok = p.kpad / 8;
    const int items = NTP * per_tok;
    for (int q0 = threadIdx.x; q0 < items; q0 += 4 * blockDim.x) {
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int q = q0 + u * blockDim.x;
        const int tok = q / per_tok, j = q % per_tok;
        v[u] = make_uint4(0, 0, 0, 0);
        if (q < items && tok < p.nt && kbase + 8 * j < p.K)
          v[u] = ldg_nc_v4(p.x + static_cast<int64_t>(tok) * p.K + kbase + 8 * j);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int q = q0 + u * blockDim.x;
        if (q < items) sts128u(xsh + (q / per_tok) * xstride + 16 * (q % per_tok), v[u]);
      }
    }
  }
  __syncthreads();
  if (warp == WC) {
    // ring position, empty-barrier parity and (tile, slab) of stage `first`,
    // advanced by counting (no division per stage)
    int slot = 0, xsl = first % p.slabs, tn = first / p.slabs;
    uint32_t parity = 0;
    for (int it = first; it < total; ++it) {
      if (!mbar_wait_warp(bar_empty + 8 * slot, parity)) return;
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      const Tile tl = tile_of(p, cta + tn * cps);
      issue_stage<G>(p, smem, ring_a + slot * p.stage, bar_full + 8 * slot, tl, sl0 + xsl);
      if (++xsl == p.slabs) {
        xsl = 0;
        ++tn;
      }
      if (++slot == stages) {
        slot = 0;
        parity ^= 1u;
      }
    }
    return;
  }
  const uint32_t tab = tab0 + static_cast<uint32_t>(warp * G::kTabBytes);
  const int rbase = 16 * warp;
  const int g = lane >> 2, t = lane & 3;
  float2 acc[NB][2];
  Tile tl{};
  int tix = 0;
  int xsl = 0, tn = 0, slot = 0;   // advanced by counting (no division per stage)
  uint32_t parity = 0;
  for (int it = 0; it < total; ++it) {
    const int sl = sl0 + xsl;
    if (xsl == 0) {
      tix = cta + tn * cps;
      tl = tile_of(p, tix);
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) acc[nb][0] = acc[nb][1] = make_float2(0.0f, 0.0f);
    }
    if (!mbar_wait_warp(bar_full + 8 * slot, parity)) return;
    const uint32_t st = ring_a + slot * p.stage;
    if (rbase < tl.rcnt) {   // warp-uniform
      build_scale_table<G>(p, tl, sl, st, rbase, tab);
      __syncwarp();
      if constexpr (F == kQ6K)
        mma_stage_q6<G, NB>(p, tl, sl, xsl * G::kSlabK, st, rbase, tab, xsh, xstride, acc);
      else
        mma_stage_q4<G, NB>(p, tl, sl, xsl * G::kSlabK, st, rbase, tab, xsh, xstride, acc);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * slot);
    if (xsl == p.slabs - 1) {
      float* y = pick(p.g.y, tl.mi);
      const int64_t N = pick(p.g.N, tl.mi);
      if (p.ksplit == 1) {
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int row = rbase + g + 8 * h;
            const float v[2] = {acc[nb][h].x, acc[nb][h].y};
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int tok = 8 * nb + 2 * t + e;
              if (row < tl.rcnt && tok < p.nt) y[static_cast<int64_t>(tok) * N + tl.row0 + row] = v[e];
            }
          }
      } else {
        float* part = static_cast<float*>(p.part) + static_cast<int64_t>(tix) * p.tile_rows * NTP;
        const int64_t seg_stride = static_cast<int64_t>(p.tiles) * p.tile_rows * NTP;
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int row = rbase + g + 8 * h;
            if (row < tl.rcnt) {
              float* q = part + kseg * seg_stride + row * NTP + 8 * nb + 2 * t;
              __stcg(q, acc[nb][h].x);
              __stcg(q + 1, acc[nb][h].y);
            }
          }
        // the consumer barrier orders every warp's stores before thread 0's
        // fence, which makes them visible device-wide before its arrival
        asm volatile("bar.sync 1, %0;" ::"r"(WC * 32) : "memory");
        if (threadIdx.x == 0) {
          __threadfence();
          last_flag = atomicAdd(p.arrivals + tix, 1u) == static_cast<unsigned>(p.ksplit - 1);
        }
        asm volatile("bar.sync 1, %0;" ::"r"(WC * 32) : "memory");
        if (last_flag) {
          __threadfence();
#pragma unroll
          for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int row = rbase + g + 8 * h;
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int tok = 8 * nb + 2 * t + e;
                if (row < tl.rcnt && tok < p.nt)
                  y[static_cast<int64_t>(tok) * N + tl.row0 + row] =
                      sum_segments(part + row * NTP + tok, seg_stride, p.ksplit);
              }
            }
          if (threadIdx.x == 0) p.arrivals[tix] = 0u;
        }
      }
    }
    if (++xsl == p.slabs) {
      xsl = 0;
      ++tn;
    }
    if (++slot == stages) {
      slot = 0;
      parity ^= 1u;
    }
  }
}

// ===================================================== single-token tensor-core kernel
//
// n_tok = 1 on large Q4_K / Q4_G128 matrices.  The products run on the
// tensor cores as mma.sync m16n8k16 (fp16 operands, fp32 accumulation), and
// the eight columns of the n8 operand carry eight SUB-BLOCKS of the one token
// instead of eight tokens.  The k slots of an mma are assigned per lane:
// slots (2t, 2t+1) of lane t (t = lane & 3) hold weights of sub-block lo(t),
// slots (2t+8, 2t+9) weights of sub-block hi(t), and B holds x at those
// slots in column lo(t) / hi(t) and zero in the other columns.  After the 16
// mmas of a super-block, D[row][n] is the dot product of sub-block n alone,
// the quantity one scale multiplies:
//   y_row += s1[n] D[row][n] + s2[n] Sx[n]
// A is exact (tc_sb_product: q 2^-24 or 16 q 2^-24, fp16 subnormals),
// so no offset term remains in D (a record of zero weights gives D = 0
// whatever its scales); x is staged in fp16 with a power-of-two scale per
// sub-block (stage_x_tc_raw) that the column scale undoes; s1 = d sc, s2 =
// -dmin m, Sx[n] the sum of x over sub-block n.  Lane t takes chunk t of the
// super-block (sub-block 2t: low nibbles, sub-block 2t+1: high nibbles);
// word m of the chunk gives mma 2m (bytes 0, 2) and 2m+1 (bytes 1, 3).  (Q5_K
// and Q6_K would need their fields assembled first, which costs more integer
// work than their CUDA-core path; they stay on gemv_stream.)
//
// gemv_tc1 (TGeo1): one CTA per SM, 4 SB consumer warps and a producer warp
// (SB = 5 where K / 256 divides by 5, else 4).  A tile is 64 rows over ALL
// of K, so no partial sum ever leaves the CTA: a stage is the tile's 64 rows
// x SB super-blocks (one tensor copy per plane), warp w takes rows 16 (w % 4)
// .. + 15 of the stage's super-block w / 4, and at the tile's end the SB
// warps of a row group add their row sums in shared memory, super-block
// column 0 to SB - 1 (a fixed order).  Tiles are
// claimed at run time (as in gemv_stream); x is staged once per CTA.
// (Splitting K across CTAs instead needs a device-scope exchange of partial
// sums whose latency ends up on the launch's critical path.)
//
// TGeo: the stage geometry of the multi-token kernel gemv_tcv (one-super-block
// stages of 16 kWC RTW rows, a producer and a split-K reducer warp).

template <int F, int SB>
struct TGeo1 {
  static constexpr int kF = F;
  static constexpr int kRowGroups = 4;              // 16-row mma tiles per tile
  static constexpr int kSlabSB = SB;                // super-blocks per stage
  static constexpr int kWC = kRowGroups * SB;       // consumer warps
  static constexpr int kThreads = (kWC + 1) * 32;   // + producer
  static constexpr int kRows = 16 * kRowGroups;
  static constexpr int kSlabK = 256 * kSlabSB;
  static constexpr int kBB = block_bytes(F);
  static constexpr int kSub = 32;   // weights per sub-block
  static_assert(F == kQ4K || F == kG128, "Q4_K and Q4_G128 only");
  static constexpr int kQBytes = (F == kG128) ? 128 * kSlabSB : kBB * kSlabSB;
  static constexpr int kPBytes = (F == kG128) ? 8 * kSlabSB : 0;
  static constexpr int round16(int b) { return (b + 15) / 16 * 16; }
  // row pitch an odd multiple of 16 bytes: the 8 rows a warp reads at once
  // start in 8 different 16-byte bank groups (the box reads 16 bytes of the
  // next stage's records, or zeros past the row)
  static constexpr int odd16(int b) { return (b / 16) % 2 ? b : b + 16; }
  static constexpr int kSlotTma = odd16(round16(kQBytes + (kQBytes % 16 ? 15 : 0)));
  static constexpr int kPSlotTma = (F == kG128) ? round16(kPBytes + (kPBytes % 16 ? 15 : 0)) : 0;
  static constexpr int kSlotBulk = odd16(round16(kQBytes + 16));
  static constexpr int kPSlotBulk = (F == kG128) ? round16(kPBytes + 16) : 0;
  // the row-sum exchange at a tile's end: two buffers of [column][row] floats
  static constexpr uint32_t kCombBytes = 2u * kSlabSB * kRows * 4u;
};

template <int F, int WC_, int RTW = 1>
struct TGeo {
  static constexpr int kF = F;
  static constexpr int kWC = WC_;
  static constexpr int kThreads = (WC_ + 2) * 32;   // + producer + reducer
  static constexpr int kRows = 16 * WC_ * RTW;        // a warp owns RTW 16-row tiles
  static_assert(kRows <= 256, "a tile is one tensor-copy box (at most 256 rows)");
  static constexpr int kSlabSB = 1;
  static constexpr int kSlabK = 256;
  static constexpr int kBB = block_bytes(F);
  static constexpr int kSub = 32;   // weights per sub-block
  static_assert(F == kQ4K || F == kG128, "Q4_K and Q4_G128 only");
  static constexpr int kQBytes = (F == kG128) ? 128 * kSlabSB : kBB * kSlabSB;
  static constexpr int kPBytes = (F == kG128) ? 8 * kSlabSB : 0;
  static constexpr int round16(int b) { return (b + 15) / 16 * 16; }
  // row pitch an odd multiple of 16 bytes: the 8 rows a warp reads at once
  // start in 8 different 16-byte bank groups
  static constexpr int odd16(int b) { return (b / 16) % 2 ? b : b + 16; }
  static constexpr int kSlotTma = odd16(round16(kQBytes + (kQBytes % 16 ? 15 : 0)));
  static constexpr int kPSlotTma = (F == kG128) ? round16(kPBytes + (kPBytes % 16 ? 15 : 0)) : 0;
  static constexpr int kSlotBulk = odd16(round16(kQBytes + 16));
  static constexpr int kPSlotBulk = (F == kG128) ? round16(kPBytes + 16) : 0;
};

// Shared layout before the ring: the staged x of the K segment (kpad values
// as fp16, each group of four positions (a, b, c, d) stored as (a, c, b, d),
// so that 32-bit entry i of a sub-block holds positions 4 (i >> 1) + (i & 1)
// and that + 2), then Sx (the fp32 sum of x over every sub-block), then the
// column scale of every sub-block (see stage_x_tc_raw), then 64 zero bytes,
// then the kernel's row-sum buffers.
//
// The zero block starts 32 bytes past a 128-byte boundary.  In a quarter-warp
// of the product one lane reads its sub-block's x (at 0 or 64 modulo 128
// bytes, plus the same 0..48 as the zero block's readers) and the other seven
// read the zero block, so the two addresses always fall in different banks.
__host__ __device__ constexpr uint32_t tc_zero_off(int kpad, int sub) {
  return ((2u * static_cast<uint32_t>(kpad) + 8u * static_cast<uint32_t>(kpad / sub) + 127u) &
          ~127u) + 32u;
}
__host__ __device__ constexpr uint32_t tc_x_only(int kpad, int sub) {
  return (tc_zero_off(kpad, sub) + 64u + 15u) & ~15u;
}

// x of a K segment for the tensor-core product (fp16 operands), with the
// sum of x over every sub-block (fp32, for the min term).  The products need
// x exactly; bf16 x is exact in fp16 within fp16's exponent range, so every
// sub-block is scaled by a power of two 2^-f chosen from its own largest |x|
// (which lands in [2^14, 2^15)): then every value of the sub-block within a
// factor 2^31 of its largest converts exactly (fp16 subnormals reach 2^-24),
// and smaller ones round (contributing less than 2^-38 of the largest |x|
// each).  The sub-block's column scale, stored beside Sx, undoes 2^-f and
// the product's own power of two: 2^(f+24) for an even sub-block (low
// nibbles, A = q 2^-24) and 2^(f+20) for an odd one (high nibbles, A =
// 16 q 2^-24).  bf16 subnormal x (below 2^-126) is not kept.
template <int S>
__device__ void stage_x_tc_raw(const uint16_t* x, int K, int kpad, uint32_t xsh, int kbase) {
  static_assert(S == 32, "one sub-block is four lanes of eight positions");
  const int nch = kpad / 8;   // 16-byte chunks (a multiple of 32)
  const uint32_t xsum = xsh + 2u * static_cast<uint32_t>(kpad);
  const uint32_t xscl = xsum + 4u * static_cast<uint32_t>(kpad / S);
  const int lane = threadIdx.x & 31;
  for (int base = static_cast<int>(threadIdx.x) & ~31; base < nch;
       base += static_cast<int>(blockDim.x)) {
    const int c = base + lane;
    const int k = kbase + 8 * c;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (k < K) v = ldg_nc_v4(x + k);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float f[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      f[2 * j] = __uint_as_float(w[j] << 16);
      f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
    float sum = 0.0f, amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      sum += f[2 * j] + f[2 * j + 1];
      amax = fmaxf(amax, fmaxf(fabsf(f[2 * j]), fabsf(f[2 * j + 1])));
    }
#pragma unroll
    for (int m = 1; m < S / 8; m <<= 1) {
      sum += __shfl_xor_sync(0xFFFFFFFFu, sum, m);
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, m));
    }
    int fs = amax > 0.0f ? static_cast<int>((__float_as_uint(amax) >> 23) & 0xFF) - 127 - 14 : 0;
    fs = fs < -100 ? -100 : (fs > 100 ? 100 : fs);
    const float down = __uint_as_float(static_cast<uint32_t>(127 - fs) << 23);   // 2^-fs, exact
    uint32_t e[4];
#pragma unroll
    for (int j = 0; j < 2; ++j) {   // entries (p0, p2), (p1, p3) of each group of four
      const __half2 a = __floats2half2_rn(f[4 * j] * down, f[4 * j + 2] * down);
      const __half2 b = __floats2half2_rn(f[4 * j + 1] * down, f[4 * j + 3] * down);
      e[2 * j] = *reinterpret_cast<const uint32_t*>(&a);
      e[2 * j + 1] = *reinterpret_cast<const uint32_t*>(&b);
    }
    sts128u(xsh + 16u * c, make_uint4(e[0], e[1], e[2], e[3]));
    if ((c & (S / 8 - 1)) == 0) {
      const int sb = c / (S / 8);
      const float scale = __uint_as_float(static_cast<uint32_t>(127 + 24 + fs - 4 * (sb & 1)) << 23);
      asm volatile("st.shared.f32 [%0], %1;" ::"r"(xsum + 4u * sb), "f"(sum) : "memory");
      asm volatile("st.shared.f32 [%0], %1;" ::"r"(xscl + 4u * sb), "f"(scale) : "memory");
    }
  }
  if (threadIdx.x < 4) sts128u(xsh + tc_zero_off(kpad, S) + 16u * threadIdx.x, make_uint4(0, 0, 0, 0));
}

template <int S>
__device__ void stage_x_tc(const Params& p, uint32_t xsh, int kbase) {
  stage_x_tc_raw<S>(p.x, p.K, p.kpad, xsh, kbase);
}

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The single-token tensor-core product of one super-block for rows g and
// g + 8 of a 16-row tile: lane t's qs chunk of each row starts at qa0 / qa1
// (32 bytes), its B operands (the staged fp16 x of its column, or the zero
// block) at xlo / xhi.  A is exact in fp16 and needs one AND per two weights:
// the low nibbles of bytes (0, 2) (mask 0x000F000F) read as fp16 are the
// subnormals q 2^-24, the high nibbles in place (mask 0x00F000F0) are
// 16 q 2^-24; bytes (1, 3) go through the same after one shift by 8.  The
// tensor cores take fp16 subnormal operands as they are, and every product
// and partial sum stays far inside fp32's normal range, so D is exactly
// 2^-24 times the sum built from q itself; the column scales of the staged x
// absorb 2^24 and the factor 16 of the high nibbles.  d[0] / d[1]: the two
// mma chains (bytes 0, 2 / bytes 1, 3); their sum per column is the dot
// product of that column's sub-block.
__device__ __forceinline__ void tc_sb_product(uint32_t qa0, uint32_t qa1, uint32_t xlo,
                                              uint32_t xhi, float (&d)[2][4]) {
  auto lo = [](uint32_t w) { return w & 0x000F000Fu; };
  auto hi = [](uint32_t w) { return w & 0x00F000F0u; };
#pragma unroll
  for (int hv = 0; hv < 2; ++hv) {   // words 4 hv .. 4 hv + 3 of the chunk
    const uint4 w0 = lds128(qa0 + 16 * hv), w8 = lds128(qa1 + 16 * hv);
    const uint4 bl0 = lds128(xlo + 32 * hv), bl1 = lds128(xlo + 32 * hv + 16);
    const uint4 bh0 = lds128(xhi + 32 * hv), bh1 = lds128(xhi + 32 * hv + 16);
    const uint32_t W[2][4] = {{w0.x, w0.y, w0.z, w0.w}, {w8.x, w8.y, w8.z, w8.w}};
    const uint32_t BL[8] = {bl0.x, bl0.y, bl0.z, bl0.w, bl1.x, bl1.y, bl1.z, bl1.w};
    const uint32_t BH[8] = {bh0.x, bh0.y, bh0.z, bh0.w, bh1.x, bh1.y, bh1.z, bh1.w};
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const uint32_t a = W[0][m], b = W[1][m];
      const uint32_t a8 = a >> 8, b8 = b >> 8;
      mma_f16(d[0], lo(a), lo(b), hi(a), hi(b), BL[2 * m], BH[2 * m]);
      mma_f16(d[1], lo(a8), lo(b8), hi(a8), hi(b8), BL[2 * m + 1], BH[2 * m + 1]);
    }
  }
}

// rotate left by r (0..31)
__device__ __forceinline__ uint32_t rotl32(uint32_t v, uint32_t r) {
  return __funnelshift_l(v, v, r);
}

// Q5_K: the fifth bit of a weight sits in qh, byte l (position l of a
// 32-position run) bit j for sub-block j, so the qh word with the same index
// as a qs word holds the fifth bits of that word's four positions.  For the
// low nibbles of sub-block j the bit goes beside the nibble, to bit 4 of each
// 16-bit half (16 2^-24 as an fp16 subnormal), for the high nibbles of
// sub-block j + 1 (kept in place, 16 q 2^-24) to bit 8 (256 2^-24): q stays
// exact (at most 31 or 496 times 2^-24).  r = the rotation that brings bit j
// of byte 0 to bit 4 (bytes 0, 2 of a word); the others follow from it.
struct Q5Rot {
  uint32_t lo02, lo13, hi02, hi13;
};
__device__ __forceinline__ Q5Rot q5_rot(int j) {   // j = the low-nibble sub-block (even)
  Q5Rot r;
  r.lo02 = static_cast<uint32_t>(4 - j) & 31u;    // bits j, 16 + j     -> 4, 20
  r.lo13 = static_cast<uint32_t>(28 - j) & 31u;   // bits 8 + j, 24 + j -> 4, 20
  r.hi02 = static_cast<uint32_t>(7 - j) & 31u;    // bits j + 1, 17 + j -> 8, 24
  r.hi13 = static_cast<uint32_t>(31 - j) & 31u;   // bits 9 + j, 25 + j -> 8, 24
  return r;
}
__device__ __forceinline__ uint32_t or_bits(uint32_t a, uint32_t q, uint32_t m) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xF8;" : "=r"(d) : "r"(a), "r"(q), "r"(m));
  return d;   // a | (q & m)
}

// tc_sb_product for Q5_K: qh0 / qh1, the rows' 32 qh bytes; rot from q5_rot(2t).
__device__ __forceinline__ void tc_sb_product_q5(uint32_t qa0, uint32_t qa1, uint32_t qh0,
                                                 uint32_t qh1, uint32_t xlo, uint32_t xhi,
                                                 const Q5Rot& rot, float (&d)[2][4]) {
  const uint32_t M4 = 0x00100010u, M8 = 0x01000100u;
#pragma unroll
  for (int hv = 0; hv < 2; ++hv) {
    const uint4 w0 = lds128(qa0 + 16 * hv), w8 = lds128(qa1 + 16 * hv);
    const uint4 h0 = lds128(qh0 + 16 * hv), h8 = lds128(qh1 + 16 * hv);
    const uint4 bl0 = lds128(xlo + 32 * hv), bl1 = lds128(xlo + 32 * hv + 16);
    const uint4 bh0 = lds128(xhi + 32 * hv), bh1 = lds128(xhi + 32 * hv + 16);
    const uint32_t W[2][4] = {{w0.x, w0.y, w0.z, w0.w}, {w8.x, w8.y, w8.z, w8.w}};
    const uint32_t H[2][4] = {{h0.x, h0.y, h0.z, h0.w}, {h8.x, h8.y, h8.z, h8.w}};
    const uint32_t BL[8] = {bl0.x, bl0.y, bl0.z, bl0.w, bl1.x, bl1.y, bl1.z, bl1.w};
    const uint32_t BH[8] = {bh0.x, bh0.y, bh0.z, bh0.w, bh1.x, bh1.y, bh1.z, bh1.w};
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      uint32_t l02[2], l13[2], h02[2], h13[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const uint32_t w = W[r][m], w8v = w >> 8, q = H[r][m];
        l02[r] = or_bits(w & 0x000F000Fu, rotl32(q, rot.lo02), M4);
        l13[r] = or_bits(w8v & 0x000F000Fu, rotl32(q, rot.lo13), M4);
        h02[r] = or_bits(w & 0x00F000F0u, rotl32(q, rot.hi02), M8);
        h13[r] = or_bits(w8v & 0x00F000F0u, rotl32(q, rot.hi13), M8);
      }
      mma_f16(d[0], l02[0], l02[1], h02[0], h02[1], BL[2 * m], BH[2 * m]);
      mma_f16(d[1], l13[0], l13[1], h13[0], h13[1], BL[2 * m + 1], BH[2 * m + 1]);
    }
  }
}

// y += s1 (cs D) + s2 Sx for rows g (h = 0) and g+8 (h = 1), columns (2t,
// 2t+1); cs, the columns' power-of-two scales, brings D to the units of x
// before s1 multiplies it (no intermediate leaves fp32's range)
__device__ __forceinline__ void tc_epilogue(float2 (&acc)[2], const float (&d)[2][4], float2 cs,
                                            float2 s1g, float2 s2g, float2 s1h, float2 s2h,
                                            float2 sx) {
  const float2 dg = __fmul2_rn(cs, make_float2(d[0][0] + d[1][0], d[0][1] + d[1][1]));
  const float2 dh = __fmul2_rn(cs, make_float2(d[0][2] + d[1][2], d[0][3] + d[1][3]));
  acc[0] = __ffma2_rn(s1g, dg, acc[0]);
  acc[0] = __ffma2_rn(s2g, sx, acc[0]);
  acc[1] = __ffma2_rn(s1h, dh, acc[1]);
  acc[1] = __ffma2_rn(s2h, sx, acc[1]);
}

// (s1, s2) of sub-blocks (2t, 2t+1) of one row: Q4_K from the record's
// header, Q4_G128 from its param plane.
template <class G>
__device__ __forceinline__ void tc_scales_q4(const Params& p, const Tile& tl, int sl, uint32_t st,
                                             int row, int s, const ScaleSel& ss, int t,
                                             float2& s1, float2& s2) {
  constexpr int F = G::kF;
  if constexpr (F == kG128) {
    const uint32_t po =
        (static_cast<uint32_t>(tl.row0 + row) * ((8u * p.nsb) & 15u) + sl * G::kPBytes) & 15u;
    const uint2 pr = lds64(st + p.pbase + row * p.pslot + po + 8 * s);
    const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&pr.x));
    const int grp = t >> 1;
    const float a = dd.x * byte_f(pr.y, grp);
    const float b = -(dd.y * byte_f(pr.y, 2 + grp));
    s1 = make_float2(a, a);
    s2 = make_float2(b, b);
  } else {
    const uint4 hdr = lds128(st + row * p.slot + G::kBB * s);
    const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&hdr.x));
    uint32_t scp, mnp;
    scale_pair6(ss, hdr.y, hdr.z, hdr.w, scp, mnp);
    s1 = __fmul2_rn(make_float2(dd.x, dd.x), bytes01_f2(scp));
    s2 = __fmul2_rn(make_float2(-dd.y, -dd.y), bytes01_f2(mnp));
  }
}

// bf16(silu(g) * u), silu(v) = v / (1 + e^-v), evaluated in fp32 and
// rounded to nearest (ties to even).
__device__ __forceinline__ uint16_t swiglu_bf16(float gv, float uv) {
  const __nv_bfloat16 hb = __float2bfloat16_rn(gv / (1.0f + expf(-gv)) * uv);
  return *reinterpret_cast<const uint16_t*>(&hb);
}

// SwiGLU mode: feature n's gate and up sums -> y_gate, y_up (fp32) and h.
__device__ __forceinline__ void swiglu_store(const Params& p, int64_t n, float gv, float uv) {
  p.g.y[0][n] = gv;
  p.g.y[1][n] = uv;
  p.h[n] = swiglu_bf16(gv, uv);
}

// h[i] = bf16(silu(g[i]) * u[i]) for i < n (the SwiGLU activation after a
// gate/up launch that did not fuse it).
__global__ void __launch_bounds__(256) swiglu_elementwise(const float* __restrict__ gv,
                                                          const float* __restrict__ uv,
                                                          uint16_t* __restrict__ h, int64_t n) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (i < n) h[i] = swiglu_bf16(gv[i], uv[i]);
}

// The reducer warp: for every unit the consumers finish (in order), publish
// its sums (tile_rows x NTP values, row-major) to the split-K scratch, count
// the arrival, and for the tile's last segment add segments 0..ksplit-1 in
// order and write y (token k of row r to y[k][row0 + r], k < n_tok).
template <int NTP>
__device__ __forceinline__ void tc_reduce(const Params& p, uint32_t psum, uint32_t part_full,
                                          uint32_t part_empty, const int* part_tile, int kseg) {
  const int lane = threadIdx.x & 31;
  const int64_t seg_stride = static_cast<int64_t>(p.tiles) * p.tile_rows * NTP;
  for (int u = 0;; ++u) {
    const int b = u & 1;
    if (!mbar_wait_warp(part_full + 8 * b, static_cast<uint32_t>(u >> 1) & 1u)) return;
    const int tix = part_tile[b];
    if (tix < 0) return;
    const Tile tl = tile_of(p, tix);
    // SwiGLU mode: all stage rows (gate rows, then up rows)
    const int n = p.swiglu ? p.tile_rows * NTP : tl.rcnt * NTP;
    float* part = static_cast<float*>(p.part) + static_cast<int64_t>(tix) * p.tile_rows * NTP;
    const uint32_t buf = psum + 4u * static_cast<uint32_t>(b * p.tile_rows * NTP);
    for (int e = lane; e < n; e += 32) {
      float v;
      asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(buf + 4u * e));
      __stcg(part + kseg * seg_stride + e, v);
    }
    // every lane's stores are visible device-wide before the arrival
    __threadfence();
    __syncwarp();
    unsigned last = 0;
    if (lane == 0)
      last = atomicAdd(p.arrivals + tix, 1u) == static_cast<unsigned>(p.ksplit - 1) ? 1u : 0u;
    last = __shfl_sync(0xFFFFFFFFu, last, 0);
    if (lane == 0) mbar_arrive(part_empty + 8 * b);   // the buffer may be refilled
    if (last) {
      __threadfence();
      // values e0 + lane + 32 i: the loads of one segment are independent, so
      // the segments stream back to back (each value still adds them in order)
      float* y = pick(p.g.y, tl.mi);
      const int64_t N = pick(p.g.N, tl.mi);
      constexpr int kR = 8;
      for (int e0 = 0; e0 < n; e0 += 32 * kR) {
        float a[kR];
#pragma unroll
        for (int i = 0; i < kR; ++i) a[i] = 0.0f;
        for (int j = 0; j < p.ksplit; ++j) {
          const float* pj = part + j * seg_stride + e0 + lane;
#pragma unroll
          for (int i = 0; i < kR; ++i)
            if (e0 + lane + 32 * i < n) a[i] += __ldcg(pj + 32 * i);
        }
        if (NTP == 1 && p.swiglu) {
          // one 256-value pass (kR = 8, tile_rows = 256): a[i], i < 4, is the
          // gate sum of feature lane + 32 i and a[i + 4] its up sum
#pragma unroll
          for (int i = 0; i < kR / 2; ++i) {
            const int r = lane + 32 * i;
            if (r < tl.rcnt) swiglu_store(p, tl.row0 + r, a[i], a[i + kR / 2]);
          }
          continue;
        }
#pragma unroll
        for (int i = 0; i < kR; ++i) {
          const int e = e0 + lane + 32 * i;
          const int row = e / NTP, k = e % NTP;
          if (e < n && k < p.nt) y[static_cast<int64_t>(k) * N + tl.row0 + row] = a[i];
        }
      }
      if (lane == 0) p.arrivals[tix] = 0u;
    }
  }
}

template <int F, int SB>
__global__ void __launch_bounds__(TGeo1<F, SB>::kThreads, 1)
    gemv_tc1(const __grid_constant__ Params p, int stages) {
  using G = TGeo1<F, SB>;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[2 * kMaxStages + 4 * G::kRowGroups];
  __shared__ int stage_tile[kMaxStages];
  const uint32_t bar_full = smem_addr(&bars[0]);
  const uint32_t bar_empty = smem_addr(&bars[kMaxStages]);
  // per row group and buffer: the group's 4 warps wrote their row sums /
  // the row sums were taken
  const uint32_t comb_full = smem_addr(&bars[2 * kMaxStages]);
  const uint32_t comb_empty = smem_addr(&bars[2 * kMaxStages + 2 * G::kRowGroups]);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t xsh = smem_addr(smem);
  const uint32_t comb = xsh + tc_x_only(p.kpad, G::kSub);   // [2][kSlabSB][kRows] floats
  const uint32_t ring_a = xsh + p.x_bytes;
  const int cta = static_cast<int>(blockIdx.x);
  const int cps = static_cast<int>(gridDim.x);
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(bar_full + 8 * s, p.tma ? 1 : 32);
      mbar_init(bar_empty + 8 * s, G::kWC);
    }
    for (int i = 0; i < 2 * G::kRowGroups; ++i) {
      mbar_init(comb_full + 8 * i, G::kSlabSB);
      mbar_init(comb_empty + 8 * i, 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const bool producer = warp == G::kWC;
  asm volatile("griddepcontrol.launch_dependents;");
  Ring ring;
  if (producer) produce_prefill<G>(p, smem, ring_a, bar_full, stage_tile, stages, cta, cps, 0, ring);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  stage_x_tc<G::kSub>(p, xsh, 0);
  __syncthreads();
  if (producer) {
    produce_rest<G>(p, smem, ring_a, bar_full, bar_empty, stage_tile, stages, cta, cps, 0, 0, ring);
    return;
  }
  const int g = lane >> 2, t = lane & 3;
  const int rg = warp % G::kRowGroups;   // rows ra + g and rb + g of every stage
  const int sc = warp / G::kRowGroups;   // super-block sc of every stage
  const int ra = 16 * rg, rb = 16 * rg + 8;
  const ScaleSel ss = scale_sel(t);
  const uint32_t xsum = xsh + 2u * static_cast<uint32_t>(p.kpad);
  const uint32_t xscl = xsum + 4u * static_cast<uint32_t>(p.kpad / 32);
  const uint32_t zero = xsh + tc_zero_off(p.kpad, 32);
  const bool act_lo = g == 2 * t, act_hi = g == 2 * t + 1;   // column g of the B operand
  float2 acc[2];
  Tile tl{};
  int xsl = 0, slot = 0, ntile = 0;
  uint32_t parity = 0;
  for (;;) {
    if (!mbar_wait_warp(bar_full + 8 * slot, parity)) return;
    if (xsl == 0) {
      const int tix = stage_tile[slot];
      if (tix < 0) return;
      tl = tile_of(p, tix);
      acc[0] = acc[1] = make_float2(0.0f, 0.0f);
    }
    const uint32_t st = ring_a + slot * p.stage;
    const int sbx = xsl * G::kSlabSB + sc;   // super-block of the row
    if (sbx < p.nsb) {
      const uint32_t xlo = act_lo ? xsh + 64u * (8 * sbx + 2 * t) : zero;
      const uint32_t xhi = act_hi ? xsh + 64u * (8 * sbx + 2 * t + 1) : zero;
      uint32_t qa[2];   // rows ra + g, rb + g: the chunk's qs bytes
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t rs = st + ((h ? rb : ra) + g) * p.slot;
        qa[h] = (F == kG128) ? rs + 128 * sc + 32 * t : rs + G::kBB * sc + 16 + 32 * t;
      }
      float d[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      tc_sb_product(qa[0], qa[1], xlo, xhi, d);
      float2 s1g, s2g, s1h, s2h;
      tc_scales_q4<G>(p, tl, xsl, st, ra + g, sc, ss, t, s1g, s2g);
      tc_scales_q4<G>(p, tl, xsl, st, rb + g, sc, ss, t, s1h, s2h);
      const float2 sx = lds_f2(xsum + 4u * (8 * sbx + 2 * t));
      const float2 cs = lds_f2(xscl + 4u * (8 * sbx + 2 * t));   // column scales
      tc_epilogue(acc, d, cs, s1g, s2g, s1h, s2h, sx);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * slot);
    if (xsl == p.slabs - 1) {
      // the tile's end: every warp leaves rows g, g+8 of its column in buffer
      // b; one warp of the row group (rotating) adds the columns in order
      // 0..3 and writes y.  In SwiGLU mode the up groups (2, 3) also take the
      // gate sums of the same features from groups 0, 1 and write h.
      const int b = ntile & 1;
      const uint32_t k = static_cast<uint32_t>(ntile >> 1);
      const uint32_t my_full = comb_full + 8u * (2 * rg + b);
      const uint32_t my_empty = comb_empty + 8u * (2 * rg + b);
      if (ntile >= 2 && !mbar_wait_warp(my_empty, (k - 1) & 1u)) return;
      const uint32_t cb = comb + 4u * static_cast<uint32_t>(b * G::kSlabSB * G::kRows);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float a = acc[h].x + acc[h].y;
        a += __shfl_xor_sync(0xFFFFFFFFu, a, 1);
        a += __shfl_xor_sync(0xFFFFFFFFu, a, 2);
        if (t == 0)
          asm volatile("st.shared.f32 [%0], %1;" ::"r"(cb + 4u * (sc * G::kRows + (h ? rb : ra) + g)),
                       "f"(a)
                       : "memory");
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(my_full);
      auto col_sum = [&](int row) {
        float v = 0.0f;
#pragma unroll
        for (int c = 0; c < G::kSlabSB; ++c) {
          float u;
          asm volatile("ld.shared.f32 %0, [%1];" : "=f"(u) : "r"(cb + 4u * (c * G::kRows + row)));
          v += u;
        }
        return v;
      };
      const bool gate_group = p.swiglu && rg < G::kRowGroups / 2;
      if (sc == (ntile % G::kSlabSB) && !gate_group) {
        if (!mbar_wait_warp(my_full, k & 1u)) return;
        if (p.swiglu) {
          // features f of this up group's rows: up row 32 + f, gate row f
          const int gq = rg - G::kRowGroups / 2;
          const uint32_t gate_full = comb_full + 8u * (2 * gq + b);
          if (!mbar_wait_warp(gate_full, k & 1u)) return;
          if (lane < 16) {
            const int f = 16 * gq + lane;
            if (f < tl.rcnt) swiglu_store(p, tl.row0 + f, col_sum(f), col_sum(G::kRows / 2 + f));
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(comb_empty + 8u * (2 * gq + b));
        } else {
          if (lane < 16) {
            const int row = ra + lane;
            if (row < tl.rcnt) pick(p.g.y, tl.mi)[tl.row0 + row] = col_sum(row);
          }
          __syncwarp();
        }
        if (lane == 0) mbar_arrive(my_empty);
      }
      ++ntile;
    }
    if (++xsl == p.slabs) xsl = 0;
    if (++slot == stages) {
      slot = 0;
      parity ^= 1u;
    }
  }
}

// ============================================= multi-token tensor-core kernel
//
// n_tok 2..16 on large Q4_K / Q4_G128 matrices (the speculative-verify
// widths): one-super-block stages of 16 WC RTW rows, tile claiming, K split
// into segments with a reducer warp (tc_reduce); two 4-warp CTAs per SM up
// to eight tokens, one 8-warp CTA beyond.  Columns of the n8 operand are
// tokens (NB blocks of eight); a warp owns two 16-row mma tiles, so every B
// fragment loaded from shared memory feeds two A fragments.  One mma covers
// 16 positions of one sub-block: lane t takes bytes 8t .. 8t+7 of a chunk,
// and word m of them gives slots (2t, 2t+1) <- bytes (0, 2) and (2t+8, 2t+9)
// <- bytes (1, 3): the low nibbles for the chunk's first sub-block, the high
// nibbles (in place) for its second; A is exact as fp16 subnormals, as in
// gemv_tc1.  Two mmas per sub-block, token block and row tile, then
//   y[tok] += s1 cs[tok] D + s2 Sx[tok],  s1 = d sc, s2 = -dmin m
// per (row, sub-block), with s1, s2 from a per-warp table built once per
// super-block (each lane decodes the four chunks of one row), and Sx and the
// column scale cs staged with x.  The staged x (stage_x_tcv_raw): token rows
// of kpad fp16 values scaled per (token, sub-block), each group of four
// positions (a, b, c, d) stored as (a, c, b, d) so that one 8-byte load gives
// a lane both B registers of an mma; row tok starts at tok (2 kpad + 128) +
// 8 ((tok & 1) + 8 ((tok >> 1) & 1)), which puts the 16 lanes of a half-warp
// load (4 tokens x 4 lanes) in 16 different 8-byte bank slots.

constexpr int kTcvRT = 2;                     // 16-row mma tiles per warp
constexpr uint32_t kTcvTabPitch = 144;        // 8 float4 + 16 bytes: the 8 g of a read in distinct banks
constexpr uint32_t kTcvTabWarp = kTcvRT * 8 * kTcvTabPitch;

__host__ __device__ constexpr uint32_t tcv_xstride(int kpad) { return 2u * kpad + 128u; }
__host__ __device__ constexpr uint32_t tcv_row(int tok, int kpad) {
  return tok * tcv_xstride(kpad) + 8u * ((tok & 1) + 8 * ((tok >> 1) & 1));
}
// shared layout before the ring: x rows | Sx [kpad/32][8 NB] | column
// scales [kpad/32][8 NB] | WC scale tables | two hand-over buffers of rows x
// 8 NB floats
__host__ __device__ constexpr uint32_t tcv_sx(int kpad, int nb) {
  return tcv_xstride(kpad) * 8u * nb;
}
__host__ __device__ constexpr uint32_t tcv_cs(int kpad, int nb) {
  return tcv_sx(kpad, nb) + 4u * (kpad / 32) * 8u * nb;
}
__host__ __device__ constexpr uint32_t tcv_tab(int kpad, int nb) {
  return tcv_cs(kpad, nb) + 4u * (kpad / 32) * 8u * nb;
}
__host__ __device__ constexpr uint32_t tcv_psum(int kpad, int nb, int wc) {
  return tcv_tab(kpad, nb) + wc * kTcvTabWarp;
}
__host__ __device__ constexpr uint32_t tcv_x_bytes(int kpad, int nb, int wc, int rows) {
  return (tcv_psum(kpad, nb, wc) + 2u * rows * 8u * nb * 4u + 127u) & ~127u;
}

// x of a K segment for the multi-token tensor-core product: per token, the
// positions as fp16 (each group of four (a, b, c, d) stored (a, c, b, d)),
// scaled per 32-position sub-block by a power of two 2^-f chosen from that
// token's largest |x| in it, as in stage_x_tc_raw (so x converts exactly
// within 2^31 of that largest); Sx, the fp32 sum of x per (sub-block, token);
// and the (sub-block, token) column scale 2^(f+24) (low-nibble sub-blocks,
// A = q 2^-24) or 2^(f+20) (high nibbles, A = 16 q 2^-24).
template <int NB>
__device__ void stage_x_tcv_raw(const uint16_t* x, int K, int nt, int kpad, uint32_t xsh,
                                int kbase) {
  constexpr int NTP = 8 * NB;
  constexpr int kInFlight = 4;    // 16-byte chunks of x a thread loads before converting them
  const int per_tok = kpad / 8;   // 16-byte chunks per token (a multiple of 32)
  const int total = NTP * per_tok;
  const int stride = static_cast<int>(blockDim.x);
  const uint32_t sxa = xsh + tcv_sx(kpad, NB);
  const uint32_t csa = xsh + tcv_cs(kpad, NB);
  const int lane = threadIdx.x & 31;
  // chunk q = token q / per_tok, positions 8 (q % per_tok) ..; a warp's 32
  // chunks always belong to one token
  for (int base = static_cast<int>(threadIdx.x) & ~31; base < total; base += kInFlight * stride) {
    uint4 v[kInFlight];
#pragma unroll
    for (int b = 0; b < kInFlight; ++b) {
      const int q = base + b * stride + lane;
      const int tok = q / per_tok, c = q % per_tok;
      const int k = kbase + 8 * c;
      v[b] = make_uint4(0, 0, 0, 0);
      if (q < total && tok < nt && k < K) v[b] = ldg_nc_v4(x + static_cast<int64_t>(tok) * K + k);
    }
#pragma unroll
    for (int b = 0; b < kInFlight; ++b) {
      if (base + b * stride >= total) break;   // warp-uniform
      const int q = base + b * stride + lane;
      const int tok = q / per_tok, c = q % per_tok;
      const uint32_t a = xsh + tcv_row(tok, kpad) + 16u * c;
      const int j = c >> 2;   // sub-block of the segment (the segment starts on an even one)
      if (tok >= nt) {
        // a token the launch does not have: its row is zero (what the
        // conversion below gives for zero x, without the work)
        asm volatile("st.shared.v2.u32 [%0], {%1, %1};" ::"r"(a), "r"(0u) : "memory");
        asm volatile("st.shared.v2.u32 [%0], {%1, %1};" ::"r"(a + 8u), "r"(0u) : "memory");
        if ((c & 3) == 0) {
          const float scale = __uint_as_float(static_cast<uint32_t>(127 + 24 - 4 * (j & 1)) << 23);
          asm volatile("st.shared.f32 [%0], %1;" ::"r"(sxa + 4u * (j * NTP + tok)), "f"(0.0f) : "memory");
          asm volatile("st.shared.f32 [%0], %1;" ::"r"(csa + 4u * (j * NTP + tok)), "f"(scale) : "memory");
        }
        continue;
      }
      const uint32_t w[4] = {v[b].x, v[b].y, v[b].z, v[b].w};
      float f[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
      }
      float sum = 0.0f, amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        sum += f[i];
        amax = fmaxf(amax, fabsf(f[i]));
      }
#pragma unroll
      for (int m = 1; m < 4; m <<= 1) {
        sum += __shfl_xor_sync(0xFFFFFFFFu, sum, m);
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, m));
      }
      int fs = amax > 0.0f ? static_cast<int>((__float_as_uint(amax) >> 23) & 0xFF) - 127 - 14 : 0;
      fs = fs < -100 ? -100 : (fs > 100 ? 100 : fs);
      const float down = __uint_as_float(static_cast<uint32_t>(127 - fs) << 23);   // 2^-fs, exact
      uint32_t e[4];
#pragma unroll
      for (int i = 0; i < 2; ++i) {   // (p0, p2), (p1, p3) of each group of four
        const __half2 lo = __floats2half2_rn(f[4 * i] * down, f[4 * i + 2] * down);
        const __half2 hi = __floats2half2_rn(f[4 * i + 1] * down, f[4 * i + 3] * down);
        e[2 * i] = *reinterpret_cast<const uint32_t*>(&lo);
        e[2 * i + 1] = *reinterpret_cast<const uint32_t*>(&hi);
      }
      // rows start on 8-byte boundaries: two 8-byte stores
      asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(a), "r"(e[0]), "r"(e[1]) : "memory");
      asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(a + 8u), "r"(e[2]), "r"(e[3]) : "memory");
      if ((c & 3) == 0) {
        const float scale = __uint_as_float(static_cast<uint32_t>(127 + 24 + fs - 4 * (j & 1)) << 23);
        asm volatile("st.shared.f32 [%0], %1;" ::"r"(sxa + 4u * (j * NTP + tok)), "f"(sum) : "memory");
        asm volatile("st.shared.f32 [%0], %1;" ::"r"(csa + 4u * (j * NTP + tok)), "f"(scale) : "memory");
      }
    }
  }
}
template <int NB>
__device__ void stage_x_tcv(const Params& p, uint32_t xsh, int kbase) {
  stage_x_tcv_raw<NB>(p.x, p.K, p.nt, p.kpad, xsh, kbase);
}

__device__ __forceinline__ void sts_f2(uint32_t a, float x, float y) {
  asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(a), "f"(x), "f"(y) : "memory");
}

// This warp's scale table for one super-block.  Entry (rt, g, j), a float4 at
// tab + (rt 8 + g) pitch + 16 j: (s1, s2) of row 16 rt + g and of row 16 rt +
// g + 8, sub-block j.  Lane l decodes the four chunks of row l of the warp.
template <class G>
__device__ __forceinline__ void tcv_scale_table(const Params& p, const Tile& tl, int sl,
                                                uint32_t st, int rbase, int s, uint32_t tab) {
  constexpr int F = G::kF;
  const int lane = threadIdx.x & 31;
  const int row = rbase + lane;
  const uint32_t te = tab + ((lane >> 4) * 8 + (lane & 7)) * kTcvTabPitch + 8u * ((lane >> 3) & 1);
  if constexpr (F == kG128) {
    const uint32_t po =
        (static_cast<uint32_t>(tl.row0 + row) * ((8u * p.nsb) & 15u) + sl * G::kPBytes) & 15u;
    const uint2 pr = lds64(st + p.pbase + row * p.pslot + po + 8 * s);
    const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&pr.x));
#pragma unroll
    for (int grp = 0; grp < 2; ++grp) {
      const float a = dd.x * byte_f(pr.y, grp);
      const float b = -(dd.y * byte_f(pr.y, 2 + grp));
#pragma unroll
      for (int j = 4 * grp; j < 4 * grp + 4; ++j) sts_f2(te + 16 * j, a, b);
    }
  } else {
    const uint4 hdr = lds128(st + row * p.slot + G::kBB * s);
    const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&hdr.x));
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t scp, mnp;
      scale_pair6(scale_sel(c), hdr.y, hdr.z, hdr.w, scp, mnp);
      const float a0 = dd.x * bytes01_f2(scp).x;
      const float a1 = dd.x * bytes01_f2(scp).y;
      sts_f2(te + 32 * c, a0, -(dd.y * bytes01_f2(mnp).x));
      sts_f2(te + 32 * c + 16, a1, -(dd.y * bytes01_f2(mnp).y));
    }
  }
}

// One stage for this warp's rows rbase .. rbase + 32, NB blocks of eight tokens.
template <class G, int NB>
__device__ __forceinline__ void tcv_stage_q4(const Params& p, const Tile& tl, int sl, int xsl,
                                             uint32_t st, int rbase, uint32_t xsh, uint32_t tab,
                                             float2 (&acc)[NB][kTcvRT][2]) {
  constexpr int F = G::kF;
  constexpr int NTP = 8 * NB;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const uint32_t sxa = xsh + tcv_sx(p.kpad, NB);
  const uint32_t csa = xsh + tcv_cs(p.kpad, NB);
  const int nrt = tl.rcnt - rbase > 16 ? 2 : 1;   // live row tiles of this warp
#pragma unroll
  for (int s = 0; s < G::kSlabSB; ++s) {
    if (sl * G::kSlabSB + s >= p.nsb) break;
    const int sbx = xsl * G::kSlabSB + s;
    tcv_scale_table<G>(p, tl, sl, st, rbase, s, tab);
    __syncwarp();
    uint32_t qa[kTcvRT][2];
#pragma unroll
    for (int rt = 0; rt < kTcvRT; ++rt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t rs = st + (rbase + 16 * rt + g + 8 * h) * p.slot;
        qa[rt][h] = (F == kG128) ? rs + 128 * s + 8 * t : rs + G::kBB * s + 16 + 8 * t;
      }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      // A registers [tile][row h][word m]: low nibbles of bytes (0, 2), (1,
      // 3); high nibbles of bytes (0, 2), (1, 3)
      uint32_t l02[kTcvRT][2][2], l13[kTcvRT][2][2], h02[kTcvRT][2][2], h13[kTcvRT][2][2];
#pragma unroll
      for (int rt = 0; rt < kTcvRT; ++rt)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint2 wv = (rt < nrt) ? lds64(qa[rt][h] + 32 * c) : make_uint2(0, 0);
          const uint32_t W[2] = {wv.x, wv.y};
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            // fp16 subnormals: q 2^-24 (low nibbles), 16 q 2^-24 (high, in place)
            const uint32_t w8 = W[m] >> 8;
            l02[rt][h][m] = W[m] & 0x000F000Fu;
            l13[rt][h][m] = w8 & 0x000F000Fu;
            h02[rt][h][m] = W[m] & 0x00F000F0u;
            h13[rt][h][m] = w8 & 0x00F000F0u;
          }
        }
      const int jlo = 8 * sbx + 2 * c;   // sub-block of the segment (low nibbles)
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        const uint32_t xr = xsh + tcv_row(8 * nb + g, p.kpad) + 2u * (256 * sbx + 64 * c + 8 * t);
        float dl[kTcvRT][4] = {}, dh[kTcvRT][4] = {};
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          const uint2 bl = lds64(xr + 8 * m);
          const uint2 bh = lds64(xr + 64 + 8 * m);
#pragma unroll
          for (int rt = 0; rt < kTcvRT; ++rt) {
            mma_f16(dl[rt], l02[rt][0][m], l02[rt][1][m], l13[rt][0][m], l13[rt][1][m], bl.x, bl.y);
            mma_f16(dh[rt], h02[rt][0][m], h02[rt][1][m], h13[rt][0][m], h13[rt][1][m], bh.x, bh.y);
          }
        }
        const float2 sxl = lds_f2(sxa + 4u * (jlo * NTP + 8 * nb + 2 * t));
        const float2 sxh = lds_f2(sxa + 4u * ((jlo + 1) * NTP + 8 * nb + 2 * t));
        const float2 csl = lds_f2(csa + 4u * (jlo * NTP + 8 * nb + 2 * t));   // column scales
        const float2 csh = lds_f2(csa + 4u * ((jlo + 1) * NTP + 8 * nb + 2 * t));
#pragma unroll
        for (int rt = 0; rt < kTcvRT; ++rt) {
          const uint32_t te = tab + (rt * 8 + g) * kTcvTabPitch + 32u * c;
          const float4 el = lds_f4(te), eh = lds_f4(te + 16);   // (s1, s2) of rows g, g + 8
          float2& a0 = acc[nb][rt][0];
          float2& a1 = acc[nb][rt][1];
          a0 = __ffma2_rn(make_float2(el.x, el.x), __fmul2_rn(csl, make_float2(dl[rt][0], dl[rt][1])), a0);
          a0 = __ffma2_rn(make_float2(el.y, el.y), sxl, a0);
          a0 = __ffma2_rn(make_float2(eh.x, eh.x), __fmul2_rn(csh, make_float2(dh[rt][0], dh[rt][1])), a0);
          a0 = __ffma2_rn(make_float2(eh.y, eh.y), sxh, a0);
          a1 = __ffma2_rn(make_float2(el.z, el.z), __fmul2_rn(csl, make_float2(dl[rt][2], dl[rt][3])), a1);
          a1 = __ffma2_rn(make_float2(el.w, el.w), sxl, a1);
          a1 = __ffma2_rn(make_float2(eh.z, eh.z), __fmul2_rn(csh, make_float2(dh[rt][2], dh[rt][3])), a1);
          a1 = __ffma2_rn(make_float2(eh.w, eh.w), sxh, a1);
        }
      }
    }
    __syncwarp();   // the table is rebuilt for the next super-block
  }
}

template <int F, int WC, int NB>
__global__ void __launch_bounds__((WC + 2) * 32, WC <= 4 ? 2 : 1)
    gemv_tcv(const __grid_constant__ Params p, int stages) {
  using G = TGeo<F, WC, kTcvRT>;
  constexpr int NTP = 8 * NB;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[2 * kMaxStages + 4];
  __shared__ int stage_tile[kMaxStages];
  __shared__ int part_tile[2];
  const uint32_t bar_full = smem_addr(&bars[0]);
  const uint32_t bar_empty = smem_addr(&bars[kMaxStages]);
  const uint32_t part_full = smem_addr(&bars[2 * kMaxStages]);
  const uint32_t part_empty = smem_addr(&bars[2 * kMaxStages + 2]);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t xsh = smem_addr(smem);
  const uint32_t tab = xsh + tcv_tab(p.kpad, NB) + warp * kTcvTabWarp;
  const uint32_t psum = xsh + tcv_psum(p.kpad, NB, WC);
  const uint32_t ring_a = xsh + p.x_bytes;
  const int kseg = static_cast<int>(blockIdx.x) % p.ksplit;
  const int cta = static_cast<int>(blockIdx.x) / p.ksplit;
  const int cps = static_cast<int>(gridDim.x) / p.ksplit;
  const int sl0 = kseg * p.slabs;
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(bar_full + 8 * s, p.tma ? 1 : 32);
      mbar_init(bar_empty + 8 * s, WC);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(part_full + 8 * b, WC);
      mbar_init(part_empty + 8 * b, 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const bool producer = warp == WC, reducer = warp == WC + 1;
  asm volatile("griddepcontrol.launch_dependents;");
  Ring ring;
  if (producer) produce_prefill<G>(p, smem, ring_a, bar_full, stage_tile, stages, cta, cps, sl0, ring);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  stage_x_tcv<NB>(p, xsh, kseg * p.kpad);
  __syncthreads();
  if (producer) {
    produce_rest<G>(p, smem, ring_a, bar_full, bar_empty, stage_tile, stages, cta, cps, kseg, sl0,
                    ring);
    return;
  }
  if (reducer) {
    if (p.ksplit > 1) tc_reduce<NTP>(p, psum, part_full, part_empty, part_tile, kseg);
    return;
  }
  const int g = lane >> 2, t = lane & 3;
  const int rbase = 16 * kTcvRT * warp;
  float2 acc[NB][kTcvRT][2];
  Tile tl{};
  int tix = 0, unit = 0;
  int xsl = 0, slot = 0;
  uint32_t parity = 0;
  // hand unit `unit` (tile tix, or -1: no more) to the reducer through
  // buffer unit & 1, once the reducer has drained that buffer's previous use
  auto hand_over = [&](bool data) -> bool {
    const int b = unit & 1;
    if (unit >= 2 && !mbar_wait_warp(part_empty + 8 * b, static_cast<uint32_t>((unit >> 1) - 1) & 1u))
      return false;
    if (data) {
      const uint32_t buf = psum + 4u * static_cast<uint32_t>(b * p.tile_rows * NTP);
#pragma unroll
      for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int rt = 0; rt < kTcvRT; ++rt)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t a = buf + 4u * ((rbase + 16 * rt + g + 8 * h) * NTP + 8 * nb + 2 * t);
            sts_f2(a, acc[nb][rt][h].x, acc[nb][rt][h].y);
          }
    }
    if (warp == 0 && lane == 0) part_tile[b] = data ? tix : -1;
    __syncwarp();
    if (lane == 0) mbar_arrive(part_full + 8 * b);
    ++unit;
    return true;
  };
  for (;;) {
    const int sl = sl0 + xsl;
    if (!mbar_wait_warp(bar_full + 8 * slot, parity)) return;
    if (xsl == 0) {
      tix = stage_tile[slot];
      if (tix < 0) {
        if (p.ksplit > 1) hand_over(false);
        return;
      }
      tl = tile_of(p, tix);
#pragma unroll
      for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int rt = 0; rt < kTcvRT; ++rt) acc[nb][rt][0] = acc[nb][rt][1] = make_float2(0.0f, 0.0f);
    }
    const uint32_t st = ring_a + slot * p.stage;
    if (rbase < tl.rcnt) tcv_stage_q4<G, NB>(p, tl, sl, xsl, st, rbase, xsh, tab, acc);
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * slot);
    if (xsl == p.slabs - 1) {
      if (p.ksplit == 1) {
        float* y = pick(p.g.y, tl.mi);
        const int64_t N = pick(p.g.N, tl.mi);
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
          for (int rt = 0; rt < kTcvRT; ++rt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int row = rbase + 16 * rt + g + 8 * h;
              const int tok = 8 * nb + 2 * t;
              if (row < tl.rcnt) {
                if (tok < p.nt) y[static_cast<int64_t>(tok) * N + tl.row0 + row] = acc[nb][rt][h].x;
                if (tok + 1 < p.nt)
                  y[static_cast<int64_t>(tok + 1) * N + tl.row0 + row] = acc[nb][rt][h].y;
              }
            }
      } else if (!hand_over(true)) {
        return;
      }
    }
    if (++xsl == p.slabs) xsl = 0;
    if (++slot == stages) {
      slot = 0;
      parity ^= 1u;
    }
  }
}

// ===================================================== small-launch kernel
//
// n_tok = 1 on Q4_K / Q4_G128 launches of a few megabytes (the attention
// projections of a decoder layer).  Such a launch streams its weights in a
// couple of microseconds, so what it costs beyond that is fixed: launch,
// waiting for the previous kernel, staging x, handing partial sums between
// CTAs.  This kernel keeps that small:
//   * one wave of CTAs (at most one per SM); CTA c owns the 16-row tiles
//     [c T / C, (c+1) T / C) over all of K, so no partial sum leaves a CTA;
//   * warp w owns slice (tile w / ks, K slice w % ks) of at most sbs
//     super-blocks; before waiting for the previous kernel it requests the
//     slice into its part of shared memory (one mbarrier per warp counts the
//     bytes), so every weight byte of the launch is requested at once, while
//     the previous kernel finishes.  Q4_K: one 2-D tensor copy of the 16 rows
//     (the number of copy instructions, not their size, is what costs here);
//     Q4_G128, or a slice wider than a tensor box: one cp.async.bulk per row;
//   * after griddepcontrol.wait the CTA stages x as gemv_tc1 does, and each
//     warp runs gemv_tc1's tensor-core product (q exact as fp16 subnormals,
//     the eight n8 columns carrying the eight sub-blocks of a super-block) on
//     its slice as soon as its bytes have landed;
//   * the ks slice sums of a row are added in slice order in shared memory
//     (a fixed order: the result does not depend on timing) and written.
// Row segments are copied at a pitch that is an odd multiple of 16 bytes, so
// the eight rows a warp reads at once fall in different bank groups.

constexpr int kSmallMaxWarps = 24;   // 768 threads: registers for the product without spills
// Q5_K's product holds the qh words too: 20 warps (102 registers a thread)
template <int F>
constexpr int small_max_warps() { return F == kQ5K ? 20 : kSmallMaxWarps; }

struct SmallParams {
  GemvGroup g;
  const uint16_t* x;
  int K, nsb;
  int tiles;                  // 16-row tiles of the group (a tile lies in one matrix)
  int tile_end[kMaxGroup];    // cumulative tile counts per matrix
  int ks;                     // K slices per tile (warps per tile)
  int sbs;                    // super-blocks per slice (the last slice may have fewer)
  int max_tiles;              // most tiles one CTA owns
  uint32_t pitch;             // shared bytes per row of a slice: records (Q4_G128: q plane)
  uint32_t ppitch;            // Q4_G128: shared bytes per row of the slice's params (+ halo)
  uint32_t warp_bytes;        // shared bytes per warp: 16 rows x (pitch + ppitch), 128-aligned
  uint32_t x_bytes;           // staged x, Sx, zero block and the slice sums, 128-aligned
  // gemv_small_mt: tokens, and the offsets of the warps' scale tables and of
  // the slice sums
  int nt;
  uint32_t tab_off, red_off;
  // Q4_K, Q5_K: a warp's slice comes in one tensor copy (16 rows x pitch bytes)
  // through the matrix's 2-D map, where the maps could be made
  int tma;
  CUtensorMap tm[kMaxGroup];
};

__device__ __forceinline__ Tile small_tile(const SmallParams& p, int t) {
  int mi = 0, base = 0;
#pragma unroll
  for (int i = 0; i < kMaxGroup - 1; ++i)
    if (i < p.g.count - 1 && t >= p.tile_end[i]) {
      mi = i + 1;
      base = p.tile_end[i];
    }
  Tile r;
  r.mi = mi;
  r.row0 = (t - base) * 16;
  r.rcnt = min(16, pick(p.g.N, mi) - r.row0);
  return r;
}

// Issue the copies of this warp's slice; returns the bytes they deliver.
// Tensor copy (Q4_K, Q5_K): lane 0 copies the 16 rows x pitch bytes from the
// slice's first record (x in 8-byte elements; the box runs 16 bytes past a
// slice whose records leave the pitch an even multiple of 16 bytes); rows
// past the matrix and bytes past a row are zero-filled and counted.
// Otherwise lane r < 16 copies row r's segment (the bytes are summed over
// the warp).  Q4_G128 param segments start on 8-byte boundaries: each is
// copied from the 16-byte boundary at or below it (the consumer skips the
// offset), and bytes past the plane's last 16-byte boundary are loaded with
// plain loads.
template <int F>
__device__ __forceinline__ uint32_t small_issue(const SmallParams& p, const Tile& tl, int sb0,
                                                int nsl, uint32_t wreg, uint32_t bar,
                                                uint8_t* smem) {
  const int lane = threadIdx.x & 31;
  if constexpr (F == kQ4K || F == kQ5K) {
    if (p.tma) {
      if (lane == 0) tma_load_2d(wreg, &p.tm[tl.mi], sb0 * (block_bytes(F) / 8), tl.row0, bar);
      return 16u * p.pitch;
    }
  }
  uint32_t tx = 0;
  if (lane < tl.rcnt) {
    const uint8_t* W = pick(p.g.W, tl.mi);
    const int64_t N = pick(p.g.N, tl.mi);
    const int64_t idx = (tl.row0 + lane) * static_cast<int64_t>(p.nsb) + sb0;
    if constexpr (F == kG128) {
      const uint32_t qb = static_cast<uint32_t>(nsl) * 128u;
      bulk_g2s(wreg + lane * p.pitch, W + idx * 128, qb, bar);
      tx += qb;
      const uint8_t* P = W + N * p.nsb * 128;
      const int64_t off = idx * 8, end = off + 8 * nsl;
      const int64_t lo = off & ~int64_t{15};
      const int64_t cap = (N * p.nsb * 8) & ~int64_t{15};
      int64_t hi = (end + 15) & ~int64_t{15};
      if (hi > cap) hi = cap;
      const uint32_t dst = wreg + 16u * p.pitch + lane * p.ppitch;
      if (hi > lo) {
        bulk_g2s(dst, P + lo, static_cast<uint32_t>(hi - lo), bar);
        tx += static_cast<uint32_t>(hi - lo);
      }
      for (int64_t b = (hi > lo ? hi : lo); b < end; ++b)
        smem[(dst - smem_addr(smem)) + (b - lo)] = __ldg(P + b);
    } else {
      const uint32_t bytes = static_cast<uint32_t>(nsl) * block_bytes(F);
      bulk_g2s(wreg + lane * p.pitch, W + idx * block_bytes(F), bytes, bar);
      tx += bytes;
    }
  }
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) tx += __shfl_xor_sync(0xFFFFFFFFu, tx, m);
  return tx;
}

// One super-block s of this warp's slice (rows g, g + 8 of the tile; lane t
// takes chunk t): gemv_tc1's product, operands from the warp's region.
template <int F>
__device__ __forceinline__ void small_sb_q4(const SmallParams& p, uint32_t wreg, int s, int sbx,
                                            int64_t idx_g, int64_t idx_g8, uint32_t xsh,
                                            const ScaleSel& ss, float2 (&acc)[2]) {
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const uint32_t xsum = xsh + 2u * static_cast<uint32_t>(p.K);
  const uint32_t xscl = xsum + 4u * static_cast<uint32_t>(p.K / 32);
  const uint32_t zero = xsh + tc_zero_off(p.K, 32);
  const bool act_lo = g == 2 * t, act_hi = g == 2 * t + 1;   // column g of the B operand
  const uint32_t xlo = act_lo ? xsh + 64u * (8 * sbx + 2 * t) : zero;
  const uint32_t xhi = act_hi ? xsh + 64u * (8 * sbx + 2 * t + 1) : zero;
  // chunk t of the qs bytes (Q5_K: after the 32 qh bytes) of rows g, g + 8
  constexpr uint32_t kQs = (F == kG128) ? 0u : (F == kQ5K ? 48u : 16u);
  uint32_t qa[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t rs = wreg + (g + 8 * h) * p.pitch;
    qa[h] = (F == kG128) ? rs + 128 * s + 32 * t : rs + block_bytes(F) * s + kQs + 32 * t;
  }
  float d[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  if constexpr (F == kQ5K) {
    const uint32_t qh0 = wreg + g * p.pitch + block_bytes(F) * s + 16;
    tc_sb_product_q5(qa[0], qa[1], qh0, qh0 + 8 * p.pitch, xlo, xhi, q5_rot(2 * t), d);
  } else {
    tc_sb_product(qa[0], qa[1], xlo, xhi, d);
  }
  // (s1, s2) of sub-blocks (2t, 2t+1) of rows g and g + 8
  float2 s1[2], s2[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t rs = wreg + (g + 8 * h) * p.pitch;
    if constexpr (F == kG128) {
      const int64_t idx = h ? idx_g8 : idx_g;
      const uint32_t pa = wreg + 16u * p.pitch + (g + 8 * h) * p.ppitch +
                          static_cast<uint32_t>((idx * 8) & 15) + 8 * s;
      const uint2 pr = lds64(pa);
      const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&pr.x));
      const int grp = t >> 1;
      const float a = dd.x * byte_f(pr.y, grp);
      const float b = -(dd.y * byte_f(pr.y, 2 + grp));
      s1[h] = make_float2(a, a);
      s2[h] = make_float2(b, b);
    } else {
      const uint4 hdr = lds128(rs + block_bytes(F) * s);
      const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&hdr.x));
      uint32_t scp, mnp;
      scale_pair6(ss, hdr.y, hdr.z, hdr.w, scp, mnp);
      s1[h] = __fmul2_rn(make_float2(dd.x, dd.x), bytes01_f2(scp));
      s2[h] = __fmul2_rn(make_float2(-dd.y, -dd.y), bytes01_f2(mnp));
    }
  }
  const float2 sx = lds_f2(xsum + 4u * (8 * sbx + 2 * t));
  const float2 cs = lds_f2(xscl + 4u * (8 * sbx + 2 * t));   // column scales
  tc_epilogue(acc, d, cs, s1[0], s2[0], s1[1], s2[1], sx);
}

template <int F>
__global__ void __launch_bounds__(small_max_warps<F>() * 32, 1)
    gemv_small(const __grid_constant__ SmallParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[kSmallMaxWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = static_cast<int>(gridDim.x);
  const int t0 = static_cast<int>(static_cast<int64_t>(blockIdx.x) * p.tiles / C);
  const int t1 = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * p.tiles / C);
  const int lt = warp / p.ks, j = warp % p.ks;
  const bool active = t0 + lt < t1;           // warp-uniform
  const int sb0 = j * p.sbs;
  const int nsl = min(p.sbs, p.nsb - sb0);    // >= 1 (no empty slices)
  const uint32_t xsh = smem_addr(smem);
  const uint32_t red = xsh + tc_x_only(p.K, 32);   // slice sums [max_tiles][ks][16]
  const uint32_t wreg = xsh + p.x_bytes + static_cast<uint32_t>(warp) * p.warp_bytes;
  const uint32_t bar = smem_addr(&bars[warp]);
  Tile tl{};
  if (active) tl = small_tile(p, t0 + lt);
  if (lane == 0) {
    mbar_init(bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  // the next kernel may start as SMs free up; it reads what this kernel
  // writes only after its own griddepcontrol.wait
  asm volatile("griddepcontrol.launch_dependents;");
  if (active) {
    const uint32_t tx = small_issue<F>(p, tl, sb0, nsl, wreg, bar, smem);
    if (lane == 0) mbar_arrive_tx(bar, tx);
  }
  // x may be produced by the previous kernel
  asm volatile("griddepcontrol.wait;" ::: "memory");
  stage_x_tc_raw<32>(p.x, p.K, p.K, xsh, 0);
  __syncthreads();
  const int g = lane >> 2, t = lane & 3;
  float v[2] = {0.0f, 0.0f};
  if (active && mbar_wait_warp(bar, 0u)) {
    const ScaleSel ss = scale_sel(t);
    const int64_t idx_g = (tl.row0 + g) * static_cast<int64_t>(p.nsb) + sb0;
    const int64_t idx_g8 = (tl.row0 + g + 8) * static_cast<int64_t>(p.nsb) + sb0;
    float2 acc[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
    for (int s = 0; s < nsl; ++s) small_sb_q4<F>(p, wreg, s, sb0 + s, idx_g, idx_g8, xsh, ss, acc);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float a = acc[h].x + acc[h].y;
      a += __shfl_xor_sync(0xFFFFFFFFu, a, 1);
      a += __shfl_xor_sync(0xFFFFFFFFu, a, 2);
      v[h] = a;
    }
  }
  if (active && t == 0) {
#pragma unroll
    for (int h = 0; h < 2; ++h)
      asm volatile("st.shared.f32 [%0], %1;" ::"r"(red + 4u * ((lt * p.ks + j) * 16 + g + 8 * h)),
                   "f"(v[h])
                   : "memory");
  }
  __syncthreads();
  // row i of the CTA's tiles: its slice sums in slice order
  const int nrows = (t1 - t0) * 16;
  for (int i = static_cast<int>(threadIdx.x); i < nrows; i += static_cast<int>(blockDim.x)) {
    const int tt = i >> 4, r = i & 15;
    const Tile ti = small_tile(p, t0 + tt);
    if (r >= ti.rcnt) continue;
    float a = 0.0f;
    for (int jj = 0; jj < p.ks; ++jj) {
      float e;
      asm volatile("ld.shared.f32 %0, [%1];" : "=f"(e) : "r"(red + 4u * ((tt * p.ks + jj) * 16 + r)));
      a += e;
    }
    pick(p.g.y, ti.mi)[ti.row0 + r] = a;
  }
}

// ------------------------------------------- small launches, 2..8 tokens
//
// gemv_small's structure -- one wave of CTAs, every warp's slice of 16 rows
// requested (one tensor copy, or row copies) before the dependency wait,
// slice sums added in shared memory in slice order -- with gemv_tcv's
// product: the tokens are the n8 columns,
// A is exact as fp16 subnormals, x is staged per token in fp16 with a
// power-of-two scale per (token, sub-block) (stage_x_tcv_raw), and each
// warp decodes its rows' (s1, s2) into a table once per super-block.  Like
// gemv_small, it needs no global scratch: at verify widths the small
// launches (attention projections) otherwise pay the split-K exchange.
constexpr int kSmallMtMaxWarps = 20;   // registers for the multi-token product

// This warp's (s1, s2) table for super-block s of its slice: entry (g, j), a
// float4 at tab + g pitch + 16 j, holds (s1, s2) of row g and of row g + 8,
// sub-block j.  Lane r < 16 decodes row r.
template <int F>
__device__ __forceinline__ void small_mt_table(const SmallParams& p, const Tile& tl, uint32_t wreg,
                                               int s, int sb0, uint32_t tab) {
  const int lane = threadIdx.x & 31;
  if (lane >= 16) return;
  const uint32_t te = tab + (lane & 7) * kTcvTabPitch + 8u * (lane >> 3);
  if constexpr (F == kG128) {
    const int64_t idx = (tl.row0 + lane) * static_cast<int64_t>(p.nsb) + sb0;
    const uint32_t pa = wreg + 16u * p.pitch + lane * p.ppitch +
                        static_cast<uint32_t>((idx * 8) & 15) + 8 * s;
    const uint2 pr = lds64(pa);
    const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&pr.x));
#pragma unroll
    for (int grp = 0; grp < 2; ++grp) {
      const float a = dd.x * byte_f(pr.y, grp);
      const float b = -(dd.y * byte_f(pr.y, 2 + grp));
#pragma unroll
      for (int j = 4 * grp; j < 4 * grp + 4; ++j) sts_f2(te + 16 * j, a, b);
    }
  } else {
    const uint4 hdr = lds128(wreg + lane * p.pitch + block_bytes(F) * s);
    const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&hdr.x));
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t scp, mnp;
      scale_pair6(scale_sel(c), hdr.y, hdr.z, hdr.w, scp, mnp);
      sts_f2(te + 32 * c, dd.x * bytes01_f2(scp).x,
             -(dd.y * bytes01_f2(mnp).x));
      sts_f2(te + 32 * c + 16, dd.x * bytes01_f2(scp).y,
             -(dd.y * bytes01_f2(mnp).y));
    }
  }
}

// Super-block s of this warp's slice (row s of the row's sb0 + s) for rows
// g, g + 8 and tokens 2t, 2t + 1: gemv_tcv's product for one 16-row tile.
template <int F>
__device__ __forceinline__ void small_mt_sb(const SmallParams& p, uint32_t wreg, int s, int sbx,
                                            uint32_t xsh, uint32_t tab, float2 (&acc)[2]) {
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const uint32_t sxa = xsh + tcv_sx(p.K, 1);
  const uint32_t csa = xsh + tcv_cs(p.K, 1);
  // bytes 8t .. 8t + 7 of each 32-byte qs chunk (Q5_K: after the 32 qh
  // bytes) of rows g, g + 8; Q5_K: the qh words of the same positions
  constexpr uint32_t kQs = (F == kG128) ? 0u : (F == kQ5K ? 48u : 16u);
  uint32_t qa[2];
  uint32_t qh[2][2] = {{0u, 0u}, {0u, 0u}};
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t rs = wreg + (g + 8 * h) * p.pitch;
    qa[h] = (F == kG128) ? rs + 128 * s + 8 * t : rs + block_bytes(F) * s + kQs + 8 * t;
    if constexpr (F == kQ5K) {
      const uint2 hv = lds64(rs + block_bytes(F) * s + 16 + 8 * t);
      qh[h][0] = hv.x;
      qh[h][1] = hv.y;
    }
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t l02[2][2], l13[2][2], h02[2][2], h13[2][2];   // [row h][word m]
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint2 wv = lds64(qa[h] + 32 * c);
      const uint32_t W[2] = {wv.x, wv.y};
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const uint32_t w8 = W[m] >> 8;
        l02[h][m] = W[m] & 0x000F000Fu;
        l13[h][m] = w8 & 0x000F000Fu;
        h02[h][m] = W[m] & 0x00F000F0u;
        h13[h][m] = w8 & 0x00F000F0u;
        if constexpr (F == kQ5K) {   // the fifth bits of sub-blocks 2c, 2c + 1
          const Q5Rot rot = q5_rot(2 * c);
          const uint32_t q = qh[h][m];
          l02[h][m] = or_bits(l02[h][m], rotl32(q, rot.lo02), 0x00100010u);
          l13[h][m] = or_bits(l13[h][m], rotl32(q, rot.lo13), 0x00100010u);
          h02[h][m] = or_bits(h02[h][m], rotl32(q, rot.hi02), 0x01000100u);
          h13[h][m] = or_bits(h13[h][m], rotl32(q, rot.hi13), 0x01000100u);
        }
      }
    }
    const int jlo = 8 * sbx + 2 * c;   // sub-block of the row (low nibbles)
    const uint32_t xr = xsh + tcv_row(g, p.K) + 2u * (256 * sbx + 64 * c + 8 * t);
    float dl[4] = {0.f, 0.f, 0.f, 0.f}, dh[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      const uint2 bl = lds64(xr + 8 * m);
      const uint2 bh = lds64(xr + 64 + 8 * m);
      mma_f16(dl, l02[0][m], l02[1][m], l13[0][m], l13[1][m], bl.x, bl.y);
      mma_f16(dh, h02[0][m], h02[1][m], h13[0][m], h13[1][m], bh.x, bh.y);
    }
    const float2 sxl = lds_f2(sxa + 4u * (jlo * 8 + 2 * t));
    const float2 sxh = lds_f2(sxa + 4u * ((jlo + 1) * 8 + 2 * t));
    const float2 csl = lds_f2(csa + 4u * (jlo * 8 + 2 * t));   // column scales
    const float2 csh = lds_f2(csa + 4u * ((jlo + 1) * 8 + 2 * t));
    const uint32_t te = tab + g * kTcvTabPitch + 32u * c;
    const float4 el = lds_f4(te), eh = lds_f4(te + 16);   // (s1, s2) of rows g, g + 8
    acc[0] = __ffma2_rn(make_float2(el.x, el.x), __fmul2_rn(csl, make_float2(dl[0], dl[1])), acc[0]);
    acc[0] = __ffma2_rn(make_float2(el.y, el.y), sxl, acc[0]);
    acc[0] = __ffma2_rn(make_float2(eh.x, eh.x), __fmul2_rn(csh, make_float2(dh[0], dh[1])), acc[0]);
    acc[0] = __ffma2_rn(make_float2(eh.y, eh.y), sxh, acc[0]);
    acc[1] = __ffma2_rn(make_float2(el.z, el.z), __fmul2_rn(csl, make_float2(dl[2], dl[3])), acc[1]);
    acc[1] = __ffma2_rn(make_float2(el.w, el.w), sxl, acc[1]);
    acc[1] = __ffma2_rn(make_float2(eh.z, eh.z), __fmul2_rn(csh, make_float2(dh[2], dh[3])), acc[1]);
    acc[1] = __ffma2_rn(make_float2(eh.w, eh.w), sxh, acc[1]);
  }
}

template <int F>
__global__ void __launch_bounds__(kSmallMtMaxWarps * 32, 1)
    gemv_small_mt(const __grid_constant__ SmallParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[kSmallMtMaxWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = static_cast<int>(gridDim.x);
  const int t0 = static_cast<int>(static_cast<int64_t>(blockIdx.x) * p.tiles / C);
  const int t1 = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * p.tiles / C);
  const int lt = warp / p.ks, j = warp % p.ks;
  const bool active = t0 + lt < t1;           // warp-uniform
  const int sb0 = j * p.sbs;
  const int nsl = min(p.sbs, p.nsb - sb0);    // >= 1 (no empty slices)
  const uint32_t xsh = smem_addr(smem);
  const uint32_t tab = xsh + p.tab_off + static_cast<uint32_t>(warp) * (8u * kTcvTabPitch);
  const uint32_t red = xsh + p.red_off;       // slice sums [max_tiles][ks][16][8]
  const uint32_t wreg = xsh + p.x_bytes + static_cast<uint32_t>(warp) * p.warp_bytes;
  const uint32_t bar = smem_addr(&bars[warp]);
  Tile tl{};
  if (active) tl = small_tile(p, t0 + lt);
  if (lane == 0) {
    mbar_init(bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  asm volatile("griddepcontrol.launch_dependents;");
  if (active) {
    const uint32_t tx = small_issue<F>(p, tl, sb0, nsl, wreg, bar, smem);
    if (lane == 0) mbar_arrive_tx(bar, tx);
  }
  // x may be produced by the previous kernel
  asm volatile("griddepcontrol.wait;" ::: "memory");
  stage_x_tcv_raw<1>(p.x, p.K, p.nt, p.K, xsh, 0);
  __syncthreads();
  const int g = lane >> 2, t = lane & 3;
  float2 acc[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
  if (active && mbar_wait_warp(bar, 0u)) {
    for (int s = 0; s < nsl; ++s) {
      small_mt_table<F>(p, tl, wreg, s, sb0, tab);
      __syncwarp();
      small_mt_sb<F>(p, wreg, s, sb0 + s, xsh, tab, acc);
      __syncwarp();   // the table is rebuilt for the next super-block
    }
  }
  if (active) {
#pragma unroll
    for (int h = 0; h < 2; ++h)
      sts_f2(red + 4u * (((lt * p.ks + j) * 16 + g + 8 * h) * 8 + 2 * t), acc[h].x, acc[h].y);
  }
  __syncthreads();
  // (row, token) i of the CTA's tiles: its slice sums in slice order
  const int nval = (t1 - t0) * 16 * 8;
  for (int i = static_cast<int>(threadIdx.x); i < nval; i += static_cast<int>(blockDim.x)) {
    const int tt = i >> 7, r = (i >> 3) & 15, k = i & 7;
    const Tile ti = small_tile(p, t0 + tt);
    if (r >= ti.rcnt || k >= p.nt) continue;
    float a = 0.0f;
    for (int jj = 0; jj < p.ks; ++jj) {
      float e;
      asm volatile("ld.shared.f32 %0, [%1];"
                   : "=f"(e)
                   : "r"(red + 4u * (((tt * p.ks + jj) * 16 + r) * 8 + k)));
      a += e;
    }
    pick(p.g.y, ti.mi)[static_cast<int64_t>(k) * pick(p.g.N, ti.mi) + ti.row0 + r] = a;
  }
}

struct DevInfo {
  int sms = 0;
  size_t smem_optin = 0;      // dynamic + static shared memory one CTA may use
  size_t smem_sm = 0;         // shared memory of one SM
  size_t smem_reserved = 0;   // shared memory the driver reserves per CTA
};

// Per-device state is kept for device ordinals below kMaxDevices; a launch on
// a higher ordinal (or when the current device cannot be read) is declined.
constexpr int kMaxDevices = 64;
int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) {
    (void)cudaGetLastError();
    return -1;
  }
  return d >= 0 && d < kMaxDevices ? d : -1;
}

// Attributes of the current device, read once per device (thread-safe);
// nullptr if the device is out of range.
const DevInfo* dev_info() {
  static DevInfo info[kMaxDevices];
  static std::once_flag once[kMaxDevices];
  const int d = current_device();
  if (d < 0) return nullptr;
  std::call_once(once[d], [d] {
    DevInfo& i = info[d];
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, d);
    i.sms = v;
    cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, d);
    i.smem_optin = static_cast<size_t>(v);
    cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerMultiprocessor, d);
    i.smem_sm = static_cast<size_t>(v);
    cudaDeviceGetAttribute(&v, cudaDevAttrReservedSharedMemoryPerBlock, d);
    i.smem_reserved = static_cast<size_t>(v);
    (void)cudaGetLastError();
  });
  return info[d].sms > 0 ? &info[d] : nullptr;
}

// Dynamic shared memory above 48 KB is opt-in per kernel and per device:
// raise `kern`'s limit on the current device to at least `smem`.
// `configured` is that kernel's per-device record of the value set.
std::mutex& attr_mutex() {
  static std::mutex m;
  return m;
}
template <typename Kern>
bool raise_smem_limit(Kern* kern, size_t smem, size_t (&configured)[kMaxDevices]) {
  const int d = current_device();
  if (d < 0) return false;
  std::lock_guard<std::mutex> lock(attr_mutex());
  if (smem <= configured[d]) return true;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  configured[d] = smem;
  return true;
}

// A launch that fails leaves no error behind for the caller's status check
// (the dispatcher then tries the next configuration).
bool launched(cudaError_t e) {
  if (e == cudaSuccess) return true;
  (void)cudaGetLastError();
  return false;
}

constexpr size_t kStaticSmem = 256;   // the kernel's static shared memory (barriers, flag), rounded up

// A nonzero tag per launch for the split-K partial sums (put_partial).
uint32_t next_tag() {
  static std::atomic<uint32_t> seq{0};
  uint32_t t = 0;
  while (t == 0) t = seq.fetch_add(1u, std::memory_order_relaxed) + 1u;
  return t;
}

// Split-K scratch of the current device: a fixed region of kMaxTiles arrival
// counters, then the partial sums.  The counter region never moves within a
// buffer, so counters stay zero across launches of any shape (partial sums of
// one launch never land on another launch's counters).  Grown on demand
// (never while the stream is being captured), zero-filled when allocated;
// kernels leave every counter they use at zero when they finish.  A grown
// buffer replaces the current one for new launches, but the old one is never
// freed: CUDA graphs captured earlier keep using it, so they stay valid.
constexpr int kMaxTiles = 1 << 16;
constexpr size_t kCounterBytes = size_t{kMaxTiles} * sizeof(unsigned int);
struct Scratch {
  void* base = nullptr;
  size_t bytes = 0;
};
Scratch g_scratch[kMaxDevices];
std::mutex& scratch_mutex() {
  static std::mutex m;
  return m;
}
void* scratch_get(size_t bytes, cudaStream_t s) {
  const int d = current_device();
  if (d < 0) return nullptr;
  std::lock_guard<std::mutex> lock(scratch_mutex());
  Scratch& sc = g_scratch[d];
  if (sc.bytes >= bytes) return sc.base;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
    (void)cudaGetLastError();
    return nullptr;
  }
  // at least 16 MB, and at least twice the previous size, so growth is rare
  size_t want = bytes < (size_t{16} << 20) ? (size_t{16} << 20) : bytes;
  if (want < 2 * sc.bytes) want = 2 * sc.bytes;
  void* p = nullptr;
  if (cudaMalloc(&p, want) != cudaSuccess || cudaMemset(p, 0, want) != cudaSuccess) {
    (void)cudaGetLastError();
    if (p != nullptr) cudaFree(p);
    return nullptr;
  }
  sc.base = p;   // the previous buffer stays allocated (see above)
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
  size_t budget = 0;   // dynamic shared memory one CTA may use at per_sm CTAs per SM
};

// CTAs per SM the streaming kernel's launch bounds allow
template <int WC>
constexpr int stream_max_per_sm() {
  return WC == 8 ? 2 : 3;
}

// Slabs of each of ksplit K segments of a row of slabs_row slabs: all equal
// but the last, which may be shorter; 0 where that would leave the last
// segment empty.
inline int segment_slabs(int slabs_row, int ksplit) {
  const int seg = (slabs_row + ksplit - 1) / ksplit;
  return (ksplit - 1) * seg < slabs_row ? seg : 0;
}

template <int F, int NT, int RT, int WC, int XM>
Plan make_plan(int K, int ksplit, bool tma) {
  using G = Geo<F, NT, RT, WC>;
  const size_t stage = stage_shape<G>(tma).bytes;
  Plan pl;
  const int slabs_row = (K / 256 + G::kSlabSB - 1) / G::kSlabSB;
  const int seg = segment_slabs(slabs_row, ksplit);
  if (seg == 0) return pl;
  const int kpad = seg * G::kSlabK;
  const size_t xb = XM == kXQ8 ? static_cast<size_t>(q8_x_bytes(NT, kpad, G::kPart))
                               : XLayout<F, NT, XM == kXBF16>::bytes(static_cast<size_t>(NT) * kpad) +
                                     static_cast<size_t>(NT) * (kpad / G::kPart) * 4;
  pl.x_bytes = static_cast<uint32_t>((xb + 127) & ~size_t{127});
  const DevInfo* dip = dev_info();
  if (dip == nullptr) return pl;
  const DevInfo& di = *dip;
  for (int per_sm = stream_max_per_sm<WC>(); per_sm >= 1; --per_sm) {
    // dynamic shared memory of one CTA when per_sm CTAs share an SM
    size_t budget = di.smem_sm / per_sm;
    budget = budget > di.smem_reserved + kStaticSmem ? budget - di.smem_reserved - kStaticSmem : 0;
    if (budget > di.smem_optin - kStaticSmem) budget = di.smem_optin - kStaticSmem;
    if (pl.x_bytes + 2 * stage > budget) continue;
    int stages = static_cast<int>((budget - pl.x_bytes) / stage);
    if (stages > kMaxStages) stages = kMaxStages;
    pl.per_sm = per_sm;
    pl.stages = stages;
    pl.smem = pl.x_bytes + static_cast<size_t>(stages) * stage;
    pl.budget = budget;
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
constexpr size_t kNoAllocScratchBytes = size_t{4} << 20;   // 4 MiB per device

// cuTensorMapEncodeTiled, fetched from the driver once (nullptr if absent).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled() {
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      (void)cudaGetLastError();
      return nullptr;
    }
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// 2-D tensor map of one plane: `rows` rows of row_bytes (a multiple of 16)
// seen as 8-byte elements; box = box_bytes (a multiple of 16) x box_rows.
// Out-of-range elements of a box read as zero.
bool encode_plane(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows,
                  uint32_t box_bytes, uint32_t box_rows) {
  const EncodeTiledFn fn = encode_tiled();
  if (fn == nullptr || row_bytes % 16 != 0 || reinterpret_cast<uintptr_t>(base) % 16 != 0 ||
      box_bytes % 16 != 0 || box_bytes / 8 > 256 || box_rows < 1 || box_rows > 256)
    return false;
  const cuuint64_t dims[2] = {row_bytes / 8, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_bytes / 8, box_rows};
  const cuuint32_t elem[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void*>(base), dims, strides, box,
            elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor copies need every plane's row stride on the 16-byte grid (always
// for Q4_K and Q5_K; Q6_K when K / 256 is a multiple of 8; the G128 param
// plane when K / 256 is even).
template <class G>
bool tma_possible(int K) {
  const int64_t nsb = K / 256;
  if (encode_tiled() == nullptr) return false;
  if ((nsb * G::kBB) % 16 != 0 && G::kF != kG128) return false;
  if (G::kF == kG128 && (nsb * 8) % 16 != 0) return false;
  return true;
}

template <int F, int NT, int RT, int WC, int XM>
bool launch_cfg(const GemvGroup& g, const uint16_t* x, int K, int n_tok, cudaStream_t s,
                int ksplit, bool tma, ScratchSrc src = ScratchSrc::kDevice,
                StaticScratch* st = nullptr) {
  using G = Geo<F, NT, RT, WC>;
  const DevInfo* dip = dev_info();
  if (dip == nullptr) return false;
  const DevInfo& di = *dip;
  Params p;
  p.g = g;
  p.x = x;
  p.K = K;
  p.nsb = K / 256;
  const int slabs_row = (p.nsb + G::kSlabSB - 1) / G::kSlabSB;
  // the last segment may be shorter: its slabs past the row are copied as
  // zeros (tensor copies) or not at all (row copies), and the consumers skip
  // super-blocks past the row
  p.slabs = segment_slabs(slabs_row, ksplit);
  if (p.slabs == 0) return false;
  p.ksplit = ksplit;
  p.kpad = p.slabs * G::kSlabK;
  p.nt = n_tok;
  p.part = nullptr;
  p.arrivals = nullptr;
  p.tag = next_tag();
  const Plan pl = make_plan<F, NT, RT, WC, XM>(K, ksplit, tma);
  if (pl.per_sm == 0) return false;
  p.tma = tma ? 1 : 0;
  p.x_bytes = pl.x_bytes;
  int per_sm = pl.per_sm;
  {
    int occ = 0;   // registers may allow fewer CTAs than shared memory does
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, gemv_stream<F, NT, RT, WC, XM>,
                                                      G::kThreads, pl.smem) == cudaSuccess &&
        occ >= 1 && occ < per_sm)
      per_sm = occ;
    (void)cudaGetLastError();
  }
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
  // even, so that both half-warps of a warp have the same number of rows in
  // every full tile (no divergence between their row loops)
  tr += tr & 1;
  if (tr > G::kRows) tr = G::kRows;
  if (tr < 1) tr = 1;
  p.tile_rows = tr;
  p.tiles = 0;
  for (int i = 0; i < kMaxGroup; ++i) {
    if (i < g.count) p.tiles += (g.N[i] + tr - 1) / tr;
    p.tile_end[i] = p.tiles;
  }
  if (cps > p.tiles) cps = p.tiles;
  // stages hold tile_rows rows: as many as the CTA's share of shared memory
  // takes (small tiles get a deep ring and request most of their K at once)
  const StageShape ss = stage_shape<G>(tma, tr);
  p.slot = ss.slot;
  p.pslot = ss.pslot;
  p.pbase = ss.pbase;
  p.stage = ss.bytes;
  int stages = static_cast<int>((pl.budget - p.x_bytes) / ss.bytes);
  if (stages > kMaxStages) stages = kMaxStages;
  if (stages < pl.stages) stages = pl.stages;
  // fixed tiles per CTA: enough to fill the ring before the previous kernel
  // has finished (claims wait for it); every further tile is claimed
  p.static_tiles = (stages + p.slabs - 1) / p.slabs;
  if (ksplit > kMaxSegs) return false;
  const size_t smem = p.x_bytes + static_cast<size_t>(stages) * ss.bytes;
  static size_t configured[kMaxDevices] = {};   // per device: dynamic smem above 48 KB is opt-in
  if (!raise_smem_limit(gemv_stream<F, NT, RT, WC, XM>, smem, configured)) return false;
  p.tx = 0;
  if (tma) {
    for (int i = 0; i < g.count; ++i) {
      const int64_t n = g.N[i];
      bool ok;
      if constexpr (F == kG128) {
        ok = encode_plane(&p.tm[i][0], g.W[i], 128 * static_cast<uint64_t>(p.nsb), n, ss.slot, tr) &&
             encode_plane(&p.tm[i][1], g.W[i] + n * p.nsb * 128, 8 * static_cast<uint64_t>(p.nsb), n,
                          ss.pslot, tr);
      } else {
        ok = encode_plane(&p.tm[i][0], g.W[i], static_cast<uint64_t>(p.nsb) * G::kBB, n, ss.slot, tr);
      }
      if (!ok) return false;
    }
    p.tx = static_cast<uint32_t>(tr) * (ss.slot + ss.pslot);
  }
  if (ksplit > 1) {
    const size_t part_bytes =
        static_cast<size_t>(ksplit) * p.tiles * p.tile_rows * NT * sizeof(uint64_t);
    if (src == ScratchSrc::kDevice) {
      if (p.tiles > kMaxTiles) return false;
      uint8_t* base = static_cast<uint8_t*>(scratch_get(kCounterBytes + part_bytes, s));
      if (base == nullptr) return false;
      p.arrivals = reinterpret_cast<unsigned int*>(base);
      p.part = base + kCounterBytes;
    } else {
      if (p.tiles > kNoAllocMaxTiles ||
          kNoAllocCounterBytes + part_bytes > kNoAllocScratchBytes) {
        st->too_large = true;
        return false;
      }
      // the array keeps the previous call's contents: clear the counters
      // this launch uses (a stream-ordered memset, not an allocation)
      if (cudaMemsetAsync(st->base, 0, static_cast<size_t>(p.tiles) * sizeof(unsigned int), s) !=
          cudaSuccess) {
        (void)cudaGetLastError();
        return false;
      }
      p.arrivals = reinterpret_cast<unsigned int*>(st->base);
      p.part = st->base + kNoAllocCounterBytes;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(cps * ksplit));
  cfg.blockDim = dim3(G::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return launched(cudaLaunchKernelEx(&cfg, gemv_stream<F, NT, RT, WC, XM>, p, stages));
}

template <int F, int NT, int RT, int WC, bool Q8 = false>
bool launch_rt(const GemvGroup& g, const uint16_t* x, int K, int n_tok, cudaStream_t s,
               ScratchSrc src = ScratchSrc::kDevice, StaticScratch* st = nullptr) {
  using G = Geo<F, NT, RT, WC>;
  // K segments: the fewest (a power of two dividing the slabs of a row, at
  // most 16) that reach the kernel's most CTAs per SM, else the fewest that
  // reach the most CTAs per SM.  Where that leaves fewer than two (tile,
  // segment) units per CTA (few rows, and a slab count with no such divisor,
  // e.g. 31), more segments with a shorter last one.
  const int slabs_row = (K / 256 + G::kSlabSB - 1) / G::kSlabSB;
  const bool tma = tma_possible<G>(K);
  constexpr int kMaxPer = stream_max_per_sm<WC>();
  if constexpr (Q8) {
    // int8 codes: one x mode
    int best_ks = 0, best_sm = 0;
    for (int ks = 1; ks <= 16 && slabs_row % ks == 0; ks *= 2) {
      const Plan pl = make_plan<F, NT, RT, WC, kXQ8>(K, ks, tma);
      if (pl.per_sm > best_sm) {
        best_sm = pl.per_sm;
        best_ks = ks;
      }
      if (best_sm == kMaxPer) break;
    }
    if (best_ks == 0) return false;
    for (int ks = best_ks;; ks = 1) {
      const bool ok = launch_cfg<F, NT, RT, WC, kXQ8>(g, x, K, n_tok, s, ks, tma, src, st);
      if (ok || ks == 1) return ok;
    }
  } else {
    int best_ks = 0, best_sm = 0;
    bool best_bf = false;
    // fp32 x first (no conversion in the consumers); bf16 x only where it
    // admits more CTAs per SM than any fp32 plan (e.g. the LM head's per-row
    // copies, whose stages with fp32 x leave room for two CTAs only)
    for (int bf = 0; bf < 2 && best_sm < kMaxPer; ++bf) {
      for (int ks = 1; ks <= 16 && slabs_row % ks == 0; ks *= 2) {
        const Plan pl = bf ? make_plan<F, NT, RT, WC, kXBF16>(K, ks, tma)
                           : make_plan<F, NT, RT, WC, kXF32>(K, ks, tma);
        if (pl.per_sm > best_sm) {
          best_sm = pl.per_sm;
          best_ks = ks;
          best_bf = bf != 0;
        }
        if (best_sm == kMaxPer) break;
      }
    }
    if (best_ks == 0) return false;
    const DevInfo* dip = dev_info();
    int64_t tiles = 0;
    for (int i = 0; i < g.count; ++i) tiles += (g.N[i] + G::kRows - 1) / G::kRows;
    // two units per CTA of the plan?
    auto enough = [&](int ks, int per_sm) {
      return dip == nullptr || tiles * ks >= 2 * static_cast<int64_t>(per_sm) * dip->sms;
    };
    if (!enough(best_ks, best_sm)) {
      // more segments (fp32 x: bf16 x with K split ran slower, e.g. 5120 x
      // 31744 Q6_K 73.7 against 41.7 us), taken while they keep at least as
      // many CTAs per SM
      for (int ks = 2 * best_ks; ks <= 16; ks *= 2) {
        if (segment_slabs(slabs_row, ks) == 0) break;
        const Plan pl = make_plan<F, NT, RT, WC, kXF32>(K, ks, tma);
        if (pl.per_sm > 0 && pl.per_sm >= best_sm) {
          best_sm = pl.per_sm;
          best_ks = ks;
          best_bf = false;
        }
        if (best_sm == kMaxPer && enough(best_ks, best_sm)) break;
      }
    }
    for (int ks = best_ks;; ks = 1) {
      const bool ok = best_bf ? launch_cfg<F, NT, RT, WC, kXBF16>(g, x, K, n_tok, s, ks, tma, src, st)
                              : launch_cfg<F, NT, RT, WC, kXF32>(g, x, K, n_tok, s, ks, tma, src, st);
      if (ok || ks == 1) return ok;   // no scratch (e.g. during capture, or beyond the fixed array): unsplit
      best_bf = static_cast<size_t>(NT) * K * 4 > 96 * 1024;
    }
  }
}

template <int F, int NT, bool Q8 = false>
bool launch_nt(const GemvGroup& g, const uint16_t* x, int K, int n_tok, cudaStream_t s,
               ScratchSrc src = ScratchSrc::kDevice, StaticScratch* st = nullptr) {
  const DevInfo* dip = dev_info();
  if (dip == nullptr) return false;
  const DevInfo& di = *dip;
  // Small matrices (fewer than 16 rows per SM) and n_tok 4 (whose x values
  // take twice the registers): 4 consumer warps x 2 rows per thread.  Large
  // matrices at n_tok 1, 2: 4 rows per thread, with 8 consumer warps for the
  // Q4 family (two CTAs per SM: more warps to hide latency) and 4 for Q6_K
  // (three CTAs per SM; measured faster than eight warps for its records).
  int64_t rows = 0;
  for (int i = 0; i < g.count; ++i) rows += g.N[i];
  if (NT == 4 || rows < 16LL * di.sms) return launch_rt<F, NT, 2, 4, Q8>(g, x, K, n_tok, s, src, st);
  if constexpr (NT == 4)
    return false;
  else if constexpr (F == kQ6K)
    return launch_rt<F, NT, 4, 4, Q8>(g, x, K, n_tok, s, src, st);
  else
    return launch_rt<F, NT, 4, 8, Q8>(g, x, K, n_tok, s, src, st);
}

// The verify kernel: tiles of 16 WC rows, slabs of two super-blocks; shared
// memory holds the per-warp scale tables, the CTA's K segment of x (bf16,
// 8 or 16 token rows) and the weight ring.  K segments: among the divisors
// of the slabs of a row (at most 16) whose x segment fits with two stages,
// the fewest that give every resident CTA work.
template <int F, int NB, int WC>
bool launch_mma(const GemvGroup& g, const uint16_t* x, int K, int n_tok, cudaStream_t s,
                ScratchSrc src = ScratchSrc::kDevice, StaticScratch* st = nullptr) {
  constexpr int NTP = 8 * NB;
  using G = MGeo<F, WC>;
  const DevInfo* dip = dev_info();
  if (dip == nullptr) return false;
  const DevInfo& di = *dip;
  const bool tma = tma_possible<G>(K);
  const StageShape full = stage_shape<G>(tma);
  Params p;
  p.g = g;
  p.x = x;
  p.K = K;
  p.nsb = K / 256;
  p.nt = n_tok;
  p.part = nullptr;
  p.arrivals = nullptr;
  p.tag = 0;
  p.tma = tma ? 1 : 0;
  p.static_tiles = 0;   // the verify kernel keeps its fixed tile order
  p.slot = full.slot;
  p.pslot = full.pslot;
  p.pbase = full.pbase;
  p.stage = full.bytes;
  int64_t rows = 0;
  for (int i = 0; i < g.count; ++i) rows += g.N[i];
  const int slabs_row = (p.nsb + G::kSlabSB - 1) / G::kSlabSB;
  auto x_bytes_of = [&](int ks) {
    const size_t seg = static_cast<size_t>(slabs_row / ks) * G::kSlabK;
    return (static_cast<size_t>(WC) * G::kTabBytes + NTP * (seg * 2 + G::kXPad) + 127) / 128 * 128;
  };
  // (CTAs per SM, fitting K-segment counts): two CTAs per SM if anything fits
  int per_sm = 0;
  size_t budget = 0;
  int fits[16];
  int nfit = 0;
  for (int ps = 2; ps >= 1 && per_sm == 0; --ps) {
    budget = di.smem_sm / ps;
    budget = budget > di.smem_reserved + kStaticSmem ? budget - di.smem_reserved - kStaticSmem : 0;
    if (budget > di.smem_optin - kStaticSmem) budget = di.smem_optin - kStaticSmem;
    nfit = 0;
    for (int ks = 1; ks <= 16 && ks <= slabs_row; ++ks)
      if (slabs_row % ks == 0 && x_bytes_of(ks) + 2 * static_cast<size_t>(full.bytes) <= budget)
        fits[nfit++] = ks;
    if (nfit > 0) per_sm = ps;
  }
  if (per_sm == 0) return false;
  {
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &occ, gemv_mma<F, NB, WC>, G::kThreads,
            x_bytes_of(fits[0]) + 2 * static_cast<size_t>(full.bytes)) == cudaSuccess &&
        occ >= 1 && occ < per_sm)
      per_sm = occ;
    (void)cudaGetLastError();
  }
  const int64_t resident = static_cast<int64_t>(per_sm) * di.sms;
  const int64_t full_tiles = (rows + G::kRows - 1) / G::kRows;
  int pick_i = nfit - 1;
  for (int i = 0; i < nfit; ++i)
    if (full_tiles * fits[i] >= resident) {
      pick_i = i;
      break;
    }
  for (;; --pick_i) {
    if (pick_i < 0) return false;
    const int ksplit = fits[pick_i];
    p.ksplit = ksplit;
    p.slabs = slabs_row / ksplit;
    p.kpad = p.slabs * G::kSlabK;
    p.x_bytes = static_cast<uint32_t>(x_bytes_of(ksplit));
    int cps = static_cast<int>(resident / ksplit);
    if (cps < 1) cps = 1;
    // balanced tiles of whole 16-row warp blocks
    const int64_t k = (rows + static_cast<int64_t>(cps) * G::kRows - 1) /
                      (static_cast<int64_t>(cps) * G::kRows);
    int tr = static_cast<int>((rows + cps * k - 1) / (cps * k));
    tr = (tr + 15) / 16 * 16;
    if (tr > G::kRows) tr = G::kRows;
    p.tile_rows = tr;
    p.tiles = 0;
    for (int i = 0; i < kMaxGroup; ++i) {
      if (i < g.count) p.tiles += (g.N[i] + tr - 1) / tr;
      p.tile_end[i] = p.tiles;
    }
    if (cps > p.tiles) cps = p.tiles;
    int stages = static_cast<int>((budget - p.x_bytes) / full.bytes);
    if (stages > kMaxStages) stages = kMaxStages;
    const size_t smem = p.x_bytes + static_cast<size_t>(stages) * full.bytes;
    static size_t configured[kMaxDevices] = {};   // per device: dynamic smem above 48 KB is opt-in
    if (!raise_smem_limit(gemv_mma<F, NB, WC>, smem, configured)) return false;
    if (ksplit > 1) {
      const size_t part_bytes =
          static_cast<size_t>(ksplit) * p.tiles * p.tile_rows * NTP * sizeof(float);
      if (src == ScratchSrc::kDevice) {
        uint8_t* base = p.tiles <= kMaxTiles
                            ? static_cast<uint8_t*>(scratch_get(kCounterBytes + part_bytes, s))
                            : nullptr;
        if (base == nullptr) continue;   // no scratch (e.g. during capture): fewer segments
        p.arrivals = reinterpret_cast<unsigned int*>(base);
        p.part = base + kCounterBytes;
      } else {
        if (p.tiles > kNoAllocMaxTiles ||
            kNoAllocCounterBytes + part_bytes > kNoAllocScratchBytes) {
          st->too_large = true;   // beyond the fixed array: fewer segments
          continue;
        }
        if (cudaMemsetAsync(st->base, 0, static_cast<size_t>(p.tiles) * sizeof(unsigned int), s) !=
            cudaSuccess) {
          (void)cudaGetLastError();
          return false;
        }
        p.arrivals = reinterpret_cast<unsigned int*>(st->base);
        p.part = st->base + kNoAllocCounterBytes;
      }
    }
    p.tx = 0;
    if (tma) {
      for (int i = 0; i < g.count; ++i) {
        const int64_t n = g.N[i];
        bool enc;
        if constexpr (F == kG128) {
          enc = encode_plane(&p.tm[i][0], g.W[i], 128 * static_cast<uint64_t>(p.nsb), n, full.slot, tr) &&
                encode_plane(&p.tm[i][1], g.W[i] + n * p.nsb * 128, 8 * static_cast<uint64_t>(p.nsb),
                             n, full.pslot, tr);
        } else {
          enc = encode_plane(&p.tm[i][0], g.W[i], static_cast<uint64_t>(p.nsb) * G::kBB, n, full.slot, tr);
        }
        if (!enc) return false;
      }
      p.tx = static_cast<uint32_t>(tr) * (full.slot + full.pslot);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(cps * ksplit));
    cfg.blockDim = dim3(G::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return launched(cudaLaunchKernelEx(&cfg, gemv_mma<F, NB, WC>, p, stages));
  }
}

// Consumer warps per CTA: 8 (one CTA per SM) for launches of 64 M weights
// or more whose rows take 2-D tensor copies; 4 (two CTAs per SM, 64-row
// tiles) for smaller ones such as the attention projections, where more,
// smaller tiles fill the GPU better, and for rows off the 16-byte grid (the
// LM head), where two producer warps per SM issue the per-row copies.
template <int F>
bool launch_verify(const GemvGroup& g, const uint16_t* x, int K, int n_tok, cudaStream_t s,
                   ScratchSrc src = ScratchSrc::kDevice, StaticScratch* st = nullptr) {
  int64_t rows = 0;
  for (int i = 0; i < g.count; ++i) rows += g.N[i];
  const bool small = rows * K < (int64_t{64} << 20) || !tma_possible<MGeo<F, 8>>(K);
  if (n_tok <= 8)
    return small ? launch_mma<F, 1, 4>(g, x, K, n_tok, s, src, st)
                 : launch_mma<F, 1, 8>(g, x, K, n_tok, s, src, st);
  return small ? launch_mma<F, 2, 4>(g, x, K, n_tok, s, src, st)
               : launch_mma<F, 2, 8>(g, x, K, n_tok, s, src, st);
}

// The single-token tensor-core kernel: one CTA per SM, 64-row tiles over all
// of K (no split-K), x of the whole row staged once per CTA.  Rows whose
// stride is off the 16-byte grid (no tensor copies), or rows too long for x
// and two stages to fit in shared memory, stay on gemv_stream.
// h != nullptr: SwiGLU mode (g = {gate, up} of one shape; tiles of 32
// features; h = bf16(silu(gate) * up) written beside y).
template <int F, int SB>
bool launch_tc1_sb(const GemvGroup& g, const uint16_t* x, int K, cudaStream_t s, uint16_t* h) {
  using G = TGeo1<F, SB>;
  const bool swiglu = h != nullptr;
  if (swiglu && (g.count != 2 || g.N[0] != g.N[1])) return false;
  const DevInfo* dip = dev_info();
  if (dip == nullptr) return false;
  const DevInfo& di = *dip;
  if (!tma_possible<G>(K)) return false;
  Params p;
  p.g = g;
  p.x = x;
  p.K = K;
  p.nsb = K / 256;
  p.nt = 1;
  p.part = nullptr;
  p.arrivals = nullptr;
  p.tag = 0;
  p.tma = 1;
  p.ksplit = 1;
  p.slabs = (p.nsb + G::kSlabSB - 1) / G::kSlabSB;
  p.kpad = p.slabs * G::kSlabK;
  const StageShape ss = stage_shape<G>(true);
  p.slot = ss.slot;
  p.pslot = ss.pslot;
  p.pbase = ss.pbase;
  p.stage = ss.bytes;
  p.tile_rows = G::kRows;
  p.swiglu = swiglu ? 1 : 0;
  p.h = h;
  p.tiles = 0;
  for (int i = 0; i < kMaxGroup; ++i) {
    if (swiglu)
      p.tiles = (g.N[0] + G::kRows / 2 - 1) / (G::kRows / 2);   // one tile holds both matrices' rows
    else if (i < g.count)
      p.tiles += (g.N[i] + G::kRows - 1) / G::kRows;
    p.tile_end[i] = p.tiles;
  }
  // the kernel's static shared memory (its barriers) comes out of the same budget
  static const size_t static_smem = [] {
    cudaFuncAttributes fa{};
    if (cudaFuncGetAttributes(&fa, gemv_tc1<F, SB>) != cudaSuccess) {
      (void)cudaGetLastError();
      return size_t{1024};
    }
    return fa.sharedSizeBytes;
  }();
  size_t budget = di.smem_sm > di.smem_reserved + static_smem
                      ? di.smem_sm - di.smem_reserved - static_smem
                      : 0;
  if (budget > di.smem_optin - static_smem) budget = di.smem_optin - static_smem;
  p.x_bytes = (tc_x_only(p.kpad, G::kSub) + G::kCombBytes + 127u) & ~127u;
  if (p.x_bytes + 2 * static_cast<size_t>(ss.bytes) > budget) return false;
  int stages = static_cast<int>((budget - p.x_bytes) / ss.bytes);
  if (stages > kMaxStages) stages = kMaxStages;
  int cps = di.sms < p.tiles ? di.sms : p.tiles;
  if (cps < 1) cps = 1;
  p.static_tiles = (stages + p.slabs - 1) / p.slabs;
  const size_t smem = p.x_bytes + static_cast<size_t>(stages) * ss.bytes;
  static size_t configured[kMaxDevices] = {};   // per device: dynamic smem above 48 KB is opt-in
  if (!raise_smem_limit(gemv_tc1<F, SB>, smem, configured)) return false;
  const uint32_t box_rows = swiglu ? G::kRows / 2 : G::kRows;
  for (int i = 0; i < g.count; ++i) {
    const int64_t n = g.N[i];
    bool ok;
    if constexpr (F == kG128) {
      ok = encode_plane(&p.tm[i][0], g.W[i], 128 * static_cast<uint64_t>(p.nsb), n, ss.slot,
                        box_rows) &&
           encode_plane(&p.tm[i][1], g.W[i] + n * p.nsb * 128, 8 * static_cast<uint64_t>(p.nsb), n,
                        ss.pslot, box_rows);
    } else {
      ok = encode_plane(&p.tm[i][0], g.W[i], static_cast<uint64_t>(p.nsb) * G::kBB, n, ss.slot,
                        box_rows);
    }
    if (!ok) return false;
  }
  p.tx = static_cast<uint32_t>(G::kRows) * (ss.slot + ss.pslot);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(cps));
  cfg.blockDim = dim3(G::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return launched(cudaLaunchKernelEx(&cfg, gemv_tc1<F, SB>, p, stages));
}
// Five super-block columns (20 consumer warps: more warps to hide the
// product's latencies) where K / 256 divides by 5, so that no stage is left
// partly empty; else four (16 warps).
template <int F>
bool launch_tc1(const GemvGroup& g, const uint16_t* x, int K, cudaStream_t s,
                uint16_t* h = nullptr) {
  return (K / 256) % 5 == 0 ? launch_tc1_sb<F, 5>(g, x, K, s, h) : launch_tc1_sb<F, 4>(g, x, K, s, h);
}

// The multi-token tensor-core kernel (n_tok 5..16, NB = 1 or 2 blocks of
// eight tokens).  K segments: the fewest whose x fits with two ring stages.
template <int F, int WC, int NB>
bool launch_tcv(const GemvGroup& g, const uint16_t* x, int K, int n_tok, cudaStream_t s,
                ScratchSrc src = ScratchSrc::kDevice, StaticScratch* st = nullptr) {
  using G = TGeo<F, WC, kTcvRT>;
  constexpr int NTP = 8 * NB;
  const DevInfo* dip = dev_info();
  if (dip == nullptr) return false;
  const DevInfo& di = *dip;
  const bool tma = tma_possible<G>(K);
  if (!tma) return false;
  Params p;
  p.g = g;
  p.x = x;
  p.K = K;
  p.nsb = K / 256;
  p.nt = n_tok;
  p.part = nullptr;
  p.arrivals = nullptr;
  p.tag = 0;
  p.tma = 1;
  const int slabs_row = (p.nsb + G::kSlabSB - 1) / G::kSlabSB;
  const StageShape ss = stage_shape<G>(true);
  p.slot = ss.slot;
  p.pslot = ss.pslot;
  p.pbase = ss.pbase;
  p.stage = ss.bytes;
  p.tile_rows = G::kRows;
  p.tiles = 0;
  for (int i = 0; i < kMaxGroup; ++i) {
    if (i < g.count) p.tiles += (g.N[i] + G::kRows - 1) / G::kRows;
    p.tile_end[i] = p.tiles;
  }
  const int per_sm = WC <= 4 ? 2 : 1;   // CTAs per SM (the launch bounds' minimum)
  size_t budget = di.smem_sm / per_sm > di.smem_reserved + kStaticSmem
                      ? di.smem_sm / per_sm - di.smem_reserved - kStaticSmem
                      : 0;
  if (budget > di.smem_optin - kStaticSmem) budget = di.smem_optin - kStaticSmem;
  auto xb = [&](int kpad) { return static_cast<size_t>(tcv_x_bytes(kpad, NB, WC, G::kRows)); };
  // the fewest K segments whose x fits: a split-K hand-over carries 8 NB
  // values per row, which costs more than the coarser tile balance
  int ksplit = 0;
  for (int ks = 1; ks <= kMaxSegs && ks <= slabs_row; ++ks) {
    if (slabs_row % ks != 0) continue;
    if (xb(slabs_row / ks * G::kSlabK) + 2 * ss.bytes > budget) continue;
    ksplit = ks;
    break;
  }
  if (ksplit == 0) return false;
  for (;; ksplit = 1) {
    p.ksplit = ksplit;
    p.slabs = slabs_row / ksplit;
    p.kpad = p.slabs * G::kSlabK;
    p.x_bytes = static_cast<uint32_t>(xb(p.kpad));
    if (p.x_bytes + 2 * ss.bytes > budget) return false;
    if (ksplit == 1) break;
    const size_t part_bytes =
        static_cast<size_t>(ksplit) * p.tiles * p.tile_rows * NTP * sizeof(float);
    if (src == ScratchSrc::kDevice) {
      if (p.tiles > kMaxTiles) continue;
      uint8_t* base = static_cast<uint8_t*>(scratch_get(kCounterBytes + part_bytes, s));
      if (base == nullptr) continue;   // no scratch (e.g. during capture): unsplit
      p.arrivals = reinterpret_cast<unsigned int*>(base);
      p.part = base + kCounterBytes;
    } else {
      if (p.tiles > kNoAllocMaxTiles ||
          kNoAllocCounterBytes + part_bytes > kNoAllocScratchBytes) {
        st->too_large = true;   // beyond the fixed array: unsplit
        continue;
      }
      if (cudaMemsetAsync(st->base, 0, static_cast<size_t>(p.tiles) * sizeof(unsigned int), s) !=
          cudaSuccess) {
        (void)cudaGetLastError();
        return false;
      }
      p.arrivals = reinterpret_cast<unsigned int*>(st->base);
      p.part = st->base + kNoAllocCounterBytes;
    }
    break;
  }
  int stages = static_cast<int>((budget - p.x_bytes) / ss.bytes);
  if (stages > kMaxStages) stages = kMaxStages;
  int cps = per_sm * di.sms / p.ksplit;
  if (cps > p.tiles) cps = p.tiles;
  if (cps < 1) cps = 1;
  p.static_tiles = (stages + p.slabs - 1) / p.slabs;
  const size_t smem = p.x_bytes + static_cast<size_t>(stages) * ss.bytes;
  static size_t configured[kMaxDevices] = {};   // per device: dynamic smem above 48 KB is opt-in
  if (!raise_smem_limit(gemv_tcv<F, WC, NB>, smem, configured)) return false;
  for (int i = 0; i < g.count; ++i) {
    const int64_t n = g.N[i];
    bool ok;
    if constexpr (F == kG128) {
      ok = encode_plane(&p.tm[i][0], g.W[i], 128 * static_cast<uint64_t>(p.nsb), n, ss.slot,
                        G::kRows) &&
           encode_plane(&p.tm[i][1], g.W[i] + n * p.nsb * 128, 8 * static_cast<uint64_t>(p.nsb), n,
                        ss.pslot, G::kRows);
    } else {
      ok = encode_plane(&p.tm[i][0], g.W[i], static_cast<uint64_t>(p.nsb) * G::kBB, n, ss.slot,
                        G::kRows);
    }
    if (!ok) return false;
  }
  p.tx = static_cast<uint32_t>(G::kRows) * (ss.slot + ss.pslot);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(cps * p.ksplit));
  cfg.blockDim = dim3(G::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return launched(cudaLaunchKernelEx(&cfg, gemv_tcv<F, WC, NB>, p, stages));
}

// The slices' tensor maps (Q4_K, Q5_K): a box of 16 rows x pitch bytes, which
// must not be wider than a row.  Leaves p.tma = 0 (row copies) otherwise.
template <int F>
void small_maps(SmallParams& p, const GemvGroup& g) {
  p.tma = 0;
  if (F != kQ4K && F != kQ5K) return;
  const uint64_t row = static_cast<uint64_t>(p.nsb) * block_bytes(F);
  if (p.pitch > row) return;
  for (int i = 0; i < g.count; ++i)
    if (!encode_plane(&p.tm[i], g.W[i], row, static_cast<uint64_t>(g.N[i]), p.pitch, 16)) return;
  p.tma = 1;
}

// The small-launch kernel: one wave, each CTA owning whole 16-row tiles
// (at most kSmallMaxTiles), each warp one (tile, K slice); the slices are
// as fine as small_max_warps<F>() warps per CTA allow.  Declines launches whose tiles do not
// fit one CTA per SM in shared memory.
constexpr int kSmallMaxTiles = 4;

template <int F>
bool launch_small(const GemvGroup& g, const uint16_t* x, int K, cudaStream_t s) {
  const DevInfo* dip = dev_info();
  if (dip == nullptr) return false;
  const DevInfo& di = *dip;
  SmallParams p;
  p.g = g;
  p.x = x;
  p.K = K;
  p.nsb = K / 256;
  p.tiles = 0;
  for (int i = 0; i < kMaxGroup; ++i) {
    if (i < g.count) p.tiles += (g.N[i] + 15) / 16;
    p.tile_end[i] = p.tiles;
  }
  const int C = p.tiles < di.sms ? p.tiles : di.sms;
  if (C < 1) return false;
  p.max_tiles = (p.tiles + C - 1) / C;
  if (p.max_tiles > kSmallMaxTiles) return false;
  int ks = small_max_warps<F>() / p.max_tiles;
  if (ks > p.nsb) ks = p.nsb;
  p.sbs = (p.nsb + ks - 1) / ks;
  p.ks = (p.nsb + p.sbs - 1) / p.sbs;   // every slice has at least one super-block
  auto odd16 = [](uint32_t b) { b = (b + 15u) / 16u * 16u; return (b / 16u) % 2u ? b : b + 16u; };
  p.pitch = odd16(static_cast<uint32_t>(p.sbs) * (F == kG128 ? 128u : block_bytes(F)));
  p.ppitch = F == kG128 ? (static_cast<uint32_t>(p.sbs) * 8u + 16u + 15u) / 16u * 16u : 0u;
  p.warp_bytes = (16u * (p.pitch + p.ppitch) + 127u) & ~127u;
  p.x_bytes = (tc_x_only(K, 32) + 4u * static_cast<uint32_t>(p.max_tiles * p.ks * 16) + 127u) & ~127u;
  const int warps = p.max_tiles * p.ks;
  const size_t smem = p.x_bytes + static_cast<size_t>(warps) * p.warp_bytes;
  if (smem + kStaticSmem > di.smem_optin) return false;
  small_maps<F>(p, g);
  static size_t configured[kMaxDevices] = {};
  if (!raise_smem_limit(gemv_small<F>, smem, configured)) return false;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(C));
  cfg.blockDim = dim3(static_cast<unsigned>(warps * 32));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return launched(cudaLaunchKernelEx(&cfg, gemv_small<F>, p));
}

// The small-launch kernel at 2..8 tokens: the same one wave of CTAs and
// slices as launch_small (at most 16 warps per CTA), x of every token staged
// once per CTA.
template <int F>
bool launch_small_mt(const GemvGroup& g, const uint16_t* x, int K, int n_tok, cudaStream_t s) {
  const DevInfo* dip = dev_info();
  if (dip == nullptr) return false;
  const DevInfo& di = *dip;
  SmallParams p;
  p.g = g;
  p.x = x;
  p.K = K;
  p.nsb = K / 256;
  p.nt = n_tok;
  p.tiles = 0;
  for (int i = 0; i < kMaxGroup; ++i) {
    if (i < g.count) p.tiles += (g.N[i] + 15) / 16;
    p.tile_end[i] = p.tiles;
  }
  const int C = p.tiles < di.sms ? p.tiles : di.sms;
  if (C < 1) return false;
  p.max_tiles = (p.tiles + C - 1) / C;
  if (p.max_tiles > kSmallMaxTiles || p.max_tiles > kSmallMtMaxWarps) return false;
  // the most warps (the shortest slices) whose layout fits shared memory
  auto odd16 = [](uint32_t b) { b = (b + 15u) / 16u * 16u; return (b / 16u) % 2u ? b : b + 16u; };
  size_t smem = 0;
  int warps = 0;
  for (int want = kSmallMtMaxWarps / p.max_tiles; want >= 1; --want) {
    const int ks = want < p.nsb ? want : p.nsb;
    p.sbs = (p.nsb + ks - 1) / ks;
    p.ks = (p.nsb + p.sbs - 1) / p.sbs;   // every slice has at least one super-block
    p.pitch = odd16(static_cast<uint32_t>(p.sbs) * (F == kG128 ? 128u : block_bytes(F)));
    p.ppitch = F == kG128 ? (static_cast<uint32_t>(p.sbs) * 8u + 16u + 15u) / 16u * 16u : 0u;
    p.warp_bytes = (16u * (p.pitch + p.ppitch) + 127u) & ~127u;
    warps = p.max_tiles * p.ks;
    p.tab_off = tcv_tab(K, 1);
    p.red_off = p.tab_off + static_cast<uint32_t>(warps) * 8u * kTcvTabPitch;
    p.x_bytes = (p.red_off + 4u * static_cast<uint32_t>(p.max_tiles * p.ks * 16 * 8) + 127u) & ~127u;
    smem = p.x_bytes + static_cast<size_t>(warps) * p.warp_bytes;
    if (smem + kStaticSmem <= di.smem_optin) break;
    smem = 0;
  }
  if (smem == 0) return false;
  small_maps<F>(p, g);
  static size_t configured[kMaxDevices] = {};
  if (!raise_smem_limit(gemv_small_mt<F>, smem, configured)) return false;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(C));
  cfg.blockDim = dim3(static_cast<unsigned>(warps * 32));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return launched(cudaLaunchKernelEx(&cfg, gemv_small_mt<F>, p));
}

// 2..8-token launches that take it: Q4_K, Q5_K and Q4_G128 launches of
// fewer than 32 M weights (the tiles must still fit one wave).
bool small_mt_eligible(int fmt, const GemvGroup& g, int K, int n_tok) {
  if (n_tok < 2 || n_tok > 8 || (fmt != kQ4K && fmt != kQ5K && fmt != kG128)) return false;
  int64_t rows = 0;
  for (int i = 0; i < g.count; ++i) rows += g.N[i];
  return rows * K < (int64_t{1} << 25);
}

// Single-token launches that take the small-launch kernel: Q4_K, Q5_K and
// Q4_G128 launches of fewer than 32 M weights (the single-token tensor-core
// kernel takes the larger Q4 ones), as long as they fit one wave
// (launch_small).
bool small_eligible(int fmt, const GemvGroup& g, int K, int n_tok) {
  if (n_tok != 1 || (fmt != kQ4K && fmt != kQ5K && fmt != kG128)) return false;
  int64_t rows = 0;
  for (int i = 0; i < g.count; ++i) rows += g.N[i];
  return rows * K < (int64_t{1} << 25);
}

// Multi-token (n_tok 2..16) launches that take the multi-token tensor-core
// kernel: Q4_K and Q4_G128 matrices of at least 32 M weights.
bool tcv_eligible(int fmt, const GemvGroup& g, int K, int n_tok) {
  if (n_tok < 2 || n_tok > 16 || (fmt != kQ4K && fmt != kG128)) return false;
  int64_t rows = 0;
  for (int i = 0; i < g.count; ++i) rows += g.N[i];
  return rows * K >= (int64_t{1} << 25);
}

template <int F>
bool launch_tcv_fmt(const GemvGroup& g, const uint16_t* x, int K, int n_tok, cudaStream_t s,
                    ScratchSrc src = ScratchSrc::kDevice, StaticScratch* st = nullptr) {
  // up to eight tokens: two CTAs of four consumer warps per SM (each with
  // half the x, so the SM keeps twice the weight stages in flight); 9..16
  // tokens: one CTA of eight consumer warps per SM
  return n_tok <= 8 ? launch_tcv<F, 4, 1>(g, x, K, n_tok, s, src, st)
                    : launch_tcv<F, 8, 2>(g, x, K, n_tok, s, src, st);
}

// Single-token launches that take the tensor-core kernel: Q4_K and Q4_G128
// matrices of at least 32 M weights (the MLP matrices of a decoder layer)
// with 64-row tiles for at least 60% of the SMs.  The kernel does not split
// K, so a tall-skinny matrix leaves SMs idle: 5120 x 32768 Q4_K (80 tiles)
// takes 34.7 us here against 31.6 us on gemv_stream, while 6656 rows (104
// tiles) still run faster here (22.3 against 24.5 us at K = 19968).
// Q5_K and Q6_K stay on gemv_stream: assembling their 5- and 6-bit fields
// costs the A operand more integer instructions than the CUDA-core path
// spends per weight (a Q5_K gate/up on this kernel: 57.3 against 58.7 us).
bool tc1_eligible(int fmt, const GemvGroup& g, int K, int n_tok) {
  if (n_tok != 1 || (fmt != kQ4K && fmt != kG128)) return false;
  int64_t rows = 0;
  for (int i = 0; i < g.count; ++i) rows += g.N[i];
  const DevInfo* di = dev_info();
  const int64_t min_tiles = di != nullptr ? (3 * static_cast<int64_t>(di->sms) + 4) / 5 : 1;
  return rows * K >= (int64_t{1} << 25) && (rows + 63) / 64 >= min_tiles;
}

template <int F>
bool launch_tc1_fmt(const GemvGroup& g, const uint16_t* x, int K, cudaStream_t s,
                    ScratchSrc src = ScratchSrc::kDevice, StaticScratch* st = nullptr) {
  (void)src;   // no split-K: no scratch
  (void)st;
  return launch_tc1<F>(g, x, K, s);
}

}  // namespace

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
// address is looked up once per device (with that device current; thread-safe)
// and cached.  nullptr if the lookup fails or the device ordinal is out of
// range.
void* noalloc_scratch_address() {
  static void* addr[kMaxDevices] = {};
  static std::once_flag once[kMaxDevices];
  const int d = current_device();
  if (d < 0) return nullptr;
  std::call_once(once[d], [d] {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) == cudaSuccess)
      addr[d] = ptr;
    else
      (void)cudaGetLastError();
  });
  return addr[d];
}

// The narrowest width the tensor cores serve.  Their cost is set by building
// the A operand from the packed weights, once per weight whatever the token
// count, while the CUDA-core kernel spends a multiply-add per weight and
// token: from three tokens on the tensor cores win everywhere (by about 2x
// in every launch of the decode step and of the Q5_K layer).  At two tokens
// the CUDA-core kernel still wins where the integer work of building A is
// largest: Q6_K (down 56.6 against 64.5 us, the LM head 369 against 495 us)
// and Q5_K on long rows (down, K = 32768: 52.9 against 57.3 us); Q4_K,
// Q4_G128 and short Q5_K rows are faster on the tensor cores.
int tensor_core_min_tokens(int fmt, int K) {
  if (fmt == kQ6K) return 3;
  if (fmt == kQ5K && K >= 16384) return 3;
  return 2;
}
}  // namespace

// The kernel choice for one request (see kq_kernels.cuh).  `noalloc`: split-K
// partial sums go to g_noalloc_scratch, and a configuration whose sums do not
// fit there gives way to one with fewer K segments or to the next kernel.
StreamResult launch_stream(int fmt, const GemvGroup& g, const uint16_t* x, int K, int n_tok,
                           cudaStream_t s, bool noalloc) {
  if (n_tok < 1 || n_tok > 16 || fmt < kQ4K || fmt > kG128) return StreamResult::kNotServed;
  StaticScratch sst{nullptr, false};
  StaticScratch* st = nullptr;
  ScratchSrc src = ScratchSrc::kDevice;
  if (noalloc) {
    sst.base = static_cast<uint8_t*>(noalloc_scratch_address());
    if (sst.base == nullptr) return StreamResult::kFailed;
    st = &sst;
    src = ScratchSrc::kStatic;
  }
  auto done = [&](bool ok) {
    return ok ? StreamResult::kLaunched
              : (sst.too_large ? StreamResult::kTooLarge : StreamResult::kNotServed);
  };
  if (n_tok >= tensor_core_min_tokens(fmt, K)) {
    // verify widths: the multi-token tensor-core kernels
    if (tcv_eligible(fmt, g, K, n_tok)) {
      const bool ok = fmt == kQ4K ? launch_tcv_fmt<kQ4K>(g, x, K, n_tok, s, src, st)
                                  : launch_tcv_fmt<kG128>(g, x, K, n_tok, s, src, st);
      if (ok) return StreamResult::kLaunched;
    }
    if (small_mt_eligible(fmt, g, K, n_tok)) {
      // needs no scratch
      const bool ok = fmt == kQ4K   ? launch_small_mt<kQ4K>(g, x, K, n_tok, s)
                      : fmt == kQ5K ? launch_small_mt<kQ5K>(g, x, K, n_tok, s)
                                    : launch_small_mt<kG128>(g, x, K, n_tok, s);
      if (ok) return StreamResult::kLaunched;
    }
    bool ok = false;
    switch (fmt) {
      case kQ4K: ok = launch_verify<kQ4K>(g, x, K, n_tok, s, src, st); break;
      case kQ5K: ok = launch_verify<kQ5K>(g, x, K, n_tok, s, src, st); break;
      case kQ6K: ok = launch_verify<kQ6K>(g, x, K, n_tok, s, src, st); break;
      default: ok = launch_verify<kG128>(g, x, K, n_tok, s, src, st); break;
    }
    if (ok) return StreamResult::kLaunched;
  } else if (small_eligible(fmt, g, K, n_tok)) {
    // needs no scratch
    const bool ok = fmt == kQ4K   ? launch_small<kQ4K>(g, x, K, s)
                    : fmt == kQ5K ? launch_small<kQ5K>(g, x, K, s)
                                  : launch_small<kG128>(g, x, K, s);
    if (ok) return StreamResult::kLaunched;
  } else if (tc1_eligible(fmt, g, K, n_tok)) {
    const bool ok = fmt == kQ4K ? launch_tc1_fmt<kQ4K>(g, x, K, s, src, st)
                                : launch_tc1_fmt<kG128>(g, x, K, s, src, st);
    if (ok) return StreamResult::kLaunched;
  }
  // the CUDA-core streaming kernel: up to four tokens per launch; wider
  // requests run as consecutive launches of up to four tokens (x and y rows
  // of a token are contiguous, so a chunk is an offset view).  Every chunk
  // has the shape of the first or fewer tokens, so if the first is served
  // the rest are too.
  auto stream_nt = [&](const GemvGroup& gc, const uint16_t* xc, int nt) {
    const int w = nt <= 1 ? 1 : (nt <= 2 ? 2 : 4);
#define KQ_CASE(F)                                                          \
  case F:                                                                   \
    return w == 1 ? launch_nt<F, 1>(gc, xc, K, nt, s, src, st)              \
                  : w == 2 ? launch_nt<F, 2>(gc, xc, K, nt, s, src, st)     \
                           : launch_nt<F, 4>(gc, xc, K, nt, s, src, st);
    switch (fmt) {
      KQ_CASE(kQ4K)
      KQ_CASE(kQ5K)
      KQ_CASE(kQ6K)
      KQ_CASE(kG128)
    }
#undef KQ_CASE
    return false;
  };
  for (int t0 = 0; t0 < n_tok; t0 += 4) {
    const int nt = n_tok - t0 < 4 ? n_tok - t0 : 4;
    GemvGroup gc = g;
    for (int i = 0; i < g.count; ++i) gc.y[i] = g.y[i] + static_cast<int64_t>(t0) * g.N[i];
    if (!stream_nt(gc, x + static_cast<int64_t>(t0) * K, nt)) {
      // nothing launched for this chunk: the caller's fallback recomputes
      // (and overwrites) every token
      return done(false);
    }
  }
  return StreamResult::kLaunched;
}

StreamResult launch_q8(int fmt, const GemvGroup& g, const uint16_t* x, int K, int n_tok,
                       cudaStream_t s) {
  if (n_tok < 1 || n_tok > 16 || fmt < kQ4K || fmt > kG128) return StreamResult::kNotServed;
  // up to four tokens per launch (x and y rows of a token are contiguous, so
  // a chunk is an offset view)
  for (int t0 = 0; t0 < n_tok; t0 += 4) {
    const int nt = n_tok - t0 < 4 ? n_tok - t0 : 4;
    const int w = nt <= 1 ? 1 : (nt <= 2 ? 2 : 4);
    GemvGroup gc = g;
    for (int i = 0; i < g.count; ++i) gc.y[i] = g.y[i] + static_cast<int64_t>(t0) * g.N[i];
    const uint16_t* xc = x + static_cast<int64_t>(t0) * K;
    bool ok = false;
#define KQ_CASE(F)                                                              \
  case F:                                                                       \
    ok = w == 1 ? launch_nt<F, 1, true>(gc, xc, K, nt, s)                       \
                : w == 2 ? launch_nt<F, 2, true>(gc, xc, K, nt, s)              \
                         : launch_nt<F, 4, true>(gc, xc, K, nt, s);             \
    break;
    switch (fmt) {
      KQ_CASE(kQ4K)
      KQ_CASE(kQ5K)
      KQ_CASE(kQ6K)
      KQ_CASE(kG128)
    }
#undef KQ_CASE
    if (!ok) return t0 == 0 ? StreamResult::kNotServed : StreamResult::kFailed;
  }
  return StreamResult::kLaunched;
}

namespace {
// The int8 codes of the dp4a path on their own: one warp per 32-position
// block, lane i quantising position i with the kernel's own steps.
__global__ void __launch_bounds__(256) quantize_x_q8_kernel(const uint16_t* __restrict__ x,
                                                            int64_t blocks, int8_t* __restrict__ xq,
                                                            float* __restrict__ dx) {
  const int64_t b = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (b >= blocks) return;   // warp-uniform
  const float v = __uint_as_float(static_cast<uint32_t>(x[32 * b + lane]) << 16);
  float amax = fabsf(v);
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, m));
  const float d = __fdiv_rn(amax, 127.0f);
  xq[32 * b + lane] = static_cast<int8_t>(q8_code(v, d));
  if (lane == 0) dx[b] = d;
}
}  // namespace

bool launch_quantize_x_q8(const uint16_t* x, int64_t n, int8_t* xq, float* dx, cudaStream_t s) {
  const int64_t blocks = n / 32;
  quantize_x_q8_kernel<<<static_cast<unsigned>((blocks * 32 + 255) / 256), 256, 0, s>>>(x, blocks, xq, dx);
  return launched(cudaGetLastError());
}

StreamResult launch_swiglu(int fmt, const GemvGroup& g, const uint16_t* x, int K, int n_tok,
                           uint16_t* h, cudaStream_t s) {
  if (g.count != 2 || g.N[0] != g.N[1]) return StreamResult::kNotServed;
  // one token on a large Q4_K / Q4_G128 pair: fused in the single-token
  // tensor-core kernel
  if (n_tok == 1 && tc1_eligible(fmt, g, K, n_tok)) {
    const bool ok =
        fmt == kQ4K ? launch_tc1<kQ4K>(g, x, K, s, h) : launch_tc1<kG128>(g, x, K, s, h);
    if (ok) return StreamResult::kLaunched;
  }
  // otherwise: the grouped GEMV, then the activation as its own kernel
  const StreamResult r = launch_gemv(fmt, g, x, K, n_tok, s, false);
  if (r != StreamResult::kLaunched) return r;
  const int64_t n = static_cast<int64_t>(n_tok) * g.N[0];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((n + 255) / 256));
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return launched(cudaLaunchKernelEx(&cfg, swiglu_elementwise, static_cast<const float*>(g.y[0]),
                                     static_cast<const float*>(g.y[1]), h, n))
             ? StreamResult::kLaunched
             : StreamResult::kFailed;
}

namespace {
// One warp waits on a shared-memory barrier that nothing ever completes,
// with the bounded wait shortened to `limit` cycles: the wait runs out, is
// counted in g_wait_timeouts like any other, and the kernel returns.  It
// exercises the failure path of the bounded waits without a GPU fault.
__global__ void __launch_bounds__(32) wait_timeout_probe(long long limit) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_addr(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  (void)mbar_wait_warp(b, 0u, limit);
}
}  // namespace

bool launch_wait_timeout_probe(unsigned int wait_us, cudaStream_t s) {
  const long long limit = static_cast<long long>(wait_us) * 2000;   // ~2 GHz SM clock
  wait_timeout_probe<<<1, 32, 0, s>>>(limit);
  return launched(cudaGetLastError());
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
    const int d = current_device();
    if (d >= 0) {
      std::lock_guard<std::mutex> lock(scratch_mutex());
      const Scratch& sc = g_scratch[d];
      if (sc.base != nullptr && cudaMemsetAsync(sc.base, 0, sc.bytes, s) != cudaSuccess) return false;
    }
    // the fixed array of kq_gemv_noalloc clears its counters on every call
    static const unsigned int zeros[2 * kMaxSegs] = {};
    if (cudaMemcpyToSymbolAsync(g_sched, zeros, sizeof(zeros), 0, cudaMemcpyHostToDevice, s) !=
        cudaSuccess)
      return false;
  }
  return cudaStreamSynchronize(s) == cudaSuccess;
}

}  // namespace kq
