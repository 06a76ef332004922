// kq_host.cpp -- host-side parts of libkq: sizes, status strings, the
// quantiser that produces test/benchmark data, and the lossless Q4_K ->
// group-128 merge.  None of this runs on the hot path.
//
// Quantiser rules (the pages define none; this library fixes them so that
// every sub-block's grid covers its weights and |w - w^| <= d*sc/2):
//   Q4_K / Q5_K (L = 15 / 31 levels above the min), per super-block:
//     mn_j = max(0, -min w), mx_j = max w over sub-block j;
//     dmin = smallest fp16 >= max_j mn_j / 63; m_j = ceil(mn_j / dmin) <= 63;
//     r_j = (mx_j + dmin*m_j) / L; d = smallest fp16 >= max_j r_j / 63;
//     sc_j = ceil(r_j / d) <= 63; q = clamp(rne((w + dmin*m_j)/(d*sc_j)), 0, L).
//   Q4_G128: the Q4_K rule with statistics over 128-weight groups.
//   Q6_K: s_j = amax_j / 31 over 16 weights; d = smallest fp16 >= max s / 127;
//     sc_j = ceil(s_j / d) <= 127; q = clamp(rne(w/(d*sc_j)) + 32, 0, 63).
// All of it in IEEE double without contraction (built with
// -ffp-contract=off), so the result is a deterministic function of the
// input bits.
//
// Merge: the daily.dev ExecuTorch summary (answer on exporting GGUF
// checkpoints) merges adjacent sub-blocks with identical scale/min into
// groups of up to 128 when lossless; the SGLang day-0 post names a Q4_K_M
// checkpoint with 128-weight groups.
#include <cmath>
#include <cstdint>
#include <cstring>

#include "../../include/kq.h"

namespace {

constexpr int kBlockBytes[4] = {144, 176, 210, 136};

bool valid_format(int f) { return f >= 0 && f <= 3; }

// fp16 value of the smallest binary16 >= v (v finite, >= 0).  Returns false
// above 65504.  Writes the encoding to *enc.
bool fp16_ceil(double v, double* out, uint16_t* enc) {
  if (v <= 0.0) {
    *out = 0.0;
    *enc = 0;
    return true;
  }
  // Spacing of the fp16 grid around v: 2^-24 below 2^-14, else
  // 2^(floor(log2 v) - 10).
  int ex = std::ilogb(v);
  int spacing_exp = ex < -14 ? -24 : ex - 10;
  double units = std::ceil(std::ldexp(v, -spacing_exp));
  double r = std::ldexp(units, spacing_exp);
  if (r > 65504.0) return false;
  int rex = std::ilogb(r);
  if (rex < -14) {
    *enc = static_cast<uint16_t>(std::ldexp(r, 24));
  } else {
    double mant = std::ldexp(r, -rex) - 1.0;           // in [0, 1)
    *enc = static_cast<uint16_t>(((rex + 15) << 10) | static_cast<int>(std::ldexp(mant, 10)));
  }
  *out = r;
  return true;
}

void put16(uint8_t* p, uint16_t v) {
  p[0] = static_cast<uint8_t>(v);
  p[1] = static_cast<uint8_t>(v >> 8);
}

struct AsymResult {
  uint16_t d_enc, dmin_enc;
  int sc[8], m[8];
  uint8_t q[256];
};

// Asymmetric (scale, min) quantisation of 256 weights with groups of `gs`.
kq_status quant_asym(const float* w, int gs, int levels, AsymResult* res) {
  const int ng = 256 / gs;
  double lo[8], hi[8];
  double mn_max = 0.0;
  for (int g = 0; g < ng; ++g) {
    const float* p = w + g * gs;
    double a = p[0], b = p[0];
    for (int i = 1; i < gs; ++i) {
      a = std::fmin(a, static_cast<double>(p[i]));
      b = std::fmax(b, static_cast<double>(p[i]));
    }
    lo[g] = a > 0.0 ? 0.0 : -a;   // mn_g = max(0, -min)
    hi[g] = b;
    if (lo[g] > mn_max) mn_max = lo[g];
  }
  double dmin;
  if (!fp16_ceil(mn_max / 63.0, &dmin, &res->dmin_enc)) return KQ_ERR_RANGE;
  double reach[8];
  double reach_max = 0.0;
  for (int g = 0; g < ng; ++g) {
    int mg = 0;
    if (dmin > 0.0) mg = static_cast<int>(std::fmin(std::ceil(lo[g] / dmin), 63.0));
    res->m[g] = mg;
    reach[g] = (hi[g] + dmin * mg) / levels;
    if (reach[g] > reach_max) reach_max = reach[g];
  }
  double d;
  if (!fp16_ceil(reach_max / 63.0, &d, &res->d_enc)) return KQ_ERR_RANGE;
  for (int g = 0; g < ng; ++g) {
    int s = 0;
    if (d > 0.0) s = static_cast<int>(std::fmax(0.0, std::fmin(std::ceil(reach[g] / d), 63.0)));
    res->sc[g] = s;
    const double step = d * s;
    const double offset = dmin * res->m[g];
    for (int i = 0; i < gs; ++i) {
      int q = 0;
      if (step > 0.0) {
        double t = std::nearbyint((static_cast<double>(w[g * gs + i]) + offset) / step);
        q = static_cast<int>(std::fmax(0.0, std::fmin(t, static_cast<double>(levels))));
      }
      res->q[g * gs + i] = static_cast<uint8_t>(q);
    }
  }
  return KQ_OK;
}

// 12-byte field: sub-block j < 4 -> low 6 bits of byte j (sc) and byte j+4
// (m); j >= 4 -> low nibbles in byte j+4 (sc low, m high nibble) and the top
// two bits in bits 6..7 of byte j-4 (sc) and byte j (m).
void pack_scale_field(const int* sc, const int* m, uint8_t* f) {
  for (int j = 0; j < 4; ++j) {
    f[j] = static_cast<uint8_t>((sc[j] & 63) | ((sc[j + 4] >> 4) << 6));
    f[j + 4] = static_cast<uint8_t>((m[j] & 63) | ((m[j + 4] >> 4) << 6));
    f[j + 8] = static_cast<uint8_t>((sc[j + 4] & 15) | ((m[j + 4] & 15) << 4));
  }
}

// 128 bytes: byte 32c + r holds weight 64c + r (low) and 64c + 32 + r (high).
void pack_q4(const uint8_t* q, uint8_t* qs) {
  for (int i = 0; i < 128; ++i) {
    const int c = i >> 5, r = i & 31;
    qs[i] = static_cast<uint8_t>((q[64 * c + r] & 15) | ((q[64 * c + 32 + r] & 15) << 4));
  }
}

kq_status quant_q4k(const float* w, uint8_t* out) {
  AsymResult a;
  kq_status st = quant_asym(w, 32, 15, &a);
  if (st != KQ_OK) return st;
  put16(out, a.d_enc);
  put16(out + 2, a.dmin_enc);
  pack_scale_field(a.sc, a.m, out + 4);
  pack_q4(a.q, out + 16);
  return KQ_OK;
}

kq_status quant_q5k(const float* w, uint8_t* out) {
  AsymResult a;
  kq_status st = quant_asym(w, 32, 31, &a);
  if (st != KQ_OK) return st;
  put16(out, a.d_enc);
  put16(out + 2, a.dmin_enc);
  pack_scale_field(a.sc, a.m, out + 4);
  uint8_t* qh = out + 16;
  for (int l = 0; l < 32; ++l) {
    uint8_t bits = 0;
    for (int k = 0; k < 8; ++k)   // bit k <- fifth bit of weight 64(k/2) + 32(k%2) + l
      bits |= static_cast<uint8_t>(((a.q[64 * (k >> 1) + 32 * (k & 1) + l] >> 4) & 1) << k);
    qh[l] = bits;
  }
  pack_q4(a.q, out + 48);
  return KQ_OK;
}

kq_status quant_q6k(const float* w, uint8_t* out) {
  double s[16];
  double s_max = 0.0;
  for (int j = 0; j < 16; ++j) {
    double amax = 0.0;
    for (int i = 0; i < 16; ++i) amax = std::fmax(amax, std::fabs(static_cast<double>(w[16 * j + i])));
    s[j] = amax / 31.0;
    if (s[j] > s_max) s_max = s[j];
  }
  double d;
  uint16_t d_enc;
  if (!fp16_ceil(s_max / 127.0, &d, &d_enc)) return KQ_ERR_RANGE;
  uint8_t q[256];
  int8_t sc[16];
  for (int j = 0; j < 16; ++j) {
    int v = 0;
    if (d > 0.0) v = static_cast<int>(std::fmin(std::ceil(s[j] / d), 127.0));
    sc[j] = static_cast<int8_t>(v);
    const double step = d * v;
    for (int i = 0; i < 16; ++i) {
      int qi = 0;
      if (step > 0.0) {
        double t = std::nearbyint(static_cast<double>(w[16 * j + i]) / step) + 32.0;
        qi = static_cast<int>(std::fmax(0.0, std::fmin(t, 63.0)));
      }
      q[16 * j + i] = static_cast<uint8_t>(qi);
    }
  }
  // ql byte 64h + 32a + l: low nibble = weight 128h + 32a + l, high nibble =
  // weight 128h + 64 + 32a + l.  qh byte 32h + l: bits 2t..2t+1 = top bits of
  // weight 128h + 32t + l.
  for (int h = 0; h < 2; ++h) {
    for (int a = 0; a < 2; ++a)
      for (int l = 0; l < 32; ++l) {
        const int base = 128 * h + 32 * a + l;
        out[64 * h + 32 * a + l] = static_cast<uint8_t>((q[base] & 15) | ((q[base + 64] & 15) << 4));
      }
    for (int l = 0; l < 32; ++l) {
      uint8_t v = 0;
      for (int t = 0; t < 4; ++t) v |= static_cast<uint8_t>((q[128 * h + 32 * t + l] >> 4) << (2 * t));
      out[128 + 32 * h + l] = v;
    }
  }
  std::memcpy(out + 192, sc, 16);
  put16(out + 208, d_enc);
  return KQ_OK;
}

// Decode (sc_j, m_j) from the 12-byte field.
void unpack_scale(const uint8_t* f, int j, int* sc, int* m) {
  if (j < 4) {
    *sc = f[j] & 63;
    *m = f[j + 4] & 63;
  } else {
    *sc = (f[j + 4] & 15) | ((f[j - 4] >> 6) << 4);
    *m = (f[j + 4] >> 4) | ((f[j] >> 6) << 4);
  }
}

}  // namespace

extern "C" {

size_t kq_block_bytes(kq_format f) {
  return valid_format(f) ? static_cast<size_t>(kBlockBytes[f]) : 0;
}

size_t kq_matrix_bytes(kq_format f, int64_t N_out, int64_t K) {
  if (!valid_format(f) || N_out <= 0 || K <= 0 || K % 256 != 0) return 0;
  return static_cast<size_t>(N_out) * static_cast<size_t>(K / 256) * kBlockBytes[f];
}

const char* kq_status_str(kq_status s) {
  switch (s) {
    case KQ_OK: return "ok";
    case KQ_ERR_ARG: return "invalid argument (null pointer, format or n_tok)";
    case KQ_ERR_SHAPE: return "invalid shape (K % 256 != 0, sizes <= 0, or mismatched K/N)";
    case KQ_ERR_ALIGN: return "device pointer not 16-byte aligned";
    case KQ_ERR_NOT_MERGEABLE: return "sub-blocks do not share (scale, min): merge to group 128 would be lossy";
    case KQ_ERR_RANGE: return "a scale exceeds the fp16 range";
    case KQ_ERR_CUDA: return "CUDA runtime or launch error";
    case KQ_ERR_UNSUPPORTED: return "unsupported request";
    case KQ_ERR_TIMEOUT: return "a kernel's bounded shared-memory wait timed out";
    case KQ_ERR_TOO_LARGE: return "request exceeds the fixed scratch of kq_gemv_noalloc";
  }
  return "unknown status";
}

kq_status kq_quantize(kq_format f, const float* W_host, int64_t N_out, int64_t K,
                      void* blocks_host) {
  if (!valid_format(f) || W_host == nullptr || blocks_host == nullptr) return KQ_ERR_ARG;
  if (N_out <= 0 || K <= 0 || K % 256 != 0) return KQ_ERR_SHAPE;
  const int64_t nsb = K / 256;
  const int64_t total = N_out * nsb;
  uint8_t* out = static_cast<uint8_t*>(blocks_host);
  for (int64_t idx = 0; idx < total; ++idx) {
    const int64_t n = idx / nsb, b = idx % nsb;
    const float* w = W_host + n * K + b * 256;
    kq_status st;
    switch (f) {
      case KQ_Q4_K: st = quant_q4k(w, out + idx * 144); break;
      case KQ_Q5_K: st = quant_q5k(w, out + idx * 176); break;
      case KQ_Q6_K: st = quant_q6k(w, out + idx * 210); break;
      default: {
        AsymResult a;
        st = quant_asym(w, 128, 15, &a);
        if (st == KQ_OK) {
          pack_q4(a.q, out + idx * 128);
          uint8_t* p = out + total * 128 + idx * 8;
          put16(p, a.d_enc);
          put16(p + 2, a.dmin_enc);
          p[4] = static_cast<uint8_t>(a.sc[0]);
          p[5] = static_cast<uint8_t>(a.sc[1]);
          p[6] = static_cast<uint8_t>(a.m[0]);
          p[7] = static_cast<uint8_t>(a.m[1]);
        }
      }
    }
    if (st != KQ_OK) return st;
  }
  return KQ_OK;
}

kq_status kq_merge_g128(const void* q4k_host, int64_t N_out, int64_t K, void* g128_host) {
  if (q4k_host == nullptr || g128_host == nullptr) return KQ_ERR_ARG;
  if (N_out <= 0 || K <= 0 || K % 256 != 0) return KQ_ERR_SHAPE;
  const int64_t total = N_out * (K / 256);
  const uint8_t* src = static_cast<const uint8_t*>(q4k_host);
  uint8_t* qplane = static_cast<uint8_t*>(g128_host);
  uint8_t* pplane = qplane + total * 128;
  for (int64_t idx = 0; idx < total; ++idx) {
    const uint8_t* blk = src + idx * 144;
    int sc[8], m[8];
    for (int j = 0; j < 8; ++j) unpack_scale(blk + 4, j, &sc[j], &m[j]);
    for (int j = 1; j < 4; ++j)
      if (sc[j] != sc[0] || m[j] != m[0] || sc[4 + j] != sc[4] || m[4 + j] != m[4])
        return KQ_ERR_NOT_MERGEABLE;
    std::memcpy(qplane + idx * 128, blk + 16, 128);
    uint8_t* p = pplane + idx * 8;
    std::memcpy(p, blk, 4);   // d, dmin
    p[4] = static_cast<uint8_t>(sc[0]);
    p[5] = static_cast<uint8_t>(sc[4]);
    p[6] = static_cast<uint8_t>(m[0]);
    p[7] = static_cast<uint8_t>(m[4]);
  }
  return KQ_OK;
}

}  // extern "C"
