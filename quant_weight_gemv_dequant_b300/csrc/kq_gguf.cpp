// kq_gguf.cpp -- host-side reader of GGUF checkpoint containers: finds the
// K-quant tensors of a file held in memory and reports where their records
// are, so that the bytes can go to the device unchanged and into kq_gemv.
//
// The pages name GGUF checkpoints as the input of the K-quant GEMV (the
// daily.dev summary, answer on exporting GGUF checkpoints; the SGLang day-0
// post, GGUF paragraph).  The container is read as the public GGUF
// description lays it out (version 2 and 3, little-endian):
//   magic "GGUF" | u32 version | u64 tensor_count | u64 kv_count
//   kv_count x (string key | u32 value_type | value)
//   tensor_count x (string name | u32 n_dims | u64 dims[n_dims] | u32 type |
//                   u64 offset)
//   padding to `alignment` | data section
// A string is u64 length + bytes (no terminator).  Value types: 0 u8, 1 i8,
// 2 u16, 3 i16, 4 u32, 5 i32, 6 f32, 7 bool (1 byte), 8 string, 9 array
// (u32 element type, u64 count, elements), 10 u64, 11 i64, 12 f64.
// `alignment` is the u32 value of the key "general.alignment" (32 when
// absent); tensor offsets are relative to the data section and multiples
// of it.  dims[0] is the length of a row (K), dims[1] the number of rows (N);
// a K-quant tensor's data are its rows one after another, each K/256
// records.  Tensor types Q4_K, Q5_K, Q6_K are 12, 13, 14; their record
// layouts are the ones written out in kq.h.
//
// Every read is checked against the buffer: a malformed or truncated file
// returns an error, never reads outside the buffer.
#include <cstdint>
#include <cstring>

#include "../../include/kq.h"

namespace {

struct Reader {
  const uint8_t* p;
  size_t size, pos;
  bool ok = true;

  bool need(uint64_t n) {
    if (!ok || n > size - pos) ok = false;
    return ok;
  }
  template <typename T>
  T get() {
    T v{};
    if (need(sizeof(T))) {
      std::memcpy(&v, p + pos, sizeof(T));
      pos += sizeof(T);
    }
    return v;
  }
  // a string: length and position; skipped
  bool str(uint64_t* len, size_t* at) {
    const uint64_t n = get<uint64_t>();
    if (!need(n)) return false;
    *len = n;
    *at = pos;
    pos += static_cast<size_t>(n);
    return true;
  }
  bool skip(uint64_t n) {
    if (!need(n)) return false;
    pos += static_cast<size_t>(n);
    return true;
  }
};

// Bytes of one scalar of a metadata value type; 0 for string / array /
// unknown.
uint64_t scalar_bytes(uint32_t t) {
  switch (t) {
    case 0: case 1: case 7: return 1;
    case 2: case 3: return 2;
    case 4: case 5: case 6: return 4;
    case 10: case 11: case 12: return 8;
    default: return 0;
  }
}

// Skip one metadata value of type t; `depth` bounds nested arrays.
bool skip_value(Reader& r, uint32_t t, int depth) {
  if (const uint64_t b = scalar_bytes(t)) return r.skip(b);
  if (t == 8) {
    uint64_t len;
    size_t at;
    return r.str(&len, &at);
  }
  if (t == 9 && depth < 4) {
    const uint32_t et = r.get<uint32_t>();
    const uint64_t n = r.get<uint64_t>();
    if (!r.ok) return false;
    if (const uint64_t b = scalar_bytes(et)) {
      if (n > (r.size - r.pos) / b) return r.ok = false;
      return r.skip(n * b);
    }
    for (uint64_t i = 0; i < n; ++i)
      if (!skip_value(r, et, depth + 1)) return false;
    return true;
  }
  return r.ok = false;
}

int format_of_ggml_type(uint32_t t) {
  switch (t) {
    case 12: return KQ_Q4_K;
    case 13: return KQ_Q5_K;
    case 14: return KQ_Q6_K;
    default: return -1;
  }
}

constexpr int kBlockBytes[3] = {144, 176, 210};

}  // namespace

extern "C" kq_status kq_gguf_index(const void* file, size_t size, kq_gguf_tensor* out,
                                   int max_tensors, int* n_tensors, uint32_t* alignment) {
  if (file == nullptr || n_tensors == nullptr || (out == nullptr && max_tensors > 0) ||
      max_tensors < 0)
    return KQ_ERR_ARG;
  Reader r{static_cast<const uint8_t*>(file), size, 0};
  if (!r.need(4) || std::memcmp(r.p, "GGUF", 4) != 0) return KQ_ERR_ARG;
  r.pos = 4;
  const uint32_t version = r.get<uint32_t>();
  if (!r.ok) return KQ_ERR_ARG;   // truncated
  if (version != 2 && version != 3) return KQ_ERR_UNSUPPORTED;
  const uint64_t nt = r.get<uint64_t>();
  const uint64_t nkv = r.get<uint64_t>();
  if (!r.ok) return KQ_ERR_ARG;
  uint32_t align = 32;
  for (uint64_t i = 0; i < nkv; ++i) {
    uint64_t klen;
    size_t kat;
    if (!r.str(&klen, &kat)) return KQ_ERR_ARG;
    const uint32_t vt = r.get<uint32_t>();
    if (!r.ok) return KQ_ERR_ARG;
    static const char kAlign[] = "general.alignment";
    if (vt == 4 && klen == sizeof(kAlign) - 1 && std::memcmp(r.p + kat, kAlign, klen) == 0) {
      align = r.get<uint32_t>();
      if (!r.ok || align == 0 || (align & (align - 1)) != 0) return KQ_ERR_ARG;
      continue;
    }
    if (!skip_value(r, vt, 0)) return KQ_ERR_ARG;
  }
  // tensor infos, first pass: check them and find where they end
  if (nt > (size - r.pos) / 24) return KQ_ERR_ARG;   // each info is at least 24 bytes
  const int want = static_cast<int>(nt < static_cast<uint64_t>(max_tensors) ? nt : max_tensors);
  const size_t info_pos = r.pos;
  for (uint64_t i = 0; i < nt; ++i) {
    uint64_t name_len;
    size_t name_at;
    if (!r.str(&name_len, &name_at)) return KQ_ERR_ARG;
    const uint32_t n_dims = r.get<uint32_t>();
    if (!r.ok || n_dims < 1 || n_dims > 4) return KQ_ERR_ARG;
    if (!r.skip(8ull * n_dims + 4 + 8)) return KQ_ERR_ARG;   // dims, type, offset
  }
  const size_t data = (r.pos + align - 1) / align * align;
  if (data > size) return KQ_ERR_ARG;
  // second pass: fill the caller's entries
  r.pos = info_pos;
  for (uint64_t i = 0; i < nt; ++i) {
    uint64_t name_len;
    size_t name_at;
    r.str(&name_len, &name_at);
    const uint32_t n_dims = r.get<uint32_t>();
    uint64_t dims[4] = {1, 1, 1, 1};
    for (uint32_t d = 0; d < n_dims; ++d) dims[d] = r.get<uint64_t>();
    const uint32_t type = r.get<uint32_t>();
    const uint64_t offset = r.get<uint64_t>();
    if (!r.ok) return KQ_ERR_ARG;
    if (offset % align != 0 || offset > size - data) return KQ_ERR_ARG;
    if (static_cast<int64_t>(i) >= want) continue;
    kq_gguf_tensor& t = out[i];
    std::memset(&t, 0, sizeof(t));
    const size_t nl = name_len < sizeof(t.name) - 1 ? static_cast<size_t>(name_len) : sizeof(t.name) - 1;
    std::memcpy(t.name, r.p + name_at, nl);
    t.ggml_type = static_cast<int32_t>(type);
    t.n_dims = static_cast<int32_t>(n_dims);
    for (int d = 0; d < 4; ++d) t.dims[d] = static_cast<int64_t>(dims[d]);
    t.data_offset = data + offset;
    t.format = format_of_ggml_type(type);
    t.bytes = 0;
    if (t.format >= 0) {
      // a 2-D (or 1-row) K-quant matrix: K = dims[0], N = product of the rest
      // (the library's limits: K <= 2^30, N < 2^31; checked factor by factor
      // so that no product overflows)
      const uint64_t K = dims[0];
      if (K == 0 || K % 256 != 0 || K > (uint64_t{1} << 30)) return KQ_ERR_SHAPE;
      uint64_t N = 1;
      for (uint32_t d = 1; d < n_dims; ++d) {
        if (dims[d] == 0 || dims[d] >= (uint64_t{1} << 31)) return KQ_ERR_SHAPE;
        N *= dims[d];
        if (N >= (uint64_t{1} << 31)) return KQ_ERR_SHAPE;
      }
      t.K = static_cast<int64_t>(K);
      t.N_out = static_cast<int64_t>(N);
      const uint64_t bytes = N * (K / 256) * kBlockBytes[t.format];
      if (bytes > size - t.data_offset) return KQ_ERR_ARG;   // truncated data
      t.bytes = bytes;
    }
  }
  *n_tensors = static_cast<int>(nt > 0x7FFFFFFF ? 0x7FFFFFFF : nt);
  if (alignment != nullptr) *alignment = align;
  return KQ_OK;
}
