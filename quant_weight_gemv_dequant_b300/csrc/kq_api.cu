// kq_api.cu -- the C ABI of libkq (declared in include/kq.h): argument
// validation, kernel selection and launches on the caller's stream.
//
// The operation (daily.dev ExecuTorch summary, answer on exporting GGUF
// checkpoints; SGLang day-0 post, GGUF paragraph): y[t][n] = sum_k w^[n][k]
// x[t][k] for K-quant weights and 1..16 bf16 activation rows.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/kq.h"
#include "kq_kernels.cuh"

namespace {

bool fmt_ok(int f) { return f >= 0 && f <= 3; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

kq_status check_matrix(int f, const void* W, int64_t N, int64_t K) {
  if (!fmt_ok(f) || W == nullptr) return KQ_ERR_ARG;
  if (N <= 0 || K <= 0 || K % 256 != 0) return KQ_ERR_SHAPE;
  if (N > (int64_t{1} << 31) - 1 || K > (int64_t{1} << 30)) return KQ_ERR_SHAPE;
  if (!aligned16(W)) return KQ_ERR_ALIGN;
  return KQ_OK;
}

kq_status check_io(const void* x, const float* y, int n_tok) {
  if (x == nullptr || y == nullptr) return KQ_ERR_ARG;
  if (n_tok < 1 || n_tok > 16) return KQ_ERR_ARG;
  if (!aligned16(x)) return KQ_ERR_ALIGN;
  if ((reinterpret_cast<uintptr_t>(y) & 3) != 0) return KQ_ERR_ALIGN;
  return KQ_OK;
}

kq_status launch_status() {
  return cudaPeekAtLastError() == cudaSuccess ? KQ_OK : KQ_ERR_CUDA;
}

kq_status status_of(kq::StreamResult r) {
  switch (r) {
    case kq::StreamResult::kLaunched: return launch_status();
    case kq::StreamResult::kTooLarge: return KQ_ERR_TOO_LARGE;
    case kq::StreamResult::kFailed: return KQ_ERR_CUDA;
    case kq::StreamResult::kNotServed: break;
  }
  return KQ_ERR_UNSUPPORTED;
}

}  // namespace

extern "C" {

kq_status kq_gemv(kq_format f, const void* W_blocks, const void* x_bf16, float* y,
                  int64_t N_out, int64_t K, int n_tok, kq_stream_t stream) {
  kq_status st = check_matrix(f, W_blocks, N_out, K);
  if (st != KQ_OK) return st;
  st = check_io(x_bf16, y, n_tok);
  if (st != KQ_OK) return st;
  kq::GemvGroup g{};
  g.count = 1;
  g.W[0] = static_cast<const uint8_t*>(W_blocks);
  g.y[0] = y;
  g.N[0] = static_cast<int>(N_out);
  return status_of(kq::launch_gemv(f, g, static_cast<const uint16_t*>(x_bf16), static_cast<int>(K),
                                   n_tok, reinterpret_cast<cudaStream_t>(stream), false));
}

kq_status kq_gemv_noalloc(kq_format f, const void* W_blocks, const void* x_bf16, float* y,
                          int64_t N_out, int64_t K, int n_tok, kq_stream_t stream) {
  kq_status st = check_matrix(f, W_blocks, N_out, K);
  if (st != KQ_OK) return st;
  st = check_io(x_bf16, y, n_tok);
  if (st != KQ_OK) return st;
  kq::GemvGroup g{};
  g.count = 1;
  g.W[0] = static_cast<const uint8_t*>(W_blocks);
  g.y[0] = y;
  g.N[0] = static_cast<int>(N_out);
  return status_of(kq::launch_gemv(f, g, static_cast<const uint16_t*>(x_bf16), static_cast<int>(K),
                                   n_tok, reinterpret_cast<cudaStream_t>(stream), true));
}

kq_status kq_gemv_multi(kq_format f, int count, const void* const* W, float* const* y,
                        const int64_t* N_out, const void* x_bf16, int64_t K, int n_tok,
                        kq_stream_t stream) {
  if (W == nullptr || y == nullptr || N_out == nullptr) return KQ_ERR_ARG;
  if (count < 1 || count > kq::kMaxGroup) return KQ_ERR_ARG;
  kq::GemvGroup g{};
  for (int i = 0; i < count; ++i) {
    kq_status st = check_matrix(f, W[i], N_out[i], K);
    if (st != KQ_OK) return st;
    st = check_io(x_bf16, y[i], n_tok);
    if (st != KQ_OK) return st;
    g.W[i] = static_cast<const uint8_t*>(W[i]);
    g.y[i] = y[i];
    g.N[i] = static_cast<int>(N_out[i]);
  }
  g.count = count;
  return status_of(kq::launch_gemv(f, g, static_cast<const uint16_t*>(x_bf16), static_cast<int>(K),
                                   n_tok, reinterpret_cast<cudaStream_t>(stream), false));
}

kq_status kq_gemv_q8(kq_format f, const void* W_blocks, const void* x_bf16, float* y,
                     int64_t N_out, int64_t K, int n_tok, kq_stream_t stream) {
  kq_status st = check_matrix(f, W_blocks, N_out, K);
  if (st != KQ_OK) return st;
  st = check_io(x_bf16, y, n_tok);
  if (st != KQ_OK) return st;
  kq::GemvGroup g{};
  g.count = 1;
  g.W[0] = static_cast<const uint8_t*>(W_blocks);
  g.y[0] = y;
  g.N[0] = static_cast<int>(N_out);
  return status_of(kq::launch_q8(f, g, static_cast<const uint16_t*>(x_bf16), static_cast<int>(K),
                                 n_tok, reinterpret_cast<cudaStream_t>(stream)));
}

kq_status kq_quantize_x_q8(const void* x_bf16, int64_t K, int n_tok, void* xq_int8, float* dx,
                           kq_stream_t stream) {
  if (x_bf16 == nullptr || xq_int8 == nullptr || dx == nullptr) return KQ_ERR_ARG;
  if (n_tok < 1 || n_tok > 16) return KQ_ERR_ARG;
  if (K <= 0 || K % 256 != 0 || K > (int64_t{1} << 30)) return KQ_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(dx) & 3) != 0 || (reinterpret_cast<uintptr_t>(x_bf16) & 1) != 0)
    return KQ_ERR_ALIGN;
  return kq::launch_quantize_x_q8(static_cast<const uint16_t*>(x_bf16), K * n_tok,
                                  static_cast<int8_t*>(xq_int8), dx,
                                  reinterpret_cast<cudaStream_t>(stream))
             ? KQ_OK
             : KQ_ERR_CUDA;
}

kq_status kq_gemv_swiglu(kq_format f, const void* W_gate, const void* W_up, const void* x_bf16,
                         float* y_gate, float* y_up, void* h_bf16, int64_t N_out, int64_t K,
                         int n_tok, kq_stream_t stream) {
  kq_status st = check_matrix(f, W_gate, N_out, K);
  if (st != KQ_OK) return st;
  st = check_matrix(f, W_up, N_out, K);
  if (st != KQ_OK) return st;
  st = check_io(x_bf16, y_gate, n_tok);
  if (st != KQ_OK) return st;
  st = check_io(x_bf16, y_up, n_tok);
  if (st != KQ_OK) return st;
  if (h_bf16 == nullptr) return KQ_ERR_ARG;
  if (!aligned16(h_bf16)) return KQ_ERR_ALIGN;
  kq::GemvGroup g{};
  g.count = 2;
  g.W[0] = static_cast<const uint8_t*>(W_gate);
  g.W[1] = static_cast<const uint8_t*>(W_up);
  g.y[0] = y_gate;
  g.y[1] = y_up;
  g.N[0] = g.N[1] = static_cast<int>(N_out);
  return status_of(kq::launch_swiglu(f, g, static_cast<const uint16_t*>(x_bf16), static_cast<int>(K),
                                     n_tok, static_cast<uint16_t*>(h_bf16),
                                     reinterpret_cast<cudaStream_t>(stream)));
}

kq_status kq_ffn_swiglu(const kq_matrix* gate, const kq_matrix* up, const kq_matrix* down,
                        const void* x_ffn, float* y_gate, float* y_up, void* h_bf16,
                        float* y_down, int n_tok, kq_stream_t stream) {
  if (gate == nullptr || up == nullptr || down == nullptr) return KQ_ERR_ARG;
  if (gate->format != up->format || gate->N_out != up->N_out || gate->K != up->K ||
      down->K != gate->N_out)
    return KQ_ERR_SHAPE;
  kq_status st = check_matrix(down->format, down->W, down->N_out, down->K);
  if (st != KQ_OK) return st;
  st = check_io(h_bf16, y_down, n_tok);
  if (st != KQ_OK) return st;
  st = kq_gemv_swiglu(gate->format, gate->W, up->W, x_ffn, y_gate, y_up, h_bf16, gate->N_out,
                      gate->K, n_tok, stream);
  if (st != KQ_OK) return st;
  return kq_gemv(down->format, down->W, h_bf16, y_down, down->N_out, down->K, n_tok, stream);
}

kq_status kq_layer_step(const kq_layer* L, const kq_layer_io* io, int n_tok, kq_stream_t stream) {
  if (L == nullptr || io == nullptr) return KQ_ERR_ARG;
  const kq_matrix* mats[7] = {&L->q, &L->k, &L->v, &L->o, &L->gate, &L->up, &L->down};
  float* ys[7] = {io->y_q, io->y_k, io->y_v, io->y_o, io->y_gate, io->y_up, io->y_down};
  const void* xs[7] = {io->x_attn, io->x_attn, io->x_attn, io->x_o, io->x_ffn, io->x_ffn, io->x_down};
  for (int i = 0; i < 7; ++i) {
    kq_status st = check_matrix(mats[i]->format, mats[i]->W, mats[i]->N_out, mats[i]->K);
    if (st != KQ_OK) return st;
    st = check_io(xs[i], ys[i], n_tok);
    if (st != KQ_OK) return st;
  }
  if (L->k.K != L->q.K || L->v.K != L->q.K || L->up.K != L->gate.K ||
      L->up.N_out != L->gate.N_out)
    return KQ_ERR_SHAPE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // Launch groups: {q, k, v} on x_attn, {o}, {gate, up} on x_ffn, {down}.
  // Matrices of one group share a launch when they share the format.
  const int groups[4][3] = {{0, 1, 2}, {3, -1, -1}, {4, 5, -1}, {6, -1, -1}};
  for (int gi = 0; gi < 4; ++gi) {
    int pending[3], np = 0;
    for (int j = 0; j < 3; ++j)
      if (groups[gi][j] >= 0) pending[np++] = groups[gi][j];
    bool done[3] = {false, false, false};
    for (int a = 0; a < np; ++a) {
      if (done[a]) continue;
      const kq_matrix* lead = mats[pending[a]];
      kq::GemvGroup g{};
      for (int b = a; b < np; ++b) {
        const kq_matrix* m = mats[pending[b]];
        if (done[b] || m->format != lead->format) continue;
        g.W[g.count] = static_cast<const uint8_t*>(m->W);
        g.y[g.count] = ys[pending[b]];
        g.N[g.count] = static_cast<int>(m->N_out);
        ++g.count;
        done[b] = true;
      }
      const kq_status st =
          status_of(kq::launch_gemv(lead->format, g, static_cast<const uint16_t*>(xs[pending[a]]),
                                    static_cast<int>(lead->K), n_tok, s, false));
      if (st != KQ_OK) return st;
    }
  }
  return KQ_OK;
}

kq_status kq_dequantize(kq_format f, const void* W_blocks, float* W_out, int64_t N_out, int64_t K,
                        kq_stream_t stream) {
  kq_status st = check_matrix(f, W_blocks, N_out, K);
  if (st != KQ_OK) return st;
  if (W_out == nullptr) return KQ_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(W_out) & 3) != 0) return KQ_ERR_ALIGN;
  kq::launch_dequant(f, static_cast<const uint8_t*>(W_blocks), W_out, static_cast<int>(N_out),
                     static_cast<int>(K), reinterpret_cast<cudaStream_t>(stream));
  return launch_status();
}

kq_status kq_test_wait_timeout(unsigned int wait_us, kq_stream_t stream) {
  if (wait_us < 1 || wait_us > 1000000) return KQ_ERR_ARG;
  return kq::launch_wait_timeout_probe(wait_us, reinterpret_cast<cudaStream_t>(stream)) ? KQ_OK
                                                                                       : KQ_ERR_CUDA;
}

kq_status kq_device_status(kq_stream_t stream) {
  unsigned int n = 0;
  if (!kq::read_wait_timeouts(&n, reinterpret_cast<cudaStream_t>(stream))) return KQ_ERR_CUDA;
  return n != 0 ? KQ_ERR_TIMEOUT : KQ_OK;
}

}  // extern "C"
