// kq_kernels.cuh -- internal launch interface between the C ABI and the
// kernels of libkq.
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

namespace kq {

constexpr int kMaxGroup = 4;

// Up to kMaxGroup matrices of one format and one K that read the same
// activations (q/k/v(/gate) or gate/up of a decoder layer) and share a launch.
struct GemvGroup {
  int count;
  const uint8_t* W[kMaxGroup];
  float* y[kMaxGroup];
  int N[kMaxGroup];
};

// Outcome of a launch request.  kNotServed: no configuration of the
// streaming / tensor-core kernels serves it (nothing was launched);
// kTooLarge: only configurations whose split-K sums exceed the fixed scratch
// array of the no-allocation path would serve it; kFailed: a CUDA call failed.
enum class StreamResult { kLaunched, kNotServed, kTooLarge, kFailed };

// The streaming and tensor-core kernels: n_tok 1 on the CUDA cores or (large
// Q4_K / Q4_G128) the tensor cores, 2..16 on the tensor cores, else the
// CUDA-core kernel in chunks of up to four tokens.  noalloc: split-K partial
// sums go to the library's fixed device array instead of the per-device
// buffer that grows with cudaMalloc.
StreamResult launch_stream(int fmt, const GemvGroup& g, const uint16_t* x, int K, int n_tok,
                           cudaStream_t stream, bool noalloc);

// launch_stream, then, for requests it does not serve, the warp-per-row
// kernel (which needs no scratch and serves every valid request).
StreamResult launch_gemv(int fmt, const GemvGroup& g, const uint16_t* x, int K, int n_tok,
                         cudaStream_t stream, bool noalloc);

// The dp4a path: x quantised to int8 per 32 positions of a token (dx =
// amax / 127, xq = rint(x / dx), binary32), integer sub-block dot products,
// on the streaming kernel in launches of up to four tokens.
StreamResult launch_q8(int fmt, const GemvGroup& g, const uint16_t* x, int K, int n_tok,
                       cudaStream_t stream);
// The codes and steps of the dp4a path alone (n a multiple of 32).
bool launch_quantize_x_q8(const uint16_t* x, int64_t n, int8_t* xq, float* dx,
                          cudaStream_t stream);

// SwiGLU input of the down projection: g = {gate, up} (same format and
// shape), y written as for launch_gemv, and h = bf16(silu(gate) * up)
// ([n_tok][N]).  Fused into the gate/up launch on the single-token
// tensor-core kernel; otherwise the grouped GEMV then an elementwise kernel.
StreamResult launch_swiglu(int fmt, const GemvGroup& g, const uint16_t* x, int K, int n_tok,
                           uint16_t* h, cudaStream_t stream);

// One warp whose bounded wait (limit ~wait_us) runs out on a barrier that
// nothing completes; the event is counted like any other timeout.
bool launch_wait_timeout_probe(unsigned int wait_us, cudaStream_t stream);

// Number of bounded waits that timed out since the last call (then cleared).
bool read_wait_timeouts(unsigned int* count, cudaStream_t stream);

void launch_dequant(int fmt, const uint8_t* W, float* out, int N, int K, cudaStream_t stream);

}  // namespace kq
