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

// One warp whose bounded wait (limit ~wait_us) runs out on a barrier that
// nothing completes; the event is counted like any other timeout.
bool launch_wait_timeout_probe(unsigned int wait_us, cudaStream_t stream);

// Number of bounded waits that timed out since the last call (then cleared).
bool read_wait_timeouts(unsigned int* count, cudaStream_t stream);

void launch_dequant(int fmt, const uint8_t* W, float* out, int N, int K, cudaStream_t stream);

}  // namespace kq
