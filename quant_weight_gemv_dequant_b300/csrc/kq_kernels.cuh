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

// Returns false if the format / n_tok combination has no kernel.
bool launch_gemv(int fmt, const GemvGroup& g, const uint16_t* x, int K, int n_tok,
                 cudaStream_t stream);

// The streaming kernels: n_tok <= 4 on the CUDA cores, 5..16 on the tensor
// cores; false if they do not serve the request.
bool launch_stream(int fmt, const GemvGroup& g, const uint16_t* x, int K, int n_tok,
                   cudaStream_t stream);

// kq_gemv_noalloc: the streaming kernels with their split-K scratch in a
// fixed device array (no allocation).  kNotServed: no configuration of these
// kernels serves the request; the caller may use a kernel that needs no
// scratch.
enum class NoAllocResult { kLaunched, kNotServed, kTooLarge, kFailed };
NoAllocResult launch_stream_noalloc(int fmt, const GemvGroup& g, const uint16_t* x, int K,
                                    int n_tok, cudaStream_t stream);

// Number of bounded waits that timed out since the last call (then cleared).
bool read_wait_timeouts(unsigned int* count, cudaStream_t stream);

void launch_dequant(int fmt, const uint8_t* W, float* out, int N, int K, cudaStream_t stream);

}  // namespace kq
