/*
 * kq.h -- C ABI of libkq: fused dequantise-and-multiply of K-quant weights
 * against 1..16 bf16 activation rows on one NVIDIA B300 (sm_103a).
 *
 * What the operation is.  The daily.dev summary "Fast on-device agentic AI
 * with Muse Glimmer on ExecuTorch" (answer "How does ExecuTorch export Muse
 * Glimmer GGUF checkpoints for CUDA and Apple Silicon?") says the CUDA backend
 * runs GGUF Q4_K/Q5_K/Q6_K weights directly as packed integer GEMV kernels and
 * that adjacent sub-blocks with the same scale/min are merged, when lossless,
 * into groups of up to 128.  The SGLang day-0 post on Muse Glimmer (paragraph
 * on the GGUF checkpoints) names a Q4_K_M checkpoint with 128-weight groups.
 * The Core AI model card for Muse-Glimmer-30B (first table and the sentence
 * under it) shows decode streaming every weight once per token (23.7 tok/s x
 * 17.9 GB = 424 GB/s), i.e. the product y = W x is weight-bandwidth bound.
 *
 * Every function computes, for t < n_tok and n < N_out,
 *     y[t][n] = sum_k  w^[n][k] * x[t][k]
 * where w^ is the dequantised weight defined by the record layouts below.
 *
 * Record layouts (all little-endian; a row of K weights is K/256
 * consecutive super-blocks; rows are stored one after another):
 *
 *  KQ_Q4_K (144 B / 256 weights)
 *     [0,2) d (fp16)  [2,4) dmin (fp16)  [4,16) scales[12]  [16,144) qs[128]
 *     sub-block j (0..7) has a 6-bit scale sc_j and 6-bit min m_j:
 *       j < 4 : sc_j = scales[j] & 63,           m_j = scales[j+4] & 63
 *       j >= 4: sc_j = (scales[j+4] & 15) | ((scales[j-4] >> 6) << 4)
 *               m_j  = (scales[j+4] >> 4) | ((scales[j]   >> 6) << 4)
 *     weight i (0..255): c = i/64, r = i%64;
 *       r < 32 : q = qs[32c+r] & 15,     j = 2c
 *       r >= 32: q = qs[32c+r-32] >> 4,  j = 2c+1
 *     w^ = d*sc_j*q - dmin*m_j
 *  KQ_Q5_K (176 B / 256 weights)
 *     [0,2) d  [2,4) dmin  [4,16) scales[12] (as Q4_K)  [16,48) qh[32]
 *     [48,176) qs[128];  weight i: c = i/64, r = i%64, l = r%32;
 *       low nibble as Q4_K (qs[32c+l], low half if r<32 else high half),
 *       fifth bit = (qh[l] >> (2c + (r>=32))) & 1,  q = nibble | bit<<4
 *     w^ = d*sc_j*q - dmin*m_j
 *  KQ_Q6_K (210 B / 256 weights)
 *     [0,128) ql  [128,192) qh  [192,208) scales[16] (int8)  [208,210) d
 *     weight i: h = i/128, t = (i%128)/32, l = i%32;
 *       nibble = ql[64h + l + 32*(t&1)], low half if t<2 else high half
 *       2 high bits = (qh[32h + l] >> 2t) & 3,  q = nibble | hb<<4
 *     w^ = d*scales[i/16]*(q-32)
 *  KQ_Q4_G128 (136 B / 256 weights, planar; this library's merged layout)
 *     one buffer = [q plane: N_out*K/2 bytes][param plane: N_out*K/256*8 B]
 *     q plane: per super-block 128 B laid out exactly as Q4_K's qs;
 *     param plane: per super-block 8 B {d fp16, dmin fp16, sc0, sc1, m0, m1};
 *     group g = i/128 (sub-blocks 4g..4g+3 of the Q4_K it came from)
 *     w^ = d*sc_g*q - dmin*m_g
 *
 * Conventions for every entry point.
 *   - The caller owns its inputs and outputs.  The library allocates device
 *     memory in exactly one place: kq_gemv (and kq_gemv_multi, kq_layer_step,
 *     which use it) grows a per-device split-K scratch buffer with cudaMalloc
 *     on the first long-row request that needs more than it holds (never
 *     while the stream is being captured; that request then runs a
 *     configuration without the buffer).  kq_gemv_noalloc never allocates.
 *   - Device pointers: W_blocks must be 16-byte aligned; x is bf16
 *     [n_tok][K] with contiguous rows (x must be 16-byte aligned and K a
 *     multiple of 256); y is fp32 [n_tok][N_out] and is overwritten.
 *   - Requirements: K % 256 == 0, K > 0, N_out > 0, 1 <= n_tok <= 16.  A
 *     violation returns a status before anything is launched.
 *   - Calls on a stream are asynchronous and never synchronise (except
 *     kq_device_status); a CUDA graph may capture them once the same shape
 *     has run outside capture.
 *   - A CUDA launch failure returns KQ_ERR_CUDA.  Nothing throws or exits
 *     across this ABI.  NaN/Inf inputs give unspecified (but in-bounds)
 *     results.
 *   - Every declaration below carries a "Source:" line: the page passage
 *     that defines the operation, or a statement that the pages define none.
 */
#ifndef KQ_H
#define KQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL means the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st* kq_stream_t;

typedef enum {
  KQ_Q4_K = 0,    /* 4-bit q, 8 sub-blocks of 32, 6-bit sc/m, fp16 d/dmin */
  KQ_Q5_K = 1,    /* as Q4_K with a fifth bit per weight                   */
  KQ_Q6_K = 2,    /* 6-bit q, 16 sub-blocks of 16, int8 sc, fp16 d          */
  KQ_Q4_G128 = 3  /* Q4_K with one (sc, m) per 128 weights, planar          */
} kq_format;

typedef enum {
  KQ_OK = 0,
  KQ_ERR_ARG = 1,           /* null pointer, bad enum, n_tok out of range  */
  KQ_ERR_SHAPE = 2,         /* K % 256 != 0, non-positive sizes, mismatch  */
  KQ_ERR_ALIGN = 3,         /* a device pointer is not 16-byte aligned     */
  KQ_ERR_NOT_MERGEABLE = 4, /* kq_merge_g128: sub-blocks differ in (sc, m) */
  KQ_ERR_RANGE = 5,         /* kq_quantize: a scale exceeds fp16 range     */
  KQ_ERR_CUDA = 6,          /* a CUDA runtime call or launch failed        */
  KQ_ERR_UNSUPPORTED = 7,   /* valid request the library cannot serve     */
  KQ_ERR_TIMEOUT = 8,       /* a kernel's bounded wait ran out (see below) */
  KQ_ERR_TOO_LARGE = 9      /* kq_gemv_noalloc: beyond its fixed scratch    */
} kq_status;

/* Bytes of one 256-weight super-block: 144 / 176 / 210 / 136.  0 for a bad
 * format.
 * Source: the pages define no sizes; these are the GGUF record sizes of the
 * formats the daily.dev summary names (answer on exporting GGUF
 * checkpoints), whose bytes per weight match the Core AI card's 17.9 GB file
 * (first table), plus this library's 136-byte merged group-128 record. */
size_t kq_block_bytes(kq_format f);

/* Bytes of an N_out x K matrix in format f (N_out*K/256 super-blocks; for
 * KQ_Q4_G128 both planes).  0 if the shape is invalid.
 * Source: none in the pages; N_out*K/256 times kq_block_bytes. */
size_t kq_matrix_bytes(kq_format f, int64_t N_out, int64_t K);

/* y[t][n] = sum_k w^[n][k] x[t][k] for t < n_tok, n < N_out.
 *   W_blocks : device, the N_out x K matrix in format f, 16-B aligned
 *   x_bf16   : device, bf16 [n_tok][K], 16-B aligned
 *   y        : device, fp32 [n_tok][N_out], overwritten
 * Accumulates in fp32.
 * Source: the daily.dev ExecuTorch summary, answer on exporting GGUF
 * checkpoints (Q4_K/Q5_K/Q6_K GEMV; group-128 merge); the Core AI card's
 * n-gram speculation paragraph and the PTE card ("Adjustments per variant")
 * for the verify widths n_tok <= 16.
 * Long rows are split over several CTAs whose partial sums go to a split-K
 * scratch buffer of the current device, allocated by the library on first
 * need (never while the stream is being captured; a capture then runs the
 * unsplit configuration) and grown by allocating a larger one; buffers are
 * never freed, so CUDA graphs captured earlier stay valid.  Row tiles are
 * handed to CTAs at run time from per-K-segment counters that live in the
 * library (zero between launches; every launch re-arms them before it ends).
 * The scratch buffer and the counters are shared by all calls on a device:
 * calls that overlap on the GPU (different streams, no ordering between
 * them) race on them.  Results do not depend on which CTA takes which tile:
 * every sum is formed in a fixed order. */
kq_status kq_gemv(kq_format f, const void* W_blocks, const void* x_bf16,
                  float* y, int64_t N_out, int64_t K, int n_tok,
                  kq_stream_t stream);

/* kq_gemv for callers that must not allocate device memory.
 * Source: none -- the pages have no counterpart; this entry point exists
 * for users of this library.  Some callers cannot call cudaMalloc at the
 * moment they compute: code running while a stream is being captured into a
 * CUDA graph, engines that hand out all device memory from their own pool
 * and forbid driver allocations after start-up, and latency-critical loops
 * that cannot afford an allocation's implicit device synchronisation.
 * kq_gemv may allocate a split-K scratch buffer on its first long-row call;
 * this variant never allocates (no cudaMalloc, cudaFree or allocating
 * library call on any path) and keeps that scratch in a fixed 4 MiB array
 * compiled into the library, which every GPU that loads the library holds
 * until the process exits.
 *   Same arguments, requirements and result as kq_gemv (within the same
 *   tolerance).  The kernels are kq_gemv's; where the fastest configuration
 *   would need more split-K sums than the array holds, a configuration with
 *   fewer K segments, or the next kernel kq_gemv would try, runs instead.
 *   Limits: a request that the streaming and tensor-core kernels can serve
 *   only with more than 16384 row tiles or more partial sums than fit in
 *   4 MiB - 64 KiB at 8 bytes each (roughly N_out * n_tok * K-segments >
 *   500000, e.g. rows of 32768 weights at 4 tokens and 200000 outputs)
 *   returns KQ_ERR_TOO_LARGE and launches nothing.
 *   Set-up: the first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current and caches it; make
 *   that first call before any stream capture.
 *   Sharing: every call uses the same array, which keeps the previous
 *   call's contents; each call clears the counters it needs (a
 *   stream-ordered memset).  Calls that overlap on the GPU (different
 *   streams, no ordering between them) race on the array and on the tile
 *   counters (as for kq_gemv). */
kq_status kq_gemv_noalloc(kq_format f, const void* W_blocks, const void* x_bf16, float* y,
                          int64_t N_out, int64_t K, int n_tok, kq_stream_t stream);

/* Several matrices of one format and one K that read the same activations,
 * computed in ONE launch: y_i = w^_i x for i < count (1 <= count <= 4).
 * Source: the Core AI card for Muse-Glimmer-30B ("The architecture, and what
 * the port had to do about it") folds q, k, v and the sigmoid attention
 * gate, which all read the pre-attention hidden state, into one qkvg
 * projection; the SwiGLU gate and up projections share their input the same
 * way.
 *   W[i]     : device, N_out[i] x K matrix in format f, 16-B aligned
 *   y[i]     : device, fp32 [n_tok][N_out[i]], overwritten
 *   x_bf16   : device, bf16 [n_tok][K], 16-B aligned
 * Same requirements and statuses as kq_gemv for each matrix. */
kq_status kq_gemv_multi(kq_format f, int count, const void* const* W, float* const* y,
                        const int64_t* N_out, const void* x_bf16, int64_t K, int n_tok,
                        kq_stream_t stream);

/* One decoder layer's seven projections.
 * Source: the Muse-Glimmer-30B Core AI card ("The architecture, and what
 * the port had to do about it") and the SGLang day-0 post (architecture
 * paragraph) describe GQA attention (q, k, v read the
 * same hidden state; o reads the attention output) and a SwiGLU FFN (gate, up
 * read the same hidden state; down reads their product).  kq_layer_step runs
 * q/k/v as one launch on x_attn, then o on x_o, gate/up as one launch on
 * x_ffn, then down on x_down, in that order on `stream`. */
typedef struct {
  kq_format format;
  const void* W;   /* device, 16-B aligned */
  int64_t N_out;
  int64_t K;
} kq_matrix;

typedef struct {
  kq_matrix q, k, v, o, gate, up, down;
} kq_layer;

typedef struct {
  const void* x_attn;  /* bf16 [n_tok][q.K]    -> q, k, v    */
  const void* x_o;     /* bf16 [n_tok][o.K]    -> o          */
  const void* x_ffn;   /* bf16 [n_tok][gate.K] -> gate, up   */
  const void* x_down;  /* bf16 [n_tok][down.K] -> down       */
  float *y_q, *y_k, *y_v, *y_o, *y_gate, *y_up, *y_down; /* fp32 [n_tok][N] */
} kq_layer_io;

/* Requirements: q.K == k.K == v.K, gate.K == up.K, gate.N_out == up.N_out,
 * plus each matrix's own requirements.  Returns the first failing status;
 * on a validation failure nothing is launched.
 * Source: the layer structure of the Core AI card's architecture section
 * (see the layer types above); the product of each launch as kq_gemv. */
kq_status kq_layer_step(const kq_layer* L, const kq_layer_io* io, int n_tok,
                        kq_stream_t stream);

/* The int8-activation (dp4a) GEMV: y[t][n] = sum_k w^[n][k] * x~[t][k],
 * where x~ = dx * xq is x quantised per 32 positions of a token:
 *     dx = amax / 127,  xq = round_to_nearest_even(x / dx)   (binary32; 0 if amax = 0)
 * with amax the largest |x| of the 32.  Every sub-block's dot product is an
 * exact integer sum (dp4a: four int8 products per instruction); the scales
 * apply in fp32.  Arguments, requirements and statuses as kq_gemv.  The
 * result differs from kq_gemv's by the activation rounding: at most
 * sum_k |w^[n][k]| dx(k) / 2 (plus the usual fp32 accumulation).
 * Source: the daily.dev summary, answer on exporting GGUF checkpoints (the
 * CUDA backend runs the K-quant weights as integer GEMV with dp4a); the
 * pages give no activation block size or rounding: per 32 (the Q4_K / Q5_K
 * sub-block) and round-to-nearest are this library's reading. */
kq_status kq_gemv_q8(kq_format f, const void* W_blocks, const void* x_bf16, float* y,
                     int64_t N_out, int64_t K, int n_tok, kq_stream_t stream);

/* The activation codes of kq_gemv_q8 alone: xq_int8 (device, int8
 * [n_tok][K]) and dx (device, fp32 [n_tok][K/32]) from x (bf16 [n_tok][K]),
 * with the kernel's own steps.  K % 256 == 0, 1 <= n_tok <= 16.
 * Source: as kq_gemv_q8. */
kq_status kq_quantize_x_q8(const void* x_bf16, int64_t K, int n_tok, void* xq_int8, float* dx,
                           kq_stream_t stream);

/* The SwiGLU activation fused into the gate/up launch:
 *     y_gate = w^_gate x,  y_up = w^_up x,
 *     h[t][n] = bf16( silu(y_gate[t][n]) * y_up[t][n] ),  silu(v) = v / (1 + e^-v)
 * (silu and the product in fp32, h rounded to nearest, ties to even): h is
 * the bf16 input of the down projection.
 *   W_gate, W_up : device, two N_out x K matrices of format f, 16-B aligned
 *   x_bf16       : device, bf16 [n_tok][K], 16-B aligned
 *   y_gate, y_up : device, fp32 [n_tok][N_out], overwritten
 *   h_bf16       : device, bf16 [n_tok][N_out], 16-B aligned, overwritten
 * One launch where the single-token tensor-core kernel serves the pair (one
 * token, Q4_K or Q4_G128, 2 * N_out * K >= 2^25): each of its tiles stages
 * the gate rows and the up rows of the same outputs, and its epilogue forms
 * h.  Otherwise the grouped GEMV and then a small elementwise kernel.
 * Statuses as kq_gemv_multi; KQ_ERR_ALIGN if h_bf16 is not 16-B aligned.
 * Source: the Core AI card's architecture section (SwiGLU feed-forward:
 * the down projection reads silu(gate) * up); silu is the standard
 * definition, which the pages do not write out. */
kq_status kq_gemv_swiglu(kq_format f, const void* W_gate, const void* W_up, const void* x_bf16,
                         float* y_gate, float* y_up, void* h_bf16, int64_t N_out, int64_t K,
                         int n_tok, kq_stream_t stream);

/* One SwiGLU feed-forward block: kq_gemv_swiglu(gate, up) into h, then
 * y_down = w^_down h (kq_gemv), on `stream`.  Requires gate and up of one
 * format and shape and down.K == gate.N_out; buffers as kq_gemv_swiglu plus
 * y_down (fp32 [n_tok][down.N_out]).  Nothing but h passes between the two
 * launches.
 * Source: as kq_gemv_swiglu (the feed-forward block of the Core AI card's
 * architecture section). */
kq_status kq_ffn_swiglu(const kq_matrix* gate, const kq_matrix* up, const kq_matrix* down,
                        const void* x_ffn, float* y_gate, float* y_up, void* h_bf16,
                        float* y_down, int n_tok, kq_stream_t stream);

/* W_out[n][k] = w^[n][k] as fp32 (device, [N_out][K]).  Every w^ of these
 * formats is computed with at most one rounding (at the subtraction of the
 * min term), so the result is bit-exact: the fp32 round-to-nearest-even of
 * the exact value.
 * Source: the dequantisation formulas of the GGUF K-quant layouts that the
 * daily.dev summary names (answer on exporting GGUF checkpoints), written out
 * above: w^ = d*sc*q - dmin*m (Q4_K, Q5_K, Q4_G128), d*sc*(q-32) (Q6_K). */
kq_status kq_dequantize(kq_format f, const void* W_blocks, float* W_out,
                        int64_t N_out, int64_t K, kq_stream_t stream);

/* Host-side quantiser for test and benchmark data (runs on the CPU, not on
 * the hot path).
 * Source: none -- the pages define no quantiser; this is this library's
 * rounding quantiser (round to nearest, scales rounded outward), the reading
 * chosen for test data.  W_host: fp32 [N_out][K]; blocks_host receives
 * kq_matrix_bytes(f, N_out, K) bytes.  Rounds q to nearest (ties to even)
 * and rounds d, dmin up to fp16 so every group's range is covered, which
 * bounds |w - w^| by half a quantisation step.  Q4_G128 takes its statistics
 * over 128-weight groups.  Returns KQ_ERR_RANGE if a scale exceeds fp16. */
kq_status kq_quantize(kq_format f, const float* W_host, int64_t N_out,
                      int64_t K, void* blocks_host);

/* Host-side lossless merge of Q4_K blocks into the KQ_Q4_G128 layout.
 * Succeeds only if, in every super-block, sub-blocks 0..3 share one (sc, m)
 * and sub-blocks 4..7 share one (sc, m); otherwise returns
 * KQ_ERR_NOT_MERGEABLE and leaves g128_host unspecified.  The merged matrix
 * dequantises to bit-identical weights.
 * Source: the daily.dev ExecuTorch summary, answer on exporting GGUF
 * checkpoints (neighbouring sub-blocks that share scale and min are merged,
 * where nothing is lost, into groups of up to 128 weights) and the SGLang
 * day-0 post, GGUF paragraph (a Q4_K_M checkpoint with 128-weight groups). */
kq_status kq_merge_g128(const void* q4k_host, int64_t N_out, int64_t K,
                        void* g128_host);

/* Device-side health check.
 * Source: none in the pages; failure detection of this library's kernels.
 * The streaming kernels hand data between warps
 * through shared-memory barriers; every wait is bounded (about two seconds),
 * and a wait that runs out makes the kernel stop early and count the event
 * in a device word instead of hanging.  This call synchronises `stream`,
 * reads and clears that count, and returns KQ_ERR_TIMEOUT if it was non-zero
 * (the outputs of the kernels since the previous call are then not valid;
 * the split-K and tile counters a stopped kernel left behind are re-armed),
 * KQ_ERR_CUDA if the read failed, KQ_OK otherwise.  Not for use inside
 * stream capture. */
kq_status kq_device_status(kq_stream_t stream);

/* Test hook for the failure path above.  Launches one warp on `stream` that
 * waits on a shared-memory barrier nothing completes, with the bounded wait
 * shortened to about wait_us microseconds (1 <= wait_us <= 1000000): the wait
 * runs out, the event is counted like any other timeout, and the kernel
 * returns.  The next kq_device_status on that stream returns KQ_ERR_TIMEOUT
 * (and re-arms the library's counters); later launches are unaffected.
 * Nothing faults and nothing hangs.  Returns KQ_ERR_ARG for wait_us out of
 * range, KQ_ERR_CUDA if the launch failed.
 * Source: none in the pages; tests this library's failure detection. */
kq_status kq_test_wait_timeout(unsigned int wait_us, kq_stream_t stream);

/* One tensor of a GGUF checkpoint (kq_gguf_index). */
typedef struct {
  char name[128];         /* tensor name (truncated to 127 bytes), 0-terminated */
  int32_t ggml_type;      /* the file's tensor type (12 Q4_K, 13 Q5_K, 14 Q6_K, ...) */
  int32_t format;         /* the kq_format of that type, or -1 if the library has none */
  int32_t n_dims;
  int64_t dims[4];        /* dims[0] = row length; unused dims are 1 */
  int64_t N_out, K;       /* K-quant tensors: rows, row length (dims[0]) */
  uint64_t data_offset;   /* byte offset of the tensor's data in the file */
  uint64_t bytes;         /* K-quant tensors: kq_matrix_bytes(format, N_out, K) */
} kq_gguf_tensor;

/* Index of a GGUF checkpoint held in host memory (file, size bytes): the
 * first min(max_tensors, count) tensors into out[], the tensor count into
 * *n_tensors, the data alignment into *alignment (may be NULL).  For a
 * Q4_K / Q5_K / Q6_K tensor, the `bytes` bytes at file + data_offset are
 * the N_out x K matrix in the layout above, ready for kq_gemv once copied
 * to the device (they are 16-B aligned on the device if the copy is).
 * Host only; nothing is allocated.  Every read is checked against `size`:
 * a truncated or malformed file returns KQ_ERR_ARG (KQ_ERR_UNSUPPORTED for
 * a version other than 2 or 3, KQ_ERR_SHAPE for a K-quant tensor whose row
 * length is not a multiple of 256).
 * Source: the daily.dev summary (answer on exporting GGUF checkpoints) and
 * the SGLang day-0 post (GGUF paragraph) name GGUF checkpoints as the input;
 * the container is read as the public GGUF description lays it out
 * (header, typed key/value metadata, tensor infos, aligned data section). */
kq_status kq_gguf_index(const void* file, size_t size, kq_gguf_tensor* out, int max_tensors,
                        int* n_tensors, uint32_t* alignment);

/* Static string for a status code.
 * Source: none in the pages. */
const char* kq_status_str(kq_status s);

#ifdef __cplusplus
}
#endif

#endif /* KQ_H */
