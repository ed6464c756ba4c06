// h3q_internal.cuh -- declarations shared by the library's translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "h3q.h"

namespace h3q {

constexpr int kQMax = 127;

// Launchers.  Each returns cudaSuccess or the launch error; arguments are
// already validated by the C-ABI layer.

// Norm segments: the K range of a row is cut into kNormSegs segments of
// norm_segment_len(K) elements (the last ones shorter or empty), each a whole
// number of the GEMM's 128-element super-stages.  The GEMM may check its
// accumulator between segments.
constexpr int kNormSegs = 4;
constexpr int kSegQuantum = 128;
__host__ __device__ constexpr int norm_segment_len(int64_t K) {
  return int(((K + kSegQuantum - 1) / kSegQuantum + kNormSegs - 1) / kNormSegs) * kSegQuantum;
}

// A2: BF16 activations -> int8 (optional) + FP32 scale + FP16-coded q (optional,
// rows of stride ldh >= K elements, the padding zeroed).  sq_max (optional):
// the activation norm maxima, ceil(M/256) * (1 + kNormSegs) words: per block
// of 256 rows the running maximum of the rows' sums of q^2, then per block
// and segment the maximum of the rows' sums over that segment (atomicMax, so
// the region must start at zero).  err (optional, a status word): with it,
// rows of 6144 < K <= 24576 take the kernel that stages them in shared
// memory, whose bounded waits report a timeout there.
cudaError_t launch_quantize_act(const uint16_t* x, int64_t M, int64_t K, int8_t* q,
                                float* scale, uint16_t* q_f16, int64_t ldh, uint32_t* sq_max,
                                cudaStream_t s, uint32_t* err = nullptr);

// A1: FP32 or BF16 weights -> int8 + FP32 scale.  A row with a non-finite
// element gets a NaN scale, which the caller turns into H3Q_ERR_NONFINITE.
cudaError_t launch_quantize_weights(const void* w, int w_dtype, int64_t N, int64_t K,
                                    int8_t* q, float* scale, cudaStream_t s);

// int8 [M, K] -> FP16-coded integers with row stride ldh (padding zeroed),
// with the activation norm maxima as launch_quantize_act.
cudaError_t launch_int8_to_f16(const int8_t* q, int64_t M, int64_t K, int64_t ldh,
                               uint16_t* out, uint32_t* sq_max, cudaStream_t s);

// Row stride (elements) of the FP16-coded activations in the linear workspace.
int64_t gemm_tc_coded_ld(int64_t K);

// Tokens per block of the activation norm maxima (the wide kernel's tile).
constexpr int kNormTokens = 256;
// Weight-norm partial maxima per 128-channel block (16 channels each).
constexpr int kNormParts = 8;
// Linears of one grouped call (they share the input).
constexpr int kMaxGroup = 4;

// The per-Linear operands of a call: G Linears with the same N and K that read
// the same activations (G = 1 for a single Linear).
struct LinearGroup {
  int G;
  const int8_t* wq[kMaxGroup];
  const float* ws[kMaxGroup];
  const uint16_t* bias[kMaxGroup];
  uint16_t* y[kMaxGroup];
  int32_t* acc[kMaxGroup];
};

// The linear workspace, in order (each part 256-byte aligned):
//   act     [M, gemm_tc_coded_ld(K)] FP16-coded activations
//   amax    [ceil(M/256)] u32: per 256 tokens, max over rows of sum(qa^2);
//           then [ceil(M/256)][kNormSegs] u32, the same per norm segment
//   status  256 bytes: word 0 error bits, word 1 fallback-list length over
//           all Linears, word 2 + g the length of Linear g's list, word 6
//           the tiles that took accumulator checkpoints, word 7 those of
//           them whose check failed (they are on the fallback list too)
//   nwpart  G x [ceil(N/128) * 8] u32: per 16 channels, max over rows of
//           sum(qw^2); then G x [ceil(N/128) * 8][kNormSegs], per segment
//   list    G x [ceil(M/128) * ceil(N/256)] uint2 {token block, channel pair}:
//           the 128 x 256 tiles the chunked kernel must finish
// act, amax and status depend on M and K only, so a call with another N
// still finds the coded activations (reuse) and the status word there.
// status starts each call at zero, amax too when the activations are coded
// anew; they are contiguous so that one memset clears them.
struct WorkspaceLayout {
  size_t act, amax, status, nwpart, list, total;
};
WorkspaceLayout workspace_layout(int64_t M, int64_t N, int64_t K, int G = 1);
// Entries of one Linear's fallback list.
size_t fallback_list_capacity(int64_t M, int64_t N);

// Weight pre-pass: nwpart as above, left unwritten when amax shows that no
// tile can need it (programmatic dependent launch after the quantiser).
cudaError_t launch_weight_norms(const LinearGroup& grp, int64_t N, int64_t K,
                                const uint32_t* amax, int64_t M, uint32_t* nwpart,
                                cudaStream_t s);

// A3 + A4 for the tiles whose FP32 sums are exact over the whole K (checked
// per tile from amax and, where that is not enough, nwpart), or provably
// exact with checks of the accumulator between norm segments; the others
// are appended to `list`, status[1] counting the entries.  status[0]: error
// bits (bounded waits).
cudaError_t launch_gemm_wide(const uint16_t* act_f16, const float* sa, const LinearGroup& grp,
                             int64_t M, int64_t N, int64_t K, const uint32_t* amax,
                             const uint32_t* nwpart, uint32_t* status, uint2* list,
                             cudaStream_t s);

// The group-wise affine comparison scheme (weight-only): y = BF16(x W^T + bias)
// with W dequantised from 8-bit codes, per channel and group of 64 inputs
// w = step q + offset (one FP32 FMA, then BF16).  x: BF16 [M, K], K a multiple
// of 64; grp.wq: the codes [N, K] (unsigned); ab[g]: [N, K/64] (step, offset)
// FP32 pairs; grp.ws and grp.acc unused.  status[0]: error bits.
cudaError_t launch_gemm_affine(const uint16_t* x, const LinearGroup& grp, const float* const* ab,
                               int64_t M, int64_t N, int64_t K, uint32_t* status, cudaStream_t s);

// Offline group-wise affine quantisation of FP32 or BF16 weights [N, K] into
// `bits`-bit codes (8 or 4; one code per byte) and (step, offset) FP32 pairs
// [N, K/64]; a group holding Inf or NaN gets a NaN step, which the caller
// turns into H3Q_ERR_NONFINITE.
cudaError_t launch_quantize_weights_affine(const void* w, int w_dtype, int bits, int64_t N,
                                           int64_t K, uint8_t* q, float* ab, cudaStream_t s);

// A3 + A4 on the tcgen05 tensor cores (exact INT32 via FP16 MMA with chunked
// FP32 accumulation) for the G Linears of grp.  act_f16: [M,
// gemm_tc_coded_ld(K)] FP16-coded INT8 activations, the padding beyond K zero.
// err: device status word (0 = ok; bits set when a bounded wait gave up).
// list == NULL: every tile of Linear 0.  Otherwise the tiles in the G lists
// (Linear g's at list + g * list_cap, list_len[g] entries, written by the wide
// kernel); the kernel exits at once when every list is empty.
cudaError_t launch_gemm_tc(const uint16_t* act_f16, const float* sa, const LinearGroup& grp,
                           int64_t M, int64_t N, int64_t K, uint32_t* err, const uint2* list,
                           const uint32_t* list_len, size_t list_cap, cudaStream_t s);

// cuTensorMapEncodeTiled, looked up through the runtime (no -lcuda); NULL if
// the driver does not provide it.
void* tensor_map_encoder();

// A3 + A4 on the legacy warp-level INT8 tensor path (mma.sync m16n8k32 s8).
cudaError_t launch_gemm_mma_s8(const int8_t* qa, const float* sa, const int8_t* qw,
                               const float* sw, const uint16_t* bias, int64_t M, int64_t N,
                               int64_t K, uint16_t* y, int32_t* acc, cudaStream_t s);

}  // namespace h3q
