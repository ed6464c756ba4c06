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

// A2: BF16 activations -> int8 (optional) + FP32 scale + FP16-coded q (optional,
// rows of stride ldh >= K elements, the padding zeroed).
cudaError_t launch_quantize_act(const uint16_t* x, int64_t M, int64_t K, int8_t* q,
                                float* scale, uint16_t* q_f16, int64_t ldh, cudaStream_t s);

// A1: FP32 or BF16 weights -> int8 + FP32 scale.  A row with a non-finite
// element gets a NaN scale, which the caller turns into H3Q_ERR_NONFINITE.
cudaError_t launch_quantize_weights(const void* w, int w_dtype, int64_t N, int64_t K,
                                    int8_t* q, float* scale, cudaStream_t s);

// int8 [M, K] -> FP16-coded integers with row stride ldh (padding zeroed).
cudaError_t launch_int8_to_f16(const int8_t* q, int64_t M, int64_t K, int64_t ldh,
                               uint16_t* out, cudaStream_t s);

// Row stride (elements) of the FP16-coded activations in the linear workspace.
int64_t gemm_tc_coded_ld(int64_t K);

// A3 + A4 on the tcgen05 tensor cores (exact INT32 via FP16 MMA with chunked
// FP32 accumulation).  act_f16: [M, gemm_tc_coded_ld(K)] FP16-coded INT8
// activations, the padding beyond K zero.
// err: device status word (0 = ok; bits set when a bounded wait gave up).
cudaError_t launch_gemm_tc(const uint16_t* act_f16, const float* sa, const int8_t* qw,
                           const float* sw, const uint16_t* bias, int64_t M, int64_t N,
                           int64_t K, uint16_t* y, int32_t* acc, uint32_t* err, cudaStream_t s);

// Byte offset of the status word inside the linear workspace.
size_t gemm_tc_status_offset(int64_t M, int64_t K);

// A3 + A4 on the legacy warp-level INT8 tensor path (mma.sync m16n8k32 s8).
cudaError_t launch_gemm_mma_s8(const int8_t* qa, const float* sa, const int8_t* qw,
                               const float* sw, const uint16_t* bias, int64_t M, int64_t N,
                               int64_t K, uint16_t* y, int32_t* acc, cudaStream_t s);

}  // namespace h3q
