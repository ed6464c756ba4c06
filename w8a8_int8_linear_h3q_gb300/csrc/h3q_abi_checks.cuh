// h3q_abi_checks.cuh -- the argument and device checks that every C-ABI entry
// point applies before it enqueues anything (defined in h3q_api.cu).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "h3q.h"

namespace h3q {

// 16-byte alignment of a base pointer (vector loads and TMA need it).
bool aligned16(const void* p);

// M, N, K within the shape rules of the C ABI (K % 16 == 0, K * 127^2 < 2^31,
// 32-bit tile coordinates).
h3q_status check_shape(int64_t M, int64_t N, int64_t K);

// The current device is an sm_103 part (the kernels are built for sm_103a only).
h3q_status check_device();

// cudaSuccess -> H3Q_OK, anything else -> H3Q_ERR_CUDA (printed when H3Q_VERBOSE is set).
h3q_status from_cuda(cudaError_t e);

}  // namespace h3q
