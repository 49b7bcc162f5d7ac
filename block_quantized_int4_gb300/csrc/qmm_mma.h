// qmm_mma.h -- internal interface between the C ABI (qmm_api.cu) and the
// warp-MMA small-batch GEMM translation unit (qmm_gemm_mma.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "qmm.h"

namespace qmm {

// True when the warp-MMA GEMM can take this product: M >= 1, K % 256 == 0,
// weight and activation pointers 16-byte aligned, and the driver exposes
// the tensor-map encoder.
bool gemm_mma_eligible(int64_t N, int64_t K, int64_t M, const void* w_qs, const void* w_d, const void* xq,
                       const void* xd);

// Enqueue y[m*ldy + n] (m < M, n < N) on `st`.  `sms` and `smem_optin` are
// the device's SM count and opt-in shared memory per block; `err` is the
// device error word (an expired bounded wait sets ERR_TIMEOUT in it).
qmm_status gemm_mma_launch(const uint8_t* w_qs, const uint16_t* w_d, int64_t N, int64_t K, int64_t M,
                           const int8_t* xq, const uint16_t* xd, float* y, int64_t ldy, int sms, int smem_optin,
                           int* err, cudaStream_t st);

}  // namespace qmm
