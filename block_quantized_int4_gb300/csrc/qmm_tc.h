// qmm_tc.h -- internal interface between the C ABI (qmm_api.cu) and the
// tensor-core GEMM translation unit (qmm_gemm_tc.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "qmm.h"

namespace qmm {

// True when the tcgen05 GEMM can take this product: 1 <= M <= 64,
// K % 256 == 0, all four operand pointers 16-byte aligned, and the driver
// exposes the tensor-map encoder.
bool gemm_tc_eligible(int64_t N, int64_t K, int64_t M, const void* w_qs, const void* w_d, const void* xq,
                      const void* xd);

// Enqueue the tcgen05 GEMM (y[m*ldy + n], m < M, n < N) on `st`; `err` is the
// device error word (bounded waits that expire set ERR_TIMEOUT in it).
qmm_status gemm_tc_launch(const uint8_t* w_qs, const uint16_t* w_d, int64_t N, int64_t K, int64_t M,
                          const int8_t* xq, const uint16_t* xd, float* y, int64_t ldy, int* err, cudaStream_t st);

// Encode a 2D tiled TMA descriptor (row-major [outer][inner] tensor of
// `dt` elements, row pitch `row_bytes`) with the driver's encoder, fetched
// through the runtime; false if the encoder is unavailable or rejects it.
bool make_tensor_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                        uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw);

}  // namespace qmm
