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

// Row plan of the 16-warp layout: rpc rows per chunk (96, 128 or 192; 0
// where the layout does not apply), nchunk chunks per CTA, nsplit CTAs per
// cluster splitting K; sms the SM count it was made for.  split192: whether
// K may be split over clusters sharing 192-row chunks (the plain entry's
// plan) or over 128-row chunks only (the workspace entry's).
struct WidePlan {
    int rpc, nchunk, nsplit, sms;
};
WidePlan gemm_wide_plan(int64_t N, int64_t K, int64_t M, int sms, bool split192);

// Bytes of the workspace of qmm_gemm_q4_0_q8_0_ws for K and M (1..16
// tokens; 0 otherwise): one record of fp16 B fragments, MMA seeds and scaled
// d_x per 16 blocks of K, then 4096 flag words for products cut evenly over
// the SMs.
size_t gemm_prep_bytes(int64_t K, int64_t M);

// The 16-warp layout with the activation prepared once into `workspace`
// (>= gemm_prep_bytes, 128-byte aligned) by a launch ahead of the product;
// plan p from gemm_wide_plan (rpc > 0), xd 16-byte aligned.  Both launches
// use programmatic dependent launch.
qmm_status gemm_prep_launch(const uint8_t* w_qs, const uint16_t* w_d, int64_t N, int64_t K, int64_t M,
                            const int8_t* xq, const uint16_t* xd, float* y, int64_t ldy, const WidePlan& p,
                            void* workspace, int smem_optin, int* err, cudaStream_t st);

// True when gemm_mma_launch (wide = true) takes the 16-warp layout for this
// product: up to 16 tokens, xd 16-byte aligned, and a row plan at one CTA
// per SM of 128 or 192 rows per CTA (ceil(N / sms) in 65..192), 96 rows for
// 9..16 tokens, several chunks of 128 or 192 rows per CTA for larger N, or
// for smaller N with long K, 128- or 192-row chunks split over K by clusters
// of 2..4 CTAs.
bool gemm_wide_planned(int64_t N, int64_t K, int64_t M, const void* xd, int sms);

// Enqueue y[m*ldy + n] (m < M, n < N) on `st`.  `sms` and `smem_optin` are
// the device's SM count and opt-in shared memory per block; `err` is the
// device error word (an expired bounded wait sets ERR_TIMEOUT in it).
// `wide`: up to 16 tokens, take the 16-warp layout where its row plan
// qualifies; otherwise (and when false) the row-group kernel.
qmm_status gemm_mma_launch(const uint8_t* w_qs, const uint16_t* w_d, int64_t N, int64_t K, int64_t M,
                           const int8_t* xq, const uint16_t* xd, float* y, int64_t ldy, int sms, int smem_optin,
                           int* err, cudaStream_t st, bool wide);

}  // namespace qmm

namespace qmm {

// True when the tensor-memory GEMM (qmm_gemm_tmem.cu, tcgen05 with the
// weight operand in TMEM; used when selected by qmm_debug_gemm_kernel) can
// take this product: 1 <= M <= 16, K % 256 == 0, all four operand pointers
// 16-byte aligned.
bool gemm_tmem_eligible(int64_t N, int64_t K, int64_t M, const void* w_qs, const void* w_d, const void* xq,
                        const void* xd);

// Row plan of the tensor-memory GEMM: nst super-tiles of H rows per CTA,
// `grid` CTAs.
void gemm_tmem_plan(int64_t N, int sms, int* H, int* nst, int64_t* grid);

// Enqueue y[m*ldy + n] (m < M <= 16, n < N) on `st`; arguments as for
// gemm_mma_launch.
qmm_status gemm_tmem_launch(const uint8_t* w_qs, const uint16_t* w_d, int64_t N, int64_t K, int64_t M,
                            const int8_t* xq, const uint16_t* xd, float* y, int64_t ldy, int sms, int smem_optin,
                            int* err, cudaStream_t st);

}  // namespace qmm
