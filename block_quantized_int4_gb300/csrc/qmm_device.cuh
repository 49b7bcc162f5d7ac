// qmm_device.cuh -- device building blocks shared by the libqmm kernels:
// the Q8_0 block quantizer, the Q4_0 nibble unpack + integer block dot, and
// small PTX wrappers.  Compiled for sm_103a only.
//
// Method: llama.cpp guide (kenji.blog/id) section 2.2 -- w ~ Delta*q,
// Delta = max|w|/7, q in [-8,7]; y ~ Delta*Delta_x*sum q*q_x with an integer
// inner sum.  Q8_0-style activations: Colibri page (kerneldigest.dev),
// "Arquitectura del Sistema".  Block of 32 with one fp16 scale: TinyLLaMA
// C++ guide (kenji.blog) section 6.1.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace qmm {

constexpr int QK = 32;
constexpr unsigned FULL = 0xffffffffu;

// Device error word bits (read back by qmm_last_device_error).
constexpr int ERR_BAD_EXPERT = 1;
constexpr int ERR_TIMEOUT = 2;

// ---------------------------------------------------------------- PTX helpers
// Streaming 16-byte load of weight bytes: read-only path, no L1 allocation
// (every weight byte is used exactly once per product).
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ unsigned short ld_stream_u16(const void* p) {
    unsigned short r;
    asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(r) : "l"(p));
    return r;
}

// dot of four unsigned bytes (a) with four signed bytes (b), plus c.
__device__ __forceinline__ int dp4a_us(unsigned a, int b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// ---------------------------------------------------------------- Q4_0 x Q8_0 block dot
// w: the 16 nibble bytes of one weight block (byte j = u[j] | u[j+16] << 4,
// u = q + 8).  xlo/xhi: the block's 32 int8 activations, elements 0..15 and
// 16..31.  Returns sum_i u_i * qx_i; the caller subtracts 8 * sum_i qx_i.
__device__ __forceinline__ int block_dot_u(uint4 w, int4 xlo, int4 xhi) {
    constexpr unsigned LO = 0x0F0F0F0Fu;
    int s = 0;
    s = dp4a_us(w.x & LO, xlo.x, s);
    s = dp4a_us(w.y & LO, xlo.y, s);
    s = dp4a_us(w.z & LO, xlo.z, s);
    s = dp4a_us(w.w & LO, xlo.w, s);
    s = dp4a_us((w.x >> 4) & LO, xhi.x, s);
    s = dp4a_us((w.y >> 4) & LO, xhi.y, s);
    s = dp4a_us((w.z >> 4) & LO, xhi.z, s);
    s = dp4a_us((w.w >> 4) & LO, xhi.w, s);
    return s;
}

// ---------------------------------------------------------------- Q8_0 quantizer
// Eight consecutive lanes (lane % 8 == 0 .. 7) hold one block of 32 values,
// four consecutive values each.  All 32 lanes of the warp must call this.
// Per block: amax, d32 = amax/127 (IEEE division), q = clamp(rha(v/d32),
// -127, 127) with round-half-away (roundf), zero block -> q = 0, d32 = 0.
// Returns the four int8 codes packed little-endian; d32 and the block's code
// sum are returned in every lane of the group.
struct Q8Quad {
    int packed;
    float d32;
    int qsum;
};

__device__ __forceinline__ int q8_code(float v, float d32, bool nonzero) {
    if (!nonzero) return 0;
    float r = roundf(__fdiv_rn(v, d32));
    r = fminf(fmaxf(r, -127.0f), 127.0f);
    return (int)r;
}

__device__ __forceinline__ Q8Quad q8_0_quad(float4 v) {
    float a = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
    a = fmaxf(a, __shfl_xor_sync(FULL, a, 1));
    a = fmaxf(a, __shfl_xor_sync(FULL, a, 2));
    a = fmaxf(a, __shfl_xor_sync(FULL, a, 4));
    const float d32 = __fdiv_rn(a, 127.0f);
    const bool nz = a != 0.0f;
    int q0 = q8_code(v.x, d32, nz), q1 = q8_code(v.y, d32, nz);
    int q2 = q8_code(v.z, d32, nz), q3 = q8_code(v.w, d32, nz);
    int s = q0 + q1 + q2 + q3;
    s += __shfl_xor_sync(FULL, s, 1);
    s += __shfl_xor_sync(FULL, s, 2);
    s += __shfl_xor_sync(FULL, s, 4);
    Q8Quad r;
    r.packed = (q0 & 0xff) | ((q1 & 0xff) << 8) | ((q2 & 0xff) << 16) | ((q3 & 0xff) << 24);
    r.d32 = d32;
    r.qsum = s;
    return r;
}

__device__ __forceinline__ unsigned short f32_to_f16_bits(float f) {
    return __half_as_ushort(__float2half_rn(f));
}

__device__ __forceinline__ float f16_bits_to_f32(unsigned short h) {
    return __half2float(__ushort_as_half(h));
}

// SwiGLU element (TinyLLaMA guide 4.4): Swish(g) * u, Swish(z) = z*sigmoid(z).
__device__ __forceinline__ float swiglu1(float g, float u) {
    return __fdiv_rn(g, 1.0f + expf(-g)) * u;
}

// ---------------------------------------------------------------- warp reduce
__device__ __forceinline__ float warp_sum(float v) {
    v += __shfl_xor_sync(FULL, v, 16);
    v += __shfl_xor_sync(FULL, v, 8);
    v += __shfl_xor_sync(FULL, v, 4);
    v += __shfl_xor_sync(FULL, v, 2);
    v += __shfl_xor_sync(FULL, v, 1);
    return v;
}

}  // namespace qmm
