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

// Sixteen times the block dot, with the -8 offset folded in: c = -128 *
// sum(q_x) seeds the high-nibble chain, and the high nibbles stay in place
// (w & 0xF0F0F0F0 contributes 16 * u_hi), so no shifts are needed:
// 16 * sum_lo + (16 * sum_hi - 128 * sum(q_x)) = 16 * sum_i q_w,i * q_x,i.
__device__ __forceinline__ int block_dot16(uint4 w, int4 xlo, int4 xhi, int c) {
    constexpr unsigned LO = 0x0F0F0F0Fu, HI = 0xF0F0F0F0u;
    int lo = dp4a_us(w.x & LO, xlo.x, 0);
    int hi = dp4a_us(w.x & HI, xhi.x, c);
    lo = dp4a_us(w.y & LO, xlo.y, lo);
    hi = dp4a_us(w.y & HI, xhi.y, hi);
    lo = dp4a_us(w.z & LO, xlo.z, lo);
    hi = dp4a_us(w.z & HI, xhi.z, hi);
    lo = dp4a_us(w.w & LO, xlo.w, lo);
    hi = dp4a_us(w.w & HI, xhi.w, hi);
    return lo * 16 + hi;
}

// Packed pair of fp32 lanes (two weight rows): acc += (a * b) * c elementwise,
// each product and sum rounded exactly as the scalar fmaf(a * b, c, acc).
__device__ __forceinline__ float2 ffma2_scaled(float2 a, float2 b, float2 c, float2 acc) {
    unsigned long long ua, ub, uc, ud, um, r;
    ua = *reinterpret_cast<unsigned long long*>(&a);
    ub = *reinterpret_cast<unsigned long long*>(&b);
    uc = *reinterpret_cast<unsigned long long*>(&c);
    ud = *reinterpret_cast<unsigned long long*>(&acc);
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(um) : "l"(ua), "l"(ub));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(um), "l"(uc), "l"(ud));
    return *reinterpret_cast<float2*>(&r);
}

// ---------------------------------------------------------------- fp16 bits
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

// ---------------------------------------------------------------- mbarrier + bulk copy
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Every wait on the device is bounded: this one gives up after `limit_ns`
// of wall time (or as soon as *abort is set) and returns false.
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;  // 2 s

// try_wait that lets the hardware suspend the thread for up to `ns` while
// the phase is incomplete (no busy polling of the issue slots)
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint64_t limit_ns = WAIT_LIMIT_NS) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait_sleep(bar, parity, 20000)) {
        if (*abort) return false;
        if (global_ns() - t0 > limit_ns) return false;
    }
    return true;
}

// Bulk copy global -> this CTA's shared memory, completion counted in bytes
// on `bar`.  dst/src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// L2 policy for weight bytes, which every product reads exactly once: evict
// them first, so that the small data that is reused (activations, residuals,
// RMSNorm weights, routing tables) stays in L2 while gigabytes of weights
// stream past.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// bulk_g2s with an L2 cache policy (see l2_evict_first_policy).
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint4 lds128(const void* p) { return *reinterpret_cast<const uint4*>(p); }

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
