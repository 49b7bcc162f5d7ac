// qmm_kernels.cuh -- the libqmm CUDA kernels (CUDA-core paths):
//   quantize_q8_0 / quantize_q4_0 / repack / swiglu+quantize   (set-up and a1, a8)
//   rows kernel: batch-1 GEMV and small-batch GEMM with dp4a   (a2-a6)
//   MoE grouping, expert-grouped GEMV and combine              (a7)
//   per-block debug dots
//
// Method: llama.cpp guide (kenji.blog/id) section 2.2; Q4_0 block format:
// TinyLLaMA C++ guide (kenji.blog) section 6.1; Q8_0-style activations and
// the routed-expert MoE: Colibri page (kerneldigest.dev), "Arquitectura del
// Sistema"; SwiGLU: TinyLLaMA guide section 4.4.
#pragma once

#include <climits>

#include "qmm_device.cuh"

namespace qmm {

// ============================================================================
// Quantizers
// ============================================================================

// Codes of one block spread over 8 lanes (4 values each).  qmax 127 (Q8_0)
// or 7 (Q4_0); codes are clamped to [qlo, qmax].
struct Quad {
    int c[4];
    float d32;
};

// Correctly rounded x / d (IEEE round to nearest) from r = RN(1/d): the
// first quotient RN(x * r) is within one ulp of x / d, the FMA gives the
// exact remainder x - q0 * d, and one more FMA lands on RN(x / d)
// (Markstein's theorem on division by FMA, as in the Handbook of
// Floating-Point Arithmetic, ch. 5).  Valid for finite normal operands
// without overflow; callers fall back to __fdiv_rn outside that range.
__device__ __forceinline__ float div_rn_fma(float x, float d, float r) {
    const float q0 = __fmul_rn(x, r);
    const float rem = __fmaf_rn(-q0, d, x);
    return __fmaf_rn(rem, r, q0);
}

// The code of one value: round-half-away of RN(v / d32), clamped.  fast:
// d32 inside the range where div_rn_fma with rc = RN(1/d32) is exact.
__device__ __forceinline__ int code_of(float v, float d32, float rc, bool fast, bool nonzero, float qmax, float qlo) {
    if (!nonzero) return 0;
    const float qf = fast ? div_rn_fma(v, d32, rc) : __fdiv_rn(v, d32);
    return (int)fminf(fmaxf(roundf(qf), qlo), qmax);
}

// Codes and scale of one block whose values v[] sit in this lane (the
// block's amax a already reduced over its lanes).  When every lane of the
// warp has a == 0 or a in [1e-28, 1e30] -- always, for finite activations and
// weights of sane magnitude -- the scale is RN(a / qmax) by the FMA-corrected
// quotient with the constant RN(1/qmax) (folded: qmax is a literal at every
// call), each quotient RN(v / d32) by div_rn_fma, and the rounding is
// floor(fl(|q| + 1/2)) for |q| >= 1/2, 0 below, which equals round-half-away
// for every float (checked exhaustively over [0, 256)), with no branch per
// value.  Otherwise the general path with the IEEE division.
template <int NV>
__device__ __forceinline__ void block_codes(const float (&v)[NV], float a, float qmax, float qlo, int (&c)[NV],
                                            float& d32) {
    const bool ok = a == 0.0f || (a >= 1.0e-28f && a <= 1.0e30f);
    if (__all_sync(FULL, ok)) {
        d32 = div_rn_fma(a, qmax, 1.0f / qmax);  // a == 0 gives 0
        const float rc = __frcp_rn(a == 0.0f ? 1.0f : d32);
        const int kpos = (int)qmax, kneg = (int)(-qlo);
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const float qf = div_rn_fma(v[i], d32, rc);
            const float aq = fabsf(qf);
            const int k = aq < 0.5f ? 0 : __float2int_rd(__fadd_rn(aq, 0.5f));
            const int cv = qf < 0.0f ? -min(k, kneg) : min(k, kpos);
            c[i] = a == 0.0f ? 0 : cv;
        }
    } else {
        d32 = __fdiv_rn(a, qmax);
        // d32 in [2^-100, 1e30] keeps 1/d32 and every quotient (|x/d32| <= qmax) in range
        const bool fast = d32 >= 7.8886091e-31f && d32 <= 1.0e30f;
        const float rc = fast ? __frcp_rn(d32) : 0.f;
#pragma unroll
        for (int i = 0; i < NV; ++i) c[i] = code_of(v[i], d32, rc, fast, a != 0.0f, qmax, qlo);
    }
}

__device__ __forceinline__ Quad quad_codes(float4 v, float qmax, float qlo) {
    float a = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
    a = fmaxf(a, __shfl_xor_sync(FULL, a, 1));
    a = fmaxf(a, __shfl_xor_sync(FULL, a, 2));
    a = fmaxf(a, __shfl_xor_sync(FULL, a, 4));
    Quad r;
    const float vv[4] = {v.x, v.y, v.z, v.w};
    block_codes<4>(vv, a, qmax, qlo, r.c, r.d32);
    return r;
}

// The same with a block spread over 4 lanes of 8 values each (lanes 4k..4k+3).
struct Oct {
    int c[8];
    float d32;
};

__device__ __forceinline__ Oct oct_codes(float4 u, float4 w, float qmax, float qlo) {
    float a = fmaxf(fmaxf(fmaxf(fabsf(u.x), fabsf(u.y)), fmaxf(fabsf(u.z), fabsf(u.w))),
                    fmaxf(fmaxf(fabsf(w.x), fabsf(w.y)), fmaxf(fabsf(w.z), fabsf(w.w))));
    a = fmaxf(a, __shfl_xor_sync(FULL, a, 1));
    a = fmaxf(a, __shfl_xor_sync(FULL, a, 2));
    Oct r;
    const float vv[8] = {u.x, u.y, u.z, u.w, w.x, w.y, w.z, w.w};
    block_codes<8>(vv, a, qmax, qlo, r.c, r.d32);
    return r;
}

// x [M][K] fp32 -> q [M][K] int8, d [M][B] fp16 bits.  Each warp handles 4
// blocks per step (8 lanes per block, one float4 per lane).
__global__ void quantize_q8_0_kernel(const float* __restrict__ x, int64_t M, int64_t K, int64_t ldx,
                                     int8_t* __restrict__ q, uint16_t* __restrict__ d) {
    // launched after the kernel that writes the input, possibly early
    // (programmatic dependent launch): nothing is read before it completes
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t B = K / QK;
    const int64_t nblk = M * B;
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t g = warp; g * 4 < nblk; g += nwarps) {
        const int64_t blk = g * 4 + (lane >> 3);
        const bool valid = blk < nblk;
        int64_t m = 0, b = 0;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (valid) {
            m = blk / B;
            b = blk - m * B;
            v = *reinterpret_cast<const float4*>(x + m * ldx + b * QK + (lane & 7) * 4);
        }
        Quad r = quad_codes(v, 127.0f, -127.0f);
        if (valid) {
            int packed = (r.c[0] & 0xff) | ((r.c[1] & 0xff) << 8) | ((r.c[2] & 0xff) << 16) | ((r.c[3] & 0xff) << 24);
            *reinterpret_cast<int*>(q + m * K + b * QK + (lane & 7) * 4) = packed;
            if ((lane & 7) == 0) d[m * B + b] = f32_to_f16_bits(r.d32);
        }
    }
}

// SwiGLU(gate, up) then Q8_0, row by row; optional fp32 h out.
__global__ void swiglu_quantize_kernel(const float* __restrict__ gate, const float* __restrict__ up, int64_t rows,
                                       int64_t K, int64_t ld, int8_t* __restrict__ q, uint16_t* __restrict__ d,
                                       float* __restrict__ h_out) {
    // launched after the kernel that writes the input, possibly early
    // (programmatic dependent launch): nothing is read before it completes
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t B = K / QK;
    const int64_t nblk = rows * B;
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t g = warp; g * 4 < nblk; g += nwarps) {
        const int64_t blk = g * 4 + (lane >> 3);
        const bool valid = blk < nblk;
        int64_t m = 0, b = 0;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (valid) {
            m = blk / B;
            b = blk - m * B;
            const int64_t off = m * ld + b * QK + (lane & 7) * 4;
            float4 gg = *reinterpret_cast<const float4*>(gate + off);
            float4 uu = *reinterpret_cast<const float4*>(up + off);
            v = make_float4(swiglu1(gg.x, uu.x), swiglu1(gg.y, uu.y), swiglu1(gg.z, uu.z), swiglu1(gg.w, uu.w));
            if (h_out) *reinterpret_cast<float4*>(h_out + off) = v;
        }
        Quad r = quad_codes(v, 127.0f, -127.0f);
        if (valid) {
            int packed = (r.c[0] & 0xff) | ((r.c[1] & 0xff) << 8) | ((r.c[2] & 0xff) << 16) | ((r.c[3] & 0xff) << 24);
            *reinterpret_cast<int*>(q + m * K + b * QK + (lane & 7) * 4) = packed;
            if ((lane & 7) == 0) d[m * B + b] = f32_to_f16_bits(r.d32);
        }
    }
}

// w [N][K] fp32 -> Q4_0 planes.  Lane i of a block group holds elements
// 4i..4i+3; lanes 0..3 (elements 0..15) pair with lanes 4..7 (16..31) to
// form bytes u[j] | u[j+16] << 4.
__global__ void quantize_q4_0_kernel(const float* __restrict__ w, int64_t N, int64_t K, int64_t ldw,
                                     uint8_t* __restrict__ qs, uint16_t* __restrict__ d) {
    const int64_t B = K / QK;
    const int64_t nblk = N * B;
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t g = warp; g * 4 < nblk; g += nwarps) {
        const int64_t blk = g * 4 + (lane >> 3);
        const bool valid = blk < nblk;
        int64_t n = 0, b = 0;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (valid) {
            n = blk / B;
            b = blk - n * B;
            v = *reinterpret_cast<const float4*>(w + n * ldw + b * QK + (lane & 7) * 4);
        }
        Quad r = quad_codes(v, 7.0f, -8.0f);
        unsigned u = (unsigned)(r.c[0] + 8) | ((unsigned)(r.c[1] + 8) << 8) | ((unsigned)(r.c[2] + 8) << 16) |
                     ((unsigned)(r.c[3] + 8) << 24);
        unsigned hi = __shfl_down_sync(FULL, u, 4);
        if (valid && (lane & 7) < 4) {
            *reinterpret_cast<unsigned*>(qs + blk * 16 + (lane & 7) * 4) = u | (hi << 4);
            if ((lane & 7) == 0) d[blk] = f32_to_f16_bits(r.d32);
        }
    }
}

// Page-format 18-byte blocks -> planes.  One thread per block.
__global__ void repack_q4_0_kernel(const uint8_t* __restrict__ blocks, int64_t nblk, uint8_t* __restrict__ qs,
                                   uint16_t* __restrict__ d) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nblk; i += (int64_t)gridDim.x * blockDim.x) {
        const uint8_t* src = blocks + i * 18;
        d[i] = (uint16_t)(src[0] | (src[1] << 8));
        unsigned wds[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            wds[k] = (unsigned)src[2 + 4 * k] | ((unsigned)src[3 + 4 * k] << 8) | ((unsigned)src[4 + 4 * k] << 16) |
                     ((unsigned)src[5 + 4 * k] << 24);
        *reinterpret_cast<uint4*>(qs + i * 16) = make_uint4(wds[0], wds[1], wds[2], wds[3]);
    }
}

// ============================================================================
// Rows kernel: y[m][n] = sum_b d_w * d_x * dot over a row tile, with the
// activation block(s) staged in shared memory and weights streamed with
// 16-byte loads.  One warp per row; lane l takes blocks l, l+32, ...
// ============================================================================

// Shared-memory image of MT activation rows over Bc blocks: 16-byte halves
// of each block in two planes (so a warp's 16-byte reads are contiguous and
// bank-conflict free), the fp32 scale and the block's code sum.
struct XTile {
    int4* lo;
    int4* hi;
    int2* sc;  // (fp32 bits of the scale, sum of the block's codes): one 8-byte read
};

__device__ __forceinline__ XTile xtile_at(void* smem, int MT, int Bc) {
    XTile t;
    t.lo = reinterpret_cast<int4*>(smem);
    t.hi = t.lo + MT * Bc;
    t.sc = reinterpret_cast<int2*>(t.hi + MT * Bc);
    return t;
}

__host__ __device__ constexpr int xtile_bytes_per_block() { return 16 + 16 + 4 + 4; }

__device__ __forceinline__ int block_qsum(int4 lo, int4 hi) {
    const int ones = 0x01010101;
    int s = 0;
    s = __dp4a(lo.x, ones, s);
    s = __dp4a(lo.y, ones, s);
    s = __dp4a(lo.z, ones, s);
    s = __dp4a(lo.w, ones, s);
    s = __dp4a(hi.x, ones, s);
    s = __dp4a(hi.y, ones, s);
    s = __dp4a(hi.z, ones, s);
    s = __dp4a(hi.w, ones, s);
    return s;
}

// Copy Q8_0 rows into the tile: tile row t <- activation row xrow[t]
// (xrow[t] < 0: zero fill).  Blocks [b0, b0 + nb).  Whole CTA.
template <int MT>
__device__ __forceinline__ void stage_q8(const XTile& xt, int Bc, const int8_t* __restrict__ xq,
                                         const uint16_t* __restrict__ xd, int64_t K, const int64_t* xrow, int b0,
                                         int nb, int tid, int nthr) {
    const int64_t B = K / QK;
    for (int i = tid; i < MT * Bc; i += nthr) {
        const int t = i / Bc, b = i - t * Bc;
        // xrow[t] by a select over the unrolled entries: a run-time index
        // would put the array in local memory
        int64_t row = -1;
#pragma unroll
        for (int tt = 0; tt < MT; ++tt)
            if (tt == t) row = xrow[tt];
        int4 lo = make_int4(0, 0, 0, 0), hi = lo;
        float s = 0.f;
        if (row >= 0 && b < nb) {
            const int8_t* src = xq + row * K + (int64_t)(b0 + b) * QK;
            lo = *reinterpret_cast<const int4*>(src);
            hi = *reinterpret_cast<const int4*>(src + 16);
            s = f16_bits_to_f32(xd[row * B + b0 + b]);
        }
        xt.lo[i] = lo;
        xt.hi[i] = hi;
        xt.sc[i] = make_int2(__float_as_int(s), block_qsum(lo, hi));
    }
}

// RMSNorm factor of one vector (TinyLLaMA guide 4.1): 1 / sqrt(mean(x^2) +
// eps).  The sum of squares is taken in one fixed order for a given thread
// count -- each thread sums x[tid], x[tid + nthr], ...; then each warp; then
// thread 0 adds the warp partials in warp order -- so every CTA normalizing
// the same vector with the same thread count gets the same factor.  Threads
// [0, nthr) take part (nthr % 32 == 0, <= 1024), synchronised with named
// barrier `bar`; red: 33 floats of shared memory.  Coherent loads (x may have
// been written by another SM of the same or the preceding launch).
__device__ __forceinline__ float rms_inv(const float* x, int64_t K, float eps, float* red, int tid, int nthr,
                                         int bar) {
    float s = 0.f;
    for (int64_t i = tid; i < K; i += nthr) {
        const float v = __ldcg(x + i);
        s = __fmaf_rn(v, v, s);
    }
    s = warp_sum(s);
    if ((tid & 31) == 0) red[tid >> 5] = s;
    asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(nthr) : "memory");
    if (tid == 0) {
        float t = 0.f;
        for (int w = 0; w < nthr / 32; ++w) t = __fadd_rn(t, red[w]);
        red[32] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(t, (float)K), eps)));
    }
    asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(nthr) : "memory");
    return red[32];
}

// Quantize one fp32 activation row (K values; or SwiGLU of gate = x[0..K),
// up = x[K..2K)) straight into tile row 0.  With gamma, the row is first
// normalized: x_i * inv * gamma_i (inv from rms_inv), each product rounded
// to fp32.  CTA 0 also writes the Q8_0 result out when xq_out/xd_out are
// given.  Whole CTA; blockDim % 32 == 0.  Coherent loads.
template <bool GATE_UP>
__device__ __forceinline__ void stage_f32(const XTile& xt, const float* __restrict__ x, int64_t K,
                                          int8_t* __restrict__ xq_out, uint16_t* __restrict__ xd_out, int tid,
                                          int nthr, const float* gamma = nullptr, float inv = 1.0f);

// RMSNorm + Q8_0 of one activation row into tile row 0 (TinyLLaMA guide
// 4.1), for rows of at most RMS_STEPS * nthr / 4 blocks (each block on 4
// lanes of 8 values): the gamma values a thread needs are loaded first
// (rms_gamma_load -- they do not depend on the activation, so a kernel loads
// them before it waits for the producer of x); then every x value is loaded
// once into registers, the sum of squares is taken from the registers in a
// fixed order (each lane over its values, then butterfly within the warp,
// then the warps in order).  The codes are those of z_i = x_i * gamma_i (a
// block's codes are the same for any positive multiple of it), formed while
// warp 0 forms 1/rms; each block's scale is then d_z * 1/rms.  Longer rows
// take rms_inv + stage_f32 (two passes).  Threads [0, nthr) of the CTA,
// named barriers bar (by the caller), bar+1 and bar+2; red: 33 floats of
// shared memory.  CTA 0 writes the Q8_0 row out when xq_out/xd_out are given.
constexpr int RMS_STEPS = 2;  // blocks per thread group of 4 in the one-pass staging

struct RmsGamma {
    float4 g[2 * RMS_STEPS];
};

// One pass when every block has its 4 lanes: K / 32 <= RMS_STEPS * nthr / 4.
__device__ __forceinline__ bool rms_one_pass(int64_t K, int nthr) { return K / QK <= RMS_STEPS * (nthr >> 2); }

// Thread t takes, in step i, values 8p..8p+7 (p = t & 3) of block
// i * nthr/4 + t/4.
__device__ __forceinline__ RmsGamma rms_gamma_load(const float* gamma, int64_t K, int tid, int nthr) {
    RmsGamma r;
    const int B = (int)(K / QK);
    const int p = tid & 3;
#pragma unroll
    for (int i = 0; i < RMS_STEPS; ++i) {
        const int b = i * (nthr >> 2) + (tid >> 2);
        const bool in = b < B && rms_one_pass(K, nthr);
        const float* g = gamma + (int64_t)b * QK + p * 8;
        r.g[2 * i] = in ? __ldg(reinterpret_cast<const float4*>(g)) : make_float4(0.f, 0.f, 0.f, 0.f);
        r.g[2 * i + 1] = in ? __ldg(reinterpret_cast<const float4*>(g + 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    return r;
}

// The one-pass staging once this thread's values are in registers: v[2i],
// v[2i+1] hold values 8p..8p+7 (p = tid & 3) of block i * nthr/4 + tid/4
// (zero past the row).
__device__ __forceinline__ void stage_rmsnorm_regs(const XTile& xt, const float4 (&v)[2 * RMS_STEPS],
                                                   const RmsGamma& gr, int64_t K, float eps, int8_t* xq_out,
                                                   uint16_t* xd_out, float* red, int tid, int nthr, int bar) {
    const int B = (int)(K / QK);
    const int lane = tid & 31, warp = tid >> 5, nwarps = nthr >> 5;
    const int p = tid & 3;
    const bool writer = blockIdx.x == 0 && blockIdx.y == 0;
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 2 * RMS_STEPS; ++i) {
        ss = __fmaf_rn(v[i].x, v[i].x, ss);
        ss = __fmaf_rn(v[i].y, v[i].y, ss);
        ss = __fmaf_rn(v[i].z, v[i].z, ss);
        ss = __fmaf_rn(v[i].w, v[i].w, ss);
    }
    ss = warp_sum(ss);
    // The sum of squares goes to warp 0 over barrier bar+1 while the other
    // warps go on: warp 0 waits for every partial, forms 1/rms and publishes
    // it over barrier bar+2, which the others wait on only at the end.
    if (lane == 0) red[warp] = ss;
    __threadfence_block();
    if (warp == 0) {
        asm volatile("bar.sync %0, %1;" ::"r"(bar + 1), "r"(nthr) : "memory");
        if (lane == 0) {
            float t = 0.f;
            for (int w = 0; w < nwarps; ++w) t = __fadd_rn(t, red[w]);
            red[32] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(t, (float)K), eps)));
        }
        __threadfence_block();
        asm volatile("bar.arrive %0, %1;" ::"r"(bar + 2), "r"(nthr) : "memory");
    } else {
        asm volatile("bar.arrive %0, %1;" ::"r"(bar + 1), "r"(nthr) : "memory");
    }
    // Q8_0 codes of z = x (.) gamma: a block's codes do not change when all of
    // its values are scaled by 1/rms, so they are formed before 1/rms is
    // known; only the block scales wait for it (d = d_z * 1/rms).
    float dz[RMS_STEPS];
    int sz[RMS_STEPS];
#pragma unroll
    for (int i = 0; i < RMS_STEPS; ++i) {
        dz[i] = 0.f;
        sz[i] = 0;
        if (i * (nthr >> 2) >= B) break;  // uniform: no block of this step exists
        const int b = i * (nthr >> 2) + (tid >> 2);
        const float4 g0 = gr.g[2 * i], g1 = gr.g[2 * i + 1];
        const float4 u = make_float4(__fmul_rn(v[2 * i].x, g0.x), __fmul_rn(v[2 * i].y, g0.y),
                                     __fmul_rn(v[2 * i].z, g0.z), __fmul_rn(v[2 * i].w, g0.w));
        const float4 w = make_float4(__fmul_rn(v[2 * i + 1].x, g1.x), __fmul_rn(v[2 * i + 1].y, g1.y),
                                     __fmul_rn(v[2 * i + 1].z, g1.z), __fmul_rn(v[2 * i + 1].w, g1.w));
        const Oct r = oct_codes(u, w, 127.0f, -127.0f);
        const int w0 = (r.c[0] & 0xff) | ((r.c[1] & 0xff) << 8) | ((r.c[2] & 0xff) << 16) | ((r.c[3] & 0xff) << 24);
        const int w1 = (r.c[4] & 0xff) | ((r.c[5] & 0xff) << 8) | ((r.c[6] & 0xff) << 16) | ((r.c[7] & 0xff) << 24);
        int sum = r.c[0] + r.c[1] + r.c[2] + r.c[3] + r.c[4] + r.c[5] + r.c[6] + r.c[7];
        sum += __shfl_xor_sync(FULL, sum, 1);
        sum += __shfl_xor_sync(FULL, sum, 2);
        dz[i] = r.d32;
        sz[i] = sum;
        if (b < B) {
            int2* plane = reinterpret_cast<int2*>(p < 2 ? &xt.lo[b] : &xt.hi[b]);
            plane[p & 1] = make_int2(w0, w1);
            if (writer && xq_out) *reinterpret_cast<int2*>(xq_out + (int64_t)b * QK + p * 8) = make_int2(w0, w1);
        }
    }
    if (warp != 0) asm volatile("bar.sync %0, %1;" ::"r"(bar + 2), "r"(nthr) : "memory");
    const float inv = red[32];
#pragma unroll
    for (int i = 0; i < RMS_STEPS; ++i) {
        const int b = i * (nthr >> 2) + (tid >> 2);
        if (b < B && p == 0) {
            const unsigned short h = f32_to_f16_bits(__fmul_rn(dz[i], inv));
            xt.sc[b] = make_int2(__float_as_int(f16_bits_to_f32(h)), sz[i]);
            if (writer && xd_out) xd_out[b] = h;
        }
    }
}

__device__ __forceinline__ void stage_f32_rmsnorm(const XTile& xt, const float* x, const float* gamma,
                                                  const RmsGamma& gr, int64_t K, float eps, int8_t* xq_out,
                                                  uint16_t* xd_out, float* red, int tid, int nthr, int bar) {
    const int B = (int)(K / QK);
    if (!rms_one_pass(K, nthr)) {
        const float inv = rms_inv(x, K, eps, red, tid, nthr, bar);
        stage_f32<false>(xt, x, K, xq_out, xd_out, tid, nthr, gamma, inv);
        return;
    }
    const int p = tid & 3;
    float4 v[2 * RMS_STEPS];
#pragma unroll
    for (int i = 0; i < RMS_STEPS; ++i) {
        const int b = i * (nthr >> 2) + (tid >> 2);
        const float* xb = x + (int64_t)b * QK + p * 8;
        v[2 * i] = b < B ? __ldcg(reinterpret_cast<const float4*>(xb)) : make_float4(0.f, 0.f, 0.f, 0.f);
        v[2 * i + 1] = b < B ? __ldcg(reinterpret_cast<const float4*>(xb + 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    stage_rmsnorm_regs(xt, v, gr, K, eps, xq_out, xd_out, red, tid, nthr, bar);
}

// Each warp of stage_f32 takes 4 blocks per step (8 lanes per block, one
// float4 per lane); STAGE_STEPS steps are loaded before any is quantized, so
// the activation costs one memory round trip per STAGE_STEPS * nwarps * 4
// blocks.  This quantizes one round: v[i] holds values part*4..part*4+3
// (part = lane & 7) of block (g0 + i * nwarps) * 4 + lane / 8.
constexpr int STAGE_STEPS = 8;

__device__ __forceinline__ void stage_f32_quantize(const XTile& xt, const float4 (&v)[STAGE_STEPS], int g0, int B,
                                                   int8_t* __restrict__ xq_out, uint16_t* __restrict__ xd_out,
                                                   int lane, int nwarps) {
    const int part = lane & 7;  // which 4 values of the block
    const bool writer = blockIdx.x == 0 && blockIdx.y == 0;
#pragma unroll
    for (int i = 0; i < STAGE_STEPS; ++i) {
        const int g = g0 + i * nwarps;
        if (g * 4 >= B) break;  // warp-uniform
        const int b = g * 4 + (lane >> 3);
        const bool valid = b < B;
        Quad r = quad_codes(v[i], 127.0f, -127.0f);
        const int packed =
            (r.c[0] & 0xff) | ((r.c[1] & 0xff) << 8) | ((r.c[2] & 0xff) << 16) | ((r.c[3] & 0xff) << 24);
        int s = r.c[0] + r.c[1] + r.c[2] + r.c[3];
        s += __shfl_xor_sync(FULL, s, 1);
        s += __shfl_xor_sync(FULL, s, 2);
        s += __shfl_xor_sync(FULL, s, 4);
        if (valid) {
            int* plane = reinterpret_cast<int*>(part < 4 ? &xt.lo[b] : &xt.hi[b]);
            plane[part & 3] = packed;
            if (part == 0) {
                const unsigned short h = f32_to_f16_bits(r.d32);
                xt.sc[b] = make_int2(__float_as_int(f16_bits_to_f32(h)), s);
                if (writer && xd_out) xd_out[b] = h;
            }
            if (writer && xq_out) *reinterpret_cast<int*>(xq_out + (int64_t)b * QK + part * 4) = packed;
        }
    }
}

template <bool GATE_UP>
__device__ __forceinline__ void stage_f32(const XTile& xt, const float* __restrict__ x, int64_t K,
                                          int8_t* __restrict__ xq_out, uint16_t* __restrict__ xd_out, int tid,
                                          int nthr, const float* gamma, float inv) {
    const int B = (int)(K / QK);
    const int lane = tid & 31;
    const int warp = tid >> 5, nwarps = nthr >> 5;
    const int part = lane & 7;  // which 4 values of the block
    for (int g0 = warp; g0 * 4 < B; g0 += nwarps * STAGE_STEPS) {
        float4 v[STAGE_STEPS];
#pragma unroll
        for (int i = 0; i < STAGE_STEPS; ++i) {
            const int b = (g0 + i * nwarps) * 4 + (lane >> 3);
            v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (b < B) {
                const int64_t off = (int64_t)b * QK + part * 4;
                v[i] = __ldcg(reinterpret_cast<const float4*>(x + off));
                if (GATE_UP) {
                    const float4 u = __ldcg(reinterpret_cast<const float4*>(x + K + off));
                    v[i] = make_float4(swiglu1(v[i].x, u.x), swiglu1(v[i].y, u.y), swiglu1(v[i].z, u.z),
                                       swiglu1(v[i].w, u.w));
                } else if (gamma) {
                    const float4 g = __ldg(reinterpret_cast<const float4*>(gamma + off));
                    v[i] = make_float4(__fmul_rn(__fmul_rn(v[i].x, inv), g.x), __fmul_rn(__fmul_rn(v[i].y, inv), g.y),
                                       __fmul_rn(__fmul_rn(v[i].z, inv), g.z), __fmul_rn(__fmul_rn(v[i].w, inv), g.w));
                }
            }
        }
        stage_f32_quantize(xt, v, g0, B, xq_out, xd_out, lane, nwarps);
    }
}

// Accumulate one weight row against MT staged activation rows, blocks
// [0, nb) of the tile (weight blocks wq/wd already offset to the tile's b0).
template <int MT>
__device__ __forceinline__ void row_accumulate(const XTile& xt, int Bc, const uint8_t* __restrict__ wq,
                                               const uint16_t* __restrict__ wd, int nb, int lane, float (&acc)[MT]) {
    constexpr int U = 4;
    int b = lane;
    for (; b + 32 * (U - 1) < nb; b += 32 * U) {
        uint4 w[U];
        float dw[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            w[u] = ld_stream_v4(wq + (int64_t)(b + 32 * u) * 16);
            dw[u] = f16_bits_to_f32(ld_stream_u16(wd + b + 32 * u));
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int bb = b + 32 * u;
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                const int i = t * Bc + bb;
                const int2 sc = xt.sc[i];
                const int dot = block_dot_u(w[u], xt.lo[i], xt.hi[i]) - 8 * sc.y;
                acc[t] = fmaf(dw[u] * __int_as_float(sc.x), (float)dot, acc[t]);
            }
        }
    }
    for (; b < nb; b += 32) {
        const uint4 w = ld_stream_v4(wq + (int64_t)b * 16);
        const float dw = f16_bits_to_f32(ld_stream_u16(wd + b));
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            const int i = t * Bc + b;
            const int2 sc = xt.sc[i];
            const int dot = block_dot_u(w, xt.lo[i], xt.hi[i]) - 8 * sc.y;
            acc[t] = fmaf(dw * __int_as_float(sc.x), (float)dot, acc[t]);
        }
    }
}

enum XMode { X_Q8 = 0, X_F32 = 1, X_SWIGLU = 2 };

struct RowsArgs {
    const uint8_t* qs;
    const uint16_t* d;
    int64_t N, K;
    int64_t M;          // tokens
    const int8_t* xq;   // X_Q8
    const uint16_t* xd;
    const float* xf;    // X_F32 / X_SWIGLU (M == 1)
    const float* residual;  // optional, added to y (fp32 modes, M == 1)
    int8_t* xq_out;     // optional Q8_0 copy of the activation (fp32 modes)
    uint16_t* xd_out;
    float* y;
    int64_t ldy;
    int chunk_blocks;   // Bc: blocks of K staged at once
};

constexpr int ROWS_THREADS = 256;
constexpr int ROWS_WARPS = ROWS_THREADS / 32;

// Grid: x = row tiles (ROWS_WARPS rows each, grid-stride), y = token groups
// of MT.  Dynamic shared memory: MT * Bc * 40 bytes.
template <int MT, int XMODE>
__global__ void __launch_bounds__(ROWS_THREADS) rows_kernel(RowsArgs a) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    // Let a dependent launch (programmatic stream serialization) start its
    // prologue; it still waits for this grid before touching our outputs.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    const int Bc = a.chunk_blocks;
    const XTile xt = xtile_at(smem_raw, MT, Bc);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t B = a.K / QK;
    const int nchunks = (int)((B + Bc - 1) / Bc);
    const int64_t m0 = (int64_t)blockIdx.y * MT;
    int64_t xrow[MT];
#pragma unroll
    for (int t = 0; t < MT; ++t) xrow[t] = (m0 + t < a.M) ? m0 + t : -1;

    // The activation is produced by the preceding kernel: wait for it.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (nchunks == 1) {
        if (XMODE == X_Q8) stage_q8<MT>(xt, Bc, a.xq, a.xd, a.K, xrow, 0, (int)B, threadIdx.x, blockDim.x);
        else stage_f32<XMODE == X_SWIGLU>(xt, a.xf, a.K, a.xq_out, a.xd_out, threadIdx.x, blockDim.x);
        __syncthreads();
    }
    const int64_t ntiles = (a.N + ROWS_WARPS - 1) / ROWS_WARPS;
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        const int64_t row = tile * ROWS_WARPS + warp;
        float acc[MT];
#pragma unroll
        for (int t = 0; t < MT; ++t) acc[t] = 0.f;
        for (int c = 0; c < nchunks; ++c) {
            const int b0 = c * Bc;
            const int nb = (int)min((int64_t)Bc, B - b0);
            if (nchunks > 1) {
                __syncthreads();
                stage_q8<MT>(xt, Bc, a.xq, a.xd, a.K, xrow, b0, nb, threadIdx.x, blockDim.x);
                __syncthreads();
            }
            if (row < a.N) row_accumulate<MT>(xt, Bc, a.qs + (row * B + b0) * 16, a.d + row * B + b0, nb, lane, acc);
        }
        if (row < a.N) {
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                float v = warp_sum(acc[t]);
                if (lane == 0 && xrow[t] >= 0) {
                    if (XMODE != X_Q8 && a.residual) v += a.residual[row];
                    a.y[xrow[t] * a.ldy + row] = v;
                }
            }
        }
    }
}

// ============================================================================
// Debug: per-block integer dots with the same unpack/dot code.
// ============================================================================
__global__ void block_dots_kernel(const uint8_t* __restrict__ qs, int64_t N, int64_t K, int64_t M,
                                  const int8_t* __restrict__ xq, int32_t* __restrict__ dots) {
    const int64_t B = K / QK;
    const int64_t total = M * N * B;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t b = i % B, n = (i / B) % N, m = i / (B * N);
        const uint4 w = *reinterpret_cast<const uint4*>(qs + (n * B + b) * 16);
        const int4 lo = *reinterpret_cast<const int4*>(xq + m * K + b * QK);
        const int4 hi = *reinterpret_cast<const int4*>(xq + m * K + b * QK + 16);
        dots[i] = block_dot_u(w, lo, hi) - 8 * block_qsum(lo, hi);
    }
}

// ============================================================================
// MoE: group slots by expert, expert-grouped rows kernel, combine.
// ============================================================================

// Workspace (int32 words): counts[E] | offsets[E+1] | cursor[E] | active[E]
// | n_active[1] | slot_list[T*k].  counts and offsets are per expert id;
// active[i] is the i-th routed expert (ascending id), cursor[i] the start of
// its slots in slot_list (i < n_active; its end is cursor[i + 1], or
// offsets[E] for the last), so a kernel can read its routing in one round
// of independent loads.
struct MoeWs {
    int* counts;
    int* offsets;
    int* cursor;
    int* active;
    int* n_active;
    int* slots;
};

__host__ __device__ inline MoeWs moe_ws(void* base, int E) {
    MoeWs w;
    w.counts = reinterpret_cast<int*>(base);
    w.offsets = w.counts + E;
    w.cursor = w.offsets + E + 1;
    w.active = w.cursor + E;
    w.n_active = w.active + E;
    w.slots = w.n_active + 1;
    return w;
}

__host__ __device__ inline size_t moe_ws_bytes(int E, int64_t nslots) {
    size_t words = (size_t)E * 4 + 2 + (size_t)nslots;
    return (words * 4 + 15) / 16 * 16;
}

// One CTA.  Counting sort of slots by expert id; slots inside one expert's
// list come out in any order (each slot's output is computed on its own,
// so the order does not change any result).
constexpr int GROUP_THREADS = 1024;

// The whole block builds the tables.  ids may have been written earlier in
// the same kernel by this block (plain loads after a block barrier).  The
// counts and cursors live in shared memory while the sort runs (up to
// GROUP_SMEM_E experts; beyond that in the workspace itself), so the only
// global-memory traffic is the final tables, written once.
constexpr int GROUP_SMEM_E = 2048;

// Few slots (one token's top-k, up to 32): each thread derives the tables of
// its experts directly from the slot ids -- counts, offsets and active
// positions by comparing against every slot -- with no scan, no atomics and
// two block barriers.  Slots of one expert keep their slot order.
constexpr int GROUP_FEW = 32;

// The tables of a few slots (nslots <= GROUP_FEW) built from their ids by
// the whole block: warp 0 holds one slot per lane and finds, with warp
// intrinsics, each slot's first occurrence and its place in the slot list;
// then every thread derives the counts, offsets and active position of its
// experts by comparing against the slots (fixed-trip, unrolled).  Every
// word the workspace layout defines is written.  f_id / f_first: GROUP_FEW
// ints of shared memory each.
__device__ __forceinline__ void moe_group_few_tables(const int32_t* ids, int nslots, int E, MoeWs w, int* f_id,
                                                     int* f_first, int* err) {
    if (threadIdx.x < 32) {
        const int s = threadIdx.x;
        int e = s < nslots ? ids[s] : -1;
        if (s < nslots && (e < 0 || e >= E)) {
            atomicOr(err, ERR_BAD_EXPERT);
            e = -1;
        }
        const unsigned same = __match_any_sync(FULL, e);
        const bool first = e >= 0 && (__ffs(same) - 1) == s;
        f_id[s] = e;
        f_first[s] = first ? 1 : 0;
        // place in the slot list: every valid slot of a lower expert, then the
        // earlier slots of the same expert
        int pos = __popc(same & ((1u << s) - 1u));
#pragma unroll
        for (int t = 0; t < GROUP_FEW; ++t) {
            const int v = __shfl_sync(FULL, e, t);
            pos += v >= 0 && v < e;
        }
        if (e >= 0) w.slots[pos] = s;
    }
    __syncthreads();
    for (int e = threadIdx.x; e <= E; e += blockDim.x) {
        int cnt = 0, below = 0, dist_below = 0;
#pragma unroll
        for (int t = 0; t < GROUP_FEW; ++t) {
            const int v = f_id[t];  // -1 past nslots
            cnt += v == e;
            below += v >= 0 && v < e;
            dist_below += f_first[t] && v < e;
        }
        if (e == E) {  // every valid slot, every routed expert
            w.offsets[E] = below;
            *w.n_active = dist_below;
            continue;
        }
        w.offsets[e] = below;
        w.counts[e] = cnt;
        if (cnt > 0) {
            w.active[dist_below] = e;
            w.cursor[dist_below] = below;
        }
    }
}

__device__ __forceinline__ void moe_group_few(const int32_t* ids, int nslots, int E, MoeWs w, int* err) {
    __shared__ int f_id[GROUP_FEW];     // slot id, or -1 (none, or an id outside [0, E))
    __shared__ int f_first[GROUP_FEW];  // 1 if no earlier slot has the same id
    moe_group_few_tables(ids, nslots, E, w, f_id, f_first, err);
}

__device__ __forceinline__ void moe_group_block(const int32_t* ids, int nslots, int E, MoeWs w, int* err) {
    if (nslots <= GROUP_FEW) {
        moe_group_few(ids, nslots, E, w, err);
        return;
    }
    __shared__ int s_cnt[GROUP_SMEM_E];
    __shared__ int s_cur[GROUP_SMEM_E];
    const bool in_smem = E <= GROUP_SMEM_E;
    int* cnt = in_smem ? s_cnt : w.counts;
    int* cur = in_smem ? s_cur : w.cursor;
    for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    for (int s = threadIdx.x; s < nslots; s += blockDim.x) {
        const int e = ids[s];
        if (e < 0 || e >= E) {
            atomicOr(err, ERR_BAD_EXPERT);
            continue;
        }
        atomicAdd(&cnt[e], 1);
    }
    __syncthreads();
    // Exclusive scans of counts (-> offsets) and of (counts > 0) (-> active
    // positions), each thread owning a contiguous chunk of experts.
    const int per = (E + blockDim.x - 1) / blockDim.x;
    const int e0 = min(E, (int)threadIdx.x * per), e1 = min(E, e0 + per);
    int csum = 0, asum = 0;
    for (int e = e0; e < e1; ++e) {
        csum += cnt[e];
        asum += cnt[e] > 0;
    }
    // block-wide exclusive scan of (csum, asum) packed into one 64-bit lane value
    long long v = ((long long)csum << 32) | (unsigned)asum;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    long long incl = v;
    for (int o = 1; o < 32; o <<= 1) {
        long long n = __shfl_up_sync(FULL, incl, o);
        if (lane >= o) incl += n;
    }
    __shared__ long long wsum[32];
    if (lane == 31) wsum[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        long long t = (lane < (int)(blockDim.x >> 5)) ? wsum[lane] : 0;
        for (int o = 1; o < 32; o <<= 1) {
            long long n = __shfl_up_sync(FULL, t, o);
            if (lane >= o) t += n;
        }
        wsum[lane] = t;  // inclusive over warps
    }
    __syncthreads();
    long long excl = incl - v + (wid > 0 ? wsum[wid - 1] : 0);
    int coff = (int)(excl >> 32), aoff = (int)(excl & 0xffffffff);
    for (int e = e0; e < e1; ++e) {
        const int c = cnt[e];
        if (in_smem) w.counts[e] = c;
        w.offsets[e] = coff;
        cur[e] = coff;
        if (c > 0) w.active[aoff++] = e;
        coff += c;
    }
    if (threadIdx.x == blockDim.x - 1) {
        w.offsets[E] = coff;
        *w.n_active = aoff;
    }
    __syncthreads();
    for (int s = threadIdx.x; s < nslots; s += blockDim.x) {
        const int e = ids[s];
        if (e < 0 || e >= E) continue;
        const int pos = atomicAdd(&cur[e], 1);
        w.slots[pos] = s;
    }
    // cursor[i]: the start of the i-th active expert's slots (the sort's own
    // cursors are no longer needed)
    __syncthreads();
    const int na = *w.n_active;
    for (int i = threadIdx.x; i < na; i += blockDim.x) w.cursor[i] = w.offsets[w.active[i]];
}

__global__ void __launch_bounds__(GROUP_THREADS) moe_group_kernel(const int32_t* __restrict__ ids, int nslots, int E,
                                                                  MoeWs w, int* err) {
    // launched after the kernel that writes the input, possibly early
    // (programmatic dependent launch): nothing is read before it completes
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    moe_group_block(ids, nslots, E, w, err);
}

// ----------------------------------------------------------------------------
// Sigmoid top-k router (Colibri page, "Arquitectura del Sistema": a sigmoid
// router picks each token's experts).  Scores s = sigmoid(logit); the k
// largest are kept, ties to the lower expert index, in decreasing order;
// gates are the kept scores divided by their sum.  sigmoid is strictly
// increasing, so the selection compares the logits themselves: no rounding
// enters it.  One warp per token: lane l holds experts l, l+32, l+64, ...
// in registers; each of the k rounds is a lane-local scan of the untaken
// experts followed by a butterfly arg-max (value, then lower index).
// ----------------------------------------------------------------------------
constexpr int ROUTE_MAX_E = 1024;
constexpr int ROUTE_MAX_K = 64;
constexpr int ROUTE_PER_LANE = ROUTE_MAX_E / 32;
constexpr int ROUTE_THREADS = 1024;

// PER_LANE: register slots per lane (E <= 32 * PER_LANE).
template <int PER_LANE = ROUTE_PER_LANE>
__device__ __forceinline__ void route_token(const float* __restrict__ lg, int E, int k, int32_t* ids, float* gates,
                                            int lane) {
    float v[PER_LANE];
    uint32_t taken = 0;  // bit i: expert lane + 32 i is chosen already, or does not exist
    const int nper = (E + 31) >> 5;  // register slots in use
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) {
        const int e = lane + 32 * i;
        v[i] = 0.f;
        if (e < E)
            v[i] = lg[e];
        else
            taken |= 1u << i;
    }
    float ssum = 0.f;
    float keep_s[ROUTE_MAX_K / 32];
    int keep_id[ROUTE_MAX_K / 32];
#pragma unroll
    for (int r = 0; r < ROUTE_MAX_K / 32; ++r) {
        keep_s[r] = 0.f;
        keep_id[r] = 0;
    }
    for (int j = 0; j < k; ++j) {
        float bv = 0.f;
        int bi = INT_MAX;  // none yet
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i) {
            if (i >= nper) break;
            if (!((taken >> i) & 1u) && (bi == INT_MAX || v[i] > bv)) {  // ascending index: ties keep the lower
                bv = v[i];
                bi = lane + 32 * i;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(FULL, bv, o);
            const int oi = __shfl_xor_sync(FULL, bi, o);
            if (oi != INT_MAX && (bi == INT_MAX || ov > bv || (ov == bv && oi < bi))) {
                bv = ov;
                bi = oi;
            }
        }
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        const float s = 1.0f / (1.0f + expf(-bv));
        ssum += s;  // every lane adds the same scores in the same order
#pragma unroll
        for (int r = 0; r < ROUTE_MAX_K / 32; ++r)
            if (j == lane + 32 * r) {
                keep_s[r] = s;
                keep_id[r] = bi;
            }
    }
#pragma unroll
    for (int r = 0; r < ROUTE_MAX_K / 32; ++r) {
        const int j = lane + 32 * r;
        if (j < k) {
            ids[j] = keep_id[r];
            gates[j] = keep_s[r] / ssum;
        }
    }
}

// The same selection and gates for a few tokens (T * k <= GROUP_FEW) and
// E <= 32 * (blockDim.x / 32) experts, with the whole block: per token, warp
// w ranks the logits of experts 32w .. 32w + 31 among themselves (value,
// then lower index) and keeps its best k as candidates; each candidate is
// then ranked among all candidates, and the one of rank j is the token's
// j-th choice.  The k best of every warp hold the k best overall, so for
// finite logits the choice is that of route_token; the gates are formed as
// there (fp32 sigmoid with expf, their sum in choice order, one division
// each).  Every step is a fixed-trip, branch-free loop of independent
// operations (one warp alone runs a dependent chain at a few cycles per
// operation, so trip counts and divisions would cost microseconds).
// ids/gates: [T][k] in shared memory; cand: 2 * 32 * (blockDim.x / 32)
// words of shared memory.  Every thread of the block.
__device__ __forceinline__ void route_few_block(const float* __restrict__ logits, int T, int E, int k, int32_t* ids,
                                                float* gates, int* cand) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (E + 31) >> 5;
    const int nc = nw * k;  // candidate slots: k per warp
    float* cv = reinterpret_cast<float*>(cand);
    int* ci = cand + 32 * (blockDim.x >> 5);
    for (int t = 0; t < T; ++t) {
        // slots a warp with fewer than k experts leaves empty rank last
        for (int c = threadIdx.x; c < nc; c += blockDim.x) {
            cv[c] = -INFINITY;
            ci[c] = INT_MAX;
        }
        __syncthreads();
        if (warp < nw) {
            const int e = 32 * warp + lane;
            const bool valid = e < E;
            const float v = valid ? logits[(int64_t)t * E + e] : -INFINITY;
            const int me = valid ? e : INT_MAX;
            int rank = 0;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float vj = __shfl_sync(FULL, v, j);
                const int ej = __shfl_sync(FULL, me, j);
                rank += (vj > v) | ((vj == v) & (ej < me));
            }
            if (valid && rank < k) {
                cv[warp * k + rank] = v;
                ci[warp * k + rank] = e;
            }
        }
        __syncthreads();
        float sc = 0.f;
        int my = -1;
        if ((int)threadIdx.x < nc) {
            const float v = cv[threadIdx.x];
            const int e = ci[threadIdx.x];
            int r0 = 0, r1 = 0, r2 = 0, r3 = 0;
            int d = 0;
            for (; d + 4 <= nc; d += 4) {
                r0 += (cv[d] > v) | ((cv[d] == v) & (ci[d] < e));
                r1 += (cv[d + 1] > v) | ((cv[d + 1] == v) & (ci[d + 1] < e));
                r2 += (cv[d + 2] > v) | ((cv[d + 2] == v) & (ci[d + 2] < e));
                r3 += (cv[d + 3] > v) | ((cv[d + 3] == v) & (ci[d + 3] < e));
            }
            for (; d < nc; ++d) r0 += (cv[d] > v) | ((cv[d] == v) & (ci[d] < e));
            const int rank = r0 + r1 + r2 + r3;
            if (e != INT_MAX && rank < k) {
                ids[t * k + rank] = e;
                sc = 1.0f / (1.0f + expf(-v));
                gates[t * k + rank] = sc;
                my = rank;
            }
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            float ssum = 0.f;
            for (int j = 0; j < k; ++j) ssum += gates[t * k + j];  // choice order, as route_token
            cv[0] = ssum;
        }
        __syncthreads();
        if (my >= 0) gates[t * k + my] = sc / cv[0];
        __syncthreads();
    }
}

// Routes tokens warp by warp; with group != 0 (one CTA) the same block then
// builds the expert grouping of the chosen ids in w.
__global__ void __launch_bounds__(ROUTE_THREADS) moe_route_kernel(const float* __restrict__ logits, int T, int E,
                                                                  int k, int32_t* ids, float* gates, MoeWs w,
                                                                  int group, int* err) {
    // launched after the kernel that writes the input, possibly early
    // (programmatic dependent launch): nothing is read before it completes
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    if (group && T * k <= GROUP_FEW && E <= (int)blockDim.x) {
        // a decode-size batch: the block-wide top-k, then the grouping, both on
        // the choices in shared memory
        __shared__ int r_ids[GROUP_FEW], r_first[GROUP_FEW];
        __shared__ float r_gates[GROUP_FEW];
        __shared__ int r_cand[2 * ROUTE_THREADS];
        __shared__ int r_fid[GROUP_FEW];
        route_few_block(logits, T, E, k, r_ids, r_gates, r_cand);
        if ((int)threadIdx.x < T * k) {
            ids[threadIdx.x] = r_ids[threadIdx.x];
            gates[threadIdx.x] = r_gates[threadIdx.x];
        }
        moe_group_few_tables(r_ids, T * k, E, w, r_fid, r_first, err);
        return;
    }
    for (int t = blockIdx.x * nw + warp; t < T; t += gridDim.x * nw)
        route_token(logits + (int64_t)t * E, E, k, ids + (int64_t)t * k, gates + (int64_t)t * k, lane);
    if (group) {
        __syncthreads();
        moe_group_block(ids, T * k, E, w, err);
    }
}

struct MoeArgs {
    const uint8_t* qs;
    const uint16_t* d;
    int64_t N, K;
    int E, k;
    const int8_t* xq;
    const uint16_t* xd;
    int x_per_slot;
    float* y;
    MoeWs ws;
    int rows_per_item;  // multiple of ROWS_WARPS
};

// Work item = (active expert a, block of rows_per_item rows).  For each
// group of MT slots routed to the expert: stage their activations, then each
// warp applies its rows (rows_per_item / ROWS_WARPS of them) to all staged
// slots.  The whole K is staged at once (host checks it fits).
template <int MT>
__global__ void __launch_bounds__(ROWS_THREADS) moe_rows_kernel(MoeArgs a) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t B = a.K / QK;
    const int Bc = (int)B;
    const XTile xt = xtile_at(smem_raw, MT, Bc);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t row_blocks = (a.N + a.rows_per_item - 1) / a.rows_per_item;
    const int n_active = *a.ws.n_active;
    const int64_t total = (int64_t)n_active * row_blocks;
    const int64_t e_qs = a.N * B * 16, e_d = a.N * B;
    for (int64_t item = blockIdx.x; item < total; item += gridDim.x) {
        const int ai = (int)(item / row_blocks);
        const int64_t r0 = (item - (int64_t)ai * row_blocks) * a.rows_per_item;
        const int e = a.ws.active[ai];
        const int s_begin = a.ws.offsets[e], s_end = a.ws.offsets[e + 1];
        const uint8_t* qs = a.qs + (int64_t)e * e_qs;
        const uint16_t* dd = a.d + (int64_t)e * e_d;
        for (int s0 = s_begin; s0 < s_end; s0 += MT) {
            int64_t xrow[MT];
            int slot[MT];
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                slot[t] = (s0 + t < s_end) ? a.ws.slots[s0 + t] : -1;
                xrow[t] = slot[t] < 0 ? -1 : (a.x_per_slot ? slot[t] : slot[t] / a.k);
            }
            __syncthreads();
            stage_q8<MT>(xt, Bc, a.xq, a.xd, a.K, xrow, 0, Bc, threadIdx.x, blockDim.x);
            __syncthreads();
            for (int64_t row = r0 + warp; row < min(a.N, r0 + a.rows_per_item); row += ROWS_WARPS) {
                float acc[MT];
#pragma unroll
                for (int t = 0; t < MT; ++t) acc[t] = 0.f;
                row_accumulate<MT>(xt, Bc, qs + row * B * 16, dd + row * B, Bc, lane, acc);
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    const float v = warp_sum(acc[t]);
                    if (lane == 0 && slot[t] >= 0) a.y[(int64_t)slot[t] * a.N + row] = v;
                }
            }
        }
    }
}

// y[t][n] = sum_j g[t][j] * z[t][j][n], j ascending.
__global__ void moe_combine_kernel(const float* __restrict__ z, const float* __restrict__ gates, int T, int k,
                                   int64_t N, float* __restrict__ y) {
    // launched after the kernel that writes the input, possibly early
    // (programmatic dependent launch): nothing is read before it completes
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t total = (int64_t)T * N;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / N, n = i - t * N;
        float acc = 0.f;
        for (int j = 0; j < k; ++j) acc = fmaf(gates[t * k + j], z[(t * k + j) * N + n], acc);
        y[i] = acc;
    }
}

}  // namespace qmm
