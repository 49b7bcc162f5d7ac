// qmm_formats.cu -- weight-format variants of the batch-1 product:
//  - per-row-scale int4 / int2 containers x Q8_0 activations (Colibri page,
//    kerneldigest.dev, "Arquitectura del Sistema": an int4 container with
//    per-row scales; int4 and int2 packing);
//  - Q4_0 weights x fp32 activations by dequantize-then-FMA (TinyLLaMA C++
//    guide, kenji.blog, section 6.2: expand the 4-bit values, multiply by the
//    scale, multiply-add with the fp32 activations).
//
// Container layout (the page gives none; this is the reading taken): row n
// holds K codes u = q + 2^(bits-1), 8/bits per byte, element i in byte
// i*bits/8 at bit (i mod 8/bits)*bits; one fp32 scale per row, delta =
// max|w_row| / (2^(bits-1) - 1), q = clamp(round-half-away(w/delta)).
//
// Both GEMVs are HBM-streaming kernels without a TMA ring: each lane reads one
// 16-byte weight unit per row with a streaming load, four rows per warp at a
// time, so every activation value loaded from shared memory serves four rows.
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <set>
#include <utility>

#include "qmm.h"
#include "qmm_device.cuh"
#include "qmm_internal.h"

namespace qmm {
namespace {

constexpr int FMT_THREADS = 256;
constexpr int FMT_WARPS = FMT_THREADS / 32;
constexpr int FMT_ROWS = 4;   // rows per warp pass
constexpr int FMT_DEPTH = 4;  // 16-byte loads per row in flight per lane (per-row GEMV)
constexpr int FMA_DEPTH = 2;  // the same for the fp32 GEMV (more registers per step)

// round half away from zero; exact for every finite float
__device__ __forceinline__ float round_half_away_f(float v) {
    const float a = fabsf(v);
    const float f = floorf(a);
    return copysignf(a - f >= 0.5f ? f + 1.0f : f, v);
}

__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, o));
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float m = red[0];
    for (int i = 1; i < (int)(blockDim.x >> 5); ++i) m = fmaxf(m, red[i]);
    __syncthreads();
    return m;
}

// ---------------------------------------------------------------------------
// Per-row quantizer: one CTA per row (grid-stride).
// ---------------------------------------------------------------------------
template <int BITS>
__global__ void __launch_bounds__(FMT_THREADS) quantize_rowwise_kernel(const float* __restrict__ w, int64_t N,
                                                                       int64_t K, int64_t ldw,
                                                                       uint8_t* __restrict__ wq, float* __restrict__ ws) {
    constexpr int PER = 8 / BITS;
    constexpr int QMAX = (1 << (BITS - 1)) - 1, QMIN = -(1 << (BITS - 1)), OFF = 1 << (BITS - 1);
    __shared__ float red[FMT_WARPS];
    const int64_t rowb = K / PER;
    for (int64_t n = blockIdx.x; n < N; n += gridDim.x) {
        const float* row = w + n * ldw;
        float amax = 0.0f;
        for (int64_t k = threadIdx.x; k < K; k += blockDim.x) amax = fmaxf(amax, fabsf(row[k]));
        amax = block_max(amax, red);
        const float delta = __fdiv_rn(amax, (float)QMAX);
        for (int64_t j = threadIdx.x; j < rowb; j += blockDim.x) {
            unsigned byte = 0;
#pragma unroll
            for (int i = 0; i < PER; ++i) {
                int r = 0;
                if (amax != 0.0f) {
                    r = (int)round_half_away_f(__fdiv_rn(row[j * PER + i], delta));
                    r = min(max(r, QMIN), QMAX);
                }
                byte |= (unsigned)(r + OFF) << (i * BITS);
            }
            wq[n * rowb + j] = (uint8_t)byte;
        }
        if (threadIdx.x == 0) ws[n] = delta;
    }
}

// ---------------------------------------------------------------------------
// Per-row codes x Q8_0 GEMV.
//
// A 16-byte weight unit holds E = 128/BITS codes (int4: 32 = one activation
// block, int2: 64 = two).  The activation is staged once per CTA, permuted so
// that each masked weight word meets its four activation codes in one dp4a
// operand, in 16-byte chunks laid out chunk-major ([chunk][unit]) so that a
// warp's 32 lanes read consecutive chunks:
//   int4: word t of a unit = elements 8t..8t+7, low nibbles the even ones and
//         high nibbles the odd ones; chunk 0 = the even codes of words 0..3,
//         chunk 1 = the odd codes.  w & 0x0F0F0F0F and w & 0xF0F0F0F0 (16 u)
//         feed dp4a unshifted: 16 * dot = 16 * lo + hi, with the hi chain
//         seeded by -128 * sum(q_x) (the -8 offset, times 16).
//   int2: word t = elements 16t..16t+15, field i (bits 2i..2i+1) of byte j =
//         element 16t + 4j + i; chunk t holds, for i = 0..3, the codes of the
//         elements of field i.  Masks 0x03.. << 2i give 4^i u; 64 * dot =
//         64 c0 + 16 c1 + 4 c2 + c3, the c3 chain seeded by -128 * sum(q_x)
//         (the -2 offset, times 64).
// Per 32-block the stage also keeps d_x (fp32) and the seed (int32).
// ---------------------------------------------------------------------------
template <int BITS>
struct RowFmt {
    static constexpr int E = 128 / BITS;   // codes per 16-byte unit
    static constexpr int NB = E / 32;      // activation blocks per unit
    static constexpr int CH = E / 16;      // 16-byte activation chunks per unit
};

template <int BITS>
__device__ __forceinline__ void stage_rowwise_x(const int8_t* __restrict__ xq, const uint16_t* __restrict__ xd, int K,
                                                uint8_t* xs, float2* meta) {
    using F = RowFmt<BITS>;
    const int U = K / F::E, B = K / QK;
    // codes: one unit per thread and step, read as 16-byte vectors and
    // rearranged with byte permutes into the unit's chunks
#pragma unroll 4
    for (int u = threadIdx.x; u < U; u += blockDim.x) {
        if (BITS == 4) {
            const uint4 a = *reinterpret_cast<const uint4*>(xq + 32 * u);       // elements 0..15
            const uint4 b = *reinterpret_cast<const uint4*>(xq + 32 * u + 16);  // 16..31
            // chunk 0: even elements of each 8-element word, chunk 1: odd ones
            const uint4 ev = make_uint4(__byte_perm(a.x, a.y, 0x6420), __byte_perm(a.z, a.w, 0x6420),
                                        __byte_perm(b.x, b.y, 0x6420), __byte_perm(b.z, b.w, 0x6420));
            const uint4 od = make_uint4(__byte_perm(a.x, a.y, 0x7531), __byte_perm(a.z, a.w, 0x7531),
                                        __byte_perm(b.x, b.y, 0x7531), __byte_perm(b.z, b.w, 0x7531));
            *reinterpret_cast<uint4*>(xs + (size_t)u * 16) = ev;
            *reinterpret_cast<uint4*>(xs + ((size_t)U + u) * 16) = od;
        } else {
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                // 16 elements e0..e15 as four words; operand i = (e_i, e_4+i, e_8+i, e_12+i)
                const uint4 v = *reinterpret_cast<const uint4*>(xq + 64 * u + 16 * t);
                const uint32_t t0 = __byte_perm(v.x, v.y, 0x5140), t1 = __byte_perm(v.z, v.w, 0x5140);
                const uint32_t t2 = __byte_perm(v.x, v.y, 0x7362), t3 = __byte_perm(v.z, v.w, 0x7362);
                *reinterpret_cast<uint4*>(xs + ((size_t)t * U + u) * 16) =
                    make_uint4(__byte_perm(t0, t1, 0x5410), __byte_perm(t0, t1, 0x7632), __byte_perm(t2, t3, 0x5410),
                               __byte_perm(t2, t3, 0x7632));
            }
        }
    }
    // per block: d_x and the seed -128 * sum(q_x)
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
        const int4 lo = *reinterpret_cast<const int4*>(xq + 32 * b);
        const int4 hi = *reinterpret_cast<const int4*>(xq + 32 * b + 16);
        int s = 0;
        s = __dp4a(lo.x, 0x01010101, s);
        s = __dp4a(lo.y, 0x01010101, s);
        s = __dp4a(lo.z, 0x01010101, s);
        s = __dp4a(lo.w, 0x01010101, s);
        s = __dp4a(hi.x, 0x01010101, s);
        s = __dp4a(hi.y, 0x01010101, s);
        s = __dp4a(hi.z, 0x01010101, s);
        s = __dp4a(hi.w, 0x01010101, s);
        meta[b] = make_float2(f16_bits_to_f32(xd[b]), __int_as_float(-128 * s));
    }
}

// One unit of one row: adds d_x * (scaled dot) of its blocks to acc.
template <int BITS>
__device__ __forceinline__ float unit_rowwise(uint4 w, const uint4* x, const float2* m, float acc) {
    const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
    if (BITS == 4) {
        const uint32_t xe[4] = {x[0].x, x[0].y, x[0].z, x[0].w};
        const uint32_t xo[4] = {x[1].x, x[1].y, x[1].z, x[1].w};
        int lo = 0, hi = __float_as_int(m[0].y);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            lo = dp4a_us(wv[t] & 0x0F0F0F0Fu, (int)xe[t], lo);
            hi = dp4a_us(wv[t] & 0xF0F0F0F0u, (int)xo[t], hi);
        }
        return fmaf(m[0].x, (float)(16 * lo + hi), acc);  // 16 * dot
    } else {
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            int c0 = 0, c1 = 0, c2 = 0, c3 = __float_as_int(m[b].y);
#pragma unroll
            for (int tt = 0; tt < 2; ++tt) {
                const int t = 2 * b + tt;
                const uint4 xv = x[t];
                c0 = dp4a_us(wv[t] & 0x03030303u, (int)xv.x, c0);
                c1 = dp4a_us(wv[t] & 0x0C0C0C0Cu, (int)xv.y, c1);
                c2 = dp4a_us(wv[t] & 0x30303030u, (int)xv.z, c2);
                c3 = dp4a_us(wv[t] & 0xC0C0C0C0u, (int)xv.w, c3);
            }
            acc = fmaf(m[b].x, (float)(64 * c0 + 16 * c1 + 4 * c2 + c3), acc);  // 64 * dot
        }
        return acc;
    }
}

template <int BITS>
__global__ void __launch_bounds__(FMT_THREADS) gemv_rowwise_kernel(const uint8_t* __restrict__ wq,
                                                                   const float* __restrict__ ws, int64_t N, int K,
                                                                   const int8_t* __restrict__ xq,
                                                                   const uint16_t* __restrict__ xd,
                                                                   float* __restrict__ y) {
    using F = RowFmt<BITS>;
    extern __shared__ __align__(16) uint8_t smem[];
    const int U = K / F::E;
    uint8_t* xs = smem;                                                   // [CH][U] x 16 B
    float2* meta = reinterpret_cast<float2*>(smem + (size_t)U * F::CH * 16);  // [K/32]
    stage_rowwise_x<BITS>(xq, xd, K, xs, meta);
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t rowb = K / (8 / BITS);
    const int64_t groups = (N + FMT_ROWS - 1) / FMT_ROWS;
    const float unscale = BITS == 4 ? 0.0625f : 0.015625f;  // 1/16, 1/64
    for (int64_t g = (int64_t)blockIdx.x * FMT_WARPS + warp; g < groups; g += (int64_t)gridDim.x * FMT_WARPS) {
        const int64_t r0 = g * FMT_ROWS;
        float acc[FMT_ROWS] = {};
        for (int u0 = lane; u0 < U; u0 += 32 * FMT_DEPTH) {
            // FMT_DEPTH steps of loads in flight before any of them is used
            uint4 wq4[FMT_DEPTH][FMT_ROWS];
#pragma unroll
            for (int dd = 0; dd < FMT_DEPTH; ++dd)
#pragma unroll
                for (int r = 0; r < FMT_ROWS; ++r) {
                    const int u = u0 + 32 * dd;
                    wq4[dd][r] = (u < U && r0 + r < N) ? ld_stream_v4(wq + (r0 + r) * rowb + (int64_t)u * 16)
                                                       : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
            for (int dd = 0; dd < FMT_DEPTH; ++dd) {
            const int u = u0 + 32 * dd;
            if (u >= U) break;
            const uint4* wv = wq4[dd];
            uint4 xv[F::CH];
#pragma unroll
            for (int c = 0; c < F::CH; ++c) xv[c] = lds128(xs + ((size_t)c * U + u) * 16);
            float2 m[F::NB];
            if (F::NB == 2) {  // both blocks' (d_x, seed) in one 16-byte load
                const float4 mm = *reinterpret_cast<const float4*>(meta + 2 * u);
                m[0] = make_float2(mm.x, mm.y);
                m[F::NB - 1] = make_float2(mm.z, mm.w);
            } else {
                m[0] = meta[u];
            }
#pragma unroll
            for (int r = 0; r < FMT_ROWS; ++r) acc[r] = unit_rowwise<BITS>(wv[r], xv, m, acc[r]);
            }
        }
#pragma unroll
        for (int r = 0; r < FMT_ROWS; ++r) {
            const float v = warp_sum(acc[r]);
            if (lane == 0 && r0 + r < N) y[r0 + r] = (ws[r0 + r] * unscale) * v;
        }
    }
}

// ---------------------------------------------------------------------------
// Q4_0 x fp32 GEMV, dequantize-then-FMA.  Lane = one Q4_0 block (16 nibble
// bytes + fp16 scale) of each of four rows; the block's 32 fp32 activations
// come from shared memory, chunk-major ([chunk c][block], chunk c = values
// 4c..4c+3), and serve all four rows.  A code becomes an exact float through
// the exponent trick: bytes (u, 0, 0, 0x4B) are the float 2^23 + u, and
// subtracting 2^23 + 8 leaves q = u - 8 exactly.  The arithmetic runs on
// packed fp32 pairs (add/fma .f32x2: each half rounds exactly like the scalar
// instruction), two values per instruction: per block two pair chains (low
// and high nibbles, 8 steps each), their four halves summed, then acc +=
// d_w * block sum.
// ---------------------------------------------------------------------------
typedef unsigned long long f32x2_t;

__device__ __forceinline__ f32x2_t pack2(uint32_t lo, uint32_t hi) {
    f32x2_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}

// (q_a, q_b) of bytes a and b of a nibble-masked word, as a packed pair
__device__ __forceinline__ f32x2_t nib2_to_q(uint32_t masked, uint32_t sel_a, uint32_t sel_b) {
    const f32x2_t m = pack2(__byte_perm(masked, 0x4B000000u, sel_a), __byte_perm(masked, 0x4B000000u, sel_b));
    const f32x2_t off = pack2(__float_as_uint(-8388616.0f), __float_as_uint(-8388616.0f));
    f32x2_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(m), "l"(off));
    return r;
}

__device__ __forceinline__ f32x2_t fma2(f32x2_t a, f32x2_t b, f32x2_t c) {
    f32x2_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

__device__ __forceinline__ float hsum2(f32x2_t v) {
    uint32_t a, b;
    asm("mov.b64 {%0, %1}, %2;" : "=r"(a), "=r"(b) : "l"(v));
    return __uint_as_float(a) + __uint_as_float(b);
}

__global__ void __launch_bounds__(FMT_THREADS) gemv_q4_0_f32_fma_kernel(const uint8_t* __restrict__ qs,
                                                                        const uint16_t* __restrict__ wd, int64_t N,
                                                                        int K, const float* __restrict__ x,
                                                                        float* __restrict__ y) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int B = K / QK;
    float4* xs = reinterpret_cast<float4*>(smem);  // [8][B]
#pragma unroll 8
    for (int idx = threadIdx.x; idx < 8 * B; idx += blockDim.x) {  // coalesced reads of x
        const int b = idx >> 3, c = idx & 7;
        xs[c * B + b] = *reinterpret_cast<const float4*>(x + 4 * idx);
    }
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t rowb = K / 2;
    const int64_t groups = (N + FMT_ROWS - 1) / FMT_ROWS;
    for (int64_t g = (int64_t)blockIdx.x * FMT_WARPS + warp; g < groups; g += (int64_t)gridDim.x * FMT_WARPS) {
        const int64_t r0 = g * FMT_ROWS;
        float acc[FMT_ROWS] = {};
        for (int b0 = lane; b0 < B; b0 += 32 * FMA_DEPTH) {
            // FMA_DEPTH steps of loads in flight before any of them is used
            uint4 wq4[FMA_DEPTH][FMT_ROWS];
            unsigned short dq4[FMA_DEPTH][FMT_ROWS];
#pragma unroll
            for (int dd = 0; dd < FMA_DEPTH; ++dd)
#pragma unroll
                for (int r = 0; r < FMT_ROWS; ++r) {
                    const int b = b0 + 32 * dd;
                    const bool in = b < B && r0 + r < N;
                    wq4[dd][r] = in ? ld_stream_v4(qs + (r0 + r) * rowb + (int64_t)b * 16)
                                    : make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
                    dq4[dd][r] = in ? ld_stream_u16(wd + (r0 + r) * B + b) : (unsigned short)0;
                }
#pragma unroll
            for (int dd = 0; dd < FMA_DEPTH; ++dd) {
            const int b = b0 + 32 * dd;
            if (b >= B) break;
            const uint4* wv = wq4[dd];
            float dv[FMT_ROWS];
#pragma unroll
            for (int r = 0; r < FMT_ROWS; ++r) dv[r] = f16_bits_to_f32(dq4[dd][r]);
            float4 xv[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) xv[c] = xs[c * B + b];
#pragma unroll
            for (int r = 0; r < FMT_ROWS; ++r) {
                const uint32_t wt[4] = {wv[r].x, wv[r].y, wv[r].z, wv[r].w};
                f32x2_t lo = 0, hi = 0;  // +0.0f pairs
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const uint32_t l = wt[t] & 0x0F0F0F0Fu, h = (wt[t] >> 4) & 0x0F0F0F0Fu;
                    const float4 xl = xv[t], xh = xv[4 + t];
                    lo = fma2(nib2_to_q(l, 0x7440u, 0x7441u), pack2(__float_as_uint(xl.x), __float_as_uint(xl.y)), lo);
                    lo = fma2(nib2_to_q(l, 0x7442u, 0x7443u), pack2(__float_as_uint(xl.z), __float_as_uint(xl.w)), lo);
                    hi = fma2(nib2_to_q(h, 0x7440u, 0x7441u), pack2(__float_as_uint(xh.x), __float_as_uint(xh.y)), hi);
                    hi = fma2(nib2_to_q(h, 0x7442u, 0x7443u), pack2(__float_as_uint(xh.z), __float_as_uint(xh.w)), hi);
                }
                acc[r] = fmaf(dv[r], hsum2(lo) + hsum2(hi), acc[r]);
            }
            }
        }
#pragma unroll
        for (int r = 0; r < FMT_ROWS; ++r) {
            const float v = warp_sum(acc[r]);
            if (lane == 0 && r0 + r < N) y[r0 + r] = v;
        }
    }
}

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

std::mutex g_mu;
std::set<std::pair<const void*, int>> g_done;

// Opt a kernel into `bytes` of dynamic shared memory (once per kernel and device).
template <typename Kern>
bool allow_smem(Kern kernel, int bytes, int optin) {
    if (bytes <= 48 * 1024) return true;
    if (bytes > optin) return false;
    int dev = 0;
    cudaGetDevice(&dev);
    const auto key = std::make_pair(reinterpret_cast<const void*>(kernel), dev);
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_done.count(key)) return true;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, optin) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    g_done.insert(key);
    return true;
}

// CTAs per SM that the kernel's registers and this shared-memory size allow
// (at most 4), times the SM count, capped by the work.
template <typename Kern>
int persistent_grid(Kern kernel, int smem, int sms, int64_t work) {
    int per_sm = 1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, FMT_THREADS, smem) != cudaSuccess) {
        cudaGetLastError();
        per_sm = 1;
    }
    per_sm = std::max(1, std::min(per_sm, 4));
    return (int)std::max<int64_t>(1, std::min<int64_t>(work, (int64_t)per_sm * sms));
}

qmm_status status_of(cudaError_t e) {
    if (e == cudaSuccess) e = cudaGetLastError();
    else cudaGetLastError();
    return e == cudaSuccess ? QMM_OK : QMM_ERR_CUDA;
}

}  // namespace
}  // namespace qmm

using namespace qmm;

extern "C" {

qmm_status qmm_quantize_rowwise(const float* w, int64_t N, int64_t K, int64_t ldw, int32_t bits, uint8_t* w_q,
                                float* w_s, void* stream) {
    if (N < 0 || K <= 0 || ldw < K || (bits != 4 && bits != 2)) return QMM_ERR_ARG;
    if (K % (bits == 4 ? 32 : 64) != 0) return QMM_ERR_SHAPE;
    if (N == 0) return QMM_OK;
    if (!w || !w_q || !w_s) return QMM_ERR_ARG;
    if (!aligned(w, 4) || !aligned(w_s, 4)) return QMM_ERR_ALIGN;
    int sms = 0, optin = 0;
    if (!device_facts(&sms, &optin)) return QMM_ERR_DEVICE;
    const int grid = (int)std::min<int64_t>(N, 8 * (int64_t)sms);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (bits == 4)
        quantize_rowwise_kernel<4><<<grid, FMT_THREADS, 0, st>>>(w, N, K, ldw, w_q, w_s);
    else
        quantize_rowwise_kernel<2><<<grid, FMT_THREADS, 0, st>>>(w, N, K, ldw, w_q, w_s);
    return status_of(cudaSuccess);
}

qmm_status qmm_gemv_rowwise_q8_0(const uint8_t* w_q, const float* w_s, int32_t bits, int64_t N, int64_t K,
                                 const int8_t* xq, const uint16_t* xd, float* y, void* stream) {
    if (N <= 0 || K <= 0 || (bits != 4 && bits != 2)) return QMM_ERR_ARG;
    if (K % (bits == 4 ? 32 : 64) != 0 || K > QMM_ROWWISE_MAX_K) return QMM_ERR_SHAPE;
    if (!w_q || !w_s || !xq || !xd || !y) return QMM_ERR_ARG;
    if (!aligned(w_q, 16) || !aligned(w_s, 4) || !aligned(xq, 16) || !aligned(xd, 2) || !aligned(y, 4))
        return QMM_ERR_ALIGN;
    int sms = 0, optin = 0;
    if (!device_facts(&sms, &optin)) return QMM_ERR_DEVICE;
    const int smem = (int)(K + (K / QK) * 8);  // permuted codes + (d_x, seed) per block
    const int64_t groups = (N + FMT_ROWS - 1) / FMT_ROWS;
    const int64_t ctas = (groups + FMT_WARPS - 1) / FMT_WARPS;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (bits == 4) {
        if (!allow_smem(gemv_rowwise_kernel<4>, smem, optin)) return QMM_ERR_SHAPE;
        const int grid = persistent_grid(gemv_rowwise_kernel<4>, smem, sms, ctas);
        gemv_rowwise_kernel<4><<<grid, FMT_THREADS, smem, st>>>(w_q, w_s, N, (int)K, xq, xd, y);
    } else {
        if (!allow_smem(gemv_rowwise_kernel<2>, smem, optin)) return QMM_ERR_SHAPE;
        const int grid = persistent_grid(gemv_rowwise_kernel<2>, smem, sms, ctas);
        gemv_rowwise_kernel<2><<<grid, FMT_THREADS, smem, st>>>(w_q, w_s, N, (int)K, xq, xd, y);
    }
    return status_of(cudaSuccess);
}

qmm_status qmm_gemv_q4_0_f32_fma(const uint8_t* w_qs, const uint16_t* w_d, int64_t N, int64_t K, const float* x,
                                 float* y, void* stream) {
    if (N <= 0 || K <= 0) return QMM_ERR_ARG;
    if (K % QK != 0 || K > QMM_F32_FMA_MAX_K) return QMM_ERR_SHAPE;
    if (!w_qs || !w_d || !x || !y) return QMM_ERR_ARG;
    if (!aligned(w_qs, 16) || !aligned(w_d, 2) || !aligned(x, 16) || !aligned(y, 4)) return QMM_ERR_ALIGN;
    int sms = 0, optin = 0;
    if (!device_facts(&sms, &optin)) return QMM_ERR_DEVICE;
    const int smem = (int)(K * 4);
    if (!allow_smem(gemv_q4_0_f32_fma_kernel, smem, optin)) return QMM_ERR_SHAPE;
    const int64_t groups = (N + FMT_ROWS - 1) / FMT_ROWS;
    const int grid = persistent_grid(gemv_q4_0_f32_fma_kernel, smem, sms, (groups + FMT_WARPS - 1) / FMT_WARPS);
    gemv_q4_0_f32_fma_kernel<<<grid, FMT_THREADS, smem, static_cast<cudaStream_t>(stream)>>>(w_qs, w_d, N, (int)K,
                                                                                            x, y);
    return status_of(cudaSuccess);
}

}  // extern "C"
