// qmm_gemm_mma.cu -- small-batch GEMM (up to 64 tokens per weight pass) of
// Q4_0 weights with Q8_0 activations on the warp-level tensor-core MMA:
// mma.sync m16n8k16 with fp16 operands and fp32 accumulation.
//
// Exact integer block dots on a float MMA: the weight codes q = u - 8 lie in
// [-8, 7] and the activation codes in [-127, 127]; both are exact in fp16
// (the weights as subnormals scaled by 2^-24, see the operand encodings
// below), every product is exact, and a block's 32-term sum is an integer of
// magnitude at most 32 * 8 * 127 = 32,512 (times 2^-24), exact in fp32.  So
// the MMA result of one block is the integer dot of the method (llama.cpp
// guide, kenji.blog/id, section 2.2: y ~ Delta * Delta_x * sum q * q_x) up to
// a power of two, and the rescale d_w * d_x * dot plus the sum over blocks
// are fp32 operations, as in the GEMV kernels.
//
// Why this instruction on sm_103a: tcgen05 has no integer MMA kind here, and
// with 8..64 token columns a 128-row tcgen05 MMA is latency-bound, whereas
// the warp MMA takes its operands from registers -- the nibbles become fp16
// in registers (no shared-memory round trip for the weights' converted
// form) and the per-block rescale is applied to the accumulator fragment in
// registers.
//
// Two layouts live here: the row-group kernel (gemm_mma_kernel, any token
// count) described next, and the 16-warp layout for up to 16 tokens
// (gemm_wide_kernel, further down), which qmm_gemm_q4_0_q8_0 takes where its
// row plan qualifies.  The workspace entry's variant of the 16-warp layout is
// in qmm_gemm_prep.cu.
//
// Row-group kernel, work layout:
//  - A CTA owns rows_per_cta consecutive weight rows (a multiple of the
//    group height R = 16, 32, 48 or 64), walked group by group; each group is
//    streamed in units of UKB blocks by a producer warp: one 2D TMA copy of
//    R rows x 8 blocks of nibbles per 8-block column (128-byte swizzled,
//    which makes the fragment loads below bank-conflict free) and one of the
//    R rows x UKB scales (swizzled over its own row pitch).
//  - Eight consumer warps.  A warp takes all R / 16 row tiles of the group
//    against up to two token tiles of 8, and 4 contiguous blocks of each
//    unit; the KP warps sharing a token group add their partial sums in
//    shared memory at the end of the group.  So each activation fragment read
//    from shared memory serves up to four row tiles.
//  - Activations: per unit, the consumer threads turn the unit's Q8_0 codes
//    of up to 8 * NT tokens into fp16 B fragments in shared memory (double
//    buffered), while the next unit's codes are already being loaded into
//    registers.
//
// Fragment mapping inside one block (k = 0..31 of the block, both halves of
// 16 go to one m16n8k16 each): lane (g, t) = (lane / 4, lane % 4) reads word
// t of a weight row's 16 nibble bytes, i.e. bytes 4t..4t+3, whose low
// nibbles are elements 4t..4t+3 and high nibbles elements 16+4t..16+4t+3.
// MMA half h uses the k slots {2t, 2t+1, 2t+8, 2t+9} <-> elements
// {4t, 4t+2, 4t+1, 4t+3} + 16h.  The same element order is used for the
// activation fragments, so each MMA sums exactly the 16 products of its
// half block.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <set>
#include <utility>

#include "qmm_device.cuh"
#include "qmm_mma.h"
#include "qmm_mma_frag.cuh"
#include "qmm_tmap.h"

namespace qmm {
namespace mmak {

using namespace frag;

constexpr int CW = 8;              // consumer warps
constexpr int NCT = CW * 32;       // consumer threads
constexpr int THREADS = NCT + 32;  // + one producer warp
constexpr int MAX_STAGES = 8;
constexpr int MAX_XITEMS = 512;    // (token, block) activation items per unit: 8 * NT * UKB

struct Args {
    int64_t N, K, M, ldy;
    const int8_t* xq;
    const uint16_t* xd;
    float* y;
    int rows_per_cta;  // a multiple of the group height
    int nstages;
    int stage_bytes;   // R * UKB * 18, rounded up to 1024
    int off_xbuf, off_xsc, off_red;  // from the 1024-aligned base; the ring starts at 1024
    int* err;
};

__device__ __forceinline__ void consumers_sync(int n) { asm volatile("bar.sync 1, %0;" ::"r"(n) : "memory"); }

// Shape of one kernel instance: NT token tiles of 8 (up to 8 * NT tokens per
// weight pass); TW row tiles of 16 per warp = the group height R / 16.
template <int NT, int TW>
struct Shape {
    static constexpr int NTW = NT < 2 ? NT : 2;          // token tiles per warp
    static constexpr int TGN = NT / NTW;                 // token groups
    static constexpr int KP = CW / TGN;                  // warps splitting the blocks of a unit
    static constexpr int R = 16 * TW;                    // rows per group
    static constexpr int UKB = 64 / NT < 32 ? 64 / NT : 32;  // blocks per unit: 32, 32, 16, 8
    static constexpr int KB_PART = UKB / KP;             // contiguous blocks per warp per unit (4)
    static constexpr int QBYTES = UKB / 8 * R * 128;     // nibble tiles of a stage
    static constexpr int STAGE = (QBYTES + R * UKB * 2 + 1023) / 1024 * 1024;
    static constexpr int XBUF = UKB * NT * 512;          // B fragments of one unit
    static constexpr int XSC = UKB * NT * 4 * 32;        // seeds and scales of one unit
    static constexpr int RED = (CW - TGN) * TW * NTW * 512;  // partial-sum slots
    static_assert(KP * TGN == CW && KB_PART == 4, "warp split");
};

template <int NT, int TW>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_mma_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_d, Args a) {
    using SH = Shape<NT, TW>;
    constexpr int NTW = SH::NTW, KP = SH::KP, R = SH::R, UKB = SH::UKB, QBYTES = SH::QBYTES;
    constexpr int XPER = (MAX_XITEMS + NCT - 1) / NCT;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(base);
    uint64_t* empty = full + MAX_STAGES;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + MAX_STAGES);
    uint8_t* ring = base + 1024;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = (int)(a.K / QK);
    const int S = a.nstages;
    const int64_t row_begin = (int64_t)blockIdx.x * a.rows_per_cta;
    const int64_t row_end = min(a.N, row_begin + a.rows_per_cta);
    const int nrows = (int)max((int64_t)0, row_end - row_begin);
    const int ngroups = (nrows + R - 1) / R;
    const int nkc = (B + UKB - 1) / UKB;
    const int nunits = ngroups * nkc;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], CW);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == CW) {
        // ---------------- producer warp: lane 0 paces the ring, lanes issue the copies
        const uint64_t pol = l2_evict_first_policy();
        int issued = 0;
        bool ok = true;
        for (int u = 0; u < nunits; ++u) {
            const int s = u % S;
            if (u >= S) {
                int w = 1;
                if (lane == 0) w = mbar_wait(&empty[s], ((u / S) - 1) & 1, abort_flag) ? 1 : 0;
                if (!__shfl_sync(FULL, w, 0)) {
                    ok = false;
                    break;
                }
            }
            const int g = u / nkc, kc = u - g * nkc;
            const int r0 = (int)(row_begin + (int64_t)g * R);
            const int b0 = kc * UKB, nbox = min(UKB, B - b0) / 8;  // K % 256 == 0: whole 8-block columns
            uint8_t* st = ring + (size_t)s * a.stage_bytes;
            if (lane == 0) mbar_arrive_expect_tx(&full[s], (uint32_t)(nbox * R * 128 + R * UKB * 2));
            __syncwarp();
            if (lane < nbox) tma2d(st + lane * R * 128, &map_q, (b0 + 8 * lane) * 16, r0, &full[s], pol);
            else if (lane == UKB / 8) tma2d(st + QBYTES, &map_d, b0, r0, &full[s], pol);
            issued = u + 1;
        }
        if (!ok && lane == 0) {
            atomicOr(a.err, ERR_TIMEOUT);
            *abort_flag = 1;
            for (int u = max(0, issued - S); u < issued; ++u) {  // let issued copies land
                const uint64_t t0 = global_ns();
                while (!mbar_try_wait(&full[u % S], (u / S) & 1) && global_ns() - t0 < WAIT_LIMIT_NS) {
                }
            }
        }
        return;
    }

    // ---------------- consumers
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int g8 = lane >> 2, t4 = lane & 3;
    const int kp = warp % KP, tg = warp / KP;
    // B fragment slot of this lane: the four 16-byte chunks of a token are
    // stored rotated by (token / 2) mod 4, so that both the per-token stores
    // and these per-lane loads are bank-conflict free
    const int fslot = (lane & ~3) | (((lane & 3) + (lane >> 3)) & 3);
    const int64_t m0 = (int64_t)blockIdx.y * (8 * NT);
    // Per buffer: B fragments [UKB][NT][32 lanes] x 16 bytes (the pair of the
    // low half, then the pair of the high half), and per token pair
    // [UKB][NT * 4] x (c even, c odd, c even, c odd | d_x even, d_x odd, -, -):
    // the MMA accumulator seed of rows g and g + 8, then the scales.
    uint8_t* xbuf = base + a.off_xbuf;
    float4* xsc = reinterpret_cast<float4*>(base + a.off_xsc);
    float* red = reinterpret_cast<float*>(base + a.off_red);  // slots of TW * NTW * 128 floats
    constexpr int XBUF_BYTES = SH::XBUF;
    constexpr int XSC_N = SH::XSC / 16;   // float4 per buffer
    constexpr int XITEMS = 8 * NT * UKB;  // (token, block) pairs of one unit
    static_assert(XITEMS <= XPER * NCT, "activation items per unit");

    uint4 px[XPER][2];
    uint32_t ps[XPER];
    // Activation codes and scale of each (token, block) item of unit column kc into registers.
    auto load_x = [&](int kc) {
        const int b0 = kc * UKB;
#pragma unroll
        for (int r = 0; r < XPER; ++r) {
            const int q = tid + NCT * r;
            px[r][0] = px[r][1] = make_uint4(0u, 0u, 0u, 0u);
            ps[r] = 0u;
            const int tok = q % (8 * NT), bl = q / (8 * NT);
            if (q < XITEMS && m0 + tok < a.M && b0 + bl < B) {
                const int64_t m = m0 + tok;
                const uint4* src = reinterpret_cast<const uint4*>(a.xq + m * a.K + (int64_t)(b0 + bl) * QK);
                px[r][0] = __ldg(src);
                px[r][1] = __ldg(src + 1);
                ps[r] = __ldg(a.xd + m * B + b0 + bl);
            }
        }
    };
    // Registers -> fragments, scales and accumulator seeds in buffer `buf`.
    auto store_x = [&](int buf) {
        uint8_t* xb = xbuf + buf * XBUF_BYTES;
        float* xs = reinterpret_cast<float*>(xsc + buf * XSC_N);
#pragma unroll
        for (int r = 0; r < XPER; ++r) {
            const int q = tid + NCT * r;
            if (q < XITEMS) {
                const int tok = q % (8 * NT), bl = q / (8 * NT);
                const uint4 lo = px[r][0], hi = px[r][1];
                int slo = __dp4a((int)lo.x, 0x01010101, 0);
                slo = __dp4a((int)lo.y, 0x01010101, slo);
                slo = __dp4a((int)lo.z, 0x01010101, slo);
                slo = __dp4a((int)lo.w, 0x01010101, slo);
                int shi = __dp4a((int)hi.x, 0x01010101, 0);
                shi = __dp4a((int)hi.y, 0x01010101, shi);
                shi = __dp4a((int)hi.z, 0x01010101, shi);
                shi = __dp4a((int)hi.w, 0x01010101, shi);
                // lane (g, t) of token tile j = tok / 8 holds word t of token g =
                // tok % 8, in chunk (t + g / 2) mod 4 of the token's 64 bytes
                uint4* dst = reinterpret_cast<uint4*>(xb + (bl * NT * 32 + tok * 4) * 16);
                const int rot = (tok >> 1) & 3;
                uint2 l, h;
                l = codes_lo_f16(lo.x), h = codes_hi_f16(hi.x);
                dst[rot] = make_uint4(l.x, l.y, h.x, h.y);
                l = codes_lo_f16(lo.y), h = codes_hi_f16(hi.y);
                dst[(rot + 1) & 3] = make_uint4(l.x, l.y, h.x, h.y);
                l = codes_lo_f16(lo.z), h = codes_hi_f16(hi.z);
                dst[(rot + 2) & 3] = make_uint4(l.x, l.y, h.x, h.y);
                l = codes_lo_f16(lo.w), h = codes_hi_f16(hi.w);
                dst[(rot + 3) & 3] = make_uint4(l.x, l.y, h.x, h.y);
                const int pr = (bl * NT * 8 + tok) >> 1, od = tok & 1;
                const float c = (float)(-8 * (slo + shi)) * 0x1p-24f;
                xs[pr * 8 + od] = c;
                xs[pr * 8 + 2 + od] = c;
                xs[pr * 8 + 4 + od] = f16_bits_to_f32((unsigned short)ps[r]) * 0x1p24f;
            }
        }
    };

    float2 acc[TW][NTW][2];
#pragma unroll
    for (int i = 0; i < TW; ++i)
#pragma unroll
        for (int j = 0; j < NTW; ++j) acc[i][j][0] = acc[i][j][1] = make_float2(0.f, 0.f);
    constexpr int DPITCH = UKB * 2;        // bytes per row of the scale tile
    constexpr int DMASK = DPITCH / 16 - 1;  // its swizzle: 16-byte chunk ^= (row * pitch / 128) & DMASK
    // This warp's blocks in every unit: 4 contiguous ones, b = 4 kp .. 4 kp + 3,
    // inside 8-block column kb = kp / 2; this lane's rows: 16 i + g8 (+ 8).
    const int kb = kp >> 1, c0 = (kp & 1) << 2;
    int doff[TW][2];  // scale-tile offsets (fp16 units) of this lane's rows, for the warp's 4 blocks
#pragma unroll
    for (int i = 0; i < TW; ++i)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            const int r = 16 * i + g8 + 8 * hr;
            doff[i][hr] = r * UKB + (((kb ^ (((r * DPITCH) >> 7) & DMASK)) << 3) | c0);
        }
    bool failed = false;

    if (nunits > 0) load_x(0);
    for (int u = 0; u < nunits; ++u) {
        const int g = u / nkc, kc = u - g * nkc, s = u % S, buf = u & 1;
        store_x(buf);
        if (u + 1 < nunits) load_x((u + 1) % nkc);
        consumers_sync(NCT);  // fragments of this unit complete (and the unit before last fully read)
        // On a timeout keep going without computing: every later wait returns
        // at once (abort flag), and the kernel ends with the error word set.
        const bool ok = !failed && mbar_wait(&full[s], (u / S) & 1, abort_flag);
        if (!ok && !failed) {
            if (lane == 0) atomicOr(a.err, ERR_TIMEOUT);
            *abort_flag = 1;
            failed = true;
        }
        const int nb = min(UKB, B - kc * UKB);
        if (ok) {
            const uint8_t* st = ring + (size_t)s * a.stage_bytes;
            const uint16_t* sd = reinterpret_cast<const uint16_t*>(st + QBYTES);
            const uint8_t* xf0 = xbuf + buf * XBUF_BYTES + (tg * NTW * 32 + fslot) * 16;
            const float4* xs0 = xsc + buf * XSC_N + (tg * NTW * 4 + t4) * 2;
            // the scales of this lane's rows for the warp's 4 blocks
            uint2 dq[TW][2];
#pragma unroll
            for (int i = 0; i < TW; ++i)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) dq[i][hr] = *reinterpret_cast<const uint2*>(sd + doff[i][hr]);
            const uint8_t* bx0 = st + kb * R * 128 + g8 * 128 + 4 * t4;
#pragma unroll
            for (int bb = 0; bb < SH::KB_PART; ++bb) {
                const int b = 4 * kp + bb;
                if (b < nb) {
                    const int sw = ((c0 + bb) ^ g8) << 4;  // 128-byte swizzle: row & 7 == g8
                    uint32_t ah[TW][2][4];
                    float dw[TW][2];
#pragma unroll
                    for (int i = 0; i < TW; ++i) {
                        const uint8_t* bx = bx0 + i * 16 * 128 + sw;
                        uint32_t q0[4], q1[4];
                        nibbles_sub(*reinterpret_cast<const uint32_t*>(bx), q0);
                        nibbles_sub(*reinterpret_cast<const uint32_t*>(bx + 8 * 128), q1);
                        ah[i][0][0] = q0[0], ah[i][0][1] = q1[0], ah[i][0][2] = q0[1], ah[i][0][3] = q1[1];
                        ah[i][1][0] = q0[2], ah[i][1][1] = q1[2], ah[i][1][2] = q0[3], ah[i][1][3] = q1[3];
#pragma unroll
                        for (int hr = 0; hr < 2; ++hr) {
                            const uint32_t wd = (bb < 2) ? dq[i][hr].x : dq[i][hr].y;
                            dw[i][hr] = f16_bits_to_f32((unsigned short)(wd >> (16 * (bb & 1))));
                        }
                    }
                    const uint8_t* xf = xf0 + b * NT * 512;
                    const float4* xs = xs0 + b * NT * 8;
#pragma unroll
                    for (int j = 0; j < NTW; ++j) {
                        const uint4 f = *reinterpret_cast<const uint4*>(xf + j * 512);
                        const float4 cq = xs[j * 8];  // accumulator seed, tokens 2t, 2t+1 of the tile
                        const float2 sx = *reinterpret_cast<const float2*>(xs + j * 8 + 1);  // their d_x
                        const float c4[4] = {cq.x, cq.y, cq.z, cq.w};
#pragma unroll
                        for (int i = 0; i < TW; ++i) {
                            float dd[4];
                            mma16816(dd, ah[i][0], f.x, f.y, c4);
                            mma16816(dd, ah[i][1], f.z, f.w, dd);  // 2^-24 x the integer block dots
                            acc[i][j][0] = ffma2_scaled(make_float2(dw[i][0], dw[i][0]), sx,
                                                        make_float2(dd[0], dd[1]), acc[i][j][0]);
                            acc[i][j][1] = ffma2_scaled(make_float2(dw[i][1], dw[i][1]), sx,
                                                        make_float2(dd[2], dd[3]), acc[i][j][1]);
                        }
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);  // stage read: the producer may refill it

        if (kc == nkc - 1) {
            // end of the group: the KP warps of (rows, tokens) meet; part 0 adds and writes y
            if (KP > 1) {
                constexpr int SLOT = TW * NTW * 128;
                const int slot0 = tg * (KP - 1);
                if (kp > 0) {
                    float* rp = red + (slot0 + kp - 1) * SLOT + lane;
#pragma unroll
                    for (int i = 0; i < TW; ++i)
#pragma unroll
                        for (int j = 0; j < NTW; ++j) {
                            float* q = rp + (i * NTW + j) * 128;
                            q[0] = acc[i][j][0].x;
                            q[32] = acc[i][j][0].y;
                            q[64] = acc[i][j][1].x;
                            q[96] = acc[i][j][1].y;
                        }
                }
                consumers_sync(NCT);
                if (kp == 0) {
#pragma unroll
                    for (int p = 1; p < KP; ++p) {
                        const float* rp = red + (slot0 + p - 1) * SLOT + lane;
#pragma unroll
                        for (int i = 0; i < TW; ++i)
#pragma unroll
                            for (int j = 0; j < NTW; ++j) {
                                const float* q = rp + (i * NTW + j) * 128;
                                acc[i][j][0].x += q[0];
                                acc[i][j][0].y += q[32];
                                acc[i][j][1].x += q[64];
                                acc[i][j][1].y += q[96];
                            }
                    }
                }
            }
            const int64_t r0 = row_begin + (int64_t)g * R;
            const int nr = (int)min((int64_t)R, row_end - r0);
            if (kp == 0 && !failed) {
#pragma unroll
                for (int i = 0; i < TW; ++i)
#pragma unroll
                    for (int j = 0; j < NTW; ++j) {
                        const int64_t m = m0 + 8 * (tg * NTW + j) + 2 * t4;
#pragma unroll
                        for (int hr = 0; hr < 2; ++hr) {
                            const int lr = 16 * i + g8 + 8 * hr;
                            if (lr >= nr) continue;
                            const int64_t row = r0 + lr;
                            if (m < a.M) a.y[m * a.ldy + row] = acc[i][j][hr].x;
                            if (m + 1 < a.M) a.y[(m + 1) * a.ldy + row] = acc[i][j][hr].y;
                        }
                    }
            }
#pragma unroll
            for (int i = 0; i < TW; ++i)
#pragma unroll
                for (int j = 0; j < NTW; ++j) acc[i][j][0] = acc[i][j][1] = make_float2(0.f, 0.f);
        }
    }
}

// ---------------------------------------------------------------- host side
template <int NT, int TW>
qmm_status launch_shape(const uint8_t* w_qs, const uint16_t* w_d, int64_t N, int64_t K, int64_t M,
                        const int8_t* xq, const uint16_t* xd, float* y, int64_t ldy, int64_t rpc, int smem_optin,
                        int* err, cudaStream_t st) {
    using SH = Shape<NT, TW>;
    const int64_t B = K / QK;
    const int64_t G = (N + rpc - 1) / rpc;
    const int fixed = 1024 + 2 * SH::XBUF + 2 * SH::XSC + SH::RED + 1024;  // header, buffers, alignment slack
    const int64_t nunits = (rpc / SH::R) * ((B + SH::UKB - 1) / SH::UKB);
    const int64_t nst = std::min<int64_t>({(int64_t)MAX_STAGES, (smem_optin - fixed) / SH::STAGE, nunits});
    if (nst < 1) return QMM_ERR_SHAPE;
    Args a = {};
    a.N = N;
    a.K = K;
    a.M = M;
    a.ldy = ldy;
    a.xq = xq;
    a.xd = xd;
    a.y = y;
    a.rows_per_cta = (int)rpc;
    a.nstages = (int)nst;
    a.stage_bytes = SH::STAGE;
    a.off_xbuf = 1024 + (int)nst * SH::STAGE;
    a.off_xsc = a.off_xbuf + 2 * SH::XBUF;
    a.off_red = a.off_xsc + 2 * SH::XSC;
    a.err = err;
    const int smem = a.off_red + SH::RED + 1024;
    const CUtensorMapSwizzle dsw = SH::UKB == 8    ? CU_TENSOR_MAP_SWIZZLE_NONE
                                   : SH::UKB == 16 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                   : CU_TENSOR_MAP_SWIZZLE_64B;
    CUtensorMap mq, md;
    if (!make_tensor_map_2d(&mq, CU_TENSOR_MAP_DATA_TYPE_UINT8, w_qs, (uint64_t)K / 2, (uint64_t)N, (uint64_t)K / 2,
                            128, (uint32_t)SH::R, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map_2d(&md, CU_TENSOR_MAP_DATA_TYPE_UINT16, w_d, (uint64_t)B, (uint64_t)N, (uint64_t)B * 2,
                            (uint32_t)SH::UKB, (uint32_t)SH::R, dsw))
        return QMM_ERR_CUDA;
    auto kern = gemm_mma_kernel<NT, TW>;
    if (smem > smem_optin || !allow_smem(kern, smem_optin)) return QMM_ERR_SHAPE;
    const dim3 grid((unsigned)G, (unsigned)((M + 8 * NT - 1) / (8 * NT)));
    kern<<<grid, THREADS, smem, st>>>(mq, md, a);
    return cudaGetLastError() == cudaSuccess ? QMM_OK : QMM_ERR_CUDA;
}

// Group height R = 16 TW rows: the tallest (TW = 4, 3, 2, 1) whose
// rows-per-CTA at one CTA per SM stays within 8% of the 16-row minimum, so
// that a CTA stages each activation unit as few times as possible.
template <int NT>
qmm_status launch_nt(const uint8_t* w_qs, const uint16_t* w_d, int64_t N, int64_t K, int64_t M, const int8_t* xq,
                     const uint16_t* xd, float* y, int64_t ldy, int sms, int smem_optin, int* err, cudaStream_t st) {
    const int64_t need = (N + sms - 1) / sms;
    const int64_t r16 = round_up(need, 16);
    auto fits = [&](int tw) { return round_up(need, 16 * tw) * 100 <= r16 * 108; };
    if (fits(4))
        return launch_shape<NT, 4>(w_qs, w_d, N, K, M, xq, xd, y, ldy, round_up(need, 64), smem_optin, err, st);
    if (fits(3))
        return launch_shape<NT, 3>(w_qs, w_d, N, K, M, xq, xd, y, ldy, round_up(need, 48), smem_optin, err, st);
    if (fits(2))
        return launch_shape<NT, 2>(w_qs, w_d, N, K, M, xq, xd, y, ldy, round_up(need, 32), smem_optin, err, st);
    return launch_shape<NT, 1>(w_qs, w_d, N, K, M, xq, xd, y, ldy, r16, smem_optin, err, st);
}


// ================================================================ wide variant
// The same arithmetic for up to 16 tokens, laid out for more warps and less
// repeated work per weight byte:
//  - 16 warps (4 per SM sub-partition, up to 128 registers each) instead of
//    8 consumers + a producer, so that the fixed-latency chains of one warp
//    (fragment load -> conversion -> two dependent MMAs -> rescale) are
//    hidden by the others;
//  - a unit is ALL rows of the CTA (RPC = 16 KPB WT rows) x 16 blocks, so the
//    activation fragments of a unit are built once per CTA instead of once
//    per row group;
//  - warp (rh, kp) takes row tiles rh WT .. rh WT + WT - 1 and the KPB
//    contiguous blocks kp KPB .. of every unit (KPB x 16 / KPB = 16 warps);
//  - one ring stage holds everything a unit reads: the nibble and scale
//    tiles of the rows and the Q8_0 codes and scales of the tokens, all by
//    TMA, S - 1 units ahead, so no load of the loop waits on L2 or HBM;
//  - weight fragments come from ldmatrix: one x4 load gives a lane its word
//    of rows g and g + 8 for two blocks, in place of four 32-bit loads;
//  - the nibbles enter the MMA as fp16 subnormals: the masked bit pattern u
//    (or 16 v) of each half word IS the fp16 value u * 2^-24 (16 v * 2^-24),
//    so a fragment register is one AND of the word (no second constant to
//    merge in); every product and block sum is that of the integer codes
//    times 2^-24, exact in fp32, and the 2^24 is folded into the staged d_x
//    (a power of two: the rescaled fp32 result is unchanged, bit for bit);
//  - the fp16 activation fragments of unit u + 1 are built from the stage
//    (warp w: block w of the unit, lane = (token, half block)) while unit u
//    is computed, handed over through mbarriers (two buffers);
//  - no producer warp: the hand-over keeps every warp within one unit of
//    the others, so once the last warp has finished unit u - 1 its stage is
//    free, and lanes 0 of warps 0..3 refill it with unit u - 1 + S (one of
//    the unit's four copies each);
//  - modes: one chunk of rows per CTA, several (large N), or a cluster of
//    CTAs splitting K over one chunk (small N, long K); see the kernel.
namespace widek {

constexpr int CW = 16;
constexpr int THREADS = CW * 32;
constexpr int UKB = 16;  // blocks per unit: two 8-block nibble columns
constexpr int MAX_STAGES = 8;

template <int NT, int WT, int KPB>
struct Shape {
    static constexpr int KP = UKB / KPB;  // warps splitting a unit's blocks
    static constexpr int RH = CW / KP;    // warps splitting the rows (= KPB)
    static constexpr int RPC = 16 * RH * WT;
    static constexpr int TK = 8 * NT;  // token rows of a launch
    // stage: nibble columns [2][RPC][128] (128-byte swizzled) | weight scales
    // [RPC][16] fp16 (32-byte swizzled) | codes [4][TK][128] (4 blocks per
    // 128-byte box, 128-byte swizzled) | activation scales [TK][16] fp16
    static constexpr int QB = 2 * RPC * 128;
    static constexpr int OFF_XQ = QB + RPC * UKB * 2;
    static constexpr int OFF_XD = OFF_XQ + 4 * TK * 128;
    static constexpr int STAGE = (OFF_XD + TK * UKB * 2 + 1023) / 1024 * 1024;
    static constexpr int XBUF = UKB * NT * 512;  // fp16 B fragments of a unit
    static constexpr int XSC = UKB * NT * 64;    // per token pair: seeds (even, odd), 2^24 d_x (even, odd)
    static constexpr int RED = RH * (KP - 1) * WT * NT * 512;  // partial sums, aliased on the ring
    static constexpr int ITEMS = UKB * TK * 2;                  // (block, token, half) staging items
    static_assert(RH * KP == CW && KPB % 2 == 0 && ITEMS % 32 == 0 && ITEMS <= THREADS, "warp split");
    static_assert(OFF_XQ % 1024 == 0 && (TK * 128) % 1024 == 0, "swizzled boxes start on 1024 bytes");
};

struct Args {
    int64_t N, K, M, ldy;
    float* y;
    int nchunk;  // row chunks of RPC rows per CTA (the last CTA may have fewer)
    int nstages;
    int off_xbuf, off_xsc;  // from the 1024-aligned base; the ring starts at 1024
    int* err;
};

// Modes: ONE chunk of rows per CTA; MULTI: the CTA walks several row chunks
// (nchunk > 1; the other instances leave that bookkeeping out, it costs
// registers at the 128 cap); SPLIT: a cluster of nsplit CTAs shares one
// chunk, rank r taking the r-th share of the units (of K), and ranks
// 1..nsplit-1 hand their sums to rank 0 through distributed shared memory,
// which adds them in rank order (deterministic) and writes y.
enum Mode { ONE = 0, MULTI = 1, SPLIT = 2 };

template <int NT, int WT, int KPB, int MODE>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_wide_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_d,
                     const __grid_constant__ CUtensorMap map_xq, const __grid_constant__ CUtensorMap map_xd, Args a) {
    using SH = Shape<NT, WT, KPB>;
    constexpr int KP = SH::KP, RPC = SH::RPC, QB = SH::QB, TK = SH::TK;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(base);  // [MAX_STAGES] TMA bytes of a stage
    uint64_t* xfull = full + MAX_STAGES;                  // [2] fragments of a unit built (16 warps)
    uint64_t* xempty = xfull + 2;                         // [2] unit computed (16 warps)
    volatile int* abort_flag = reinterpret_cast<volatile int*>(xempty + 2);
    uint8_t* ring = base + 1024;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = (int)(a.K / QK);
    const int S = a.nstages;  // >= 2
    constexpr bool multi = MODE == MULTI, split = MODE == SPLIT;
    // units of a chunk this CTA takes: u_lo .. u_lo + nunits - 1 (all of K
    // but with SPLIT)
    int nunits = (B + UKB - 1) / UKB, u_lo = 0;
    uint32_t rank = 0, nsplit = 1;
    if constexpr (split) {
        asm("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
        asm("mov.u32 %0, %%cluster_nctarank;" : "=r"(nsplit));
        const int per = (nunits + (int)nsplit - 1) / (int)nsplit;
        u_lo = min(nunits, (int)rank * per);
        nunits = min(nunits, u_lo + per) - u_lo;
    }
    // this CTA's chunks of RPC rows: chunk0 .. chunk0 + nck - 1, walked one
    // after the other through one unit sequence v = chunk * nunits + unit
    const int64_t chunk0 = multi ? (int64_t)blockIdx.x * a.nchunk : split ? (int64_t)(blockIdx.x / nsplit)
                                                                         : (int64_t)blockIdx.x;
    const int nck = multi ? (int)min((int64_t)a.nchunk, (a.N + RPC - 1) / RPC - chunk0) : 1;
    const int V = multi ? nck * nunits : nunits;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&xfull[b], CW);
            mbar_init(&xempty[b], CW);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // The four copies of unit u into stage u % S (nibble columns, weight
    // scales, activation codes, activation scales), one each by lane 0 of
    // warps 0..3, in parallel (one thread issuing all of them serialises
    // their issue cost on the path every warp waits for).  Warp 0 announces
    // the unit's bytes; a copy may land before that (the barrier's byte
    // count may go negative, and its phase cannot complete before warp 0
    // arrives).  Boxes past K (a last half unit) or past the rows are
    // zero-filled and count in full.  The activations come from the kernel
    // before: only the first unit's weight copies go out before that wait.
    const bool issuer = lane == 0 && warp < 4;
    const uint64_t pol = l2_evict_first_policy();
    auto issue = [&](int v, bool weights, bool acts) {
        const int ck = multi ? v / nunits : 0;
        const int s = v % S, b0 = (u_lo + v - ck * nunits) * UKB;
        const int row_begin = (int)((chunk0 + ck) * RPC);
        uint8_t* st = ring + (size_t)s * SH::STAGE;
        if (warp == 0 && weights) {
            mbar_arrive_expect_tx(&full[s], (uint32_t)(2 * RPC * 128 + RPC * UKB * 2 + 4 * TK * 128 + TK * UKB * 2));
            tma3d_ef(st, &map_q, 0, (int)row_begin, b0 / 8, &full[s], pol);
        } else if (warp == 1 && weights) {
            tma2d(st + QB, &map_d, b0, (int)row_begin, &full[s], pol);
        } else if (warp == 2 && acts) {
            tma3d_keep(st + SH::OFF_XQ, &map_xq, 0, (int)blockIdx.y * TK, b0 / 4, &full[s]);
        } else if (warp == 3 && acts) {
            tma2d_keep(st + SH::OFF_XD, &map_xd, b0, (int)blockIdx.y * TK, &full[s]);
        }
    };
    int issued = min(S, V);
    if (issuer && V > 0) issue(0, true, false);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (issuer && V > 0) {
        issue(0, false, true);
        for (int v = 1; v < issued; ++v) issue(v, true, true);
    }

    const int g8 = lane >> 2, t4 = lane & 3;
    const int kp = warp % KP, rh = warp / KP;
    const int fb = kp * KPB, kb = fb >> 3, c0 = fb & 7;  // first block of the warp; its column, slot in it
    const int64_t m0 = (int64_t)blockIdx.y * TK;
    uint8_t* xbuf = base + a.off_xbuf;
    float4* xsc = reinterpret_cast<float4*>(base + a.off_xsc);
    constexpr int XSC_N = SH::XSC / 16;

    // staging item of this thread: block sb of the unit, token st_tok, half block sh
    const bool stager = warp * 32 < SH::ITEMS;  // warp-uniform
    const int sh = lane & 1, st_tok = (lane >> 1) & (TK - 1), sb = (warp * 32 + lane) / (2 * TK);
    // its 16 code bytes in a stage: box sb / 4, row st_tok, 16-byte chunk
    // (2 (sb % 4) + sh) ^ (st_tok % 8) of the 128-byte swizzle
    const int xq_off = SH::OFF_XQ + (sb >> 2) * TK * 128 + st_tok * 128 + ((((sb & 3) * 2 + sh) ^ (st_tok & 7)) << 4);
    const int xd_off = SH::OFF_XD + (st_tok * UKB + sb) * 2;
    const uint32_t x_mul = sh ? 0x2C002C00u : 0x3C003C00u;  // 1/16 or 1
    const uint32_t x_add = sh ? 0xD480D480u : 0xE480E480u;  // -72 or -1152
    // Unit u's fp16 B fragments and (seed, d_x) pairs into buffer buf.
    auto stage_x = [&](int v, int buf) {
        const uint8_t* st = ring + (size_t)(v % S) * SH::STAGE;
        const uint4 px = lds128(st + xq_off);
        int sum = __dp4a((int)px.x, 0x01010101, 0);
        sum = __dp4a((int)px.y, 0x01010101, sum);
        sum = __dp4a((int)px.z, 0x01010101, sum);
        sum = __dp4a((int)px.w, 0x01010101, sum);
        const int other = __shfl_xor_sync(FULL, sum, 1);
        // lane (g, t) of token tile j = tok / 8 holds word t of token g = tok % 8,
        // in chunk (t + g / 2) mod 4 of the token's 64 bytes; this thread writes
        // the low or high 8 bytes of each chunk
        uint8_t* dst = xbuf + buf * SH::XBUF + (sb * NT * 32 + st_tok * 4) * 16 + sh * 8;
        const int rot = (st_tok >> 1) & 3;
        const uint32_t w4[4] = {px.x, px.y, px.z, px.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            // (1152 + x) * mul + add = x (low half) or x / 16 (high half), exact
            uint2 p;
            p.x = hfma2((w4[t] & 0x00FF00FFu) ^ 0x64806480u, x_mul, x_add);
            p.y = hfma2(((w4[t] >> 8) & 0x00FF00FFu) ^ 0x64806480u, x_mul, x_add);
            *reinterpret_cast<uint2*>(dst + ((rot + t) & 3) * 16) = p;
        }
        if (sh == 0) {
            float* xs = reinterpret_cast<float*>(xsc + buf * XSC_N);
            const int pr = (sb * TK + st_tok) >> 1, od = st_tok & 1;
            // MMA seed: the products carry 2^-24 and the codes u = q + 8, so
            // -8 * 2^-24 * (sum of the block's codes) leaves 2^-24 * sum q x
            xs[pr * 4 + od] = (float)(-8 * (sum + other)) * 0x1p-24f;
            xs[pr * 4 + 2 + od] = f16_bits_to_f32(*reinterpret_cast<const uint16_t*>(st + xd_off)) * 0x1p24f;
        }
    };
    // B fragment slot of this lane (the rotation above, read back)
    const int fslot = (lane & ~3) | (((lane & 3) + (lane >> 3)) & 3);

    float2 acc[WT][NT][2];
#pragma unroll
    for (int i = 0; i < WT; ++i)
#pragma unroll
        for (int j = 0; j < NT; ++j) acc[i][j][0] = acc[i][j][1] = make_float2(0.f, 0.f);
    // scale-tile offsets (fp16 units) of this lane's rows: the tile is
    // [RPC][16] fp16, 32-byte swizzled (16-byte chunk ^= (row >> 2) & 1)
    int doff[WT][2];
    // ldmatrix row addresses: lane l gives row l % 8 of matrix l / 8 = (row
    // half hr, block of the pair bsel); both stay fixed, only the tile moves
    uint32_t qaddr[WT];
    {
        const int hr = (lane >> 3) & 1, bsel = lane >> 4, rr = lane & 7;
#pragma unroll
        for (int i = 0; i < WT; ++i) {
            const int rt = (rh * WT + i) * 16;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int r = rt + g8 + 8 * h;
                doff[i][h] = r * UKB + (((kb ^ ((r >> 2) & 1)) << 3) | c0);
            }
            const int r = rt + 8 * hr + rr;
            qaddr[i] = (uint32_t)(kb * RPC * 128 + r * 128 + (((c0 + bsel) ^ rr) << 4));
        }
    }
    bool failed = false;
    auto fail = [&]() {
        if (!failed) {
            if (lane == 0) atomicOr(a.err, ERR_TIMEOUT);
            *abort_flag = 1;
            failed = true;
        }
    };

    // The KP warps of each row set add their sums of a chunk in shared memory
    // (`red`: a stage every warp has finished with, which no copy fills until
    // this returns); kp 0 writes y.  Every thread calls this at the same
    // points (it holds two CTA barriers).
    constexpr int SLOT = WT * NT * 128;  // floats per warp
    // kp > 0 warps' sums into red, then added into kp 0's acc (one barrier)
    auto reduce_partials = [&](float* red) {
        if (kp > 0) {
            float* rp = red + (rh * (KP - 1) + kp - 1) * SLOT + lane;
#pragma unroll
            for (int i = 0; i < WT; ++i)
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    float* q = rp + (i * NT + j) * 128;
                    q[0] = acc[i][j][0].x;
                    q[32] = acc[i][j][0].y;
                    q[64] = acc[i][j][1].x;
                    q[96] = acc[i][j][1].y;
                }
        }
        asm volatile("bar.sync 1, %0;" ::"r"(THREADS) : "memory");
        if (kp == 0) {
#pragma unroll 1
            for (int p = 1; p < KP; ++p) {
                const float* rp = red + (rh * (KP - 1) + p - 1) * SLOT + lane;
#pragma unroll
                for (int i = 0; i < WT; ++i)
#pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        const float* q = rp + (i * NT + j) * 128;
                        acc[i][j][0].x += q[0];
                        acc[i][j][0].y += q[32];
                        acc[i][j][1].x += q[64];
                        acc[i][j][1].y += q[96];
                    }
            }
        }
    };
    // kp 0 warps write their rows of the chunk starting at row_begin
    auto store_rows = [&](int64_t row_begin) {
        if (kp == 0 && !failed) {
#pragma unroll
            for (int i = 0; i < WT; ++i)
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    const int64_t m = m0 + 8 * j + 2 * t4;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int64_t row = row_begin + (rh * WT + i) * 16 + g8 + 8 * h;
                        if (row >= a.N) continue;
                        if (m < a.M) a.y[m * a.ldy + row] = acc[i][j][h].x;
                        if (m + 1 < a.M) a.y[(m + 1) * a.ldy + row] = acc[i][j][h].y;
                    }
                }
        }
    };
    // a chunk's sums out through red, acc cleared; every thread calls this
    // at the same points (it holds two CTA barriers)
    auto reduce_store = [&](int64_t row_begin, float* red) {
        reduce_partials(red);
        store_rows(row_begin);
        asm volatile("bar.sync 1, %0;" ::"r"(THREADS) : "memory");  // red read before the stage is refilled
#pragma unroll
        for (int i = 0; i < WT; ++i)
#pragma unroll
            for (int j = 0; j < NT; ++j) acc[i][j][0] = acc[i][j][1] = make_float2(0.f, 0.f);
    };

    // prologue: unit 0's fragments built
    if (V > 0) {
        if (!wait_phase(&full[0], 0, abort_flag)) fail();
        if (stager && !failed) stage_x(0, 0);
        __syncwarp();
        if (lane == 0) mbar_arrive(&xfull[0]);
    }
    int u = 0, ck = 0;  // unit inside the chunk, chunk of this CTA
    for (int v = 0; v < V; ++v) {
        const int s = v % S, buf = v & 1;
        // every warp has finished unit v - 1: its stage may be refilled and
        // its fragment buffer (buf ^ 1) overwritten
        if (v >= 1 && !failed && !wait_phase(&xempty[buf ^ 1], ((v - 1) >> 1) & 1, abort_flag)) fail();
        // a chunk ended with unit v - 1: its sums out, through that unit's stage
        if constexpr (multi) {
            if (v >= 1 && u == 0)
                reduce_store((chunk0 + ck - 1) * RPC,
                             reinterpret_cast<float*>(ring + (size_t)((v - 1) % S) * SH::STAGE));
        }
        if (v >= 1 && issued < V && !failed) {
            if (issuer) issue(issued, true, true);
            ++issued;
        }
        // unit v: its stage was waited for before its fragments were built
        if (!failed && !wait_phase(&xfull[buf], (v >> 1) & 1, abort_flag)) fail();
        const int nb = min(UKB, B - (u_lo + u) * UKB);
        const bool work = !failed && fb < nb;
        const uint8_t* st = ring + (size_t)s * SH::STAGE;
        const uint32_t st_u32 = smem_u32(st);
        const uint8_t* xf0 = xbuf + buf * SH::XBUF + fslot * 16;
        const float4* xs0 = xsc + buf * XSC_N + t4;
        // the weight scales of this lane's rows for the warp's KPB blocks
        uint32_t dq[WT][2][KPB / 2];
        if (work) {
            const uint16_t* sd = reinterpret_cast<const uint16_t*>(st + QB);
#pragma unroll
            for (int i = 0; i < WT; ++i)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if constexpr (KPB == 4) {
                        const uint2 v = *reinterpret_cast<const uint2*>(sd + doff[i][h]);
                        dq[i][h][0] = v.x;
                        dq[i][h][1] = v.y;
                    } else {
                        dq[i][h][0] = *reinterpret_cast<const uint32_t*>(sd + doff[i][h]);
                    }
                }
        }
        // blocks fb + 2 bp and fb + 2 bp + 1 of unit u against all row tiles
        auto compute_pair = [&](int bp) {
            // the word of rows g and g + 8 of each row tile for both blocks
            uint32_t wq[WT][4];
#pragma unroll
            for (int i = 0; i < WT; ++i) ldsm_x4(st_u32 + (qaddr[i] ^ (uint32_t)(bp << 5)), wq[i]);
#pragma unroll
            for (int bs = 0; bs < 2; ++bs) {
                const int b = fb + 2 * bp + bs;  // block inside the unit
                const uint8_t* xf = xf0 + b * NT * 512;
                const float4* xs = xs0 + b * NT * 4;
                uint4 f[NT];
                float4 cs[NT];
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    f[j] = *reinterpret_cast<const uint4*>(xf + j * 512);
                    cs[j] = xs[j * 4];
                }
#pragma unroll
                for (int i = 0; i < WT; ++i) {
                    uint32_t q0[4], q1[4];
                    nibbles_sub(wq[i][2 * bs], q0);
                    nibbles_sub(wq[i][2 * bs + 1], q1);
                    const uint32_t a0[4] = {q0[0], q1[0], q0[1], q1[1]};
                    const uint32_t a1[4] = {q0[2], q1[2], q0[3], q1[3]};
                    float dw[2];
#pragma unroll
                    for (int h = 0; h < 2; ++h) dw[h] = f16_bits_to_f32((unsigned short)(dq[i][h][bp] >> (16 * bs)));
#pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        const float c4[4] = {cs[j].x, cs[j].y, cs[j].x, cs[j].y};
                        const float2 sx = make_float2(cs[j].z, cs[j].w);
                        float dd[4];
                        mma16816(dd, a0, f[j].x, f[j].y, c4);
                        mma16816(dd, a1, f[j].z, f[j].w, dd);  // 2^-24 x the integer block dots
                        acc[i][j][0] =
                            ffma2_scaled(make_float2(dw[0], dw[0]), sx, make_float2(dd[0], dd[1]), acc[i][j][0]);
                        acc[i][j][1] =
                            ffma2_scaled(make_float2(dw[1], dw[1]), sx, make_float2(dd[2], dd[3]), acc[i][j][1]);
                    }
                }
            }
        };
        if (work) compute_pair(0);
        // unit v + 1's fragments, between the two halves of unit v's work so
        // that their latency hides behind it
        if (v + 1 < V) {
            if (!failed && !wait_phase(&full[(v + 1) % S], ((v + 1) / S) & 1, abort_flag)) fail();
            if (stager && !failed) stage_x(v + 1, buf ^ 1);
            __syncwarp();
            if (lane == 0) mbar_arrive(&xfull[buf ^ 1]);
        }
        if constexpr (KPB == 4) {
            if (work) compute_pair(1);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&xempty[buf]);  // unit read: its stage and fragments may be reused
        if (++u == nunits) {
            u = 0;
            if constexpr (multi) ++ck;
        }
    }
    if (failed && tid == 0) {  // copies still in flight land before the ring is reused or the CTA exits
        for (int w = max(0, issued - S); w < issued; ++w) {
            const uint64_t t0 = global_ns();
            while (!mbar_try_wait(&full[w % S], (w / S) & 1) && global_ns() - t0 < WAIT_LIMIT_NS) {
            }
        }
    }

    // ---------------- the last chunk's sums, through the ring (every warp has
    // finished reading it and no copy fills it any more: each was waited for)
    __syncthreads();
    if constexpr (split) {
        // this CTA's sums in kp 0's acc; then (after every CTA of the cluster
        // has done so, so rank 0's ring is free) ranks > 0 write theirs into
        // rank 0's ring, slot (rank - 1, rh), and rank 0 adds them in order
        float* red = reinterpret_cast<float*>(ring);
        reduce_partials(red);
        cluster_sync_all();
        if (rank > 0 && kp == 0) {
            uint32_t dst;
            asm("mapa.shared::cluster.u32 %0, %1, 0;"
                : "=r"(dst)
                : "r"(smem_u32(red + ((rank - 1) * SH::RH + rh) * SLOT + lane)));
#pragma unroll
            for (int i = 0; i < WT; ++i)
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    const uint32_t q = dst + (uint32_t)((i * NT + j) * 128 * 4);
                    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(q), "f"(acc[i][j][0].x) : "memory");
                    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(q + 128), "f"(acc[i][j][0].y) : "memory");
                    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(q + 256), "f"(acc[i][j][1].x) : "memory");
                    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(q + 384), "f"(acc[i][j][1].y) : "memory");
                }
        }
        cluster_sync_all();
        if (rank == 0 && kp == 0) {
#pragma unroll 1
            for (uint32_t r = 1; r < nsplit; ++r) {
                const float* rp = red + ((r - 1) * SH::RH + rh) * SLOT + lane;
#pragma unroll
                for (int i = 0; i < WT; ++i)
#pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        const float* q = rp + (i * NT + j) * 128;
                        acc[i][j][0].x += q[0];
                        acc[i][j][0].y += q[32];
                        acc[i][j][1].x += q[64];
                        acc[i][j][1].y += q[96];
                    }
            }
            store_rows(chunk0 * RPC);
        }
    } else {
        if (V > 0) reduce_store((chunk0 + nck - 1) * RPC, reinterpret_cast<float*>(ring));
    }
}

template <int NT, int WT, int KPB, int MODE>
qmm_status launch(const uint8_t* w_qs, const uint16_t* w_d, int64_t N, int64_t K, int64_t M, const int8_t* xq,
                  const uint16_t* xd, float* y, int64_t ldy, int nchunk, int nsplit, int smem_optin, int* err,
                  cudaStream_t st) {
    using SH = Shape<NT, WT, KPB>;
    if ((MODE == MULTI) != (nchunk > 1) || (MODE == SPLIT) != (nsplit > 1) || nsplit > 8) return QMM_ERR_SHAPE;
    const int64_t B = K / QK;
    const int64_t nunits = ((B + UKB - 1) / UKB + nsplit - 1) / nsplit * nchunk;
    // a chunk that ends before the last adds its sums in one stage; the
    // ranks of a split hand theirs to rank 0's ring
    if (nchunk > 1 && SH::RED > SH::STAGE) return QMM_ERR_SHAPE;
    const int fixed = 1024 + 2 * SH::XBUF + 2 * SH::XSC + 1024;  // barriers, buffers, alignment slack
    const int64_t nst = std::min<int64_t>({(int64_t)MAX_STAGES, (smem_optin - fixed) / SH::STAGE, nunits + 1});
    if (nst < 2) return QMM_ERR_SHAPE;
    // the ring also holds the final partial sums
    const int64_t ring = std::max<int64_t>({nst * SH::STAGE, (int64_t)SH::RED,
                                            (int64_t)(nsplit - 1) * SH::RH * WT * NT * 512});
    Args a = {};
    a.N = N;
    a.K = K;
    a.M = M;
    a.ldy = ldy;
    a.y = y;
    a.nchunk = nchunk;
    a.nstages = (int)nst;
    a.off_xbuf = 1024 + (int)ring;
    a.off_xsc = a.off_xbuf + 2 * SH::XBUF;
    a.err = err;
    const int64_t smem = a.off_xsc + 2 * SH::XSC + 1024;
    if (smem > smem_optin) return QMM_ERR_SHAPE;
    CUtensorMap mq, md, mxq, mxd;
    // nibbles as [K / 256 chunks of 128 bytes][N rows][128]: one box = the
    // unit's two columns; codes as [K / 128][M][128]: one box = its 4 blocks
    // of 4 (each a 128-byte row per token)
    const uint64_t dq3[3] = {128, (uint64_t)N, (uint64_t)K / 256}, sq3[2] = {(uint64_t)K / 2, 128};
    const uint32_t bq3[3] = {128, (uint32_t)SH::RPC, 2};
    const uint64_t dx3[3] = {128, (uint64_t)M, (uint64_t)K / 128}, sx3[2] = {(uint64_t)K, 128};
    const uint32_t bx3[3] = {128, (uint32_t)SH::TK, 4};
    if (!make_tensor_map_3d(&mq, CU_TENSOR_MAP_DATA_TYPE_UINT8, w_qs, dq3, sq3, bq3, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map_2d(&md, CU_TENSOR_MAP_DATA_TYPE_UINT16, w_d, (uint64_t)B, (uint64_t)N, (uint64_t)B * 2,
                            (uint32_t)UKB, (uint32_t)SH::RPC, CU_TENSOR_MAP_SWIZZLE_32B) ||
        !make_tensor_map_3d(&mxq, CU_TENSOR_MAP_DATA_TYPE_UINT8, xq, dx3, sx3, bx3, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map_2d(&mxd, CU_TENSOR_MAP_DATA_TYPE_UINT16, xd, (uint64_t)B, (uint64_t)M, (uint64_t)B * 2,
                            (uint32_t)UKB, (uint32_t)SH::TK, CU_TENSOR_MAP_SWIZZLE_NONE))
        return QMM_ERR_CUDA;
    auto kern = gemm_wide_kernel<NT, WT, KPB, MODE>;
    if (!allow_smem(kern, smem_optin)) return QMM_ERR_SHAPE;
    const int64_t chunks = (N + SH::RPC - 1) / SH::RPC;
    const dim3 grid((unsigned)((chunks + nchunk - 1) / nchunk * nsplit), (unsigned)((M + SH::TK - 1) / SH::TK));
    if (MODE != SPLIT) {
        kern<<<grid, THREADS, (int)smem, st>>>(mq, md, mxq, mxd, a);
    } else {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = grid;
        cfg.blockDim = dim3(THREADS);
        cfg.dynamicSmemBytes = (size_t)smem;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)nsplit;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, kern, mq, md, mxq, mxd, a) != cudaSuccess) {
            cudaGetLastError();
            return QMM_ERR_CUDA;
        }
    }
    return cudaGetLastError() == cudaSuccess ? QMM_OK : QMM_ERR_CUDA;
}

// Row plan at one CTA per SM: chunks of `rpc` rows (two or three row tiles
// per warp), `nchunk` of them per CTA, or rpc = 0 where the layout does not
// qualify.  It is used when its rows per CTA (nchunk * rpc) exceed those of
// the row-group kernel's 16-row granule by at most 8%.
//  - up to 192 rows per CTA: one chunk of 128 or 192 rows, or 96 rows (three
//    32-row sets, 8 warps splitting a unit's blocks) for 9..16 tokens only
//    (with 8 or fewer the row-group kernel measured faster there: 14336 x
//    4096 14.5 against 15.1 us at 8 tokens, 20.7 against 18.5 at 16).  With
//    one row tile per warp the per-unit hand-over and staging cost more
//    than the 16 warps save (8192 x 28672 at 16 tokens 91 us against 69 us,
//    4096 x 14336 40 against 28), and 256 rows leave room for two stages.
//  - more: several chunks of 128 or 192 rows, whichever needs fewer rows
//    per CTA (192 on a tie).
//  - fewer rows (at most 64 per SM): chunks of 128 or 192 rows, each shared
//    by a cluster of nsplit = min(4, SMs / chunks) >= 2 CTAs splitting K,
//    when every rank gets at least 6 units of 16 blocks; of the two, the
//    one with fewer rows x units on the busiest CTA, 192-row chunks counted
//    at 0.9 for their cheaper blocks (three row tiles per warp: 8192 x 28672
//    at 16 tokens 59.9 -> 51.7 us, 4 tokens 43.1 -> 37.0).  Clusters of up
//    to 4 CTAs of one SM each pack a GB300's 152 SMs (76, 46 and 36 of them
//    at once: 152, 138, 144 CTAs); of 5 to 8, 28, 23, 15 and 15 fit (140,
//    138, 105, 120 CTAs), and 5-CTA clusters behind the workspace entry's
//    preparation launch measured 19-28% slower than 3-CTA ones.  With
//    split192 false only 128-row chunks are split: the workspace entry's
//    plan, where 3-CTA clusters placed behind the previous product's tail
//    varied from run to run (the batch-16 dense set 0.296-0.311 ms against
//    0.300 steady with 2-CTA clusters).
struct Plan {
    int rpc = 0, nchunk = 1, nsplit = 1;
};

Plan plan_rows(int64_t N, int64_t K, int64_t M, int sms, bool split192 = true) {
    Plan p;
    const int64_t need = (N + sms - 1) / sms;
    const int64_t r16 = round_up(need, 16);
    const auto ok = [&](int64_t rows) { return rows * 100 <= r16 * 108; };
    if (need <= 64) {
        const int64_t units = (K / QK + UKB - 1) / UKB;
        int64_t best = 0;  // rows x units of the busiest CTA, 192-row chunks weighted 0.9
        for (const int rpc : {192, 128}) {
            if (rpc == 192 && !split192) continue;
            const int64_t chunks = (N + rpc - 1) / rpc;
            const int64_t ns = std::min<int64_t>(4, sms / chunks);
            if (ns < 2 || units < 6 * ns) continue;
            const int64_t cost = rpc * ((units + ns - 1) / ns) * (rpc == 192 ? 9 : 10);
            if (best == 0 || cost < best) {
                best = cost;
                p.rpc = rpc;
                p.nsplit = (int)ns;
            }
        }
        return p;
    }
    if (need <= 192) {
        if (ok(round_up(need, 64))) p.rpc = need <= 128 ? 128 : 192;
        else if (M > 8 && need <= 96 && ok(round_up(need, 32))) p.rpc = 96;
        return p;
    }
    const int64_t n128 = ((N + 127) / 128 + sms - 1) / sms, n192 = ((N + 191) / 192 + sms - 1) / sms;
    if (n192 * 192 <= n128 * 128) {
        p.rpc = 192;
        p.nchunk = (int)n192;
    } else {
        p.rpc = 128;
        p.nchunk = (int)n128;
    }
    if (!ok((int64_t)p.rpc * p.nchunk) || p.nchunk > (1 << 20)) p = Plan();
    return p;
}

template <int NT>
bool plan_launch(const uint8_t* w_qs, const uint16_t* w_d, int64_t N, int64_t K, int64_t M, const int8_t* xq,
                 const uint16_t* xd, float* y, int64_t ldy, int sms, int smem_optin, int* err, cudaStream_t st,
                 qmm_status* out) {
    if (reinterpret_cast<uintptr_t>(xd) % 16 != 0) return false;
    const Plan p = plan_rows(N, K, M, sms);
    const int nc = p.nchunk, ns = p.nsplit;
    switch (p.rpc) {
        case 128:
            *out = ns > 1   ? launch<NT, 2, 4, SPLIT>(w_qs, w_d, N, K, M, xq, xd, y, ldy, 1, ns, smem_optin, err, st)
                   : nc > 1 ? launch<NT, 2, 4, MULTI>(w_qs, w_d, N, K, M, xq, xd, y, ldy, nc, 1, smem_optin, err, st)
                            : launch<NT, 2, 4, ONE>(w_qs, w_d, N, K, M, xq, xd, y, ldy, 1, 1, smem_optin, err, st);
            return true;
        case 192:
            *out = ns > 1   ? launch<NT, 3, 4, SPLIT>(w_qs, w_d, N, K, M, xq, xd, y, ldy, 1, ns, smem_optin, err, st)
                   : nc > 1 ? launch<NT, 3, 4, MULTI>(w_qs, w_d, N, K, M, xq, xd, y, ldy, nc, 1, smem_optin, err, st)
                            : launch<NT, 3, 4, ONE>(w_qs, w_d, N, K, M, xq, xd, y, ldy, 1, 1, smem_optin, err, st);
            return true;
        case 96:  // one chunk only
            *out = launch<NT, 3, 2, ONE>(w_qs, w_d, N, K, M, xq, xd, y, ldy, 1, 1, smem_optin, err, st);
            return true;
        default: return false;
    }
}

}  // namespace widek

}  // namespace mmak

WidePlan gemm_wide_plan(int64_t N, int64_t K, int64_t M, int sms, bool split192) {
    const mmak::widek::Plan p = mmak::widek::plan_rows(N, K, M, sms, split192);
    return WidePlan{p.rpc, p.nchunk, p.nsplit, sms};
}

bool gemm_wide_planned(int64_t N, int64_t K, int64_t M, const void* xd, int sms) {
    return M >= 1 && M <= 16 && reinterpret_cast<uintptr_t>(xd) % 16 == 0 && mmak::widek::plan_rows(N, K, M, sms).rpc > 0;
}

bool gemm_mma_eligible(int64_t N, int64_t K, int64_t M, const void* w_qs, const void* w_d, const void* xq,
                       const void* xd) {
    auto al = [](const void* p, uintptr_t n) { return reinterpret_cast<uintptr_t>(p) % n == 0; };
    return N >= 1 && N < (int64_t(1) << 31) && M >= 1 && K >= 256 && K % 256 == 0 && al(w_qs, 16) && al(w_d, 16) &&
           al(xq, 16) && al(xd, 2);
}

qmm_status gemm_mma_launch(const uint8_t* w_qs, const uint16_t* w_d, int64_t N, int64_t K, int64_t M,
                           const int8_t* xq, const uint16_t* xd, float* y, int64_t ldy, int sms, int smem_optin,
                           int* err, cudaStream_t st, bool wide) {
    qmm_status s = QMM_OK;
    if (wide && M <= 8 && mmak::widek::plan_launch<1>(w_qs, w_d, N, K, M, xq, xd, y, ldy, sms, smem_optin, err, st, &s))
        return s;
    if (wide && M > 8 && M <= 16 &&
        mmak::widek::plan_launch<2>(w_qs, w_d, N, K, M, xq, xd, y, ldy, sms, smem_optin, err, st, &s))
        return s;
    if (M <= 8) return mmak::launch_nt<1>(w_qs, w_d, N, K, M, xq, xd, y, ldy, sms, smem_optin, err, st);
    if (M <= 16) return mmak::launch_nt<2>(w_qs, w_d, N, K, M, xq, xd, y, ldy, sms, smem_optin, err, st);
    if (M <= 32) return mmak::launch_nt<4>(w_qs, w_d, N, K, M, xq, xd, y, ldy, sms, smem_optin, err, st);
    return mmak::launch_nt<8>(w_qs, w_d, N, K, M, xq, xd, y, ldy, sms, smem_optin, err, st);
}

}  // namespace qmm
