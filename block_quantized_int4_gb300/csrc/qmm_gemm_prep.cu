// qmm_gemm_prep.cu -- the small-batch GEMM (up to 16 tokens) with its
// activation operand prepared once per call (qmm_gemm_q4_0_q8_0_ws).
//
// Same arithmetic as the 16-warp layout of qmm_gemm_mma.cu (exact integer
// block dots on mma.sync m16n8k16 with the weight nibbles as fp16
// subnormals, fp32 rescale per block; llama.cpp guide, kenji.blog/id,
// section 2.2: y ~ Delta * Delta_x * sum q * q_x), and the same row plans.
// What differs is where the activation's fp16 B fragments come from:
//  - a small launch ahead of the product turns the Q8_0 codes and scales of
//    the (up to 16) token rows into the fragments, MMA seeds and scaled d_x
//    of every 16-block unit of K, once, into a caller-owned workspace;
//  - each ring stage of the product then carries, beside the unit's weight
//    tiles, that unit's prepared record (one bulk copy from L2), so no CTA
//    converts activation codes and no warp waits for another to have done
//    so: the per-unit hand-over of the staged layout disappears;
//  - a stage is refilled by the last warp to finish with it (a per-stage
//    arrival counter), so no warp is held to the pace of the slowest one
//    except through the ring's depth.
// The fp32 results are those of the staged layout bit for bit (same
// fragments, same MMA and accumulation order, same reductions) under the same
// row plan.  The plans differ in two places: under the EVEN mode below, a
// row chunk cut between two CTAs sums its two parts separately (then added
// in one fixed order: the same bits every call); and K is split over
// clusters sharing 128-row chunks only (the plain entry also splits 192-row
// chunks).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "qmm_device.cuh"
#include "qmm_mma.h"
#include "qmm_mma_frag.cuh"
#include "qmm_tmap.h"

namespace qmm {
namespace prepk {

using namespace frag;

constexpr int CW = 16;
constexpr int THREADS = CW * 32;
constexpr int UKB = 16;  // blocks per unit
constexpr int MAX_STAGES = 8;
// Modes: ONE chunk of rows per CTA; MULTI: nchunk chunks per CTA; SPLIT: a
// cluster of CTAs splitting one chunk's K; EVEN: the (chunk, unit) sequence
// of the whole product cut into equal runs, one per CTA.  A chunk cut between
// two CTAs: the later CTA meets the chunk's end at the start of its run, so
// it stores its partial sums into y and raises the chunk's flag in the
// workspace; the earlier CTA meets the chunk's start at the end of its run,
// long after, adds those partial sums to its own (one fixed order) and
// writes y.
enum Mode { ONE = 0, MULTI = 1, SPLIT = 2, EVEN = 3 };
constexpr int MAX_FLAGS = 4096;  // chunks an EVEN product may have (one flag word each)

// One unit's prepared record for NT token tiles (TK = 8 NT token rows):
//   fragments [16 blocks][NT tiles][32 lanes] x 16 bytes: lane (g, t) of
//     tile j holds token 8 j + g's word t of the block's low half as the fp16
//     pairs (x0, x2), (x1, x3), then word t of the high half divided by 16,
//     likewise (the B operand of the block's two m16n8k16 MMAs);
//   pairs [16 blocks][NT * 4] float4: for tokens (8 j + 2 t, 8 j + 2 t + 1):
//     the MMA seeds -8 * 2^-24 * (sum of the block's codes) and 2^24 d_x.
template <int NT>
struct Rec {
    static constexpr int FRAG = UKB * NT * 512;
    static constexpr int BYTES = FRAG + UKB * NT * 64;
};

// ---------------------------------------------------------------- preparation
// One CTA per unit; thread = (block of the unit, token, half block).  Tokens
// at or past M and blocks past K give zero codes, seeds and scales.
template <int NT>
__global__ void __launch_bounds__(UKB * 16 * NT) prep_kernel(const int8_t* __restrict__ xq,
                                                             const uint16_t* __restrict__ xd, int64_t K, int64_t M,
                                                             uint8_t* __restrict__ rec, int* __restrict__ flags) {
    constexpr int TK = 8 * NT;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the codes come from the kernel before
    if (blockIdx.x == 0)  // the EVEN mode's chunk flags start lowered
        for (int i = threadIdx.x; i < MAX_FLAGS; i += blockDim.x) flags[i] = 0;
    const int B = (int)(K / QK);
    const int tid = threadIdx.x, sh = tid & 1, tok = (tid >> 1) & (TK - 1), bl = tid / (2 * TK);
    const int b = blockIdx.x * UKB + bl;
    uint4 px = make_uint4(0u, 0u, 0u, 0u);
    uint32_t ps = 0u;
    if (tok < M && b < B) {
        px = __ldg(reinterpret_cast<const uint4*>(xq + (int64_t)tok * K + (int64_t)b * QK) + sh);
        ps = __ldg(xd + (int64_t)tok * B + b);
    }
    int sum = __dp4a((int)px.x, 0x01010101, 0);
    sum = __dp4a((int)px.y, 0x01010101, sum);
    sum = __dp4a((int)px.z, 0x01010101, sum);
    sum = __dp4a((int)px.w, 0x01010101, sum);
    const int other = __shfl_xor_sync(FULL, sum, 1);
    uint8_t* r = rec + (size_t)blockIdx.x * Rec<NT>::BYTES;
    // (1152 + x) * mul + add = x (low half) or x / 16 (high half), exact
    const uint32_t mul = sh ? 0x2C002C00u : 0x3C003C00u, add = sh ? 0xD480D480u : 0xE480E480u;
    const uint32_t w4[4] = {px.x, px.y, px.z, px.w};
    uint8_t* dst = r + (size_t)(bl * NT * 32 + tok * 4) * 16 + sh * 8;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        uint2 p;
        p.x = hfma2((w4[t] & 0x00FF00FFu) ^ 0x64806480u, mul, add);
        p.y = hfma2(((w4[t] >> 8) & 0x00FF00FFu) ^ 0x64806480u, mul, add);
        *reinterpret_cast<uint2*>(dst + t * 16) = p;
    }
    if (sh == 0) {
        float* xs = reinterpret_cast<float*>(r + Rec<NT>::FRAG);
        const int pr = (bl * TK + tok) >> 1, od = tok & 1;
        xs[pr * 4 + od] = (float)(-8 * (sum + other)) * 0x1p-24f;
        xs[pr * 4 + 2 + od] = f16_bits_to_f32((unsigned short)ps) * 0x1p24f;
    }
}

// ---------------------------------------------------------------- product
template <int NT, int WT, int KPB>
struct Shape {
    static constexpr int KP = UKB / KPB;  // warps splitting a unit's blocks
    static constexpr int RH = CW / KP;    // warps splitting the rows
    static constexpr int RPC = 16 * RH * WT;
    static constexpr int QB = 2 * RPC * 128;             // nibble columns [2][RPC][128], 128-byte swizzled
    static constexpr int OFF_REC = QB + RPC * UKB * 2;  // after the weight scales [RPC][16] fp16, 32-byte swizzled
    static constexpr int STAGE = (OFF_REC + Rec<NT>::BYTES + 1023) / 1024 * 1024;
    static constexpr int TX = OFF_REC + Rec<NT>::BYTES;  // bytes a unit's copies deliver
    static constexpr int RED = RH * (KP - 1) * WT * NT * 512;
    static_assert(RH * KP == CW && KPB % 2 == 0 && OFF_REC % 16 == 0, "warp split");
};

struct Args {
    int64_t N, K, M, ldy;
    float* y;
    const uint8_t* rec;  // prepared records, one per unit of K
    int* flags;          // EVEN: one word per chunk, lowered by the preparation launch
    int64_t units_total;  // EVEN: chunks x units per chunk
    int nchunk, nstages;
    int* err;
};

template <int NT, int WT, int KPB, int MODE>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_prep_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_d, Args a) {
    using SH = Shape<NT, WT, KPB>;
    constexpr int KP = SH::KP, RPC = SH::RPC, QB = SH::QB;
    constexpr bool multi = MODE == MULTI, split = MODE == SPLIT, even = MODE == EVEN;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(base);                    // [MAX_STAGES] a unit's bytes landed
    unsigned* done = reinterpret_cast<unsigned*>(full + MAX_STAGES);       // [MAX_STAGES] warps done, ever
    volatile int* abort_flag = reinterpret_cast<volatile int*>(done + MAX_STAGES);
    uint8_t* ring = base + 1024;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = (int)(a.K / QK);
    const int S = a.nstages;
    int nunits = (B + UKB - 1) / UKB, u_lo = 0;  // units of a chunk this CTA takes
    uint32_t rank = 0, nsplit = 1;
    if constexpr (split) {
        asm("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
        asm("mov.u32 %0, %%cluster_nctarank;" : "=r"(nsplit));
        const int per = (nunits + (int)nsplit - 1) / (int)nsplit;
        u_lo = min(nunits, (int)rank * per);
        nunits = min(nunits, u_lo + per) - u_lo;
    }
    // EVEN: this CTA's run [g0, g1) of the product's (chunk, unit) sequence
    const int64_t g0 = even ? a.units_total * blockIdx.x / gridDim.x : 0;
    const int64_t g1 = even ? a.units_total * (blockIdx.x + 1) / gridDim.x : 0;
    const int64_t chunk0 = even    ? g0 / nunits
                           : multi ? (int64_t)blockIdx.x * a.nchunk
                           : split ? (int64_t)(blockIdx.x / nsplit)
                                   : (int64_t)blockIdx.x;
    const int u0 = even ? (int)(g0 - chunk0 * nunits) : 0;  // first unit, inside its chunk
    const int nck = multi ? (int)min((int64_t)a.nchunk, (a.N + RPC - 1) / RPC - chunk0) : 1;
    const int V = even ? (int)(g1 - g0) : multi ? nck * nunits : nunits;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            done[s] = 0u;
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // The copies of unit v into stage v % S, from lanes 0..2 of one warp in
    // parallel: the nibble columns (3D box) with the unit's byte count, the
    // weight scales, and the prepared record (a bulk copy from L2).  Weights
    // are evicted first from L2; the records, read by every CTA, are not.
    const uint64_t pol = l2_evict_first_policy();
    auto issue = [&](int v, bool weights, bool acts) {
        int64_t c;
        int u;
        if constexpr (even) {
            const int64_t g = g0 + v;
            c = g / nunits;
            u = (int)(g - c * nunits);
        } else {
            const int ck = multi ? v / nunits : 0;
            c = chunk0 + ck;
            u = u_lo + v - ck * nunits;
        }
        const int s = v % S, b0 = u * UKB;
        const int row_begin = (int)(c * RPC);
        uint8_t* st = ring + (size_t)s * SH::STAGE;
        if (lane == 0 && weights) {
            mbar_arrive_expect_tx(&full[s], (uint32_t)SH::TX);
            tma3d_ef(st, &map_q, 0, row_begin, b0 / 8, &full[s], pol);
        } else if (lane == 1 && weights) {
            tma2d(st + QB, &map_d, b0, row_begin, &full[s], pol);
        } else if (lane == 2 && acts) {
            bulk_g2s(st + SH::OFF_REC, a.rec + (size_t)u * Rec<NT>::BYTES, (uint32_t)Rec<NT>::BYTES, &full[s]);
        }
    };
    int issued = min(S, V);
    if (warp == 0 && V > 0) issue(0, true, false);
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the records come from the preparation launch
    if (warp == 0 && V > 0) {
        issue(0, false, true);
        for (int v = 1; v < issued; ++v) issue(v, true, true);
    }

    const int g8 = lane >> 2, t4 = lane & 3;
    const int kp = warp % KP, rh = warp / KP;
    const int fb = kp * KPB, kb = fb >> 3, c0 = fb & 7;  // first block of the warp; its column, slot in it
    const int64_t m0 = (int64_t)blockIdx.y * (8 * NT);

    float2 acc[WT][NT][2];
#pragma unroll
    for (int i = 0; i < WT; ++i)
#pragma unroll
        for (int j = 0; j < NT; ++j) acc[i][j][0] = acc[i][j][1] = make_float2(0.f, 0.f);
    // scale-tile offsets (fp16 units) of this lane's rows; ldmatrix row
    // addresses (lane l: row l % 8 of matrix l / 8 = (row half, block of the pair))
    int doff[WT][2];
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

    constexpr int SLOT = WT * NT * 128;  // floats per warp
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

    int u = u0, ck = 0;  // unit inside the chunk, chunk of this CTA (from chunk0)
    for (int v = 0; v < V; ++v) {
        const int s = v % S;
        if (!failed && !wait_phase(&full[s], (v / S) & 1, abort_flag)) {
            if (lane == 0) atomicOr(a.err, ERR_TIMEOUT);
            *abort_flag = 1;
            failed = true;
        }
        const int nb = min(UKB, B - (u_lo + u) * UKB);
        if (!failed && fb < nb) {
            const uint8_t* st = ring + (size_t)s * SH::STAGE;
            const uint32_t st_u32 = smem_u32(st);
            const uint16_t* sd = reinterpret_cast<const uint16_t*>(st + QB);
            const uint8_t* xf0 = st + SH::OFF_REC + lane * 16;
            const float4* xs0 = reinterpret_cast<const float4*>(st + SH::OFF_REC + Rec<NT>::FRAG) + t4;
            uint32_t dq[WT][2][KPB / 2];
#pragma unroll
            for (int i = 0; i < WT; ++i)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if constexpr (KPB == 4) {
                        const uint2 q = *reinterpret_cast<const uint2*>(sd + doff[i][h]);
                        dq[i][h][0] = q.x;
                        dq[i][h][1] = q.y;
                    } else {
                        dq[i][h][0] = *reinterpret_cast<const uint32_t*>(sd + doff[i][h]);
                    }
                }
#pragma unroll
            for (int bp = 0; bp < KPB / 2; ++bp) {
                uint32_t wq[WT][4];
#pragma unroll
                for (int i = 0; i < WT; ++i) ldsm_x4(st_u32 + (qaddr[i] ^ (uint32_t)(bp << 5)), wq[i]);
#pragma unroll
                for (int bs = 0; bs < 2; ++bs) {
                    const int b = fb + 2 * bp + bs;
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
            }
        }
        // The stage is released: the last warp to do so refills it with unit
        // v + S (at a chunk's end the refill waits for the chunk's sums, which
        // go through this stage).  The counter only grows: after the n-th use
        // of stage s the last arrival sees (n + 1) * 16 - 1.
        const bool chunk_end = (multi && u == nunits - 1) || (even && (u == nunits - 1 || v == V - 1));
        __syncwarp();
        unsigned prev = 0;
        if (lane == 0) {
            __threadfence_block();  // this warp's reads of the stage come first
            prev = atomicAdd(&done[s], 1u);
            __threadfence_block();
        }
        prev = __shfl_sync(FULL, prev, 0);
        if (prev == (unsigned)((v / S + 1) * CW - 1) && !chunk_end && v + S < V) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(v + S, true, true);
        }
        if constexpr (multi || even) {
            if (chunk_end) {
                const int64_t c = chunk0 + ck;
                // EVEN: which ends of chunk c this CTA's run holds
                const bool has_start = !even || c * nunits >= g0, has_end = !even || (c + 1) * nunits <= g1;
                asm volatile("bar.sync 1, %0;" ::"r"(THREADS) : "memory");  // every warp done with the chunk
                reduce_partials(reinterpret_cast<float*>(ring + (size_t)s * SH::STAGE));
                if (!has_end) {
                    // the end of the chunk was the next CTA's, done at the start of
                    // its run: wait for its partial sums in y (bounded), add them
                    if (tid == 0) {
                        const uint64_t t0 = global_ns();
                        int f = 0;
                        while (!*abort_flag) {
                            asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(f) : "l"(a.flags + c) : "memory");
                            if (f || global_ns() - t0 > WAIT_LIMIT_NS) break;
                        }
                        if (!f) {
                            atomicOr(a.err, ERR_TIMEOUT);
                            *abort_flag = 1;
                        }
                    }
                    asm volatile("bar.sync 1, %0;" ::"r"(THREADS) : "memory");
                    if (*abort_flag) failed = true;
                    if (kp == 0 && !failed) {
#pragma unroll
                        for (int i = 0; i < WT; ++i)
#pragma unroll
                            for (int j = 0; j < NT; ++j) {
                                const int64_t m = m0 + 8 * j + 2 * t4;
#pragma unroll
                                for (int h = 0; h < 2; ++h) {
                                    const int64_t row = c * RPC + (rh * WT + i) * 16 + g8 + 8 * h;
                                    if (row >= a.N) continue;
                                    if (m < a.M) acc[i][j][h].x += __ldcg(a.y + m * a.ldy + row);
                                    if (m + 1 < a.M) acc[i][j][h].y += __ldcg(a.y + (m + 1) * a.ldy + row);
                                }
                            }
                    }
                }
                store_rows(c * RPC);  // whole chunk or its start (with the end added): final; its end only: partial
                asm volatile("bar.sync 1, %0;" ::"r"(THREADS) : "memory");  // the sums read before the refill
                if (!has_start && tid == 0) {  // the partial sums are in y: raise the chunk's flag
                    __threadfence();
                    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(a.flags + c), "r"(1) : "memory");
                }
#pragma unroll
                for (int i = 0; i < WT; ++i)
#pragma unroll
                    for (int j = 0; j < NT; ++j) acc[i][j][0] = acc[i][j][1] = make_float2(0.f, 0.f);
                if (warp == 0 && v + S < V) {
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    issue(v + S, true, true);
                }
            }
        }
        if (++u == nunits) {
            u = 0;
            if constexpr (multi || even) ++ck;
        }
    }
    if (failed && tid == 0) {  // copies still in flight land before the ring is reused or the CTA exits
        for (int w = max(0, V - S); w < V; ++w) {
            const uint64_t t0 = global_ns();
            while (!mbar_try_wait(&full[w % S], (w / S) & 1) && global_ns() - t0 < WAIT_LIMIT_NS) {
            }
        }
    }

    // ---------------- the last chunk's sums (through the ring, which no copy fills any more)
    __syncthreads();
    if constexpr (split) {
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
    } else if constexpr (!multi && !even) {
        if (V > 0) {
            reduce_partials(reinterpret_cast<float*>(ring));
            store_rows(chunk0 * RPC);
        }
    }
}

// Launch with programmatic dependent launch (and a cluster for SPLIT).
template <typename Kern, typename... Args>
cudaError_t launch_ex(Kern kernel, dim3 grid, int threads, size_t smem, cudaStream_t st, int cluster, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    int n = 1;
    if (cluster > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = (unsigned)cluster;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        n = 2;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Everything the product needs is checked and encoded first; only then are
// the preparation launch and the product launched, so a call that fails
// before its launches enqueues nothing.
template <int NT, int WT, int KPB, int MODE>
qmm_status launch(const uint8_t* w_qs, const uint16_t* w_d, int64_t N, int64_t K, int64_t M, const int8_t* xq,
                  const uint16_t* xd, float* y, int64_t ldy, uint8_t* rec, int nchunk, int nsplit, int smem_optin,
                  int* err, cudaStream_t st, int sms_even = 0) {
    using SH = Shape<NT, WT, KPB>;
    if ((MODE == MULTI) != (nchunk > 1) || (MODE == SPLIT) != (nsplit > 1) || nsplit > 8) return QMM_ERR_SHAPE;
    if ((nchunk > 1 || MODE == EVEN) && SH::RED > SH::STAGE) return QMM_ERR_SHAPE;
    const int64_t B = K / QK;
    const int64_t units_all = (B + UKB - 1) / UKB;
    const int64_t chunks = (N + SH::RPC - 1) / SH::RPC;
    // EVEN: one run per SM, each at least a chunk long (so a chunk is cut at
    // most once), and one flag word per chunk
    if (MODE == EVEN && (chunks < sms_even || chunks > MAX_FLAGS)) return QMM_ERR_SHAPE;
    const int64_t units = MODE == EVEN ? (chunks * units_all + sms_even - 1) / sms_even
                                       : (units_all + nsplit - 1) / nsplit * nchunk;
    const int fixed = 1024 + 1024;  // barriers and counters, alignment slack
    const int64_t nst = std::min<int64_t>({(int64_t)MAX_STAGES, (smem_optin - fixed) / SH::STAGE, units});
    if (nst < 1) return QMM_ERR_SHAPE;
    const int64_t ring = std::max<int64_t>({nst * SH::STAGE, (int64_t)SH::RED,
                                            (int64_t)(nsplit - 1) * SH::RH * WT * NT * 512});
    const int64_t smem = 1024 + ring + 1024;
    if (smem > smem_optin) return QMM_ERR_SHAPE;
    Args a = {};
    a.N = N;
    a.K = K;
    a.M = M;
    a.ldy = ldy;
    a.y = y;
    a.rec = rec;
    a.flags = reinterpret_cast<int*>(rec + units_all * Rec<NT>::BYTES);
    a.units_total = chunks * units_all;
    a.nchunk = nchunk;
    a.nstages = (int)nst;
    a.err = err;
    CUtensorMap mq, md;
    const uint64_t dq3[3] = {128, (uint64_t)N, (uint64_t)K / 256}, sq3[2] = {(uint64_t)K / 2, 128};
    const uint32_t bq3[3] = {128, (uint32_t)SH::RPC, 2};
    if (!make_tensor_map_3d(&mq, CU_TENSOR_MAP_DATA_TYPE_UINT8, w_qs, dq3, sq3, bq3, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map_2d(&md, CU_TENSOR_MAP_DATA_TYPE_UINT16, w_d, (uint64_t)B, (uint64_t)N, (uint64_t)B * 2,
                            (uint32_t)UKB, (uint32_t)SH::RPC, CU_TENSOR_MAP_SWIZZLE_32B))
        return QMM_ERR_CUDA;
    auto kern = gemm_prep_kernel<NT, WT, KPB, MODE>;
    if (!allow_smem(kern, smem_optin)) return QMM_ERR_SHAPE;
    const dim3 grid(MODE == EVEN ? (unsigned)sms_even : (unsigned)((chunks + nchunk - 1) / nchunk * nsplit), 1);
    if (launch_ex(prep_kernel<NT>, dim3((unsigned)units_all), UKB * 16 * NT, 0, st, 1, xq, xd, K, M, rec,
                  a.flags) != cudaSuccess) {
        cudaGetLastError();
        return QMM_ERR_CUDA;
    }
    if (launch_ex(kern, grid, THREADS, (size_t)smem, st, nsplit, mq, md, a) != cudaSuccess) {
        cudaGetLastError();
        return QMM_ERR_CUDA;
    }
    return QMM_OK;
}

template <int NT>
qmm_status launch_nt(const uint8_t* w_qs, const uint16_t* w_d, int64_t N, int64_t K, int64_t M, const int8_t* xq,
                     const uint16_t* xd, float* y, int64_t ldy, const WidePlan& p, uint8_t* ws, int smem_optin,
                     int* err, cudaStream_t st) {
    const int nc = p.nchunk, ns = p.nsplit;
    // several chunks per CTA: the even cut over the SMs of 192-row chunks,
    // where every SM's run is at least a chunk long and the busiest CTA's
    // rows drop by 3% or more (lm_head 128256 rows: 896 -> 844 per SM, 16
    // tokens 182.0 -> 175.7 us; at 58000 rows, 384 -> 383, the cut's own
    // cost made it 2-4% slower)
    if (nc > 1) {
        const int64_t c192 = (N + 191) / 192;
        if (c192 >= p.sms && c192 <= MAX_FLAGS && c192 * 192 * 100 <= (int64_t)nc * p.rpc * p.sms * 97)
            return launch<NT, 3, 4, EVEN>(w_qs, w_d, N, K, M, xq, xd, y, ldy, ws, 1, 1, smem_optin, err, st, p.sms);
    }
    switch (p.rpc) {
        case 128:
            return ns > 1 ? launch<NT, 2, 4, SPLIT>(w_qs, w_d, N, K, M, xq, xd, y, ldy, ws, 1, ns, smem_optin, err, st)
                   : nc > 1
                       ? launch<NT, 2, 4, MULTI>(w_qs, w_d, N, K, M, xq, xd, y, ldy, ws, nc, 1, smem_optin, err, st)
                       : launch<NT, 2, 4, ONE>(w_qs, w_d, N, K, M, xq, xd, y, ldy, ws, 1, 1, smem_optin, err, st);
        case 192:
            return ns > 1   ? launch<NT, 3, 4, SPLIT>(w_qs, w_d, N, K, M, xq, xd, y, ldy, ws, 1, ns, smem_optin, err, st)
                   : nc > 1 ? launch<NT, 3, 4, MULTI>(w_qs, w_d, N, K, M, xq, xd, y, ldy, ws, nc, 1, smem_optin, err, st)
                            : launch<NT, 3, 4, ONE>(w_qs, w_d, N, K, M, xq, xd, y, ldy, ws, 1, 1, smem_optin, err, st);
        case 96: return launch<NT, 3, 2, ONE>(w_qs, w_d, N, K, M, xq, xd, y, ldy, ws, 1, 1, smem_optin, err, st);
        default: return QMM_ERR_SHAPE;
    }
}

}  // namespace prepk

size_t gemm_prep_bytes(int64_t K, int64_t M) {
    if (M < 1 || M > 16 || K <= 0) return 0;
    const int64_t units = (K / QK + prepk::UKB - 1) / prepk::UKB;
    return (size_t)units * (size_t)(M <= 8 ? prepk::Rec<1>::BYTES : prepk::Rec<2>::BYTES) +
           (size_t)prepk::MAX_FLAGS * sizeof(int);
}

qmm_status gemm_prep_launch(const uint8_t* w_qs, const uint16_t* w_d, int64_t N, int64_t K, int64_t M,
                            const int8_t* xq, const uint16_t* xd, float* y, int64_t ldy, const WidePlan& p,
                            void* workspace, int smem_optin, int* err, cudaStream_t st) {
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    return M <= 8 ? prepk::launch_nt<1>(w_qs, w_d, N, K, M, xq, xd, y, ldy, p, ws, smem_optin, err, st)
                  : prepk::launch_nt<2>(w_qs, w_d, N, K, M, xq, xd, y, ldy, p, ws, smem_optin, err, st);
}

}  // namespace qmm
