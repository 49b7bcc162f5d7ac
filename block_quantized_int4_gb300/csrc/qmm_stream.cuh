// qmm_stream.cuh -- streaming GEMV / small-batch GEMM for Q4_0 x Q8_0.
//
// Each CTA owns a contiguous range of weight rows and walks it in groups of
// RB (<= 32) rows; a group is streamed in K chunks of up to 64 blocks.  One
// (group, chunk) "unit" is two 2D TMA copies -- the nibble tile (RB rows x
// 1 KB) and the scale tile (RB rows x 128 B) -- issued by one producer
// thread into a ring of shared-memory stages.  Sixteen consumer warps each
// own two adjacent rows of the group (2w, 2w+1: a gate/up pair stays in one
// warp) for the whole K range: per chunk a lane loads the staged activation
// of its two blocks (lane, lane+32) once into registers and applies it to
// both rows with dp4a; no cross-warp reduction is needed.  After the last
// chunk the warp reduces each row across lanes and writes y (plus a
// residual, or SwiGLU of a gate/up pair).  With a Q8_0 output the CTA's row
// range covers whole 32-output blocks, and the CTA quantizes its own
// outputs, so the next GEMV of a chain only copies its activation.
//
// Decode chains: the producer starts copying before the kernel waits on the
// preceding grid (griddepcontrol.wait), so under programmatic dependent
// launch a kernel's weight stream overlaps the kernel before it; only the
// activation read waits.
//
// Method: llama.cpp guide (kenji.blog/id) section 2.2, y ~ Delta*Delta_x *
// sum q*q_x per block of 32; block format: TinyLLaMA C++ guide (kenji.blog)
// section 6.1; SwiGLU of the gate/up pair: TinyLLaMA guide section 4.4.
#pragma once

#include <cuda.h>

#include "qmm_kernels.cuh"

namespace qmm {

enum YMode { Y_PLAIN = 0, Y_SWIGLU_PAIRS = 1 };

constexpr int SW = 16;  // consumer warps (two rows each)
constexpr int STREAM_THREADS = (SW + 1) * 32;
constexpr int STREAM_HDR = 256;  // barriers + flags
constexpr int STREAM_MAX_STAGES = 8;
constexpr int GROUP_ROWS = 32;   // rows per group (2 per consumer warp)
constexpr int CHUNK_KB = 64;     // K blocks per unit (2 per lane)
constexpr int STAGE_Q = GROUP_ROWS * CHUNK_KB * 16;  // 32 KB
constexpr int STAGE_D = GROUP_ROWS * CHUNK_KB * 2;   //  4 KB
constexpr int STAGE_BYTES = STAGE_Q + STAGE_D;

struct StreamArgs {
    int64_t N, K, M;
    const int8_t* xq;    // X_Q8: [M][K]
    const uint16_t* xd;  // X_Q8: [M][B]
    const float* xf;     // X_F32 / X_SWIGLU: [K] (or [2K])
    const float* residual;  // optional [N] (Y_PLAIN, M == 1)
    int8_t* xq_out;
    uint16_t* xd_out;
    float* y;            // may be NULL when a Q8_0 output is requested
    int64_t ldy;
    int8_t* yq;          // QOUT: Q8_0 codes of the output [N_out]
    uint16_t* yd;        // QOUT: Q8_0 scales [N_out / 32]
    int rows_per_cta;    // even
    int rb;              // rows per group = TMA box rows (even, <= 32)
    int ckb;             // K blocks per chunk = TMA box width in blocks (multiple of 8, <= 64)
    int nstages;
    int xtile_bytes;     // multiple of 128
    int* err;
};

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// Up to two CTAs per SM for the batch-1 variants (<= 60 registers), so a
// chained kernel's CTA fits beside the one before it.
template <int MT, int XMODE, int YMODE, bool QOUT>
__global__ void __launch_bounds__(STREAM_THREADS, MT <= 2 ? 2 : 1)
    stream_rows_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_d,
                       StreamArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + STREAM_MAX_STAGES;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + STREAM_MAX_STAGES);
    const int B = (int)(a.K / QK);
    const XTile xt = xtile_at(smem + STREAM_HDR, MT, B);
    uint8_t* ring = smem + STREAM_HDR + a.xtile_bytes;
    float* ybuf = reinterpret_cast<float*>(ring + (size_t)a.nstages * STAGE_BYTES);  // QOUT: this CTA's outputs
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    const int RB = a.rb, CKB = a.ckb;
    const int64_t row_begin = (int64_t)blockIdx.x * a.rows_per_cta;
    const int64_t row_end = min(a.N, row_begin + a.rows_per_cta);
    const int nrows = (int)max((int64_t)0, row_end - row_begin);
    const int ngroups = (nrows + RB - 1) / RB;
    const int nkc = (B + CKB - 1) / CKB;
    const int nunits = ngroups * nkc;
    const int S = a.nstages;
    const uint32_t unit_bytes = (uint32_t)(RB * CKB * 18);  // full boxes, OOB parts zero-filled

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], SW);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == SW) {
        // ---------------- producer: weights only, independent of earlier grids
        if (lane == 0) {
            int issued = 0;
            bool ok = true;
            for (int u = 0; u < nunits; ++u) {
                const int s = u % S;
                if (u >= S && !mbar_wait(&empty[s], ((u / S) - 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                const int g = u / nkc, kc = u - g * nkc;
                const int r0 = (int)(row_begin + (int64_t)g * RB);
                uint8_t* st = ring + (size_t)s * STAGE_BYTES;
                mbar_arrive_expect_tx(&full[s], unit_bytes);
                tma_load_2d(st, &map_q, kc * CKB * 4, r0, &full[s]);           // u32 columns
                tma_load_2d(st + STAGE_Q, &map_d, kc * CKB, r0, &full[s]);     // fp16 columns
                issued = u + 1;
            }
            if (!ok) {
                atomicOr(a.err, ERR_TIMEOUT);
                *abort_flag = 1;
                for (int u = max(0, issued - S); u < issued; ++u) {  // let issued copies land
                    const uint64_t t0 = global_ns();
                    while (!mbar_try_wait(&full[u % S], (u / S) & 1) && global_ns() - t0 < WAIT_LIMIT_NS) {
                    }
                }
            }
        }
        return;
    }

    // ---------------- consumers
    asm volatile("griddepcontrol.wait;" ::: "memory");
    constexpr int NTHR = SW * 32;
    const int64_t m0 = (int64_t)blockIdx.y * MT;
    int64_t xrow[MT];
#pragma unroll
    for (int t = 0; t < MT; ++t) xrow[t] = (m0 + t < a.M) ? m0 + t : -1;
    if (XMODE == X_Q8) stage_q8<MT>(xt, B, a.xq, a.xd, a.K, xrow, 0, B, tid, NTHR);
    else stage_f32<XMODE == X_SWIGLU>(xt, a.xf, a.K, a.xq_out, a.xd_out, tid, NTHR);
    asm volatile("bar.sync 1, %0;" ::"r"(NTHR) : "memory");

    // this warp's rows inside a group
    const int lr0 = 2 * warp, lr1 = 2 * warp + 1;
    constexpr int OPR = YMODE == Y_SWIGLU_PAIRS ? 2 : 1;  // rows per output
    bool failed = false;
    for (int g = 0; g < ngroups; ++g) {
        const int64_t r0 = row_begin + (int64_t)g * RB;
        const int nr = (int)min((int64_t)RB, row_end - r0);
        float acc0[MT], acc1[MT];
#pragma unroll
        for (int t = 0; t < MT; ++t) acc0[t] = acc1[t] = 0.f;
        for (int kc = 0; kc < nkc; ++kc) {
            const int u = g * nkc + kc, s = u % S;
            // On a timeout keep going without computing: every later wait returns
            // at once (abort flag), and the kernel ends with the error word set.
            const bool ok = !failed && mbar_wait(&full[s], (u / S) & 1, abort_flag);
            if (!ok && !failed) {
                if (lane == 0) atomicOr(a.err, ERR_TIMEOUT);
                *abort_flag = 1;
                failed = true;
            }
            const int b0 = kc * CKB, nb = min(CKB, B - b0);
            if (ok && lr0 < nr) {
                const uint8_t* stq = ring + (size_t)s * STAGE_BYTES;
                const uint16_t* std_ = reinterpret_cast<const uint16_t*>(stq + STAGE_Q);
                const bool has1 = lr1 < nr;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int bl = lane + 32 * h;  // block inside the chunk
                    if (bl >= nb) break;
                    const uint4 w0 = lds128(stq + (lr0 * CKB + bl) * 16);
                    const uint4 w1 = has1 ? lds128(stq + (lr1 * CKB + bl) * 16) : make_uint4(0, 0, 0, 0);
                    const float d0 = f16_bits_to_f32(std_[lr0 * CKB + bl]);
                    const float d1 = has1 ? f16_bits_to_f32(std_[lr1 * CKB + bl]) : 0.f;
#pragma unroll
                    for (int t = 0; t < MT; ++t) {
                        const int i = t * B + b0 + bl;
                        const int4 xl = xt.lo[i], xh = xt.hi[i];
                        const float xs = xt.s[i];
                        const int xc = 8 * xt.sum[i];
                        const int p0 = block_dot_u(w0, xl, xh) - xc;
                        const int p1 = block_dot_u(w1, xl, xh) - xc;
                        acc0[t] = fmaf(d0 * xs, (float)p0, acc0[t]);
                        acc1[t] = fmaf(d1 * xs, (float)p1, acc1[t]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        // reduce the warp's two rows across lanes, write
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            acc0[t] = warp_sum(acc0[t]);
            acc1[t] = warp_sum(acc1[t]);
        }
        if (lane == 0 && !failed && lr0 < nr) {
            const bool has1 = lr1 < nr;
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                if (xrow[t] < 0) continue;
                if (YMODE == Y_SWIGLU_PAIRS) {
                    const float v = swiglu1(acc0[t], acc1[t]);
                    const int64_t o = (r0 + lr0) / 2;
                    if (a.y) a.y[xrow[t] * a.ldy + o] = v;
                    if (QOUT) ybuf[o - row_begin / 2] = v;
                } else {
                    const int64_t row = r0 + lr0;
                    const float v0 = acc0[t] + (a.residual ? a.residual[row] : 0.f);
                    const float v1 = has1 ? acc1[t] + (a.residual ? a.residual[row + 1] : 0.f) : 0.f;
                    if (a.y) {
                        a.y[xrow[t] * a.ldy + row] = v0;
                        if (has1) a.y[xrow[t] * a.ldy + row + 1] = v1;
                    }
                    if (QOUT) {
                        ybuf[row - row_begin] = v0;
                        if (has1) ybuf[row + 1 - row_begin] = v1;
                    }
                }
            }
        }
    }
    if (QOUT) {
        // Q8_0 of this CTA's outputs (whole blocks of 32; M == 1): warp w takes
        // blocks 4w.., eight lanes per block, same rounding as the quantizers.
        asm volatile("bar.sync 1, %0;" ::"r"(NTHR) : "memory");
        const int nout = nrows / OPR;
        const int nblk = nout / QK;
        const int64_t out0 = row_begin / OPR;
        for (int blk0 = warp * 4; blk0 < nblk; blk0 += SW * 4) {
            const int blk = blk0 + (lane >> 3), part = lane & 7;
            const bool valid = blk < nblk && !failed;
            const float4 v = valid ? *reinterpret_cast<const float4*>(ybuf + blk * QK + part * 4)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
            const Quad r = quad_codes(v, 127.0f, -127.0f);
            if (valid) {
                const int packed = (r.c[0] & 0xff) | ((r.c[1] & 0xff) << 8) | ((r.c[2] & 0xff) << 16) |
                                   ((r.c[3] & 0xff) << 24);
                *reinterpret_cast<int*>(a.yq + (out0 + blk * QK) + part * 4) = packed;
                if (part == 0) a.yd[out0 / QK + blk] = f32_to_f16_bits(r.d32);
            }
        }
    }
}

}  // namespace qmm
