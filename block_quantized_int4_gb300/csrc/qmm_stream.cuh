// qmm_stream.cuh -- streaming GEMV / small-batch GEMM for Q4_0 x Q8_0.
//
// Each CTA owns a contiguous range of weight rows.  One producer warp moves
// the range's nibble and scale bytes HBM -> shared memory with bulk copies
// (the copy engine, no registers) into a ring of stages; eight consumer
// warps quantize / stage the activation, then apply every row of a stage to
// it with dp4a, two rows per warp at a time, and release the stage.
//
// Decode chains: the producer starts copying before the kernel waits on the
// preceding grid (griddepcontrol.wait), so with programmatic dependent
// launch a kernel's weight stream overlaps the kernel before it; only the
// activation read waits.  Weights never depend on earlier kernels.
//
// Method: llama.cpp guide (kenji.blog/id) section 2.2, y ~ Delta*Delta_x *
// sum q*q_x per block of 32; block format: TinyLLaMA C++ guide (kenji.blog)
// section 6.1; SwiGLU of the gate/up pair: TinyLLaMA guide section 4.4.
#pragma once

#include "qmm_kernels.cuh"

namespace qmm {

enum YMode { Y_PLAIN = 0, Y_SWIGLU_PAIRS = 1 };

constexpr int STREAM_CONSUMER_WARPS = 8;
constexpr int STREAM_THREADS = (STREAM_CONSUMER_WARPS + 1) * 32;
constexpr int STREAM_HDR = 256;  // barriers + flags at the start of shared memory
constexpr int STREAM_MAX_STAGES = 15;

struct StreamArgs {
    const uint8_t* qs;   // [N][K/2]
    const uint16_t* d;   // [N][B]
    int64_t N, K, M;
    const int8_t* xq;    // X_Q8: [M][K]
    const uint16_t* xd;  // X_Q8: [M][B]
    const float* xf;     // X_F32 / X_SWIGLU: [K] (or [2K])
    const float* residual;  // optional [N] (Y_PLAIN, M == 1)
    int8_t* xq_out;
    uint16_t* xd_out;
    float* y;
    int64_t ldy;
    int rows_per_cta;    // even
    int stage_rows;      // even
    int nstages;
    int stage_bytes;     // multiple of 128
    int xtile_bytes;     // multiple of 128
    int* err;
};

// Apply two weight rows (in shared memory) to MT staged activations.
template <int MT>
__device__ __forceinline__ void pair_accumulate(const XTile& xt, int B, const uint8_t* q0, const uint8_t* q1,
                                                const uint16_t* d0, const uint16_t* d1, bool has1, int lane,
                                                float (&a0)[MT], float (&a1)[MT]) {
    for (int b = lane; b < B; b += 32) {
        const uint4 w0 = lds128(q0 + b * 16);
        const uint4 w1 = has1 ? lds128(q1 + b * 16) : make_uint4(0, 0, 0, 0);
        const float s0 = f16_bits_to_f32(d0[b]);
        const float s1 = has1 ? f16_bits_to_f32(d1[b]) : 0.f;
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            const int i = t * B + b;
            const int4 lo = xt.lo[i], hi = xt.hi[i];
            const float xs = xt.s[i];
            const int c8 = 8 * xt.sum[i];
            const int dot0 = block_dot_u(w0, lo, hi) - c8;
            const int dot1 = block_dot_u(w1, lo, hi) - c8;
            a0[t] = fmaf(s0 * xs, (float)dot0, a0[t]);
            a1[t] = fmaf(s1 * xs, (float)dot1, a1[t]);
        }
    }
}

template <int MT, int XMODE, int YMODE>
__global__ void __launch_bounds__(STREAM_THREADS) stream_rows_kernel(StreamArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + STREAM_MAX_STAGES;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + STREAM_MAX_STAGES);
    const int B = (int)(a.K / QK);
    const XTile xt = xtile_at(smem + STREAM_HDR, MT, B);
    uint8_t* ring = smem + STREAM_HDR + a.xtile_bytes;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    const int64_t row_begin = (int64_t)blockIdx.x * a.rows_per_cta;
    const int64_t row_end = min(a.N, row_begin + a.rows_per_cta);
    const int nrows = (int)(row_end - row_begin);
    const int nchunks = (nrows + a.stage_rows - 1) / a.stage_rows;
    const int S = a.nstages;
    const int64_t qrow = a.K / 2;           // nibble bytes per row
    const int64_t drow = (int64_t)B * 2;    // scale bytes per row
    const int dpart = a.stage_rows * (int)qrow;  // offset of the scale part in a stage

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], STREAM_CONSUMER_WARPS);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == STREAM_CONSUMER_WARPS) {
        // ---------------- producer: weights only, no dependence on earlier grids
        if (lane == 0) {
            int issued = 0;
            bool ok = true;
            for (int c = 0; c < nchunks; ++c) {
                const int s = c % S;
                if (c >= S && !mbar_wait(&empty[s], ((c / S) - 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                const int64_t r0 = row_begin + (int64_t)c * a.stage_rows;
                const int nr = (int)min((int64_t)a.stage_rows, row_end - r0);
                const uint32_t bq = (uint32_t)(nr * qrow), bd = (uint32_t)(nr * drow);
                uint8_t* st = ring + (size_t)s * a.stage_bytes;
                mbar_arrive_expect_tx(&full[s], bq + bd);
                bulk_g2s(st, a.qs + r0 * qrow, bq, &full[s]);
                bulk_g2s(st + dpart, a.d + r0 * B, bd, &full[s]);
                issued = c + 1;
            }
            if (!ok) {
                atomicOr(a.err, ERR_TIMEOUT);
                *abort_flag = 1;
                // let the copies already issued land before the CTA can exit
                for (int c = max(0, issued - S); c < issued; ++c) {
                    const int s = c % S;
                    const uint64_t t0 = global_ns();
                    while (!mbar_try_wait(&full[s], (c / S) & 1) && global_ns() - t0 < WAIT_LIMIT_NS) {
                    }
                }
            }
        }
        return;
    }

    // ---------------- consumers
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int nthr = STREAM_CONSUMER_WARPS * 32;
    const int64_t m0 = (int64_t)blockIdx.y * MT;
    int64_t xrow[MT];
#pragma unroll
    for (int t = 0; t < MT; ++t) xrow[t] = (m0 + t < a.M) ? m0 + t : -1;
    if (XMODE == X_Q8) stage_q8<MT>(xt, B, a.xq, a.xd, a.K, xrow, 0, B, tid, nthr);
    else stage_f32<XMODE == X_SWIGLU>(xt, a.xf, a.K, blockIdx.x == 0 ? a.xq_out : nullptr,
                                      blockIdx.x == 0 ? a.xd_out : nullptr, tid, nthr);
    asm volatile("bar.sync 1, %0;" ::"r"(nthr) : "memory");

    for (int c = 0; c < nchunks; ++c) {
        const int s = c % S;
        if (!mbar_wait(&full[s], (c / S) & 1, abort_flag)) {
            if (lane == 0) atomicOr(a.err, ERR_TIMEOUT);
            *abort_flag = 1;
            return;
        }
        const int64_t r0 = row_begin + (int64_t)c * a.stage_rows;
        const int nr = (int)min((int64_t)a.stage_rows, row_end - r0);
        const uint8_t* st = ring + (size_t)s * a.stage_bytes;
        const uint16_t* sd = reinterpret_cast<const uint16_t*>(st + dpart);
        for (int p = warp * 2; p < nr; p += 2 * STREAM_CONSUMER_WARPS) {
            const bool has1 = p + 1 < nr;
            float a0[MT], a1[MT];
#pragma unroll
            for (int t = 0; t < MT; ++t) a0[t] = a1[t] = 0.f;
            pair_accumulate<MT>(xt, B, st + p * qrow, st + (p + 1) * qrow, sd + p * B, sd + (p + 1) * B, has1,
                                lane, a0, a1);
            const int64_t row = r0 + p;
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                const float v0 = warp_sum(a0[t]);
                const float v1 = warp_sum(a1[t]);
                if (lane == 0 && xrow[t] >= 0) {
                    if (YMODE == Y_SWIGLU_PAIRS) {
                        a.y[xrow[t] * a.ldy + row / 2] = swiglu1(v0, v1);
                    } else {
                        float o0 = v0, o1 = v1;
                        if (a.residual) {
                            o0 += a.residual[row];
                            if (has1) o1 += a.residual[row + 1];
                        }
                        a.y[xrow[t] * a.ldy + row] = o0;
                        if (has1) a.y[xrow[t] * a.ldy + row + 1] = o1;
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
}

}  // namespace qmm
