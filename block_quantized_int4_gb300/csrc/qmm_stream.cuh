// qmm_stream.cuh -- streaming GEMV / small-batch GEMM for Q4_0 x Q8_0.
//
// Each CTA owns a contiguous range of weight rows, taken 32 rows at a time
// (one row per lane) and 64 K blocks at a time (a "unit").  A producer warp
// moves each unit's nibble and scale bytes HBM -> shared memory with bulk
// copies (one per row segment, into padded rows so that the 32 lanes'
// 16-byte reads fall in distinct bank groups), through a ring of stages.
// Eight consumer warps each own one eighth of the unit's K blocks: lane l
// accumulates row l over its warp's blocks with dp4a against the staged
// activation (a warp-uniform broadcast read), then the eight partial sums of
// every row are added in a fixed order.  No per-row shuffle reduction.
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

#include "qmm_kernels.cuh"

namespace qmm {

enum YMode { Y_PLAIN = 0, Y_SWIGLU_PAIRS = 1 };

constexpr int SW = 8;                       // consumer warps
constexpr int STREAM_THREADS = (SW + 1) * 32;
constexpr int STREAM_HDR = 256;             // barriers + flags
constexpr int STREAM_MAX_STAGES = 8;
constexpr int UNIT_ROWS = 32;               // rows per unit (one per lane)
constexpr int UNIT_KB = 64;                 // K blocks per unit (8 per consumer warp)
constexpr int QSTR = UNIT_KB * 16 + 16;     // padded nibble row in a stage
constexpr int DSTR = UNIT_KB * 2 + 16;      // padded scale row in a stage
constexpr int STAGE_BYTES = UNIT_ROWS * (QSTR + DSTR);  // 37,888

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
    int nstages;
    int xtile_bytes;     // multiple of 128
    int* err;
};

template <int MT, int XMODE, int YMODE>
__global__ void __launch_bounds__(STREAM_THREADS) stream_rows_kernel(StreamArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + STREAM_MAX_STAGES;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + STREAM_MAX_STAGES);
    const int B = (int)(a.K / QK);
    const XTile xt = xtile_at(smem + STREAM_HDR, MT, B);
    uint8_t* ring = smem + STREAM_HDR + a.xtile_bytes;
    float* part = reinterpret_cast<float*>(ring + (size_t)a.nstages * STAGE_BYTES);  // [SW][32][MT]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    const int64_t row_begin = (int64_t)blockIdx.x * a.rows_per_cta;
    const int64_t row_end = min(a.N, row_begin + a.rows_per_cta);
    const int nrows = (int)max((int64_t)0, row_end - row_begin);
    const int ngroups = (nrows + UNIT_ROWS - 1) / UNIT_ROWS;
    const int nkc = (B + UNIT_KB - 1) / UNIT_KB;  // K chunks per group
    const int nunits = ngroups * nkc;
    const int S = a.nstages;
    const int64_t qrow = a.K / 2;

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
                const int64_t r0 = row_begin + (int64_t)g * UNIT_ROWS;
                const int nr = (int)min((int64_t)UNIT_ROWS, row_end - r0);
                const int b0 = kc * UNIT_KB, nb = min(UNIT_KB, B - b0);
                uint8_t* st = ring + (size_t)s * STAGE_BYTES;
                mbar_arrive_expect_tx(&full[s], (uint32_t)(nr * nb * 18));
                const uint8_t* qsrc = a.qs + r0 * qrow + b0 * 16;
                const uint16_t* dsrc = a.d + r0 * B + b0;
                for (int r = 0; r < nr; ++r) {
                    bulk_g2s(st + r * QSTR, qsrc + r * qrow, (uint32_t)(nb * 16), &full[s]);
                    bulk_g2s(st + UNIT_ROWS * QSTR + r * DSTR, dsrc + (int64_t)r * B, (uint32_t)(nb * 2), &full[s]);
                }
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

    constexpr int J = UNIT_KB / SW;  // blocks per warp per unit
    for (int g = 0; g < ngroups; ++g) {
        const int64_t r0 = row_begin + (int64_t)g * UNIT_ROWS;
        const int nr = (int)min((int64_t)UNIT_ROWS, row_end - r0);
        float acc[MT], acc2[MT];
#pragma unroll
        for (int t = 0; t < MT; ++t) acc[t] = acc2[t] = 0.f;
        for (int kc = 0; kc < nkc; ++kc) {
            const int u = g * nkc + kc, s = u % S;
            // On a timeout keep going without computing: every later wait returns
            // at once (abort flag) and all warps still meet at the named barriers.
            const bool ok = mbar_wait(&full[s], (u / S) & 1, abort_flag);
            if (!ok) {
                if (lane == 0) atomicOr(a.err, ERR_TIMEOUT);
                *abort_flag = 1;
            }
            const int b0 = kc * UNIT_KB, nb = min(UNIT_KB, B - b0);
            const int jb = warp * J;  // this warp's first block in the unit
            if (ok && lane < nr && jb < nb) {
                const uint8_t* st = ring + (size_t)s * STAGE_BYTES;
                const uint8_t* qr = st + lane * QSTR;
                // eight scales of this row, one 16-byte read
                const uint4 dv = lds128(st + UNIT_ROWS * QSTR + lane * DSTR + jb * 2);
                const unsigned short* dh = reinterpret_cast<const unsigned short*>(&dv);
#pragma unroll
                for (int j = 0; j < J; ++j) {
                    const int bl = jb + j;  // nb is a multiple of 8, so all J blocks are valid
                    const uint4 w = lds128(qr + bl * 16);
                    const float dw = f16_bits_to_f32(dh[j]);
#pragma unroll
                    for (int t = 0; t < MT; ++t) {
                        const int i = t * B + b0 + bl;
                        const int dot = block_dot_u(w, xt.lo[i], xt.hi[i]) - 8 * xt.sum[i];
                        if (j & 1) acc2[t] = fmaf(dw * xt.s[i], (float)dot, acc2[t]);
                        else acc[t] = fmaf(dw * xt.s[i], (float)dot, acc[t]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        // fixed-order reduction of the eight warps' partial sums
#pragma unroll
        for (int t = 0; t < MT; ++t) part[(warp * 32 + lane) * MT + t] = acc[t] + acc2[t];
        asm volatile("bar.sync 1, %0;" ::"r"(NTHR) : "memory");
        if (warp == 0) {
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                float v = 0.f;
#pragma unroll
                for (int w = 0; w < SW; ++w) v += part[(w * 32 + lane) * MT + t];
                const int64_t row = r0 + lane;
                if (YMODE == Y_SWIGLU_PAIRS) {
                    const float up = __shfl_down_sync(FULL, v, 1);
                    if ((lane & 1) == 0 && lane < nr && xrow[t] >= 0) a.y[xrow[t] * a.ldy + row / 2] = swiglu1(v, up);
                } else if (lane < nr && xrow[t] >= 0) {
                    if (a.residual) v += a.residual[row];
                    a.y[xrow[t] * a.ldy + row] = v;
                }
            }
        }
        asm volatile("bar.sync 1, %0;" ::"r"(NTHR) : "memory");
    }
}

}  // namespace qmm
