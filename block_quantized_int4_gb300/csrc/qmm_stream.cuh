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

enum YMode { Y_PLAIN = 0, Y_SWIGLU_PAIRS = 1, Y_RUNTIME = 2 };
// XMODE = X_RUNTIME / YMODE = Y_RUNTIME: the input and output forms are read
// from StreamArgs (xmode, ymode, qout) at run time, so one compiled kernel
// serves every op of a decode chain (one code image for the instruction caches).
constexpr int X_RUNTIME = 3;

// Tiling constants (overridable at build time for tuning sweeps).
#ifndef QMM_STREAM_WARPS
#define QMM_STREAM_WARPS 8
#endif
#ifndef QMM_STREAM_CHUNK_KB
#define QMM_STREAM_CHUNK_KB 64
#endif
constexpr int SW = QMM_STREAM_WARPS;  // consumer warps (four rows each)
constexpr int STREAM_THREADS = (SW + 1) * 32;
constexpr int STREAM_HDR = 512;  // barriers, flags, reduction scratch (from byte 256)
constexpr int STREAM_MAX_STAGES = 8;
constexpr int GROUP_ROWS = 4 * SW;              // rows per group (4 per consumer warp)
constexpr int CHUNK_KB = QMM_STREAM_CHUNK_KB;   // K blocks per unit (CHUNK_KB / 32 per lane)
constexpr int STAGE_Q = GROUP_ROWS * CHUNK_KB * 16;  // 32 KB
constexpr int STAGE_D = GROUP_ROWS * CHUNK_KB * 2;   //  4 KB
constexpr int STAGE_BYTES = STAGE_Q + STAGE_D;

struct StreamArgs {
    int64_t N, K, M;
    const int8_t* xq;    // X_Q8: [M][K]
    const uint16_t* xd;  // X_Q8: [M][B]
    const float* xf;     // X_F32 / X_SWIGLU: [K] (or [2K])
    const float* residual;  // optional [N] (Y_PLAIN, M == 1)
    const float* gamma;     // X_F32: RMSNorm weight [K] (normalize x first), or NULL
    float eps;              // its epsilon
    int8_t* xq_out;
    uint16_t* xd_out;
    float* y;            // may be NULL when a Q8_0 output is requested
    int64_t ldy;
    int xmode, ymode, qout;  // the forms, read when the kernel is compiled with X_RUNTIME / Y_RUNTIME
    int8_t* yq;          // QOUT: Q8_0 codes of the output [N_out]
    uint16_t* yd;        // QOUT: Q8_0 scales [N_out / 32]
    int rows_per_cta;    // even
    int rb;              // rows per group = TMA box rows (even, <= 32)
    int ckb;             // K blocks per chunk = TMA box width in blocks (multiple of 8, <= 64)
    int nstages;
    int stage_bytes;     // ring stage: nibbles of rb x ckb blocks, then their scales (each part 128-aligned)
    int stage_q;         // offset of the scales in a stage
    int xtile_bytes;     // multiple of 128
    int* err;
    int ybuf_bytes;      // QOUT: shared-memory bytes of the CTA's outputs (after the ring)
    int rbuf;            // the CTA's residual values are read into shared memory (after ybuf) up front
    uint64_t wait_ns;    // limit of every bounded wait of the kernel (WAIT_LIMIT_NS normally)
    int withhold_last;   // test of the bounded waits: the producer never issues its last unit
};

// 2D tile copy of weight bytes, evicted first from L2 (l2_evict_first_policy).
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, "
        "{%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// A warp's four weight rows of one K block, read out of a ring stage into
// registers (so the stage can be handed back to the producer before the
// arithmetic): q points at this lane's block of the warp's first row, rows
// are qrs bytes apart; dd likewise, drs elements apart.
struct Quad4 {
    uint4 w[4];
    float d[4];
};

// Rows 16 and 17 further on are read only when the stage holds them (hi):
// a stage sized to a short row group ends before them.
__device__ __forceinline__ Quad4 quad_load(const uint8_t* q, int qrs, const uint16_t* dd, int drs, bool hi = true) {
    Quad4 r;
    r.w[0] = lds128(q);
    r.w[1] = lds128(q + qrs);
    r.d[0] = f16_bits_to_f32(dd[0]);
    r.d[1] = f16_bits_to_f32(dd[drs]);
    if (hi) {
        r.w[2] = lds128(q + 16 * qrs);
        r.w[3] = lds128(q + 17 * qrs);
        r.d[2] = f16_bits_to_f32(dd[16 * drs]);
        r.d[3] = f16_bits_to_f32(dd[17 * drs]);
    } else {
        r.w[2] = r.w[3] = make_uint4(0u, 0u, 0u, 0u);
        r.d[2] = r.d[3] = 0.0f;
    }
    return r;
}

// The four rows against MT staged activations: each activation block (two
// 16-byte halves and its scale/code-sum pair) is read once for all four
// rows.  acc[t][0] holds rows (r0, r1), acc[t][1] rows (r2, r3).  The block
// dot is taken as 16 * dot (block_dot16) and the scale as d_w * d_x / 16:
// the same fp32 product and sum as d_w * d_x * dot.
template <int MT>
__device__ __forceinline__ void quad_compute(const Quad4& q, const XTile& xt, int B, int ib, float2 (&acc)[MT][2],
                                             int mt = MT) {
#pragma unroll
    for (int t = 0; t < MT; ++t) {
        if (t >= mt) break;  // warp-uniform: tokens past mt are absent
        const int i = t * B + ib;
        const int4 xl = xt.lo[i], xh = xt.hi[i];
        const int2 sc = xt.sc[i];
        const float xs16 = __int_as_float(sc.x) * 0.0625f;
        const int c = -128 * sc.y;
        const float2 xs2 = make_float2(xs16, xs16);
        const int D0 = block_dot16(q.w[0], xl, xh, c), D1 = block_dot16(q.w[1], xl, xh, c);
        const int D2 = block_dot16(q.w[2], xl, xh, c), D3 = block_dot16(q.w[3], xl, xh, c);
        acc[t][0] = ffma2_scaled(make_float2(q.d[0], q.d[1]), xs2, make_float2((float)D0, (float)D1), acc[t][0]);
        acc[t][1] = ffma2_scaled(make_float2(q.d[2], q.d[3]), xs2, make_float2((float)D2, (float)D3), acc[t][1]);
    }
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
    const int xmode = XMODE == X_RUNTIME ? a.xmode : XMODE;
    const int ymode = YMODE == Y_RUNTIME ? a.ymode : YMODE;
    const bool qout = XMODE == X_RUNTIME ? a.qout != 0 : QOUT;
    const int B = (int)(a.K / QK);
    const XTile xt = xtile_at(smem + STREAM_HDR, MT, B);
    uint8_t* ring = smem + STREAM_HDR + a.xtile_bytes;
    float* ybuf = reinterpret_cast<float*>(ring + (size_t)a.nstages * a.stage_bytes);  // QOUT: this CTA's outputs
    float* rbuf = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ybuf) + a.ybuf_bytes);  // residual slice
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
            const uint64_t pol = l2_evict_first_policy();
            int issued = 0;
            bool ok = true;
            // withhold_last: the last unit is never issued (no expect_tx, no
            // copy), so its consumers' bounded waits run out -- the test of the
            // timeout path; every issued copy still lands before the CTA ends
            const int nissue = a.withhold_last ? nunits - 1 : nunits;
            for (int u = 0; u < nissue; ++u) {
                const int s = u % S;
                if (u >= S && !mbar_wait(&empty[s], ((u / S) - 1) & 1, abort_flag, a.wait_ns)) {
                    ok = false;
                    break;
                }
                const int g = u / nkc, kc = u - g * nkc;
                const int r0 = (int)(row_begin + (int64_t)g * RB);
                uint8_t* st = ring + (size_t)s * a.stage_bytes;
                mbar_arrive_expect_tx(&full[s], unit_bytes);
                tma_load_2d(st, &map_q, kc * CKB * 4, r0, &full[s], pol);           // u32 columns
                tma_load_2d(st + a.stage_q, &map_d, kc * CKB, r0, &full[s], pol);     // fp16 columns
                issued = u + 1;
            }
            if (!ok) {
                atomicOr(a.err, ERR_TIMEOUT);
                *abort_flag = 1;
            }
            if (!ok || a.withhold_last) {
                for (int u = max(0, issued - S); u < issued; ++u) {  // let issued copies land
                    const uint64_t t0 = global_ns();
                    while (!mbar_try_wait(&full[u % S], (u / S) & 1) && global_ns() - t0 < a.wait_ns) {
                    }
                }
            }
        }
        return;
    }

    // ---------------- consumers
    constexpr int NTHR = SW * 32;
    // RMSNorm weights do not depend on the preceding kernel: load them first
    RmsGamma gr;
    if (xmode == X_F32 && a.gamma) gr = rms_gamma_load(a.gamma, a.K, tid, NTHR);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // the residual values of this CTA's rows are read now, their latency
    // overlapping the staging's, and kept in shared memory for the epilogue
    // (read there, they would add a memory round trip at the very end)
    const float rv = a.rbuf && tid < nrows ? __ldcg(a.residual + row_begin + tid) : 0.f;
    const int64_t m0 = (int64_t)blockIdx.y * MT;
    int64_t xrow[MT];
#pragma unroll
    for (int t = 0; t < MT; ++t) xrow[t] = (m0 + t < a.M) ? m0 + t : -1;
    if (xmode == X_Q8) stage_q8<MT>(xt, B, a.xq, a.xd, a.K, xrow, 0, B, tid, NTHR);
    else if (xmode == X_F32 && a.gamma)
        stage_f32_rmsnorm(xt, a.xf, a.gamma, gr, a.K, a.eps, a.xq_out, a.xd_out, reinterpret_cast<float*>(smem + 256),
                          tid, NTHR, 1);
    else if (xmode == X_SWIGLU)
        stage_f32<true>(xt, a.xf, a.K, a.xq_out, a.xd_out, tid, NTHR);
    else
        stage_f32<false>(xt, a.xf, a.K, a.xq_out, a.xd_out, tid, NTHR);
    if (a.rbuf) {
        if (tid < nrows) rbuf[tid] = rv;
        for (int i = tid + NTHR; i < nrows; i += NTHR) rbuf[i] = __ldcg(a.residual + row_begin + i);
    }
    asm volatile("bar.sync 1, %0;" ::"r"(NTHR) : "memory");

    // this warp's rows inside a group: pairs (2w, 2w+1) and (2w+16, 2w+17),
    // so a gate/up pair always sits in one warp
    const int rA = 2 * warp, rB = 2 * warp + 16;
    const bool hi_rows = rB < RB;  // the stage holds this warp's second row pair (RB is even)
    const int OPR = ymode == Y_SWIGLU_PAIRS ? 2 : 1;  // rows per output
    bool failed = false;
    for (int g = 0; g < ngroups; ++g) {
        const int64_t r0 = row_begin + (int64_t)g * RB;
        const int nr = (int)min((int64_t)RB, row_end - r0);
        float2 acc[MT][2];
#pragma unroll
        for (int t = 0; t < MT; ++t) acc[t][0] = acc[t][1] = make_float2(0.f, 0.f);
        for (int kc = 0; kc < nkc; ++kc) {
            const int u = g * nkc + kc, s = u % S;
            // On a timeout keep going without computing: every later wait returns
            // at once (abort flag), and the kernel ends with the error word set.
            const bool ok = !failed && mbar_wait(&full[s], (u / S) & 1, abort_flag, a.wait_ns);
            if (!ok && !failed) {
                if (lane == 0) atomicOr(a.err, ERR_TIMEOUT);
                *abort_flag = 1;
                failed = true;
            }
            const int b0 = kc * CKB, nb = min(CKB, B - b0);
            // rows past nr hold stale or zero-filled bytes: computed, never written
            constexpr int H = CHUNK_KB / 32;
            Quad4 qd[H];
            const bool work = ok && rA < nr;
            if (work) {
                const uint8_t* stq = ring + (size_t)s * a.stage_bytes + (rA * CKB + lane) * 16;
                const uint16_t* std_ = reinterpret_cast<const uint16_t*>(ring + (size_t)s * a.stage_bytes + a.stage_q) +
                                       rA * CKB + lane;
#pragma unroll
                for (int h = 0; h < H; ++h)
                    if (lane + 32 * h < nb) qd[h] = quad_load(stq + 512 * h, CKB * 16, std_ + 32 * h, CKB, hi_rows);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);  // stage read: the producer may refill it
            if (work) {
#pragma unroll
                for (int h = 0; h < H; ++h)
                    if (lane + 32 * h < nb) quad_compute<MT>(qd[h], xt, B, b0 + lane + 32 * h, acc);
            }
        }
        // reduce the warp's four rows across lanes, write
        float v[MT][4];
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            v[t][0] = warp_sum(acc[t][0].x);
            v[t][1] = warp_sum(acc[t][0].y);
            v[t][2] = warp_sum(acc[t][1].x);
            v[t][3] = warp_sum(acc[t][1].y);
        }
        if (lane == 0 && !failed) {
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                if (xrow[t] < 0) continue;
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    const int lr = p ? rB : rA;
                    if (lr >= nr) continue;
                    const int64_t row = r0 + lr;
                    if (ymode == Y_SWIGLU_PAIRS) {
                        const float h = swiglu1(v[t][2 * p], v[t][2 * p + 1]);
                        const int64_t o = row / 2;
                        if (a.y) a.y[xrow[t] * a.ldy + o] = h;
                        if (qout) ybuf[o - row_begin / 2] = h;
                    } else {
                        const bool has1 = lr + 1 < nr;
                        const float r0v = a.rbuf ? rbuf[row - row_begin] : a.residual ? a.residual[row] : 0.f;
                        const float r1v =
                            !has1 ? 0.f : a.rbuf ? rbuf[row + 1 - row_begin] : a.residual ? a.residual[row + 1] : 0.f;
                        const float o0 = v[t][2 * p] + r0v;
                        const float o1 = has1 ? v[t][2 * p + 1] + r1v : 0.f;
                        if (a.y) {
                            a.y[xrow[t] * a.ldy + row] = o0;
                            if (has1) a.y[xrow[t] * a.ldy + row + 1] = o1;
                        }
                        if (qout) {
                            ybuf[row - row_begin] = o0;
                            if (has1) ybuf[row + 1 - row_begin] = o1;
                        }
                    }
                }
            }
        }
    }
    if (qout) {
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

// ============================================================================
// MoE expert-grouped GEMV on the same streaming scheme.  The rows of all
// active experts (in the order of the device-built active list) form one row
// space; CTA c takes the slice [c*R/G, (c+1)*R/G) of it, so a CTA meets only
// a few expert boundaries and restages the routed activations only there.
// Weights of all E experts are one 2D tensor [E*N rows][K/2 bytes].  A row
// group is applied to MT of the expert's slots per pass; an expert with more
// routed slots is streamed once per MT slots.  With pairs, each expert's rows
// interleave its gate and up projections (row 2i gate, 2i + 1 up; a pair
// always sits in one warp) and the output is SwiGLU of each pair (TinyLLaMA
// guide section 4.4): the expert FFN's first half in one launch.
// ============================================================================
struct MoeStreamArgs {
    int64_t N, K;
    int E, k;
    int nslots;       // T * k
    int slots_smem;   // the slot list is copied into shared memory (nslots <= MOE_SMEM_SLOTS)
    const int8_t* xq;
    const uint16_t* xd;
    const float* xf;  // fp32 activation rows instead of xq/xd (Q8_0 formed while staging), or NULL
    int x_per_slot;
    float* y;   // [T*k][N], or [T*k][N/2] with pairs
    int pairs;  // rows 2i, 2i+1 of each expert are a (gate, up) pair: y = SwiGLU of the pair
    MoeWs ws;
    int rb, ckb, nstages, xtile_bytes;
    int* err;
    // Launch chaining (programmatic dependent launch):
    //  - late_trigger: let dependents start only after this grid's wait for
    //    its predecessor (the gate/up launch after the router, so that the
    //    grouping is complete before the down launch can start);
    //  - tables_ready: the grouping was complete before this grid could start
    //    (the down launch after such a gate/up launch): it is read, and the
    //    producer streams weights, before the wait; only the consumers, which
    //    read the activations, wait.
    int late_trigger, tables_ready;
};

// The unit sequence of one CTA, walked identically by producer and consumers:
// segments (the rows of one active expert inside the CTA's slice), then per
// segment its slot passes (MT slots each), then per pass the segment's row
// groups and K chunks.  So a pass stages its activations once for all the
// segment's rows.
constexpr int MOE_SMEM_SLOTS = 1024;

struct MoeCursor {
    // 32-bit positions: the host admits this kernel only when E * N < 2^31
    int gr, gr1;  // position in the row space, end of this CTA's slice
    int N;
    int n_active, total;  // routed experts; valid slots (end of the last span)
    // current segment: expert e, rows [r, r + nrows), slots [sbeg, send)
    int e, nrows, sbeg, send;
    int r;
    // active: expert of each active index; start: first slot of each active
    // index -- shared-memory copies of the grouping
    __device__ bool next_segment(const int* active, const int* start) {
        if (gr >= gr1) return false;
        const int ai = gr / N;
        r = gr - ai * N;
        nrows = min(N - r, gr1 - gr);
        e = active[ai];
        sbeg = start[ai];
        send = ai + 1 < n_active ? start[ai + 1] : total;
        gr += nrows;
        return true;
    }
};

template <int MT>
__global__ void __launch_bounds__(STREAM_THREADS, 2)
    moe_stream_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_d,
                      MoeStreamArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + STREAM_MAX_STAGES;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + STREAM_MAX_STAGES);
    const int B = (int)(a.K / QK);
    const XTile xt = xtile_at(smem + STREAM_HDR, MT, B);
    uint8_t* ring = smem + STREAM_HDR + a.xtile_bytes;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int S = a.nstages, CKB = a.ckb;
    const int nkc = (B + CKB - 1) / CKB;
    const uint32_t unit_bytes = (uint32_t)(a.rb * CKB * 18);

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], SW);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (!a.late_trigger) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // the grouping written by the kernel before (unless complete before this grid started)
    if (!a.tables_ready) asm volatile("griddepcontrol.wait;" ::: "memory");

    // The routing, read once into shared memory in one round of independent
    // loads (the walk below consults it for every row group): the active
    // experts and the start of each one's slots, for every possible active
    // index (those past n_active are not used), the count and the end, and
    // (when short enough) the slot list itself.  Read from L2 (.cg), so that
    // no line an earlier grid left in this SM's L1 is used.
    int* s_active = reinterpret_cast<int*>(ring + (size_t)S * STAGE_BYTES);
    int* s_start = s_active + a.E;
    int* s_slots = s_start + a.E;
    int* s_count = s_slots + (a.slots_smem ? a.nslots : 0);  // n_active, total
    for (int i = tid; i < a.E; i += blockDim.x) {
        s_active[i] = __ldcg(a.ws.active + i);
        s_start[i] = __ldcg(a.ws.cursor + i);
    }
    if (a.slots_smem)
        for (int i = tid; i < a.nslots; i += blockDim.x) s_slots[i] = __ldcg(a.ws.slots + i);
    if (tid == 0) {
        s_count[0] = __ldcg(a.ws.n_active);
        s_count[1] = __ldcg(a.ws.offsets + a.E);
    }
    __syncthreads();
    if (a.late_trigger) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int n_active = s_count[0];
    const int* slot_list = a.slots_smem ? s_slots : a.ws.slots;
    const int64_t total = (int64_t)n_active * a.N;
    MoeCursor cur;
    cur.n_active = n_active;
    cur.total = s_count[1];
    if (a.pairs) {  // slices of whole (gate, up) row pairs (N is even)
        const int64_t tp = total / 2;
        cur.gr = 2 * (int)(tp * blockIdx.x / gridDim.x);
        cur.gr1 = 2 * (int)(tp * (blockIdx.x + 1) / gridDim.x);
    } else {
        cur.gr = (int)(total * blockIdx.x / gridDim.x);
        cur.gr1 = (int)(total * (blockIdx.x + 1) / gridDim.x);
    }
    cur.N = (int)a.N;


    if (warp == SW) {
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();
            int u = 0, issued = 0;
            bool ok = true;
            while (ok && cur.next_segment(s_active, s_start)) {
                const int nsb = (cur.send - cur.sbeg + MT - 1) / MT;
                const int ngroups = (cur.nrows + a.rb - 1) / a.rb;
                for (int sb = 0; sb < nsb && ok; ++sb)
                    for (int g = 0; g < ngroups && ok; ++g) {
                        const int row = (int)((int64_t)cur.e * a.N + cur.r + (int64_t)g * a.rb);
                        for (int kc = 0; kc < nkc; ++kc, ++u) {
                            const int s = u % S;
                            if (u >= S && !mbar_wait(&empty[s], ((u / S) - 1) & 1, abort_flag)) {
                                ok = false;
                                break;
                            }
                            uint8_t* st = ring + (size_t)s * STAGE_BYTES;
                            mbar_arrive_expect_tx(&full[s], unit_bytes);
                            tma_load_2d(st, &map_q, kc * CKB * 4, row, &full[s], pol);
                            tma_load_2d(st + STAGE_Q, &map_d, kc * CKB, row, &full[s], pol);
                            issued = u + 1;
                        }
                    }
            }
            if (!ok) {
                atomicOr(a.err, ERR_TIMEOUT);
                *abort_flag = 1;
                for (int v = max(0, issued - S); v < issued; ++v) {
                    const uint64_t t0 = global_ns();
                    while (!mbar_try_wait(&full[v % S], (v / S) & 1) && global_ns() - t0 < WAIT_LIMIT_NS) {
                    }
                }
            }
        }
        return;
    }

    constexpr int NTHR = SW * 32;
    const int rA = 2 * warp, rB = 2 * warp + 16;
    int u = 0;
    bool failed = false;
    if (a.tables_ready) asm volatile("griddepcontrol.wait;" ::: "memory");  // the activations
    while (cur.next_segment(s_active, s_start)) {
        const int nslots = cur.send - cur.sbeg;
        const int nsb = (nslots + MT - 1) / MT;
        const int ngroups = (cur.nrows + a.rb - 1) / a.rb;
        for (int sb = 0; sb < nsb; ++sb) {
            const int mt = min(MT, nslots - sb * MT);  // slots in this pass
            int slot[MT];
            int64_t xrow[MT];
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                const int j = sb * MT + t;
                slot[t] = j < nslots ? slot_list[cur.sbeg + j] : -1;
                xrow[t] = slot[t] < 0 ? -1 : (a.x_per_slot ? slot[t] : slot[t] / a.k);
            }
            asm volatile("bar.sync 1, %0;" ::"r"(NTHR) : "memory");  // everyone is done with the old tile
            if (a.xf) {
                // Q8_0 of each fp32 row as qmm_quantize_q8_0 would form it
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    XTile r = xt;
                    r.lo += t * B;
                    r.hi += t * B;
                    r.sc += t * B;
                    if (xrow[t] >= 0) {
                        stage_f32<false>(r, a.xf + xrow[t] * a.K, a.K, nullptr, nullptr, tid, NTHR);
                    } else {
                        for (int b = tid; b < B; b += NTHR) {
                            r.lo[b] = r.hi[b] = make_int4(0, 0, 0, 0);
                            r.sc[b] = make_int2(0, 0);
                        }
                    }
                }
            } else {
                stage_q8<MT>(xt, B, a.xq, a.xd, a.K, xrow, 0, B, tid, NTHR);
            }
            asm volatile("bar.sync 1, %0;" ::"r"(NTHR) : "memory");
            for (int g = 0; g < ngroups; ++g) {
                const int64_t r0 = cur.r + (int64_t)g * a.rb;
                const int nr = (int)min((int64_t)a.rb, cur.r + cur.nrows - r0);
                float2 acc[MT][2];
#pragma unroll
                for (int t = 0; t < MT; ++t) acc[t][0] = acc[t][1] = make_float2(0.f, 0.f);
                for (int kc = 0; kc < nkc; ++kc, ++u) {
                    const int s = u % S;
                    const bool ok = !failed && mbar_wait(&full[s], (u / S) & 1, abort_flag);
                    if (!ok && !failed) {
                        if (lane == 0) atomicOr(a.err, ERR_TIMEOUT);
                        *abort_flag = 1;
                        failed = true;
                    }
                    const int b0 = kc * CKB, nb = min(CKB, B - b0);
                    constexpr int H = CHUNK_KB / 32;
                    const bool work = ok && rA < nr;
                    const uint8_t* stq = ring + (size_t)s * STAGE_BYTES + (rA * CKB + lane) * 16;
                    const uint16_t* std_ =
                        reinterpret_cast<const uint16_t*>(ring + (size_t)s * STAGE_BYTES + STAGE_Q) + rA * CKB + lane;
                    // one 32-block half of the chunk in registers at a time (the
                    // four-slot kernel would not fit two in its register budget);
                    // the stage goes back to the producer once its last half is read
#pragma unroll
                    for (int h = 0; h < H; ++h) {
                        const bool here = work && lane + 32 * h < nb;
                        Quad4 qd;
                        if (here) qd = quad_load(stq + 512 * h, CKB * 16, std_ + 32 * h, CKB);
                        if (h == H - 1) {
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&empty[s]);
                        }
                        if (here) quad_compute<MT>(qd, xt, B, b0 + lane + 32 * h, acc, mt);
                    }
                }
                float v[MT][4];
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    v[t][0] = warp_sum(acc[t][0].x);
                    v[t][1] = warp_sum(acc[t][0].y);
                    v[t][2] = warp_sum(acc[t][1].x);
                    v[t][3] = warp_sum(acc[t][1].y);
                }
                if (a.pairs && !failed) {
                    // rows (rA, rA + 1) and (rB, rB + 1) are (gate, up) pairs (r0,
                    // rA, rB and nr are even); every lane holds the sums, so lane
                    // 2t + p evaluates the SwiGLU of slot t's pair p
                    const int tl = lane >> 1, p = lane & 1;
                    float g = 0.f, uu = 0.f;
                    int sl = -1;
#pragma unroll
                    for (int t = 0; t < MT; ++t)
                        if (t == tl) {
                            g = p ? v[t][2] : v[t][0];
                            uu = p ? v[t][3] : v[t][1];
                            sl = slot[t];
                        }
                    const int lr = p ? rB : rA;
                    if (tl < MT && sl >= 0 && lr < nr)
                        a.y[(int64_t)sl * (a.N / 2) + (r0 + lr) / 2] = swiglu1(g, uu);
                } else if (!failed) {
                    // lane 4t + q writes slot t's row q of the warp (rA, rA + 1, rB, rB + 1)
                    const int tl = lane >> 2, q = lane & 3;
                    float o = 0.f;
                    int sl = -1;
#pragma unroll
                    for (int t = 0; t < MT; ++t)
                        if (t == tl) {
                            o = q == 0 ? v[t][0] : q == 1 ? v[t][1] : q == 2 ? v[t][2] : v[t][3];
                            sl = slot[t];
                        }
                    const int lr = (q < 2 ? rA : rB) + (q & 1);
                    if (tl < MT && sl >= 0 && lr < nr) a.y[(int64_t)sl * a.N + r0 + lr] = o;
                }
            }
        }
    }
}

}  // namespace qmm
