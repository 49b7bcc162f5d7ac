// qmm_chain.cuh -- a chain of dependent batch-1 GEMVs (one decode step's
// projections) in one persistent cooperative launch.
//
// Each op is the fused GEMV of the streaming kernel (Q8_0 or fp32 activation
// in, the fp32 one optionally RMSNorm-ed first; fp32 and/or Q8_0 out,
// optional residual add, optional SwiGLU of row pairs).  Op i reads what op
// i-1 (or any earlier op) wrote; op i starts on a CTA once every CTA has
// finished op i-1, signalled through a per-op completion counter in global
// memory.  The weights do not depend on the
// activations, so each CTA's producer warp streams the weight rows of all its
// ops back to back into the shared-memory ring -- across op boundaries, while
// the consumers are still waiting for the previous op -- and the only serial
// part left per op is: wait for the counter, stage the activation, finish the
// rows whose weights are already on chip, write and signal.
//
// Rows: op i's N rows are split in contiguous slices of rows_per_cta over
// the CTAs (whole 32-output blocks when the op writes Q8_0, so each CTA
// quantizes its own outputs).  Weights come in with 1D bulk copies, one per
// row of a 32-row group and K chunk (the slice of a row is contiguous).
//
// Method: as the streaming kernel (llama.cpp guide, kenji.blog/id, section
// 2.2; block format: TinyLLaMA C++ guide, kenji.blog, section 6.1; SwiGLU:
// TinyLLaMA guide section 4.4; RMSNorm: TinyLLaMA guide section 4.1).
#pragma once

#include "qmm_stream.cuh"

namespace qmm {

constexpr int CHAIN_MAX_OPS = 96;

struct ChainOp {
    const uint8_t* qs;
    const uint16_t* d;
    const float* xf;        // fp32 activation [K], or NULL: Q8_0 activation xq/xd
    const float* gamma;     // with xf: RMSNorm weight [K] (x is normalized first), or NULL
    const int8_t* xq;       // with xf: optional output of the staged Q8_0 activation (CTA 0 writes it)
    const uint16_t* xd;
    const float* residual;  // optional [N_out] (not with pairs)
    float* y;               // optional fp32 output [N_out]
    int8_t* yq;             // optional Q8_0 output [N_out], with yd [N_out / 32]
    uint16_t* yd;
    int N, K;               // K % 256 == 0
    int rows_per_cta;       // even; a multiple of 32 * (pairs ? 2 : 1) with a Q8_0 output
    int ckb;                // K blocks per unit: min(64, K / 32), a multiple of 8
    int pairs;              // SwiGLU of row pairs (2n, 2n+1) -> output n
    float eps;              // RMSNorm epsilon
};

struct ChainArgs {
    ChainOp ops[CHAIN_MAX_OPS];
    int n_ops;
    int nstages;
    int xtile_bytes;      // room for the largest op's staged activation (multiple of 128)
    unsigned* counters;   // [n_ops]: zero before the launch, left zero after a normal end
    int* err;
};

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Q8_0 activation row into the tile with coherent (L2) loads: the row was
// written by an earlier op of this launch on other SMs.
__device__ __forceinline__ void chain_stage_q8(const XTile& xt, const int8_t* xq, const uint16_t* xd, int B, int tid,
                                               int nthr) {
    for (int b = tid; b < B; b += nthr) {
        const int4 lo = __ldcg(reinterpret_cast<const int4*>(xq + (int64_t)b * QK));
        const int4 hi = __ldcg(reinterpret_cast<const int4*>(xq + (int64_t)b * QK + 16));
        const float s = f16_bits_to_f32(__ldcg(reinterpret_cast<const unsigned short*>(xd + b)));
        xt.lo[b] = lo;
        xt.hi[b] = hi;
        xt.sc[b] = make_int2(__float_as_int(s), block_qsum(lo, hi));
    }
}

// Rows of op `o` owned by CTA `c`: [r0, r1).
__device__ __forceinline__ void chain_rows(const ChainOp& o, int c, int& r0, int& r1) {
    const int64_t b = (int64_t)c * o.rows_per_cta;
    r0 = (int)min((int64_t)o.N, b);
    r1 = (int)min((int64_t)o.N, b + o.rows_per_cta);
}

__global__ void __launch_bounds__(STREAM_THREADS, 1) gemv_chain_kernel(const __grid_constant__ ChainArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + STREAM_MAX_STAGES;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + STREAM_MAX_STAGES);
    uint8_t* xbase = smem + STREAM_HDR;
    uint8_t* ring = xbase + a.xtile_bytes;
    float* ybuf = reinterpret_cast<float*>(ring + (size_t)a.nstages * STAGE_BYTES);  // this CTA's outputs of an op
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int S = a.nstages;
    const unsigned G = gridDim.x;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], SW);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == SW) {
        // ---------------- producer warp: every op's weight rows, back to back
        const uint64_t pol = l2_evict_first_policy();
        int u = 0, issued = 0;
        bool ok = true;
        for (int i = 0; i < a.n_ops && ok; ++i) {
            const ChainOp& o = a.ops[i];
            int r0, r1;
            chain_rows(o, blockIdx.x, r0, r1);
            const int B = o.K / QK, ckb = o.ckb;
            const int ngroups = (r1 - r0 + GROUP_ROWS - 1) / GROUP_ROWS, nkc = (B + ckb - 1) / ckb;
            for (int g = 0; g < ngroups && ok; ++g) {
                const int gr = r0 + g * GROUP_ROWS, nr = min(GROUP_ROWS, r1 - gr);
                for (int kc = 0; kc < nkc; ++kc, ++u) {
                    const int s = u % S;
                    if (u >= S) {
                        int w = 1;
                        if (lane == 0) w = mbar_wait(&empty[s], ((u / S) - 1) & 1, abort_flag) ? 1 : 0;
                        if (!__shfl_sync(FULL, w, 0)) {
                            ok = false;
                            break;
                        }
                    }
                    const int b0 = kc * ckb, nb = min(ckb, B - b0);  // nb % 8 == 0
                    uint8_t* st = ring + (size_t)s * STAGE_BYTES;
                    if (lane == 0) mbar_arrive_expect_tx(&full[s], (uint32_t)(nr * nb * 18));
                    __syncwarp();
                    if (lane < nr) {
                        const int64_t row = gr + lane;
                        bulk_g2s_hint(st + lane * ckb * 16, o.qs + row * (o.K / 2) + (int64_t)b0 * 16,
                                      (uint32_t)nb * 16, &full[s], pol);
                        bulk_g2s_hint(st + STAGE_Q + lane * ckb * 2, o.d + row * B + b0, (uint32_t)nb * 2, &full[s],
                                      pol);
                    }
                    issued = u + 1;
                }
            }
        }
        if (!ok && lane == 0) {
            atomicOr(a.err, ERR_TIMEOUT);
            *abort_flag = 1;
            for (int v = max(0, issued - S); v < issued; ++v) {  // let issued copies land
                const uint64_t t0 = global_ns();
                while (!mbar_try_wait(&full[v % S], (v / S) & 1) && global_ns() - t0 < WAIT_LIMIT_NS) {
                }
            }
        }
        return;
    }

    // ---------------- consumers
    constexpr int NTHR = SW * 32;
    const int rA = 2 * warp, rB = 2 * warp + 16;  // this warp's row pairs in a 32-row group
    bool failed = false;
    int u = 0;
    for (int i = 0; i < a.n_ops; ++i) {
        const ChainOp& o = a.ops[i];
        int r0, r1;
        chain_rows(o, blockIdx.x, r0, r1);
        const int B = o.K / QK, ckb = o.ckb;
        const int opr = o.pairs ? 2 : 1;
        const bool qout = o.yq != nullptr;
        if (r1 > r0) {
            // RMSNorm weights do not depend on earlier ops: load them before waiting
            RmsGamma gr;
            if (o.xf && o.gamma) gr = rms_gamma_load(o.gamma, o.K, tid, NTHR);
            if (i > 0 && tid == 0) {
                // wait until every CTA has finished op i-1 (bounded)
                if (!failed) {
                    const uint64_t t0 = global_ns();
                    while (ld_acquire_u32(&a.counters[i - 1]) < G) {
                        if (*abort_flag || global_ns() - t0 > WAIT_LIMIT_NS) {
                            atomicOr(a.err, ERR_TIMEOUT);
                            *abort_flag = 1;
                            break;
                        }
                        __nanosleep(64);
                    }
                }
            }
            asm volatile("bar.sync 1, %0;" ::"r"(NTHR) : "memory");
            failed = failed || *abort_flag;
            const XTile xt = xtile_at(xbase, 1, B);
            // Staged by every consumer thread even after a timeout: the staging
            // meets named barriers with all of them, and threads may see the
            // abort flag at different moments (later work is skipped instead).
            if (o.xf && o.gamma) {
                stage_f32_rmsnorm(xt, o.xf, o.gamma, gr, o.K, o.eps, const_cast<int8_t*>(o.xq),
                                  const_cast<uint16_t*>(o.xd), reinterpret_cast<float*>(smem + 256), tid, NTHR, 1);
            } else if (o.xf) {
                stage_f32<false>(xt, o.xf, o.K, const_cast<int8_t*>(o.xq), const_cast<uint16_t*>(o.xd), tid, NTHR);
            } else {
                chain_stage_q8(xt, o.xq, o.xd, B, tid, NTHR);
            }
            asm volatile("bar.sync 1, %0;" ::"r"(NTHR) : "memory");

            const int ngroups = (r1 - r0 + GROUP_ROWS - 1) / GROUP_ROWS, nkc = (B + ckb - 1) / ckb;
            for (int g = 0; g < ngroups; ++g) {
                const int gr = r0 + g * GROUP_ROWS, nr = min(GROUP_ROWS, r1 - gr);
                float2 acc[1][2];
                acc[0][0] = acc[0][1] = make_float2(0.f, 0.f);
                for (int kc = 0; kc < nkc; ++kc, ++u) {
                    const int s = u % S;
                    const bool ok = !failed && mbar_wait(&full[s], (u / S) & 1, abort_flag);
                    if (!ok && !failed) {
                        if (lane == 0) atomicOr(a.err, ERR_TIMEOUT);
                        *abort_flag = 1;
                        failed = true;
                    }
                    const int b0 = kc * ckb, nb = min(ckb, B - b0);
                    constexpr int H = CHUNK_KB / 32;
                    Quad4 qd[H];
                    const bool work = ok && rA < nr;
                    if (work) {
                        const uint8_t* stq = ring + (size_t)s * STAGE_BYTES + (rA * ckb + lane) * 16;
                        const uint16_t* std_ =
                            reinterpret_cast<const uint16_t*>(ring + (size_t)s * STAGE_BYTES + STAGE_Q) + rA * ckb +
                            lane;
#pragma unroll
                        for (int h = 0; h < H; ++h)
                            if (lane + 32 * h < nb) qd[h] = quad_load(stq + 512 * h, ckb * 16, std_ + 32 * h, ckb);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[s]);  // stage read: the producer may refill it
                    if (work) {
#pragma unroll
                        for (int h = 0; h < H; ++h)
                            if (lane + 32 * h < nb) quad_compute<1>(qd[h], xt, B, b0 + lane + 32 * h, acc);
                    }
                }
                // reduce the warp's four rows across lanes, write (rows past nr hold
                // stale bytes: computed, never written)
                const float v0 = warp_sum(acc[0][0].x), v1 = warp_sum(acc[0][0].y);
                const float v2 = warp_sum(acc[0][1].x), v3 = warp_sum(acc[0][1].y);
                if (lane == 0 && !failed) {
                    const float v[4] = {v0, v1, v2, v3};
#pragma unroll
                    for (int p = 0; p < 2; ++p) {
                        const int lr = p ? rB : rA;
                        if (lr >= nr) continue;
                        const int row = gr + lr;
                        if (o.pairs) {
                            const float hv = swiglu1(v[2 * p], v[2 * p + 1]);
                            const int on = row / 2;
                            if (o.y) o.y[on] = hv;
                            if (qout) ybuf[on - r0 / 2] = hv;
                        } else {
                            const bool has1 = lr + 1 < nr;
                            const float o0 = v[2 * p] + (o.residual ? __ldcg(o.residual + row) : 0.f);
                            const float o1 = has1 ? v[2 * p + 1] + (o.residual ? __ldcg(o.residual + row + 1) : 0.f)
                                                  : 0.f;
                            if (o.y) {
                                o.y[row] = o0;
                                if (has1) o.y[row + 1] = o1;
                            }
                            if (qout) {
                                ybuf[row - r0] = o0;
                                if (has1) ybuf[row + 1 - r0] = o1;
                            }
                        }
                    }
                }
            }
            if (qout) {
                // Q8_0 of this CTA's outputs (whole blocks of 32): 8 lanes per block
                asm volatile("bar.sync 1, %0;" ::"r"(NTHR) : "memory");
                const int nblk = (r1 - r0) / opr / QK;
                const int out0 = r0 / opr;
                for (int blk0 = warp * 4; blk0 < nblk; blk0 += SW * 4) {
                    const int blk = blk0 + (lane >> 3), part = lane & 7;
                    const bool valid = blk < nblk && !failed;
                    const float4 v = valid ? *reinterpret_cast<const float4*>(ybuf + blk * QK + part * 4)
                                           : make_float4(0.f, 0.f, 0.f, 0.f);
                    const Quad r = quad_codes(v, 127.0f, -127.0f);
                    if (valid) {
                        const int packed = (r.c[0] & 0xff) | ((r.c[1] & 0xff) << 8) | ((r.c[2] & 0xff) << 16) |
                                           ((r.c[3] & 0xff) << 24);
                        *reinterpret_cast<int*>(o.yq + (out0 + blk * QK) + part * 4) = packed;
                        if (part == 0) o.yd[out0 / QK + blk] = f32_to_f16_bits(r.d32);
                    }
                }
            }
        }
        // signal: this CTA is done with op i (its outputs written)
        asm volatile("bar.sync 1, %0;" ::"r"(NTHR) : "memory");
        if (tid == 0) {
            __threadfence();
            const unsigned prev = atomicAdd(&a.counters[i], 1u);
            if (i == a.n_ops - 1 && prev == G - 1) {
                // the last CTA to finish the last op: every CTA is past every
                // wait, so the counters can be put back to zero for the next launch
                for (int j = 0; j < a.n_ops; ++j) a.counters[j] = 0u;
                __threadfence();
            }
        }
    }
}

}  // namespace qmm
