// qmm_decode.cuh -- qmm_decode_chain (include/qmm.h): a decode step's chain
// of dependent batch-1 GEMVs (TinyLLaMA C++ guide, section 5.2 layer graph:
// RMSNorm, QKV, O + residual, RMSNorm, gate/up with SwiGLU, down + residual,
// final RMSNorm, lm_head) in one persistent launch, one CTA per SM.
//
// Why one launch: at batch 1 each projection reads a few MB of weights, about
// a microsecond of HBM time, but a launch boundary or a grid-wide barrier
// costs as much again before the next projection can start.  Here the two
// things a projection waits for are decoupled:
//  - weights do not depend on activations: each CTA's producer warp streams
//    the weight rows of all its ops back to back into one shared-memory ring
//    (a byte ring with per-unit barriers, so a unit takes exactly its bytes),
//    running ahead across op boundaries while the consumers wait;
//  - activations travel through flagged buffers in the workspace: every
//    output value is stored together with a 32-bit flag in one 64-bit word
//    (single-copy atomic), the flag naming the op and the call.  A consumer
//    thread spins on exactly the words it needs, so an op starts on a CTA the
//    moment its input has landed, without a counter, a fence or a barrier
//    across CTAs.
// Each CTA then stages the activation (RMSNorm and Q8_0 as the streaming
// kernel does, same arithmetic, same thread layout and order), takes its rows
// from the ring, and writes its outputs (residual add, SwiGLU of row pairs)
// as flagged words for the ops that read them.  Rows are split evenly over
// the CTAs in row pairs.  Per-row arithmetic, the Q8_0 rule and the RMSNorm
// reduction order are those of the streaming kernel, so the results are
// bit-identical to the same ops launched one by one.
//
// Method: llama.cpp guide (kenji.blog/id) section 2.2, y ~ Delta*Delta_x *
// sum q*q_x per block of 32; block format: TinyLLaMA C++ guide (kenji.blog)
// section 6.1; RMSNorm section 4.1, SwiGLU section 4.4.
//
// Included once, by qmm_api.cu (the translation unit of the kernels it uses).
#pragma once

#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>

#include "qmm.h"
#include "qmm_internal.h"
#include "qmm_stream.cuh"

namespace qmm {
namespace dec {

constexpr int MAX_OPS = QMM_DECODE_MAX_OPS;
constexpr int NSLOT = 16;           // ring units in flight at most
constexpr int NTHR = SW * 32;       // consumer threads
constexpr int HDR = 1024;           // barriers, flags, reduction scratch, producer bookkeeping
constexpr int OFF_ABORT = 256;      // int: this CTA gave up
constexpr int OFF_RED = 512;        // 33 floats: RMSNorm reduction
constexpr int OFF_RANGES = 768;     // int2[NSLOT]: byte range of each unit in flight (producer)
constexpr uint32_t FLAGS_PER_CALL = 128;  // > MAX_OPS: flag = epoch * 128 + op + 1

struct Op {
    const uint8_t* qs;
    const uint16_t* d;
    const float* x;         // plain fp32 input (src < 0), else null
    const uint64_t* fsrc;   // flagged input (src >= 0), else null
    const float* xres;      // plain fp32 residual, or null
    const uint64_t* fres;   // flagged residual, or null
    uint64_t* fout;         // this op's flagged output (a later op reads it), or null
    const float* gamma;     // RMSNorm weight of the input, or null
    float* y;               // plain fp32 copy of the output, or null
    int8_t* xq;             // the staged Q8_0 activation (CTA 0 writes it), or null
    uint16_t* xd;
    float eps;
    int N, K;
    int src, res;           // op whose output is the input / residual (-1: none or plain)
    int ckb;                // K blocks per ring unit: min(64, K / 32)
    int pairs;              // SwiGLU of row pairs (2n, 2n + 1) -> output n
};

struct Args {
    Op ops[MAX_OPS];
    int n_ops;
    int ring_bytes;         // multiple of 128
    int xtile_bytes;        // multiple of 128
    unsigned* ctl;          // workspace words: [0] call epoch, [1] CTAs done, [2] abort
    int* err;
    uint64_t wait_ns;
};

// ---------------------------------------------------------------- flagged words
__device__ __forceinline__ uint64_t fword(float v, uint32_t flag) {
    return ((uint64_t)flag << 32) | __float_as_uint(v);
}

__device__ __forceinline__ void fstore1(uint64_t* p, float v, uint32_t flag) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(fword(v, flag)) : "memory");
}

__device__ __forceinline__ void fstore2(uint64_t* p, float v0, float v1, uint32_t flag) {  // p 16-byte aligned
    asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(fword(v0, flag)), "l"(fword(v1, flag))
                 : "memory");
}

__device__ __forceinline__ ulonglong2 fload2(const uint64_t* p) {  // p 16-byte aligned
    ulonglong2 r;
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(r.x), "=l"(r.y) : "l"(p) : "memory");
    return r;
}

__device__ __forceinline__ bool fok(ulonglong2 r, uint32_t flag) {
    return (uint32_t)(r.x >> 32) == flag && (uint32_t)(r.y >> 32) == flag;
}

__device__ __forceinline__ float2 fval(ulonglong2 r) {
    return make_float2(__uint_as_float((uint32_t)r.x), __uint_as_float((uint32_t)r.y));
}

// Bounded spin of one thread on flagged words: gives up after the wait
// limit, or once this CTA or any other has given up.
struct Spin {
    uint64_t t0;
    int n;
    __device__ __forceinline__ bool again(const Args& a, volatile int* abort_flag) {
        if (*abort_flag) return false;
        if (t0 == 0) t0 = global_ns();
        if ((++n & 15) == 0) {
            if (*reinterpret_cast<volatile unsigned*>(a.ctl + 2)) return false;
            if (global_ns() - t0 > a.wait_ns) return false;
        }
        return true;
    }
};

__device__ __forceinline__ void give_up(const Args& a, volatile int* abort_flag) {
    if (!*abort_flag) {
        *abort_flag = 1;
        atomicOr(a.err, ERR_TIMEOUT);
        atomicExch(a.ctl + 2, 1u);
    }
}

// ---------------------------------------------------------------- staging from flagged words
// RMSNorm + Q8_0 of a flagged row (K / 32 <= RMS_STEPS * NTHR / 4): the
// values each thread takes in stage_rmsnorm_regs, read once every flag
// matches; then the same register-level staging.
__device__ __forceinline__ void stage_flagged_rmsnorm(const XTile& xt, const uint64_t* src, uint32_t flag,
                                                      const RmsGamma& gr, int K, float eps, int8_t* xq_out,
                                                      uint16_t* xd_out, float* red, int tid, const Args& a,
                                                      volatile int* abort_flag) {
    const int B = K / QK;
    const int p = tid & 3;
    ulonglong2 r[RMS_STEPS][4];
    Spin sp = {0, 0};
    unsigned pending = 0;  // words still to read: bit 4i + j (only those are read again)
#pragma unroll
    for (int i = 0; i < RMS_STEPS; ++i)
        if (i * (NTHR >> 2) + (tid >> 2) < B) pending |= 0xfu << (4 * i);
    for (;;) {
#pragma unroll
        for (int i = 0; i < RMS_STEPS; ++i) {
            const uint64_t* w = src + (int64_t)(i * (NTHR >> 2) + (tid >> 2)) * QK + p * 8;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (pending & (1u << (4 * i + j))) {
                    r[i][j] = fload2(w + 2 * j);
                    if (fok(r[i][j], flag)) pending &= ~(1u << (4 * i + j));
                }
        }
        if (!pending) break;
        if (!sp.again(a, abort_flag)) {
            give_up(a, abort_flag);
            break;
        }
    }
    float4 v[2 * RMS_STEPS];
#pragma unroll
    for (int i = 0; i < RMS_STEPS; ++i) {
        const int b = i * (NTHR >> 2) + (tid >> 2);
        if (b < B) {
            const float2 v0 = fval(r[i][0]), v1 = fval(r[i][1]), v2 = fval(r[i][2]), v3 = fval(r[i][3]);
            v[2 * i] = make_float4(v0.x, v0.y, v1.x, v1.y);
            v[2 * i + 1] = make_float4(v2.x, v2.y, v3.x, v3.y);
        } else {
            v[2 * i] = v[2 * i + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    // every thread reaches the staging's barriers, given up or not
    stage_rmsnorm_regs(xt, v, gr, K, eps, xq_out, xd_out, red, tid, NTHR, 1);
}

// Q8_0 of a flagged row: the rounds of stage_f32, each read once every flag
// of the round matches.
__device__ __forceinline__ void stage_flagged_f32(const XTile& xt, const uint64_t* src, uint32_t flag, int K,
                                                  int8_t* xq_out, uint16_t* xd_out, int tid, const Args& a,
                                                  volatile int* abort_flag) {
    const int B = K / QK;
    const int lane = tid & 31, warp = tid >> 5, nwarps = NTHR >> 5;
    const int part = lane & 7;
    for (int g0 = warp; g0 * 4 < B; g0 += nwarps * STAGE_STEPS) {
        ulonglong2 r[STAGE_STEPS][2];
        Spin sp = {0, 0};
        unsigned pending = 0;  // words still to read: bit 2i + j (only those are read again)
#pragma unroll
        for (int i = 0; i < STAGE_STEPS; ++i)
            if ((g0 + i * nwarps) * 4 + (lane >> 3) < B) pending |= 3u << (2 * i);
        for (;;) {
#pragma unroll
            for (int i = 0; i < STAGE_STEPS; ++i) {
                const uint64_t* w = src + (int64_t)((g0 + i * nwarps) * 4 + (lane >> 3)) * QK + part * 4;
#pragma unroll
                for (int j = 0; j < 2; ++j)
                    if (pending & (1u << (2 * i + j))) {
                        r[i][j] = fload2(w + 2 * j);
                        if (fok(r[i][j], flag)) pending &= ~(1u << (2 * i + j));
                    }
            }
            if (!pending) break;
            if (!sp.again(a, abort_flag)) {
                give_up(a, abort_flag);
                break;
            }
        }
        float4 v[STAGE_STEPS];
#pragma unroll
        for (int i = 0; i < STAGE_STEPS; ++i) {
            const int b = (g0 + i * nwarps) * 4 + (lane >> 3);
            if (b < B) {
                const float2 v0 = fval(r[i][0]), v1 = fval(r[i][1]);
                v[i] = make_float4(v0.x, v0.y, v1.x, v1.y);
            } else {
                v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        stage_f32_quantize(xt, v, g0, B, xq_out, xd_out, lane, nwarps);
    }
}

// ---------------------------------------------------------------- the ring
// Rows of op o owned by CTA c: row pairs split evenly, [r0, r1).
__device__ __forceinline__ void op_rows(const Op& o, int c, int G, int& r0, int& r1) {
    const int64_t P = o.N / 2;
    r0 = (int)(2 * (P * c / G));
    r1 = (int)(2 * (P * (c + 1) / G));
}

// Bytes of a unit of nr rows: nibbles (nr x ckb x 16) then scales (nr x ckb x 2).
__device__ __forceinline__ int unit_bytes(int nr, int ckb) { return (nr * ckb * 18 + 127) & ~127; }

// Place the next unit of `bytes` in the ring after `head` (wrapping to 0 when
// it does not fit before the end); both sides walk the same sequence.
__device__ __forceinline__ int ring_place(int& head, int bytes, int ring_bytes) {
    const int at = head + bytes <= ring_bytes ? head : 0;
    head = at + bytes;
    return at;
}

__global__ void __launch_bounds__(STREAM_THREADS, 1) decode_chain_kernel(const __grid_constant__ Args a) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + NSLOT;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_ABORT);
    float* red = reinterpret_cast<float*>(smem + OFF_RED);
    int2* ranges = reinterpret_cast<int2*>(smem + OFF_RANGES);
    uint8_t* xbase = smem + HDR;
    uint8_t* ring = xbase + a.xtile_bytes;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = gridDim.x, c = blockIdx.x;

    if (tid == 0) {
        for (int s = 0; s < NSLOT; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], SW);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    // the call's flags: written by the last CTA of the previous call, so stable here
    const uint32_t base = *reinterpret_cast<volatile unsigned*>(a.ctl) * FLAGS_PER_CALL + 1u;

    if (warp == SW) {
        // ---------------- producer warp: the weight rows of every op, back to back
        const uint64_t pol = l2_evict_first_policy();
        int u = 0, tail = 0, head = 0;
        bool ok = true;
        for (int i = 0; i < a.n_ops && ok; ++i) {
            const Op& o = a.ops[i];
            int r0, r1;
            op_rows(o, c, G, r0, r1);
            const int B = o.K / QK, ckb = o.ckb, nkc = (B + ckb - 1) / ckb;
            for (int gr = r0; gr < r1 && ok; gr += GROUP_ROWS) {
                const int nr = min(GROUP_ROWS, r1 - gr);
                for (int kc = 0; kc < nkc; ++kc, ++u) {
                    const int bytes = unit_bytes(nr, ckb);
                    const int at = ring_place(head, bytes, a.ring_bytes);
                    if (lane == 0) {
                        // a free slot, and none of the unit's bytes under a unit
                        // still in flight: units leave the ring in order, so wait
                        // for the oldest until no unit in flight overlaps
                        while (ok && tail < u) {
                            bool clash = u - tail >= NSLOT;
                            for (int v = tail; v < u && !clash; ++v) {
                                const int2 rg = ranges[v % NSLOT];
                                clash = rg.x < at + bytes && at < rg.y;
                            }
                            if (!clash) break;
                            ok = mbar_wait(&empty[tail % NSLOT], (tail / NSLOT) & 1, abort_flag, a.wait_ns);
                            if (ok) ++tail;
                        }
                        ranges[u % NSLOT] = make_int2(at, at + bytes);
                    }
                    ok = __shfl_sync(FULL, ok ? 1 : 0, 0) != 0;
                    if (!ok) break;
                    const int b0 = kc * ckb, nb = min(ckb, B - b0);
                    uint8_t* st = ring + at;
                    const int s = u % NSLOT;
                    if (lane == 0) mbar_arrive_expect_tx(&full[s], (uint32_t)(nr * nb * 18));
                    __syncwarp();
                    if (lane < nr) {
                        const int64_t row = gr + lane;
                        bulk_g2s_hint(st + lane * ckb * 16, o.qs + row * (o.K / 2) + (int64_t)b0 * 16,
                                      (uint32_t)nb * 16, &full[s], pol);
                        bulk_g2s_hint(st + nr * ckb * 16 + lane * ckb * 2, o.d + row * B + b0, (uint32_t)nb * 2,
                                      &full[s], pol);
                    }
                }
            }
        }
        if (!ok && lane == 0) {
            give_up(a, abort_flag);
            // let the copies in flight land before the CTA can end
            for (int v = max(tail, u - NSLOT); v < u; ++v) {
                const uint64_t t0 = global_ns();
                while (!mbar_try_wait(&full[v % NSLOT], (v / NSLOT) & 1) && global_ns() - t0 < a.wait_ns) {
                }
            }
        }
        return;
    }

    // ---------------- consumers (8 warps)
    const int rA = 2 * warp, rB = 2 * warp + 16;  // this warp's row pairs in a 32-row group
    int u = 0, head = 0;
    for (int i = 0; i < a.n_ops; ++i) {
        const Op& o = a.ops[i];
        const int B = o.K / QK, ckb = o.ckb, nkc = (B + ckb - 1) / ckb;
        const uint32_t my_flag = base + (uint32_t)i;
        // RMSNorm weights do not depend on earlier ops: load them before waiting
        RmsGamma gr;
        if (o.gamma) gr = rms_gamma_load(o.gamma, o.K, tid, NTHR);
        const XTile xt = xtile_at(xbase, 1, B);
        asm volatile("bar.sync 1, %0;" ::"r"(NTHR) : "memory");  // the previous op is done with the tile
        // Staged by every consumer thread even after a give-up: the staging
        // meets named barriers with all of them (later work is skipped).
        if (o.fsrc) {
            const uint32_t f = base + (uint32_t)o.src;
            if (o.gamma)
                stage_flagged_rmsnorm(xt, o.fsrc, f, gr, o.K, o.eps, o.xq, o.xd, red, tid, a, abort_flag);
            else
                stage_flagged_f32(xt, o.fsrc, f, o.K, o.xq, o.xd, tid, a, abort_flag);
        } else if (o.gamma) {
            stage_f32_rmsnorm(xt, o.x, o.gamma, gr, o.K, o.eps, o.xq, o.xd, red, tid, NTHR, 1);
        } else {
            stage_f32<false>(xt, o.x, o.K, o.xq, o.xd, tid, NTHR);
        }
        asm volatile("bar.sync 1, %0;" ::"r"(NTHR) : "memory");
        bool failed = *abort_flag != 0;

        int r0, r1;
        op_rows(o, c, G, r0, r1);
        for (int gr0 = r0; gr0 < r1; gr0 += GROUP_ROWS) {
            const int nr = min(GROUP_ROWS, r1 - gr0);  // even
            float2 acc[1][2];
            acc[0][0] = acc[0][1] = make_float2(0.f, 0.f);
            for (int kc = 0; kc < nkc; ++kc, ++u) {
                const int at = ring_place(head, unit_bytes(nr, ckb), a.ring_bytes);
                const int s = u % NSLOT;
                bool ok = !failed && mbar_wait(&full[s], (u / NSLOT) & 1, abort_flag, a.wait_ns);
                ok = __all_sync(FULL, ok);
                if (!ok && !failed) {
                    if (lane == 0) give_up(a, abort_flag);
                    failed = true;
                }
                const int b0 = kc * ckb, nb = min(ckb, B - b0);
                constexpr int H = CHUNK_KB / 32;
                Quad4 qd[H];
                const bool work = ok && rA < nr;
                if (work) {
                    const uint8_t* stq = ring + at + (rA * ckb + lane) * 16;
                    const uint16_t* std_ = reinterpret_cast<const uint16_t*>(ring + at + nr * ckb * 16) + rA * ckb + lane;
#pragma unroll
                    for (int h = 0; h < H; ++h)
                        if (lane + 32 * h < nb) qd[h] = quad_load(stq + 512 * h, ckb * 16, std_ + 32 * h, ckb, rB < nr);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);  // unit read: the producer may reuse its bytes
                if (work) {
#pragma unroll
                    for (int h = 0; h < H; ++h)
                        if (lane + 32 * h < nb) quad_compute<1>(qd[h], xt, B, b0 + lane + 32 * h, acc);
                }
            }
            // reduce the warp's four rows across lanes, write
            const float v0 = warp_sum(acc[0][0].x), v1 = warp_sum(acc[0][0].y);
            const float v2 = warp_sum(acc[0][1].x), v3 = warp_sum(acc[0][1].y);
            if (lane == 0 && !failed) {
                const float v[4] = {v0, v1, v2, v3};
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    const int lr = p ? rB : rA;
                    if (lr >= nr) continue;
                    const int row = gr0 + lr;
                    if (o.pairs) {
                        const float hv = swiglu1(v[2 * p], v[2 * p + 1]);
                        if (o.fout) fstore1(o.fout + row / 2, hv, my_flag);
                        if (o.y) o.y[row / 2] = hv;
                    } else {
                        float2 rv = make_float2(0.f, 0.f);
                        if (o.fres) {
                            // read before by this CTA's staging of an earlier op: its flags match
                            const uint32_t f = base + (uint32_t)o.res;
                            Spin sp = {0, 0};
                            ulonglong2 w = fload2(o.fres + row);
                            while (!fok(w, f)) {
                                if (!sp.again(a, abort_flag)) {
                                    give_up(a, abort_flag);
                                    break;
                                }
                                w = fload2(o.fres + row);
                            }
                            rv = fval(w);
                        } else if (o.xres) {
                            rv = make_float2(__ldcg(o.xres + row), __ldcg(o.xres + row + 1));
                        }
                        const float o0 = v[2 * p] + rv.x, o1 = v[2 * p + 1] + rv.y;
                        if (o.fout) fstore2(o.fout + row, o0, o1, my_flag);
                        if (o.y) {
                            o.y[row] = o0;
                            o.y[row + 1] = o1;
                        }
                    }
                }
            }
        }
    }
    // the call is over for this CTA; the last CTA to finish advances the
    // epoch (every CTA read it at its start) and clears the counters
    asm volatile("bar.sync 1, %0;" ::"r"(NTHR) : "memory");
    if (tid == 0) {
        __threadfence();
        const unsigned prev = atomicAdd(a.ctl + 1, 1u);
        if (prev == (unsigned)G - 1) {
            a.ctl[1] = 0u;
            a.ctl[2] = 0u;
            a.ctl[0] = a.ctl[0] + 1u;
            __threadfence();
        }
    }
}

}  // namespace dec
}  // namespace qmm

namespace {

using namespace qmm;

std::atomic<unsigned long long> g_decode_wait_ns{WAIT_LIMIT_NS};

inline bool al(const void* p, uintptr_t n) { return reinterpret_cast<uintptr_t>(p) % n == 0; }

int64_t n_out(const qmm_chain_op& o) { return (o.flags & QMM_Y_SWIGLU_PAIRS) ? o.N / 2 : o.N; }

// Validates the chain and marks which ops' outputs later ops read.
qmm_status validate_chain(const qmm_chain_op* ops, int32_t n_ops, bool* read_later) {
    if (!ops || n_ops < 1 || n_ops > QMM_DECODE_MAX_OPS) return QMM_ERR_ARG;
    for (int i = 0; i < n_ops; ++i) read_later[i] = false;
    for (int i = 0; i < n_ops; ++i) {
        const qmm_chain_op& o = ops[i];
        if (o.flags & ~QMM_Y_SWIGLU_PAIRS) return QMM_ERR_ARG;
        if (!o.w_qs || !o.w_d) return QMM_ERR_ARG;
        if (o.N < 2 || o.N % 2 || o.N >= ((int64_t)1 << 31) || o.K < 256 || o.K % 256 || o.K > QMM_DECODE_MAX_K)
            return QMM_ERR_SHAPE;
        const bool pairs = o.flags & QMM_Y_SWIGLU_PAIRS;
        if (o.src < -1 || o.src >= i || o.residual < -2 || o.residual >= i) return QMM_ERR_ARG;
        if ((o.src == -1 || o.residual == -2) && !o.x) return QMM_ERR_ARG;
        if (o.src >= 0 && n_out(ops[o.src]) < o.K) return QMM_ERR_SHAPE;
        if (o.residual >= 0 && n_out(ops[o.residual]) < o.N) return QMM_ERR_SHAPE;
        if (pairs && o.residual != -1) return QMM_ERR_ARG;
        if (o.norm_w && !(o.norm_eps >= 0.0f)) return QMM_ERR_ARG;
        if (o.norm_w && o.K > 4096) return QMM_ERR_SHAPE;  // the one-pass RMSNorm staging
        if ((o.xq == nullptr) != (o.xd == nullptr)) return QMM_ERR_ARG;
        if (!al(o.w_qs, 16) || !al(o.w_d, 16) || (o.x && !al(o.x, 16)) || (o.norm_w && !al(o.norm_w, 16)) ||
            (o.y && !al(o.y, 4)) || (o.xq && !al(o.xq, 16)) || (o.xd && !al(o.xd, 2)))
            return QMM_ERR_ALIGN;
        if (o.src >= 0) read_later[o.src] = true;
        if (o.residual >= 0) read_later[o.residual] = true;
    }
    return QMM_OK;
}

constexpr size_t CTL_BYTES = 256;

size_t flagged_bytes(int64_t n) { return (size_t)(n * 8 + 15) / 16 * 16; }

}  // namespace

extern "C" {

qmm_status qmm_decode_chain_workspace_size(const qmm_chain_op* ops, int32_t n_ops, size_t* bytes) {
    if (!bytes) return QMM_ERR_ARG;
    bool read_later[QMM_DECODE_MAX_OPS];
    const qmm_status v = validate_chain(ops, n_ops, read_later);
    if (v != QMM_OK) return v;
    size_t total = CTL_BYTES;
    for (int i = 0; i < n_ops; ++i)
        if (read_later[i]) total += flagged_bytes(n_out(ops[i]));
    *bytes = total;
    return QMM_OK;
}

qmm_status qmm_decode_chain(const qmm_chain_op* ops, int32_t n_ops, void* workspace, size_t workspace_bytes,
                            void* stream) {
    static_assert(QMM_DECODE_MAX_OPS <= (int)dec::FLAGS_PER_CALL - 1, "flags per call");
    bool read_later[QMM_DECODE_MAX_OPS];
    qmm_status v = validate_chain(ops, n_ops, read_later);
    if (v != QMM_OK) return v;
    size_t need = CTL_BYTES;
    for (int i = 0; i < n_ops; ++i)
        if (read_later[i]) need += flagged_bytes(n_out(ops[i]));
    if (!workspace || workspace_bytes < need) return QMM_ERR_WORKSPACE;
    if (!al(workspace, 16)) return QMM_ERR_ALIGN;
    int sms = 0, optin = 0;
    if (!device_facts(&sms, &optin)) return QMM_ERR_DEVICE;

    dec::Args a = {};
    a.n_ops = n_ops;
    uint8_t* wsb = static_cast<uint8_t*>(workspace);
    uint64_t* fbuf[QMM_DECODE_MAX_OPS] = {};
    size_t off = CTL_BYTES;
    int64_t maxB = 0;
    for (int i = 0; i < n_ops; ++i) {
        if (read_later[i]) {
            fbuf[i] = reinterpret_cast<uint64_t*>(wsb + off);
            off += flagged_bytes(n_out(ops[i]));
        }
        maxB = std::max<int64_t>(maxB, ops[i].K / QK);
    }
    for (int i = 0; i < n_ops; ++i) {
        const qmm_chain_op& o = ops[i];
        dec::Op& d = a.ops[i];
        d.qs = o.w_qs;
        d.d = o.w_d;
        d.N = (int)o.N;
        d.K = (int)o.K;
        d.src = o.src;
        d.res = o.residual;
        d.x = o.src == -1 ? o.x : nullptr;
        d.fsrc = o.src >= 0 ? fbuf[o.src] : nullptr;
        d.xres = o.residual == -2 ? o.x : nullptr;
        d.fres = o.residual >= 0 ? fbuf[o.residual] : nullptr;
        d.fout = fbuf[i];
        d.gamma = o.norm_w;
        d.eps = o.norm_eps;
        d.y = o.y;
        d.xq = o.xq;
        d.xd = o.xd;
        d.ckb = (int)std::min<int64_t>(CHUNK_KB, o.K / QK);
        d.pairs = (o.flags & QMM_Y_SWIGLU_PAIRS) ? 1 : 0;
    }
    a.xtile_bytes = (int)((maxB * xtile_bytes_per_block() + 127) / 128 * 128);
    a.ring_bytes = (optin - dec::HDR - a.xtile_bytes) / 128 * 128;
    if (a.ring_bytes < GROUP_ROWS * CHUNK_KB * 18) return QMM_ERR_SHAPE;  // one full unit must fit
    a.ctl = static_cast<unsigned*>(workspace);
    a.err = device_error_word();
    a.wait_ns = g_decode_wait_ns.load();
    const int smem = dec::HDR + a.xtile_bytes + a.ring_bytes;
    // opt the kernel into the full shared memory once per device (later calls
    // are a lookup, safe during stream capture)
    static std::atomic<int> attr_done[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return QMM_ERR_DEVICE;
    }
    if (!attr_done[dev].load()) {
        if (cudaFuncSetAttribute(dec::decode_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, optin) !=
            cudaSuccess) {
            cudaGetLastError();
            return QMM_ERR_SHAPE;
        }
        attr_done[dev].store(1);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)sms);
    cfg.blockDim = dim3(STREAM_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // every CTA resident: they wait on one another's outputs
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, dec::decode_chain_kernel, a);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return QMM_ERR_CUDA;
    }
    return cudaGetLastError() == cudaSuccess ? QMM_OK : QMM_ERR_CUDA;
}

qmm_status qmm_debug_decode_wait(uint64_t limit_ns, uint64_t* previous_limit_ns) {
    if (limit_ns < 1000ull || limit_ns > 10000000000ull) return QMM_ERR_ARG;
    const unsigned long long old = g_decode_wait_ns.exchange(limit_ns);
    if (previous_limit_ns) *previous_limit_ns = old;
    return QMM_OK;
}

}  // extern "C"
