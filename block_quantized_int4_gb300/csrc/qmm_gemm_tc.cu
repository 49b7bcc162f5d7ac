// qmm_gemm_tc.cu -- batched Q4_0 x Q8_0 GEMM on the 5th-generation tensor
// cores (tcgen05.mma, accumulators in TMEM), for 16..64 tokens.
//
// Y[m][n] = sum_b d_w[n][b] * d_x[m][b] * dot_b(n, m): every 32-wide K block
// has its own scale pair (llama.cpp guide, kenji.blog/id, section 2.2), so the
// integer block dots cannot be accumulated across blocks inside the tensor
// core.  Each K block is one MMA group into its own TMEM column slice; the
// epilogue warps read the slice back and apply d_w * d_x in fp32.
//
// Exactness: the MMA runs kind::f16 on bf16 operands that hold small
// integers exactly -- A = 128 + u (u = q + 8, the stored nibble), B = q_x --
// plus one correction MMA that adds -136 * sum(q_x), so the fp32 sum in TMEM
// is the exact integer dot sum q_w * q_x (all partial sums < 2^21).
//
// Pipeline (one CTA = 128 weight rows x NTOK tokens x its K range):
//   warp 0      TMA producer: nibble tile (128B swizzle), scale tile, Q8_0
//               activation tile and its scales, 8 K blocks per stage
//   warp 1      TMEM allocation; lane 0 issues the MMAs
//   warps 2-5   converters: nibbles -> bf16 A tile, int8 -> bf16 B tile and
//               correction rows, fp32 scales for the epilogue
//   warps 6-9   epilogue: tcgen05.ld per K block, y += d_w*d_x*dot
// Every mbarrier wait is bounded (2 s); on expiry the kernel sets the device
// error word, drains its own copies / MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "qmm.h"
#include "qmm_device.cuh"
#include "qmm_tc.h"

namespace qmm {
namespace tc {

constexpr int ROWS = 128;           // MMA M (weight rows per CTA)
constexpr int KB_STAGE = 8;         // K blocks per TMA stage
constexpr int RAW_STAGES = 2;
constexpr int CONV_BUFS_MAX = 16;   // converted K blocks in flight (per NTOK, see conv_bufs)
constexpr int THREADS = 320;
constexpr int WARP_TMA = 0, WARP_MMA = 1, WARP_CONV0 = 2, WARP_EPI0 = 6;
constexpr int NCONV = 4, NEPI = 4;

// converted K blocks in flight: as many as shared memory allows
__host__ __device__ constexpr int conv_bufs(int ntok) { return ntok <= 16 ? 16 : ntok <= 32 ? 12 : 8; }
// K blocks converted per handshake with the MMA warp (divides KB_STAGE and conv_bufs)
__host__ __device__ constexpr int conv_group(int ntok) { return ntok <= 16 ? 8 : 4; }

struct Layout {
    // byte offsets in dynamic shared memory (base aligned to 1024)
    int raw, raw_stage, a_nib, a_d, x_q, x_d;  // raw stage parts (relative to stage base)
    int conv, conv_stride, conv_a, conv_b;     // conversion buffers
    int aextra;                                 // constant correction A tile
    int scal, scal_stride;                      // per-slot fp32 scales (dw[128], dx[NTOK])
    int bars, total;
};

__host__ __device__ inline Layout layout(int ntok, int slots) {
    // Conversion buffers and the constant correction tile come first and the
    // raw TMA stages after them, so every MMA operand read stays inside the
    // allocation with room to spare.
    Layout L;
    L.conv = 0;
    L.conv_a = 0;                                // 4 chunks x 128 rows x 16 B
    L.conv_b = ROWS * 64;                        // 6 chunks x ntok x 16 B
    L.conv_stride = (L.conv_b + 6 * ntok * 16 + 127) / 128 * 128;
    L.aextra = L.conv + conv_bufs(ntok) * L.conv_stride;  // 2 chunks x 128 rows x 16 B
    L.a_nib = 0;                                 // 128 rows x 128 B, 128B-swizzled (1024-aligned)
    L.a_d = ROWS * 128;                          // 128 rows x 8 fp16
    L.x_q = L.a_d + ROWS * 16;                   // ntok rows x 256 B int8
    L.x_d = L.x_q + ntok * 256;                  // ntok rows x 8 fp16
    L.raw_stage = (L.x_d + ntok * 16 + 1023) / 1024 * 1024;
    L.raw = (L.aextra + 2 * ROWS * 16 + 1023) / 1024 * 1024;
    L.scal = L.raw + RAW_STAGES * L.raw_stage;
    L.scal_stride = (ROWS + ntok) * 4;
    L.bars = (L.scal + slots * L.scal_stride + 127) / 128 * 128;
    L.total = L.bars + 1024;
    return L;
}

// mbarrier slots inside the barrier area
struct Bars {
    uint64_t* raw_full;    // [RAW_STAGES]    TMA bytes
    uint64_t* raw_empty;   // [RAW_STAGES]    converters (4 warps)
    uint64_t* conv_full;   // [CONV_BUFS_MAX] converters (4 warps)
    uint64_t* conv_empty;  // [CONV_BUFS_MAX] MMA commit
    uint64_t* tm_full;     // [slots]       MMA commit
    uint64_t* tm_empty;    // [slots]       epilogue (4 warps)
    uint64_t* sc_full;     // [slots]       converters (4 warps)
    uint64_t* mma_done;    // [1]           final MMA commit
    uint32_t* tmem_base;
    volatile int* abort;
};

__device__ inline Bars bars_at(uint8_t* p, int slots) {
    Bars b;
    uint64_t* q = reinterpret_cast<uint64_t*>(p);
    b.raw_full = q;
    b.raw_empty = q + RAW_STAGES;
    b.conv_full = b.raw_empty + RAW_STAGES;
    b.conv_empty = b.conv_full + CONV_BUFS_MAX;
    b.tm_full = b.conv_empty + CONV_BUFS_MAX;
    b.tm_empty = b.tm_full + slots;
    b.sc_full = b.tm_empty + slots;
    b.mma_done = b.sc_full + slots;
    b.tmem_base = reinterpret_cast<uint32_t*>(b.mma_done + 1);
    b.abort = reinterpret_cast<volatile int*>(b.tmem_base + 1);
    return b;
}

struct Args {
    int64_t N, K, M;
    float* y;
    int64_t ldy;
    int ntok_slots;  // TMEM slots (K blocks in flight between MMA and epilogue)
    int* err;
};

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ uint64_t umma_desc(const void* smem_ptr, uint32_t lbo, uint32_t sbo) {
    const uint64_t addr = smem_u32(smem_ptr);
    return ((addr >> 4) & 0x3FFFull) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46);  // version 1, no swizzle
}

__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, int accum) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accum)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 16 consecutive TMEM columns of this thread's lane; completes at tmem_wait_ld()
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// bf16 pair from two small integers (exact for |v| < 256)
__device__ __forceinline__ uint32_t bf16x2_from_ints(int lo, int hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"((float)hi), "f"((float)lo));
    return r;
}

// ---------------------------------------------------------------- kernel
template <int NTOK>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap map_wq, const __grid_constant__ CUtensorMap map_wd,
                   const __grid_constant__ CUtensorMap map_xq, const __grid_constant__ CUtensorMap map_xd, Args a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int SL = a.ntok_slots;
    constexpr int CB = conv_bufs(NTOK);
    const Layout L = layout(NTOK, SL);
    const Bars br = bars_at(smem + L.bars, SL);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t n0 = (int64_t)blockIdx.x * ROWS;
    const int nkb = (int)(a.K / QK);        // K blocks
    const int nstage = nkb / KB_STAGE;      // host guarantees nkb % 8 == 0

    if (tid == 0) {
        for (int i = 0; i < RAW_STAGES; ++i) {
            mbar_init(&br.raw_full[i], 1);
            mbar_init(&br.raw_empty[i], NCONV);
        }
        for (int i = 0; i < CB; ++i) {
            mbar_init(&br.conv_full[i], NCONV);
            mbar_init(&br.conv_empty[i], 1);
        }
        for (int i = 0; i < SL; ++i) {
            mbar_init(&br.tm_full[i], 1);
            mbar_init(&br.tm_empty[i], NEPI);
            mbar_init(&br.sc_full[i], NCONV);
        }
        mbar_init(br.mma_done, 1);
        *br.abort = 0;
        fence_mbar_init();
    }
    // constant parts: correction A tile (136, 136, 0...) and the zero 6th chunk of each B buffer
    for (int i = tid; i < 2 * ROWS; i += THREADS) {
        uint4 v = make_uint4(0, 0, 0, 0);
        if (i < ROWS) v.x = 0x43084308u;  // bf16(136) twice: K elements 0 and 1 of chunk 0
        *reinterpret_cast<uint4*>(smem + L.aextra + i * 16) = v;
    }
    for (int cb = 0; cb < CB; ++cb)
        for (int i = tid; i < 2 * NTOK; i += THREADS)
            *reinterpret_cast<uint4*>(smem + L.conv + cb * L.conv_stride + L.conv_b + (4 * NTOK + i) * 16) =
                make_uint4(0, 0, 0, 0);
    if (warp == WARP_MMA) {
        const uint32_t ncols = (uint32_t)(SL * NTOK);
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(br.tmem_base)),
                     "r"(ncols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *br.tmem_base;

    if (warp == WARP_TMA) {
        if (lane == 0) {
            int issued = 0;
            bool ok = true;
            const uint32_t stage_bytes = ROWS * 128 + ROWS * 16 + NTOK * 256 + NTOK * 16;
            for (int s = 0; s < nstage; ++s) {
                const int r = s % RAW_STAGES;
                if (s >= RAW_STAGES && !mbar_wait(&br.raw_empty[r], ((s / RAW_STAGES) - 1) & 1, br.abort)) {
                    ok = false;
                    break;
                }
                uint8_t* st = smem + L.raw + r * L.raw_stage;
                mbar_arrive_expect_tx(&br.raw_full[r], stage_bytes);
                const int kb0 = s * KB_STAGE;
                tma_load_2d(st + L.a_nib, &map_wq, kb0 * 16, (int)n0, &br.raw_full[r]);
                tma_load_2d(st + L.a_d, &map_wd, kb0, (int)n0, &br.raw_full[r]);
                tma_load_2d(st + L.x_q, &map_xq, kb0 * 32, 0, &br.raw_full[r]);
                tma_load_2d(st + L.x_d, &map_xd, kb0, 0, &br.raw_full[r]);
                issued = s + 1;
            }
            if (!ok) {
                atomicOr(a.err, ERR_TIMEOUT);
                *br.abort = 1;
            }
            // copies already issued must land before the CTA can exit
            for (int s = max(0, issued - RAW_STAGES); s < issued; ++s) {
                const uint64_t t0 = global_ns();
                while (!mbar_try_wait(&br.raw_full[s % RAW_STAGES], (s / RAW_STAGES) & 1) &&
                       global_ns() - t0 < WAIT_LIMIT_NS) {
                }
            }
        }
    } else if (warp == WARP_MMA) {
        if (lane == 0) {
            // idesc: D f32, A/B bf16, both K-major, N = NTOK, M = 128
            const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(NTOK >> 3) << 17) |
                                   ((uint32_t)(ROWS >> 4) << 24);
            bool ok = true;
            int done = 0;
            constexpr int CG = conv_group(NTOK), NSLOT = CB / CG;
            for (int g = 0; g * CG < nkb && ok; ++g) {
                if (!mbar_wait(&br.conv_full[g % NSLOT], (g / NSLOT) & 1, br.abort)) { ok = false; break; }
                for (int jj = 0; jj < CG; ++jj) {
                    const int j = g * CG + jj, cb = j % CB, sl = j % SL;
                    if (j >= SL && !mbar_wait(&br.tm_empty[sl], ((j / SL) - 1) & 1, br.abort)) { ok = false; break; }
                    tc_fence_after();
                    const uint8_t* cbuf = smem + L.conv + cb * L.conv_stride;
                    const uint32_t d = tmem + (uint32_t)(sl * NTOK);
                    const uint32_t lbo_a = ROWS * 16, lbo_b = NTOK * 16;
                    umma_f16(d, umma_desc(cbuf + L.conv_a, lbo_a, 128), umma_desc(cbuf + L.conv_b, lbo_b, 128), idesc,
                             0);
                    umma_f16(d, umma_desc(cbuf + L.conv_a + 2 * ROWS * 16, lbo_a, 128),
                             umma_desc(cbuf + L.conv_b + 2 * NTOK * 16, lbo_b, 128), idesc, 1);
                    umma_f16(d, umma_desc(smem + L.aextra, lbo_a, 128),
                             umma_desc(cbuf + L.conv_b + 4 * NTOK * 16, lbo_b, 128), idesc, 1);
                    umma_commit(&br.tm_full[sl]);
                    done = j + 1;
                }
                if (ok) umma_commit(&br.conv_empty[g % NSLOT]);  // the group's buffers may be refilled
            }
            if (!ok) {
                atomicOr(a.err, ERR_TIMEOUT);
                *br.abort = 1;
            }
            if (done > 0) {  // all issued MMAs complete before TMEM is freed
                umma_commit(br.mma_done);
                const uint64_t t0 = global_ns();
                while (!mbar_try_wait(br.mma_done, 0) && global_ns() - t0 < WAIT_LIMIT_NS) {
                }
            }
        }
    } else if (warp < WARP_EPI0) {
        // ---------------- converters: thread r (0..127) owns weight row r;
        // CG K blocks per handshake (one wait, one proxy fence, one arrive)
        const int r = tid - WARP_CONV0 * 32;
        constexpr int CG = conv_group(NTOK), NSLOT = CB / CG;
        for (int g = 0; g * CG < nkb; ++g) {
            const int j0 = g * CG;
            const int s = j0 / KB_STAGE, rs = s % RAW_STAGES;
            // every lane waits (acquire), then the warp agrees, so the warp-wide
            // shuffles below are never reached by only part of it
            bool ok = true;
            if (j0 % KB_STAGE == 0) ok = mbar_wait(&br.raw_full[rs], (s / RAW_STAGES) & 1, br.abort);
            if (ok && g >= NSLOT) ok = mbar_wait(&br.conv_empty[g % NSLOT], ((g / NSLOT) - 1) & 1, br.abort);
            // scale slots of this group are free once the epilogue released the last of them
            const int jl = j0 + CG - 1;
            if (ok && jl >= SL) ok = mbar_wait(&br.tm_empty[jl % SL], ((jl / SL) - 1) & 1, br.abort);
            if (!__all_sync(0xffffffffu, ok)) {
                *br.abort = 1;
                break;
            }
            const uint8_t* st = smem + L.raw + rs * L.raw_stage;
            const uint16_t* wd = reinterpret_cast<const uint16_t*>(st + L.a_d);
            const uint16_t* xdp = reinterpret_cast<const uint16_t*>(st + L.x_d);
#pragma unroll 2
            for (int jj = 0; jj < CG; ++jj) {
                const int j = j0 + jj, bi = j % KB_STAGE, cb = j % CB, sl = j % SL;
                uint8_t* cbuf = smem + L.conv + cb * L.conv_stride;
                float* sc = reinterpret_cast<float*>(smem + L.scal + sl * L.scal_stride);
                // A: 16 nibble bytes of (row r, block bi), 128B-swizzled tile
                const uint4 w = lds128(st + L.a_nib + r * 128 + ((bi ^ (r & 7)) << 4));
                const uint32_t C = 0x43u, LO = 0x0F0F0F0Fu;
                const uint32_t lo0 = w.x & LO, lo1 = w.y & LO, lo2 = w.z & LO, lo3 = w.w & LO;
                const uint32_t hi0 = (w.x >> 4) & LO, hi1 = (w.y >> 4) & LO, hi2 = (w.z >> 4) & LO,
                               hi3 = (w.w >> 4) & LO;
                uint8_t* ca = cbuf + L.conv_a + r * 16;
                *reinterpret_cast<uint4*>(ca + 0 * ROWS * 16) =
                    make_uint4(__byte_perm(lo0, C, 0x4140), __byte_perm(lo0, C, 0x4342), __byte_perm(lo1, C, 0x4140),
                               __byte_perm(lo1, C, 0x4342));
                *reinterpret_cast<uint4*>(ca + 1 * ROWS * 16) =
                    make_uint4(__byte_perm(lo2, C, 0x4140), __byte_perm(lo2, C, 0x4342), __byte_perm(lo3, C, 0x4140),
                               __byte_perm(lo3, C, 0x4342));
                *reinterpret_cast<uint4*>(ca + 2 * ROWS * 16) =
                    make_uint4(__byte_perm(hi0, C, 0x4140), __byte_perm(hi0, C, 0x4342), __byte_perm(hi1, C, 0x4140),
                               __byte_perm(hi1, C, 0x4342));
                *reinterpret_cast<uint4*>(ca + 3 * ROWS * 16) =
                    make_uint4(__byte_perm(hi2, C, 0x4140), __byte_perm(hi2, C, 0x4342), __byte_perm(hi3, C, 0x4140),
                               __byte_perm(hi3, C, 0x4342));
                sc[r] = f16_bits_to_f32(wd[r * KB_STAGE + bi]);
                // B: 4 threads per token, 8 activations each
                for (int t = r; t < 4 * NTOK; t += NCONV * 32) {
                    const int tok = t >> 2, c = t & 3;
                    const uint2 q8 = *reinterpret_cast<const uint2*>(st + L.x_q + tok * 256 + bi * 32 + c * 8);
                    int v[8];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        v[i] = (int)(int8_t)(q8.x >> (8 * i));
                        v[4 + i] = (int)(int8_t)(q8.y >> (8 * i));
                    }
                    *reinterpret_cast<uint4*>(cbuf + L.conv_b + (c * NTOK + tok) * 16) =
                        make_uint4(bf16x2_from_ints(v[0], v[1]), bf16x2_from_ints(v[2], v[3]),
                                   bf16x2_from_ints(v[4], v[5]), bf16x2_from_ints(v[6], v[7]));
                    int sum = v[0] + v[1] + v[2] + v[3] + v[4] + v[5] + v[6] + v[7];
                    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
                    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
                    if (c == 0) {
                        // -sum = -64*hi - lo exactly, both bf16-exact; the A tile holds 136 twice
                        const int hi = sum >> 6, lo = sum - 64 * hi;
                        *reinterpret_cast<uint4*>(cbuf + L.conv_b + (4 * NTOK + tok) * 16) =
                            make_uint4(bf16x2_from_ints(-64 * hi, -lo), 0u, 0u, 0u);
                    } else if (c == 1) {
                        sc[ROWS + tok] = f16_bits_to_f32(xdp[tok * KB_STAGE + bi]);
                    }
                }
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&br.conv_full[g % NSLOT]);
                for (int jj = 0; jj < CG; ++jj) mbar_arrive(&br.sc_full[(j0 + jj) % SL]);
                if ((j0 + CG) % KB_STAGE == 0) mbar_arrive(&br.raw_empty[rs]);
            }
        }
    } else {
        // ---------------- epilogue: thread owns row (warp % 4) * 32 + lane
        // G K blocks per round: wait for all G slots, issue every TMEM load,
        // one wait, then the fp32 scale-and-add.
        constexpr int G = NTOK >= 64 ? 1 : 64 / NTOK;
        const int q = warp & 3;
        const int row = q * 32 + lane;
        float acc[NTOK];
#pragma unroll
        for (int t = 0; t < NTOK; ++t) acc[t] = 0.f;
        bool ok = true;
        for (int j0 = 0; j0 < nkb; j0 += G) {
            const int ng = min(G, nkb - j0);
            bool got = true;
            for (int g = 0; g < ng && got; ++g) {
                const int j = j0 + g, sl = j % SL;
                got = mbar_wait(&br.tm_full[sl], (j / SL) & 1, br.abort) &&
                      mbar_wait(&br.sc_full[sl], (j / SL) & 1, br.abort);
            }
            if (!__all_sync(0xffffffffu, got)) {  // tcgen05.ld below is warp-collective
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t v[G][NTOK];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                if (g < ng) {
                    const int sl = (j0 + g) % SL;
#pragma unroll
                    for (int t0 = 0; t0 < NTOK; t0 += 16)
                        tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(sl * NTOK + t0), &v[g][t0]);
                }
            }
            tmem_wait_ld();
#pragma unroll
            for (int g = 0; g < G; ++g) {
                if (g < ng) {
                    const int sl = (j0 + g) % SL;
                    const float* sc = reinterpret_cast<const float*>(smem + L.scal + sl * L.scal_stride);
                    const float dw = sc[row];
                    const float4* sx = reinterpret_cast<const float4*>(sc + ROWS);
#pragma unroll
                    for (int t4 = 0; t4 < NTOK / 4; ++t4) {
                        const float4 dx = sx[t4];
                        acc[4 * t4 + 0] = fmaf(dw * dx.x, __uint_as_float(v[g][4 * t4 + 0]), acc[4 * t4 + 0]);
                        acc[4 * t4 + 1] = fmaf(dw * dx.y, __uint_as_float(v[g][4 * t4 + 1]), acc[4 * t4 + 1]);
                        acc[4 * t4 + 2] = fmaf(dw * dx.z, __uint_as_float(v[g][4 * t4 + 2]), acc[4 * t4 + 2]);
                        acc[4 * t4 + 3] = fmaf(dw * dx.w, __uint_as_float(v[g][4 * t4 + 3]), acc[4 * t4 + 3]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                for (int g = 0; g < ng; ++g) mbar_arrive(&br.tm_empty[(j0 + g) % SL]);
        }
        if (!ok) {
            if (lane == 0) atomicOr(a.err, ERR_TIMEOUT);
            *br.abort = 1;
        } else if (n0 + row < a.N) {
#pragma unroll
            for (int t = 0; t < NTOK; ++t)
                if (t < a.M) a.y[(int64_t)t * a.ldy + n0 + row] = acc[t];
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == WARP_MMA) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"((uint32_t)(SL * NTOK))
                     : "memory");
    }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        cudaGetLastError();
    });
    return fn;
}

bool make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
              uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
    return make_tensor_map_2d(m, dt, base, inner, outer, row_bytes, box_inner, box_outer, sw);
}

}  // namespace tc

bool make_tensor_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                        uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
    auto fn = tc::encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t es[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace tc {

template <int NTOK>
qmm_status launch_ntok(const uint8_t* w_qs, const uint16_t* w_d, int64_t N, int64_t K, int64_t M, const int8_t* xq,
                       const uint16_t* xd, float* y, int64_t ldy, int* err, cudaStream_t st) {
    const int64_t B = K / QK;
    CUtensorMap mwq, mwd, mxq, mxd;
    if (!make_map(&mwq, CU_TENSOR_MAP_DATA_TYPE_UINT8, w_qs, (uint64_t)K / 2, (uint64_t)N, (uint64_t)K / 2, 128, ROWS,
                  CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&mwd, CU_TENSOR_MAP_DATA_TYPE_UINT16, w_d, (uint64_t)B, (uint64_t)N, (uint64_t)B * 2, KB_STAGE, ROWS,
                  CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map(&mxq, CU_TENSOR_MAP_DATA_TYPE_UINT8, xq, (uint64_t)K, (uint64_t)M, (uint64_t)K, KB_STAGE * 32, NTOK,
                  CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map(&mxd, CU_TENSOR_MAP_DATA_TYPE_UINT16, xd, (uint64_t)B, (uint64_t)M, (uint64_t)B * 2, KB_STAGE, NTOK,
                  CU_TENSOR_MAP_SWIZZLE_NONE))
        return QMM_ERR_CUDA;
    const int slots = std::min(16, 512 / NTOK);
    const Layout L = layout(NTOK, slots);
    const int smem = L.total + 1024;  // + alignment slack
    auto kern = gemm_tc_kernel<NTOK>;
    static std::once_flag attr_once;
    static bool attr_ok = false;
    std::call_once(attr_once, [&] {
        attr_ok = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) == cudaSuccess;
    });
    if (!attr_ok || smem > 227 * 1024) {
        cudaGetLastError();
        return QMM_ERR_SHAPE;
    }
    Args a;
    a.N = N;
    a.K = K;
    a.M = M;
    a.y = y;
    a.ldy = ldy;
    a.ntok_slots = slots;
    a.err = err;
    dim3 grid((unsigned)((N + ROWS - 1) / ROWS));
    kern<<<grid, THREADS, smem, st>>>(mwq, mwd, mxq, mxd, a);
    return cudaGetLastError() == cudaSuccess ? QMM_OK : QMM_ERR_CUDA;
}

}  // namespace tc

qmm_status gemm_tc_launch(const uint8_t* w_qs, const uint16_t* w_d, int64_t N, int64_t K, int64_t M,
                          const int8_t* xq, const uint16_t* xd, float* y, int64_t ldy, int* err, cudaStream_t st) {
    if (M <= 16) return tc::launch_ntok<16>(w_qs, w_d, N, K, M, xq, xd, y, ldy, err, st);
    if (M <= 32) return tc::launch_ntok<32>(w_qs, w_d, N, K, M, xq, xd, y, ldy, err, st);
    return tc::launch_ntok<64>(w_qs, w_d, N, K, M, xq, xd, y, ldy, err, st);
}

bool gemm_tc_eligible(int64_t N, int64_t K, int64_t M, const void* w_qs, const void* w_d, const void* xq,
                      const void* xd) {
    auto al = [](const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; };
    return M >= 1 && M <= 64 && K % 256 == 0 && N >= 1 && N < (int64_t(1) << 31) && K < (int64_t(1) << 31) &&
           al(w_qs, 16) && al(w_d, 16) && al(xq, 16) && al(xd, 16) && tc::encode_fn() != nullptr;
}

}  // namespace qmm
