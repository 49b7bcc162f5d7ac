// qmm_gemm_mma.cu -- small-batch GEMM (up to 64 tokens per weight pass) of
// Q4_0 weights with Q8_0 activations on the warp-level tensor-core MMA:
// mma.sync m16n8k16 with fp16 operands and fp32 accumulation.
//
// Exact integer block dots on a float MMA: the weight codes q = u - 8 lie in
// [-8, 7] and the activation codes in [-127, 127]; both are exact in fp16,
// every product is exact, and a block's 32-term sum is an integer of
// magnitude at most 32 * 8 * 127 = 32,512, exact in fp32.  So the MMA result
// of one block is the integer dot of the method (llama.cpp guide,
// kenji.blog/id, section 2.2: y ~ Delta * Delta_x * sum q * q_x), and the
// rescale d_w * d_x * dot plus the sum over blocks are fp32 operations, as in
// the GEMV kernels.
//
// Why this instruction on sm_103a: tcgen05 has no integer MMA kind here, and
// with 8..64 token columns a 128-row tcgen05 MMA is latency-bound, whereas
// the warp MMA takes its operands from registers -- the nibbles become fp16
// in registers (no shared-memory round trip for the weights' converted
// form) and the per-block rescale is applied to the accumulator fragment in
// registers.
//
// Work layout:
//  - A CTA owns rows_per_cta consecutive weight rows (a multiple of 16),
//    walked in groups of up to 128 rows = 8 row tiles of 16.  A group is
//    streamed in units of UKB blocks by a producer warp: per row tile, one
//    2D TMA copy of 16 rows x 8 blocks of nibbles (128-byte swizzled, which
//    makes the fragment loads below bank-conflict free) per 8 blocks, and
//    one of the 16 rows x UKB scales (swizzled over its own row pitch).
//  - Eight consumer warps.  In a full group warp w owns row tile w for the
//    whole K range.  In a CTA's last group of T < 8 tiles, warp w takes tile
//    w % T and every P-th block of each unit (P = warps on that tile); their
//    partial sums meet in shared memory at the end of the group.
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
#include "qmm_tc.h"

namespace qmm {
namespace mmak {

constexpr int CW = 8;              // consumer warps
constexpr int NCT = CW * 32;       // consumer threads
constexpr int THREADS = NCT + 32;  // + one producer warp
constexpr int GROUP_TILES = CW;    // row tiles of 16 per full group
constexpr int GROUP_ROWS = 16 * GROUP_TILES;
constexpr int MAX_STAGES = 8;
constexpr int XPER = 2;            // activation items per consumer thread per unit (8 * NT * UKB <= 512)
constexpr int SPER = 1;            // scale items per consumer thread per unit (4 * NT * UKB <= 256)

// Blocks per unit for NT token tiles: the unit's fp16 fragments (NT * UKB *
// 512 bytes) stay at 32 KB or less.
__host__ __device__ constexpr int unit_blocks(int nt) { return nt >= 8 ? 8 : nt >= 4 ? 16 : 32; }

struct Args {
    int64_t N, K, M, ldy;
    const int8_t* xq;
    const uint16_t* xd;
    float* y;
    int rows_per_cta;  // a multiple of 16
    int nstages;
    int stage_bytes;   // GROUP_ROWS * UKB * 18, rounded up to 1024
    int off_xbuf, off_xsc, off_red;  // from the 1024-aligned base; the ring starts at 1024
    int* err;
};

__device__ __forceinline__ void tma2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, %0;" ::"r"(NCT) : "memory"); }

__device__ __forceinline__ uint32_t hadd2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t r;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}

// fp16 bit patterns used below: 0x6400 = 1024 (unit spacing, so OR-ing a
// small integer n into the mantissa gives 1024 + n exactly); 0xE408 = -1032,
// 0xE480 = -1152, 0x2C00 = 1/16, 0xD480 = -72.
//
// One word of a weight row (bytes 4t..4t+3 of a block, byte i = u_i | v_i << 4
// with u = element 4t+i, v = element 16+4t+i, codes stored as q + 8) -> the
// four fp16 pairs (q of elements (4t, 4t+2), (4t+1, 4t+3), and the same +16).
// Low nibbles: (1024 + u) - 1032 = u - 8.  High nibbles stay in place:
// (1024 + 16 v) / 16 - 72 = v - 8.  All exact.
__device__ __forceinline__ void nibbles_to_f16(uint32_t w, uint32_t (&o)[4]) {
    const uint32_t w8 = w >> 8;
    o[0] = hadd2((w & 0x000F000Fu) ^ 0x64006400u, 0xE408E408u);
    o[1] = hadd2((w8 & 0x000F000Fu) ^ 0x64006400u, 0xE408E408u);
    o[2] = hfma2((w & 0x00F000F0u) ^ 0x64006400u, 0x2C002C00u, 0xD480D480u);
    o[3] = hfma2((w8 & 0x00F000F0u) ^ 0x64006400u, 0x2C002C00u, 0xD480D480u);
}

// One word of activation codes (four int8 x0..x3) -> B fragment registers
// (x0, x2) and (x1, x3) as fp16 pairs: (1024 + (x + 128)) - 1152 = x, exact
// (x ^ 0x80 = x + 128 for a two's-complement byte).
__device__ __forceinline__ uint2 codes_to_f16(uint32_t x) {
    uint2 r;
    r.x = hadd2((x & 0x00FF00FFu) ^ 0x64806480u, 0xE480E480u);
    r.y = hadd2(((x >> 8) & 0x00FF00FFu) ^ 0x64806480u, 0xE480E480u);
    return r;
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                         const float (&c)[4]) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
          "f"(c[3]));
}

template <int NT>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_mma_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_d, Args a) {
    constexpr int UKB = unit_blocks(NT);
    constexpr int QBYTES = UKB / 8 * GROUP_ROWS * 128;  // nibble tiles of one stage
    constexpr int U = NT >= 4 ? 2 : 4;                   // blocks in flight per warp
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
    const int ntiles = (nrows + 15) / 16;
    const int ngroups = (ntiles + GROUP_TILES - 1) / GROUP_TILES;
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
        // ---------------- producer warp: lane 0 paces the ring, all lanes issue copies
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
            const int tiles = min(GROUP_TILES, ntiles - g * GROUP_TILES);
            const int r0 = (int)(row_begin + (int64_t)g * GROUP_ROWS);
            const int b0 = kc * UKB, nb = min(UKB, B - b0);
            const int nbox = (nb + 7) / 8;  // 8-block columns wholly past K are not copied
            uint8_t* st = ring + (size_t)s * a.stage_bytes;
            if (lane == 0) mbar_arrive_expect_tx(&full[s], (uint32_t)(tiles * 16 * (nbox * 128 + UKB * 2)));
            __syncwarp();
            const int nq = tiles * nbox;
            for (int i = lane; i < nq + tiles; i += 32) {
                if (i < nq) {
                    const int t = i / nbox, j = i - t * nbox;
                    tma2d(st + j * GROUP_ROWS * 128 + t * 16 * 128, &map_q, (b0 + 8 * j) * 16, r0 + 16 * t, &full[s]);
                } else {
                    const int t = i - nq;
                    tma2d(st + QBYTES + t * 16 * UKB * 2, &map_d, b0, r0 + 16 * t, &full[s]);
                }
            }
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
    const int64_t m0 = (int64_t)blockIdx.y * (8 * NT);
    uint8_t* xbuf = base + a.off_xbuf;  // 2 x [UKB][2 halves][NT][32 lanes] uint2 fragments
    float2* xsc = reinterpret_cast<float2*>(base + a.off_xsc);  // 2 x [UKB][NT][4] (d_x of tokens 2t, 2t+1)
    float* red = reinterpret_cast<float*>(base + a.off_red);    // [7 slots][NT][4][32] partial sums
    constexpr int XBUF_BYTES = UKB * 2 * NT * 256;
    constexpr int XSC_N = UKB * NT * 4;
    constexpr int XITEMS = 8 * NT * UKB, SITEMS = 4 * NT * UKB;
    static_assert(XITEMS <= XPER * NCT && SITEMS <= SPER * NCT, "activation items per unit");

    uint4 px[XPER][2];
    uint32_t ps[SPER];
    // Activation codes and scales of unit column kc into registers.
    auto load_x = [&](int kc) {
        const int b0 = kc * UKB;
#pragma unroll
        for (int r = 0; r < XPER; ++r) {
            const int q = tid + NCT * r;
            px[r][0] = px[r][1] = make_uint4(0u, 0u, 0u, 0u);
            const int tok = q % (8 * NT), bl = q / (8 * NT);
            if (q < XITEMS && m0 + tok < a.M && b0 + bl < B) {
                const uint4* src = reinterpret_cast<const uint4*>(a.xq + (m0 + tok) * a.K + (int64_t)(b0 + bl) * QK);
                px[r][0] = __ldg(src);
                px[r][1] = __ldg(src + 1);
            }
        }
#pragma unroll
        for (int r = 0; r < SPER; ++r) {
            const int i = tid + NCT * r;
            ps[r] = 0u;
            const int bl = i / (4 * NT), j = (i >> 2) % NT, tt = i & 3;
            const int64_t m = m0 + 8 * j + 2 * tt;
            if (i < SITEMS && b0 + bl < B) {
                const uint32_t lo = m < a.M ? __ldg(a.xd + m * B + b0 + bl) : 0u;
                const uint32_t hi = m + 1 < a.M ? __ldg(a.xd + (m + 1) * B + b0 + bl) : 0u;
                ps[r] = lo | (hi << 16);
            }
        }
    };
    // Registers -> fp16 fragments and fp32 scale pairs in buffer `buf`.
    auto store_x = [&](int buf) {
        uint8_t* xb = xbuf + buf * XBUF_BYTES;
#pragma unroll
        for (int r = 0; r < XPER; ++r) {
            const int q = tid + NCT * r;
            if (q < XITEMS) {
                const int tok = q % (8 * NT), bl = q / (8 * NT);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint4 v = px[r][h];
                    const uint2 f0 = codes_to_f16(v.x), f1 = codes_to_f16(v.y);
                    const uint2 f2 = codes_to_f16(v.z), f3 = codes_to_f16(v.w);
                    uint4* dst = reinterpret_cast<uint4*>(xb + (bl * 2 + h) * NT * 256 + tok * 32);
                    dst[0] = make_uint4(f0.x, f0.y, f1.x, f1.y);
                    dst[1] = make_uint4(f2.x, f2.y, f3.x, f3.y);
                }
            }
        }
        float2* xs = xsc + buf * XSC_N;
#pragma unroll
        for (int r = 0; r < SPER; ++r) {
            const int i = tid + NCT * r;
            if (i < SITEMS)
                xs[i] = make_float2(f16_bits_to_f32((unsigned short)(ps[r] & 0xffffu)),
                                    f16_bits_to_f32((unsigned short)(ps[r] >> 16)));
        }
    };

    const float zero[4] = {0.f, 0.f, 0.f, 0.f};
    float2 acc[NT][2];
#pragma unroll
    for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = make_float2(0.f, 0.f);
    constexpr int DPITCH = UKB * 2;        // bytes per row of the scale tile
    constexpr int DMASK = DPITCH / 16 - 1;  // its swizzle: 16-byte chunk ^= (row * pitch / 128) & DMASK
    bool failed = false;

    // One block: nibble words of rows ra, ra + 8 and their scales -> MMAs
    // against every token tile -> rescaled into the accumulators.
    auto block = [&](const uint8_t* st, const uint8_t* xb, const float2* xs, int b, int ra, int dsw_a, int dsw_b) {
        const uint8_t* box = st + (b >> 3) * GROUP_ROWS * 128;
        const int sw = (((b & 7) ^ g8) << 4) + 4 * t4;  // 128-byte swizzle: row & 7 == g8
        const uint32_t w0 = *reinterpret_cast<const uint32_t*>(box + ra * 128 + sw);
        const uint32_t w1 = *reinterpret_cast<const uint32_t*>(box + (ra + 8) * 128 + sw);
        const uint16_t* sd = reinterpret_cast<const uint16_t*>(st + QBYTES);
        const int dchunk = b >> 3, dlo = b & 7;
        const float dw0 = f16_bits_to_f32(sd[ra * UKB + (((dchunk ^ dsw_a) << 3) | dlo)]);
        const float dw1 = f16_bits_to_f32(sd[(ra + 8) * UKB + (((dchunk ^ dsw_b) << 3) | dlo)]);
        uint32_t q0[4], q1[4];
        nibbles_to_f16(w0, q0);
        nibbles_to_f16(w1, q1);
        const uint32_t ah0[4] = {q0[0], q1[0], q0[1], q1[1]};  // elements 0..15 of the block
        const uint32_t ah1[4] = {q0[2], q1[2], q0[3], q1[3]};  // elements 16..31
        const uint8_t* xbb = xb + b * 2 * NT * 256;
        const float2* xsb = xs + b * NT * 4;
        const float2 dwa = make_float2(dw0, dw0), dwb = make_float2(dw1, dw1);
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            const uint2 f0 = *reinterpret_cast<const uint2*>(xbb + j * 256);
            const uint2 f1 = *reinterpret_cast<const uint2*>(xbb + (NT + j) * 256);
            float dd[4];
            mma16816(dd, ah0, f0.x, f0.y, zero);
            mma16816(dd, ah1, f1.x, f1.y, dd);  // exact integer block dots
            const float2 sx = xsb[j * 4];       // d_x of tokens 2t, 2t+1
            acc[j][0] = ffma2_scaled(dwa, sx, make_float2(dd[0], dd[1]), acc[j][0]);  // row ra
            acc[j][1] = ffma2_scaled(dwb, sx, make_float2(dd[2], dd[3]), acc[j][1]);  // row ra + 8
        }
    };

    if (nunits > 0) load_x(0);
    for (int u = 0; u < nunits; ++u) {
        const int g = u / nkc, kc = u - g * nkc, s = u % S, buf = u & 1;
        const int T = min(GROUP_TILES, ntiles - g * GROUP_TILES);  // tiles in this group
        const int tile = warp % T, part = warp / T;
        const int P = (CW - tile + T - 1) / T;  // warps on this warp's tile
        const int ra = 16 * tile + g8;           // this lane's rows in the group: ra and ra + 8
        const int dsw_a = ((ra * DPITCH) >> 7) & DMASK, dsw_b = (((ra + 8) * DPITCH) >> 7) & DMASK;
        store_x(buf);
        if (u + 1 < nunits) load_x((u + 1) % nkc);
        consumers_sync();  // fragments of this unit complete (and the unit before last fully read)
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
            const uint8_t* xb = xbuf + buf * XBUF_BYTES + lane * 8;
            const float2* xs = xsc + buf * XSC_N + t4;
            int b = part;
            for (; b + (U - 1) * P < nb; b += U * P) {
#pragma unroll
                for (int i = 0; i < U; ++i) block(st, xb, xs, b + i * P, ra, dsw_a, dsw_b);
            }
            for (; b < nb; b += P) block(st, xb, xs, b, ra, dsw_a, dsw_b);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);  // stage read: the producer may refill it

        if (kc == nkc - 1) {
            // end of the group: a split tile's partial sums meet in slot
            // (part - 1) * T + tile; the part-0 warp adds them and writes y
            if (T < GROUP_TILES) {
                if (part > 0) {
                    float* rp = red + ((part - 1) * T + tile) * NT * 128 + lane;
#pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        rp[j * 128 + 0] = acc[j][0].x;
                        rp[j * 128 + 32] = acc[j][0].y;
                        rp[j * 128 + 64] = acc[j][1].x;
                        rp[j * 128 + 96] = acc[j][1].y;
                    }
                }
                consumers_sync();
                if (part == 0) {
                    for (int p = 1; p < P; ++p) {
                        const float* rp = red + ((p - 1) * T + tile) * NT * 128 + lane;
#pragma unroll
                        for (int j = 0; j < NT; ++j) {
                            acc[j][0].x += rp[j * 128 + 0];
                            acc[j][0].y += rp[j * 128 + 32];
                            acc[j][1].x += rp[j * 128 + 64];
                            acc[j][1].y += rp[j * 128 + 96];
                        }
                    }
                }
            }
            const int64_t r0 = row_begin + (int64_t)g * GROUP_ROWS;
            const int nr = (int)min((int64_t)GROUP_ROWS, row_end - r0);
            if (part == 0 && !failed) {
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    const int64_t m = m0 + 8 * j + 2 * t4;
#pragma unroll
                    for (int hr = 0; hr < 2; ++hr) {
                        const int lr = ra + 8 * hr;
                        if (lr >= nr) continue;
                        const int64_t row = r0 + lr;
                        if (m < a.M) a.y[m * a.ldy + row] = acc[j][hr].x;
                        if (m + 1 < a.M) a.y[(m + 1) * a.ldy + row] = acc[j][hr].y;
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = make_float2(0.f, 0.f);
        }
    }
}

// ---------------------------------------------------------------- host side
std::mutex g_attr_mu;
std::set<std::pair<const void*, int>> g_attr_done;

// Opt a kernel into `bytes` (the device's opt-in maximum) of dynamic shared
// memory, once per (kernel, device).
template <typename Kern>
bool allow_smem(Kern kernel, int bytes) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lk(g_attr_mu);
    const auto key = std::make_pair(reinterpret_cast<const void*>(kernel), dev);
    if (g_attr_done.count(key)) return true;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    g_attr_done.insert(key);
    return true;
}

inline int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

template <int NT>
qmm_status launch_nt(const uint8_t* w_qs, const uint16_t* w_d, int64_t N, int64_t K, int64_t M, const int8_t* xq,
                     const uint16_t* xd, float* y, int64_t ldy, int sms, int smem_optin, int* err, cudaStream_t st) {
    constexpr int UKB = unit_blocks(NT);
    const int64_t B = K / QK;
    // Rows per CTA: the fewest row tiles that cover N with one CTA per SM.
    const int64_t rpc = round_up((N + sms - 1) / sms, 16);
    const int64_t G = (N + rpc - 1) / rpc;
    const int stage = (int)round_up((int64_t)GROUP_ROWS * UKB * 18, 1024);
    const int xbuf = 2 * UKB * 2 * NT * 256;
    const int xsc = 2 * UKB * NT * 4 * 8;
    const int redb = (CW - 1) * NT * 128 * 4;
    const int fixed = 1024 + xbuf + xsc + redb + 1024;  // header, buffers, alignment slack
    const int64_t nunits = ((rpc + GROUP_ROWS - 1) / GROUP_ROWS) * ((B + UKB - 1) / UKB);
    const int64_t nst = std::min<int64_t>({(int64_t)MAX_STAGES, (smem_optin - fixed) / stage, nunits});
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
    a.stage_bytes = stage;
    a.off_xbuf = 1024 + (int)nst * stage;
    a.off_xsc = a.off_xbuf + xbuf;
    a.off_red = a.off_xsc + xsc;
    a.err = err;
    const int smem = a.off_red + redb + 1024;
    const CUtensorMapSwizzle dsw = UKB == 8 ? CU_TENSOR_MAP_SWIZZLE_NONE
                                   : UKB == 16 ? CU_TENSOR_MAP_SWIZZLE_32B
                                               : CU_TENSOR_MAP_SWIZZLE_64B;
    CUtensorMap mq, md;
    if (!make_tensor_map_2d(&mq, CU_TENSOR_MAP_DATA_TYPE_UINT8, w_qs, (uint64_t)K / 2, (uint64_t)N, (uint64_t)K / 2,
                            128, 16, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map_2d(&md, CU_TENSOR_MAP_DATA_TYPE_UINT16, w_d, (uint64_t)B, (uint64_t)N, (uint64_t)B * 2,
                            (uint32_t)UKB, 16, dsw))
        return QMM_ERR_CUDA;
    auto kern = gemm_mma_kernel<NT>;
    if (smem > smem_optin || !allow_smem(kern, smem_optin)) return QMM_ERR_SHAPE;
    const dim3 grid((unsigned)G, (unsigned)((M + 8 * NT - 1) / (8 * NT)));
    kern<<<grid, THREADS, smem, st>>>(mq, md, a);
    return cudaGetLastError() == cudaSuccess ? QMM_OK : QMM_ERR_CUDA;
}

}  // namespace mmak

bool gemm_mma_eligible(int64_t N, int64_t K, int64_t M, const void* w_qs, const void* w_d, const void* xq,
                       const void* xd) {
    auto al = [](const void* p, uintptr_t n) { return reinterpret_cast<uintptr_t>(p) % n == 0; };
    return N >= 1 && N < (int64_t(1) << 31) && M >= 1 && K >= 256 && K % 256 == 0 && al(w_qs, 16) && al(w_d, 16) &&
           al(xq, 16) && al(xd, 2);
}

qmm_status gemm_mma_launch(const uint8_t* w_qs, const uint16_t* w_d, int64_t N, int64_t K, int64_t M,
                           const int8_t* xq, const uint16_t* xd, float* y, int64_t ldy, int sms, int smem_optin,
                           int* err, cudaStream_t st) {
    if (M <= 8) return mmak::launch_nt<1>(w_qs, w_d, N, K, M, xq, xd, y, ldy, sms, smem_optin, err, st);
    if (M <= 16) return mmak::launch_nt<2>(w_qs, w_d, N, K, M, xq, xd, y, ldy, sms, smem_optin, err, st);
    if (M <= 32) return mmak::launch_nt<4>(w_qs, w_d, N, K, M, xq, xd, y, ldy, sms, smem_optin, err, st);
    return mmak::launch_nt<8>(w_qs, w_d, N, K, M, xq, xd, y, ldy, sms, smem_optin, err, st);
}

}  // namespace qmm
