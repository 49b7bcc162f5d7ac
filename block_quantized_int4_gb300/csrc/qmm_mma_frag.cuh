// qmm_mma_frag.cuh -- pieces shared by the warp-MMA GEMM translation units
// (qmm_gemm_mma.cu, qmm_gemm_prep.cu): TMA tile copies, the fp16 operand
// encodings of the weight nibbles and activation codes, the m16n8k16 MMA,
// ldmatrix, a bounded mbarrier wait, the cluster barrier, and the host-side
// shared-memory opt-in.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>
#include <set>
#include <utility>

#include "qmm_device.cuh"

namespace qmm {
namespace frag {

// 2D tile copy of weight bytes, evicted first from L2 (l2_evict_first_policy).
__device__ __forceinline__ void tma2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                      uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, "
        "{%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

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

// Operand encodings (fp16 bit patterns; 0xE480 = -1152, 0x2C00 = 1/16,
// 0xD480 = -72).
//
// Weights: one word of a weight row (bytes 4t..4t+3 of a block, byte i =
// u_i | v_i << 4 with u = element 4t+i, v = element 16+4t+i, codes stored as
// q + 8) -> four fp16 pairs by masking alone, as fp16 subnormals: a half
// word holding the bit pattern n is the fp16 value n * 2^-24, so
//   o[0] = u * 2^-24 for elements (4t, 4t+2), o[1] the same for (4t+1, 4t+3),
//   o[2] = 16 v * 2^-24 for elements (16+4t, 16+4t+2), o[3] for (16+4t+1, ..+3),
// each one AND of the word with one constant.
// Activations: the low half block as x itself, the high half as x / 16 (exact:
// (1152 + x) / 16 - 72).  Then the low-half MMA sums 2^-24 u x = 2^-24 (q + 8) x
// and the high-half MMA sums 2^-24 16 v x / 16 = 2^-24 (q + 8) x, so seeding
// the accumulator with c = -8 * 2^-24 * (sum x_lo + sum x_hi) leaves exactly
// 2^-24 * sum q * x: every product is an integer times 2^-24 and every
// partial sum an integer below 2^23 in magnitude times 2^-24, exact in fp32.
// The 2^24 goes into the staged activation scale (a power of two, so the
// rescaled fp32 result is the same as with unscaled integers, bit for bit).
__device__ __forceinline__ void nibbles_sub(uint32_t w, uint32_t (&o)[4]) {
    const uint32_t w8 = w >> 8;
    o[0] = w & 0x000F000Fu;
    o[1] = w8 & 0x000F000Fu;
    o[2] = w & 0x00F000F0u;
    o[3] = w8 & 0x00F000F0u;
}

// One word of activation codes (four int8 x0..x3) -> the B fragment pair
// (x0, x2), (x1, x3) as fp16: (1024 + (x + 128)) - 1152 = x (x ^ 0x80 = x + 128
// for a two's-complement byte).
__device__ __forceinline__ uint2 codes_lo_f16(uint32_t x) {
    uint2 r;
    r.x = hadd2((x & 0x00FF00FFu) ^ 0x64806480u, 0xE480E480u);
    r.y = hadd2(((x >> 8) & 0x00FF00FFu) ^ 0x64806480u, 0xE480E480u);
    return r;
}

// The same pairs divided by 16: (1152 + x) / 16 - 72 = x / 16, exact.
__device__ __forceinline__ uint2 codes_hi_f16(uint32_t x) {
    uint2 r;
    r.x = hfma2((x & 0x00FF00FFu) ^ 0x64806480u, 0x2C002C00u, 0xD480D480u);
    r.y = hfma2(((x >> 8) & 0x00FF00FFu) ^ 0x64806480u, 0x2C002C00u, 0xD480D480u);
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

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// 2D tile copy that stays in L2 (the activation codes: every CTA reads them).
__device__ __forceinline__ void tma2d_keep(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// 3D tile copies (the nibble columns of a unit in one box, the code boxes
// of a unit in one box): weights evicted first, activation codes kept.
__device__ __forceinline__ void tma3d_ef(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, "
        "{%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma3d_keep(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// Every wait is bounded; a plain try_wait lets the hardware hold the warp
// until the phase completes (or its own short limit passes).
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, volatile int* abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort || global_ns() - t0 > WAIT_LIMIT_NS) return false;
    }
    return true;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- host side
inline std::mutex g_attr_mu;
inline std::set<std::pair<const void*, int>> g_attr_done;

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

}  // namespace frag
}  // namespace qmm
