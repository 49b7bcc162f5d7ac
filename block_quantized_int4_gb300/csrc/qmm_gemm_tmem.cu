// qmm_gemm_tmem.cu -- small-batch GEMM (2..16 tokens) of Q4_0 weights with
// Q8_0 activations on the 5th-generation tensor cores: tcgen05.mma kind::f16
// with the weight operand A held in tensor memory and fp32 block dots
// accumulated in tensor memory.
//
// Method (llama.cpp guide, kenji.blog/id, section 2.2): y ~ Delta * Delta_x *
// sum q * q_x per block of 32, fp32 sum over the blocks; Q4_0 block format of
// the TinyLLaMA C++ guide (kenji.blog) section 6.1.  Every 32-wide block has
// its own scale pair, so one block is one MMA pair into its own TMEM slice,
// read back and rescaled in fp32 by the thread that owns the row.
//
// Exactness: the weight codes go to fp16 as q = u - 8 (elements 0..15 of a
// block) and 16 q (elements 16..31), the activation codes as x and x / 16;
// all are exact in fp16, every product q * x is exact, and a block's 32-term
// sum has magnitude at most 32 * 8 * 127 = 32,512, exact in fp32.  So the
// two K=16 MMAs of a block leave the integer block dot itself in TMEM.
//
// Why A lives in TMEM: the converted weights are written once per block by
// the thread that owns the row (tcgen05.st from registers) and read by the
// MMA from tensor memory, so the 128-row fp16 tile never passes through
// shared memory, whose bandwidth bounded a design that staged it there.
//
// Work layout (one CTA per SM):
//  - A CTA owns nst consecutive super-tiles of H <= 256 weight rows (two MMA
//    tiles of 128 rows) and walks each over all of K in chunks of 8 blocks.
//  - warp 17: TMA producer.  Per chunk one stage: the nibble tile (H rows x
//    128 B, 128-byte swizzled), its scales (H x 8 fp16), the chunk's Q8_0
//    codes of the 16 token rows and their scales (rows >= M are zero-filled).
//  - warps 0..15: worker w owns rows 128 ((w / 4) % 2) + 32 (w % 4) + lane of
//    the super-tile, i.e. TMEM lanes 32 (w % 4) .. + 31 of MMA tile
//    (w / 4) % 2, and the blocks of parity w / 8 of every chunk: two workers
//    share each row, each with its own sums, added through shared memory at
//    the end of a super-tile (per-pair mbarriers, bounded waits).  For its
//    block j a worker reads the dot slice of block j (tcgen05.ld), writes the
//    fp16 codes of block j + 8 into the slice the MMA of block j has
//    finished with (tcgen05.st), signals, and then adds d_w * d_x * dot into
//    its 16 per-token fp32 sums.  Warps 0..7 also turn block w of each
//    chunk's activation codes into the fp16 B operand in shared memory.
//  - warps 16 and 18: one lane each issues the MMAs of one tile (warp 16
//    also allocates TMEM): per block, two M=128 N=16 K=16 MMAs into the
//    block's slice, then one commit to that tile's barrier.
// TMEM: 8 slots (block mod 8) x 2 tiles x (16 columns of A + 16 of D).
// Every wait is bounded; on expiry the kernel sets the device error word,
// lets its own copies and MMAs finish, frees TMEM and returns.
//
// Measured on GB300 (16 tokens, 28672 x 8192): 84 us per call (8 workers:
// 115-117 us) against 44.5 us for the warp-MMA kernel's 16-warp layout, so
// the library routes to this kernel only when asked (qmm_debug_gemm_kernel).
// Each tcgen05.mma costs the tensor core about 45 cycles whatever N (16..64),
// K and operand kind, so the 1024 MMAs of a 192-row share take ~23 us; the
// bound that binds is the workers' per-block work (nibble conversion, TMEM
// store and load, rescale), about as many instructions per row and block as
// the warp-MMA kernel's register path spends, with the TMEM round trip on
// top.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <set>
#include <utility>

#include "qmm_device.cuh"
#include "qmm_mma.h"
#include "qmm_tmap.h"

namespace qmm {
namespace tmk {

constexpr int NTOK = 16;      // MMA N: token columns per launch
constexpr int KB = 8;         // K blocks per chunk (one 128-byte nibble box column); also the TMEM slot count
constexpr int WORKERS = 16;   // worker warps: two per TMEM lane quarter of each tile, one per parity of the blocks
constexpr int PER_BLOCK = 8;  // worker warps that write the A slice of one block (4 lane quarters x 2 tiles)
constexpr int WARP_MMA = 16, WARP_TMA = 17, WARP_MMA1 = 18;  // MMA issuers of tile 0 and tile 1
constexpr int THREADS = 19 * 32;
constexpr int RED_BYTES = 2 * 128 * NTOK * 4;  // the odd-block warps' sums of a super-tile, per row
constexpr int MAX_STAGES = 8;
constexpr uint32_t TMEM_COLS = 512;
constexpr int XQ_BYTES = NTOK * KB * 32;  // activation codes of one chunk
constexpr int XD_BYTES = NTOK * KB * 2;   // their scales
constexpr int BBUF = KB * 1024;           // fp16 B operand of one chunk: [block][half][k chunk][token][16 B]
constexpr int SXB = KB * NTOK * 4;        // d_x of one chunk as fp32: [block][token]
constexpr int NBARS = 2 * MAX_STAGES + 2 + 3 * KB + 2 + 2 * PER_BLOCK;

struct Args {
    int64_t N, K, M, ldy;
    float* y;
    int H;            // rows per super-tile = TMA box height (multiple of 8, <= 256)
    int nst;          // super-tiles per CTA
    int nstages;
    int stage_bytes;  // H * 144 + XQ_BYTES + XD_BYTES, rounded up to 1024
    int off_bbuf, off_sx, off_red, off_bar;  // from the 1024-aligned base
    int* err;
};

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ void tma2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// weight bytes are read once per product: evicted first from L2
__device__ __forceinline__ void tma2d_ef(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, "
        "{%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Shared-memory matrix descriptor, no swizzle, K-major core matrices of
// 8 rows x 16 bytes: lbo = byte distance of core matrices adjacent in K,
// sbo = in the M/N direction.
__device__ __forceinline__ uint64_t smem_desc(const void* p, uint32_t lbo, uint32_t sbo) {
    const uint64_t addr = smem_u32(p);
    return ((addr >> 4) & 0x3FFFull) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46);
}

// D[tmem] (+)= A[tmem] * B[smem]; ACC = 0 overwrites D
template <int ACC>
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "n"(ACC)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 16 consecutive TMEM columns of this thread's lane (warp-collective)
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Wait for this thread's TMEM loads, naming their destination registers, so
// that no use of them is scheduled before the wait.
__device__ __forceinline__ void tmem_wait_ld_regs(uint32_t (&r)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15])
                 :
                 : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

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

// Operand encodings (fp16 bit patterns).  0x6400 is 1024 with unit spacing,
// so OR-ing (here: xor-ing into the zero mantissa) a small integer n gives
// 1024 + n exactly.
//
// Weights: word i of a row's 16 block bytes (byte 4i + p = u | v << 4, u the
// code of element 4i + p, v of element 16 + 4i + p, codes stored as q + 8)
// gives four fp16 pairs:
//   a[2i]     = q of elements (4i, 4i + 2)      (1024 + u) - 1032
//   a[2i + 1] = q of elements (4i + 1, 4i + 3)
//   a[8 + 2i], a[9 + 2i]: the same for elements 16 + ..., as 16 q = (1024 + 16 v) - 1152.
// TMEM column c of a row holds K slots (2c, 2c + 1) of the MMA (low half
// first), so the block's first MMA takes columns 0..7 and the second 8..15.
constexpr uint32_t F16_NEG1032 = 0xE408E408u, F16_NEG1152 = 0xE480E480u;

__device__ __forceinline__ void weights_f16(uint4 w, uint32_t (&a)[16]) {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t w0 = ws[i], w8 = ws[i] >> 8;
        a[2 * i] = hadd2((w0 & 0x000F000Fu) ^ 0x64006400u, F16_NEG1032);
        a[2 * i + 1] = hadd2((w8 & 0x000F000Fu) ^ 0x64006400u, F16_NEG1032);
        a[8 + 2 * i] = hadd2((w0 & 0x00F000F0u) ^ 0x64006400u, F16_NEG1152);
        a[9 + 2 * i] = hadd2((w8 & 0x00F000F0u) ^ 0x64006400u, F16_NEG1152);
    }
}

// Activations: one word of four codes x0..x3 -> the pairs (x0, x2), (x1, x3),
// times `mul` (1 for elements 0..15, 1/16 for 16..31): (1152 + x) * mul -
// 1152 * mul, exact either way ((x ^ 0x80) = x + 128 for a two's-complement byte).
__device__ __forceinline__ uint2 codes_f16(uint32_t x, uint32_t mul, uint32_t add) {
    uint2 r;
    r.x = hfma2((x & 0x00FF00FFu) ^ 0x64806480u, mul, add);
    r.y = hfma2(((x >> 8) & 0x00FF00FFu) ^ 0x64806480u, mul, add);
    return r;
}

// Every lane waits (acquire), then the warp agrees, so a warp-collective
// tcgen05 instruction after it is reached by all lanes or by none.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
    const bool ok = mbar_wait(bar, parity, abort);
    return __all_sync(FULL, ok);
}

__global__ void __launch_bounds__(THREADS, 1)
    gemm_tmem_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_d,
                     const __grid_constant__ CUtensorMap map_xq, const __grid_constant__ CUtensorMap map_xd, Args a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + a.off_bar);
    uint64_t* raw_full = bars;                  // [MAX_STAGES] TMA bytes of a stage
    uint64_t* raw_empty = bars + MAX_STAGES;    // [MAX_STAGES] 8 worker warps done with a stage
    uint64_t* b_full = raw_empty + MAX_STAGES;  // [2] 8 worker warps staged a chunk's B operand
    uint64_t* ready = b_full + 2;               // [KB] 8 worker warps: A written, D read
    uint64_t* full = ready + KB;                // [2][KB] MMA commit per tile: D of the slot's block complete
    uint64_t* mma_done = full + 2 * KB;         // [2]  final MMA commit per issuer
    uint64_t* red_full = mma_done + 2;          // [8] odd-block warp of a row slice wrote its sums
    uint64_t* red_empty = red_full + PER_BLOCK; // [8] even-block warp of it has read them
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NBARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = a.nstages, H = a.H;
    const int nch = (int)(a.K / (QK * KB));  // chunks per super-tile (K % 256 == 0)
    const int64_t row_cta = (int64_t)blockIdx.x * a.nst * H;
    // super-tiles of this CTA that hold rows (the last CTA may hold fewer)
    const int nst = (int)min((int64_t)a.nst, (a.N - row_cta + H - 1) / H);
    const int total = nst * nch;

    if (tid == 0) {
        for (int s = 0; s < MAX_STAGES; ++s) {
            mbar_init(&raw_full[s], 1);
            mbar_init(&raw_empty[s], WORKERS);
        }
        for (int i = 0; i < 2; ++i) mbar_init(&b_full[i], KB);  // warps 0..7 stage one block each
        for (int j = 0; j < KB; ++j) {
            mbar_init(&ready[j], PER_BLOCK);
            mbar_init(&full[j], 1);
            mbar_init(&full[KB + j], 1);
        }
        mbar_init(&mma_done[0], 1);
        mbar_init(&mma_done[1], 1);
        for (int p = 0; p < PER_BLOCK; ++p) {
            mbar_init(&red_full[p], 1);
            mbar_init(&red_empty[p], 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == WARP_MMA) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == WARP_TMA) {
        if (lane == 0) {
            asm volatile("griddepcontrol.wait;" ::: "memory");  // activations come from the kernel before
            const uint64_t pol = l2_evict_first_policy();
            const uint32_t bytes = (uint32_t)(H * 144 + XQ_BYTES + XD_BYTES);
            int issued = 0;
            bool ok = true;
            for (int gc = 0; gc < total; ++gc) {
                const int s = gc % S;
                if (gc >= S && !mbar_wait(&raw_empty[s], ((gc / S) - 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                const int st = gc / nch, c = gc - st * nch;
                const int row = (int)(row_cta + (int64_t)st * H);
                uint8_t* sp = base + (size_t)s * a.stage_bytes;
                mbar_arrive_expect_tx(&raw_full[s], bytes);
                tma2d_ef(sp, &map_q, c * 128, row, &raw_full[s], pol);
                tma2d_ef(sp + H * 128, &map_d, c * KB, row, &raw_full[s], pol);
                tma2d(sp + H * 144, &map_xq, c * KB * 32, (int)(blockIdx.y * NTOK), &raw_full[s]);
                tma2d(sp + H * 144 + XQ_BYTES, &map_xd, c * KB, (int)(blockIdx.y * NTOK), &raw_full[s]);
                issued = gc + 1;
            }
            if (!ok) {
                atomicOr(a.err, ERR_TIMEOUT);
                *abort_flag = 1;
            }
            for (int gc = max(0, issued - S); gc < issued; ++gc) {  // copies in flight land before exit
                const uint64_t t0 = global_ns();
                while (!mbar_try_wait(&raw_full[gc % S], (gc / S) & 1) && global_ns() - t0 < WAIT_LIMIT_NS) {
                }
            }
        }
    } else if (warp == WARP_MMA || warp == WARP_MMA1) {
        // one issuer per MMA tile: the tensor core takes instructions from
        // both while each thread waits out its own issue latency
        const int t = warp == WARP_MMA ? 0 : 1;
        if (lane == 0) {
            // D fp32, A and B fp16, both K-major, N = 16, M = 128
            constexpr uint32_t idesc = (1u << 4) | ((uint32_t)(NTOK >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
            // descriptor of block 0 of B buffer 0; the address field counts 16-byte units
            const uint64_t bdesc0 = smem_desc(base + a.off_bbuf, 256, 128);
            bool ok = true, any = false;
            int st = 0, c = 0;
            bool two = min((int64_t)H, a.N - row_cta) > 128;
            for (int gc = 0; gc < total && ok; ++gc) {
                if (!mbar_wait(&b_full[gc & 1], (gc >> 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint64_t bd = bdesc0 + (uint64_t)((gc & 1) * (BBUF >> 4));
                const uint32_t ph = gc & 1;
#pragma unroll
                for (int jj = 0; jj < KB; ++jj) {
                    if (!mbar_wait(&ready[jj], ph, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (t == 0 || two) {
                        const uint32_t col = tmem + (uint32_t)(jj * 64 + t * 32);
                        mma_ts<0>(col + 16, col, bd + (uint64_t)(jj * 64), idesc);
                        mma_ts<1>(col + 16, col + 8, bd + (uint64_t)(jj * 64 + 32), idesc);
                    }
                    mma_commit(&full[t * KB + jj]);  // arrives at once when nothing was issued
                    any = true;
                }
                if (++c == nch) {  // next super-tile
                    c = 0;
                    ++st;
                    two = min((int64_t)H, a.N - (row_cta + (int64_t)st * H)) > 128;
                }
            }
            if (!ok) {
                atomicOr(a.err, ERR_TIMEOUT);
                *abort_flag = 1;
            }
            if (any) {  // every issued MMA completes before TMEM is freed
                mma_commit(&mma_done[t]);
                const uint64_t t0 = global_ns();
                while (!mbar_try_wait(&mma_done[t], 0) && global_ns() - t0 < WAIT_LIMIT_NS) {
                }
            }
        }
    } else {
        // ---------------- workers: warp w owns TMEM lane quarter q = w & 3 of tile
        // (w >> 2) & 1, and the blocks of parity hf = w >> 3 of every chunk, so
        // two warps share each row's work and every SM sub-partition holds four
        // workers; the two keep their own sums, added at the end of a super-tile
        const int q = warp & 3, tile = (warp >> 2) & 1, hf = warp >> 3;
        const int rl = tile * 128 + q * 32 + lane;  // row inside the super-tile
        const int rs = min(rl, H - 1);              // its shared-memory row (lanes past H read a valid row)
        const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(tile * 32);
        uint64_t* fullt = full + tile * KB;  // this tile's MMA commits
        float* sx = reinterpret_cast<float*>(base + a.off_sx);
        float* red = reinterpret_cast<float*>(base + a.off_red) + ((tile * 128 + q * 32 + lane) * NTOK);
        // the super-tile's rows reach this warp
        auto active = [&](int st) { return row_cta + (int64_t)st * H + tile * 128 + q * 32 < min(a.N, row_cta + (int64_t)(st + 1) * H); };
        // B operand and d_x of chunk gc from its stage (warps 0..7): warp w
        // takes block w, lane = (half, token)
        auto stage_b = [&](int gc) {
            const uint8_t* sp = base + (size_t)(gc % S) * a.stage_bytes;
            const int half = lane >> 4, tok = lane & 15;
            const uint4 x = lds128(sp + H * 144 + tok * (KB * 32) + warp * 32 + half * 16);
            const uint32_t mul = half ? 0x2C002C00u : 0x3C003C00u;  // 1/16 or 1
            const uint32_t add = half ? 0xD480D480u : 0xE480E480u;  // -72 or -1152
            const uint2 p0 = codes_f16(x.x, mul, add), p1 = codes_f16(x.y, mul, add);
            const uint2 p2 = codes_f16(x.z, mul, add), p3 = codes_f16(x.w, mul, add);
            uint8_t* bb = base + a.off_bbuf + (gc & 1) * BBUF + warp * 1024 + half * 512 + tok * 16;
            *reinterpret_cast<uint4*>(bb) = make_uint4(p0.x, p0.y, p1.x, p1.y);
            *reinterpret_cast<uint4*>(bb + 256) = make_uint4(p2.x, p2.y, p3.x, p3.y);
            if (half == 0) {
                const uint16_t* xd = reinterpret_cast<const uint16_t*>(sp + H * 144 + XQ_BYTES);
                sx[(gc % 3) * (SXB / 4) + warp * NTOK + tok] = f16_bits_to_f32(xd[tok * KB + warp]);
            }
            fence_async_smem();  // visible to the MMA's reads
            __syncwarp();
            if (lane == 0) mbar_arrive(&b_full[gc & 1]);
        };
        // fp16 codes of block jj of the stage's rows -> this warp's A slice of slot jj
        auto convert = [&](const uint8_t* sp, int jj) {
            const uint4 w = lds128(sp + rs * 128 + ((jj ^ (rs & 7)) << 4));
            uint32_t av[16];
            weights_f16(w, av);
            tmem_st16(tl + (uint32_t)(jj * 64), av);
        };

        float2 acc[NTOK / 2];
#pragma unroll
        for (int t = 0; t < NTOK / 2; ++t) acc[t] = make_float2(0.f, 0.f);
        const int ngrp = (int)min((int64_t)(NTOK / 4), (a.M + 3) / 4);  // token groups of 4 holding tokens
        bool ok = total > 0;
        uint4 sc_cur = make_uint4(0u, 0u, 0u, 0u), sc_next = sc_cur;
        uint32_t v[16];
        if (ok) {
            // chunk 0: B operand, A of this warp's 4 blocks, the rows' scales
            ok = warp_wait(&raw_full[0], 0, abort_flag);
            if (ok) {
                const uint8_t* sp = base;
                if (warp < KB) stage_b(0);
                const bool act = active(0);
                if (act) sc_cur = lds128(sp + H * 128 + rs * 16);
#pragma unroll
                for (int jj = hf; jj < KB; jj += 2) {
                    if (act) {
                        convert(sp, jj);
                        tmem_wait_st();
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ready[jj]);
                }
                if (lane == 0) mbar_arrive(&raw_empty[0]);
                // the dot slice of this warp's first block on its way
                ok = warp_wait(&fullt[hf], 0, abort_flag);
                tc_fence_after();
                if (ok && act) tmem_ld16(tl + (uint32_t)(hf * 64) + 16u, v);
            }
        }
        // Iteration (gc, jj) rescales block j = 8 gc + jj and converts block
        // j + 8 into the slot the MMA of block j has finished with.  The TMEM
        // load of block j was issued at the end of this warp's iteration before,
        // and the store of block j + 8 completes while block j is rescaled.
        // Chunk-level positions advance by counters (no divisions in the loop):
        // st / c = super-tile and chunk inside it of gc; sn / pn = stage and
        // its phase parity of chunk gn; x3 = gc mod 3.
        int st = 0, c = 0, sn = S > 1 ? 1 : 0, pn = S > 1 ? 0 : 1, x3 = 0;
        bool act = ok && active(0);
        for (int gc = 0; gc < total && ok; ++gc) {
            const int gn = gc + 1;
            const bool has_next = gn < total;
            const bool actn = has_next && active(c + 1 == nch ? st + 1 : st);
            const uint8_t* spn = base + (size_t)sn * a.stage_bytes;
            if (has_next && !(ok = warp_wait(&raw_full[sn], pn, abort_flag))) break;
            // every warp's d_x of chunk gc is visible (its phase cannot have
            // moved on: chunk gc + 2 is staged only after this warp signals below)
            if (!(ok = warp_wait(&b_full[gc & 1], (gc >> 1) & 1, abort_flag))) break;
            const float* sxc = sx + x3 * (SXB / 4);
            const uint8_t* nib = spn + rs * 128;
            const int r7 = rs & 7;
#pragma unroll
            for (int jj = hf; jj < KB; jj += 2) {
                // chunk gn's B buffer held chunk gc - 1, whose MMAs are complete
                // (the commit waited for before this block's load covers every earlier MMA)
                if (jj == 0 && has_next && warp < KB) stage_b(gn);
                if (actn) {
                    const uint4 w = lds128(nib + ((jj ^ r7) << 4));
                    uint32_t av[16];
                    weights_f16(w, av);
                    tmem_st16(tl + (uint32_t)(jj * 64), av);
                }
                if (jj + 2 >= KB && actn) sc_next = lds128(spn + H * 128 + rs * 16);
                if (act) {
                    tmem_wait_ld_regs(v);
                    const uint32_t sw = jj < 2 ? sc_cur.x : jj < 4 ? sc_cur.y : jj < 6 ? sc_cur.z : sc_cur.w;
                    const float dw = f16_bits_to_f32((unsigned short)(sw >> (16 * (jj & 1))));
                    const float2 dw2 = make_float2(dw, dw);
                    const float4* dx = reinterpret_cast<const float4*>(sxc + jj * NTOK);
#pragma unroll
                    for (int i = 0; i < NTOK / 4; ++i) {
                        if (i >= ngrp) break;  // warp-uniform: no tokens past M
                        const float4 d4 = dx[i];
                        acc[2 * i] = ffma2_scaled(dw2, make_float2(d4.x, d4.y),
                                                  make_float2(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1])),
                                                  acc[2 * i]);
                        acc[2 * i + 1] = ffma2_scaled(
                            dw2, make_float2(d4.z, d4.w),
                            make_float2(__uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3])), acc[2 * i + 1]);
                    }
                }
                if (actn) tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0 && has_next) {
                    mbar_arrive(&ready[jj]);
                    if (jj + 2 >= KB) mbar_arrive(&raw_empty[sn]);
                }
                // this warp's next block's dot slice: (gc, jj + 2), or its first of chunk gn
                const bool wrap = jj + 2 >= KB;
                if (!wrap || has_next) {
                    const int jn = wrap ? hf : jj + 2;
                    if (!(ok = warp_wait(&fullt[jn], (wrap ? gn : gc) & 1, abort_flag))) break;
                    tc_fence_after();
                    if (wrap ? actn : act) tmem_ld16(tl + (uint32_t)(jn * 64 + 16), v);
                }
            }
            if (!ok) break;
            sc_cur = sc_next;
            if (++sn == S) {
                sn = 0;
                pn ^= 1;
            }
            x3 = x3 == 2 ? 0 : x3 + 1;
            if (++c == nch) {
                // end of the super-tile: the odd-block warp of each row slice hands
                // its sums to the even-block warp (warp - 8), which writes the rows
                const int pair = warp & 7;
                if (hf == 1) {
                    if (st > 0 && !(ok = warp_wait(&red_empty[pair], (st - 1) & 1, abort_flag))) break;
#pragma unroll
                    for (int t = 0; t < NTOK / 2; ++t) reinterpret_cast<float2*>(red)[t] = acc[t];
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&red_full[pair]);
                } else {
                    if (!(ok = warp_wait(&red_full[pair], st & 1, abort_flag))) break;
                    const int64_t row = row_cta + (int64_t)st * H + rl;
#pragma unroll
                    for (int t = 0; t < NTOK / 2; ++t) {
                        const float2 o = reinterpret_cast<const float2*>(red)[t];
                        acc[t].x += o.x;
                        acc[t].y += o.y;
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&red_empty[pair]);
                    if (act && rl < H && row < a.N) {
#pragma unroll
                        for (int t = 0; t < NTOK / 2; ++t) {
                            if (2 * t < a.M) a.y[(int64_t)(2 * t) * a.ldy + row] = acc[t].x;
                            if (2 * t + 1 < a.M) a.y[(int64_t)(2 * t + 1) * a.ldy + row] = acc[t].y;
                        }
                    }
                }
#pragma unroll
                for (int t = 0; t < NTOK / 2; ++t) acc[t] = make_float2(0.f, 0.f);
                c = 0;
                ++st;
            }
            act = actn;
        }
        if (!ok && total > 0) {
            if (lane == 0) atomicOr(a.err, ERR_TIMEOUT);
            *abort_flag = 1;
        }
        tmem_wait_ld();  // no load of this warp still in flight when TMEM is freed
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == WARP_MMA)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
}

// ---------------------------------------------------------------- host side
std::mutex g_mu;
std::set<int> g_attr_devices;

bool allow_smem(int bytes) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_attr_devices.count(dev)) return true;
    if (cudaFuncSetAttribute(gemm_tmem_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    g_attr_devices.insert(dev);
    return true;
}

}  // namespace tmk

// Super-tile plan: one CTA per SM, each with nst super-tiles of H rows
// (H a multiple of 8, at most 256), as few super-tiles as that allows.
void gemm_tmem_plan(int64_t N, int sms, int* H, int* nst, int64_t* grid) {
    const int64_t need = (N + sms - 1) / sms;
    const int64_t n = (need + 255) / 256;
    const int64_t h = ((need + n - 1) / n + 7) / 8 * 8;
    *H = (int)h;
    *nst = (int)n;
    *grid = (N + n * h - 1) / (n * h);
}

bool gemm_tmem_eligible(int64_t N, int64_t K, int64_t M, const void* w_qs, const void* w_d, const void* xq,
                        const void* xd) {
    auto al = [](const void* p, uintptr_t n) { return reinterpret_cast<uintptr_t>(p) % n == 0; };
    return N >= 1 && N < (int64_t(1) << 31) && M >= 1 && M <= tmk::NTOK && K >= 256 && K % 256 == 0 &&
           K < (int64_t(1) << 31) && al(w_qs, 16) && al(w_d, 16) && al(xq, 16) && al(xd, 16);
}

qmm_status gemm_tmem_launch(const uint8_t* w_qs, const uint16_t* w_d, int64_t N, int64_t K, int64_t M,
                            const int8_t* xq, const uint16_t* xd, float* y, int64_t ldy, int sms, int smem_optin,
                            int* err, cudaStream_t st) {
    using namespace tmk;
    int H = 0, nst = 0;
    int64_t grid = 0;
    gemm_tmem_plan(N, sms, &H, &nst, &grid);
    const int64_t B = K / QK;
    Args a = {};
    a.N = N;
    a.K = K;
    a.M = M;
    a.ldy = ldy;
    a.y = y;
    a.H = H;
    a.nst = nst;
    a.stage_bytes = (H * 144 + XQ_BYTES + XD_BYTES + 1023) / 1024 * 1024;
    const int fixed = 2 * BBUF + 3 * SXB + RED_BYTES + 1024 + 1024;  // B buffers, d_x, sums, barriers, slack
    const int64_t chunks = (int64_t)nst * (K / (QK * KB));
    const int64_t ns = std::min<int64_t>({(int64_t)MAX_STAGES, (smem_optin - fixed) / a.stage_bytes, chunks});
    if (ns < 1 || grid > 0x7fffffff) return QMM_ERR_SHAPE;
    a.nstages = (int)ns;
    a.off_bbuf = (int)ns * a.stage_bytes;
    a.off_sx = a.off_bbuf + 2 * BBUF;
    a.off_red = a.off_sx + 3 * SXB;
    a.off_bar = a.off_red + RED_BYTES;
    a.err = err;
    const int smem = a.off_bar + 1024 + 1024;
    CUtensorMap mq, md, mxq, mxd;
    if (!make_tensor_map_2d(&mq, CU_TENSOR_MAP_DATA_TYPE_UINT8, w_qs, (uint64_t)K / 2, (uint64_t)N, (uint64_t)K / 2,
                            128, (uint32_t)H, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map_2d(&md, CU_TENSOR_MAP_DATA_TYPE_UINT16, w_d, (uint64_t)B, (uint64_t)N, (uint64_t)B * 2, KB,
                            (uint32_t)H, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_tensor_map_2d(&mxq, CU_TENSOR_MAP_DATA_TYPE_UINT8, xq, (uint64_t)K, (uint64_t)M, (uint64_t)K, KB * 32,
                            NTOK, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_tensor_map_2d(&mxd, CU_TENSOR_MAP_DATA_TYPE_UINT16, xd, (uint64_t)B, (uint64_t)M, (uint64_t)B * 2, KB,
                            NTOK, CU_TENSOR_MAP_SWIZZLE_NONE))
        return QMM_ERR_CUDA;
    if (smem > smem_optin || !allow_smem(smem_optin)) return QMM_ERR_SHAPE;
    gemm_tmem_kernel<<<dim3((unsigned)grid, 1), THREADS, smem, st>>>(mq, md, mxq, mxd, a);
    return cudaGetLastError() == cudaSuccess ? QMM_OK : QMM_ERR_CUDA;
}

}  // namespace qmm

