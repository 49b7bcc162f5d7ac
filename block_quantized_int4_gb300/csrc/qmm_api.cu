// qmm_api.cu -- the C ABI of libqmm (declared in include/qmm.h): argument
// validation on the host, launch configuration, error reporting.  Every
// entry enqueues work on the caller's stream and returns; nothing here
// allocates device memory or synchronises (except qmm_last_device_error).
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <set>
#include <utility>

#include "qmm.h"
#include "qmm_internal.h"
#include "qmm_kernels.cuh"
#include "qmm_stream.cuh"
#include "qmm_mma.h"
#include "qmm_tmap.h"

using namespace qmm;

// Device error word: bit ERR_BAD_EXPERT / ERR_TIMEOUT, or-ed by kernels.
static __device__ int g_err_word;

namespace {

constexpr int MAX_DEVICES = 64;

struct DevInfo {
    bool ready = false;
    bool ok = false;
    int sms = 0;
    int smem_optin = 0;
    int smem_per_sm = 0;
    int* err = nullptr;  // device address of g_err_word
};

std::mutex g_mu;
DevInfo g_dev[MAX_DEVICES];

// Small-batch GEMM kernel choice (qmm_debug_gemm_kernel), process-wide.
std::atomic<int> g_gemm_kernel{QMM_GEMM_KERNEL_AUTO};

// Bounded-wait test settings of the streaming kernel (qmm_debug_stream_wait).
std::atomic<unsigned long long> g_stream_wait_ns{WAIT_LIMIT_NS};
std::atomic<int> g_stream_withhold{0};

// Per-device facts, looked up once.  Requires an sm_103 device.
const DevInfo* device_info() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) {
        cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    DevInfo& d = g_dev[dev];
    if (!d.ready) {
        d.ready = true;
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
        void* p = nullptr;
        const bool sym = cudaGetSymbolAddress(&p, g_err_word) == cudaSuccess;
        d.err = static_cast<int*>(p);
        d.ok = (major == 10 && minor == 3) && sym && d.sms > 0;
        cudaGetLastError();
    }
    return d.ok ? &d : nullptr;
}

}  // namespace

int* qmm::device_error_word() {
    const DevInfo* d = device_info();
    return d ? d->err : nullptr;
}

bool qmm::device_facts(int* sms, int* smem_optin) {
    const DevInfo* d = device_info();
    if (!d) return false;
    *sms = d->sms;
    *smem_optin = d->smem_optin;
    return true;
}

namespace {

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline qmm_status launch_status() {
    return cudaGetLastError() == cudaSuccess ? QMM_OK : QMM_ERR_CUDA;
}

inline cudaStream_t S(void* s) { return static_cast<cudaStream_t>(s); }

// Opt a kernel into the device's full dynamic shared memory, once per
// (kernel, device); later calls are a lookup (safe during stream capture).
std::mutex g_attr_mu;
std::set<std::pair<const void*, int>> g_attr_done;

template <typename K>
bool smem_optin(K kernel, int bytes, int optin) {
    if (bytes <= 48 * 1024) return true;
    if (bytes > optin) return false;
    int dev = 0;
    cudaGetDevice(&dev);
    const auto key = std::make_pair(reinterpret_cast<const void*>(kernel), dev);
    std::lock_guard<std::mutex> lk(g_attr_mu);
    if (g_attr_done.count(key)) return true;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, optin) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    g_attr_done.insert(key);
    return true;
}

// Prefer the largest shared-memory carve-out for a kernel, once per (kernel,
// device): launches of one kernel with small and large shared-memory needs
// then share an SM configuration, so a chained launch's CTAs can become
// resident beside those of the launch before it instead of waiting for the
// SM to drain and be reconfigured.
std::set<std::pair<const void*, int>> g_carve_done;

template <typename K>
bool max_carveout(K kernel) {
    int dev = 0;
    cudaGetDevice(&dev);
    const auto key = std::make_pair(reinterpret_cast<const void*>(kernel), dev);
    std::lock_guard<std::mutex> lk(g_attr_mu);
    if (g_carve_done.count(key)) return true;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared) !=
        cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    g_carve_done.insert(key);
    return true;
}

int grid_for(int64_t work_items, int per_sm, int sms) {
    int64_t g = std::min<int64_t>(work_items, (int64_t)sms * per_sm);
    return (int)std::max<int64_t>(g, 1);
}

// Launch with or without programmatic dependent launch.
template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                   Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    if (pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Rows-kernel dispatch over the token-group width MT.
template <int MT, int XM>
qmm_status rows_launch(const DevInfo* di, RowsArgs a, bool pdl, cudaStream_t st) {
    const int64_t B = a.K / QK;
    const int per_block = xtile_bytes_per_block();
    // Stage all of K when it fits, else chunks of a multiple of 32 blocks.
    int64_t cap = (int64_t)std::min(di->smem_optin, 200 * 1024) / (MT * per_block);
    int64_t Bc = B <= cap ? B : std::max<int64_t>(32, cap / 32 * 32);
    if (XM != X_Q8 && Bc < B) return QMM_ERR_SHAPE;  // fp32 prologue needs the whole row on chip
    a.chunk_blocks = (int)Bc;
    const int smem = (int)(MT * Bc * per_block);
    auto kern = rows_kernel<MT, XM>;
    if (!smem_optin(kern, smem, di->smem_optin)) return QMM_ERR_SHAPE;
    const int64_t ntiles = (a.N + ROWS_WARPS - 1) / ROWS_WARPS;
    const int per_sm = std::max(1, std::min(8, (di->smem_optin / std::max(smem, 1))));
    dim3 grid(grid_for(ntiles, per_sm, di->sms), (unsigned)((a.M + MT - 1) / MT));
    cudaError_t e = launch(kern, grid, dim3(ROWS_THREADS), smem, st, pdl, a);
    return e == cudaSuccess ? launch_status() : (cudaGetLastError(), QMM_ERR_CUDA);
}

bool valid_k(int64_t K) { return K > 0 && K % QK == 0 && K <= (int64_t)1 << 30; }

// Streaming kernel: eligible when the scale plane can be bulk-copied in row
// segments (B % 8 == 0, i.e. K % 256 == 0; d 16-byte aligned) and the staged
// activation tile fits: up to 64 KB at two CTAs per SM; for two tokens up to
// 96 KB at one CTA per SM (a 220 KB ring: 8192 x 28672 at 2 tokens 35.8 ->
// 32.6 us against the row kernel, the batch-2 dense set 0.185 -> 0.181 ms).
constexpr int STREAM_XTILE_CAP = 64 * 1024;
constexpr int STREAM_XTILE_CAP_ONE_CTA = 96 * 1024;
constexpr int64_t CHAIN_MATRIX_BYTES = 16ll << 20;  // up to this, one CTA per SM and room for a neighbour CTA

bool stream_eligible(int64_t N, int64_t K, const void* qs, const void* d, int MT) {
    const int64_t B = K / QK;
    return (B % 8 == 0) && aligned(qs, 16) && aligned(d, 16) && N < (int64_t(1) << 31) &&
           (int64_t)MT * B * xtile_bytes_per_block() <= (MT == 2 ? STREAM_XTILE_CAP_ONE_CTA : STREAM_XTILE_CAP);
}

inline int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

template <int MT, int XM, int YM, bool QOUT>
qmm_status stream_launch(const DevInfo* di, const uint8_t* qs, const uint16_t* d, StreamArgs a, bool pdl,
                         cudaStream_t st) {
    const int64_t B = a.K / QK;
    const int64_t row_bytes = a.K / 2 + B * 2;
    const bool qout = XM == X_RUNTIME ? a.qout != 0 : QOUT;
    const int64_t opr = (YM == Y_RUNTIME ? a.ymode : YM) == Y_SWIGLU_PAIRS ? 2 : 1;
    // rows per CTA: even; with a Q8_0 output, whole blocks of 32 outputs
    const int64_t align = qout ? QK * opr : 2;
    // Large matrices: two CTAs per SM (more warps to hide latency); small
    // ones (decode chains): one per SM, leaving room for the next kernel.
#ifndef QMM_STREAM_BIG_CTAS_PER_SM
#define QMM_STREAM_BIG_CTAS_PER_SM 2
#endif
#ifndef QMM_STREAM_BIG_SMEM_KB
#define QMM_STREAM_BIG_SMEM_KB 110
#endif
    const bool chain_sized = a.N * row_bytes <= CHAIN_MATRIX_BYTES;
    // an activation tile above the two-CTA cap: one CTA per SM
    const bool one_cta = (int64_t)MT * B * xtile_bytes_per_block() > STREAM_XTILE_CAP;
    const int64_t ctas = chain_sized || one_cta ? di->sms : QMM_STREAM_BIG_CTAS_PER_SM * (int64_t)di->sms;
    // A CTA's weights arrive through its one producer lane, so in a decode
    // chain fewer bytes per CTA finish sooner: a Q8_0-output launch, a
    // one-token launch of the fused (chain) entries, and a one- or two-token
    // product of more than 4096 rows (the kernel fits two CTAs per SM up to
    // two tokens) take the smallest row count (whole 32-output blocks with a
    // Q8_0 output, else pairs) that keeps about two CTAs per SM at most
    // (TinyLLaMA gate/up: 176 CTAs of 64 rows instead of 88 of 128, the
    // decode step 462 -> 422 us; O and down: 256 CTAs of 8 rows instead of
    // 147 of 14, 0.361 -> 0.358 ms; 5632 x 2048 alone 4.80 -> 4.25 us at one
    // token, 5.75 -> 5.08 at two; but 2048-row products alone 1-3% slower:
    // 2048 x 2048 3.27 -> 3.30).  With 4 tokens the kernel holds one CTA per
    // SM, and twice the CTAs ran in two waves (2048 x 5632 7.1 -> 10.8 us).
    const bool two_per_sm = qout || (MT == 1 && XM == X_RUNTIME) || (MT <= 2 && a.N > 4096);
    const int64_t rpc = chain_sized && two_per_sm
                            ? std::max<int64_t>(align, round_up((a.N + 2 * ctas - 1) / (2 * ctas), align))
                            : round_up((a.N + ctas - 1) / ctas, align);
    const int64_t G = (a.N + rpc - 1) / rpc;
    const int rb = (int)std::min<int64_t>(GROUP_ROWS, rpc);
    const int ckb = (int)std::min<int64_t>(CHUNK_KB, B);
    const int64_t xtile = round_up((int64_t)MT * B * xtile_bytes_per_block(), 128);
    const int64_t ybuf = qout ? round_up(rpc / opr * 4, 128) : 0;
    const bool rpre = a.residual != nullptr && a.M == 1 && opr == 1;
    const int64_t rbuf = rpre ? round_up(rpc * 4, 128) : 0;
    const int64_t nunits = ((rpc + rb - 1) / rb) * ((B + ckb - 1) / ckb);
    // a ring stage holds one TMA box pair (rb rows x ckb blocks): sized to it,
    // so short row groups leave room for more stages
    const int64_t stage_q = round_up((int64_t)rb * ckb * 16, 128);
    const int64_t stage_bytes = stage_q + round_up((int64_t)rb * ckb * 2, 128);
    // Small matrices (decode chains): stay under ~112 KB so the next chained
    // kernel's CTA is resident beside this one and prefetches its weights
    // (two such CTAs and their 1 KB reservations fill the SM's 228 KB).
    const int64_t cap = chain_sized ? 112 * 1024 : one_cta ? 220 * 1024 : QMM_STREAM_BIG_SMEM_KB * 1024;
    const int64_t room = (cap - STREAM_HDR - xtile - ybuf - rbuf) / stage_bytes;
    const int64_t nst = std::min<int64_t>({nunits, room, (int64_t)STREAM_MAX_STAGES});
    if (nst < 1) return QMM_ERR_SHAPE;
    CUtensorMap mq, md;
    if (!make_tensor_map_2d(&mq, CU_TENSOR_MAP_DATA_TYPE_UINT32, qs, (uint64_t)a.K / 8, (uint64_t)a.N,
                            (uint64_t)a.K / 2, (uint32_t)ckb * 4, (uint32_t)rb, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_tensor_map_2d(&md, CU_TENSOR_MAP_DATA_TYPE_UINT16, d, (uint64_t)B, (uint64_t)a.N, (uint64_t)B * 2,
                            (uint32_t)ckb, (uint32_t)rb, CU_TENSOR_MAP_SWIZZLE_NONE))
        return QMM_ERR_CUDA;
    const int smem = (int)(STREAM_HDR + xtile + nst * stage_bytes + ybuf + rbuf);
    a.rows_per_cta = (int)rpc;
    a.ybuf_bytes = (int)ybuf;
    a.rbuf = rpre ? 1 : 0;
    a.stage_bytes = (int)stage_bytes;
    a.stage_q = (int)stage_q;
    a.rb = rb;
    a.ckb = ckb;
    a.nstages = (int)nst;
    a.xtile_bytes = (int)xtile;
    a.err = di->err;
    a.wait_ns = g_stream_wait_ns.load();
    a.withhold_last = g_stream_withhold.load();
    auto kern = stream_rows_kernel<MT, XM, YM, QOUT>;
    if (!smem_optin(kern, smem, di->smem_optin) || !max_carveout(kern)) return QMM_ERR_SHAPE;
    dim3 grid((unsigned)G, (unsigned)((a.M + MT - 1) / MT));
    cudaError_t e = launch(kern, grid, dim3(STREAM_THREADS), smem, st, pdl, mq, md, a);
    return e == cudaSuccess ? launch_status() : (cudaGetLastError(), QMM_ERR_CUDA);
}

// Batch-1 fused launch: one compiled kernel for every (input form, output
// form) combination, the forms passed at run time -- a decode chain runs one
// code image from launch to launch.
template <int XM>
qmm_status fused_dispatch(const DevInfo* di, const uint8_t* qs, const uint16_t* d, StreamArgs a, bool pairs, bool qout,
                          bool pdl, cudaStream_t st) {
    a.xmode = XM;
    a.ymode = pairs ? Y_SWIGLU_PAIRS : Y_PLAIN;
    a.qout = qout ? 1 : 0;
    return stream_launch<1, X_RUNTIME, Y_RUNTIME, false>(di, qs, d, a, pdl, st);
}

}  // namespace

// ============================================================================
extern "C" {

const char* qmm_status_string(int s) {
    switch (s) {
        case QMM_OK: return "QMM_OK";
        case QMM_ERR_ARG: return "QMM_ERR_ARG: null pointer or negative size";
        case QMM_ERR_SHAPE: return "QMM_ERR_SHAPE: K not a positive multiple of 32, empty, or too large";
        case QMM_ERR_ALIGN: return "QMM_ERR_ALIGN: pointer misaligned for the documented layout";
        case QMM_ERR_DEVICE: return "QMM_ERR_DEVICE: current device is not sm_103";
        case QMM_ERR_CUDA: return "QMM_ERR_CUDA: CUDA runtime call or launch failed";
        case QMM_ERR_TIMEOUT: return "QMM_ERR_TIMEOUT: a bounded device-side wait gave up";
        case QMM_ERR_BAD_EXPERT_ID: return "QMM_ERR_BAD_EXPERT_ID: expert id outside [0, E) skipped";
        case QMM_ERR_WORKSPACE: return "QMM_ERR_WORKSPACE: workspace missing or too small";
        case QMM_ERR_SCRATCH_LIMIT:
            return "QMM_ERR_SCRATCH_LIMIT: needs more than the fixed scratch (QMM_MOE_STATIC_SCRATCH_BYTES)";
        default: return "QMM_ERR_UNKNOWN";
    }
}

int qmm_abi_version(void) { return QMM_ABI_VERSION; }

qmm_status qmm_quantize_q4_0(const float* w, int64_t N, int64_t K, int64_t ldw, uint8_t* qs, uint16_t* d,
                             void* stream) {
    if (N < 0 || ldw < K) return QMM_ERR_ARG;
    if (!valid_k(K)) return QMM_ERR_SHAPE;
    if (N == 0) return QMM_OK;
    if (!w || !qs || !d) return QMM_ERR_ARG;
    if (!aligned(w, 16) || ldw % 4 || !aligned(qs, 16) || !aligned(d, 2)) return QMM_ERR_ALIGN;
    const DevInfo* di = device_info();
    if (!di) return QMM_ERR_DEVICE;
    const int64_t warps = (N * (K / QK) + 3) / 4;
    quantize_q4_0_kernel<<<grid_for((warps + 7) / 8, 16, di->sms), 256, 0, S(stream)>>>(w, N, K, ldw, qs, d);
    return launch_status();
}

qmm_status qmm_repack_q4_0(const uint8_t* blocks, int64_t N, int64_t K, uint8_t* qs, uint16_t* d, void* stream) {
    if (N < 0) return QMM_ERR_ARG;
    if (!valid_k(K)) return QMM_ERR_SHAPE;
    if (N == 0) return QMM_OK;
    if (!blocks || !qs || !d) return QMM_ERR_ARG;
    if (!aligned(qs, 16) || !aligned(d, 2)) return QMM_ERR_ALIGN;
    const DevInfo* di = device_info();
    if (!di) return QMM_ERR_DEVICE;
    const int64_t nblk = N * (K / QK);
    repack_q4_0_kernel<<<grid_for((nblk + 255) / 256, 16, di->sms), 256, 0, S(stream)>>>(blocks, nblk, qs, d);
    return launch_status();
}

qmm_status qmm_quantize_q8_0(const float* x, int64_t M, int64_t K, int64_t ldx, int8_t* q, uint16_t* d,
                             void* stream) {
    if (M < 0 || ldx < K) return QMM_ERR_ARG;
    if (!valid_k(K)) return QMM_ERR_SHAPE;
    if (M == 0) return QMM_OK;
    if (!x || !q || !d) return QMM_ERR_ARG;
    if (!aligned(x, 16) || ldx % 4 || !aligned(q, 16) || !aligned(d, 2)) return QMM_ERR_ALIGN;
    const DevInfo* di = device_info();
    if (!di) return QMM_ERR_DEVICE;
    const int64_t warps = (M * (K / QK) + 3) / 4;
    // programmatic dependent launch: the kernel waits for its predecessor
    const cudaError_t e = launch(quantize_q8_0_kernel, dim3(grid_for((warps + 7) / 8, 16, di->sms)), dim3(256), 0,
                                 S(stream), true, x, M, K, ldx, q, d);
    return e == cudaSuccess ? launch_status() : (cudaGetLastError(), QMM_ERR_CUDA);
}

qmm_status qmm_swiglu_quantize_q8_0(const float* gate, const float* up, int64_t rows, int64_t K, int64_t ld,
                                    int8_t* q, uint16_t* d, float* h_out, void* stream) {
    if (rows < 0 || ld < K) return QMM_ERR_ARG;
    if (!valid_k(K)) return QMM_ERR_SHAPE;
    if (rows == 0) return QMM_OK;
    if (!gate || !up || !q || !d) return QMM_ERR_ARG;
    if (!aligned(gate, 16) || !aligned(up, 16) || ld % 4 || !aligned(q, 16) || !aligned(d, 2) ||
        (h_out && !aligned(h_out, 16)))
        return QMM_ERR_ALIGN;
    const DevInfo* di = device_info();
    if (!di) return QMM_ERR_DEVICE;
    const int64_t warps = (rows * (K / QK) + 3) / 4;
    const cudaError_t e = launch(swiglu_quantize_kernel, dim3(grid_for((warps + 7) / 8, 16, di->sms)), dim3(256), 0,
                                 S(stream), true, gate, up, rows, K, ld, q, d, h_out);
    return e == cudaSuccess ? launch_status() : (cudaGetLastError(), QMM_ERR_CUDA);
}

qmm_status qmm_gemv_q4_0_q8_0(const uint8_t* w_qs, const uint16_t* w_d, int64_t N, int64_t K, const int8_t* xq,
                              const uint16_t* xd, float* y, void* stream) {
    return qmm_gemm_q4_0_q8_0(w_qs, w_d, N, K, 1, xq, xd, y, N, stream);
}

qmm_status qmm_gemv_q4_0_f32(const uint8_t* w_qs, const uint16_t* w_d, int64_t N, int64_t K, const float* x,
                             const float* residual, float* y, int8_t* xq_out, uint16_t* xd_out, int flags,
                             void* stream) {
    if (N < 0 || (flags & ~(QMM_X_SWIGLU | QMM_Y_SWIGLU_PAIRS | QMM_CHAIN))) return QMM_ERR_ARG;
    if (!valid_k(K) || N == 0 || K > 40960) return QMM_ERR_SHAPE;
    if (!w_qs || !w_d || !x || !y) return QMM_ERR_ARG;
    const bool xs = flags & QMM_X_SWIGLU, ys = flags & QMM_Y_SWIGLU_PAIRS, pdl = flags & QMM_CHAIN;
    if (ys && (N % 2 || residual)) return QMM_ERR_ARG;
    if (!aligned(w_qs, 16) || !aligned(w_d, 2) || !aligned(x, 16) || !aligned(y, 4) ||
        (residual && !aligned(residual, 4)) || (xq_out && !aligned(xq_out, 16)) || (xd_out && !aligned(xd_out, 2)))
        return QMM_ERR_ALIGN;
    const DevInfo* di = device_info();
    if (!di) return QMM_ERR_DEVICE;
    cudaStream_t st = S(stream);
    if (stream_eligible(N, K, w_qs, w_d, 1)) {
        StreamArgs a = {};
        a.N = N;
        a.K = K;
        a.M = 1;
        a.xf = x;
        a.residual = residual;
        a.xq_out = xq_out;
        a.xd_out = xd_out;
        a.y = y;
        a.ldy = ys ? N / 2 : N;
        return xs ? fused_dispatch<X_SWIGLU>(di, w_qs, w_d, a, ys, false, pdl, st)
                  : fused_dispatch<X_F32>(di, w_qs, w_d, a, ys, false, pdl, st);
    }
    if (ys) return QMM_ERR_SHAPE;  // paired rows need the streaming kernel (K % 256 == 0, d 16-byte aligned)
    RowsArgs a = {};
    a.qs = w_qs;
    a.d = w_d;
    a.N = N;
    a.K = K;
    a.M = 1;
    a.xf = x;
    a.residual = residual;
    a.xq_out = xq_out;
    a.xd_out = xd_out;
    a.y = y;
    a.ldy = N;
    return xs ? rows_launch<1, X_SWIGLU>(di, a, pdl, st) : rows_launch<1, X_F32>(di, a, pdl, st);
}

qmm_status qmm_gemv_fused(const uint8_t* w_qs, const uint16_t* w_d, int64_t N, int64_t K, const float* x,
                          const int8_t* xq, const uint16_t* xd, const float* residual, float* y, int8_t* yq,
                          uint16_t* yd, int flags, void* stream) {
    if (N < 0 || (flags & ~(QMM_X_SWIGLU | QMM_Y_SWIGLU_PAIRS | QMM_CHAIN))) return QMM_ERR_ARG;
    if (!valid_k(K) || N == 0 || K > 40960) return QMM_ERR_SHAPE;
    const bool xs = flags & QMM_X_SWIGLU, ys = flags & QMM_Y_SWIGLU_PAIRS, pdl = flags & QMM_CHAIN;
    const bool qout = yq != nullptr || yd != nullptr;
    if (!w_qs || !w_d || (!x && (!xq || !xd)) || (!y && !qout) || (qout && (!yq || !yd))) return QMM_ERR_ARG;
    if (xs && !x) return QMM_ERR_ARG;
    if (ys && (N % 2 || residual)) return QMM_ERR_ARG;
    const int64_t nout = ys ? N / 2 : N;
    if (qout && nout % QK) return QMM_ERR_SHAPE;
    if (!aligned(w_qs, 16) || !aligned(w_d, 16) || (x && !aligned(x, 16)) || (xq && !aligned(xq, 16)) ||
        (xd && !aligned(xd, 2)) || (y && !aligned(y, 4)) || (residual && !aligned(residual, 4)) ||
        (yq && !aligned(yq, 16)) || (yd && !aligned(yd, 2)))
        return QMM_ERR_ALIGN;
    if (!stream_eligible(N, K, w_qs, w_d, 1)) return QMM_ERR_SHAPE;
    const DevInfo* di = device_info();
    if (!di) return QMM_ERR_DEVICE;
    StreamArgs a = {};
    a.N = N;
    a.K = K;
    a.M = 1;
    a.xf = x;
    a.xq = xq;
    a.xd = xd;
    a.residual = residual;
    a.y = y;
    a.ldy = nout;
    a.yq = yq;
    a.yd = yd;
    cudaStream_t st = S(stream);
    if (x) return xs ? fused_dispatch<X_SWIGLU>(di, w_qs, w_d, a, ys, qout, pdl, st)
                     : fused_dispatch<X_F32>(di, w_qs, w_d, a, ys, qout, pdl, st);
    return fused_dispatch<X_Q8>(di, w_qs, w_d, a, ys, qout, pdl, st);
}

qmm_status qmm_gemm_q4_0_q8_0(const uint8_t* w_qs, const uint16_t* w_d, int64_t N, int64_t K, int64_t M,
                              const int8_t* xq, const uint16_t* xd, float* y, int64_t ldy, void* stream) {
    if (N < 0 || M < 0 || ldy < N) return QMM_ERR_ARG;
    if (!valid_k(K) || N == 0 || M == 0 || M > 65535 * 8) return QMM_ERR_SHAPE;
    if (!w_qs || !w_d || !xq || !xd || !y) return QMM_ERR_ARG;
    if (!aligned(w_qs, 16) || !aligned(w_d, 2) || !aligned(xq, 16) || !aligned(xd, 2) || !aligned(y, 4))
        return QMM_ERR_ALIGN;
    const DevInfo* di = device_info();
    if (!di) return QMM_ERR_DEVICE;
    RowsArgs a = {};
    a.qs = w_qs;
    a.d = w_d;
    a.N = N;
    a.K = K;
    a.M = M;
    a.xq = xq;
    a.xd = xd;
    a.y = y;
    a.ldy = ldy;
    cudaStream_t st = S(stream);
    // Two or more tokens: mostly a tensor-core kernel (exact fp16 products,
    // fp32 block sums).  By default the warp-MMA kernel, which streams the
    // weights once per 64 tokens; the tcgen05 kernel (weight operand in
    // tensor memory, up to 16 tokens) when selected, which measures slower
    // at every shape (its per-block TMEM read-back and rescale cost as much
    // as the warp kernel's register path, on top of the tensor core's fixed
    // cost per instruction).
    if (M >= 2 && ldy >= N) {
        const int pick = g_gemm_kernel.load();
        if (pick == QMM_GEMM_KERNEL_TMEM) {
            if (!gemm_tmem_eligible(N, K, M, w_qs, w_d, xq, xd)) return QMM_ERR_SHAPE;
            return gemm_tmem_launch(w_qs, w_d, N, K, M, xq, xd, y, ldy, di->sms, di->smem_optin, di->err, st);
        }
        // 2..4 tokens: the batch-1 GEMV's streaming path (its row-kernel
        // fallback where the activation tile does not fit), where it measured
        // faster than warp MMA (x = stream / MMA, us): 2 tokens on every
        // shape (28672x8192 23.2/31.9 against the 16-warp layout, 8192x28672
        // 32.6 at one CTA per SM, where the 16-warp layout splitting K over
        // clusters takes 37.0 at 4 tokens, 2048x5632 6.0/8.0, 2560x2048 4.0/5.0,
        // 5632x2048 5.7/5.7); 3-4 tokens when N <= 4096 or K >= 8192, the
        // activation tile fits and the 16-warp layout does not apply
        // (2048x5632 7.0/8.1, 2560x2048 4.4/4.9; but 5632x2048 6.4/5.6, and
        // 28672x8192 41.7 against 31.9 for the 16-warp layout).  From 8
        // tokens warp MMA wins everywhere.
        const bool wide = pick != QMM_GEMM_KERNEL_MMA_GROUPS && gemm_wide_planned(N, K, M, xd, di->sms);
        const bool prefer_stream =
            pick == QMM_GEMM_KERNEL_AUTO &&
            (M == 2 || (M <= 4 && !wide && (N <= 4096 || K >= 8192) && stream_eligible(N, K, w_qs, w_d, 4)));
        if (pick != QMM_GEMM_KERNEL_STREAM && !prefer_stream && gemm_mma_eligible(N, K, M, w_qs, w_d, xq, xd))
            return gemm_mma_launch(w_qs, w_d, N, K, M, xq, xd, y, ldy, di->sms, di->smem_optin, di->err, st, wide);
    }
    const int mt = M == 1 ? 1 : M == 2 ? 2 : M <= 4 ? 4 : 8;
    const bool streamable = stream_eligible(N, K, w_qs, w_d, mt);
    if (streamable) {
        StreamArgs s = {};
        s.N = N;
        s.K = K;
        s.M = M;
        s.xq = xq;
        s.xd = xd;
        s.y = y;
        s.ldy = ldy;
        switch (mt) {
            case 1: return stream_launch<1, X_Q8, Y_PLAIN, false>(di, w_qs, w_d, s, false, st);
            case 2: return stream_launch<2, X_Q8, Y_PLAIN, false>(di, w_qs, w_d, s, false, st);
            case 4: return stream_launch<4, X_Q8, Y_PLAIN, false>(di, w_qs, w_d, s, false, st);
            default: return stream_launch<8, X_Q8, Y_PLAIN, false>(di, w_qs, w_d, s, false, st);
        }
    }
    if (M == 1) return rows_launch<1, X_Q8>(di, a, false, st);
    if (M == 2) return rows_launch<2, X_Q8>(di, a, false, st);
    if (M <= 4) return rows_launch<4, X_Q8>(di, a, false, st);
    return rows_launch<8, X_Q8>(di, a, false, st);
}

qmm_status qmm_gemm_workspace_size(int64_t K, int64_t M, size_t* bytes) {
    if (!bytes || M < 0) return QMM_ERR_ARG;
    if (!valid_k(K)) return QMM_ERR_SHAPE;
    *bytes = gemm_prep_bytes(K, M);
    return QMM_OK;
}

qmm_status qmm_gemm_q4_0_q8_0_ws(const uint8_t* w_qs, const uint16_t* w_d, int64_t N, int64_t K, int64_t M,
                                 const int8_t* xq, const uint16_t* xd, float* y, int64_t ldy, void* workspace,
                                 size_t workspace_bytes, void* stream) {
    // qmm_gemm_q4_0_q8_0's checks, in its order, then the workspace's
    if (N < 0 || M < 0 || ldy < N) return QMM_ERR_ARG;
    if (!valid_k(K) || N == 0 || M == 0 || M > 65535 * 8) return QMM_ERR_SHAPE;
    if (!w_qs || !w_d || !xq || !xd || !y) return QMM_ERR_ARG;
    if (!aligned(w_qs, 16) || !aligned(w_d, 2) || !aligned(xq, 16) || !aligned(xd, 2) || !aligned(y, 4))
        return QMM_ERR_ALIGN;
    const size_t need = gemm_prep_bytes(K, M);
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned(workspace, 128))) return QMM_ERR_WORKSPACE;
    const DevInfo* di = device_info();
    if (!di) return QMM_ERR_DEVICE;
    // The prepared path where qmm_gemm_q4_0_q8_0 would take the 16-warp
    // layout (same kernel choice, same results bit for bit); elsewhere the
    // workspace is not used.
    const int pick = g_gemm_kernel.load();
    if (need > 0 && M >= 3 && (pick == QMM_GEMM_KERNEL_AUTO || pick == QMM_GEMM_KERNEL_MMA) && aligned(xd, 16) &&
        gemm_mma_eligible(N, K, M, w_qs, w_d, xq, xd)) {
        const WidePlan p = gemm_wide_plan(N, K, M, di->sms, false);
        if (p.rpc > 0)
            return gemm_prep_launch(w_qs, w_d, N, K, M, xq, xd, y, ldy, p, workspace, di->smem_optin, di->err,
                                    S(stream));
    }
    return qmm_gemm_q4_0_q8_0(w_qs, w_d, N, K, M, xq, xd, y, ldy, stream);
}

}  // extern "C"

namespace {

// Host checks of one qmm_gemv_op.
qmm_status validate_op(const qmm_gemv_op& o) {
    if (o.N <= 0 || (o.flags & ~QMM_Y_SWIGLU_PAIRS)) return QMM_ERR_ARG;
    if (!valid_k(o.K) || o.K % 256 != 0 || o.K > 40960 || o.N >= (int64_t(1) << 31)) return QMM_ERR_SHAPE;
    const bool pairs = o.flags & QMM_Y_SWIGLU_PAIRS;
    const bool qout = o.yq != nullptr || o.yd != nullptr;
    if (!o.w_qs || !o.w_d || (!o.x && (!o.xq || !o.xd)) || (!o.y && !qout) || (qout && (!o.yq || !o.yd)))
        return QMM_ERR_ARG;
    if (o.x && (o.xq == nullptr) != (o.xd == nullptr)) return QMM_ERR_ARG;
    if (o.norm_w && (!o.x || !(o.norm_eps >= 0.0f))) return QMM_ERR_ARG;
    if (pairs && (o.N % 2 || o.residual)) return QMM_ERR_ARG;
    const int64_t nout = pairs ? o.N / 2 : o.N;
    if (qout && nout % QK) return QMM_ERR_SHAPE;
    if (!aligned(o.w_qs, 16) || !aligned(o.w_d, 16) || (o.x && !aligned(o.x, 16)) ||
        (o.norm_w && !aligned(o.norm_w, 16)) || (o.xq && !aligned(o.xq, 16)) || (o.xd && !aligned(o.xd, 2)) ||
        (o.y && !aligned(o.y, 4)) || (o.residual && !aligned(o.residual, 4)) || (o.yq && !aligned(o.yq, 16)) ||
        (o.yd && !aligned(o.yd, 2)))
        return QMM_ERR_ALIGN;
    return QMM_OK;
}

// One checked op as one launch of the streaming kernel.
qmm_status launch_op(const qmm_gemv_op& o, int flags, const DevInfo* di, void* stream) {
    const bool pairs = o.flags & QMM_Y_SWIGLU_PAIRS, qout = o.yq != nullptr;
    StreamArgs a = {};
    a.N = o.N;
    a.K = o.K;
    a.M = 1;
    a.xf = o.x;
    a.gamma = o.x ? o.norm_w : nullptr;
    a.eps = o.norm_eps;
    if (o.x) {
        a.xq_out = const_cast<int8_t*>(o.xq);
        a.xd_out = const_cast<uint16_t*>(o.xd);
    } else {
        a.xq = o.xq;
        a.xd = o.xd;
    }
    a.residual = o.residual;
    a.y = o.y;
    a.ldy = pairs ? o.N / 2 : o.N;
    a.yq = o.yq;
    a.yd = o.yd;
    const bool pdl = flags & QMM_CHAIN;
    cudaStream_t st = S(stream);
    return o.x ? fused_dispatch<X_F32>(di, o.w_qs, o.w_d, a, pairs, qout, pdl, st)
               : fused_dispatch<X_Q8>(di, o.w_qs, o.w_d, a, pairs, qout, pdl, st);
}

}  // namespace

extern "C" {

qmm_status qmm_gemv_fused_op(const qmm_gemv_op* op, int flags, void* stream) {
    if (!op || (flags & ~QMM_CHAIN)) return QMM_ERR_ARG;
    const qmm_status v = validate_op(*op);
    if (v != QMM_OK) return v;
    const DevInfo* di = device_info();
    if (!di) return QMM_ERR_DEVICE;
    return launch_op(*op, flags, di, stream);
}

qmm_status qmm_gemv_fused_ops(const qmm_gemv_op* ops, int32_t n, int flags, void* stream) {
    if (n < 0 || (n > 0 && !ops) || (flags & ~QMM_CHAIN)) return QMM_ERR_ARG;
    for (int32_t i = 0; i < n; ++i) {
        const qmm_status v = validate_op(ops[i]);
        if (v != QMM_OK) return v;
    }
    if (n == 0) return QMM_OK;
    const DevInfo* di = device_info();
    if (!di) return QMM_ERR_DEVICE;
    for (int32_t i = 0; i < n; ++i) {
        const qmm_status s = launch_op(ops[i], flags, di, stream);
        if (s != QMM_OK) return s;
    }
    return QMM_OK;
}

qmm_status qmm_debug_gemm_kernel(int kernel, int* previous) {
    if (kernel < QMM_GEMM_KERNEL_AUTO || kernel > QMM_GEMM_KERNEL_MMA_GROUPS) return QMM_ERR_ARG;
    const int old = g_gemm_kernel.exchange(kernel);
    if (previous) *previous = old;
    return QMM_OK;
}

qmm_status qmm_debug_stream_wait(uint64_t limit_ns, int withhold_last_copy, uint64_t* previous_limit_ns) {
    if (limit_ns < 1000ull || limit_ns > 10000000000ull || (withhold_last_copy != 0 && withhold_last_copy != 1))
        return QMM_ERR_ARG;
    const unsigned long long old = g_stream_wait_ns.exchange(limit_ns);
    g_stream_withhold.store(withhold_last_copy);
    if (previous_limit_ns) *previous_limit_ns = old;
    return QMM_OK;
}

qmm_status qmm_debug_block_dots(const uint8_t* w_qs, int64_t N, int64_t K, int64_t M, const int8_t* xq,
                                int32_t* dots, void* stream) {
    if (N < 0 || M < 0) return QMM_ERR_ARG;
    if (!valid_k(K) || N == 0 || M == 0) return QMM_ERR_SHAPE;
    if (!w_qs || !xq || !dots) return QMM_ERR_ARG;
    if (!aligned(w_qs, 16) || !aligned(xq, 16) || !aligned(dots, 4)) return QMM_ERR_ALIGN;
    const DevInfo* di = device_info();
    if (!di) return QMM_ERR_DEVICE;
    const int64_t total = M * N * (K / QK);
    block_dots_kernel<<<grid_for((total + 255) / 256, 16, di->sms), 256, 0, S(stream)>>>(w_qs, N, K, M, xq, dots);
    return launch_status();
}

qmm_status qmm_moe_workspace_size(int32_t E, int32_t T, int32_t k, size_t* bytes) {
    if (!bytes || E <= 0 || T < 0 || k <= 0) return QMM_ERR_ARG;
    *bytes = moe_ws_bytes(E, (int64_t)T * k);
    return QMM_OK;
}

}  // extern "C"

namespace {

// Argument checks shared by qmm_moe_gemv and qmm_moe_gemv_pregrouped (ids
// is checked by the former only).
qmm_status moe_check(const uint8_t* w_qs, const uint16_t* w_d, int32_t E, int64_t N, int64_t K, int32_t T, int32_t k,
                     const int8_t* xq, const uint16_t* xd, float* y, void* workspace, size_t workspace_bytes) {
    if (E <= 0 || N <= 0 || T < 0 || k <= 0) return QMM_ERR_ARG;
    if (!valid_k(K) || (int64_t)T * k > (1 << 24)) return QMM_ERR_SHAPE;
    if (T == 0) return QMM_OK;
    if (!w_qs || !w_d || !xq || !xd || !y) return QMM_ERR_ARG;
    if (!workspace || workspace_bytes < moe_ws_bytes(E, (int64_t)T * k)) return QMM_ERR_WORKSPACE;
    if (!aligned(w_qs, 16) || !aligned(w_d, 2) || !aligned(xq, 16) || !aligned(xd, 2) || !aligned(y, 4) ||
        !aligned(workspace, 16))
        return QMM_ERR_ALIGN;
    return QMM_OK;
}

// Whether the streaming expert GEMV takes this expert tensor (the fp32 and
// SwiGLU-pair forms require it).
bool moe_streamable(const uint8_t* w_qs, const uint16_t* w_d, int32_t E, int64_t N, int64_t K) {
    const int64_t B = K / QK;
    return (B % 8 == 0) && aligned(w_qs, 16) && aligned(w_d, 16) && (int64_t)E * N < (int64_t(1) << 31) &&
           E <= 2048 && 4 * B * xtile_bytes_per_block() <= STREAM_XTILE_CAP;
}

// Ring stages of the streaming expert GEMV (0: it does not fit), and the
// sizes that decide them: slots per weight pass, activation tile, tables.
struct MoeStreamSizes {
    int mt;
    int64_t xtile, tables, nst;
};
MoeStreamSizes moe_stream_sizes(int32_t E, int64_t K, int64_t nslots) {
    MoeStreamSizes z;
    const int64_t B = K / QK;
    // Slots per weight pass: four once slots outnumber a quarter of the
    // experts (experts with several slots are then common, and each pass
    // streams the expert's weights once), else one.  Measured on the
    // GLM-scale layer, top-8 of 256: 16 tokens 0.518 ms with four per pass,
    // 0.552 with two, 0.665 with one; 1 token fastest with one.
    z.mt = nslots * 4 > (int64_t)E ? 4 : 1;
    z.xtile = round_up((int64_t)z.mt * B * xtile_bytes_per_block(), 128);
    // routing tables in shared memory: active list and slot starts (E each),
    // the slot list when short, count and end
    z.tables = round_up((int64_t)E * 8 + (nslots <= MOE_SMEM_SLOTS ? nslots * 4 : 0) + 8, 128);
    // two CTAs per SM (110 KB each): more warps to hide the dot-product latency
    z.nst = std::max<int64_t>(
        0, std::min<int64_t>((110 * 1024 - STREAM_HDR - z.xtile - z.tables) / STAGE_BYTES, STREAM_MAX_STAGES));
    return z;
}

// Launch chaining of moe_apply (MoeStreamArgs late_trigger / tables_ready).
constexpr int CHAIN_LATE_TRIGGER = 1, CHAIN_TABLES_READY = 2;

// The expert GEMV on routing tables already built in the workspace.
// pairs: rows 2i, 2i + 1 of each expert are a (gate, up) pair and y gets
// SwiGLU of each pair ([T*k][N/2]); xf: fp32 activation rows quantized while
// staging, in place of xq/xd.  Both on the streaming kernel only.  chain:
// CHAIN_* bits, only for launches whose order on the stream the caller
// fixes (qmm_moe_layer_f32).
qmm_status moe_apply(const DevInfo* di, const uint8_t* w_qs, const uint16_t* w_d, int32_t E, int64_t N, int64_t K,
                     int32_t T, int32_t k, const int8_t* xq, const uint16_t* xd, int x_per_slot, float* y,
                     MoeWs ws, cudaStream_t st, bool pairs = false, const float* xf = nullptr, int chain = 0) {
    const int64_t B = K / QK;
    const int64_t nslots = (int64_t)T * k;
    const bool streamable = moe_streamable(w_qs, w_d, E, N, K);
    if (streamable) {
        MoeStreamArgs m = {};
        m.N = N;
        m.K = K;
        m.E = E;
        m.k = k;
        m.xq = xq;
        m.xd = xd;
        m.xf = xf;
        m.x_per_slot = x_per_slot;
        m.nslots = (int)nslots;
        m.slots_smem = nslots <= MOE_SMEM_SLOTS ? 1 : 0;
        m.y = y;
        m.pairs = pairs ? 1 : 0;
        m.ws = ws;
        m.rb = GROUP_ROWS;
        m.ckb = (int)std::min<int64_t>(CHUNK_KB, B);
        m.err = di->err;
        m.late_trigger = (chain & CHAIN_LATE_TRIGGER) ? 1 : 0;
        m.tables_ready = (chain & CHAIN_TABLES_READY) ? 1 : 0;
        const MoeStreamSizes z = moe_stream_sizes(E, K, nslots);
        const int mt = z.mt;
        const int64_t xtile = z.xtile, tables = z.tables, nst = z.nst;
        if (nst < 1) return QMM_ERR_SHAPE;
        m.nstages = (int)nst;
        m.xtile_bytes = (int)xtile;
        const int smem = (int)(STREAM_HDR + xtile + nst * STAGE_BYTES + tables);
        CUtensorMap mq, md;
        if (!make_tensor_map_2d(&mq, CU_TENSOR_MAP_DATA_TYPE_UINT32, w_qs, (uint64_t)K / 8, (uint64_t)E * N,
                                (uint64_t)K / 2, (uint32_t)m.ckb * 4, GROUP_ROWS, CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !make_tensor_map_2d(&md, CU_TENSOR_MAP_DATA_TYPE_UINT16, w_d, (uint64_t)B, (uint64_t)E * N,
                                (uint64_t)B * 2, (uint32_t)m.ckb, GROUP_ROWS, CU_TENSOR_MAP_SWIZZLE_NONE))
            return QMM_ERR_CUDA;
        // With one slot per pass (few routed slots), programmatic dependent
        // launch: the kernel's CTAs start while its predecessor finishes and
        // read the routing tables and activations once it has completed
        // (GLM-scale layer, 1 token: 51.6 -> 50.2 us).  With four slots per
        // pass it measured slower (16 tokens: 0.468 -> 0.509 ms), so those
        // launches wait for the predecessor as usual.
        cudaError_t e;
        dim3 grid(2 * di->sms);
        if (mt == 4) {
            if (!smem_optin(moe_stream_kernel<4>, smem, di->smem_optin)) return QMM_ERR_SHAPE;
            e = launch(moe_stream_kernel<4>, grid, dim3(STREAM_THREADS), smem, st, false, mq, md, m);
        } else {
            if (!smem_optin(moe_stream_kernel<1>, smem, di->smem_optin)) return QMM_ERR_SHAPE;
            e = launch(moe_stream_kernel<1>, grid, dim3(STREAM_THREADS), smem, st, true, mq, md, m);
        }
        return e == cudaSuccess ? launch_status() : (cudaGetLastError(), QMM_ERR_CUDA);
    }

    if (pairs || xf || chain) return QMM_ERR_SHAPE;  // the fallback: plain rows of Q8_0 activations only
    MoeArgs a = {};
    a.qs = w_qs;
    a.d = w_d;
    a.N = N;
    a.K = K;
    a.E = E;
    a.k = k;
    a.xq = xq;
    a.xd = xd;
    a.x_per_slot = x_per_slot;
    a.y = y;
    a.ws = ws;
    a.rows_per_item = 8 * ROWS_WARPS;
    const int per_block = xtile_bytes_per_block();
    const int64_t cap = std::min(di->smem_optin, 200 * 1024);
    // Token-group width: widest that stages the whole K.
    int mt = 8;
    while (mt > 1 && (int64_t)mt * B * per_block > cap) mt /= 2;
    if ((int64_t)mt * B * per_block > cap) return QMM_ERR_SHAPE;
    // Tokens per expert on average decides how wide a group is useful.
    const int64_t max_slots = std::min<int64_t>(nslots, 8);
    while (mt > 1 && mt / 2 >= max_slots) mt /= 2;
    const int smem = (int)(mt * B * per_block);
    const int64_t row_blocks = (N + a.rows_per_item - 1) / a.rows_per_item;
    const int64_t max_items = std::min<int64_t>(E, nslots) * row_blocks;
    const int per_sm = std::max(1, std::min(4, di->smem_optin / std::max(smem, 1)));
    dim3 grid(grid_for(max_items, per_sm, di->sms));
    cudaError_t e;
    switch (mt) {
        case 8:
            if (!smem_optin(moe_rows_kernel<8>, smem, di->smem_optin)) return QMM_ERR_SHAPE;
            e = launch(moe_rows_kernel<8>, grid, dim3(ROWS_THREADS), smem, st, false, a);
            break;
        case 4:
            if (!smem_optin(moe_rows_kernel<4>, smem, di->smem_optin)) return QMM_ERR_SHAPE;
            e = launch(moe_rows_kernel<4>, grid, dim3(ROWS_THREADS), smem, st, false, a);
            break;
        case 2:
            if (!smem_optin(moe_rows_kernel<2>, smem, di->smem_optin)) return QMM_ERR_SHAPE;
            e = launch(moe_rows_kernel<2>, grid, dim3(ROWS_THREADS), smem, st, false, a);
            break;
        default:
            if (!smem_optin(moe_rows_kernel<1>, smem, di->smem_optin)) return QMM_ERR_SHAPE;
            e = launch(moe_rows_kernel<1>, grid, dim3(ROWS_THREADS), smem, st, false, a);
            break;
    }
    return e == cudaSuccess ? launch_status() : (cudaGetLastError(), QMM_ERR_CUDA);
}

}  // namespace

extern "C" {

qmm_status qmm_moe_gemv(const uint8_t* w_qs, const uint16_t* w_d, int32_t E, int64_t N, int64_t K, const int32_t* ids,
                        int32_t T, int32_t k, const int8_t* xq, const uint16_t* xd, int x_per_slot, float* y,
                        void* workspace, size_t workspace_bytes, void* stream) {
    qmm_status s = moe_check(w_qs, w_d, E, N, K, T, k, xq, xd, y, workspace, workspace_bytes);
    if (s != QMM_OK || T == 0) return s;
    if (!ids) return QMM_ERR_ARG;
    if (!aligned(ids, 4)) return QMM_ERR_ALIGN;
    const DevInfo* di = device_info();
    if (!di) return QMM_ERR_DEVICE;
    cudaStream_t st = S(stream);
    MoeWs ws = moe_ws(workspace, E);
    if (launch(moe_group_kernel, dim3(1), dim3(GROUP_THREADS), 0, st, true, ids, T * k, E, ws, di->err) !=
        cudaSuccess) {
        cudaGetLastError();
        return QMM_ERR_CUDA;
    }
    s = launch_status();
    if (s != QMM_OK) return s;
    return moe_apply(di, w_qs, w_d, E, N, K, T, k, xq, xd, x_per_slot, y, ws, st);
}

qmm_status qmm_moe_group_ids(const int32_t* ids, int32_t T, int32_t k, int32_t E, void* workspace,
                             size_t workspace_bytes, void* stream) {
    if (E <= 0 || T < 0 || k <= 0) return QMM_ERR_ARG;
    if ((int64_t)T * k > (1 << 24)) return QMM_ERR_SHAPE;
    if (T == 0) return QMM_OK;
    if (!ids || !workspace) return QMM_ERR_ARG;
    if (workspace_bytes < moe_ws_bytes(E, (int64_t)T * k)) return QMM_ERR_WORKSPACE;
    if (!aligned(ids, 4) || !aligned(workspace, 16)) return QMM_ERR_ALIGN;
    const DevInfo* di = device_info();
    if (!di) return QMM_ERR_DEVICE;
    if (launch(moe_group_kernel, dim3(1), dim3(GROUP_THREADS), 0, S(stream), true, ids, T * k, E,
               moe_ws(workspace, E), di->err) != cudaSuccess) {
        cudaGetLastError();
        return QMM_ERR_CUDA;
    }
    return launch_status();
}

qmm_status qmm_moe_gemv_pregrouped(const uint8_t* w_qs, const uint16_t* w_d, int32_t E, int64_t N, int64_t K,
                                   int32_t T, int32_t k, const int8_t* xq, const uint16_t* xd, int x_per_slot,
                                   float* y, const void* workspace, size_t workspace_bytes, void* stream) {
    void* wsp = const_cast<void*>(workspace);
    qmm_status s = moe_check(w_qs, w_d, E, N, K, T, k, xq, xd, y, wsp, workspace_bytes);
    if (s != QMM_OK || T == 0) return s;
    const DevInfo* di = device_info();
    if (!di) return QMM_ERR_DEVICE;
    return moe_apply(di, w_qs, w_d, E, N, K, T, k, xq, xd, x_per_slot, y, moe_ws(wsp, E), S(stream));
}

qmm_status qmm_moe_gemv_gate_up(const uint8_t* w_qs, const uint16_t* w_d, int32_t E, int64_t N, int64_t K, int32_t T,
                                int32_t k, const float* x, const int8_t* xq, const uint16_t* xd, int x_per_slot,
                                float* h, const void* workspace, size_t workspace_bytes, void* stream) {
    void* wsp = const_cast<void*>(workspace);
    // with an fp32 x the Q8_0 planes are not read: check x in their place
    const int8_t* cq = x ? reinterpret_cast<const int8_t*>(x) : xq;
    const uint16_t* cd = x ? reinterpret_cast<const uint16_t*>(x) : xd;
    qmm_status s = moe_check(w_qs, w_d, E, N, K, T, k, cq, cd, h, wsp, workspace_bytes);
    if (s != QMM_OK || T == 0) return s;
    if (N % 2) return QMM_ERR_SHAPE;
    const DevInfo* di = device_info();
    if (!di) return QMM_ERR_DEVICE;
    return moe_apply(di, w_qs, w_d, E, N, K, T, k, xq, xd, x_per_slot, h, moe_ws(wsp, E), S(stream), true, x);
}

qmm_status qmm_moe_gemv_pregrouped_f32(const uint8_t* w_qs, const uint16_t* w_d, int32_t E, int64_t N, int64_t K,
                                       int32_t T, int32_t k, const float* x, int x_per_slot, float* y,
                                       const void* workspace, size_t workspace_bytes, void* stream) {
    void* wsp = const_cast<void*>(workspace);
    qmm_status s = moe_check(w_qs, w_d, E, N, K, T, k, reinterpret_cast<const int8_t*>(x),
                             reinterpret_cast<const uint16_t*>(x), y, wsp, workspace_bytes);
    if (s != QMM_OK || T == 0) return s;
    const DevInfo* di = device_info();
    if (!di) return QMM_ERR_DEVICE;
    return moe_apply(di, w_qs, w_d, E, N, K, T, k, nullptr, nullptr, x_per_slot, y, moe_ws(wsp, E), S(stream), false,
                     x);
}

qmm_status qmm_moe_router_topk(const float* logits, int32_t T, int32_t E, int32_t k, int32_t* ids, float* gates,
                               void* workspace, size_t workspace_bytes, void* stream) {
    if (T < 0 || E <= 0 || k <= 0) return QMM_ERR_ARG;
    if (E > QMM_ROUTER_MAX_EXPERTS || k > QMM_ROUTER_MAX_K || k > E || (int64_t)T * k > (1 << 24) ||
        (int64_t)T * E > (int64_t(1) << 40))
        return QMM_ERR_SHAPE;
    if (T == 0) return QMM_OK;
    if (!logits || !ids || !gates) return QMM_ERR_ARG;
    if (workspace && workspace_bytes < moe_ws_bytes(E, (int64_t)T * k)) return QMM_ERR_WORKSPACE;
    if (!aligned(logits, 4) || !aligned(ids, 4) || !aligned(gates, 4) || (workspace && !aligned(workspace, 16)))
        return QMM_ERR_ALIGN;
    const DevInfo* di = device_info();
    if (!di) return QMM_ERR_DEVICE;
    static_assert(QMM_ROUTER_MAX_EXPERTS == ROUTE_MAX_E && QMM_ROUTER_MAX_K == ROUTE_MAX_K, "router limits");
    const int warps = ROUTE_THREADS / 32;
    // Grouping needs every token's ids in one block; without it, one warp
    // per token over as many CTAs as that takes (up to 4 per SM).
    const int grid = workspace ? 1 : (int)std::min<int64_t>(((int64_t)T + warps - 1) / warps, 4 * (int64_t)di->sms);
    const MoeWs ws = workspace ? moe_ws(workspace, E) : MoeWs{};
    // The grouping CTA: one warp per token, 8 to 32 warps (fewer warps make
    // its block barriers and scan cheaper when few tokens are routed)
    const int threads = workspace ? (int)std::min<int64_t>(ROUTE_THREADS, std::max<int64_t>(256, 32 * (int64_t)T))
                                  : ROUTE_THREADS;
    const cudaError_t e = launch(moe_route_kernel, dim3(grid), dim3(threads), 0, S(stream), true, logits, T, E, k, ids,
                                 gates, ws, workspace ? 1 : 0, di->err);
    return e == cudaSuccess ? launch_status() : (cudaGetLastError(), QMM_ERR_CUDA);
}

qmm_status qmm_moe_combine(const float* z, const float* gates, int32_t T, int32_t k, int64_t N, float* y,
                           void* stream) {
    if (T < 0 || k <= 0 || N <= 0) return QMM_ERR_ARG;
    if (T == 0) return QMM_OK;
    if (!z || !gates || !y) return QMM_ERR_ARG;
    if (!aligned(z, 4) || !aligned(gates, 4) || !aligned(y, 4)) return QMM_ERR_ALIGN;
    const DevInfo* di = device_info();
    if (!di) return QMM_ERR_DEVICE;
    const int64_t total = (int64_t)T * N;
    const cudaError_t e = launch(moe_combine_kernel, dim3(grid_for((total + 255) / 256, 16, di->sms)), dim3(256), 0,
                                 S(stream), true, z, gates, T, k, N, y);
    return e == cudaSuccess ? launch_status() : (cudaGetLastError(), QMM_ERR_CUDA);
}

qmm_status qmm_moe_layer_f32(const float* logits, int32_t T, int32_t E, int32_t k, const uint8_t* gu_qs,
                             const uint16_t* gu_d, const uint8_t* down_qs, const uint16_t* down_d, int64_t H,
                             int64_t F, const float* x, int32_t* ids, float* gates, float* h, float* z, float* y,
                             void* workspace, size_t workspace_bytes, void* stream) {
    // every check of the four launches before the first
    if (T < 0 || E <= 0 || k <= 0 || H <= 0 || F <= 0) return QMM_ERR_ARG;
    if (E > QMM_ROUTER_MAX_EXPERTS || k > QMM_ROUTER_MAX_K || k > E || (int64_t)T * k > (1 << 24) ||
        (int64_t)T * E > (int64_t(1) << 40) || !valid_k(H) || !valid_k(F))
        return QMM_ERR_SHAPE;
    if (T == 0) return QMM_OK;
    if (!logits || !ids || !gates || !gu_qs || !gu_d || !down_qs || !down_d || !x || !h || !z || !y)
        return QMM_ERR_ARG;
    const int64_t nslots = (int64_t)T * k;
    if (!workspace || workspace_bytes < moe_ws_bytes(E, nslots)) return QMM_ERR_WORKSPACE;
    if (!aligned(logits, 4) || !aligned(ids, 4) || !aligned(gates, 4) || !aligned(workspace, 16) ||
        !aligned(gu_qs, 16) || !aligned(down_qs, 16) || !aligned(gu_d, 2) || !aligned(down_d, 2) ||
        !aligned(x, 16) || !aligned(h, 16) || !aligned(z, 4) || !aligned(y, 4))
        return QMM_ERR_ALIGN;
    if (!moe_streamable(gu_qs, gu_d, E, 2 * F, H) || !moe_streamable(down_qs, down_d, E, H, F) ||
        moe_stream_sizes(E, H, nslots).nst < 1 || moe_stream_sizes(E, F, nslots).nst < 1)
        return QMM_ERR_SHAPE;
    const DevInfo* di = device_info();
    if (!di) return QMM_ERR_DEVICE;
    qmm_status s = qmm_moe_router_topk(logits, T, E, k, ids, gates, workspace, workspace_bytes, stream);
    if (s != QMM_OK) return s;
    const MoeWs ws = moe_ws(workspace, E);
    // The gate/up launch lets its dependents start only once the router has
    // completed, so the down launch reads the grouping and streams weights
    // before its own wait (which only its activation reads need).
    s = moe_apply(di, gu_qs, gu_d, E, 2 * F, H, T, k, nullptr, nullptr, 0, h, ws, S(stream), true, x,
                  CHAIN_LATE_TRIGGER);
    if (s != QMM_OK) return s;
    s = moe_apply(di, down_qs, down_d, E, H, F, T, k, nullptr, nullptr, 1, z, ws, S(stream), false, h,
                  CHAIN_TABLES_READY);
    if (s != QMM_OK) return s;
    return qmm_moe_combine(z, gates, T, k, H, y, stream);
}

qmm_status qmm_last_device_error(void* stream) {
    const DevInfo* di = device_info();
    if (!di) return QMM_ERR_DEVICE;
    if (cudaStreamSynchronize(S(stream)) != cudaSuccess) {
        cudaGetLastError();
        return QMM_ERR_CUDA;
    }
    int v = 0;
    if (cudaMemcpy(&v, di->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return QMM_ERR_CUDA;
    if (v) {
        const int zero = 0;
        if (cudaMemcpy(di->err, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return QMM_ERR_CUDA;
    }
    if (v & ERR_TIMEOUT) return QMM_ERR_TIMEOUT;
    if (v & ERR_BAD_EXPERT) return QMM_ERR_BAD_EXPERT_ID;
    return QMM_OK;
}

}  // extern "C"
