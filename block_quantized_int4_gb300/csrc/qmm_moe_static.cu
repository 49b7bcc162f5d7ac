// qmm_moe_static.cu -- qmm_moe_gemv_static (include/qmm.h): the MoE expert
// GEMV with its routing tables in a fixed device array owned by the library
// instead of a caller workspace.  Allocates nothing; the work itself is
// qmm_moe_gemv's, handed this array as its workspace.
#include <cuda_runtime.h>

#include <mutex>

#include "qmm.h"

// Routing tables of qmm_moe_gemv (expert counts, offsets, cursors, active
// list, slot list).  A __device__ variable exists once in each device's copy
// of the module, so every device has its own.  It need not start at zero:
// the grouping kernel rewrites every word before anything reads it.
static __device__ __align__(256) unsigned char g_moe_scratch[QMM_MOE_STATIC_SCRATCH_BYTES];

namespace {

constexpr int MAX_DEVICES = 64;

std::mutex g_mu;
void* g_scratch[MAX_DEVICES];  // device address of g_moe_scratch per device, null until looked up

// Device address of g_moe_scratch on the current device, looked up on the
// first call for that device and cached.
qmm_status scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) {
        cudaGetLastError();
        return QMM_ERR_DEVICE;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_moe_scratch);
        if (e != cudaSuccess || !p) {
            cudaGetLastError();
            int major = 0, minor = 0;
            cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
            cudaGetLastError();
            return (major == 10 && minor == 3) ? QMM_ERR_CUDA : QMM_ERR_DEVICE;
        }
        g_scratch[dev] = p;
    }
    *out = g_scratch[dev];
    return QMM_OK;
}

}  // namespace

extern "C" {

qmm_status qmm_moe_gemv_static(const uint8_t* w_qs, const uint16_t* w_d, int32_t E, int64_t N, int64_t K,
                               const int32_t* ids, int32_t T, int32_t k, const int8_t* xq, const uint16_t* xd,
                               int x_per_slot, float* y, void* stream) {
    // The workspace entry's host checks, in its order, so that both return
    // the same status for the same bad arguments; then the scratch limit.
    if (E <= 0 || N <= 0 || T < 0 || k <= 0) return QMM_ERR_ARG;
    if (K <= 0 || K % QMM_QK != 0 || K > ((int64_t)1 << 30) || (int64_t)T * k > (1 << 24)) return QMM_ERR_SHAPE;
    if (T == 0) return QMM_OK;
    if (!w_qs || !w_d || !xq || !xd || !y) return QMM_ERR_ARG;
    const auto misaligned = [](const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a != 0; };
    if (misaligned(w_qs, 16) || misaligned(w_d, 2) || misaligned(xq, 16) || misaligned(xd, 2) || misaligned(y, 4))
        return QMM_ERR_ALIGN;
    // the workspace entry checks ids after the other pointers
    if (!ids) return QMM_ERR_ARG;
    if (misaligned(ids, 4)) return QMM_ERR_ALIGN;
    size_t need = 0;
    qmm_status s = qmm_moe_workspace_size(E, T, k, &need);
    if (s != QMM_OK) return s;
    if (need > (size_t)QMM_MOE_STATIC_SCRATCH_BYTES) return QMM_ERR_SCRATCH_LIMIT;
    void* scratch = nullptr;
    if ((s = scratch_address(&scratch)) != QMM_OK) return s;
    return qmm_moe_gemv(w_qs, w_d, E, N, K, ids, T, k, xq, xd, x_per_slot, y, scratch,
                        (size_t)QMM_MOE_STATIC_SCRATCH_BYTES, stream);
}

}  // extern "C"
