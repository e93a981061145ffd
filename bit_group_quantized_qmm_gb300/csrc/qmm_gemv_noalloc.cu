// qmm_gemv_noalloc.cu -- the M = 1 GEMV for callers that cannot allocate
// device memory.
//
// qmm_gemv splits a small layer's K range over several CTAs and combines their
// partial sums in a caller-supplied workspace. Some callers have no way to
// provide one: code embedded in a host program that owns every device
// allocation and forbids its plug-ins to allocate, or a latency-critical loop
// that must never reach cudaMalloc (which may synchronise the whole device).
// This entry point runs the same kernel with its scratch in a fixed,
// file-scope device array instead, so it allocates nothing.
//
// The array is kStaticScratchBytes (1 MiB) on every device that loads the
// library and stays until the process exits. All calls share it: it keeps the
// last call's contents, the split-K counters are cleared on the stream before
// every call, and calls that overlap on the GPU (different streams, or
// different host threads) race on it.
#include <cuda_runtime.h>

#include <initializer_list>
#include <mutex>

#include "qmm.h"
#include "qmm_internal.h"

namespace qmm {
namespace {

constexpr size_t kStaticScratchBytes = QMM_GEMV_STATIC_SCRATCH_BYTES;
static_assert(kStaticScratchBytes == (size_t)1 << 20, "scratch size is part of the ABI");

// The scratch. Host code must not use this name as a device address: it is a
// host-side stand-in; the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) uint8_t g_gemv_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per
// device (this is the only CUDA call the set-up makes).
qmm_status scratch_address(void** out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return QMM_ERR_UNSUPPORTED_DEVICE;
    }
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_gemv_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return QMM_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return QMM_OK;
}

}  // namespace
}  // namespace qmm

extern "C" qmm_status qmm_gemv_static_scratch(const qmm_weight_desc* w, const void* packed, const int8_t* a,
                                              const float* sx, float* y, qmm_stream stream)
{
    using namespace qmm;
    if (!w) return QMM_ERR_INVALID_ARG;
    const size_t need = qmm_gemv_workspace_size(w);
    if (qmm_packed_size(w) == 0)
        return w->variant == QMM_W4A8 || w->variant == QMM_AFFINE || w->variant == QMM_CQ4 ? QMM_ERR_UNSUPPORTED_SHAPE
                                                                                           : QMM_ERR_INVALID_ARG;
    if (need > kStaticScratchBytes) return QMM_ERR_WORKSPACE;
    if (need == 0) return qmm_gemv(w, packed, a, sx, y, nullptr, 0, stream);   // no split: no scratch used
    // validate everything qmm_gemv validates before touching the device
    if (w->variant != QMM_W4A8 && w->variant != QMM_CQ4) return QMM_ERR_UNSUPPORTED_SHAPE;
    if (!packed || !a || !sx || !y) return QMM_ERR_INVALID_ARG;
    for (const void* p : {packed, static_cast<const void*>(a), static_cast<const void*>(sx),
                          static_cast<const void*>(y)})
        if (reinterpret_cast<uintptr_t>(p) & 15u) return QMM_ERR_MISALIGNED;
    // the device probe first: an unsupported device gets the code qmm_gemv gives
    // it, before any CUDA call of the set-up
    qmm_status st = static_cast<qmm_status>(probe_current_device());
    if (st != QMM_OK) return st;
    void* scratch = nullptr;
    st = scratch_address(&scratch);
    if (st != QMM_OK) return st;
    // the split-K counters sit at the end of the workspace and must start at zero
    const size_t T = (size_t)(w->N + 127) / 128;
    const size_t counters = T * sizeof(unsigned);
    if (cudaMemsetAsync(static_cast<uint8_t*>(scratch) + need - counters, 0, counters,
                        static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return QMM_ERR_CUDA;
    }
    return qmm_gemv(w, packed, a, sx, y, scratch, need, stream);
}
