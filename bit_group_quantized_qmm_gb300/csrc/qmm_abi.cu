// qmm_abi.cu -- the extern "C" boundary of libqmm_gb300: argument checks,
// device probe, tensor maps and kernel launches. Declarations and the meaning
// of every argument are in include/qmm.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <string.h>

#include <mutex>

#include "qmm.h"
#include "qmm_cq4.cuh"
#include "qmm_internal.h"

namespace qmm {

// Device error word; kernels set bits in it instead of hanging (bounded waits).
__device__ int g_status_word;

namespace {

struct DeviceInfo {
    bool probed = false;
    bool supported = false;
    int num_sms = 0;
    int* status = nullptr;
};

std::mutex g_mutex;
DeviceInfo g_devices[kMaxDevices];
thread_local int32_t g_last_kernel = QMM_KERNEL_NONE;
int g_pdl = 1;
int g_a_in_smem = 0;
int g_narrow = QMM_NARROW_AUTO;
int g_fault = 0;   // test-only fault injection point (0: none)
int g_rows_max = 8;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool desc_ok(const qmm_weight_desc* w)
{
    if (!w || w->N < 1 || w->K < 1) return false;
    if (w->variant == QMM_W4A8 || w->variant == QMM_CQ4) return w->group == 64 || w->group == 128;
    if (w->variant == QMM_AFFINE) return w->group == 64;
    return false;
}

// Variants whose activations take the symmetric int8 prepass (W4A8 weights
// and codebook weights).
bool int8_act(int32_t variant) { return variant == QMM_W4A8 || variant == QMM_CQ4; }

qmm_status shape_ok(const qmm_weight_desc* w)
{
    if (!w) return QMM_ERR_INVALID_ARG;
    if (w->variant != QMM_W4A8 && w->variant != QMM_AFFINE && w->variant != QMM_CQ4) return QMM_ERR_INVALID_ARG;
    if (w->N < 1 || w->K < 1) return QMM_ERR_INVALID_ARG;
    if (!desc_ok(w)) return QMM_ERR_UNSUPPORTED_SHAPE;
    if (w->K % w->group != 0) return QMM_ERR_UNSUPPORTED_SHAPE;
    return QMM_OK;
}

// Probe the current device once: compute capability 10.3 is required.
qmm_status device_ctx(qmm_stream stream, LaunchCtx* ctx)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return QMM_ERR_UNSUPPORTED_DEVICE;
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo& d = g_devices[dev];
    if (!d.probed) {
        d.probed = true;
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
            cudaGetLastError();
            return QMM_ERR_UNSUPPORTED_DEVICE;
        }
        d.supported = prop.major == 10 && prop.minor == 3;
        d.num_sms = prop.multiProcessorCount;
        if (d.supported) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) {
                cudaGetLastError();
                d.supported = false;
            }
            d.status = static_cast<int*>(p);
        }
    }
    if (!d.supported) return QMM_ERR_UNSUPPORTED_DEVICE;
    ctx->stream = static_cast<cudaStream_t>(stream);
    ctx->pdl = g_pdl != 0;
    ctx->device = dev;
    ctx->num_sms = d.num_sms;
    ctx->status = d.status;
    return QMM_OK;
}

std::mutex g_smem_mutex;

}  // namespace

int probe_current_device()
{
    LaunchCtx c;
    return (int)device_ctx(nullptr, &c);
}

cudaError_t ensure_smem_bytes(KernelSmem& ks, const LaunchCtx& c, const void* kern, size_t smem,
                              bool nonportable_cluster)
{
    std::lock_guard<std::mutex> lock(g_smem_mutex);
    std::atomic<size_t>& have = ks.bytes[c.device];
    if (smem <= have.load(std::memory_order_relaxed)) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (nonportable_cluster) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    have.store(smem, std::memory_order_release);
    return cudaSuccess;
}

namespace {

qmm_status launched(cudaError_t e, int32_t kernel)
{
    if (e != cudaSuccess) {
        cudaGetLastError();
        return QMM_ERR_CUDA;
    }
    g_last_kernel = kernel;
    return QMM_OK;
}

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

// fp16 [M][K] activations, boxes of 64 (k) x m_tile (rows), 128-byte swizzle.
// The last few encodings of each host thread are kept (keyed by pointer,
// shape and box): a caller that repeats a call skips the driver's encoding.
struct ActMapEntry {
    const void* ptr;
    int M, K, m_tile;
    CUtensorMap map;
};
constexpr int kActMapCache = 8;
thread_local ActMapEntry t_act_maps[kActMapCache] = {};
thread_local int t_act_next = 0;

bool act_tensor_map_encode(CUtensorMap* map, const void* act16, int M, int K, int m_tile);

bool act_tensor_map(CUtensorMap* map, const void* act16, int M, int K, int m_tile)
{
    for (const ActMapEntry& e : t_act_maps)
        if (e.ptr == act16 && e.M == M && e.K == K && e.m_tile == m_tile) {
            *map = e.map;
            return true;
        }
    if (!act_tensor_map_encode(map, act16, M, K, m_tile)) return false;
    ActMapEntry& slot = t_act_maps[t_act_next];
    t_act_next = (t_act_next + 1) % kActMapCache;
    slot.ptr = act16;
    slot.M = M;
    slot.K = K;
    slot.m_tile = m_tile;
    slot.map = *map;
    return true;
}

bool act_tensor_map_encode(CUtensorMap* map, const void* act16, int M, int K, int m_tile)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)m_tile};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(act16), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 [K][K] rotation viewed as 32 floats x K rows x K/32 k-chunks (strides
// 4 B, 4K B, 128 B), boxes of 32 x 16 rows x 16 chunks, 128-byte swizzle: one
// box is 16 rows x 512 k laid out chunk by chunk; k beyond K reads zeros.
bool rotation_tensor_map(CUtensorMap* map, const float* R, int K)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {32, (cuuint64_t)K, (cuuint64_t)(K / 32)};
    cuuint64_t strides[2] = {(cuuint64_t)K * 4, 128};
    cuuint32_t box[3] = {32, 16, 16};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(R), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tile shape of the tensor-core GEMM for M activation rows.
GemmShape gemm_shape(int M, int N, int K, bool a_in_smem)
{
    GemmShape sh;
    sh.M = M;
    sh.N = N;
    sh.K = K;
    const int tiles_m = (M + kMaxMTile - 1) / kMaxMTile;
    int mt = (M + tiles_m - 1) / tiles_m;
    mt = (mt + 15) / 16 * 16;
    if (mt < 16) mt = 16;
    sh.m_tile = mt;
    sh.mt_count = (M + mt - 1) / mt;
    sh.num_tiles = ((N + 127) / 128) * sh.mt_count;
    sh.d_stride = (mt + 31) / 32 * 32;
    const int cols = 2 * sh.d_stride + (a_in_smem ? 0 : 64);
    int alloc = 32;
    while (alloc < cols) alloc <<= 1;
    sh.tmem_cols = alloc;
    return sh;
}

}  // namespace
}  // namespace qmm

using namespace qmm;

extern "C" {

size_t qmm_packed_size(const qmm_weight_desc* w)
{
    if (shape_ok(w) != QMM_OK) return 0;
    const size_t T = (size_t)(w->N + 127) / 128;
    const size_t CB = (size_t)64 * w->group + 256 + (w->variant == QMM_AFFINE ? 256 : 0);
    return T * (size_t)(w->K / w->group) * CB + (w->variant == QMM_CQ4 ? (size_t)kCq4TrailerBytes : 0);
}

qmm_status qmm_pack_weights(const qmm_weight_desc* w, const uint8_t* q, const uint16_t* scales,
                            const uint16_t* biases, void* packed, qmm_stream stream)
{
    qmm_status st = shape_ok(w);
    if (st != QMM_OK) return st;
    if (w->variant == QMM_CQ4) return QMM_ERR_INVALID_ARG;   // needs its codebook: qmm_pack_weights_cq4
    if (!q || !scales || !packed) return QMM_ERR_INVALID_ARG;
    if ((w->variant == QMM_AFFINE) != (biases != nullptr)) return QMM_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(scales) || !aligned16(packed) || (biases && !aligned16(biases)))
        return QMM_ERR_MISALIGNED;
    LaunchCtx c;
    if ((st = device_ctx(stream, &c)) != QMM_OK) return st;
    return launched(launch_pack(c, w->variant, w->N, w->K, w->group, q, scales, biases, static_cast<uint8_t*>(packed)),
                    QMM_KERNEL_PACK);
}

qmm_status qmm_pack_weights_cq4(const qmm_weight_desc* w, const uint8_t* idx, const int8_t* codebook,
                                float cb_scale, const uint16_t* scales, void* packed, qmm_stream stream)
{
    qmm_status st = shape_ok(w);
    if (st != QMM_OK) return st;
    if (w->variant != QMM_CQ4) return QMM_ERR_INVALID_ARG;
    if (!idx || !codebook || !scales || !packed || !isfinite(cb_scale)) return QMM_ERR_INVALID_ARG;
    if (!aligned16(idx) || !aligned16(scales) || !aligned16(packed)) return QMM_ERR_MISALIGNED;
    LaunchCtx c;
    if ((st = device_ctx(stream, &c)) != QMM_OK) return st;
    return launched(launch_pack_cq4(c, w->N, w->K, w->group, idx, codebook, cb_scale, scales,
                                    static_cast<uint8_t*>(packed)),
                    QMM_KERNEL_PACK);
}

qmm_status qmm_pack_weights_interleaved4(const qmm_weight_desc* w, int32_t chunk_k, const uint8_t* panels,
                                        const uint16_t* scales, const uint16_t* biases, const int8_t* codebook,
                                        float cb_scale, void* packed, qmm_stream stream)
{
    qmm_status st = shape_ok(w);
    if (st != QMM_OK) return st;
    if (chunk_k != 8 && chunk_k != 16 && chunk_k != 32 && chunk_k != 64 && chunk_k != 128)
        return QMM_ERR_INVALID_ARG;
    if (w->K % chunk_k != 0) return QMM_ERR_UNSUPPORTED_SHAPE;
    if (!panels || !scales || !packed) return QMM_ERR_INVALID_ARG;
    if ((w->variant == QMM_AFFINE) != (biases != nullptr)) return QMM_ERR_INVALID_ARG;
    if ((w->variant == QMM_CQ4) != (codebook != nullptr)) return QMM_ERR_INVALID_ARG;
    if (w->variant == QMM_CQ4 && !isfinite(cb_scale)) return QMM_ERR_INVALID_ARG;
    if (!aligned16(panels) || !aligned16(scales) || !aligned16(packed) || (biases && !aligned16(biases)))
        return QMM_ERR_MISALIGNED;
    LaunchCtx c;
    if ((st = device_ctx(stream, &c)) != QMM_OK) return st;
    return launched(launch_pack_il4(c, w->variant, w->N, w->K, w->group, chunk_k, panels, scales, biases, codebook,
                                    cb_scale, static_cast<uint8_t*>(packed)),
                    QMM_KERNEL_PACK);
}

qmm_status qmm_prep_act(int32_t variant, int32_t M, int32_t K, int32_t group, int32_t hadamard, const void* x,
                        int32_t x_dtype, int8_t* a, uint16_t* a16, float* sx, int32_t* asum, float* gsum,
                        uint16_t* x16, qmm_stream stream)
{
    if (M < 1 || K < 1 || !x) return QMM_ERR_INVALID_ARG;
    if (x_dtype != QMM_DTYPE_F32 && x_dtype != QMM_DTYPE_F16 && x_dtype != QMM_DTYPE_BF16) return QMM_ERR_INVALID_ARG;
    if (!aligned16(x)) return QMM_ERR_MISALIGNED;
    qmm_status st;
    LaunchCtx c;
    if (int8_act(variant)) {
        if (group != 64 && group != 128) return QMM_ERR_UNSUPPORTED_SHAPE;
        if (K % group) return QMM_ERR_UNSUPPORTED_SHAPE;
        if (hadamard != 0 && hadamard != group) return QMM_ERR_UNSUPPORTED_SHAPE;
        if (!sx || gsum || x16) return QMM_ERR_INVALID_ARG;
        if ((a && !aligned16(a)) || (a16 && !aligned16(a16)) || !aligned16(sx) || (asum && !aligned16(asum)))
            return QMM_ERR_MISALIGNED;
        if ((st = device_ctx(stream, &c)) != QMM_OK) return st;
        return launched(launch_prep_w4a8(c, M, K, group, hadamard, x, x_dtype, a, a16, sx, asum),
                        QMM_KERNEL_PREP_W4A8);
    }
    if (variant == QMM_AFFINE) {
        if (group != 64 || K % 64 || hadamard != 0) return QMM_ERR_UNSUPPORTED_SHAPE;
        if (!gsum || a || a16 || sx || asum) return QMM_ERR_INVALID_ARG;
        if (!aligned16(gsum) || (x16 && !aligned16(x16))) return QMM_ERR_MISALIGNED;
        if ((st = device_ctx(stream, &c)) != QMM_OK) return st;
        return launched(launch_prep_affine(c, M, K, x, x_dtype, gsum, x16), QMM_KERNEL_PREP_AFFINE);
    }
    return QMM_ERR_INVALID_ARG;
}

qmm_status qmm_prep_act_rotated(int32_t M, int32_t K, int32_t group, const float* R, const void* x,
                                int32_t x_dtype, int8_t* a, uint16_t* a16, float* sx, int32_t* asum,
                                qmm_stream stream)
{
    if (M < 1 || K < 1 || !R || !x || !sx) return QMM_ERR_INVALID_ARG;
    if (x_dtype != QMM_DTYPE_F32 && x_dtype != QMM_DTYPE_F16 && x_dtype != QMM_DTYPE_BF16) return QMM_ERR_INVALID_ARG;
    if (group != 64 && group != 128) return QMM_ERR_UNSUPPORTED_SHAPE;
    if (K % 128 != 0) return QMM_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(R) || !aligned16(x) || !aligned16(sx) || (a && !aligned16(a)) || (a16 && !aligned16(a16)) ||
        (asum && !aligned16(asum)))
        return QMM_ERR_MISALIGNED;
    qmm_status st;
    LaunchCtx c;
    if ((st = device_ctx(stream, &c)) != QMM_OK) return st;
    CUtensorMap map;
    if (!rotation_tensor_map(&map, R, K)) return QMM_ERR_CUDA;
    return launched(launch_prep_rotated(c, map, M, K, group, x, x_dtype, a, a16, sx, asum, g_fault == 1),
                    QMM_KERNEL_PREP_ROTATED);
}

size_t qmm_gemv_workspace_size(const qmm_weight_desc* w)
{
    if (shape_ok(w) != QMM_OK || !int8_act(w->variant)) return 0;
    return gemv_workspace_bytes(w->N, w->K, w->group);
}

qmm_status qmm_gemv(const qmm_weight_desc* w, const void* packed, const int8_t* a, const float* sx, float* y,
                    void* workspace, size_t workspace_bytes, qmm_stream stream)
{
    qmm_status st = shape_ok(w);
    if (st != QMM_OK) return st;
    if (!int8_act(w->variant)) return QMM_ERR_UNSUPPORTED_SHAPE;
    if (!packed || !a || !sx || !y) return QMM_ERR_INVALID_ARG;
    if (!aligned16(packed) || !aligned16(a) || !aligned16(sx) || !aligned16(y) ||
        (workspace && !aligned16(workspace)))
        return QMM_ERR_MISALIGNED;
    if (workspace && workspace_bytes < gemv_workspace_bytes(w->N, w->K, w->group)) return QMM_ERR_WORKSPACE;
    LaunchCtx c;
    if ((st = device_ctx(stream, &c)) != QMM_OK) return st;
    const bool cq4 = w->variant == QMM_CQ4;
    return launched(launch_gemv(c, cq4, w->N, w->K, w->group, static_cast<const uint8_t*>(packed), a, sx, y,
                                nullptr, workspace, workspace_bytes),
                    cq4 ? QMM_KERNEL_GEMV_CQ4 : QMM_KERNEL_GEMV_W4A8);
}

qmm_status qmm_gemv_fused(const qmm_weight_desc* w, const void* packed, const void* x, int32_t x_dtype,
                          int32_t hadamard, float* y, int8_t* a_out, float* sx_out, qmm_stream stream)
{
    qmm_status st = shape_ok(w);
    if (st != QMM_OK) return st;
    if (!int8_act(w->variant)) return QMM_ERR_UNSUPPORTED_SHAPE;
    if (hadamard != 0 && hadamard != w->group) return QMM_ERR_UNSUPPORTED_SHAPE;
    if (x_dtype != QMM_DTYPE_F32 && x_dtype != QMM_DTYPE_F16 && x_dtype != QMM_DTYPE_BF16) return QMM_ERR_INVALID_ARG;
    if (!packed || !x || !y) return QMM_ERR_INVALID_ARG;
    if (!aligned16(packed) || !aligned16(x) || !aligned16(y) || (a_out && !aligned16(a_out)) ||
        (sx_out && !aligned16(sx_out)))
        return QMM_ERR_MISALIGNED;
    const int max_k = 16 * (w->group == 64 ? 44 : 22) * w->group;
    if (w->K > max_k) return QMM_ERR_UNSUPPORTED_SHAPE;
    LaunchCtx c;
    if ((st = device_ctx(stream, &c)) != QMM_OK) return st;
    return launched(launch_gemv_fused(c, w->variant == QMM_CQ4, w->N, w->K, w->group, hadamard, static_cast<const uint8_t*>(packed), x,
                                      x_dtype, y, a_out, sx_out),
                    QMM_KERNEL_GEMV_FUSED);
}

qmm_status qmm_gemv_fused_siblings(int32_t count, const qmm_weight_desc* w, const void* const* packed,
                                   const void* x, int32_t x_dtype, int32_t hadamard, float* const* y,
                                   int8_t* a_out, float* sx_out, qmm_stream stream)
{
    if (count < 1 || count > QMM_MAX_SIBLINGS || count > kMaxSiblings || !w || !packed || !y || !x)
        return QMM_ERR_INVALID_ARG;
    int N[QMM_MAX_SIBLINGS];
    const uint8_t* blobs[QMM_MAX_SIBLINGS];
    float* ys[QMM_MAX_SIBLINGS];
    for (int i = 0; i < count; ++i) {
        qmm_status st = shape_ok(&w[i]);
        if (st != QMM_OK) return st;
        if (!int8_act(w[i].variant) || w[i].variant != w[0].variant || w[i].K != w[0].K ||
            w[i].group != w[0].group)
            return QMM_ERR_UNSUPPORTED_SHAPE;
        if (!packed[i] || !y[i]) return QMM_ERR_INVALID_ARG;
        if (!aligned16(packed[i]) || !aligned16(y[i])) return QMM_ERR_MISALIGNED;
        N[i] = w[i].N;
        blobs[i] = static_cast<const uint8_t*>(packed[i]);
        ys[i] = y[i];
    }
    if (hadamard != 0 && hadamard != w[0].group) return QMM_ERR_UNSUPPORTED_SHAPE;
    if (x_dtype != QMM_DTYPE_F32 && x_dtype != QMM_DTYPE_F16 && x_dtype != QMM_DTYPE_BF16) return QMM_ERR_INVALID_ARG;
    if (!aligned16(x) || (a_out && !aligned16(a_out)) || (sx_out && !aligned16(sx_out))) return QMM_ERR_MISALIGNED;
    const int max_k = 16 * (w[0].group == 64 ? 44 : 22) * w[0].group;
    if (w[0].K > max_k) return QMM_ERR_UNSUPPORTED_SHAPE;
    LaunchCtx c;
    qmm_status st = device_ctx(stream, &c);
    if (st != QMM_OK) return st;
    return launched(launch_gemv_fused_set(c, w[0].variant == QMM_CQ4, count, N, w[0].K, w[0].group, hadamard, blobs, x, x_dtype, ys, a_out,
                                          sx_out),
                    QMM_KERNEL_GEMV_FUSED_SIBLINGS);
}

static qmm_status gemm_common(const qmm_weight_desc* w, const void* packed, int32_t M, const void* act16,
                              const float* act_scale, float* Y, int32_t* P, qmm_stream stream)
{
    qmm_status st = shape_ok(w);
    if (st != QMM_OK) return st;
    if (M < 1 || !packed || !act16 || (!P && (!act_scale || !Y))) return QMM_ERR_INVALID_ARG;
    if (!aligned16(packed) || !aligned16(act16) || (act_scale && !aligned16(act_scale)) || (Y && !aligned16(Y)) ||
        (P && !aligned16(P)))
        return QMM_ERR_MISALIGNED;
    if (w->K % 64) return QMM_ERR_UNSUPPORTED_SHAPE;
    LaunchCtx c;
    if ((st = device_ctx(stream, &c)) != QMM_OK) return st;
    const uint8_t* blob = static_cast<const uint8_t*>(packed);
    const bool cq4 = w->variant == QMM_CQ4;
    if (int8_act(w->variant) && !P && M <= g_rows_max) {
        const cudaError_t e = launch_gemm_rows(c, cq4, w->group, M, w->N, w->K, blob,
                                               static_cast<const uint16_t*>(act16), act_scale, Y);
        if (e != cudaErrorNotSupported) return launched(e, QMM_KERNEL_GEMM_ROWS);
    }
    const bool many_tiles = (w->N + 127) / 128 >= 512;
    if (w->variant == QMM_W4A8 && !P && M <= 16 && w->group == 128 &&
        (g_narrow == QMM_NARROW_ALWAYS || (g_narrow == QMM_NARROW_AUTO && many_tiles))) {
        const cudaError_t e = launch_gemm_narrow_e4m3(c, M, w->N, w->K, blob, static_cast<const uint16_t*>(act16),
                                                      act_scale, Y);
        if (e != cudaErrorNotSupported) return launched(e, QMM_KERNEL_GEMM_NARROW_E4M3);
    }
    if (int8_act(w->variant) && !P && M <= 32 &&
        (g_narrow == QMM_NARROW_ALWAYS || g_narrow == QMM_NARROW_F16 ||
         (g_narrow == QMM_NARROW_AUTO && w->variant == QMM_W4A8 && many_tiles))) {
        CUtensorMap nmap;
        if (!act_tensor_map(&nmap, act16, M, w->K, (M + 7) & ~7)) return QMM_ERR_CUDA;
        const cudaError_t e = launch_gemm_narrow(c, cq4, w->group, nmap, M, w->N, w->K, blob, act_scale, Y);
        if (e != cudaErrorNotSupported) return launched(e, QMM_KERNEL_GEMM_NARROW);
    }
    const bool a_smem = g_a_in_smem != 0;
    GemmShape sh = gemm_shape(M, w->N, w->K, a_smem);
    CUtensorMap map;
    if (!act_tensor_map(&map, act16, M, w->K, sh.m_tile)) return QMM_ERR_CUDA;
    if (w->variant == QMM_W4A8)
        return launched(launch_gemm_w4a8(c, w->group, map, sh, blob, act_scale, Y, P, a_smem), QMM_KERNEL_GEMM_W4A8);
    if (cq4)
        return launched(launch_gemm_cq4(c, w->group, map, sh, blob, act_scale, Y, P, a_smem), QMM_KERNEL_GEMM_CQ4);
    if (P) return QMM_ERR_UNSUPPORTED_SHAPE;
    return launched(launch_gemm_affine(c, map, sh, blob, act_scale, Y, a_smem), QMM_KERNEL_GEMM_AFFINE);
}

qmm_status qmm_gemm(const qmm_weight_desc* w, const void* packed, int32_t M, const uint16_t* act16,
                    const float* act_scale, float* Y, qmm_stream stream)
{
    if (!act_scale || !Y) return QMM_ERR_INVALID_ARG;
    return gemm_common(w, packed, M, act16, act_scale, Y, nullptr, stream);
}

qmm_status qmm_debug_partials(const qmm_weight_desc* w, const void* packed, int32_t M, int32_t path,
                              const void* act, int32_t* P, qmm_stream stream)
{
    qmm_status st = shape_ok(w);
    if (st != QMM_OK) return st;
    if (!int8_act(w->variant)) return QMM_ERR_UNSUPPORTED_SHAPE;
    if (!packed || !act || !P || M < 1) return QMM_ERR_INVALID_ARG;
    if (path == QMM_PATH_GEMV) {
        if (M != 1) return QMM_ERR_INVALID_ARG;
        if (!aligned16(packed) || !aligned16(act) || !aligned16(P)) return QMM_ERR_MISALIGNED;
        LaunchCtx c;
        if ((st = device_ctx(stream, &c)) != QMM_OK) return st;
        const bool cq4 = w->variant == QMM_CQ4;
        return launched(launch_gemv(c, cq4, w->N, w->K, w->group, static_cast<const uint8_t*>(packed),
                                    static_cast<const int8_t*>(act), nullptr, nullptr, P, nullptr, 0),
                        cq4 ? QMM_KERNEL_GEMV_CQ4 : QMM_KERNEL_GEMV_W4A8);
    }
    if (path == QMM_PATH_GEMM) return gemm_common(w, packed, M, act, nullptr, nullptr, P, stream);
    return QMM_ERR_INVALID_ARG;
}

const char* qmm_status_string(qmm_status s)
{
    switch (s) {
    case QMM_OK: return "ok";
    case QMM_ERR_INVALID_ARG: return "invalid argument";
    case QMM_ERR_UNSUPPORTED_SHAPE: return "unsupported shape or group size";
    case QMM_ERR_UNSUPPORTED_DEVICE: return "unsupported device (compute capability 10.3 required)";
    case QMM_ERR_MISALIGNED: return "device pointer not 16-byte aligned";
    case QMM_ERR_CUDA: return "CUDA call failed";
    case QMM_ERR_TIMEOUT: return "a kernel gave up a bounded wait";
    case QMM_ERR_WORKSPACE: return "workspace too small";
    }
    return "unknown status";
}

int32_t qmm_last_kernel_id(void) { return g_last_kernel; }

qmm_status qmm_device_status(qmm_stream stream, int32_t* flags)
{
    LaunchCtx c;
    qmm_status st = device_ctx(stream, &c);
    if (st != QMM_OK) return st;
    if (cudaStreamSynchronize(c.stream) != cudaSuccess) {
        cudaGetLastError();
        return QMM_ERR_CUDA;
    }
    int word = 0;
    if (cudaMemcpy(&word, c.status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return QMM_ERR_CUDA;
    }
    const int zero = 0;
    if (word && cudaMemcpy(c.status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaGetLastError();
        return QMM_ERR_CUDA;
    }
    if (flags) *flags = word;
    return word ? QMM_ERR_TIMEOUT : QMM_OK;
}

void qmm_set_pdl(int32_t enable) { g_pdl = enable ? 1 : 0; }

void qmm_set_fault_injection(int32_t point) { g_fault = point == 1 ? 1 : 0; }

void qmm_set_gemm_weight_operand(int32_t in_shared_memory) { g_a_in_smem = in_shared_memory ? 1 : 0; }

void qmm_set_gemm_narrow(int32_t mode)
{
    g_narrow = mode == QMM_NARROW_OFF || mode == QMM_NARROW_ALWAYS || mode == QMM_NARROW_F16 ? mode
                                                                                          : QMM_NARROW_AUTO;
}

void qmm_set_gemm_rows_max(int32_t max_rows) { g_rows_max = max_rows < 0 ? 0 : (max_rows > 16 ? 16 : max_rows); }

}  // extern "C"
