// qmm_internal.h -- launchers shared between the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>
#include <utility>

namespace qmm {

constexpr int kMaxDevices = 64;   // device ordinals the library serves

struct LaunchCtx {
    cudaStream_t stream;
    bool pdl;         // launch with programmatic stream serialization
    int device;       // current device ordinal, < kMaxDevices
    int num_sms;
    int* status;      // device error word
};

// A kernel's dynamic shared-memory limit is a per-device function attribute,
// and CUDA sets it rather than raising it. Each launcher keeps one KernelSmem
// per kernel instantiation (a function-local static); ensure_smem raises the
// limit on the launch's device when the launch needs more than was set there.
// The fast path is one atomic load; raising is serialised by a mutex, so two
// threads never lower the limit under each other.
struct KernelSmem {
    std::atomic<size_t> bytes[kMaxDevices] = {};
};

cudaError_t ensure_smem_bytes(KernelSmem& ks, const LaunchCtx& c, const void* kern, size_t smem,
                              bool nonportable_cluster);

template <typename... Params>
cudaError_t ensure_smem(KernelSmem& ks, const LaunchCtx& c, void (*kern)(Params...), size_t smem,
                        bool nonportable_cluster = false)
{
    if (smem <= ks.bytes[c.device].load(std::memory_order_acquire)) return cudaSuccess;
    return ensure_smem_bytes(ks, c, reinterpret_cast<const void*>(kern), smem, nonportable_cluster);
}

// Launch `kern` on the context's stream, with programmatic dependent launch
// when enabled.
template <typename... Params, typename... Args>
cudaError_t launch(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem, const LaunchCtx& c,
                   Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = c.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = c.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// The library's probe of the current device (compute capability 10.3, looked
// up once per device): 0 (QMM_OK) when it is supported, else the qmm_status
// code every entry point returns for it.
int probe_current_device();

cudaError_t launch_pack(const LaunchCtx& c, int variant, int N, int K, int group, const uint8_t* q,
                        const uint16_t* scales, const uint16_t* biases, uint8_t* blob);

// Codebook 4-bit weights: raw index nibbles + trailer (16 host levels, cb_scale).
cudaError_t launch_pack_cq4(const LaunchCtx& c, int N, int K, int group, const uint8_t* idx, const int8_t* levels,
                            float cb_scale, const uint16_t* scales, uint8_t* blob);

// 4-row panel input (any variant): chunk_k weights per row per k-chunk.
cudaError_t launch_pack_il4(const LaunchCtx& c, int variant, int N, int K, int group, int chunk_k,
                            const uint8_t* panels, const uint16_t* scales, const uint16_t* biases,
                            const int8_t* levels, float cb_scale, uint8_t* blob);

cudaError_t launch_prep_w4a8(const LaunchCtx& c, int M, int K, int group, int hadamard, const void* x, int x_dtype,
                             int8_t* a, uint16_t* a16, float* sx, int32_t* asum);

// Full-K rotation z = R x (fp32, ascending fused multiply-adds), then per-group
// int8 quantization. K % 128 == 0, group 64 or 128.
// r_map: qmm_abi's rotation_tensor_map of R.
// skip_first_box: test-only fault injection (the first stage, box of R and rows of x, is never
// requested, so the kernel's bounded waits run out and it sets the timeout bit).
cudaError_t launch_prep_rotated(const LaunchCtx& c, const CUtensorMap& r_map, int M, int K, int group,
                                const void* x, int x_dtype, int8_t* a, uint16_t* a16, float* sx, int32_t* asum,
                                bool skip_first_box = false);

cudaError_t launch_prep_affine(const LaunchCtx& c, int M, int K, const void* x, int x_dtype, float* gsum,
                               uint16_t* x16);

// Number of K-slices the GEMV splits a weight into (1 = no split).
int gemv_ksplit(int N, int K, int group);
size_t gemv_workspace_bytes(int N, int K, int group);

// y = W a (M = 1). P_debug != nullptr: write raw group partials instead.
// cq4: the blob holds codebook indices and a trailer (else symmetric W4A8).
cudaError_t launch_gemv(const LaunchCtx& c, bool cq4, int N, int K, int group, const uint8_t* blob, const int8_t* a,
                        const float* sx, float* y, int32_t* P_debug, void* ws, size_t ws_bytes);

// Largest activation-row tile of the tensor-core GEMM (MMA N).
constexpr int kMaxMTile = 128;

// One-kernel decode GEMV: prepass of x and GEMV (optional code/scale outputs).
// Fused prepass + GEMV over up to kMaxSiblings weight matrices that share x,
// K and the group size (one launch; matrix i writes y[i]).
constexpr int kMaxSiblings = 8;
cudaError_t launch_gemv_fused_set(const LaunchCtx& c, bool cq4, int count, const int* N, int K, int group, int hadamard,
                                  const uint8_t* const* blob, const void* x, int x_dtype, float* const* y,
                                  int8_t* a_out, float* sx_out);
cudaError_t launch_gemv_fused(const LaunchCtx& c, bool cq4, int N, int K, int group, int hadamard, const uint8_t* blob,
                              const void* x, int x_dtype, float* y, int8_t* a_out, float* sx_out);

struct GemmShape {
    int M, N, K;
    int m_tile;      // activation rows per tile (MMA N), multiple of 16, <= kMaxMTile
    int mt_count;    // ceil(M / m_tile)
    int num_tiles;   // row tiles x mt_count
    int d_stride;    // tensor-memory columns per accumulator buffer
    int tmem_cols;   // allocated tensor-memory columns (power of two)
    int bs;          // k-step stages in use (<= the instance's maximum)
};

cudaError_t launch_gemm_w4a8(const LaunchCtx& c, int group, const CUtensorMap& map, const GemmShape& sh,
                             const uint8_t* blob, const float* sx, float* Y, int32_t* P, bool a_in_smem);
cudaError_t launch_gemm_cq4(const LaunchCtx& c, int group, const CUtensorMap& map, const GemmShape& sh,
                            const uint8_t* blob, const float* sx, float* Y, int32_t* P, bool a_in_smem);
// W4A8 / CQ4 GEMM for 1 <= M <= 32 on the tensor cores with the weights in the
// MMA's N slot. map: act_tensor_map of act16 with boxes of M rounded up to 8 rows.
cudaError_t launch_gemm_narrow(const LaunchCtx& c, bool cq4, int group, const CUtensorMap& map, int M, int N, int K,
                               const uint8_t* blob, const float* sx, float* Y);
// W4A8 GEMM for M <= 16, group 128, on the tensor cores with the weights in the
// MMA's N slot and e4m3 operands; cudaErrorNotSupported when K is too long for
// its shared memory (the caller then uses the fp16 form).
cudaError_t launch_gemm_narrow_e4m3(const LaunchCtx& c, int M, int N, int K, const uint8_t* blob,
                                    const uint16_t* act16, const float* sx, float* Y);
// W4A8 / CQ4 GEMM for M <= 16 on the CUDA cores; cudaErrorNotSupported when the
// shape does not fit it (the caller then uses the tensor-core kernel).
cudaError_t launch_gemm_rows(const LaunchCtx& c, bool cq4, int group, int M, int N, int K, const uint8_t* blob,
                             const uint16_t* act16, const float* sx, float* Y);
cudaError_t launch_gemm_affine(const LaunchCtx& c, const CUtensorMap& map, const GemmShape& sh,
                               const uint8_t* blob, const float* gsum, float* Y, bool a_in_smem);

}  // namespace qmm
