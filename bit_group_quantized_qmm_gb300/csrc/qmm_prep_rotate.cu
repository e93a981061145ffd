// qmm_prep_rotate.cu -- activation prepass with a full K x K orthogonal
// rotation, then per-group int8 quantization.
//
// Source: cactus PR #697 "SME2 acceleration for CQ4 matmul, prefill
// attention, and orthogonal embeddings", Summary: the orthogonal-rotation
// CQ4 lm_head runs on the same fused GEMV through an exact virtual 128-wide
// group view, with the rotation applied in phase A (before the weight
// stream); "Orthogonal embedding dequantization": the rotation is a K x K
// matvec accumulated in fp32.
//
// z[m][i] = sum_k R[i][k] x[m][k] is accumulated in fp32 with one fused
// multiply-add per term in ascending k, so the codes decided from z are the
// same bits on every run and equal the plain sequential sum. One dot product
// is one dependent chain of K FMAs; the work is spread so that the matrix
// streams from every SM instead:
//   - a cluster of 8 CTAs owns 128 consecutive outputs i (one or two
//     quantization groups), each CTA 16 of them, for up to 8 activation rows;
//     its 16 rows of R (16 * K * 4 bytes) stream through a ring of 512-wide
//     k-stages, one 32 KB TMA box per stage (a 3-D view of R: 32 floats x 16
//     rows x 16 k-chunks, 128-byte swizzle, so that a warp reading the same k
//     of 16 rows hits distinct banks); the first ring's worth is issued before
//     the dependency wait (R is a constant operand);
//   - thread (r, mm) runs the chain of output i0 + r for activation row mm,
//     32 k per step from registers loaded one step ahead;
//   - a group's amax is the max of its CTAs' partial maxima, exchanged through
//     distributed shared memory (max is exact in any order); the group's first
//     CTA sums the code partials (integers) and writes sx and the code sums.
// Every wait is bounded; a timed-out CTA still takes part in the cluster
// barriers (so no CTA of the cluster waits on it) and writes nothing.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "qmm_internal.h"
#include "qmm_ptx.cuh"

namespace qmm {

namespace {

constexpr int kRotThreads = 128;
constexpr int kRotCluster = 8;                    // CTAs per 128 outputs
constexpr int kRotRows = 128 / kRotCluster;       // outputs per CTA
constexpr int kRotMB = 8;                         // activation rows per CTA
constexpr int kRotChunks = 16;                    // 32-wide k-chunks per stage
constexpr int kRotCK = 32 * kRotChunks;           // k per stage
constexpr int kRotStages = 3;
constexpr int kRotRBytes = kRotChunks * kRotRows * 128;   // one TMA box
static_assert(kRotRBytes % 1024 == 0, "swizzle alignment");
static_assert(kRotThreads == kRotRows * kRotMB, "one thread per (output, row)");

// A stage holds the R box and the x rows of the launch's row blocks (at most
// kRotMB; fewer for small M, which leaves room for a second CTA per SM).
inline int rot_stage_bytes(int M, int es)
{
    const int rows = M < kRotMB ? M : kRotMB;
    return kRotRBytes + rows * kRotCK * es;   // a multiple of 1024: the next R box stays aligned
}

inline size_t rot_smem_bytes(int stage_bytes)
{
    return 1024 + (size_t)kRotStages * stage_bytes + 8 * kRotStages + 2 * 4 * kRotMB + 16;
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

// Four consecutive activations of row mm, k .. k+3, from a stage.
template <int XDT>
__device__ __forceinline__ float4 stage_x4(const uint8_t* xs, int mm, int k);

template <>
__device__ __forceinline__ float4 stage_x4<0>(const uint8_t* xs, int mm, int k)
{
    return *reinterpret_cast<const float4*>(xs + ((size_t)mm * kRotCK + k) * 4);
}
template <>
__device__ __forceinline__ float4 stage_x4<1>(const uint8_t* xs, int mm, int k)
{
    const uint2 u = *reinterpret_cast<const uint2*>(xs + ((size_t)mm * kRotCK + k) * 2);
    const float2 lo = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
    const float2 hi = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
}
template <>
__device__ __forceinline__ float4 stage_x4<2>(const uint8_t* xs, int mm, int k)
{
    const uint2 u = *reinterpret_cast<const uint2*>(xs + ((size_t)mm * kRotCK + k) * 2);
    const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
}

// R of row r, k-chunk j of a stage (32 floats), and x of row mm for the same k.
template <int XDT>
__device__ __forceinline__ void load_chunk(const uint8_t* st, int r, int mm, int j, float4 (&rv)[8], float4 (&xv)[8])
{
    const uint8_t* line = st + (size_t)(j * kRotRows + r) * 128;   // 128-byte swizzle: unit u at u ^ (line & 7)
#pragma unroll
    for (int u = 0; u < 8; ++u) rv[u] = *reinterpret_cast<const float4*>(line + ((u ^ (r & 7)) << 4));
#pragma unroll
    for (int u = 0; u < 8; ++u) xv[u] = stage_x4<XDT>(st + kRotRBytes, mm, 32 * j + 4 * u);
}

__device__ __forceinline__ float fma_chunk(float acc, const float4 (&rv)[8], const float4 (&xv)[8])
{
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        acc = __fmaf_rn(rv[u].x, xv[u].x, acc);
        acc = __fmaf_rn(rv[u].y, xv[u].y, acc);
        acc = __fmaf_rn(rv[u].z, xv[u].z, acc);
        acc = __fmaf_rn(rv[u].w, xv[u].w, acc);
    }
    return acc;
}

// Grid (K/128 * 8, ceil(M/8)), cluster (8, 1, 1), 128 threads. r_map: R as
// 32 floats x K rows x K/32 k-chunks (strides 4, 4K, 128 bytes), box 32 x 16 x 16.
template <int GROUP, int XDT>
__global__ void __launch_bounds__(kRotThreads) prep_rotate_kernel(const __grid_constant__ CUtensorMap r_map, int M,
                                                                  int K, const void* __restrict__ x,
                                                                  int8_t* __restrict__ a, __half* __restrict__ a16,
                                                                  float* __restrict__ sx,
                                                                  int32_t* __restrict__ asum, int stage_bytes,
                                                                  int skip_first_box, int* status)
{
    constexpr int ES = XDT == 0 ? 4 : 2;            // bytes per activation
    constexpr int CPG = GROUP / kRotRows;           // CTAs per quantization group (4 or 8)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + (size_t)kRotStages * stage_bytes);
    float* pamax = reinterpret_cast<float*>(full + kRotStages);   // [kRotMB] partial maxima
    int* psum = reinterpret_cast<int*>(pamax + kRotMB);            // [kRotMB] partial code sums
    int* pok = psum + kRotMB;   // every stage of this CTA arrived (read by the whole cluster)

    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int r = t & (kRotRows - 1), mm = t / kRotRows;
    const uint32_t rank = cluster_ctarank();
    const int i0 = (blockIdx.x / kRotCluster) * 128 + (int)rank * kRotRows;
    const int m0 = blockIdx.y * kRotMB;
    const int mrows = min(kRotMB, M - m0);
    const int nstage = (K + kRotCK - 1) / kRotCK;
    const int G = K / GROUP;

    if (t == 0) {
        prefetch_tensormap(&r_map);
        for (int s = 0; s < kRotStages; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
    }
    __syncthreads();
    // the GEMV/GEMM that reads the codes may start streaming its weights now;
    // its own dependency wait still waits for this grid to finish
    pdl_trigger();

    // k-width of stage c (a multiple of 128; the TMA box beyond K is zero-filled)
    auto width = [&](int c) { return min(kRotCK, K - c * kRotCK); };
    // warp 0 fills stage c: lane 0 the R box, lanes 16.. the x rows
    auto issue_r = [&](int c) {
        uint8_t* st = ring + (size_t)(c % kRotStages) * stage_bytes;
        if (lane == 0) {
            mbar_arrive_expect_tx(&full[c % kRotStages], (uint32_t)(kRotRBytes + mrows * width(c) * ES));
            // fault injection (tests): the first box is expected but never requested
            if (!(skip_first_box && c == 0)) tma_load_3d(st, &r_map, 0, i0, c * kRotChunks, &full[c % kRotStages]);
        }
    };
    auto issue_x = [&](int c) {
        if (skip_first_box && c == 0) return;   // injected: stage 0 gets no copies at all
        uint8_t* st = ring + (size_t)(c % kRotStages) * stage_bytes + kRotRBytes;
        const int j = lane - 16;
        if (j >= 0 && j < mrows)
            bulk_g2s(st + (size_t)j * kRotCK * ES,
                     static_cast<const uint8_t*>(x) + ((size_t)(m0 + j) * K + (size_t)c * kRotCK) * ES,
                     (uint32_t)(width(c) * ES), &full[c % kRotStages]);
    };

    const int first = nstage < kRotStages ? nstage : kRotStages;
    if (warp == 0)
        for (int c = 0; c < first; ++c) issue_r(c);   // the rotation is constant: before the wait
    pdl_wait();                                      // x comes from the previous kernel
    if (warp == 0) {
        __syncwarp();   // every expect_tx precedes the copies that complete it
        for (int c = 0; c < first; ++c) issue_x(c);
    }

    const bool active = 2 * warp < mrows;   // warp-uniform: some row of this warp is real
    const int mx = mm < mrows ? mm : 0;      // rows past M read row 0 (the stage holds mrows rows)
    float acc = 0.f;
    int ok = 1;
    int consumed = 0;
    for (int c = 0; c < nstage; ++c) {
        const int s = c % kRotStages;
        if (ok && !mbar_wait(&full[s], (uint32_t)(c / kRotStages) & 1u, status, nullptr)) ok = 0;
        ok = __syncthreads_and(ok);   // everyone is past stage c - 1 and sees stage c
        if (!ok) break;
        consumed = c + 1;
        if (warp == 0 && c >= 1 && c - 1 + kRotStages < nstage) {
            issue_r(c - 1 + kRotStages);
            __syncwarp();
            issue_x(c - 1 + kRotStages);
        }
        if (active) {
            const uint8_t* st = ring + (size_t)s * stage_bytes;
            const int nj = width(c) / 32;   // 4, 8, 12 or 16 chunks
            float4 ra[8], xa[8], rb[8], xb[8];
            load_chunk<XDT>(st, r, mx, 0, ra, xa);
            for (int j = 0; j < nj; j += 2) {   // nj is even
                load_chunk<XDT>(st, r, mx, j + 1, rb, xb);
                acc = fma_chunk(acc, ra, xa);
                if (j + 2 < nj) load_chunk<XDT>(st, r, mx, j + 2, ra, xa);
                acc = fma_chunk(acc, rb, xb);
            }
        }
    }
    if (!ok && warp == 0 && lane == 0) {
        // copies may still be in flight into stages that were never consumed
        const int upto = consumed >= 1 ? consumed - 1 + kRotStages : kRotStages;
        const int issued = nstage < upto ? nstage : upto;
        for (int c = consumed; c < issued; ++c) {
            if (skip_first_box && c == 0) continue;   // nothing was requested for it
            mbar_wait(&full[c % kRotStages], (uint32_t)(c / kRotStages) & 1u, status, nullptr);
        }
    }
    // the cluster's CTAs combine their partial maxima and code sums: none of
    // them writes anything unless every CTA of the cluster saw all its stages
    if (t == 0) *pok = ok;

    // ---- group amax: partial maxima of this CTA's 16 outputs per row
    const bool valid = mm < mrows;
    float pa = fabsf(acc);
#pragma unroll
    for (int o = kRotRows / 2; o > 0; o >>= 1) pa = fmaxf(pa, __shfl_xor_sync(0xffffffffu, pa, o));
    if (r == 0) pamax[mm] = pa;
    cluster_sync_all();
    for (uint32_t j = 0; j < kRotCluster; ++j) ok &= ld_shared_cluster_s32(map_shared_rank(smem_u32(pok), j));
    const uint32_t g_first = rank / CPG * CPG;
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < CPG; ++j)
        amax = fmaxf(amax, ld_shared_cluster_f32(map_shared_rank(smem_u32(pamax + mm), g_first + j)));

    int code = 0;
    float s = 0.f;
    if (amax != 0.f) {
        s = __fdiv_rn(amax, 127.0f);
        float q = rintf(__fdiv_rn(acc, s));
        q = fminf(fmaxf(q, -127.f), 127.f);
        code = (int)q;
    }
    ok = __syncthreads_and(ok);   // every thread of the CTA agrees before writing
    if (ok && valid) {
        const size_t at = (size_t)(m0 + mm) * K + i0 + r;
        if (a) a[at] = (int8_t)code;
        if (a16) a16[at] = __int2half_rn(code);
    }
    int ps = code;
#pragma unroll
    for (int o = kRotRows / 2; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
    if (r == 0) psum[mm] = ps;
    cluster_sync_all();
    if (ok && valid && r == 0 && rank == g_first) {
        int sum = 0;
        for (int j = 0; j < CPG; ++j) sum += ld_shared_cluster_s32(map_shared_rank(smem_u32(psum + mm), g_first + j));
        const int g = i0 / GROUP;
        sx[(size_t)(m0 + mm) * G + g] = s;
        if (asum) asum[(size_t)(m0 + mm) * G + g] = sum;
    }
    cluster_sync_all();   // no CTA leaves while another still reads its shared memory
}

template <int GROUP, int XDT>
cudaError_t launch_rot_t(const LaunchCtx& c, const CUtensorMap& map, int M, int K, const void* x, int8_t* a,
                         __half* a16, float* sx, int32_t* asum, int skip)
{
    auto kern = prep_rotate_kernel<GROUP, XDT>;
    const int stage_bytes = rot_stage_bytes(M, XDT == 0 ? 4 : 2);
    const size_t smem = rot_smem_bytes(stage_bytes);
    static KernelSmem configured;
    const cudaError_t e = ensure_smem(configured, c, kern, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(K / 128 * kRotCluster), (unsigned)((M + kRotMB - 1) / kRotMB));
    cfg.blockDim = dim3(kRotThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = c.stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = kRotCluster;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
    if (c.pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, map, M, K, x, a, a16, sx, asum, stage_bytes, skip, c.status);
}

template <int GROUP>
cudaError_t launch_rot_g(const LaunchCtx& c, const CUtensorMap& map, int M, int K, const void* x, int xdt,
                         int8_t* a, __half* a16, float* sx, int32_t* asum, int skip)
{
    if (xdt == 0) return launch_rot_t<GROUP, 0>(c, map, M, K, x, a, a16, sx, asum, skip);
    if (xdt == 1) return launch_rot_t<GROUP, 1>(c, map, M, K, x, a, a16, sx, asum, skip);
    return launch_rot_t<GROUP, 2>(c, map, M, K, x, a, a16, sx, asum, skip);
}

}  // namespace

cudaError_t launch_prep_rotated(const LaunchCtx& c, const CUtensorMap& r_map, int M, int K, int group,
                                const void* x, int x_dtype, int8_t* a, uint16_t* a16, float* sx, int32_t* asum,
                                bool skip_first_box)
{
    if (K % 128 != 0 || M < 1) return cudaErrorInvalidValue;
    __half* h = reinterpret_cast<__half*>(a16);
    const int skip = skip_first_box ? 1 : 0;
    if (group == 64) return launch_rot_g<64>(c, r_map, M, K, x, x_dtype, a, h, sx, asum, skip);
    if (group == 128) return launch_rot_g<128>(c, r_map, M, K, x, x_dtype, a, h, sx, asum, skip);
    return cudaErrorInvalidValue;
}

}  // namespace qmm
