// qmm_gemv.cu -- M = 1 decode GEMV of the symmetric W4A8 variant.
//
// cactus PR #697 "SME2 acceleration for CQ4 matmul, prefill attention, and
// orthogonal embeddings", Summary: the M = 1 path streams packed nibbles (half
// the weight bytes) and is DRAM-bound at large layers; raw integer group
// partials are rescaled by the caller's scales (the per-group partials contract
// in the review thread).
//
// Design on GB300: each CTA owns one 128-row tile of the packed blob and a
// contiguous range of its groups (split-K across CTAs when the layer has too
// few row tiles to fill the GPU). One producer warp streams the tile's chunks
// (nibbles + scales, contiguous in the blob) into a ring of shared-memory
// stages with 1-D bulk copies, so a CTA keeps tens of KB of HBM reads in
// flight with one instruction per chunk. Eight compute warps read 16-byte
// pieces conflict-free (a warp reads 512 contiguous bytes: 32 rows x one
// piece), expand nibbles to signed bytes (16*q, exact) with one shift and two
// logic ops per 8 weights, and accumulate exact int32 group partials with
// dp4a against activations staged once per CTA in the order the expansion
// consumes them. Each group partial is rescaled once in fp32. Split-K slices
// are combined by the last CTA of a tile in a fixed order (deterministic).
// Codebook (CQ4) blobs take the same loop with the nibbles looked up in the
// matrix's 16 int8 levels instead (cb_scale folded into the staged sx).
#include <cuda_fp16.h>

#include "qmm_cq4.cuh"
#include "qmm_internal.h"
#include "qmm_ptx.cuh"

namespace qmm {

constexpr int kGemvComputeThreads = 256;
constexpr int kGemvThreads = kGemvComputeThreads + 32;   // + producer warp
constexpr int kGemvTargetCtas = 3 * 152;                   // CTAs wanted in flight

template <int GROUP>
struct GemvCfg {
    static constexpr int PP = GROUP / 32;                  // 16-byte pieces per row and group
    static constexpr int CB = 64 * GROUP + 256;            // chunk bytes (nibbles + scales)
    // stages (about 52 KB for group 64; group 128 keeps 34 KB so that more CTAs
    // share an SM: measured 34.3 us against 35.0 with 6 on the lm_head GEMV)
    static constexpr int RING = GROUP == 64 ? 12 : 4;
    // The two compute halves take alternate groups, so stage i % RING must
    // always be read by the same half: with an odd ring a stage's phases would
    // alternate between the halves and a half running ahead could take a later
    // phase of the same parity for its own (ring = ng when ng < RING has no
    // stage reuse).
    static_assert(RING % 2 == 0, "even ring");
};

// Signed bytes 16*q of the low / high nibble of each byte of w (offset-binary
// nibbles u = q + 8: flipping bit 3 of the nibble gives q's two's complement).
__device__ __forceinline__ int nib_lo16(uint32_t w) { return (int)(((w << 4) ^ 0x80808080u) & 0xF0F0F0F0u); }
__device__ __forceinline__ int nib_hi16(uint32_t w) { return (int)((w ^ 0x80808080u) & 0xF0F0F0F0u); }

static size_t gemv_smem_bytes(int ring, int cb, int ng, int group)
{
    return (size_t)ring * cb + (size_t)ng * group + (size_t)ng * 4 + 128 * 4 + 2 * ring * 8 + 16 + 64;
}

// Barrier among the 256 compute threads only (the producer warp never joins).
__device__ __forceinline__ void compute_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// Grid (T, ksplit); CTA (t, s) handles groups [g0, g1) of row tile t.
template <int GROUP, bool DEBUG, bool CQ>
__global__ void __launch_bounds__(kGemvThreads)
    gemv_kernel(int N, int K, int ksplit, const uint8_t* __restrict__ blob, const int8_t* __restrict__ a,
                const float* __restrict__ sx, float* __restrict__ y, int32_t* __restrict__ P,
                float* __restrict__ ws_part, unsigned* __restrict__ ws_count, int* status)
{
    using C = GemvCfg<GROUP>;
    const int G = K / GROUP;
    const int t = blockIdx.x, s = blockIdx.y;
    const int g0 = (int)((long long)G * s / ksplit), g1 = (int)((long long)G * (s + 1) / ksplit);
    const int ng = g1 - g0;
    const int ring = ng < C::RING ? ng : C::RING;
    const int Npad = gridDim.x * 128;

    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* stages = smem;
    uint32_t* aperm = reinterpret_cast<uint32_t*>(smem + (size_t)ring * C::CB);   // permuted codes
    float* sxs = reinterpret_cast<float*>(aperm + ng * GROUP / 4);               // [ng]
    float* red = sxs + ng;                                                        // [128]
    uint64_t* full = reinterpret_cast<uint64_t*>((reinterpret_cast<uintptr_t>(red + 128) + 7) & ~uintptr_t(7));
    uint64_t* empty = full + ring;
    int* flags = reinterpret_cast<int*>(empty + ring);   // [0] abort, [1] last-CTA flag
    volatile int* abort = flags;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    pdl_trigger();
    if (tid == 0) {
        for (int i = 0; i < ring; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 4);   // the 4 warps of one half read each stage
        }
        flags[0] = 0;
        flags[1] = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kGemvComputeThreads / 32) {
        // producer: weights do not depend on the previous kernel, so the
        // copies start before the dependency wait
        if (lane == 0) {
            const uint8_t* src = blob + ((size_t)t * G + g0) * C::CB;
            int issued = 0;
            for (int i = 0; i < ng; ++i) {
                const int st = i % ring;
                if (i >= ring && !mbar_wait(&empty[st], ((i / ring) - 1) & 1, status, abort)) break;
                // the chunk lies inside the blob
                if (!in_range((size_t)t * G + g0 + i < (size_t)((N + 127) / 128) * G, status)) break;
                mbar_arrive_expect_tx(&full[st], C::CB);
                bulk_g2s(stages + (size_t)st * C::CB, src + (size_t)i * C::CB, C::CB, &full[st]);
                ++issued;
            }
            // the CTA must not exit with copies in flight: wait for the last ones
            for (int i = issued - ring > 0 ? issued - ring : 0; i < issued; ++i)
                mbar_wait(&full[i % ring], (i / ring) & 1, status, nullptr);
        }
        return;
    }

    // compute warps: stage activations (permuted for the dp4a pairing) and scales
    Cq4Book book = {};
    if (CQ) book = cq4_load(blob + cq4_trailer_offset(N, K, GROUP));
    pdl_wait();
    {
        const uint2* src = reinterpret_cast<const uint2*>(a + (size_t)g0 * GROUP);
        for (int i = tid; i < ng * GROUP / 8; i += kGemvComputeThreads) {
            const uint2 w = src[i];
            if (CQ) {
                aperm[2 * i] = __byte_perm(w.x, w.y, 0x6420);       // k = 0, 2, 4, 6
                aperm[2 * i + 1] = __byte_perm(w.x, w.y, 0x7531);   // k = 1, 3, 5, 7
            } else {
                aperm[2 * i] = __byte_perm(w.x, w.y, 0x5140);       // k = 0, 4, 1, 5
                aperm[2 * i + 1] = __byte_perm(w.x, w.y, 0x7362);   // k = 2, 6, 3, 7
            }
        }
        if (!DEBUG)   // the partials hook passes no scales
            for (int i = tid; i < ng; i += kGemvComputeThreads) sxs[i] = CQ ? sx[g0 + i] * book.scale : sx[g0 + i];
    }
    compute_sync();

    const int r = tid & 127, h = tid >> 7;
    const int n = t * 128 + r;
    float acc = 0.f;
    for (int i = h; i < ng; i += 2) {
        const int st = i % ring;
        if (!mbar_wait(&full[st], (i / ring) & 1, status, abort)) break;
        const uint8_t* c = stages + (size_t)st * C::CB;
        int dp = 0;
#pragma unroll
        for (int p = 0; p < C::PP; ++p) {
            const uint4 w = *reinterpret_cast<const uint4*>(c + p * 2048 + r * 16);
            const uint4* ap = reinterpret_cast<const uint4*>(aperm + (i * GROUP + 32 * p) / 4);
            const uint4 a0 = ap[0], a1 = ap[1];
            if (CQ) {
                uint32_t lo, hi;
                cq4_expand(book, w.x, lo, hi);
                dp = __dp4a((int)lo, (int)a0.x, dp);
                dp = __dp4a((int)hi, (int)a0.y, dp);
                cq4_expand(book, w.y, lo, hi);
                dp = __dp4a((int)lo, (int)a0.z, dp);
                dp = __dp4a((int)hi, (int)a0.w, dp);
                cq4_expand(book, w.z, lo, hi);
                dp = __dp4a((int)lo, (int)a1.x, dp);
                dp = __dp4a((int)hi, (int)a1.y, dp);
                cq4_expand(book, w.w, lo, hi);
                dp = __dp4a((int)lo, (int)a1.z, dp);
                dp = __dp4a((int)hi, (int)a1.w, dp);
            } else {
                dp = __dp4a(nib_lo16(w.x), (int)a0.x, dp);
                dp = __dp4a(nib_hi16(w.x), (int)a0.y, dp);
                dp = __dp4a(nib_lo16(w.y), (int)a0.z, dp);
                dp = __dp4a(nib_hi16(w.y), (int)a0.w, dp);
                dp = __dp4a(nib_lo16(w.z), (int)a1.x, dp);
                dp = __dp4a(nib_hi16(w.z), (int)a1.y, dp);
                dp = __dp4a(nib_lo16(w.w), (int)a1.z, dp);
                dp = __dp4a(nib_hi16(w.w), (int)a1.w, dp);
            }
        }
        const int Pg = CQ ? dp : dp >> 4;   // symmetric: exact, every product carried a factor 16
        if (DEBUG) {
            if (n < N) P[(size_t)n * G + g0 + i] = Pg;
        } else {
            const float sw = __half2float(reinterpret_cast<const __half*>(c + 64 * GROUP)[r]);
            acc = fmaf((float)Pg, sw * sxs[i], acc);
        }
        // release the stage (one arrival per warp; the 4 warps of this half read it)
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
    }
    if (DEBUG) return;

    if (h == 1) red[r] = acc;
    compute_sync();
    if (h == 0) {
        const float yv = acc + red[r];
        if (ksplit == 1) {
            if (n < N) y[n] = yv;
        } else {
            ws_part[(size_t)s * Npad + n] = yv;
        }
    }
    if (ksplit > 1) {
        __threadfence();
        compute_sync();
        if (tid == 0) {
            const unsigned prev = atomicAdd(&ws_count[t], 1u);
            flags[1] = (prev == (unsigned)ksplit - 1) ? 1 : 0;
        }
        compute_sync();
        if (flags[1]) {
            __threadfence();
            if (h == 0) {
                float yv = 0.f;
                for (int k = 0; k < ksplit; ++k) yv += __ldcg(&ws_part[(size_t)k * Npad + n]);
                if (n < N) y[n] = yv;
            }
            if (tid == 0) ws_count[t] = 0;
        }
    }
}

int gemv_ksplit(int N, int K, int group)
{
    const int T = (N + 127) / 128, G = K / group;
    int ks = (kGemvTargetCtas + T - 1) / T;
    if (ks > G) ks = G;
    if (ks < 1) ks = 1;
    return ks;
}

size_t gemv_workspace_bytes(int N, int K, int group)
{
    const int ks = gemv_ksplit(N, K, group);
    if (ks == 1) return 0;
    const size_t T = (size_t)(N + 127) / 128;
    return (size_t)ks * T * 128 * sizeof(float) + T * sizeof(unsigned);
}

template <int GROUP, bool DEBUG, bool CQ>
static cudaError_t launch_gemv_t(const LaunchCtx& c, int N, int K, int ksplit, const uint8_t* blob, const int8_t* a,
                                 const float* sx, float* y, int32_t* P, float* ws_part, unsigned* ws_count)
{
    using C = GemvCfg<GROUP>;
    const int T = (N + 127) / 128, G = K / GROUP;
    const int ng_max = (G + ksplit - 1) / ksplit;
    const int ring = ng_max < C::RING ? ng_max : C::RING;
    const size_t smem = gemv_smem_bytes(ring, C::CB, ng_max, GROUP);
    auto kern = gemv_kernel<GROUP, DEBUG, CQ>;
    static KernelSmem configured;
    const cudaError_t e = ensure_smem(configured, c, kern, smem);
    if (e != cudaSuccess) return e;
    return launch(kern, dim3(T, ksplit), dim3(kGemvThreads), smem, c, N, K, ksplit, blob, a, sx, y, P, ws_part,
                  ws_count, c.status);
}

template <int GROUP, bool CQ>
static cudaError_t launch_gemv_g(const LaunchCtx& c, int N, int K, int ks, const uint8_t* blob, const int8_t* a,
                                 const float* sx, float* y, int32_t* P_debug, float* part, unsigned* count)
{
    if (P_debug) return launch_gemv_t<GROUP, true, CQ>(c, N, K, 1, blob, a, sx, y, P_debug, nullptr, nullptr);
    return launch_gemv_t<GROUP, false, CQ>(c, N, K, ks, blob, a, sx, y, nullptr, part, count);
}

cudaError_t launch_gemv(const LaunchCtx& c, bool cq4, int N, int K, int group, const uint8_t* blob, const int8_t* a,
                        const float* sx, float* y, int32_t* P_debug, void* ws, size_t ws_bytes)
{
    int ks = 1;
    float* part = nullptr;
    unsigned* count = nullptr;
    if (!P_debug && ws) {
        ks = gemv_ksplit(N, K, group);
        if (ks > 1) {
            if (ws_bytes < gemv_workspace_bytes(N, K, group)) return cudaErrorInvalidValue;
            const size_t T = (size_t)(N + 127) / 128;
            part = static_cast<float*>(ws);
            count = reinterpret_cast<unsigned*>(static_cast<uint8_t*>(ws) + (size_t)ks * T * 128 * sizeof(float));
        }
    }
    if (group == 64)
        return cq4 ? launch_gemv_g<64, true>(c, N, K, ks, blob, a, sx, y, P_debug, part, count)
                   : launch_gemv_g<64, false>(c, N, K, ks, blob, a, sx, y, P_debug, part, count);
    if (group == 128)
        return cq4 ? launch_gemv_g<128, true>(c, N, K, ks, blob, a, sx, y, P_debug, part, count)
                   : launch_gemv_g<128, false>(c, N, K, ks, blob, a, sx, y, P_debug, part, count);
    return cudaErrorInvalidValue;
}

}  // namespace qmm
