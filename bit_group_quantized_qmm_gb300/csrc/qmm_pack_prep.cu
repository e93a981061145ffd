// qmm_pack_prep.cu -- weight repack and activation prepass kernels.
//
// Weight repack: cactus PR #697 "SME2 acceleration for CQ4 matmul, prefill
// attention, and orthogonal embeddings" (the packed weight cache is built once
// per weight and is the one runtime format); geistlib issue #500 "native W*A8
// int8 GEMM for prefill", Design sketch item 2 (repack at resolve time).
// Activation prepass: cactus PR #697, Summary (parallel Hadamard transform and
// int8 activation quantization ahead of the GEMV); TensorFold PR #3215
// "simd_qmm on Metal: X's group sums and half operands from a prepass", What
// this changes (group sums by the tiles' tree, X written once as half).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <string.h>

#include "qmm_internal.h"
#include "qmm_ptx.cuh"

namespace qmm {

// ------------------------------------------------------------------ repack

// Input word: 8 nibbles, byte i holding k = 2i (low) and k = 2i+1 (high).
// Output word: slots 0-3 take k = 0, 2, 4, 6 (the low nibbles), slots 4-7
// take k = 1, 3, 5, 7 (the high nibbles). In that order the fp16 expansion
// yields (k, k+1) pairs and the dp4a expansion pairs with permuted activations.
__device__ __forceinline__ uint32_t repack_word(uint32_t w)
{
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        lo |= ((w >> (8 * i)) & 0xFu) << (4 * i);
        hi |= ((w >> (8 * i + 4)) & 0xFu) << (4 * i);
    }
    return lo | (hi << 16);
}

// Source layouts. il4_cb == 0: row-major nibble bytes [N][K/2] and scales
// [N][G]. il4_cb > 0: 4-row panels (cactus PR #697, follow-up on the
// orthogonal lm_head: the production INTERLEAVED_4ROW layout keeps rows in
// blocks of four, block nb at byte nb*2K, its bytes ordered by k-chunk; scales
// of block nb, group g, row ni at (nb*G + g)*4 + ni). Chunk c of a block holds
// the four rows' il4_cb bytes (2*il4_cb weights) in row order.
__device__ __forceinline__ size_t src_byte(int n, int kb, int K, int il4_cb)
{
    if (il4_cb == 0) return (size_t)n * (K / 2) + kb;
    return (size_t)(n >> 2) * (2 * K) + (size_t)(kb / il4_cb) * (4 * il4_cb) + (size_t)(n & 3) * il4_cb +
           (size_t)(kb % il4_cb);
}

__device__ __forceinline__ size_t src_scale(int n, int g, int G, int il4_cb)
{
    if (il4_cb == 0) return (size_t)n * G + g;
    return ((size_t)(n >> 2) * G + g) * 4 + (size_t)(n & 3);
}

// One thread per 16-byte piece of the blob (row r, piece p, group g, tile t).
// VARIANT 0 symmetric, 1 affine, 2 codebook (CQ4: raw indices, and the first
// thread writes the trailer: levels, cb_scale, zero padding).
template <int VARIANT, int GROUP>
__global__ void __launch_bounds__(256) pack_kernel(int N, int K, const uint8_t* __restrict__ q,
                                                   const uint16_t* __restrict__ scales,
                                                   const uint16_t* __restrict__ biases, uint8_t* __restrict__ blob,
                                                   uint4 levels, float cb_scale, int il4_cb)
{
    constexpr int PP = GROUP / 32;
    constexpr int CB = 64 * GROUP + 256 + (VARIANT == 1 ? 256 : 0);
    // No early trigger: the GEMV and GEMM kernels stream packed weights before
    // their own dependency wait, so a kernel queued right after this one may
    // start only once every byte of the blob is written.
    pdl_wait();
    const int G = K / GROUP;
    const int T = (N + 127) / 128;
    const long long total = (long long)T * G * PP * 128;
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= total) return;
    if (VARIANT == 2 && idx == 0) {
        uint4* tr = reinterpret_cast<uint4*>(blob + (size_t)T * G * CB);   // after the T*G chunks
        tr[0] = levels;
        tr[1] = make_uint4(__float_as_uint(cb_scale), 0u, 0u, 0u);
    }
    const int r = (int)(idx % 128);
    long long rest = idx / 128;
    const int p = (int)(rest % PP);
    rest /= PP;
    const int g = (int)(rest % G);
    const int t = (int)(rest / G);
    const int n = t * 128 + r;
    uint8_t* chunk = blob + ((size_t)t * G + g) * CB;

    // offset binary for the symmetric variant: q + 8 == q ^ 8 on 4 bits
    const uint32_t flip = VARIANT == 0 ? 0x88888888u : 0u;
    uint4 out;
    if (n < N) {
        const int kb = (g * GROUP + 32 * p) / 2;
        uint4 in;
        if (il4_cb == 0 || il4_cb >= 16) {
            // the piece's 16 bytes are contiguous (16-byte aligned) in the source
            in = *reinterpret_cast<const uint4*>(q + src_byte(n, kb, K, il4_cb));
        } else {
            // narrow chunks: each aligned 4-byte word lies inside one chunk
            in.x = *reinterpret_cast<const uint32_t*>(q + src_byte(n, kb, K, il4_cb));
            in.y = *reinterpret_cast<const uint32_t*>(q + src_byte(n, kb + 4, K, il4_cb));
            in.z = *reinterpret_cast<const uint32_t*>(q + src_byte(n, kb + 8, K, il4_cb));
            in.w = *reinterpret_cast<const uint32_t*>(q + src_byte(n, kb + 12, K, il4_cb));
        }
        out.x = repack_word(in.x) ^ flip;
        out.y = repack_word(in.y) ^ flip;
        out.z = repack_word(in.z) ^ flip;
        out.w = repack_word(in.w) ^ flip;
    } else {
        out = make_uint4(flip, flip, flip, flip);
    }
    *reinterpret_cast<uint4*>(chunk + p * 2048 + r * 16) = out;
    if (p == 0) {
        const uint16_t s = n < N ? scales[src_scale(n, g, G, il4_cb)] : 0;
        *reinterpret_cast<uint16_t*>(chunk + 64 * GROUP + 2 * r) = s;
        if (VARIANT == 1) {
            const uint16_t b = n < N ? biases[src_scale(n, g, G, il4_cb)] : 0;
            *reinterpret_cast<uint16_t*>(chunk + 64 * GROUP + 256 + 2 * r) = b;
        }
    }
}

template <int VARIANT, int GROUP>
static cudaError_t launch_pack_t(const LaunchCtx& c, int N, int K, const uint8_t* q, const uint16_t* s,
                                 const uint16_t* b, uint8_t* blob, uint4 levels, float cb_scale, int il4_cb)
{
    const long long total = (long long)((N + 127) / 128) * (K / GROUP) * (GROUP / 32) * 128;
    const int threads = 256;
    const long long blocks = (total + threads - 1) / threads;
    return launch(pack_kernel<VARIANT, GROUP>, dim3((unsigned)blocks), dim3(threads), 0, c, N, K, q, s, b, blob,
                  levels, cb_scale, il4_cb);
}

static cudaError_t launch_pack_any(const LaunchCtx& c, int variant, int N, int K, int group, const uint8_t* q,
                                   const uint16_t* scales, const uint16_t* biases, uint8_t* blob, uint4 lv,
                                   float cb_scale, int il4_cb)
{
    if (variant == 0 && group == 64) return launch_pack_t<0, 64>(c, N, K, q, scales, biases, blob, lv, 0.f, il4_cb);
    if (variant == 0 && group == 128) return launch_pack_t<0, 128>(c, N, K, q, scales, biases, blob, lv, 0.f, il4_cb);
    if (variant == 1 && group == 64) return launch_pack_t<1, 64>(c, N, K, q, scales, biases, blob, lv, 0.f, il4_cb);
    if (variant == 2 && group == 64) return launch_pack_t<2, 64>(c, N, K, q, scales, nullptr, blob, lv, cb_scale, il4_cb);
    if (variant == 2 && group == 128)
        return launch_pack_t<2, 128>(c, N, K, q, scales, nullptr, blob, lv, cb_scale, il4_cb);
    return cudaErrorInvalidValue;
}

cudaError_t launch_pack(const LaunchCtx& c, int variant, int N, int K, int group, const uint8_t* q,
                        const uint16_t* scales, const uint16_t* biases, uint8_t* blob)
{
    if (variant == 2) return cudaErrorInvalidValue;
    return launch_pack_any(c, variant, N, K, group, q, scales, biases, blob, uint4{}, 0.f, 0);
}

cudaError_t launch_pack_cq4(const LaunchCtx& c, int N, int K, int group, const uint8_t* idx, const int8_t* levels,
                            float cb_scale, const uint16_t* scales, uint8_t* blob)
{
    uint4 lv;
    memcpy(&lv, levels, 16);
    return launch_pack_any(c, 2, N, K, group, idx, scales, nullptr, blob, lv, cb_scale, 0);
}

cudaError_t launch_pack_il4(const LaunchCtx& c, int variant, int N, int K, int group, int chunk_k,
                            const uint8_t* panels, const uint16_t* scales, const uint16_t* biases,
                            const int8_t* levels, float cb_scale, uint8_t* blob)
{
    uint4 lv{};
    if (variant == 2) memcpy(&lv, levels, 16);
    return launch_pack_any(c, variant, N, K, group, panels, scales, biases, blob, lv, cb_scale, chunk_k / 2);
}

// ------------------------------------------------------------------ loads

template <int XDT>
__device__ __forceinline__ float load_x(const void* x, size_t i);

template <>
__device__ __forceinline__ float load_x<0>(const void* x, size_t i)
{
    return static_cast<const float*>(x)[i];
}
template <>
__device__ __forceinline__ float load_x<1>(const void* x, size_t i)
{
    return __half2float(static_cast<const __half*>(x)[i]);
}
template <>
__device__ __forceinline__ float load_x<2>(const void* x, size_t i)
{
    return __bfloat162float(static_cast<const __nv_bfloat16*>(x)[i]);
}

// ------------------------------------------------------------------ W4A8 prep

// One warp per (row m, group g); lane l holds inputs l*E .. l*E+E-1.
template <int GROUP, int XDT>
__global__ void __launch_bounds__(256) prep_w4a8_kernel(int M, int K, int hadamard, float rot_scale,
                                                        const void* __restrict__ x, int8_t* __restrict__ a,
                                                        __half* __restrict__ a16, float* __restrict__ sx,
                                                        int32_t* __restrict__ asum)
{
    constexpr int E = GROUP / 32;
    pdl_trigger();
    pdl_wait();
    const int G = K / GROUP;
    const long long wid = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (wid >= (long long)M * G) return;   // uniform per warp
    const int m = (int)(wid / G), g = (int)(wid % G);
    const size_t base = (size_t)m * K + (size_t)g * GROUP + (size_t)lane * E;

    float v[E];
#pragma unroll
    for (int e = 0; e < E; ++e) v[e] = load_x<XDT>(x, base + e);

    if (hadamard) {
        // unnormalised Walsh-Hadamard butterflies, stages h = 1, 2, 4, ...
#pragma unroll
        for (int h = 1; h < GROUP; h <<= 1) {
            if (h < E) {
#pragma unroll
                for (int e = 0; e < E; ++e)
                    if ((e & h) == 0) {
                        const float lo = v[e], hi = v[e + h];
                        v[e] = __fadd_rn(lo, hi);
                        v[e + h] = __fsub_rn(lo, hi);
                    }
            } else {
                const int lm = h / E;
                const bool upper = (lane & lm) != 0;
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const float o = __shfl_xor_sync(0xffffffffu, v[e], lm);
                    v[e] = upper ? __fsub_rn(o, v[e]) : __fadd_rn(v[e], o);
                }
            }
        }
    }

    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(v[e]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));

    int codes[E];
    float scale = 0.f;
    if (amax == 0.f) {
#pragma unroll
        for (int e = 0; e < E; ++e) codes[e] = 0;
    } else {
        const float s = __fdiv_rn(amax, 127.0f);
#pragma unroll
        for (int e = 0; e < E; ++e) {
            float r = rintf(__fdiv_rn(v[e], s));
            r = fminf(fmaxf(r, -127.f), 127.f);
            codes[e] = (int)r;
        }
        scale = __fmul_rn(s, rot_scale);
    }

    int sum = 0;
#pragma unroll
    for (int e = 0; e < E; ++e) sum += codes[e];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);

    if (a) {
        uint32_t packed = 0;
#pragma unroll
        for (int e = 0; e < E; ++e) packed |= ((uint32_t)codes[e] & 0xFFu) << (8 * e);
        if (E == 2)
            *reinterpret_cast<uint16_t*>(a + base) = (uint16_t)packed;
        else
            *reinterpret_cast<uint32_t*>(a + base) = packed;
    }
    if (a16) {
#pragma unroll
        for (int e = 0; e < E; e += 2)
            *reinterpret_cast<__half2*>(a16 + base + e) =
                __halves2half2(__int2half_rn(codes[e]), __int2half_rn(codes[e + 1]));
    }
    if (lane == 0) {
        sx[(size_t)m * G + g] = scale;
        if (asum) asum[(size_t)m * G + g] = sum;
    }
}

template <int GROUP>
static cudaError_t launch_prep_w4a8_t(const LaunchCtx& c, int M, int K, int hadamard, const void* x, int xdt,
                                      int8_t* a, uint16_t* a16, float* sx, int32_t* asum)
{
    const float rot = hadamard ? (float)(1.0 / sqrt((double)GROUP)) : 1.0f;
    const long long warps = (long long)M * (K / GROUP);
    const int threads = 256;
    const unsigned blocks = (unsigned)((warps * 32 + threads - 1) / threads);
    __half* h16 = reinterpret_cast<__half*>(a16);
    if (xdt == 0)
        return launch(prep_w4a8_kernel<GROUP, 0>, dim3(blocks), dim3(threads), 0, c, M, K, hadamard, rot, x, a, h16,
                      sx, asum);
    if (xdt == 1)
        return launch(prep_w4a8_kernel<GROUP, 1>, dim3(blocks), dim3(threads), 0, c, M, K, hadamard, rot, x, a, h16,
                      sx, asum);
    return launch(prep_w4a8_kernel<GROUP, 2>, dim3(blocks), dim3(threads), 0, c, M, K, hadamard, rot, x, a, h16, sx,
                  asum);
}

cudaError_t launch_prep_w4a8(const LaunchCtx& c, int M, int K, int group, int hadamard, const void* x, int x_dtype,
                             int8_t* a, uint16_t* a16, float* sx, int32_t* asum)
{
    if (group == 64) return launch_prep_w4a8_t<64>(c, M, K, hadamard, x, x_dtype, a, a16, sx, asum);
    if (group == 128) return launch_prep_w4a8_t<128>(c, M, K, hadamard, x, x_dtype, a, a16, sx, asum);
    return cudaErrorInvalidValue;
}

// ------------------------------------------------------------------ affine prep

// Eight lanes per 64-input group: lane j sums inputs 8j .. 8j+7 left to right,
// then the tree ((c0+c1)+(c2+c3))+((c4+c5)+(c6+c7)) by butterflies over the
// eight lanes (fp32 addition is commutative, so each butterfly level forms
// exactly the tree's pairs).
template <int XDT>
__global__ void __launch_bounds__(256) prep_affine_kernel(int M, int K, const void* __restrict__ x,
                                                          float* __restrict__ gsum, __half* __restrict__ x16)
{
    pdl_trigger();
    pdl_wait();
    const int G = K / 64;
    const long long gid = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 3;
    const int j = threadIdx.x & 7;
    const bool valid = gid < (long long)M * G;
    const int m = valid ? (int)(gid / G) : 0, g = valid ? (int)(gid % G) : 0;
    const size_t base = (size_t)m * K + (size_t)g * 64 + (size_t)j * 8;
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = valid ? load_x<XDT>(x, base + i) : 0.f;
    float c = v[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) c = __fadd_rn(c, v[i]);
    c = __fadd_rn(c, __shfl_xor_sync(0xffffffffu, c, 1));
    c = __fadd_rn(c, __shfl_xor_sync(0xffffffffu, c, 2));
    c = __fadd_rn(c, __shfl_xor_sync(0xffffffffu, c, 4));
    if (valid && j == 0) gsum[(size_t)m * G + g] = c;
    if (valid && x16) {
        __half2 h[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
        *reinterpret_cast<uint4*>(x16 + base) = *reinterpret_cast<uint4*>(h);
    }
}

cudaError_t launch_prep_affine(const LaunchCtx& c, int M, int K, const void* x, int x_dtype, float* gsum,
                               uint16_t* x16)
{
    const long long lanes = (long long)M * (K / 64) * 8;
    const int threads = 256;
    const unsigned blocks = (unsigned)((lanes + threads - 1) / threads);
    __half* h = reinterpret_cast<__half*>(x16);
    if (x_dtype == 0) return launch(prep_affine_kernel<0>, dim3(blocks), dim3(threads), 0, c, M, K, x, gsum, h);
    if (x_dtype == 1) return launch(prep_affine_kernel<1>, dim3(blocks), dim3(threads), 0, c, M, K, x, gsum, h);
    return launch(prep_affine_kernel<2>, dim3(blocks), dim3(threads), 0, c, M, K, x, gsum, h);
}

}  // namespace qmm
