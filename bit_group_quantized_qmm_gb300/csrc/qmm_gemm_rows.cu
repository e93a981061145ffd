// qmm_gemm_rows.cu -- the W4A8 GEMM for a few activation rows (M <= 16) on
// the CUDA cores: exact int32 group partials with dp4a, one pass over the
// packed weights for all rows.
//
// cactus PR #697 "SME2 acceleration for CQ4 matmul, prefill attention, and
// orthogonal embeddings", Summary: partials are raw integer dot products of
// the int4 weights and int8 codes, rescaled in fp32 per group; geistlib issue
// #500 "native W*A8 int8 GEMM for prefill", Design sketch: one activation
// quantization shared by the GEMV and the GEMM, no dequantized weights.
//
// GB300 design. At a handful of rows the GEMM is a weight stream (the whole
// lm_head blob per call) with at most 16 multiply-adds per weight: the tensor
// core path spends its time expanding nibbles per 128 x 64 block for one MMA,
// while the dp4a loop of the GEMV consumes each expanded weight word once per
// row from registers. So this kernel is the GEMV's structure with M rows:
// grid = 128-row tiles x K-slices, the slices of a tile forming one
// thread-block cluster; a producer warp issues the slice's packed chunks as
// 1-D bulk copies before the dependency wait (weights do not depend on the
// previous kernel); the compute warps stage the slice's activation codes
// (given as their exact fp16 image, the GEMM's operand format) as int8 in the
// dp4a order, then each thread takes one weight row and half the groups,
// expands each 16-byte nibble piece once and runs it against every row's
// codes. The halves meet in shared memory, the slices in the cluster's first
// CTA through distributed shared memory, in a fixed order: deterministic, no
// workspace, no atomics. Codebook (CQ4) blobs take the same loop with each
// piece's indices looked up in the matrix's 16 int8 levels, the codes staged
// in the lookup's order and cb_scale applied once per output.
//
// Shapes with many row tiles (an lm_head: thousands of tiles) run a streaming
// form instead: a grid of resident CTAs, each taking tiles t = blockIdx.x,
// blockIdx.x + gridDim.x, ... over the whole of K. The codes of all K are
// staged once per CTA, the producer streams the chunks of successive tiles
// through two rings of stages (one per half of the compute threads: half h
// takes one contiguous half of the groups of every tile), so a CTA pays its
// set-up once and never waits for a tile's first bytes after the first.
// The halves meet once per tile in shared memory; no K-split, no cluster.
#include <cuda_fp16.h>

#include "qmm.h"
#include "qmm_cq4.cuh"
#include "qmm_internal.h"
#include "qmm_ptx.cuh"

namespace qmm {

namespace {

constexpr int kComputeThreads = 256;
constexpr int kThreads = kComputeThreads + 32;   // + producer warp
constexpr int kTargetCtas = 2 * 152;
constexpr int kMaxCluster = 8;                    // portable cluster size

template <int GROUP, int MR>
struct Cfg {
    static constexpr int PP = GROUP / 32;         // 16-byte pieces per row and group
    static constexpr int CB = 64 * GROUP + 256;   // packed chunk bytes
    static constexpr int NG_MAX = GROUP == 64 ? 24 : 12;   // most chunks a CTA may hold
    // preferred chunks per CTA: with up to 4 rows the loop is light and long
    // CTAs keep more bytes in flight; with more rows, short CTAs give the
    // SM more of them to overlap (measured on the lm_head shape)
    static constexpr int NG_CAP = MR <= 4 ? NG_MAX : (GROUP == 64 ? 8 : 4);
};

__device__ __forceinline__ int nib_lo16(uint32_t w) { return (int)(((w << 4) ^ 0x80808080u) & 0xF0F0F0F0u); }
__device__ __forceinline__ int nib_hi16(uint32_t w) { return (int)((w ^ 0x80808080u) & 0xF0F0F0F0u); }
__device__ __forceinline__ void compute_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// Fixed header (same offsets in every CTA of a launch): the slices' partial
// sums [ksplit][MR][128] (used in the first CTA of a cluster), the halves'
// sums [MR][128], flags, the cluster barrier and one barrier per chunk.
__host__ __device__ inline size_t header_bytes(int ksplit, int mr, int ng_max)
{
    const size_t b = (size_t)ksplit * mr * 512 + (size_t)mr * 512 + 16 + 8 + 8 * (size_t)ng_max;
    return (b + 127) / 128 * 128;
}

size_t smem_bytes(int ksplit, int mr, int ng_max, int group, int cb)
{
    return header_bytes(ksplit, mr, ng_max) + (size_t)ng_max * cb + (size_t)ng_max * mr * group +
           (size_t)ng_max * mr * 4 + 16;
}

// int8 of an exact fp16 integer code
__device__ __forceinline__ uint32_t code_byte(uint16_t h)
{
    return (uint32_t)__half2int_rn(__ushort_as_half(h)) & 0xFFu;
}

// Grid (T, ksplit), cluster (1, ksplit): CTA (t, s) handles groups [g0, g1) of
// tile t for all M (<= MR) rows.
template <int GROUP, int MR, bool CQ>
__global__ void __launch_bounds__(kThreads)
    gemm_rows_kernel(int M, int N, int K, int ksplit, int ng_max, const uint8_t* __restrict__ blob,
                     const uint16_t* __restrict__ act16, const float* __restrict__ sx, float* __restrict__ Y,
                     int* status)
{
    using C = Cfg<GROUP, MR>;
    const int G = K / GROUP;
    const int t = blockIdx.x, s = blockIdx.y;
    const int g0 = (int)((long long)G * s / ksplit), g1 = (int)((long long)G * (s + 1) / ksplit);
    const int ng = g1 - g0;

    extern __shared__ __align__(128) uint8_t smem[];
    float* parts = reinterpret_cast<float*>(smem);                 // [ksplit][MR][128]
    float* red = parts + (size_t)ksplit * MR * 128;                 // [MR][128]
    int* flags = reinterpret_cast<int*>(red + MR * 128);           // [4]
    uint64_t* sums_in = reinterpret_cast<uint64_t*>(flags + 4);     // slices' sums arrived (first CTA)
    uint64_t* full = sums_in + 1;                                   // [ng_max]
    uint8_t* stages = smem + header_bytes(ksplit, MR, ng_max);
    uint8_t* aperm = stages + (size_t)ng_max * C::CB;               // [ng][MR][GROUP] codes, dp4a order
    float* sxs = reinterpret_cast<float*>(aperm + (size_t)ng_max * MR * GROUP);   // [ng][MR]
    volatile int* abort = flags;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    pdl_trigger();
    if (tid == 0) {
        for (int i = 0; i < ng; ++i) mbar_init(&full[i], 1);
        // the other slices' sums land with st.async, completing their bytes on
        // this barrier
        mbar_init(sums_in, 1);
        if (ksplit > 1 && s == 0) mbar_arrive_expect_tx(sums_in, (uint32_t)(ksplit - 1) * MR * 512u);
        flags[0] = 0;
        fence_barrier_init();
    }
    // the other slices arrive on sums_in only once it is initialised
    if (ksplit > 1)
        cluster_sync_all();
    else
        __syncthreads();

    if (warp == kComputeThreads / 32) {
        // producer: the whole slice, before the dependency wait
        if (lane == 0) {
            const uint8_t* src = blob + ((size_t)t * G + g0) * C::CB;
            const size_t n_chunks = (size_t)((N + 127) / 128) * G;
            for (int i = 0; i < ng; ++i) {
                // the chunk lies inside the blob (a skipped chunk leaves its
                // consumers to their bounded waits)
                if (!in_range((size_t)t * G + g0 + i < n_chunks, status)) continue;
                mbar_arrive_expect_tx(&full[i], C::CB);
                bulk_g2s(stages + (size_t)i * C::CB, src + (size_t)i * C::CB, C::CB, &full[i]);
            }
            // the CTA must not exit with copies in flight
            for (int i = 0; i < ng; ++i)
                if (!QMM_CHECKS || (size_t)t * G + g0 + i < n_chunks) mbar_wait(&full[i], 0, status, nullptr);
        }
        __syncwarp();
        return;
    }

    // ---------------------------------------------------------- stage codes
    Cq4Book book = {};
    if (CQ) book = cq4_load(blob + cq4_trailer_offset(N, K, GROUP));
    // warm the slice's codes in L2 first (a prefetch returns no data, so it
    // may run before the dependency wait)
    if (tid < M)
        bulk_prefetch_l2(act16 + (size_t)tid * K + (size_t)g0 * GROUP, (uint32_t)(ng * GROUP * 2));
    pdl_wait();   // codes and scales come from the previous kernel
    {
        constexpr int B8 = GROUP / 8;   // 8-blocks per group
        for (int w = tid; w < ng * MR * B8; w += kComputeThreads) {
            const int c8 = w % B8, rest = w / B8;
            const int m = rest % MR, i = rest / MR;
            uint2 perm = make_uint2(0u, 0u);
            if (m < M) {
                const uint4 hv = *reinterpret_cast<const uint4*>(act16 + (size_t)m * K + (size_t)(g0 + i) * GROUP +
                                                                 (size_t)c8 * 8);
                const uint32_t b0 = code_byte((uint16_t)hv.x), b1 = code_byte((uint16_t)(hv.x >> 16));
                const uint32_t b2 = code_byte((uint16_t)hv.y), b3 = code_byte((uint16_t)(hv.y >> 16));
                const uint32_t b4 = code_byte((uint16_t)hv.z), b5 = code_byte((uint16_t)(hv.z >> 16));
                const uint32_t b6 = code_byte((uint16_t)hv.w), b7 = code_byte((uint16_t)(hv.w >> 16));
                if (CQ)   // lookup order of an 8-block: k = 0, 2, 4, 6 | 1, 3, 5, 7
                    perm = make_uint2(b0 | (b2 << 8) | (b4 << 16) | (b6 << 24),
                                      b1 | (b3 << 8) | (b5 << 16) | (b7 << 24));
                else      // dp4a order of an 8-block: k = 0, 4, 1, 5 | 2, 6, 3, 7
                    perm = make_uint2(b0 | (b4 << 8) | (b1 << 16) | (b5 << 24),
                                      b2 | (b6 << 8) | (b3 << 16) | (b7 << 24));
            }
            *reinterpret_cast<uint2*>(aperm + ((size_t)i * MR + m) * GROUP + (size_t)c8 * 8) = perm;
        }
        for (int w = tid; w < ng * MR; w += kComputeThreads) {
            const int m = w % MR, i = w / MR;
            sxs[w] = m < M ? sx[(size_t)m * G + g0 + i] : 0.f;
        }
    }
    compute_sync();

    // ---------------------------------------------------------- partials
    const int r = tid & 127, h = tid >> 7;
    float acc[MR];
#pragma unroll
    for (int m = 0; m < MR; ++m) acc[m] = 0.f;
    for (int i = h; i < ng; i += 2) {
        if (!mbar_wait(&full[i], 0, status, abort)) break;
        const uint8_t* c = stages + (size_t)i * C::CB;
        // the row's GROUP weights as bytes: 16 * q in the blob's slot order
        // (symmetric) or the looked-up levels (codebook)
        int wv[8 * C::PP];
#pragma unroll
        for (int p = 0; p < C::PP; ++p) {
            const uint4 w = *reinterpret_cast<const uint4*>(c + p * 2048 + r * 16);
            if (CQ) {
                uint32_t lo, hi;
                cq4_expand(book, w.x, lo, hi);
                wv[8 * p + 0] = (int)lo;
                wv[8 * p + 1] = (int)hi;
                cq4_expand(book, w.y, lo, hi);
                wv[8 * p + 2] = (int)lo;
                wv[8 * p + 3] = (int)hi;
                cq4_expand(book, w.z, lo, hi);
                wv[8 * p + 4] = (int)lo;
                wv[8 * p + 5] = (int)hi;
                cq4_expand(book, w.w, lo, hi);
                wv[8 * p + 6] = (int)lo;
                wv[8 * p + 7] = (int)hi;
            } else {
                wv[8 * p + 0] = nib_lo16(w.x);
                wv[8 * p + 1] = nib_hi16(w.x);
                wv[8 * p + 2] = nib_lo16(w.y);
                wv[8 * p + 3] = nib_hi16(w.y);
                wv[8 * p + 4] = nib_lo16(w.z);
                wv[8 * p + 5] = nib_hi16(w.z);
                wv[8 * p + 6] = nib_lo16(w.w);
                wv[8 * p + 7] = nib_hi16(w.w);
            }
        }
        const float sw = __half2float(reinterpret_cast<const __half*>(c + 64 * GROUP)[r]);
        // one dp4a chain per row, interleaved piece by piece
        int dp[MR];
#pragma unroll
        for (int m = 0; m < MR; ++m) dp[m] = 0;
        const uint4* ap = reinterpret_cast<const uint4*>(aperm + (size_t)i * MR * GROUP);
#pragma unroll
        for (int p = 0; p < C::PP; ++p) {
#pragma unroll
            for (int m = 0; m < MR; ++m) {
                const uint4 a0 = ap[m * (GROUP / 16) + 2 * p], a1 = ap[m * (GROUP / 16) + 2 * p + 1];
                dp[m] = __dp4a(wv[8 * p + 0], (int)a0.x, dp[m]);
                dp[m] = __dp4a(wv[8 * p + 1], (int)a0.y, dp[m]);
                dp[m] = __dp4a(wv[8 * p + 2], (int)a0.z, dp[m]);
                dp[m] = __dp4a(wv[8 * p + 3], (int)a0.w, dp[m]);
                dp[m] = __dp4a(wv[8 * p + 4], (int)a1.x, dp[m]);
                dp[m] = __dp4a(wv[8 * p + 5], (int)a1.y, dp[m]);
                dp[m] = __dp4a(wv[8 * p + 6], (int)a1.z, dp[m]);
                dp[m] = __dp4a(wv[8 * p + 7], (int)a1.w, dp[m]);
            }
        }
#pragma unroll
        for (int m = 0; m < MR; ++m) acc[m] = fmaf((float)(CQ ? dp[m] : dp[m] >> 4), sw * sxs[i * MR + m], acc[m]);
    }

    // ---------------------------------------------------------- reduce, store
    if (h == 1) {
#pragma unroll
        for (int m = 0; m < MR; ++m) red[m * 128 + r] = acc[m];
    }
    compute_sync();
    const int n = t * 128 + r;
    if (h == 0) {
#pragma unroll
        for (int m = 0; m < MR; ++m) {
            const float v = acc[m] + red[m * 128 + r];
            if (ksplit == 1) {
                if (m < M && n < N) Y[(size_t)m * N + n] = CQ ? v * book.scale : v;
            } else {
                parts[((size_t)s * MR + m) * 128 + r] = v;   // this slice's sums, locally first
            }
        }
    }
    if (ksplit > 1) {
        if (s != 0) {
            // the slice's MR x 128 sums go to the first CTA of the cluster as
            // asynchronous 16-byte stores that complete on its barrier
            compute_sync();
            const float4* src = reinterpret_cast<const float4*>(parts + (size_t)s * MR * 128);
            const uint32_t dst = map_shared_rank(smem_u32(parts + (size_t)s * MR * 128), 0u);
            const uint32_t bar = map_shared_rank(smem_u32(sums_in), 0u);
            for (int j = tid; j < MR * 32; j += kComputeThreads) st_async_cluster_v4(dst + 16u * j, src[j], bar);
        } else if (tid < 128) {
            // the first CTA adds the slices in order once all have arrived
            mbar_wait_cluster(sums_in, 0, status);
#pragma unroll
            for (int m = 0; m < MR; ++m) {
                float v = 0.f;
                for (int k = 0; k < ksplit; ++k) v += parts[((size_t)k * MR + m) * 128 + tid];
                if (m < M && t * 128 + tid < N) Y[(size_t)m * N + t * 128 + tid] = CQ ? v * book.scale : v;
            }
        }
    }
}

// ------------------------------------------------------------------ streaming form
constexpr int kStreamMinTiles = 512;          // row tiles from which a launch streams
constexpr int kStreamCodesMax = 64 * 1024;    // staged code bytes a CTA may hold (K x rows)

// RPT weight rows per thread (r, r + 128 / RPT): each broadcast load of codes
// from shared memory feeds 8 * RPT dp4a. The 256 compute threads form
// NS = 2 * RPT group sets of 128 / RPT threads; set q takes groups
// [G * q / NS, G * (q + 1) / NS) of every tile through its own ring of RS stages.
template <int GROUP, int RPT>
struct StreamCfg {
    static constexpr int PP = GROUP / 32;
    static constexpr int CB = 64 * GROUP + 256;
    static constexpr int NS = 2 * RPT;                     // group sets
    static constexpr int TPS = kComputeThreads / NS;       // threads per set
    // stages per set: about 50 KB in all, at least two per set
    static constexpr int RS = (GROUP == 64 ? 12 : 6) / NS < 2 ? 2 : (GROUP == 64 ? 12 : 6) / NS;
};

// Header: the sums of sets 1 .. NS-1 [2][NS-1][MR][128] (double-buffered by
// tile), flags, full and empty barriers of every ring; padded to 128 bytes.
__host__ __device__ inline size_t stream_header_bytes(int mr, int ns, int rs)
{
    const size_t b = (size_t)2 * (ns - 1) * mr * 512 + 16 + (size_t)2 * ns * rs * 8;
    return (b + 127) / 128 * 128;
}

size_t stream_smem_bytes(int G, int mr, int group, int cb, int ns, int rs)
{
    return stream_header_bytes(mr, ns, rs) + (size_t)ns * rs * cb + (size_t)G * mr * group + (size_t)G * mr * 4 + 16;
}

// Grid (P): CTA b takes row tiles b, b + P, ... with all G groups; set q of
// the compute threads reads only its own ring, so each ring has one consumer
// set and the stage phases advance in order.
template <int GROUP, int MR, int RPT, bool CQ>
__global__ void __launch_bounds__(kThreads)
    gemm_rows_stream_kernel(int M, int N, int K, const uint8_t* __restrict__ blob, const uint16_t* __restrict__ act16,
                            const float* __restrict__ sx, float* __restrict__ Y, int* status)
{
    using C = StreamCfg<GROUP, RPT>;
    constexpr int NS = C::NS, RS = C::RS, RSTRIDE = 128 / RPT;
    const int G = K / GROUP, T = (N + 127) / 128;

    extern __shared__ __align__(128) uint8_t smem[];
    float* red = reinterpret_cast<float*>(smem);                              // [2][NS-1][MR][128]
    int* flags = reinterpret_cast<int*>(red + 2 * (NS - 1) * MR * 128);        // [4]
    uint64_t* full = reinterpret_cast<uint64_t*>(flags + 4);                   // [NS][RS]
    uint64_t* empty = full + NS * RS;                                          // [NS][RS]
    uint8_t* stages = smem + stream_header_bytes(MR, NS, RS);                  // [NS][RS][CB]
    uint8_t* aperm = stages + (size_t)NS * RS * C::CB;                         // [G][MR][GROUP] codes, dp4a order
    float* sxs = reinterpret_cast<float*>(aperm + (size_t)G * MR * GROUP);    // [G][MR]
    volatile int* abort = flags;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    pdl_trigger();
    if (tid == 0) {
        for (int i = 0; i < NS * RS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], C::TPS / 32);   // the warps of one set read each stage
        }
        flags[0] = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kComputeThreads / 32) {
        // producer: the chunks of all sets interleaved, tile after tile;
        // weights do not depend on the previous kernel, so this starts before
        // the dependency wait
        if (lane == 0) {
            // per ring: chunks issued, next stage, parity of its next empty wait
            uint32_t n[NS], ph[NS];
            int st[NS];
#pragma unroll
            for (int q = 0; q < NS; ++q) {
                n[q] = 0u;
                ph[q] = 0u;
                st[q] = 0;
            }
            const int imax = (G + NS - 1) / NS;
            bool stop = false;
            for (int t = blockIdx.x; t < T && !stop; t += gridDim.x) {
                const uint8_t* tile = blob + (size_t)t * G * C::CB;
                for (int i = 0; i < imax && !stop; ++i) {
#pragma unroll
                    for (int q = 0; q < NS; ++q) {
                        const int ga = G * q / NS, gz = G * (q + 1) / NS;
                        if (stop || ga + i >= gz) continue;
                        if (n[q] >= (uint32_t)RS && !mbar_wait(&empty[q * RS + st[q]], ph[q], status, abort)) {
                            stop = true;
                            continue;
                        }
                        if (!in_range((size_t)t * G + ga + i < (size_t)T * G, status)) {
                            stop = true;
                            continue;
                        }
                        uint64_t* f = &full[q * RS + st[q]];
                        mbar_arrive_expect_tx(f, C::CB);
                        bulk_g2s(stages + (size_t)(q * RS + st[q]) * C::CB, tile + (size_t)(ga + i) * C::CB, C::CB, f);
                        ++n[q];
                        if (++st[q] == RS) {
                            st[q] = 0;
                            if (n[q] > (uint32_t)RS) ph[q] ^= 1u;
                        }
                    }
                }
            }
            // the CTA must not exit with copies in flight: wait for the last ones
#pragma unroll
            for (int q = 0; q < NS; ++q)
                for (uint32_t c = n[q] > (uint32_t)RS ? n[q] - RS : 0u; c < n[q]; ++c)
                    mbar_wait(&full[q * RS + c % RS], (c / RS) & 1u, status, nullptr);
        }
        __syncwarp();
        return;
    }

    // ---------------------------------------------------------- stage codes (all of K)
    Cq4Book book = {};
    if (CQ) book = cq4_load(blob + cq4_trailer_offset(N, K, GROUP));
    if (tid < M) bulk_prefetch_l2(act16 + (size_t)tid * K, (uint32_t)(K * 2));
    pdl_wait();   // codes and scales come from the previous kernel
    {
        constexpr int B8 = GROUP / 8;   // 8-blocks per group
        for (int w = tid; w < G * MR * B8; w += kComputeThreads) {
            const int c8 = w % B8, rest = w / B8;
            const int m = rest % MR, i = rest / MR;
            uint2 perm = make_uint2(0u, 0u);
            if (m < M) {
                const uint4 hv =
                    *reinterpret_cast<const uint4*>(act16 + (size_t)m * K + (size_t)i * GROUP + (size_t)c8 * 8);
                const uint32_t b0 = code_byte((uint16_t)hv.x), b1 = code_byte((uint16_t)(hv.x >> 16));
                const uint32_t b2 = code_byte((uint16_t)hv.y), b3 = code_byte((uint16_t)(hv.y >> 16));
                const uint32_t b4 = code_byte((uint16_t)hv.z), b5 = code_byte((uint16_t)(hv.z >> 16));
                const uint32_t b6 = code_byte((uint16_t)hv.w), b7 = code_byte((uint16_t)(hv.w >> 16));
                if (CQ)   // lookup order of an 8-block: k = 0, 2, 4, 6 | 1, 3, 5, 7
                    perm = make_uint2(b0 | (b2 << 8) | (b4 << 16) | (b6 << 24),
                                      b1 | (b3 << 8) | (b5 << 16) | (b7 << 24));
                else      // dp4a order of an 8-block: k = 0, 4, 1, 5 | 2, 6, 3, 7
                    perm = make_uint2(b0 | (b4 << 8) | (b1 << 16) | (b5 << 24),
                                      b2 | (b6 << 8) | (b3 << 16) | (b7 << 24));
            }
            *reinterpret_cast<uint2*>(aperm + ((size_t)i * MR + m) * GROUP + (size_t)c8 * 8) = perm;
        }
        for (int w = tid; w < G * MR; w += kComputeThreads) {
            const int m = w % MR, i = w / MR;
            sxs[w] = m < M ? sx[(size_t)m * G + i] : 0.f;
        }
    }
    compute_sync();

    // ---------------------------------------------------------- tiles
    const int q = tid / C::TPS, r = tid % C::TPS;   // set, first weight row
    const int ga = G * q / NS, nq = G * (q + 1) / NS - ga;
    uint64_t* fullq = full + q * RS;
    uint64_t* emptyq = empty + q * RS;
    const uint8_t* stagesq = stages + (size_t)q * RS * C::CB;
    int st = 0;
    uint32_t ph = 0u;
    bool ok = true;
    int lt = 0;
    for (int t = blockIdx.x; t < T; t += gridDim.x, ++lt) {
        float acc[RPT][MR];
#pragma unroll
        for (int rr = 0; rr < RPT; ++rr)
#pragma unroll
            for (int m = 0; m < MR; ++m) acc[rr][m] = 0.f;
        // after a failed wait the loop still runs every tile's barrier (all
        // sets must meet), with no further waits or stores
        for (int i = 0; i < nq && ok; ++i) {
            if (!mbar_wait(&fullq[st], ph, status, abort)) {
                ok = false;
                break;
            }
            const uint8_t* c = stagesq + (size_t)st * C::CB;
            const int g = ga + i;
            float sw[RPT];
#pragma unroll
            for (int rr = 0; rr < RPT; ++rr)
                sw[rr] = __half2float(reinterpret_cast<const __half*>(c + 64 * GROUP)[r + RSTRIDE * rr]);
            int dp[RPT][MR];
#pragma unroll
            for (int rr = 0; rr < RPT; ++rr)
#pragma unroll
                for (int m = 0; m < MR; ++m) dp[rr][m] = 0;
            const uint4* ap = reinterpret_cast<const uint4*>(aperm + (size_t)g * MR * GROUP);
#pragma unroll
            for (int p = 0; p < C::PP; ++p) {
                // the rows' 32 weights of this piece as bytes: 16 * q in the
                // blob's slot order (symmetric) or the looked-up levels (codebook)
                int wv[RPT][8];
#pragma unroll
                for (int rr = 0; rr < RPT; ++rr) {
                    const uint4 w = *reinterpret_cast<const uint4*>(c + p * 2048 + (r + RSTRIDE * rr) * 16);
                    if (CQ) {
                        uint32_t lo, hi;
                        cq4_expand(book, w.x, lo, hi);
                        wv[rr][0] = (int)lo;
                        wv[rr][1] = (int)hi;
                        cq4_expand(book, w.y, lo, hi);
                        wv[rr][2] = (int)lo;
                        wv[rr][3] = (int)hi;
                        cq4_expand(book, w.z, lo, hi);
                        wv[rr][4] = (int)lo;
                        wv[rr][5] = (int)hi;
                        cq4_expand(book, w.w, lo, hi);
                        wv[rr][6] = (int)lo;
                        wv[rr][7] = (int)hi;
                    } else {
                        wv[rr][0] = nib_lo16(w.x);
                        wv[rr][1] = nib_hi16(w.x);
                        wv[rr][2] = nib_lo16(w.y);
                        wv[rr][3] = nib_hi16(w.y);
                        wv[rr][4] = nib_lo16(w.z);
                        wv[rr][5] = nib_hi16(w.z);
                        wv[rr][6] = nib_lo16(w.w);
                        wv[rr][7] = nib_hi16(w.w);
                    }
                }
                if (p == C::PP - 1) {
                    // every byte of the stage is in registers: release it
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&emptyq[st]);
                }
#pragma unroll
                for (int m = 0; m < MR; ++m) {
                    const uint4 a0 = ap[m * (GROUP / 16) + 2 * p], a1 = ap[m * (GROUP / 16) + 2 * p + 1];
#pragma unroll
                    for (int rr = 0; rr < RPT; ++rr) {
                        dp[rr][m] = __dp4a(wv[rr][0], (int)a0.x, dp[rr][m]);
                        dp[rr][m] = __dp4a(wv[rr][1], (int)a0.y, dp[rr][m]);
                        dp[rr][m] = __dp4a(wv[rr][2], (int)a0.z, dp[rr][m]);
                        dp[rr][m] = __dp4a(wv[rr][3], (int)a0.w, dp[rr][m]);
                        dp[rr][m] = __dp4a(wv[rr][4], (int)a1.x, dp[rr][m]);
                        dp[rr][m] = __dp4a(wv[rr][5], (int)a1.y, dp[rr][m]);
                        dp[rr][m] = __dp4a(wv[rr][6], (int)a1.z, dp[rr][m]);
                        dp[rr][m] = __dp4a(wv[rr][7], (int)a1.w, dp[rr][m]);
                    }
                }
            }
            if (++st == RS) {
                st = 0;
                ph ^= 1u;
            }
#pragma unroll
            for (int rr = 0; rr < RPT; ++rr)
#pragma unroll
                for (int m = 0; m < MR; ++m)
                    acc[rr][m] = fmaf((float)(CQ ? dp[rr][m] : dp[rr][m] >> 4), sw[rr] * sxs[g * MR + m], acc[rr][m]);
        }
        // the sets meet: sets 1 .. NS-1 park their sums (buffer by tile parity,
        // so a set one tile ahead never overwrites unread sums), set 0 adds
        // them in set order and stores
        float* rb = red + (size_t)(lt & 1) * (NS - 1) * MR * 128;
        if (q > 0) {
#pragma unroll
            for (int rr = 0; rr < RPT; ++rr)
#pragma unroll
                for (int m = 0; m < MR; ++m) rb[((size_t)(q - 1) * MR + m) * 128 + r + RSTRIDE * rr] = acc[rr][m];
        }
        compute_sync();
        if (q == 0 && ok) {
#pragma unroll
            for (int rr = 0; rr < RPT; ++rr) {
                const int row = r + RSTRIDE * rr, n = t * 128 + row;
#pragma unroll
                for (int m = 0; m < MR; ++m) {
                    float v = acc[rr][m];
#pragma unroll
                    for (int k = 0; k < NS - 1; ++k) v += rb[((size_t)k * MR + m) * 128 + row];
                    if (m < M && n < N) Y[(size_t)m * N + n] = CQ ? v * book.scale : v;
                }
            }
        }
    }
}

// Two weight rows per thread from 4 activation rows up: with one, the code
// loads keep the shared-memory pipe about as busy as the dp4a pipe (measured
// on the lm_head shape, M = 8: 68.8 -> 65.0 us; M = 16: 124 -> 119 us). One
// row for M <= 2, where the weight stream is the limit.
template <int MR>
constexpr int stream_rpt()
{
    return MR >= 4 ? 2 : 1;
}

template <int GROUP, int MR, bool CQ>
cudaError_t run_stream(const LaunchCtx& c, int M, int N, int K, const uint8_t* blob, const uint16_t* act16,
                       const float* sx, float* Y)
{
    constexpr int RPT = stream_rpt<MR>();
    using C = StreamCfg<GROUP, RPT>;
    auto kern = gemm_rows_stream_kernel<GROUP, MR, RPT, CQ>;
    const int T = (N + 127) / 128, G = K / GROUP;
    const size_t smem = stream_smem_bytes(G, MR, GROUP, C::CB, C::NS, C::RS);
    static KernelSmem configured;
    cudaError_t e = ensure_smem(configured, c, kern, smem);
    if (e != cudaSuccess) return e;
    // blocks per SM for this shared-memory size (the same on every supported
    // device), cached as one word: shared-memory bytes << 8 | blocks
    static std::atomic<uint64_t> occ_cache{0};
    const uint64_t cached = occ_cache.load(std::memory_order_relaxed);
    int nb = (cached >> 8) == (uint64_t)smem ? (int)(cached & 0xFF) : 0;
    if (nb == 0) {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kern, kThreads, smem);
        if (e != cudaSuccess) return e;
        if (nb < 1) return cudaErrorNotSupported;
        occ_cache.store(((uint64_t)smem << 8) | (uint64_t)(nb & 0xFF), std::memory_order_relaxed);
    }
    const int P = T < nb * c.num_sms ? T : nb * c.num_sms;
    return launch(kern, dim3(P), dim3(kThreads), smem, c, M, N, K, blob, act16, sx, Y, c.status);
}

template <int GROUP, int MR, bool CQ>
cudaError_t run(const LaunchCtx& c, int M, int N, int K, const uint8_t* blob, const uint16_t* act16,
                const float* sx, float* Y)
{
    using C = Cfg<GROUP, MR>;
    auto kern = gemm_rows_kernel<GROUP, MR, CQ>;
    const int T = (N + 127) / 128, G = K / GROUP;
    if (T >= kStreamMinTiles && (size_t)K * MR <= (size_t)kStreamCodesMax)
        return run_stream<GROUP, MR, CQ>(c, M, N, K, blob, act16, sx, Y);
    int ks = (kTargetCtas + T - 1) / T;
    const int ks_ng = (G + C::NG_CAP - 1) / C::NG_CAP;
    if (ks < ks_ng) ks = ks_ng;
    if (ks > G) ks = G;
    if (ks > kMaxCluster) ks = kMaxCluster;
    if (ks < 1) ks = 1;
    const int ng_max = (G + ks - 1) / ks;
    if (ng_max > C::NG_MAX) return cudaErrorNotSupported;   // K too large: the tensor-core path takes it
    const size_t smem = smem_bytes(ks, MR, ng_max, GROUP, C::CB);
    static KernelSmem configured;
    const cudaError_t e = ensure_smem(configured, c, kern, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(T, ks);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = c.stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 1;
    attr[na].val.clusterDim.y = ks;
    attr[na].val.clusterDim.z = 1;
    ++na;
    if (c.pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, M, N, K, ks, ng_max, blob, act16, sx, Y, c.status);
}

template <int GROUP, bool CQ>
cudaError_t dispatch(const LaunchCtx& c, int M, int N, int K, const uint8_t* blob, const uint16_t* act16,
                     const float* sx, float* Y)
{
    if (M <= 2) return run<GROUP, 2, CQ>(c, M, N, K, blob, act16, sx, Y);
    if (M <= 4) return run<GROUP, 4, CQ>(c, M, N, K, blob, act16, sx, Y);
    if (M <= 8) return run<GROUP, 8, CQ>(c, M, N, K, blob, act16, sx, Y);
    if (M <= 16) return run<GROUP, 16, CQ>(c, M, N, K, blob, act16, sx, Y);
    return cudaErrorNotSupported;
}

}  // namespace

cudaError_t launch_gemm_rows(const LaunchCtx& c, bool cq4, int group, int M, int N, int K, const uint8_t* blob,
                             const uint16_t* act16, const float* sx, float* Y)
{
    if (group == 64)
        return cq4 ? dispatch<64, true>(c, M, N, K, blob, act16, sx, Y)
                   : dispatch<64, false>(c, M, N, K, blob, act16, sx, Y);
    if (group == 128)
        return cq4 ? dispatch<128, true>(c, M, N, K, blob, act16, sx, Y)
                   : dispatch<128, false>(c, M, N, K, blob, act16, sx, Y);
    return cudaErrorInvalidValue;
}

}  // namespace qmm
