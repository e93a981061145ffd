// qmm_gemv_fused.cu -- one-kernel M = 1 decode GEMV of the symmetric W4A8
// variant: activation prepass and weight streaming in a single launch.
//
// cactus PR #697 "SME2 acceleration for CQ4 matmul, prefill attention, and
// orthogonal embeddings", Summary: the M = 1 path is one dispatch in two
// phases — phase A applies the Hadamard transform and quantizes the
// activations to int8 per group, phase B streams the packed nibbles through
// the integer partials leaf — and the dispatch itself was a measurable tax on
// calls of tens of microseconds.
//
// GB300 design. A CTA owns one 128-row tile and a contiguous range of its
// groups. Before waiting on the previous kernel (programmatic dependent
// launch) a producer warp issues 1-D bulk copies of all the CTA's packed
// chunks into shared memory, so a layer's weights stream while its
// predecessor finishes. After the wait, phase A quantizes only the CTA's own
// groups (quantization is per group, so no other CTA's input is needed), writing
// the codes straight into the permuted order the dp4a expansion reads;
// phase B is the exact int32 group-partial loop of the plain GEMV. The
// K-slices of a tile form one thread-block cluster and are summed through
// distributed shared memory in a fixed order by the cluster's first CTA: no
// global workspace, no atomics, deterministic results.
//
// Codebook (CQ4) blobs run the same kernel: phase A writes the codes in the
// order the table lookup consumes them, phase B looks the nibbles up in the
// matrix's 16 int8 levels, and the sum is multiplied by cb_scale once.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "qmm.h"
#include "qmm_cq4.cuh"
#include "qmm_internal.h"
#include "qmm_ptx.cuh"

namespace qmm {

namespace {

constexpr int kComputeThreads = 256;
constexpr int kThreads = kComputeThreads + 32;   // + producer warp
// Launch shape, measured on the 32-layer Gemma-shaped decode step (ms per
// step, alternating best-of rounds). K-slices per tile: ceil(kTargetCtas /
// tiles), at most one 16-CTA cluster (about 1.3 CTAs per SM: 0.380 against
// 0.426 at 2 per SM), raised so that a CTA holds at most kMaxGroupsPerCta
// groups as long as the grid stays within kCtasPerSm resident CTAs per SM;
// and when the whole grid fits that way, each CTA takes at least
// kMinSmemPerCta of shared memory, so that no SM holds more than kCtasPerSm of
// them (the block scheduler otherwise stacked up to 5 gate_up CTAs on an SM
// whose weight copies then landed last). K-slices of gate_up / down / q / o
// become 4 / 16 / 13 / 16 (from 3 / 16 / 13 / 16): 0.361 against 0.382 with
// at most 4 CTAs per SM, 0.366 with at most 3, 0.394 with at most 5; at most
// 5 or 4 groups per CTA 0.373 / 0.374, the split alone 0.391, a floor allowing
// only 2 per SM 0.43.
constexpr int kTargetCtas = 200;
constexpr int kMaxGroupsPerCta = 6;
constexpr int kCtasPerSm = 4;
constexpr size_t kMinSmemPerCta = 45 * 1024;   // 5 x (45 + 1) KB exceeds an SM's 228 KB
constexpr int kMaxCluster = 16;
constexpr int kMaxNg = 48;                          // chunks a CTA may hold
// parts (16 x 512 B), red (512 B), flags (16 B), kMaxNg barriers, padded to 128 B
constexpr size_t kHeaderBytes = 9216;
static_assert(kHeaderBytes % 128 == 0 && kHeaderBytes >= (kMaxCluster + 1) * 512 + 16 + 8 * kMaxNg, "header layout");

template <int GROUP>
struct Cfg {
    static constexpr int PP = GROUP / 32;
    static constexpr int CB = 64 * GROUP + 256;
};

__device__ __forceinline__ int nib_lo16(uint32_t w) { return (int)(((w << 4) ^ 0x80808080u) & 0xF0F0F0F0u); }
__device__ __forceinline__ int nib_hi16(uint32_t w) { return (int)((w ^ 0x80808080u) & 0xF0F0F0F0u); }
__device__ __forceinline__ void compute_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

template <int XDT>
__device__ __forceinline__ float load_in(const void* x, size_t i)
{
    if (XDT == 0) return static_cast<const float*>(x)[i];
    if (XDT == 1) return __half2float(static_cast<const __half*>(x)[i]);
    return __bfloat162float(static_cast<const __nv_bfloat16*>(x)[i]);
}

// The weight matrices of one launch (siblings share x, K and the group size):
// matrix i owns grid rows [tile0[i], tile0[i + 1]).
struct FusedSet {
    int count;
    int tile0[kMaxSiblings + 1];
    int N[kMaxSiblings];
    const uint8_t* blob[kMaxSiblings];
    float* y[kMaxSiblings];
};

size_t smem_bytes(int ring, int cb, int ng, int group)
{
    return kHeaderBytes + (size_t)ring * cb + (size_t)ng * group + (size_t)ng * 4 + 16;
}

// Grid (sum of the matrices' tiles, ksplit), cluster (1, ksplit): CTA (b, s)
// handles groups [g0, g1) of tile t of the matrix that owns grid row b.
// EPL inputs per lane in phase A: 8 for long slices; GROUP/32 (a whole warp per
// group, fewer serial divisions per lane) for short ones.
template <int GROUP, int XDT, int EPL, bool CQ>
__global__ void __launch_bounds__(kThreads)
    gemv_fused_kernel(const __grid_constant__ FusedSet set, int K, int ksplit, int hadamard, float rot_scale,
                      const void* __restrict__ x, int8_t* __restrict__ a_out, float* __restrict__ sx_out, int* status)
{
    using C = Cfg<GROUP>;
    const int G = K / GROUP;
    int mi = 0;
    while (mi + 1 < set.count && (int)blockIdx.x >= set.tile0[mi + 1]) ++mi;
    const int t = blockIdx.x - set.tile0[mi], s = blockIdx.y;
    const int N = set.N[mi];
    const uint8_t* __restrict__ blob = set.blob[mi];
    float* __restrict__ y = set.y[mi];
    const int g0 = (int)((long long)G * s / ksplit), g1 = (int)((long long)G * (s + 1) / ksplit);
    const int ng = g1 - g0;
    const int ring = ng;   // the launcher keeps a CTA's whole slice resident

    // Fixed offsets first: every CTA of the cluster stores its partial sums
    // into the first CTA's `parts` at the same offset, and ng differs between
    // the K-slices.
    extern __shared__ __align__(128) uint8_t smem[];
    float* parts = reinterpret_cast<float*>(smem);                            // [kMaxCluster][128] (rank 0)
    float* red = parts + kMaxCluster * 128;                                    // [128]
    int* flags = reinterpret_cast<int*>(red + 128);                            // [2]
    uint64_t* sums_in = reinterpret_cast<uint64_t*>(flags + 2);                // slices' sums arrived (rank 0)
    uint64_t* full = sums_in + 1;                                              // [kMaxNg]
    uint8_t* stages = smem + kHeaderBytes;
    uint8_t* aperm = stages + (size_t)ring * C::CB;                            // permuted codes, ng*GROUP bytes
    float* sxs = reinterpret_cast<float*>(aperm + (size_t)ng * GROUP);        // [ng]
    volatile int* abort = flags;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    pdl_trigger();
    if (tid == 0) {
        for (int i = 0; i < ring; ++i) mbar_init(&full[i], 1);
        // the other slices' sums land with st.async, each completing its bytes
        // on this barrier; the phase completes when all (ksplit - 1) x 512
        // bytes are in
        mbar_init(sums_in, 1);
        if (ksplit > 1 && s == 0) mbar_arrive_expect_tx(sums_in, (uint32_t)(ksplit - 1) * 512u);
        flags[0] = 0;
        fence_barrier_init();
    }
    // the other slices may arrive on sums_in only once it is initialised: a
    // cluster barrier here, before the dependency wait, keeps it off the
    // critical path
    if (ksplit > 1)
        cluster_sync_all();
    else
        __syncthreads();

    if (warp == kComputeThreads / 32) {
        // producer: the whole slice, before the dependency wait
        if (lane == 0) {
            const uint8_t* src = blob + ((size_t)t * G + g0) * C::CB;
            for (int i = 0; i < ng; ++i) {
                // the chunk lies inside the blob (a skipped chunk is never
                // waited for below: its consumers' bounded waits run out)
                if (!in_range((size_t)t * G + g0 + i < (size_t)((N + 127) / 128) * G, status)) continue;
                mbar_arrive_expect_tx(&full[i], C::CB);
                bulk_g2s(stages + (size_t)i * C::CB, src + (size_t)i * C::CB, C::CB, &full[i]);
            }
            // the CTA must not exit with copies in flight
            for (int i = 0; i < ng; ++i)
                if (!QMM_CHECKS || (size_t)t * G + g0 + i < (size_t)((N + 127) / 128) * G)
                    mbar_wait(&full[i], 0, status, nullptr);
        }
        __syncwarp();
    } else {
        Cq4Book book = {};
        if (CQ) book = cq4_load(blob + cq4_trailer_offset(N, K, GROUP));
        // ---------------------------------------------------------- phase A
        // LPG lanes per group, EPL consecutive inputs per lane; GPW groups per
        // warp. Transform stages below EPL run inside the lane, the others
        // across lanes, in the ascending order of the page's butterfly.
        // The slice of x is warmed in L2 before the dependency wait (a
        // prefetch returns no data; the loads after the wait read the lines
        // the previous kernel wrote).
        constexpr int XSZ = XDT == 0 ? 4 : 2;
        if (tid == 0)
            bulk_prefetch_l2(static_cast<const uint8_t*>(x) + (size_t)g0 * GROUP * XSZ, (uint32_t)(ng * GROUP * XSZ));
        pdl_wait();
        constexpr int LPG = GROUP / EPL, GPW = 32 / LPG;
        static_assert(LPG <= 32 && EPL >= 2, "phase A layout");
        const int sub = lane / LPG, cl = lane % LPG;
        for (int i0 = warp * GPW; i0 < ng; i0 += (kComputeThreads / 32) * GPW) {
            const int i = i0 + sub;
            const bool valid = i < ng;
            const int g = g0 + (valid ? i : 0);
            const size_t base = (size_t)g * GROUP + (size_t)cl * EPL;
            float v[EPL];
            if (XDT == 0 && EPL == 8) {
                const float4 p0 = reinterpret_cast<const float4*>(static_cast<const float*>(x) + base)[0];
                const float4 p1 = reinterpret_cast<const float4*>(static_cast<const float*>(x) + base)[1];
                v[0] = p0.x; v[1] = p0.y; v[2] = p0.z; v[3] = p0.w;
                v[4] = p1.x; v[5] = p1.y; v[6] = p1.z; v[7] = p1.w;
            } else if (XDT == 0 && EPL == 4) {
                const float4 p0 = *reinterpret_cast<const float4*>(static_cast<const float*>(x) + base);
                v[0] = p0.x; v[1] = p0.y; v[2] = p0.z; v[3] = p0.w;
            } else if (XDT == 0 && EPL == 2) {
                const float2 p0 = *reinterpret_cast<const float2*>(static_cast<const float*>(x) + base);
                v[0] = p0.x; v[1] = p0.y;
            } else {
#pragma unroll
                for (int e = 0; e < EPL; ++e) v[e] = load_in<XDT>(x, base + e);
            }
            if (hadamard) {
#pragma unroll
                for (int h = 1; h < EPL; h <<= 1)
#pragma unroll
                    for (int e = 0; e < EPL; ++e)
                        if ((e & h) == 0) {
                            const float lo = v[e], hi = v[e + h];
                            v[e] = __fadd_rn(lo, hi);
                            v[e + h] = __fsub_rn(lo, hi);
                        }
#pragma unroll
                for (int lm = 1; lm < LPG; lm <<= 1) {
                    const bool upper = (cl & lm) != 0;
#pragma unroll
                    for (int e = 0; e < EPL; ++e) {
                        const float o = __shfl_xor_sync(0xffffffffu, v[e], lm);
                        v[e] = upper ? __fsub_rn(o, v[e]) : __fadd_rn(v[e], o);
                    }
                }
            }
            float amax = 0.f;
#pragma unroll
            for (int e = 0; e < EPL; ++e) amax = fmaxf(amax, fabsf(v[e]));
#pragma unroll
            for (int o = 1; o < LPG; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            float scale = 0.f;
            uint32_t b[EPL];
            if (amax == 0.f) {
#pragma unroll
                for (int e = 0; e < EPL; ++e) b[e] = 0;
            } else {
                const float sc = __fdiv_rn(amax, 127.0f);
#pragma unroll
                for (int e = 0; e < EPL; ++e) {
                    float r = rintf(__fdiv_rn(v[e], sc));
                    r = fminf(fmaxf(r, -127.f), 127.f);
                    b[e] = (uint32_t)(int)r & 0xFFu;
                }
                scale = __fmul_rn(sc, rot_scale);
            }
            if (valid) {
                uint8_t* blk = aperm + (size_t)i * GROUP + (size_t)(cl * EPL / 8) * 8;
                if (EPL == 8 && CQ) {
                    // lookup order of an 8-block: k = 0, 2, 4, 6 | 1, 3, 5, 7
                    *reinterpret_cast<uint2*>(blk) = make_uint2(b[0] | (b[2] << 8) | (b[4] << 16) | (b[6] << 24),
                                                                b[1] | (b[3] << 8) | (b[5] << 16) | (b[7] << 24));
                } else if (EPL == 8) {
                    // dp4a order of an 8-block: k = 0, 4, 1, 5 | 2, 6, 3, 7
                    *reinterpret_cast<uint2*>(blk) = make_uint2(b[0] | (b[4] << 8) | (b[1] << 16) | (b[5] << 24),
                                                                b[2] | (b[6] << 8) | (b[3] << 16) | (b[7] << 24));
                } else {
                    // this lane's EPL inputs k = k0 .. k0+EPL-1 of an 8-block, at
                    // their positions in the dp4a (or lookup) order
#pragma unroll
                    for (int e = 0; e < EPL; ++e) {
                        const int k = (cl * EPL + e) & 7;
                        blk[CQ ? 4 * (k & 1) + (k >> 1) : 2 * (k & 3) + (k >> 2)] = (uint8_t)b[e];
                    }
                }
                if (a_out) {
                    if (EPL == 8)
                        *reinterpret_cast<uint2*>(a_out + base) =
                            make_uint2(b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24),
                                       b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24));
                    else
#pragma unroll
                        for (int e = 0; e < EPL; ++e) a_out[base + e] = (int8_t)b[e];
                }
                if (cl == 0) {
                    sxs[i] = scale;
                    if (sx_out) sx_out[g] = scale;
                }
            }
        }
        compute_sync();

        // ---------------------------------------------------------- phase B
        const int r = tid & 127, h = tid >> 7;
        float acc = 0.f;
        // one group's exact partial as four independent dp4a chains (one per
        // 32-bit word of a piece; integer sums, so the order is free)
        auto partial = [&](int i) {
            const uint8_t* c = stages + (size_t)i * C::CB;
            int d0 = 0, d1 = 0, d2 = 0, d3 = 0;
#pragma unroll
            for (int p = 0; p < C::PP; ++p) {
                const uint4 w = *reinterpret_cast<const uint4*>(c + p * 2048 + r * 16);
                const uint4* ap = reinterpret_cast<const uint4*>(aperm + (size_t)i * GROUP + 32 * p);
                const uint4 a0 = ap[0], a1 = ap[1];
                if (CQ) {
                    uint32_t lo, hi;
                    cq4_expand(book, w.x, lo, hi);
                    d0 = __dp4a((int)lo, (int)a0.x, d0);
                    d0 = __dp4a((int)hi, (int)a0.y, d0);
                    cq4_expand(book, w.y, lo, hi);
                    d1 = __dp4a((int)lo, (int)a0.z, d1);
                    d1 = __dp4a((int)hi, (int)a0.w, d1);
                    cq4_expand(book, w.z, lo, hi);
                    d2 = __dp4a((int)lo, (int)a1.x, d2);
                    d2 = __dp4a((int)hi, (int)a1.y, d2);
                    cq4_expand(book, w.w, lo, hi);
                    d3 = __dp4a((int)lo, (int)a1.z, d3);
                    d3 = __dp4a((int)hi, (int)a1.w, d3);
                } else {
                    d0 = __dp4a(nib_lo16(w.x), (int)a0.x, d0);
                    d0 = __dp4a(nib_hi16(w.x), (int)a0.y, d0);
                    d1 = __dp4a(nib_lo16(w.y), (int)a0.z, d1);
                    d1 = __dp4a(nib_hi16(w.y), (int)a0.w, d1);
                    d2 = __dp4a(nib_lo16(w.z), (int)a1.x, d2);
                    d2 = __dp4a(nib_hi16(w.z), (int)a1.y, d2);
                    d3 = __dp4a(nib_lo16(w.w), (int)a1.z, d3);
                    d3 = __dp4a(nib_hi16(w.w), (int)a1.w, d3);
                }
            }
            const int dp = (d0 + d1) + (d2 + d3);
            return CQ ? dp : dp >> 4;   // symmetric: every product carried a factor 16
        };
        // two groups per step (independent dp4a chains), added in group order
        for (int i = h; i < ng; i += 4) {
            const bool two = i + 2 < ng;
            if (!mbar_wait(&full[i], 0, status, abort)) break;
            if (two && !mbar_wait(&full[i + 2], 0, status, abort)) break;
            const int dp0 = partial(i);
            const int dp1 = two ? partial(i + 2) : 0;
            const float sw0 = __half2float(reinterpret_cast<const __half*>(stages + (size_t)i * C::CB + 64 * GROUP)[r]);
            acc = fmaf((float)dp0, sw0 * sxs[i], acc);
            if (two) {
                const float sw1 =
                    __half2float(reinterpret_cast<const __half*>(stages + (size_t)(i + 2) * C::CB + 64 * GROUP)[r]);
                acc = fmaf((float)dp1, sw1 * sxs[i + 2], acc);
            }
        }
        if (h == 1) red[r] = acc;
        compute_sync();
        if (h == 0) {
            const float v = acc + red[r];
            if (ksplit == 1) {
                if (t * 128 + r < N) y[t * 128 + r] = CQ ? v * book.scale : v;
            } else {
                parts[s * 128 + r] = v;   // this slice's sums, locally first
            }
        }
        if (ksplit > 1) {
            if (s != 0) {
                // the slice's 128 sums go to the first CTA of the cluster as 32
                // asynchronous 16-byte stores that complete on its barrier
                compute_sync();
                if (warp == 0) {
                    const float4 v4 = reinterpret_cast<const float4*>(parts + s * 128)[lane];
                    st_async_cluster_v4(map_shared_rank(smem_u32(parts + s * 128 + 4 * lane), 0u), v4,
                                        map_shared_rank(smem_u32(sums_in), 0u));
                }
            } else if (tid < 128) {
                // the first CTA adds the slices in order once all have arrived
                mbar_wait_cluster(sums_in, 0, status);
                float v = 0.f;
                for (int k = 0; k < ksplit; ++k) v += parts[k * 128 + tid];
                if (t * 128 + tid < N) y[t * 128 + tid] = CQ ? v * book.scale : v;
            }
        }
    }
}

// K-slices per tile (see kTargetCtas), at most 16 (one cluster), and few
// enough groups per CTA for its shared memory (44 chunks of group 64, 22 of
// group 128).
int fused_ksplit(int T, int K, int group, int num_sms)
{
    const int G = K / group;
    int ks = (kTargetCtas + T - 1) / T;
    const int by_groups = (G + kMaxGroupsPerCta - 1) / kMaxGroupsPerCta;
    if (by_groups > ks && (long long)T * by_groups <= (long long)kCtasPerSm * num_sms) ks = by_groups;
    if (ks > G) ks = G;
    if (ks > kMaxCluster) ks = kMaxCluster;
    if (ks < 1) ks = 1;
    const int max_ng = group == 64 ? 44 : 22;
    while ((G + ks - 1) / ks > max_ng && ks < kMaxCluster && ks < G) ++ks;
    return ks;
}

template <int GROUP, int XDT, int EPL, bool CQ>
cudaError_t run(const LaunchCtx& c, const FusedSet& set, int K, int hadamard, const void* x, int8_t* a_out,
                float* sx_out)
{
    using C = Cfg<GROUP>;
    auto kern = gemv_fused_kernel<GROUP, XDT, EPL, CQ>;
    const int G = K / GROUP, T = set.tile0[set.count];
    const int ks = fused_ksplit(T, K, GROUP, c.num_sms);
    const int ng_max = (G + ks - 1) / ks;
    if (ng_max > (GROUP == 64 ? 44 : 22)) return cudaErrorInvalidValue;   // K too large for one cluster per tile
    size_t smem = smem_bytes(ng_max, C::CB, ng_max, GROUP);
    if ((long long)T * ks <= (long long)kCtasPerSm * c.num_sms && smem < kMinSmemPerCta) smem = kMinSmemPerCta;
    static KernelSmem configured;
    const cudaError_t e = ensure_smem(configured, c, kern, smem, /*nonportable_cluster=*/true);
    if (e != cudaSuccess) return e;
    const float rot = hadamard ? (float)(1.0 / sqrt((double)GROUP)) : 1.0f;
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
    return cudaLaunchKernelEx(&cfg, kern, set, K, ks, hadamard, rot, x, a_out, sx_out, c.status);
}

template <int GROUP, int EPL, bool CQ>
cudaError_t run_dtype(const LaunchCtx& c, const FusedSet& set, int K, int hadamard, const void* x, int x_dtype,
                      int8_t* a_out, float* sx_out)
{
    if (x_dtype == 0) return run<GROUP, 0, EPL, CQ>(c, set, K, hadamard, x, a_out, sx_out);
    if (x_dtype == 1) return run<GROUP, 1, EPL, CQ>(c, set, K, hadamard, x, a_out, sx_out);
    return run<GROUP, 2, EPL, CQ>(c, set, K, hadamard, x, a_out, sx_out);
}

template <bool CQ>
cudaError_t run_group(const LaunchCtx& c, const FusedSet& set, int K, int group, int hadamard, const void* x,
                      int x_dtype, int8_t* a_out, float* sx_out)
{
    // short slices (at most 16 groups per CTA) quantize with a warp per group
    const int ks = fused_ksplit(set.tile0[set.count], K, group, c.num_sms);
    const bool short_slice = (K / group + ks - 1) / ks <= 16;
    if (group == 64)
        return short_slice ? run_dtype<64, 2, CQ>(c, set, K, hadamard, x, x_dtype, a_out, sx_out)
                           : run_dtype<64, 8, CQ>(c, set, K, hadamard, x, x_dtype, a_out, sx_out);
    if (group == 128)
        return short_slice ? run_dtype<128, 4, CQ>(c, set, K, hadamard, x, x_dtype, a_out, sx_out)
                           : run_dtype<128, 8, CQ>(c, set, K, hadamard, x, x_dtype, a_out, sx_out);
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_gemv_fused_set(const LaunchCtx& c, bool cq4, int count, const int* N, int K, int group, int hadamard,
                                  const uint8_t* const* blob, const void* x, int x_dtype, float* const* y,
                                  int8_t* a_out, float* sx_out)
{
    if (count < 1 || count > kMaxSiblings) return cudaErrorInvalidValue;
    FusedSet set = {};
    set.count = count;
    set.tile0[0] = 0;
    for (int i = 0; i < count; ++i) {
        set.N[i] = N[i];
        set.blob[i] = blob[i];
        set.y[i] = y[i];
        set.tile0[i + 1] = set.tile0[i] + (N[i] + 127) / 128;
    }
    return cq4 ? run_group<true>(c, set, K, group, hadamard, x, x_dtype, a_out, sx_out)
               : run_group<false>(c, set, K, group, hadamard, x, x_dtype, a_out, sx_out);
}

cudaError_t launch_gemv_fused(const LaunchCtx& c, bool cq4, int N, int K, int group, int hadamard, const uint8_t* blob,
                              const void* x, int x_dtype, float* y, int8_t* a_out, float* sx_out)
{
    return launch_gemv_fused_set(c, cq4, 1, &N, K, group, hadamard, &blob, x, x_dtype, &y, a_out, sx_out);
}

}  // namespace qmm
