// qmm_gemm.cuh -- tensor-core GEMM of both variants on sm_103a (tcgen05).
//
// Sources: cactus PR #697 "SME2 acceleration for CQ4 matmul, prefill
// attention, and orthogonal embeddings", Summary ("Fused SME2 GEMM (M>1)":
// raw int32 partials with a separate fp32 rescale); geistlib issue #500
// "native W*A8 int8 GEMM for prefill" (no fp32 intermediate, no dequantized
// weights in DRAM); TensorFold PR #3215 "simd_qmm on Metal: X's group sums and
// half operands from a prepass" (affine tiles on the prepass's group sums and
// half X).
//
// GB300 design. The tensor cores of sm_103a have no int8 MMA kind, so both
// variants use tcgen05.mma kind::f16 with operands that carry the integers
// exactly: int4 weights and int8 activation codes are exact in fp16, products
// are exact, and a 64- or 128-wide group sum stays below 2^24, so the fp32
// accumulator holds the exact int32 group partial. Weights sit in the MMA's M
// slot (128 rows of the packed tile), activations in its N slot (m_tile rows,
// 16..128), so one kernel serves decode-sized and prefill-sized M.
//
// Warp roles (512 threads, one CTA per SM, persistent over tiles):
//   warps 0-3   expand: packed nibbles (smem) -> fp16 weight operand, written
//               to tensor memory with tcgen05.st (or to 128-byte-swizzled
//               shared memory); one tensor-memory lane quadrant per warp.
//               They copy each group's scales to a small ring of their own
//               and release the packed chunk at once, so the chunk ring is
//               not held for the length of the MMA and epilogue pipeline.
//   warps 4-11  epilogue: read each group's partials from tensor memory,
//               rescale in fp32 into register accumulators (at most 64 per
//               thread: m_tile <= 128, two warpgroups), store Y
//   warp 12     weight producer: 1-D bulk copies of packed chunks
//   warp 13     MMA issuer; owns the tensor-memory allocation
//   warp 14     activation-scale loader (sx or S per group, cp.async)
//   warp 15     activation producer: TMA tiles of the fp16 activations
//               (128-byte swizzle), in a ring deep enough that these small
//               loads never wait behind the weight chunks
// Accumulators are double-buffered per group in tensor memory so the MMAs of
// group g+1 run while the epilogue rescales group g. Every wait is bounded.
#pragma once

#include <cuda_fp16.h>

#include "qmm_internal.h"
#include "qmm_ptx.cuh"

namespace qmm {

constexpr int kGemmThreads = 512;

// Pipeline depths. Narrow tiles (m_tile <= 64: decode-sized M) are bound by
// the latency of the expand -> MMA -> epilogue hand-offs, so they keep more
// k-steps and groups in flight; wide tiles are bound by tensor-memory space.
template <int VARIANT, int GROUP, int MAXC>
struct GemmCfg {
    static constexpr bool NARROW = MAXC <= 32;
    static constexpr int CB = 64 * GROUP + 256 + (VARIANT == 1 ? 256 : 0);
    static constexpr int KSG = GROUP / 64;                                   // 64-wide k-steps per group
    static constexpr int RS = NARROW ? (GROUP == 128 ? 10 : 16) : (GROUP == 128 ? 8 : 12);  // packed chunks
    static constexpr int KS = NARROW ? 8 : 4;   // k-step stages: weight operand + activation tile together
    static constexpr int DS = NARROW ? 4 : 3;                                // accumulator buffers
    static constexpr int XS = 16;                                            // activation-scale stages
    static constexpr int SR = 8;                                             // weight-scale copies
    static constexpr int SCB = VARIANT == 1 ? 512 : 256;                     // bytes per copy
};

// k-step stages in use: the weight operand in shared memory takes 16 KB per
// stage, so that variant keeps fewer.
template <int VARIANT, int GROUP, int MAXC>
inline int gemm_kstages(bool a_in_smem)
{
    using C = GemmCfg<VARIANT, GROUP, MAXC>;
    return a_in_smem && C::KS > 4 ? 4 : C::KS;
}

template <int VARIANT, int GROUP, int MAXC>
inline size_t gemm_smem_bytes(int m_tile, bool a_in_smem)
{
    using C = GemmCfg<VARIANT, GROUP, MAXC>;
    const int ks = gemm_kstages<VARIANT, GROUP, MAXC>(a_in_smem);
    size_t b = 1024;                                     // alignment slack
    b += (size_t)ks * m_tile * 128;
    if (a_in_smem) b += (size_t)ks * 16384;
    b += (size_t)C::RS * C::CB;
    b += (size_t)C::XS * m_tile * 4;
    b += (size_t)C::SR * C::SCB;
    b += 8 * (2 * C::RS + 2 * C::KS + 2 * C::DS + 2 * C::XS + 2 * C::SR + 1) + 64;
    return b;
}

// Tensor-memory columns: DS accumulators (+ AS weight-operand stages).
template <int VARIANT, int GROUP, int MAXC>
inline int gemm_tmem_cols(int d_stride, bool a_in_smem)
{
    using C = GemmCfg<VARIANT, GROUP, MAXC>;
    const int cols = C::DS * d_stride + (a_in_smem ? 0 : 32 * C::KS);
    int alloc = 32;
    while (alloc < cols) alloc <<= 1;
    return alloc;
}

// fp16 pairs (k, k+1) of one packed word (slot order of the blob): exact
// integers via the 1024 + u trick. OFF = 8 for offset-binary symmetric
// weights, 0 for unsigned affine weights.
template <int OFF>
__device__ __forceinline__ void expand_word(uint32_t w, uint32_t* out)
{
    constexpr uint32_t kMagic = 0x64006400u;                           // fp16 1024, 1024
    constexpr uint32_t kSubLo = OFF == 8 ? 0x64086408u : 0x64006400u;  // 1032 or 1024
    constexpr uint32_t kMulHi = 0x2C002C00u;                           // 1/16
    constexpr uint32_t kSubHi = OFF == 8 ? 0xD480D480u : 0xD400D400u;  // -72 or -64
    const uint32_t w2 = w >> 8;
    uint32_t lo0 = (w & 0x000F000Fu) | kMagic;     // slots 0, 4 -> k0, k1
    uint32_t hi0 = (w & 0x00F000F0u) | kMagic;     // slots 1, 5 -> k2, k3 (x16)
    uint32_t lo1 = (w2 & 0x000F000Fu) | kMagic;    // slots 2, 6 -> k4, k5
    uint32_t hi1 = (w2 & 0x00F000F0u) | kMagic;    // slots 3, 7 -> k6, k7 (x16)
    const uint32_t sub_lo = kSubLo, mul_hi = kMulHi, sub_hi = kSubHi;
    __half2 r0 = __hsub2(*reinterpret_cast<__half2*>(&lo0), *reinterpret_cast<const __half2*>(&sub_lo));
    __half2 r1 = __hfma2(*reinterpret_cast<__half2*>(&hi0), *reinterpret_cast<const __half2*>(&mul_hi),
                         *reinterpret_cast<const __half2*>(&sub_hi));
    __half2 r2 = __hsub2(*reinterpret_cast<__half2*>(&lo1), *reinterpret_cast<const __half2*>(&sub_lo));
    __half2 r3 = __hfma2(*reinterpret_cast<__half2*>(&hi1), *reinterpret_cast<const __half2*>(&mul_hi),
                         *reinterpret_cast<const __half2*>(&sub_hi));
    out[0] = *reinterpret_cast<uint32_t*>(&r0);
    out[1] = *reinterpret_cast<uint32_t*>(&r1);
    out[2] = *reinterpret_cast<uint32_t*>(&r2);
    out[3] = *reinterpret_cast<uint32_t*>(&r3);
}

// Packed fp32 pairs (fma.rn.f32x2 / mul.rn.f32x2: two lanes of fp32 per
// instruction; each element rounds exactly as the scalar operation).
__device__ __forceinline__ unsigned long long pack2(float a, float b)
{
    return (unsigned long long)__float_as_uint(a) | ((unsigned long long)__float_as_uint(b) << 32);
}

// (p0 * s0, p1 * s1) for raw fp32 bit patterns p0, p1
__device__ __forceinline__ unsigned long long mul_pair(uint32_t p0, uint32_t p1, float s0, float s1)
{
    unsigned long long d;
    const unsigned long long a = (unsigned long long)p0 | ((unsigned long long)p1 << 32);
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(pack2(s0, s1)));
    return d;
}

// (acc0, acc1) += t * (w, w)
__device__ __forceinline__ void fma_pair(float& acc0, float& acc1, unsigned long long t, float w)
{
    unsigned long long c = pack2(acc0, acc1), d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(t), "l"(pack2(w, w)), "l"(c));
    acc0 = __uint_as_float((uint32_t)d);
    acc1 = __uint_as_float((uint32_t)(d >> 32));
}

// (acc0, acc1) += (v0, v1) * (w, w)
__device__ __forceinline__ void fma_pair_v(float& acc0, float& acc1, float v0, float v1, float w)
{
    fma_pair(acc0, acc1, pack2(v0, v1), w);
}

// (acc0, acc1) += (p0, p1) * (w, w) for raw fp32 bit patterns
__device__ __forceinline__ void fma_pair_u(float& acc0, float& acc1, uint32_t p0, uint32_t p1, float w)
{
    fma_pair(acc0, acc1, (unsigned long long)p0 | ((unsigned long long)p1 << 32), w);
}

template <int VARIANT, int GROUP, bool A_TMEM, bool DEBUG, int MAXC>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap act_map, const GemmShape sh, const uint8_t* __restrict__ blob,
                const float* __restrict__ act_scale, float* __restrict__ Y, int32_t* __restrict__ P, int* status)
{
    using C = GemmCfg<VARIANT, GROUP, MAXC>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int m_tile = sh.m_tile;
    const int b_bytes = m_tile * 128;
    uint8_t* bst = base;
    const int KSr = sh.bs;   // k-step stages in use
    uint8_t* ast = bst + (size_t)KSr * b_bytes;
    uint8_t* raw = ast + (A_TMEM ? 0 : (size_t)KSr * 16384);
    float* xs = reinterpret_cast<float*>(raw + (size_t)C::RS * C::CB);
    uint8_t* scr = reinterpret_cast<uint8_t*>(xs + C::XS * m_tile);   // per-group weight scales (+ biases)
    uint64_t* bars =
        reinterpret_cast<uint64_t*>((reinterpret_cast<uintptr_t>(scr + C::SR * C::SCB) + 7) & ~uintptr_t(7));
    uint64_t* raw_full = bars;
    uint64_t* raw_empty = raw_full + C::RS;
    uint64_t* k_full = raw_empty + C::RS;    // weight operand expanded + activation tile landed
    uint64_t* k_empty = k_full + C::KS;      // the k-step's MMAs retired
    uint64_t* d_full = k_empty + C::KS;
    uint64_t* d_empty = d_full + C::DS;
    uint64_t* x_full = d_empty + C::DS;
    uint64_t* x_empty = x_full + C::XS;
    uint64_t* s_full = x_empty + C::XS;      // weight scales of a group copied
    uint64_t* s_empty = s_full + C::SR;
    uint64_t* done = s_empty + C::SR;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = sh.K / GROUP;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::RS; ++i) {
            mbar_init(&raw_full[i], 1);
            mbar_init(&raw_empty[i], 4);   // expand warps, once they have read the chunk
        }
        for (int i = 0; i < C::SR; ++i) {
            mbar_init(&s_full[i], 4);      // expand warps
            mbar_init(&s_empty[i], 8);     // epilogue warps
        }
        for (int i = 0; i < KSr; ++i) {
            mbar_init(&k_full[i], 5);      // 4 expand warps + the activation producer (with its bytes)
            mbar_init(&k_empty[i], 1);     // MMA commit
        }
        for (int i = 0; i < C::DS; ++i) {
            mbar_init(&d_full[i], 1);      // MMA commit
            mbar_init(&d_empty[i], 8);     // epilogue warps
        }
        for (int i = 0; i < C::XS; ++i) {
            mbar_init(&x_full[i], 32);     // loader lanes
            mbar_init(&x_empty[i], 8);     // epilogue warps
        }
        mbar_init(done, 1);
        *abort = 0;
        fence_barrier_init();
    }
    if (warp == 15 && lane == 0) prefetch_tensormap(&act_map);
    if (warp == 13) {
        tmem_alloc(tmem_slot, (uint32_t)sh.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_trigger();

    if (warp == 12) {
        // ---------------------------------------------------------- weight producer
        if (lane == 0) {
            int rc = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < sh.num_tiles; tile += gridDim.x) {
                const int nt = tile / sh.mt_count;
                for (int g = 0; g < G; ++g) {
                    const int rs = rc % C::RS;
                    if (!mbar_wait(&raw_empty[rs], ((rc / C::RS) & 1) ^ 1, status, abort)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&raw_full[rs], C::CB);
                    bulk_g2s(raw + (size_t)rs * C::CB, blob + ((size_t)nt * G + g) * C::CB, C::CB, &raw_full[rs]);
                    ++rc;
                }
            }
            // no copy may still be landing when the CTA exits
            for (int i = rc - C::RS > 0 ? rc - C::RS : 0; i < rc; ++i)
                mbar_wait(&raw_full[i % C::RS], (i / C::RS) & 1, status, nullptr);
        }
    } else if (warp == 15) {
        // ---------------------------------------------------------- activation producer
        if (lane == 0) {
            pdl_wait();   // activations come from the previous kernel
            int bc = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < sh.num_tiles; tile += gridDim.x) {
                const int mt = tile % sh.mt_count;
                for (int kstep = 0; kstep < G * C::KSG; ++kstep) {
                    const int bs = bc % KSr;
                    if (!mbar_wait(&k_empty[bs], ((bc / KSr) & 1) ^ 1, status, abort)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&k_full[bs], (uint32_t)b_bytes);
                    tma_load_2d(bst + (size_t)bs * b_bytes, &act_map, kstep * 64, mt * m_tile, &k_full[bs]);
                    ++bc;
                }
            }
            for (int i = bc - KSr > 0 ? bc - KSr : 0; i < bc; ++i)
                mbar_wait(&k_full[i % KSr], (i / KSr) & 1, status, nullptr);
        }
    } else if (warp == 13) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_f16_f32(128, m_tile);
            int kc = 0, dc = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < sh.num_tiles; tile += gridDim.x) {
                for (int g = 0; ok && g < G; ++g) {
                    const int db = dc % C::DS;
                    if (!mbar_wait(&d_empty[db], ((dc / C::DS) & 1) ^ 1, status, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem + (uint32_t)(db * sh.d_stride);
                    for (int j = 0; j < C::KSG; ++j) {
                        const int ks = kc % KSr;
                        if (!mbar_wait(&k_full[ks], (kc / KSr) & 1, status, abort)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t bdesc = sdesc_sw128(smem_u32(bst + (size_t)ks * b_bytes));
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint32_t accum = (j > 0 || kk > 0) ? 1u : 0u;
                            if (A_TMEM) {
                                const uint32_t a_tmem = tmem + (uint32_t)(C::DS * sh.d_stride + 32 * ks + 8 * kk);
                                mma_f16_ts(d_tmem, a_tmem, bdesc + 2 * kk, idesc, accum);
                            } else {
                                const uint64_t adesc = sdesc_sw128(smem_u32(ast + (size_t)ks * 16384));
                                mma_f16_ss(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, accum);
                            }
                        }
                        tc_commit(&k_empty[ks]);
                        ++kc;
                    }
                    if (!ok) break;
                    tc_commit(&d_full[db]);
                    ++dc;
                }
            }
            // every issued MMA must retire before the allocation is released
            tc_commit(done);
            mbar_wait(done, 0, status, nullptr);
        }
    } else if (warp == 14) {
        // ---------------------------------------------------------- scale loader
        pdl_wait();
        // no copy may still be landing when the CTA exits (checked below)
        int xc = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < sh.num_tiles; tile += gridDim.x) {
            const int mt = tile % sh.mt_count;
            const int m0 = mt * m_tile;
            for (int g = 0; g < G; ++g) {
                const int s = xc % C::XS;
                if (!mbar_wait(&x_empty[s], ((xc / C::XS) & 1) ^ 1, status, abort)) {
                    ok = false;
                    break;
                }
                // asynchronous copies: the loader never waits for the data, the
                // slot's barrier completes when every lane's copies have landed
                float* dst = xs + (size_t)s * m_tile;
                for (int c = lane; c < m_tile; c += 32) {
                    const int m = m0 + c;
                    // rows beyond M, and the partials hook (no scales), read nothing: zero
                    const bool have = !DEBUG && m < sh.M;
                    cp_async_4(dst + c, have ? static_cast<const void*>(act_scale + (size_t)m * G + g)
                                             : static_cast<const void*>(blob),
                               have ? 4u : 0u);
                }
                cp_async_arrive(&x_full[s]);
                ++xc;
            }
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
    } else if (warp < 4) {
        // ---------------------------------------------------------- expand
        const int r = threadIdx.x;   // weight row within the tile == tensor-memory lane
        int kc = 0, rc = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < sh.num_tiles; tile += gridDim.x) {
            for (int g = 0; ok && g < G; ++g) {
                const int rs = rc % C::RS;
                if (!mbar_wait(&raw_full[rs], (rc / C::RS) & 1, status, abort)) {
                    ok = false;
                    break;
                }
                const uint8_t* ch = raw + (size_t)rs * C::CB;
                {
                    // the epilogue gets this group's scales (and biases) in a ring of
                    // its own, so the chunk can be released as soon as it has been read
                    const int ss = rc % C::SR;
                    if (!mbar_wait(&s_empty[ss], ((rc / C::SR) & 1) ^ 1, status, abort)) {
                        ok = false;
                        break;
                    }
                    uint16_t* dst = reinterpret_cast<uint16_t*>(scr + (size_t)ss * C::SCB);
                    const uint16_t* src = reinterpret_cast<const uint16_t*>(ch + 64 * GROUP);
                    dst[r] = src[r];
                    if (VARIANT == 1) dst[128 + r] = src[128 + r];
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&s_full[ss]);
                }
                for (int j = 0; j < C::KSG; ++j) {
                    const int as = kc % KSr;
                    if (!mbar_wait(&k_empty[as], ((kc / KSr) & 1) ^ 1, status, abort)) {
                        ok = false;
                        break;
                    }
                    const uint4 p0 = *reinterpret_cast<const uint4*>(ch + (2 * j) * 2048 + r * 16);
                    const uint4 p1 = *reinterpret_cast<const uint4*>(ch + (2 * j + 1) * 2048 + r * 16);
                    uint32_t hv[32];
                    constexpr int OFF = VARIANT == 0 ? 8 : 0;
                    expand_word<OFF>(p0.x, hv + 0);
                    expand_word<OFF>(p0.y, hv + 4);
                    expand_word<OFF>(p0.z, hv + 8);
                    expand_word<OFF>(p0.w, hv + 12);
                    expand_word<OFF>(p1.x, hv + 16);
                    expand_word<OFF>(p1.y, hv + 20);
                    expand_word<OFF>(p1.z, hv + 24);
                    expand_word<OFF>(p1.w, hv + 28);
                    if (A_TMEM) {
                        const uint32_t taddr =
                            tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)(C::DS * sh.d_stride + 32 * as);   // as < KS
                        tmem_st32(taddr, hv);
                        tmem_st_wait();
                        tc_fence_before();
                    } else {
                        uint8_t* row = ast + (size_t)as * 16384 + r * 128;
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            *reinterpret_cast<uint4*>(row + ((c ^ (r & 7)) * 16)) =
                                make_uint4(hv[4 * c], hv[4 * c + 1], hv[4 * c + 2], hv[4 * c + 3]);
                        fence_proxy_async_smem();
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&k_full[as]);
                    ++kc;
                }
                if (!ok) break;
                if (lane == 0) mbar_arrive(&raw_empty[rs]);   // the warp's reads of the chunk are done
                ++rc;
            }
        }
    } else if (warp < 12) {
        // ---------------------------------------------------------- epilogue
        const int q = warp & 3;             // tensor-memory lane quadrant
        const int half = (warp - 4) >> 2;   // column half
        const int r = 32 * q + lane;
        const int ncol = m_tile >> 1;
        const int c0 = half * ncol;
        const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
        int dc = 0, rc = 0, xc = 0;
        bool ok = true;
        pdl_wait();   // outputs may still be read by the previous kernel
        for (int tile = blockIdx.x; ok && tile < sh.num_tiles; tile += gridDim.x) {
            const int nt = tile / sh.mt_count, mt = tile % sh.mt_count;
            const int n = nt * 128 + r;
            const int m0 = mt * m_tile + c0;
            float acc[MAXC];
#pragma unroll
            for (int c = 0; c < MAXC; ++c) acc[c] = 0.f;
            for (int g = 0; g < G; ++g) {
                const int db = dc % C::DS, ss = rc % C::SR, xsi = xc % C::XS;
                if (!mbar_wait(&d_full[db], (dc / C::DS) & 1, status, abort) ||
                    !mbar_wait(&s_full[ss], (rc / C::SR) & 1, status, abort) ||
                    !mbar_wait(&x_full[xsi], (xc / C::XS) & 1, status, abort)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const __half* sc = reinterpret_cast<const __half*>(scr + (size_t)ss * C::SCB);
                const float sw = __half2float(sc[r]);
                const float bw = VARIANT == 1 ? __half2float(sc[128 + r]) : 0.f;
                const float* sxv = xs + (size_t)xsi * m_tile + c0;
                const uint32_t dcol = lane_base + (uint32_t)(db * sh.d_stride + c0);
                // BATCH columns at a time: up to BATCH/8 loads of 8 columns, one wait
                constexpr int BATCH = 32;
#pragma unroll
                for (int cb = 0; cb < MAXC; cb += BATCH) {
                    if (cb < ncol) {
                        uint32_t v[32];
#pragma unroll
                        for (int q8 = 0; q8 < BATCH / 8; ++q8)
                            if (cb + 8 * q8 < MAXC && cb + 8 * q8 < ncol) tmem_ld8_at(dcol + cb + 8 * q8, v, 8 * q8);
                        tmem_ld_wait32(v);
#pragma unroll
                        for (int e4 = 0; e4 < BATCH; e4 += 4) {
                            if (cb + e4 < MAXC && cb + e4 < ncol) {
                                const float4 s4 = *reinterpret_cast<const float4*>(sxv + cb + e4);
                                const int c = cb + e4;
                                if (DEBUG) {
#pragma unroll
                                    for (int e = 0; e < 4; ++e) {
                                        const int m = m0 + c + e;
                                        if (m < sh.M && n < sh.N)
                                            P[((size_t)m * sh.N + n) * G + g] = __float2int_rn(__uint_as_float(v[e4 + e]));
                                    }
                                } else if (VARIANT == 0) {
                                    // acc += (P * sx) * sw, two columns per packed instruction
                                    fma_pair(acc[c], acc[c + 1], mul_pair(v[e4], v[e4 + 1], s4.x, s4.y), sw);
                                    fma_pair(acc[c + 2], acc[c + 3], mul_pair(v[e4 + 2], v[e4 + 3], s4.z, s4.w), sw);
                                } else {
                                    // acc += S * b + P * s
                                    fma_pair_v(acc[c], acc[c + 1], s4.x, s4.y, bw);
                                    fma_pair_v(acc[c + 2], acc[c + 3], s4.z, s4.w, bw);
                                    fma_pair_u(acc[c], acc[c + 1], v[e4], v[e4 + 1], sw);
                                    fma_pair_u(acc[c + 2], acc[c + 3], v[e4 + 2], v[e4 + 3], sw);
                                }
                            }
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&d_empty[db]);
                    mbar_arrive(&s_empty[ss]);
                    mbar_arrive(&x_empty[xsi]);
                }
                ++dc;
                ++rc;
                ++xc;
            }
            if (!DEBUG && ok && n < sh.N) {
#pragma unroll
                for (int c = 0; c < MAXC; ++c) {
                    const int m = m0 + c;
                    if (c < ncol && m < sh.M) Y[(size_t)m * sh.N + n] = acc[c];
                }
            }
        }
    }

    // ------------------------------------------------------------------ teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 13) {
        tc_fence_after();
        tmem_dealloc(tmem, (uint32_t)sh.tmem_cols);
    }
}

// Host side: configure and launch one instance of gemm_kernel.
template <int VARIANT, int GROUP, bool A_TMEM, bool DEBUG, int MAXC>
cudaError_t run_gemm(const LaunchCtx& c, const CUtensorMap& map, const GemmShape& sh_in, const uint8_t* blob,
                     const float* act_scale, float* Y, int32_t* P)
{
    auto kern = gemm_kernel<VARIANT, GROUP, A_TMEM, DEBUG, MAXC>;
    GemmShape sh = sh_in;
    sh.tmem_cols = gemm_tmem_cols<VARIANT, GROUP, MAXC>(sh.d_stride, !A_TMEM);
    sh.bs = gemm_kstages<VARIANT, GROUP, MAXC>(!A_TMEM);
    const size_t smem = gemm_smem_bytes<VARIANT, GROUP, MAXC>(sh.m_tile, !A_TMEM);
    static size_t configured = 0;
    cudaError_t e;
    if (smem > configured) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured = smem;
    }
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kGemmThreads, smem);
    if (e != cudaSuccess) return e;
    if (occ < 1) return cudaErrorInvalidConfiguration;
    int per_sm = occ;
    if (per_sm * sh.tmem_cols > 512) per_sm = 512 / sh.tmem_cols;
    const int grid = sh.num_tiles < c.num_sms * per_sm ? sh.num_tiles : c.num_sms * per_sm;
    return launch(kern, dim3(grid), dim3(kGemmThreads), smem, c, map, sh, blob, act_scale, Y, P, c.status);
}

}  // namespace qmm
