// qmm_gemm_narrow.cu -- tensor-core GEMM of the int8-activation variants
// (symmetric W4A8, codebook CQ4) for up to 32 activation rows, with the
// weights in the MMA's N slot.
//
// Sources: cactus PR #697 "SME2 acceleration for CQ4 matmul, prefill
// attention, and orthogonal embeddings", Summary ("Fused SME2 GEMM (M>1)":
// raw int32 partials with a separate fp32 rescale; CQ4 indices expanded
// in-engine, cb_scale folded into one rescale); geistlib issue #500 "native
// W*A8 int8 GEMM for prefill" (no dequantized weights in DRAM).
//
// GB300 design. With few activation rows, putting the weights in the MMA's
// M slot (128 rows) and the activations in its N slot leaves each MMA with
// N = 16..32: every tcgen05.mma costs its issue and operand hand-off for
// almost no work, and the pipeline ran at one MMA per ~180 cycles. Here the
// roles are swapped: one MMA covers 256 weight rows (N = 256) and 128
// activation rows (M = 128), so a 64-wide k-step of 256 weight rows is 4 MMAs
// (a microbenchmark with the weight operand refilled from shared memory every
// k-step ran them at the isolated rate, ~130 cycles each). The activation
// tile (at most 32 rows; boxes of M rounded up to 8 rows) is loaded four
// times, at rows 0, 32, 64 and 96 of the operand, so every tensor-memory lane
// quadrant holds all activation rows and the rescale of a group's 256 columns
// spreads over the four quadrants (each quadrant's two epilogue warps take 64
// of the columns).
//
// Per k-step: 8 expand warps decode the 256 rows' nibbles (or codebook
// indices) into fp16 integers in the 128-byte-swizzled K-major layout of the
// B operand; the activation producer lands the four TMA boxes (64 k wide); the
// MMA warp issues 4 MMAs into the group's accumulator (256 tensor-memory
// columns, two buffers). Per group the epilogue rescales the exact fp32
// partials, acc += (P * sx) * sw in group order: the operations and order of
// the other tensor-core kernel, so the outputs are the same bits. The
// activation scales of every group are staged once in shared memory.
// Persistent over pairs of 128-row weight tiles; every wait bounded. Shared
// memory carries the fp16 weight operand twice (stored, then read by the
// MMAs) and bounds the kernel at ~2.5x the MMA time.
#include <cuda_fp16.h>

#include "qmm.h"
#include "qmm_gemm.cuh"

namespace qmm {

namespace {

constexpr int kNwExpandWarps = 8;
constexpr int kNwEpiWarps = 8;
constexpr int kNwThreads = 32 * (kNwExpandWarps + kNwEpiWarps + 3);   // + weight producer, activation producer, MMA
constexpr int kNwRows = 256;            // weight rows per MMA (N)
constexpr int kNwMaxM = 32;             // activation rows
constexpr int kNwAStage = 128 * 128;    // activation operand: 128 rows x 64 k fp16
constexpr int kNwBStage = kNwRows * 128;
constexpr int kNwRA = 3, kNwRX = 4, kNwDS = 2;

template <int GROUP>
struct NwCfg {
    static constexpr int CB = 64 * GROUP + 256;   // packed chunk (one 128-row tile, one group)
    static constexpr int KSG = GROUP / 64;        // k-steps per group
    static constexpr int RW = GROUP == 64 ? 4 : 3;   // chunk-pair stages
    static constexpr int RB = GROUP == 64 ? 4 : 3;   // expanded weight-operand stages (32 KB each)
    static constexpr int XB = kNwRows * 4;        // scale stage: sw of the 256 rows
};

// Fixed part; the activation scales of all groups (G x 32 fp32) follow.
template <int GROUP>
constexpr size_t nw_smem_fixed()
{
    using C = NwCfg<GROUP>;
    return 1024 + (size_t)kNwRA * kNwAStage + (size_t)C::RB * kNwBStage + (size_t)C::RW * 2 * C::CB +
           (size_t)kNwRX * C::XB + 8 * (2 * C::RW + 2 * kNwRA + 2 * C::RB + 2 * kNwRX + 2 * kNwDS + 1) + 16;
}

// acc += ((p0, p1) * (sx, sx)) * (sw0, sw1): the other tensor-core kernel's
// operations (partial times the activation scale, then a fused multiply-add
// with the weight scale), two columns per instruction.
__device__ __forceinline__ void acc_pair(unsigned long long& acc, uint32_t p0, uint32_t p1, unsigned long long sx2,
                                         float sw0, float sw1)
{
    asm("{\n\t.reg .b64 t, w;\n\t"
        "mov.b64 t, {%1, %2};\n\t"
        "mov.b64 w, {%3, %4};\n\t"
        "mul.rn.f32x2 t, t, %5;\n\t"
        "fma.rn.f32x2 %0, t, w, %0;\n\t}"
        : "+l"(acc)
        : "r"(p0), "r"(p1), "f"(sw0), "f"(sw1), "l"(sx2));
}

// Grid (P): CTA b takes weight-tile pairs b, b + P, ... (rows 256 tp ..
// 256 tp + 255) over all of K.
template <int VARIANT, int GROUP>
__global__ void __launch_bounds__(kNwThreads, 1)
    gemm_narrow_kernel(const __grid_constant__ CUtensorMap act_map, int M, int N, int K,
                       const uint8_t* __restrict__ blob, const float* __restrict__ sx, float* __restrict__ Y,
                       int* status)
{
    using C = NwCfg<GROUP>;
    constexpr int KSG = C::KSG, RW = C::RW;
    const int G = K / GROUP, T = (N + 127) / 128, TP = (T + 1) / 2;
    const int box_rows = (M + 7) & ~7;   // rows of the activation map's box

    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* ast = base;                                          // [RA][128 rows][128 B]
    uint8_t* bst = ast + (size_t)kNwRA * kNwAStage;              // [RB][256 rows][128 B]
    uint8_t* wst = bst + (size_t)C::RB * kNwBStage;              // [RW][2 chunks]
    uint8_t* xst = wst + (size_t)RW * 2 * C::CB;                  // [RX][sw 256 | sx 32] fp32
    uint64_t* bars = reinterpret_cast<uint64_t*>(xst + (size_t)kNwRX * C::XB);
    uint64_t* w_full = bars;                 // chunk pair landed (producer, with its bytes)
    uint64_t* w_empty = w_full + RW;         // expand warps have read it
    uint64_t* a_full = w_empty + RW;         // activation boxes landed
    uint64_t* a_empty = a_full + kNwRA;      // MMA commit
    uint64_t* b_full = a_empty + kNwRA;      // expand warps stored the k-step's weights
    uint64_t* b_empty = b_full + C::RB;      // MMA commit
    uint64_t* x_full = b_empty + C::RB;      // expand warps stored the group's scales
    uint64_t* x_empty = x_full + kNwRX;      // epilogue warps are done with them
    uint64_t* d_full = x_empty + kNwRX;      // MMA commit after the group's last k-step
    uint64_t* d_empty = d_full + kNwDS;      // epilogue warps loaded the partials
    uint64_t* done = d_empty + kNwDS;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
    float* sx_all = reinterpret_cast<float*>(tmem_slot + 4);   // [G][32] activation scales

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int kProducer = kNwExpandWarps + kNwEpiWarps, kActProducer = kProducer + 1, kMma = kProducer + 2;

    if (threadIdx.x == 0) {
        for (int i = 0; i < RW; ++i) {
            mbar_init(&w_full[i], 1);
            mbar_init(&w_empty[i], kNwExpandWarps);
        }
        for (int i = 0; i < kNwRA; ++i) {
            mbar_init(&a_full[i], 1);
            mbar_init(&a_empty[i], 1);
        }
        for (int i = 0; i < C::RB; ++i) {
            mbar_init(&b_full[i], kNwExpandWarps);
            mbar_init(&b_empty[i], 1);
        }
        for (int i = 0; i < kNwRX; ++i) {
            mbar_init(&x_full[i], kNwExpandWarps);
            mbar_init(&x_empty[i], kNwEpiWarps);
        }
        for (int i = 0; i < kNwDS; ++i) {
            mbar_init(&d_full[i], 1);
            mbar_init(&d_empty[i], kNwEpiWarps);
        }
        mbar_init(done, 1);
        *abort = 0;
        fence_barrier_init();
    }
    if (warp == kActProducer && lane == 0) prefetch_tensormap(&act_map);
    if (warp == kMma) {
        tmem_alloc(tmem_slot, 512u);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_trigger();

    if (warp == kProducer) {
        // ---------------------------------------------------------- weight producer
        if (lane == 0) {
            int ws = 0, issued = 0;
            uint32_t wph = 0;
            bool ok = true;
            for (int tp = blockIdx.x; ok && tp < TP; tp += gridDim.x) {
                const bool two = 2 * tp + 1 < T;
                const uint8_t* src0 = blob + (size_t)(2 * tp) * G * C::CB;
                for (int g = 0; g < G; ++g) {
                    if (!mbar_wait(&w_empty[ws], wph ^ 1u, status, abort)) {
                        ok = false;
                        break;
                    }
                    // both chunks lie inside the blob
                    if (!in_range((size_t)(2 * tp + (two ? 1 : 0)) * G + g < (size_t)T * G, status)) {
                        *abort = 1;
                        ok = false;
                        break;
                    }
                    uint8_t* dst = wst + (size_t)ws * 2 * C::CB;
                    mbar_arrive_expect_tx(&w_full[ws], (uint32_t)(two ? 2 * C::CB : C::CB));
                    bulk_g2s(dst, src0 + (size_t)g * C::CB, C::CB, &w_full[ws]);
                    if (two) bulk_g2s(dst + C::CB, src0 + (size_t)(G + g) * C::CB, C::CB, &w_full[ws]);
                    ++issued;
                    ring_next<RW>(ws, wph);
                }
            }
            // no copy may still be landing when the CTA exits
            for (int i = issued - RW > 0 ? issued - RW : 0; i < issued; ++i)
                mbar_wait(&w_full[i % RW], (i / RW) & 1, status, nullptr);
        }
    } else if (warp == kActProducer) {
        // ---------------------------------------------------------- activation producer
        if (lane == 0) {
            pdl_wait();   // the codes come from the previous kernel
            int as = 0, issued = 0;
            uint32_t aph = 0;
            bool ok = true;
            for (int tp = blockIdx.x; ok && tp < TP; tp += gridDim.x) {
                for (int k0 = 0; k0 < K; k0 += 64) {
                    if (!mbar_wait(&a_empty[as], aph ^ 1u, status, abort)) {
                        ok = false;
                        break;
                    }
                    uint8_t* dst = ast + (size_t)as * kNwAStage;
                    // boxes of M rounded up to 8 rows: lanes at or past M in each
                    // quadrant are never stored, so their operand rows may hold anything
                    mbar_arrive_expect_tx(&a_full[as], (uint32_t)(4 * box_rows * 128));
#pragma unroll
                    for (int c = 0; c < 4; ++c) tma_load_2d(dst + c * 4096, &act_map, k0, 0, &a_full[as]);
                    ++issued;
                    ring_next<kNwRA>(as, aph);
                }
            }
            for (int i = issued - kNwRA > 0 ? issued - kNwRA : 0; i < issued; ++i)
                mbar_wait(&a_full[i % kNwRA], (i / kNwRA) & 1, status, nullptr);
        }
    } else if (warp == kMma) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_f16_f32(128, kNwRows);
            int as = 0, bs = 0, db = 0;
            uint32_t aph = 0, bph = 0, dph = 0;
            bool ok = true;
            for (int tp = blockIdx.x; ok && tp < TP; tp += gridDim.x) {
                for (int g = 0; ok && g < G; ++g) {
                    if (!mbar_wait(&d_empty[db], dph ^ 1u, status, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem + (uint32_t)(db * kNwRows);
#pragma unroll
                    for (int j = 0; j < KSG; ++j) {
                        if (!mbar_wait(&a_full[as], aph, status, abort) || !mbar_wait(&b_full[bs], bph, status, abort)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t adesc = sdesc_sw128(smem_u32(ast + (size_t)as * kNwAStage));
                        const uint64_t bdesc = sdesc_sw128(smem_u32(bst + (size_t)bs * kNwBStage));
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_f16_ss(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, (j > 0 || kk > 0) ? 1u : 0u);
                        tc_commit(&a_empty[as]);
                        tc_commit(&b_empty[bs]);
                        ring_next<kNwRA>(as, aph);
                        ring_next<C::RB>(bs, bph);
                    }
                    if (!ok) break;
                    tc_commit(&d_full[db]);
                    ring_next<kNwDS>(db, dph);
                }
            }
            // every issued MMA must retire before the allocation is released
            tc_commit(done);
            mbar_wait(done, 0, status, nullptr);
        }
    } else if (warp < kNwExpandWarps) {
        // ---------------------------------------------------------- expand
        // thread t: row t of the 256-row operand (tile t / 128 of the pair)
        const int t = threadIdx.x, half = t >> 7, r = t & 127;
        Cq4Book book = {};
        if (VARIANT == 2) book = cq4_load(blob + cq4_trailer_offset(N, K, GROUP), 0x80808080u);
        pdl_wait();   // sx comes from the previous kernel
        // every group's activation scales, once (rows beyond M: zero); the
        // epilogue reads them after the group's x_full, which these warps
        // arrive on after this
        for (int i = t; i < G * kNwMaxM; i += 32 * kNwExpandWarps) {
            const int m = i % kNwMaxM, gi = i / kNwMaxM;
            sx_all[i] = m < M ? sx[(size_t)m * G + gi] : 0.f;
        }
        int ws = 0, bs = 0, xs = 0;
        uint32_t wph = 0, bph = 0, xph = 0;
        bool ok = true;
        for (int tp = blockIdx.x; ok && tp < TP; tp += gridDim.x) {
            for (int g = 0; ok && g < G; ++g) {
                if (!mbar_wait(&w_full[ws], wph, status, abort) || !mbar_wait(&x_empty[xs], xph ^ 1u, status, abort)) {
                    ok = false;
                    break;
                }
                const uint8_t* ch = wst + (size_t)ws * 2 * C::CB + (size_t)half * C::CB;
                // the group's weight scale of this row
                float* xsp = reinterpret_cast<float*>(xst + (size_t)xs * C::XB);
                xsp[t] = __half2float(reinterpret_cast<const __half*>(ch + 64 * GROUP)[r]);
                __syncwarp();
                if (lane == 0) mbar_arrive(&x_full[xs]);
                ring_next<kNwRX>(xs, xph);
#pragma unroll
                for (int j = 0; j < KSG; ++j) {
                    if (!mbar_wait(&b_empty[bs], bph ^ 1u, status, abort)) {
                        ok = false;
                        break;
                    }
                    const uint4 p0 = *reinterpret_cast<const uint4*>(ch + (2 * j) * 2048 + r * 16);
                    const uint4 p1 = *reinterpret_cast<const uint4*>(ch + (2 * j + 1) * 2048 + r * 16);
                    if (j == KSG - 1) {
                        // the chunk's last words are loaded: release it before the
                        // expansion, so that the producer refills the stage meanwhile
                        // (an ordered asm statement taking every loaded word keeps
                        // the arrive after the loads)
                        asm volatile("" ::"r"(p0.x), "r"(p0.y), "r"(p0.z), "r"(p0.w), "r"(p1.x), "r"(p1.y), "r"(p1.z),
                                     "r"(p1.w));
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&w_empty[ws]);
                    }
                    uint32_t hv[32];
                    if (VARIANT == 2) {
                        expand_word_cq4(book, p0.x, hv + 0);
                        expand_word_cq4(book, p0.y, hv + 4);
                        expand_word_cq4(book, p0.z, hv + 8);
                        expand_word_cq4(book, p0.w, hv + 12);
                        expand_word_cq4(book, p1.x, hv + 16);
                        expand_word_cq4(book, p1.y, hv + 20);
                        expand_word_cq4(book, p1.z, hv + 24);
                        expand_word_cq4(book, p1.w, hv + 28);
                    } else {
                        expand_word<8>(p0.x, hv + 0);
                        expand_word<8>(p0.y, hv + 4);
                        expand_word<8>(p0.z, hv + 8);
                        expand_word<8>(p0.w, hv + 12);
                        expand_word<8>(p1.x, hv + 16);
                        expand_word<8>(p1.y, hv + 20);
                        expand_word<8>(p1.z, hv + 24);
                        expand_word<8>(p1.w, hv + 28);
                    }
                    uint8_t* row = bst + (size_t)bs * kNwBStage + (size_t)t * 128;
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<uint4*>(row + ((c ^ (t & 7)) * 16)) =
                            make_uint4(hv[4 * c], hv[4 * c + 1], hv[4 * c + 2], hv[4 * c + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&b_full[bs]);
                    ring_next<C::RB>(bs, bph);
                }
                ring_next<RW>(ws, wph);
            }
        }
    } else {
        // ---------------------------------------------------------- epilogue
        // warp (quadrant q, column half h): activation row = lane (every
        // quadrant holds all of them), weight rows c0 .. c0 + 31 of the pair
        const int e = warp - kNwExpandWarps, q = warp & 3, h = e >> 2;
        const int c0 = 64 * q + 32 * h;
        const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)c0;
        const float out_scale =
            VARIANT == 2 ? *reinterpret_cast<const float*>(blob + cq4_trailer_offset(N, K, GROUP) + 16) : 1.f;
        int db = 0, xs = 0;
        uint32_t dph = 0, xph = 0;
        // the 32 columns read from either accumulator buffer lie inside the
        // 512-column allocation
        bool ok = in_range((kNwDS - 1) * kNwRows + c0 + 32 <= 512, status);
        if (!ok) *abort = 1;
        pdl_wait();   // outputs may still be read by the previous kernel
        for (int tp = blockIdx.x; ok && tp < TP; tp += gridDim.x) {
            unsigned long long acc[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) acc[c] = 0ull;
            for (int g = 0; g < G; ++g) {
                if (!mbar_wait(&d_full[db], dph, status, abort) || !mbar_wait(&x_full[xs], xph, status, abort)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float* xsp = reinterpret_cast<const float*>(xst + (size_t)xs * C::XB);
                const unsigned long long sx2 = splat2(sx_all[g * kNwMaxM + lane]);
                // two rounds of 16 columns (fewer live registers)
#pragma unroll
                for (int hc = 0; hc < 32; hc += 16) {
                    uint32_t v[16];
                    tmem_ld8_at(lane_base + (uint32_t)(db * kNwRows + hc), v, 0);
                    tmem_ld8_at(lane_base + (uint32_t)(db * kNwRows + hc + 8), v, 8);
                    tmem_ld_wait_n(v);
#pragma unroll
                    for (int c4 = 0; c4 < 16; c4 += 4) {
                        const float4 w4 = *reinterpret_cast<const float4*>(xsp + c0 + hc + c4);
                        acc_pair(acc[(hc + c4) / 2], v[c4], v[c4 + 1], sx2, w4.x, w4.y);
                        acc_pair(acc[(hc + c4) / 2 + 1], v[c4 + 2], v[c4 + 3], sx2, w4.z, w4.w);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&d_empty[db]);
                ring_next<kNwDS>(db, dph);
                __syncwarp();
                if (lane == 0) mbar_arrive(&x_empty[xs]);
                ring_next<kNwRX>(xs, xph);
            }
            if (ok && lane < M) {
                const int n0 = 256 * tp + c0;
                float* yrow = Y + (size_t)lane * N;
                float o[32];
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const uint32_t bits = (uint32_t)(c & 1 ? acc[c / 2] >> 32 : acc[c / 2]);
                    o[c] = VARIANT == 2 ? __uint_as_float(bits) * out_scale : __uint_as_float(bits);
                }
                if ((N & 3) == 0 && n0 + 32 <= N) {
                    // 16-byte stores (row starts are 16-byte aligned when N % 4 == 0)
#pragma unroll
                    for (int c = 0; c < 32; c += 4)
                        *reinterpret_cast<float4*>(yrow + n0 + c) = make_float4(o[c], o[c + 1], o[c + 2], o[c + 3]);
                } else {
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        if (n0 + c < N) yrow[n0 + c] = o[c];
                }
            }
        }
    }

    // ------------------------------------------------------------------ teardown
    tc_fence_before();
    __syncthreads();
    if (warp == kMma) {
        tc_fence_after();
        tmem_dealloc(tmem, 512u);
    }
}

template <int VARIANT, int GROUP>
cudaError_t run_narrow(const LaunchCtx& c, const CUtensorMap& map, int M, int N, int K, const uint8_t* blob,
                       const float* sx, float* Y)
{
    auto kern = gemm_narrow_kernel<VARIANT, GROUP>;
    const size_t smem = nw_smem_fixed<GROUP>() + (size_t)(K / GROUP) * kNwMaxM * 4;
    if (smem > 227 * 1024) return cudaErrorNotSupported;   // K too long: the general kernel takes it
    static KernelSmem configured;
    const cudaError_t e = ensure_smem(configured, c, kern, smem);
    if (e != cudaSuccess) return e;
    const int T = (N + 127) / 128, TP = (T + 1) / 2;
    const int grid = TP < c.num_sms ? TP : c.num_sms;
    return launch(kern, dim3(grid), dim3(kNwThreads), smem, c, map, M, N, K, blob, sx, Y, c.status);
}

}  // namespace

cudaError_t launch_gemm_narrow(const LaunchCtx& c, bool cq4, int group, const CUtensorMap& map, int M, int N, int K,
                               const uint8_t* blob, const float* sx, float* Y)
{
    if (M < 1 || M > kNwMaxM || K % 64 != 0) return cudaErrorInvalidValue;
    if (group == 64) return cq4 ? run_narrow<2, 64>(c, map, M, N, K, blob, sx, Y) : run_narrow<0, 64>(c, map, M, N, K, blob, sx, Y);
    if (group == 128)
        return cq4 ? run_narrow<2, 128>(c, map, M, N, K, blob, sx, Y) : run_narrow<0, 128>(c, map, M, N, K, blob, sx, Y);
    return cudaErrorInvalidValue;
}

}  // namespace qmm
