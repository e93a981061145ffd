// qmm_gemm.cuh -- tensor-core GEMM of both variants on sm_103a (tcgen05).
//
// Sources: cactus PR #697 "SME2 acceleration for CQ4 matmul, prefill
// attention, and orthogonal embeddings", Summary ("Fused SME2 GEMM (M>1)":
// raw int32 partials with a separate fp32 rescale); geistlib issue #500
// "native W*A8 int8 GEMM for prefill" (no fp32 intermediate, no dequantized
// weights in DRAM); TensorFold PR #3215 "simd_qmm on Metal: X's group sums and
// half operands from a prepass" (affine tiles on the prepass's group sums and
// half X). Codebook (CQ4) weights: cactus PR #697, Summary (in-engine 4-bit
// codebook expansion, cb_scale folded into one fp32 rescale).
//
// GB300 design. The tensor cores of sm_103a have no int8 MMA kind, so both
// variants use tcgen05.mma kind::f16 with operands that carry the integers
// exactly: int4 weights and int8 activation codes are exact in fp16, products
// are exact, and a 64- or 128-wide group sum stays below 2^24, so the fp32
// accumulator holds the exact int32 group partial. Weights sit in the MMA's M
// slot (128 rows of the packed tile), activations in its N slot (m_tile rows,
// 16..128), so one kernel serves decode-sized and prefill-sized M.
//
// Every group's partials must be rescaled on their own (sw differs per row and
// group, sx per activation row and group), so the epilogue reads the whole
// accumulator from tensor memory once per group: 2 fp32 operations per
// partial against 64 (g64) tensor-core MACs. That rescale, not the MMA, sets
// the pace on wide tiles, so it gets the fewest instructions:
//   - a thread keeps its running sums (up to 64 columns) as packed fp32 pairs
//     (fma.rn.f32x2 / mul.rn.f32x2: two columns per instruction, each rounded
//     as the scalar operation) and reads all of a group's columns with one
//     tensor-memory round trip; the epilogue warpgroups raise their register
//     budget with setmaxnreg to hold both;
//   - every column of the instance is loaded and rescaled without column
//     guards (guarded loops scheduled 1.4x slower);
//   - one scale stage per group carries the weight scales (+ biases) and the
//     activation scales, filled by one loader warp with asynchronous copies:
//     the epilogue waits on two barriers per group (partials, scales), and
//     the expand warps only expand.
// Warp roles (512 threads, one CTA per SM, persistent over tiles):
//   warps 0-3   expand: packed nibbles (smem) -> fp16 weight operand, written
//               to tensor memory with tcgen05.st (or to 128-byte-swizzled
//               shared memory); one tensor-memory lane quadrant per warp
//   warps 4-11  epilogue: rescale each group's partials into register sums
//               (two warpgroups = two column halves), store Y per tile
//   (tiles of at most 32 activation rows instead run 8 expand warps, two sets
//   taking alternate groups, and one epilogue warpgroup, warps 8-11: there
//   the per-group expand chain, not the rescale, is the critical path)
//   warp 12     weight producer: 1-D bulk copies of packed chunks
//   warp 13     MMA issuer; owns the tensor-memory allocation
//   warp 14     scale loader (weight scales from the blob, sx or S per group)
//   warp 15     activation producer: TMA tiles of the fp16 activations
// Ring positions advance incrementally (no division on the issue paths).
// Every wait is bounded.
#pragma once

#include <cuda_fp16.h>

#include "qmm_cq4.cuh"
#include "qmm_internal.h"
#include "qmm_ptx.cuh"

namespace qmm {

// VARIANT: 0 symmetric W4A8, 1 affine, 2 codebook (CQ4: the symmetric
// variant's layout and rescale with looked-up levels, times cb_scale at the
// store).
constexpr int kGemmThreads = 512;
// Register budgets after setmaxnreg: the expand and single-role warpgroups drop
// to 80 per thread, the epilogue warpgroups rise to 176 (a whole group's 64
// columns and their 64 running sums in registers). With 4 expand warps the
// four warpgroups sum to exactly the launch's 512 x 128 registers; with 8 the
// one epilogue warpgroup needs less than is freed.
constexpr int kGemmRegsLow = 80;
constexpr int kGemmRegsHigh = 176;
static_assert(128 * (2 * kGemmRegsLow + 2 * kGemmRegsHigh) <= kGemmThreads * 128, "register split");

// Pipeline depths. Narrow tiles (m_tile <= 64: decode-sized M) keep more
// k-steps and groups in flight; wide tiles are bound by tensor-memory space.
template <int VARIANT, int GROUP, int MAXC>
struct GemmCfg {
    static constexpr bool NARROW = MAXC <= 32;
    static constexpr int CB = 64 * GROUP + 256 + (VARIANT == 1 ? 256 : 0);
    static constexpr int KSG = GROUP / 64;                                   // 64-wide k-steps per group
    static constexpr int RS = NARROW ? (GROUP == 128 ? 10 : 16) : (GROUP == 128 ? 8 : 12);  // packed chunks
    static constexpr int KS_TMEM = NARROW ? 8 : 4;   // k-step stages, weight operand in tensor memory
    static constexpr int KS_SMEM = 4;                // k-step stages, weight operand in shared memory
    static constexpr int DS = MAXC <= 48 ? 4 : 3;    // accumulator buffers
    // Narrow tiles relay the accumulator-buffer wait through the expand warps:
    // there the MMA-issuing thread's loop is the critical path (two mbarrier
    // waits, four MMAs and two commits per group, each wait ~150 cycles of
    // that thread), while the expand warps have slack.
    static constexpr bool RELAY = NARROW;
    // epilogue columns per tensor-memory round trip: the whole group
    static constexpr int EB = MAXC;
    static constexpr int XS = 16;                    // scale stages
    static constexpr int SWB = VARIANT == 1 ? 512 : 256;   // weight scales (+ biases) bytes per stage
};

template <int VARIANT, int GROUP, int MAXC>
constexpr int gemm_kstages(bool a_in_smem)
{
    return a_in_smem ? GemmCfg<VARIANT, GROUP, MAXC>::KS_SMEM : GemmCfg<VARIANT, GROUP, MAXC>::KS_TMEM;
}

template <int VARIANT, int GROUP, int MAXC>
inline size_t gemm_smem_bytes(int m_tile, int d_stride, bool a_in_smem)
{
    using C = GemmCfg<VARIANT, GROUP, MAXC>;
    const int ks = gemm_kstages<VARIANT, GROUP, MAXC>(a_in_smem);
    size_t b = 1024;                                     // alignment slack
    b += (size_t)ks * m_tile * 128;
    if (a_in_smem) b += (size_t)ks * 16384;
    b += (size_t)C::RS * C::CB;
    b += (size_t)C::XS * (C::SWB + 4 * d_stride);
    b += 8 * (2 * C::RS + 2 * ks + 2 * C::DS + 2 * C::XS + 1) + 64;
    return b;
}

// Tensor-memory columns: DS accumulators (+ the weight-operand stages).
template <int VARIANT, int GROUP, int MAXC>
inline int gemm_tmem_cols(int d_stride, bool a_in_smem)
{
    using C = GemmCfg<VARIANT, GROUP, MAXC>;
    const int cols = C::DS * d_stride + (a_in_smem ? 0 : 32 * C::KS_TMEM);
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

// fp16 pairs (k, k+1) of one packed word of codebook indices. The levels are
// looked up as unsigned bytes u = c + 128 (the book is loaded with its bytes
// XOR 0x80), placed under the fp16 exponent of 1024 (1024 + u is exact) and
// offset by 1152: exact integers c in [-128, 127].
__device__ __forceinline__ void expand_word_cq4(const Cq4Book& book, uint32_t w, uint32_t* out)
{
    uint32_t lo, hi;   // u of k = 0, 2, 4, 6 and of k = 1, 3, 5, 7
    cq4_expand(book, w, lo, hi);
    constexpr uint32_t kExp = 0x64646464u;
    const uint32_t t0 = prmt(lo, hi, 0x5140u);   // u0 u1 u2 u3
    const uint32_t t1 = prmt(lo, hi, 0x7362u);   // u4 u5 u6 u7
    uint32_t f[4] = {prmt(t0, kExp, 0x4140u), prmt(t0, kExp, 0x4342u), prmt(t1, kExp, 0x4140u),
                     prmt(t1, kExp, 0x4342u)};
    const uint32_t off = 0x64806480u;   // fp16 1152, 1152
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __half2 r = __hsub2(*reinterpret_cast<__half2*>(&f[i]), *reinterpret_cast<const __half2*>(&off));
        out[i] = *reinterpret_cast<uint32_t*>(&r);
    }
}

// Running sums of two columns as one packed fp32 pair.
__device__ __forceinline__ unsigned long long splat2(float w)
{
    unsigned long long d;
    asm("mov.b64 %0, {%1, %1};" : "=l"(d) : "f"(w));
    return d;
}

// W4A8: acc += ((p0, p1) * (s0, s1)) * (w, w), p the raw fp32 partials.
__device__ __forceinline__ void acc_w4a8(unsigned long long& acc, uint32_t p0, uint32_t p1, float s0, float s1,
                                         unsigned long long w2)
{
    asm("{\n\t.reg .b64 t, s;\n\t"
        "mov.b64 t, {%1, %2};\n\t"
        "mov.b64 s, {%3, %4};\n\t"
        "mul.rn.f32x2 t, t, s;\n\t"
        "fma.rn.f32x2 %0, t, %5, %0;\n\t}"
        : "+l"(acc)
        : "r"(p0), "r"(p1), "f"(s0), "f"(s1), "l"(w2));
}

// Affine: acc += (S0, S1) * (b, b), then acc += (p0, p1) * (s, s).
__device__ __forceinline__ void acc_affine(unsigned long long& acc, uint32_t p0, uint32_t p1, float S0, float S1,
                                           unsigned long long b2, unsigned long long s2)
{
    asm("{\n\t.reg .b64 t, u;\n\t"
        "mov.b64 u, {%3, %4};\n\t"
        "fma.rn.f32x2 %0, u, %5, %0;\n\t"
        "mov.b64 t, {%1, %2};\n\t"
        "fma.rn.f32x2 %0, t, %6, %0;\n\t}"
        : "+l"(acc)
        : "r"(p0), "r"(p1), "f"(S0), "f"(S1), "l"(b2), "l"(s2));
}

template <int S>
__device__ __forceinline__ void ring_next(int& i, uint32_t& ph)
{
    if (++i == S) {
        i = 0;
        ph ^= 1u;
    }
}

template <int VARIANT, int GROUP, bool A_TMEM, bool DEBUG, int MAXC, int EXPW>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap act_map, const GemmShape sh, const uint8_t* __restrict__ blob,
                const float* __restrict__ act_scale, float* __restrict__ Y, int32_t* __restrict__ P, int* status)
{
    using C = GemmCfg<VARIANT, GROUP, MAXC>;
    constexpr int KS = A_TMEM ? C::KS_TMEM : C::KS_SMEM;
    constexpr int RS = C::RS, DS = C::DS, XS = C::XS, KSG = C::KSG;
    // With the relay, the commit that frees a group's last k-step stage also
    // tells the epilogue that the group's partials are complete (one commit
    // per group fewer for the MMA-issuing thread). The epilogue then waits on
    // that stage's barrier, whose next phase needs the MMAs of a group that in
    // turn needs the epilogue to have released a later group's buffer, so the
    // phase it waits for cannot be overtaken when KS >= KSG * (DS + 1).
    // Measured: prefill M = 16 11.6 -> 11.0 µs; the affine GEMM at M = 64 went
    // from 74.4 to 76.0 µs, so the affine variant keeps its own commit.
    constexpr bool SHARED_COMMIT = C::RELAY && VARIANT != 1 && KS >= KSG * (DS + 1);
    // EXPW expand warps (4, or 8 = two sets taking alternate groups), then
    // 12 - EXPW epilogue warps (two column halves with 8, one with 4)
    static_assert(EXPW == 4 || EXPW == 8, "expand warps");
    constexpr int EPIW = 12 - EXPW;
    constexpr int EB = C::EB;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int m_tile = sh.m_tile;
    const int b_bytes = m_tile * 128;
    const int ssb = C::SWB + 4 * sh.d_stride;   // bytes per scale stage (sx region: d_stride floats)
    uint8_t* bst = base;
    uint8_t* ast = bst + (size_t)KS * b_bytes;
    uint8_t* raw = ast + (A_TMEM ? 0 : (size_t)KS * 16384);
    uint8_t* scs = raw + (size_t)RS * C::CB;
    uint64_t* bars =
        reinterpret_cast<uint64_t*>((reinterpret_cast<uintptr_t>(scs + (size_t)XS * ssb) + 7) & ~uintptr_t(7));
    uint64_t* raw_full = bars;
    uint64_t* raw_empty = raw_full + RS;
    uint64_t* k_full = raw_empty + RS;    // weight operand expanded + activation tile landed
    uint64_t* k_empty = k_full + KS;      // the k-step's MMAs retired
    uint64_t* d_full = k_empty + KS;      // a group's partials complete
    uint64_t* d_empty = d_full + DS;      // the epilogue's loads of them landed
    uint64_t* x_full = d_empty + DS;      // a group's scales landed
    uint64_t* x_empty = x_full + XS;      // the epilogue is done with them
    uint64_t* done = x_empty + XS;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = sh.K / GROUP;
    const size_t n_chunks = (size_t)((sh.N + 127) / 128) * G;   // chunks in the blob

    if (threadIdx.x == 0) {
        for (int i = 0; i < RS; ++i) {
            mbar_init(&raw_full[i], 1);
            mbar_init(&raw_empty[i], 4);   // expand warps, once they have read the chunk
        }
        for (int i = 0; i < KS; ++i) {
            mbar_init(&k_full[i], 5);      // 4 expand warps + the activation producer (with its bytes)
            mbar_init(&k_empty[i], 1);     // MMA commit
        }
        for (int i = 0; i < DS; ++i) {
            mbar_init(&d_full[i], 1);      // MMA commit
            mbar_init(&d_empty[i], EPIW);  // epilogue warps
        }
        for (int i = 0; i < XS; ++i) {
            mbar_init(&x_full[i], 32);     // loader lanes
            mbar_init(&x_empty[i], EPIW);  // epilogue warps
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
    const uint32_t a_col0 = (uint32_t)(DS * sh.d_stride);   // first weight-operand column
    pdl_trigger();

    if (warp >= 12) {
        setmaxnreg_dec<kGemmRegsLow>();   // one instruction for the whole warpgroup
        if (warp == 12) {
            // ------------------------------------------------------ weight producer
            if (lane == 0) {
                int rs = 0, issued = 0;
                uint32_t rph = 0;
                bool ok = true;
                for (int tile = blockIdx.x; ok && tile < sh.num_tiles; tile += gridDim.x) {
                    const uint8_t* src = blob + (size_t)(tile / sh.mt_count) * G * C::CB;
                    for (int g = 0; g < G; ++g) {
                        if (!mbar_wait(&raw_empty[rs], rph ^ 1u, status, abort)) {
                            ok = false;
                            break;
                        }
                        // the chunk lies inside the blob
                        if (!in_range((size_t)(tile / sh.mt_count) * G + g < n_chunks, status)) {
                            *abort = 1;
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&raw_full[rs], C::CB);
                        bulk_g2s(raw + (size_t)rs * C::CB, src + (size_t)g * C::CB, C::CB, &raw_full[rs]);
                        ++issued;
                        ring_next<RS>(rs, rph);
                    }
                }
                // no copy may still be landing when the CTA exits
                for (int i = issued - RS > 0 ? issued - RS : 0; i < issued; ++i)
                    mbar_wait(&raw_full[i % RS], (i / RS) & 1, status, nullptr);
            }
        } else if (warp == 13) {
            // ------------------------------------------------------ MMA issuer
            if (lane == 0) {
                const uint32_t idesc = idesc_f16_f32(128, m_tile);
                int ks = 0, db = 0;
                uint32_t kph = 0, dph = 0;
                // accumulators below the weight-operand stages, stages inside
                // the allocation
                bool ok = in_range(DS * sh.d_stride <= (int)a_col0 && m_tile <= sh.d_stride &&
                                       (!A_TMEM || (int)a_col0 + 32 * KS <= sh.tmem_cols),
                                   status);
                if (!ok) *abort = 1;
                for (int tile = blockIdx.x; ok && tile < sh.num_tiles; tile += gridDim.x) {
                    for (int g = 0; ok && g < G; ++g) {
                        // the group's accumulator buffer has been drained (with the
                        // relay, the first k-step's barrier below implies it)
                        if (!C::RELAY && !mbar_wait(&d_empty[db], dph ^ 1u, status, abort)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t d_tmem = tmem + (uint32_t)(db * sh.d_stride);
#pragma unroll
                        for (int j = 0; j < KSG; ++j) {
                            if (!mbar_wait(&k_full[ks], kph, status, abort)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            const uint64_t bdesc = sdesc_sw128(smem_u32(bst + (size_t)ks * b_bytes));
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk) {
                                const uint32_t accum = (j > 0 || kk > 0) ? 1u : 0u;
                                if (A_TMEM) {
                                    mma_f16_ts(d_tmem, tmem + a_col0 + (uint32_t)(32 * ks + 8 * kk), bdesc + 2 * kk,
                                               idesc, accum);
                                } else {
                                    const uint64_t adesc = sdesc_sw128(smem_u32(ast + (size_t)ks * 16384));
                                    mma_f16_ss(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, accum);
                                }
                            }
                            tc_commit(&k_empty[ks]);
                            ring_next<KS>(ks, kph);
                        }
                        if (!ok) break;
                        if (!SHARED_COMMIT) tc_commit(&d_full[db]);
                        ring_next<DS>(db, dph);
                    }
                }
                // every issued MMA must retire before the allocation is released
                tc_commit(done);
                mbar_wait(done, 0, status, nullptr);
            }
        } else if (warp == 14) {
            // ------------------------------------------------------ scale loader
            pdl_wait();   // sx / S come from the previous kernel
            int xs = 0;
            uint32_t xph = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < sh.num_tiles; tile += gridDim.x) {
                const int nt = tile / sh.mt_count, mt = tile - nt * sh.mt_count;
                const int m0 = mt * m_tile;
                const uint8_t* wsrc = blob + (size_t)nt * G * C::CB + 64 * GROUP;
                for (int g = 0; g < G; ++g) {
                    if (!mbar_wait(&x_empty[xs], xph ^ 1u, status, abort)) {
                        ok = false;
                        break;
                    }
                    // asynchronous copies: the slot's barrier completes when every
                    // lane's copies have landed
                    if (!in_range((size_t)nt * G + g < n_chunks, status)) {
                        *abort = 1;
                        ok = false;
                        break;
                    }
                    uint8_t* st = scs + (size_t)xs * ssb;
                    const uint8_t* ws = wsrc + (size_t)g * C::CB;
#pragma unroll
                    for (int j = lane; j < C::SWB / 4; j += 32) cp_async_4(st + 4 * j, ws + 4 * j, 4u);
                    float* sxd = reinterpret_cast<float*>(st + C::SWB);
                    for (int c = lane; c < m_tile; c += 32) {
                        const int m = m0 + c;
                        // rows beyond M, and the partials hook (no scales), read nothing: zero
                        const bool have = !DEBUG && m < sh.M;
                        cp_async_4(sxd + c, have ? static_cast<const void*>(act_scale + (size_t)m * G + g)
                                                 : static_cast<const void*>(blob),
                                   have ? 4u : 0u);
                    }
                    cp_async_arrive(&x_full[xs]);
                    ring_next<XS>(xs, xph);
                }
            }
            asm volatile("cp.async.wait_all;" ::: "memory");
        } else {
            // ------------------------------------------------------ activation producer
            if (lane == 0) {
                pdl_wait();   // activations come from the previous kernel
                int ks = 0, issued = 0;
                uint32_t kph = 0;
                bool ok = true;
                for (int tile = blockIdx.x; ok && tile < sh.num_tiles; tile += gridDim.x) {
                    const int row0 = (tile % sh.mt_count) * m_tile;
                    for (int kstep = 0; kstep < G * KSG; ++kstep) {
                        if (!mbar_wait(&k_empty[ks], kph ^ 1u, status, abort)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&k_full[ks], (uint32_t)b_bytes);
                        tma_load_2d(bst + (size_t)ks * b_bytes, &act_map, kstep * 64, row0, &k_full[ks]);
                        ++issued;
                        ring_next<KS>(ks, kph);
                    }
                }
                for (int i = issued - KS > 0 ? issued - KS : 0; i < issued; ++i)
                    mbar_wait(&k_full[i % KS], (i / KS) & 1, status, nullptr);
            }
        }
    } else if (warp < EXPW) {
        setmaxnreg_dec<kGemmRegsLow>();
        // ---------------------------------------------------------- expand
        const int wq = warp & 3;           // tensor-memory lane quadrant
        const int r = 32 * wq + lane;      // weight row within the tile == tensor-memory lane
        const int set = warp >> 2;         // with two sets, set s takes the groups g % 2 == s
        Cq4Book book = {};
        if (VARIANT == 2) book = cq4_load(blob + cq4_trailer_offset(sh.N, sh.K, GROUP), 0x80808080u);
        int rs = 0, ks = 0, turn = 0, db = 0;
        uint32_t rph = 0, kph = 0, dph = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < sh.num_tiles; tile += gridDim.x) {
            for (int g = 0; ok && g < G; ++g) {
                if (EXPW == 8) {
                    const bool mine = turn == set;
                    turn ^= 1;
                    if (!mine) {   // the other set's group: only the ring positions move
#pragma unroll
                        for (int j = 0; j < KSG; ++j) ring_next<KS>(ks, kph);
                        ring_next<RS>(rs, rph);
                        ring_next<DS>(db, dph);
                        continue;
                    }
                }
                if (!mbar_wait(&raw_full[rs], rph, status, abort)) {
                    ok = false;
                    break;
                }
                const uint8_t* ch = raw + (size_t)rs * C::CB;
#pragma unroll
                for (int j = 0; j < KSG; ++j) {
                    if (!mbar_wait(&k_empty[ks], kph ^ 1u, status, abort)) {
                        ok = false;
                        break;
                    }
                    const uint4 p0 = *reinterpret_cast<const uint4*>(ch + (2 * j) * 2048 + r * 16);
                    const uint4 p1 = *reinterpret_cast<const uint4*>(ch + (2 * j + 1) * 2048 + r * 16);
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
                        constexpr int OFF = VARIANT == 0 ? 8 : 0;
                        expand_word<OFF>(p0.x, hv + 0);
                        expand_word<OFF>(p0.y, hv + 4);
                        expand_word<OFF>(p0.z, hv + 8);
                        expand_word<OFF>(p0.w, hv + 12);
                        expand_word<OFF>(p1.x, hv + 16);
                        expand_word<OFF>(p1.y, hv + 20);
                        expand_word<OFF>(p1.z, hv + 24);
                        expand_word<OFF>(p1.w, hv + 28);
                    }
                    if (j == KSG - 1) {
                        // the chunk's words are all in registers (the decode used them)
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&raw_empty[rs]);
                    }
                    if (A_TMEM) {
                        tmem_st32(tmem + ((uint32_t)(32 * wq) << 16) + a_col0 + (uint32_t)(32 * ks), hv);
                        tmem_st_wait();
                        tc_fence_before();
                    } else {
                        uint8_t* row = ast + (size_t)ks * 16384 + r * 128;
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            *reinterpret_cast<uint4*>(row + ((c ^ (r & 7)) * 16)) =
                                make_uint4(hv[4 * c], hv[4 * c + 1], hv[4 * c + 2], hv[4 * c + 3]);
                        fence_proxy_async_smem();
                    }
                    // relay: the group's first k-step is released to the MMA warp
                    // only once the epilogue has drained the group's accumulator
                    // buffer (one lane of the set's first warp waits)
                    if (C::RELAY && j == 0 && wq == 0 && lane == 0 && !mbar_wait(&d_empty[db], dph ^ 1u, status, abort))
                        ok = false;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&k_full[ks]);
                    ring_next<KS>(ks, kph);
                }
                ring_next<RS>(rs, rph);
                ring_next<DS>(db, dph);
            }
        }
    } else {
        // ---------------------------------------------------------- epilogue
        setmaxnreg_inc<kGemmRegsHigh>();
        const int q = warp & 3;                 // tensor-memory lane quadrant
        const int half = (warp - EXPW) >> 2;    // column half (always 0 with one epilogue warpgroup)
        const int r = 32 * q + lane;
        const int ncol = EPIW == 8 ? m_tile >> 1 : m_tile;
        const int c0 = half * ncol;
        const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)c0;
        int db = 0, xs = 0, kse = 0;
        uint32_t dph = 0, xph = 0, kphe = 0;
        // the columns read per group lie inside the accumulator buffer and the
        // scale stage's activation-scale region (the raw-partials hook reads
        // only live columns)
        bool ok = in_range(DEBUG || c0 + MAXC <= sh.d_stride, status);
        if (!ok) *abort = 1;
        const float out_scale =
            VARIANT == 2 ? *reinterpret_cast<const float*>(blob + cq4_trailer_offset(sh.N, sh.K, GROUP) + 16) : 1.f;
        pdl_wait();   // outputs may still be read by the previous kernel
        for (int tile = blockIdx.x; ok && tile < sh.num_tiles; tile += gridDim.x) {
            const int nt = tile / sh.mt_count, mt = tile - nt * sh.mt_count;
            const int n = nt * 128 + r;
            const int m0 = mt * m_tile + c0;
            unsigned long long acc[MAXC / 2];
#pragma unroll
            for (int c = 0; c < MAXC / 2; ++c) acc[c] = 0ull;
            for (int g = 0; g < G; ++g) {
                // the group's partials are complete: its own barrier, or with the
                // shared commit the barrier of its last k-step's stage
                uint64_t* part_done = &d_full[db];
                uint32_t part_ph = dph;
                if (SHARED_COMMIT) {
#pragma unroll
                    for (int j = 0; j < KSG - 1; ++j) ring_next<KS>(kse, kphe);
                    part_done = &k_empty[kse];
                    part_ph = kphe;
                    ring_next<KS>(kse, kphe);
                }
                if (!mbar_wait(part_done, part_ph, status, abort) || !mbar_wait(&x_full[xs], xph, status, abort)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint8_t* st = scs + (size_t)xs * ssb;
                const float* sxv = reinterpret_cast<const float*>(st + C::SWB) + c0;
                const unsigned long long w2 = splat2(__half2float(reinterpret_cast<const __half*>(st)[r]));
                const unsigned long long b2 =
                    VARIANT == 1 ? splat2(__half2float(reinterpret_cast<const __half*>(st)[128 + r])) : 0ull;
                const uint32_t dcol = lane_base + (uint32_t)(db * sh.d_stride);
                // All MAXC columns are loaded and rescaled, live or not: the
                // accumulator buffer and the scale stage extend to d_stride
                // columns (>= c0 + MAXC, checked on the host), columns past
                // ncol are never stored, and a loop without column guards
                // schedules far better (measured 1.4x on the prefill shape).
                // The partials hook keeps the guards (it serves every m_tile).
#pragma unroll
                for (int cb = 0; cb < MAXC; cb += EB) {
                    if (DEBUG && cb >= ncol) break;
                    uint32_t v[EB];
#pragma unroll
                    for (int q8 = 0; q8 < EB / 8; ++q8)
                        if (!DEBUG || cb + 8 * q8 < ncol) tmem_ld8_at(dcol + cb + 8 * q8, v, 8 * q8);
                    tmem_ld_wait_n(v);
#pragma unroll
                    for (int e4 = 0; e4 < EB; e4 += 4) {
                        if (DEBUG) {
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int c = cb + e4 + e, m = m0 + c;
                                if (c < ncol && m < sh.M && n < sh.N)
                                    P[((size_t)m * sh.N + n) * G + g] = __float2int_rn(__uint_as_float(v[e4 + e]));
                            }
                        } else {
                            const float4 s4 = *reinterpret_cast<const float4*>(sxv + cb + e4);
                            const int c = (cb + e4) / 2;
                            if (VARIANT != 1) {
                                acc_w4a8(acc[c], v[e4], v[e4 + 1], s4.x, s4.y, w2);
                                acc_w4a8(acc[c + 1], v[e4 + 2], v[e4 + 3], s4.z, s4.w, w2);
                            } else {
                                acc_affine(acc[c], v[e4], v[e4 + 1], s4.x, s4.y, b2, w2);
                                acc_affine(acc[c + 1], v[e4 + 2], v[e4 + 3], s4.z, s4.w, b2, w2);
                            }
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&d_empty[db]);
                ring_next<DS>(db, dph);
                __syncwarp();
                if (lane == 0) mbar_arrive(&x_empty[xs]);
                ring_next<XS>(xs, xph);
            }
            if (!DEBUG && ok && n < sh.N) {
#pragma unroll
                for (int c = 0; c < MAXC; ++c) {
                    const int m = m0 + c;
                    const uint32_t bits = (uint32_t)(c & 1 ? acc[c / 2] >> 32 : acc[c / 2]);
                    if (c < ncol && m < sh.M)
                        Y[(size_t)m * sh.N + n] = VARIANT == 2 ? __uint_as_float(bits) * out_scale : __uint_as_float(bits);
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
template <int VARIANT, int GROUP, bool A_TMEM, bool DEBUG, int MAXC, int EXPW = 4>
cudaError_t run_gemm(const LaunchCtx& c, const CUtensorMap& map, const GemmShape& sh_in, const uint8_t* blob,
                     const float* act_scale, float* Y, int32_t* P)
{
    auto kern = gemm_kernel<VARIANT, GROUP, A_TMEM, DEBUG, MAXC, EXPW>;
    GemmShape sh = sh_in;
    sh.tmem_cols = gemm_tmem_cols<VARIANT, GROUP, MAXC>(sh.d_stride, !A_TMEM);
    sh.bs = gemm_kstages<VARIANT, GROUP, MAXC>(!A_TMEM);
    const size_t smem = gemm_smem_bytes<VARIANT, GROUP, MAXC>(sh.m_tile, sh.d_stride, !A_TMEM);
    // the epilogue reads MAXC columns from its first column on: they must lie
    // inside the accumulator buffer (and the scale stage's sx region)
    const int first_col = EXPW == 8 ? 0 : sh.m_tile / 2;
    if (!DEBUG && first_col + MAXC > sh.d_stride) return cudaErrorInvalidValue;
    static KernelSmem configured;
    cudaError_t e = ensure_smem(configured, c, kern, smem);
    if (e != cudaSuccess) return e;
    static std::atomic<int> regs_seen{0};
    int regs = regs_seen.load(std::memory_order_relaxed);
    if (regs == 0) {
        // the setmaxnreg split draws on the launch's 128 registers per thread
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, kern);
        if (e != cudaSuccess) return e;
        regs = fa.numRegs;
        regs_seen.store(regs, std::memory_order_relaxed);
    }
    if (regs * kGemmThreads != 65536) return cudaErrorInvalidConfiguration;
    // blocks per SM for this shared-memory size (the same on every supported
    // device), asked once and cached as one word: shared-memory bytes << 8 | blocks
    static std::atomic<uint64_t> occ_cache{0};
    const uint64_t cached = occ_cache.load(std::memory_order_relaxed);
    int occ = (cached >> 8) == (uint64_t)smem ? (int)(cached & 0xFF) : 0;
    if (occ == 0) {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kGemmThreads, smem);
        if (e != cudaSuccess) return e;
        if (occ < 1) return cudaErrorInvalidConfiguration;
        occ_cache.store(((uint64_t)smem << 8) | (uint64_t)(occ & 0xFF), std::memory_order_relaxed);
    }
    int per_sm = occ;
    if (per_sm * sh.tmem_cols > 512) per_sm = 512 / sh.tmem_cols;
    const int grid = sh.num_tiles < c.num_sms * per_sm ? sh.num_tiles : c.num_sms * per_sm;
    return launch(kern, dim3(grid), dim3(kGemmThreads), smem, c, map, sh, blob, act_scale, Y, P, c.status);
}

}  // namespace qmm
