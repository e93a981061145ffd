// qmm_gemm_narrow_e4m3.cu -- tensor-core GEMM of the symmetric W4A8 variant
// for up to 16 activation rows, group 128, with the weights in the MMA's N
// slot and both operands in e4m3 (tcgen05.mma kind::f8f6f4).
//
// Sources: cactus PR #697 "SME2 acceleration for CQ4 matmul, prefill
// attention, and orthogonal embeddings", Summary ("Fused SME2 GEMM (M>1)":
// raw int32 partials, then a separate fp32 rescale); geistlib issue #500
// "native W*A8 int8 GEMM for prefill" (no dequantized weights in DRAM).
//
// GB300 design. The fp16 form of the weights-in-N kernel (qmm_gemm_narrow.cu)
// spends its time moving the expanded 16-bit weight operand through shared
// memory and issuing one MMA per 16 k. Here every operand byte is an e4m3
// number, and every value involved is a small integer that e4m3 holds exactly:
//   - weights: the offset-binary nibble u = q + 8 in [0, 15];
//   - activations: the int8 code a = 16 hi + lo, split into two planes,
//     16 hi with hi = floor(a / 16) in [-8, 7], and lo = a mod 16 in [0, 15].
// A kind::f8f6f4 MMA takes 32 k per instruction and sums these products
// exactly in fp32 (a probe over worst-case operands, sums up to 2^20, matched
// integer arithmetic everywhere), and the weight operand is one byte per
// weight instead of two.
//
// The activation operand stage holds, in each of the four tensor-memory lane
// quadrants (rows 32 c .. 32 c + 31), the hi plane of activation rows 0..15
// followed by their lo plane. Per 32-k chunk two MMAs accumulate into the
// same columns: one reads the stage as it is, the other through a descriptor
// 16 rows further on, so that lanes 32 c .. 32 c + 15 first take the hi rows
// and then the lo rows. Those lanes end with sum_k a u exactly (the other
// lanes hold sums nobody reads), and the raw partial is
//   P = sum_k a u - 8 sum_k a,
// an exact integer in fp32. The group sums of a are formed with the planes.
// The epilogue subtracts 8 sum a and rescales acc += (P * sx) * sw in group
// order: the same operations on the same exact partials as the other
// tensor-core kernels, so the outputs are the same bits.
//
// Per 128-k group: 8 expand warps turn 256 rows of nibbles into e4m3 bytes
// (two byte permutes and an OR per 4 weights: a selector nibble with bit 3
// set makes prmt replicate the sign of the picked byte, which is 0 for
// these positive tables, so each lookup yields zero where the other half of
// the table applies). The activation warp copies the group's planes from
// shared memory into the four lane-quadrant copies of the operand. The MMA
// warp issues 8 MMAs into the group's accumulator (256 columns, two buffers).
//
// The planes of all of K are built once per block at its start (the codes
// are the same for every weight tile) in a k order that matches the
// expanded weights: within each 8-k block, k = 0, 2, 4, 6, 1, 3, 5, 7. That is
// the order of the nibble slots in a packed word.
//
// The packed weights arrive by bulk copies of chunk pairs into a two-stage
// ring (all the shared memory the operand stages and the planes leave), so a
// chunk's refill can start only when its previous use releases it, and the
// refill's latency paces the groups. The expand warps therefore release a
// chunk as soon as its words are in registers, before the lookups, and the
// producer prefetches the chunks six groups ahead into L2.
//
// Persistent over pairs of 128-row weight tiles; every wait bounded.
#include <cuda_fp16.h>

#include "qmm.h"
#include "qmm_e4m3.cuh"
#include "qmm_gemm.cuh"

namespace qmm {

namespace {

using namespace e4m3;

constexpr int kE8Group = 128;
constexpr int kE8ExpandWarps = 8;
constexpr int kE8EpiWarps = 8;
constexpr int kE8Threads = 32 * (kE8ExpandWarps + kE8EpiWarps + 3);   // + weight producer, activation, MMA
constexpr int kE8Rows = 256;                  // weight rows per MMA (N)
constexpr int kE8MaxM = 16;                   // activation rows
constexpr int kE8CB = 64 * kE8Group + 256;    // packed chunk: one 128-row tile, one group
constexpr int kE8AStage = 128 * 128;          // activation operand: 4 x 32 rows x 128 k
constexpr int kE8APad = 16 * 128;             // the lo-plane descriptor reads 16 rows past a stage
constexpr int kE8BStage = kE8Rows * 128;      // weight operand: 256 rows x 128 k
constexpr int kE8Plane = 32 * 128;            // one group's hi and lo rows
constexpr int kE8XB = kE8Rows * 4;            // scale stage: sw of the 256 rows
constexpr int kE8RA = 2, kE8RB = 3, kE8RW = 2, kE8RX = 4, kE8DS = 2;
constexpr int kE8Prefetch = 6;               // groups ahead of the bulk copies, into L2
constexpr int kE8Bars = 2 * kE8RW + 2 * kE8RA + 2 * kE8RB + 2 * kE8RX + 2 * kE8DS + 2;

size_t e8_smem_bytes(int G)
{
    return 1024 + (size_t)kE8RA * kE8AStage + kE8APad + (size_t)kE8RB * kE8BStage + (size_t)G * kE8Plane +
           (size_t)kE8RW * 2 * kE8CB + (size_t)kE8RX * kE8XB + 8 * kE8Bars + 16 + (size_t)2 * G * kE8MaxM * 4;
}

// Grid (P): block b takes weight-tile pairs b, b + P, ... over all of K.
__global__ void __launch_bounds__(kE8Threads, 1)
    gemm_narrow_e4m3_kernel(int M, int N, int K, const uint8_t* __restrict__ blob, const uint16_t* __restrict__ act16,
                            const float* __restrict__ sx, float* __restrict__ Y, int* status)
{
    const int G = K / kE8Group, T = (N + 127) / 128, TP = (T + 1) / 2;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* ast = base;                                        // [RA][128 rows][128 B]
    uint8_t* bst = ast + (size_t)kE8RA * kE8AStage + kE8APad;  // [RB][256 rows][128 B]
    uint8_t* res = bst + (size_t)kE8RB * kE8BStage;            // [G][32 rows][128 B] planes
    uint8_t* wst = res + (size_t)G * kE8Plane;                  // [RW][2 chunks]
    uint8_t* xst = wst + (size_t)kE8RW * 2 * kE8CB;            // [RX][sw of 256 rows]
    uint64_t* bars = reinterpret_cast<uint64_t*>(xst + (size_t)kE8RX * kE8XB);
    uint64_t* w_full = bars;                 // chunk pair landed
    uint64_t* w_empty = w_full + kE8RW;      // expand warps have read it
    uint64_t* a_full = w_empty + kE8RW;      // activation operand stored
    uint64_t* a_empty = a_full + kE8RA;      // MMA commit
    uint64_t* b_full = a_empty + kE8RA;      // expand warps stored the group's weights
    uint64_t* b_empty = b_full + kE8RB;      // MMA commit
    uint64_t* x_full = b_empty + kE8RB;      // expand warps stored the group's weight scales
    uint64_t* x_empty = x_full + kE8RX;      // epilogue warps are done with them
    uint64_t* d_full = x_empty + kE8RX;      // MMA commit after the group's MMAs
    uint64_t* d_empty = d_full + kE8DS;      // epilogue warps loaded the partials
    uint64_t* done = d_empty + kE8DS;
    uint64_t* planes_ready = done + 1;       // epilogue warps built the planes and group sums
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(planes_ready + 1);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
    float* sx_all = reinterpret_cast<float*>(tmem_slot + 4);   // [G][16] activation scales
    float* corr = sx_all + (size_t)G * kE8MaxM;                // [G][16] 8 * sum of the group's codes

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int kProducer = kE8ExpandWarps + kE8EpiWarps, kAct = kProducer + 1, kMma = kProducer + 2;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kE8RW; ++i) {
            mbar_init(&w_full[i], 1);
            mbar_init(&w_empty[i], kE8ExpandWarps);
        }
        for (int i = 0; i < kE8RA; ++i) {
            mbar_init(&a_full[i], 1);
            mbar_init(&a_empty[i], 1);
        }
        for (int i = 0; i < kE8RB; ++i) {
            mbar_init(&b_full[i], kE8ExpandWarps);
            mbar_init(&b_empty[i], 1);
        }
        for (int i = 0; i < kE8RX; ++i) {
            mbar_init(&x_full[i], kE8ExpandWarps);
            mbar_init(&x_empty[i], kE8EpiWarps);
        }
        for (int i = 0; i < kE8DS; ++i) {
            mbar_init(&d_full[i], 1);
            mbar_init(&d_empty[i], kE8EpiWarps);
        }
        mbar_init(done, 1);
        mbar_init(planes_ready, kE8EpiWarps);
        *abort = 0;
        fence_barrier_init();
    }
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
                const uint8_t* src0 = blob + (size_t)(2 * tp) * G * kE8CB;
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
                    uint8_t* dst = wst + (size_t)ws * 2 * kE8CB;
                    mbar_arrive_expect_tx(&w_full[ws], (uint32_t)(two ? 2 * kE8CB : kE8CB));
                    bulk_g2s(dst, src0 + (size_t)g * kE8CB, kE8CB, &w_full[ws]);
                    if (two) bulk_g2s(dst + kE8CB, src0 + (size_t)(G + g) * kE8CB, kE8CB, &w_full[ws]);
                    // the chunks kE8Prefetch groups ahead into L2: one block per SM
                    // holds only kE8RW chunk pairs in shared memory, too few bytes
                    // in flight to cover HBM latency at full bandwidth
                    {
                        const int ahead = issued + kE8Prefetch, tpa = (int)blockIdx.x + (ahead / G) * (int)gridDim.x;
                        if (tpa < TP) {
                            const uint8_t* srca = blob + (size_t)(2 * tpa) * G * kE8CB + (size_t)(ahead % G) * kE8CB;
                            bulk_prefetch_l2(srca, kE8CB);
                            if (2 * tpa + 1 < T) bulk_prefetch_l2(srca + (size_t)G * kE8CB, kE8CB);
                        }
                    }
                    ++issued;
                    ring_next<kE8RW>(ws, wph);
                }
            }
            // no copy may still be landing when the block exits
            for (int i = issued - kE8RW > 0 ? issued - kE8RW : 0; i < issued; ++i)
                mbar_wait(&w_full[i % kE8RW], (i / kE8RW) & 1, status, nullptr);
        }
    } else if (warp == kAct) {
        // ---------------------------------------------------------- activation operand
        // lane l copies plane row l (hi of row l, or lo of row l - 16) of the
        // group into rows l, 32 + l, 64 + l, 96 + l of the operand: the
        // 128-byte swizzle depends on the row mod 8 only, so the 16-byte
        // pieces move unchanged
        bool ok = mbar_wait(planes_ready, 0, status, abort);
        int as = 0;
        uint32_t aph = 0;
        for (int tp = blockIdx.x; ok && tp < TP; tp += gridDim.x) {
            for (int g = 0; g < G; ++g) {
                if (!mbar_wait(&a_empty[as], aph ^ 1u, status, abort)) {
                    ok = false;
                    break;
                }
                // lane l moves piece (c + l) mod 8 in step c: the eight lanes of
                // each shared-memory wavefront then touch eight different
                // 16-byte bank groups (rows are 128 bytes apart)
                const uint8_t* src = res + (size_t)g * kE8Plane + lane * 128;
                uint8_t* dst = ast + (size_t)as * kE8AStage + lane * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const int pc = 16 * ((c + lane) & 7);
                    const uint4 u = *reinterpret_cast<const uint4*>(src + pc);
#pragma unroll
                    for (int q = 0; q < 4; ++q) *reinterpret_cast<uint4*>(dst + q * 4096 + pc) = u;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&a_full[as]);
                ring_next<kE8RA>(as, aph);
            }
        }
    } else if (warp == kMma) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_f16_f32(128, kE8Rows);   // format fields 0: e4m3 A and B
            int as = 0, bs = 0, db = 0;
            uint32_t aph = 0, bph = 0, dph = 0;
            bool ok = true;
            for (int tp = blockIdx.x; ok && tp < TP; tp += gridDim.x) {
                for (int g = 0; g < G; ++g) {
                    if (!mbar_wait(&d_empty[db], dph ^ 1u, status, abort) ||
                        !mbar_wait(&a_full[as], aph, status, abort) || !mbar_wait(&b_full[bs], bph, status, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem + (uint32_t)(db * kE8Rows);
                    const uint64_t adesc = sdesc_sw128(smem_u32(ast + (size_t)as * kE8AStage));
                    const uint64_t bdesc = sdesc_sw128(smem_u32(bst + (size_t)bs * kE8BStage));
                    // per 32-k chunk: the hi rows, then the lo rows (the
                    // descriptor 16 rows = 2048 bytes further on) into the same lanes
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        mma_e4m3_ss(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, kk > 0 ? 1u : 0u);
                        mma_e4m3_ss(d_tmem, adesc + 128 + 2 * kk, bdesc + 2 * kk, idesc, 1u);
                    }
                    tc_commit(&a_empty[as]);
                    tc_commit(&b_empty[bs]);
                    tc_commit(&d_full[db]);
                    ring_next<kE8RA>(as, aph);
                    ring_next<kE8RB>(bs, bph);
                    ring_next<kE8DS>(db, dph);
                }
            }
            // every issued MMA must retire before the allocation is released
            tc_commit(done);
            mbar_wait(done, 0, status, nullptr);
        }
    } else if (warp < kE8ExpandWarps) {
        // ---------------------------------------------------------- expand
        // thread t: row t of the 256-row operand (tile t / 128 of the pair)
        const int t = threadIdx.x, half = t >> 7, r = t & 127;
        pdl_wait();   // sx comes from the previous kernel
        // every group's activation scales, once (rows beyond M: zero); the
        // epilogue reads them after the group's x_full, which these warps
        // arrive on after this
        for (int i = t; i < G * kE8MaxM; i += 32 * kE8ExpandWarps) {
            const int m = i % kE8MaxM, gi = i / kE8MaxM;
            sx_all[i] = m < M ? sx[(size_t)m * G + gi] : 0.f;
        }
        int ws = 0, bs = 0, xs = 0;
        uint32_t wph = 0, bph = 0, xph = 0;
        bool ok = true;
        for (int tp = blockIdx.x; ok && tp < TP; tp += gridDim.x) {
            for (int g = 0; g < G; ++g) {
                if (!mbar_wait(&w_full[ws], wph, status, abort) || !mbar_wait(&x_empty[xs], xph ^ 1u, status, abort)) {
                    ok = false;
                    break;
                }
                const uint8_t* ch = wst + (size_t)ws * 2 * kE8CB + (size_t)half * kE8CB;
                // the group's weight scale of this row
                float* xsp = reinterpret_cast<float*>(xst + (size_t)xs * kE8XB);
                xsp[t] = __half2float(reinterpret_cast<const __half*>(ch + 64 * kE8Group)[r]);
                __syncwarp();
                if (lane == 0) mbar_arrive(&x_full[xs]);
                ring_next<kE8RX>(xs, xph);
                if (!mbar_wait(&b_empty[bs], bph ^ 1u, status, abort)) {
                    ok = false;
                    break;
                }
                // piece p (16 bytes) of the row holds k = 32 p .. 32 p + 31, word
                // i of it k = 32 p + 8 i .. + 7; its 8 output bytes land at 32 p + 8 i
                // the row's 16 words, and the first step of their lookup, which
                // needs every loaded value: only then is the chunk released, so
                // that the producer can refill the stage while the lookups run
                // (with two chunk stages, the refill's latency paces the kernel)
                uint32_t w[16], xw[16];
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    const uint4 v = *reinterpret_cast<const uint4*>(ch + p * 2048 + r * 16);
                    w[4 * p] = v.x;
                    w[4 * p + 1] = v.y;
                    w[4 * p + 2] = v.z;
                    w[4 * p + 3] = v.w;
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) xw[i] = w[i] ^ 0x88888888u;
                // the release must follow the loads: an ordered asm statement
                // that takes every loaded value keeps the arrive after them
                asm volatile("" ::"r"(xw[0]), "r"(xw[1]), "r"(xw[2]), "r"(xw[3]), "r"(xw[4]), "r"(xw[5]), "r"(xw[6]),
                             "r"(xw[7]), "r"(xw[8]), "r"(xw[9]), "r"(xw[10]), "r"(xw[11]), "r"(xw[12]), "r"(xw[13]),
                             "r"(xw[14]), "r"(xw[15]));
                __syncwarp();
                if (lane == 0) mbar_arrive(&w_empty[ws]);
                uint32_t o[32];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    o[2 * i] = e4m3_u4(w[i], xw[i]);
                    o[2 * i + 1] = e4m3_u4(w[i] >> 16, xw[i] >> 16);
                }
                uint8_t* row = bst + (size_t)bs * kE8BStage + (size_t)t * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<uint4*>(row + ((c ^ (t & 7)) * 16)) =
                        make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&b_full[bs]);
                ring_next<kE8RB>(bs, bph);
                ring_next<kE8RW>(ws, wph);
            }
        }
    } else {
        // ---------------------------------------------------------- epilogue
        const int e = warp - kE8ExpandWarps;
        // the planes of all groups and 8 * (group sums), once: thread (m, j)
        // converts the 8-k block j of row m in every group
        {
            const int te = threadIdx.x - 32 * kE8ExpandWarps, m = te >> 4, j = te & 15;
            const bool live = m < M;
            pdl_wait();   // the codes come from the previous kernel
            const uint16_t* arow = act16 + (size_t)(live ? m : 0) * K + 8 * j;
            const uint32_t c1536 = 0x66006600u;   // fp16 1536 + a: low byte = a (two's complement)
            // four groups' codes in flight per round trip
            uint4 hb[4];
            for (int g = 0; g < G; ++g) {
                if ((g & 3) == 0) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        hb[i] = live && g + i < G ? __ldg(reinterpret_cast<const uint4*>(arow + (size_t)(g + i) * kE8Group))
                                                  : make_uint4(0u, 0u, 0u, 0u);
                }
                uint4 h = hb[0];
#pragma unroll
                for (int i = 1; i < 4; ++i)
                    if ((g & 3) == i) h = hb[i];
                uint32_t w4[4] = {h.x, h.y, h.z, h.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    __half2 v = __hadd2(*reinterpret_cast<__half2*>(&w4[i]), *reinterpret_cast<const __half2*>(&c1536));
                    w4[i] = *reinterpret_cast<uint32_t*>(&v);   // bytes 0, 2: codes of k = 2i, 2i + 1
                }
                const uint32_t x = prmt(w4[0], w4[1], 0x6240u);   // k = 0, 2, 1, 3
                const uint32_t y = prmt(w4[2], w4[3], 0x6240u);   // k = 4, 6, 5, 7
                const uint32_t ca = prmt(x, y, 0x5410u);          // k = 0, 2, 4, 6
                const uint32_t cb = prmt(x, y, 0x7632u);          // k = 1, 3, 5, 7
                uint32_t ha, la, hb, lb;
                split_codes(ca, ha, la);
                split_codes(cb, hb, lb);
                int sum = __dp4a((int)ca, 0x01010101, __dp4a((int)cb, 0x01010101, 0));
                sum += __shfl_xor_sync(0xffffffffu, sum, 8);
                sum += __shfl_xor_sync(0xffffffffu, sum, 4);
                sum += __shfl_xor_sync(0xffffffffu, sum, 2);
                sum += __shfl_xor_sync(0xffffffffu, sum, 1);
                if (j == 0) corr[g * kE8MaxM + m] = 8.f * (float)sum;
                // bytes 8 j .. 8 j + 7 of rows m (hi) and 16 + m (lo); row mod 8 = m mod 8
                const int off = (((j >> 1) ^ (m & 7)) << 4) + ((j & 1) << 3);
                uint8_t* pg = res + (size_t)g * kE8Plane;
                *reinterpret_cast<uint2*>(pg + m * 128 + off) = make_uint2(ha, hb);
                *reinterpret_cast<uint2*>(pg + (16 + m) * 128 + off) = make_uint2(la, lb);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(planes_ready);
        }
        // warp (quadrant q, column half h): lane m < 16 holds row m's sums of
        // weight rows c0 .. c0 + 31 (lanes 16-31 compute on sums nobody reads
        // and store nothing)
        const int q = warp & 3, hcol = e >> 2;
        const int c0 = 64 * q + 32 * hcol;
        const int m = lane & 15;
        const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)c0;
        int db = 0, xs = 0;
        uint32_t dph = 0, xph = 0;
        // the 32 columns read from either accumulator buffer lie inside the
        // 512-column allocation
        bool ok = in_range((kE8DS - 1) * kE8Rows + c0 + 32 <= 512, status);
        if (!ok) *abort = 1;
        // every warp's group sums are in place
        if (ok && !mbar_wait(planes_ready, 0, status, abort)) ok = false;
        for (int tp = blockIdx.x; ok && tp < TP; tp += gridDim.x) {
            unsigned long long acc[16];   // columns (2 i, 2 i + 1)
#pragma unroll
            for (int i = 0; i < 16; ++i) acc[i] = 0ull;
            for (int g = 0; g < G; ++g) {
                if (!mbar_wait(&d_full[db], dph, status, abort) || !mbar_wait(&x_full[xs], xph, status, abort)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float* xsp = reinterpret_cast<const float*>(xst + (size_t)xs * kE8XB) + c0;
                const unsigned long long sx2 = splat2(sx_all[g * kE8MaxM + m]);
                const unsigned long long c2 = splat2(corr[g * kE8MaxM + m]);
                const uint32_t ta = lane_base + (uint32_t)(db * kE8Rows);
                // two rounds of 16 columns (fewer live registers)
#pragma unroll
                for (int hc = 0; hc < 32; hc += 16) {
                    uint32_t v[16];
                    tmem_ld8_at(ta + hc, v, 0);
                    tmem_ld8_at(ta + hc + 8, v, 8);
                    tmem_ld_wait_n(v);
#pragma unroll
                    for (int c4 = 0; c4 < 16; c4 += 4) {
                        const float4 w4 = *reinterpret_cast<const float4*>(xsp + hc + c4);
                        acc_pair_corr(acc[(hc + c4) / 2], v[c4], v[c4 + 1], c2, sx2, w4.x, w4.y);
                        acc_pair_corr(acc[(hc + c4) / 2 + 1], v[c4 + 2], v[c4 + 3], c2, sx2, w4.z, w4.w);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&d_empty[db]);
                ring_next<kE8DS>(db, dph);
                __syncwarp();
                if (lane == 0) mbar_arrive(&x_empty[xs]);
                ring_next<kE8RX>(xs, xph);
            }
            if (!ok) break;
            if (lane < 16 && m < M) {
                const int n0 = 256 * tp + c0;
                float* yrow = Y + (size_t)m * N;
                float o[32];
#pragma unroll
                for (int c = 0; c < 32; ++c)
                    o[c] = __uint_as_float((uint32_t)(c & 1 ? acc[c / 2] >> 32 : acc[c / 2]));
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

}  // namespace

cudaError_t launch_gemm_narrow_e4m3(const LaunchCtx& c, int M, int N, int K, const uint8_t* blob,
                                    const uint16_t* act16, const float* sx, float* Y)
{
    if (M < 1 || M > kE8MaxM || K % kE8Group != 0) return cudaErrorInvalidValue;
    const size_t smem = e8_smem_bytes(K / kE8Group);
    if (smem > 227 * 1024) return cudaErrorNotSupported;   // K too long: the fp16 form takes it
    auto kern = gemm_narrow_e4m3_kernel;
    static KernelSmem configured;
    const cudaError_t e = ensure_smem(configured, c, kern, smem);
    if (e != cudaSuccess) return e;
    const int T = (N + 127) / 128, TP = (T + 1) / 2;
    const int grid = TP < c.num_sms ? TP : c.num_sms;
    return launch(kern, dim3(grid), dim3(kE8Threads), smem, c, M, N, K, blob, act16, sx, Y, c.status);
}

}  // namespace qmm
