// qmm_e4m3.cuh -- e4m3 encodings of the small integers on the W4A8 path, for
// the tcgen05.mma kind::f8f6f4 GEMMs: the offset-binary weight nibbles
// u = q + 8 in [0, 15] and the two planes of an int8 activation code,
// a = 16 hi + lo (16 hi, hi in [-8, 7], and lo in [0, 15]); all of them are
// exact e4m3 numbers, so the MMA's sums are the exact integer sums.
#pragma once

#include "qmm_cq4.cuh"   // prmt
#include "qmm_gemm.cuh"

namespace qmm {
namespace e4m3 {

// e4m3 bytes of u = 0..7 and 8..15 (u = 1: 0x38, 2: 0x40, ..., 8: 0x50, 15: 0x57).
constexpr uint32_t kU0 = 0x44403800u, kU1 = 0x4E4C4A48u, kU2 = 0x53525150u, kU3 = 0x57565554u;
// e4m3 bytes of 16 h for the nibble n = h mod 16: n = 0..7 (h = n) and 8..15 (h = n - 16).
constexpr uint32_t kP0 = 0x64605800u, kP1 = 0x6E6C6A68u, kN0 = 0xEAECEEF0u, kN1 = 0xD8E0E4E8u;

// e4m3 of the four nibbles u in selector bits 0-15 (byte e <- nibble e).
__device__ __forceinline__ uint32_t e4m3_u4(uint32_t s, uint32_t sx)
{
    return prmt(kU0, kU1, s) | prmt(kU2, kU3, sx);
}

// The eight weights of a packed word: bytes of k = 0, 2, 4, 6 and of 1, 3, 5, 7.
__device__ __forceinline__ void expand_word_e4m3(uint32_t w, uint32_t& a, uint32_t& b)
{
    const uint32_t x = w ^ 0x88888888u;
    a = e4m3_u4(w, x);
    b = e4m3_u4(w >> 16, x >> 16);
}

// Selector of the four low nibbles of the bytes of v (byte e -> nibble e).
__device__ __forceinline__ uint32_t nibble_sel(uint32_t v)
{
    const uint32_t t = v & 0x0F0F0F0Fu;
    return prmt(t | (t >> 4), 0u, 0x0020u);
}

// Hi and lo planes of four int8 codes (bytes of c): e4m3(16 floor(a / 16)) and e4m3(a mod 16).
__device__ __forceinline__ void split_codes(uint32_t c, uint32_t& hi, uint32_t& lo)
{
    const uint32_t sl = nibble_sel(c);
    lo = e4m3_u4(sl, sl ^ 0x8888u);
    const uint32_t sh = nibble_sel(c >> 4);
    const uint32_t s7 = sh & 0x7777u;
    hi = prmt(prmt(kP0, kP1, s7), prmt(kN0, kN1, s7), ((sh >> 1) & 0x4444u) | 0x3210u);
}

// acc += (((d0, d1) - (c, c)) * (sx, sx)) * (sw0, sw1): the partials P = d - c
// (exact), then the other tensor-core kernels' rescale (partial times the
// activation scale, then a fused multiply-add with the weight scale), two
// columns per instruction.
__device__ __forceinline__ void acc_pair_corr(unsigned long long& acc, uint32_t d0, uint32_t d1,
                                              unsigned long long c2, unsigned long long sx2, float sw0, float sw1)
{
    asm("{\n\t.reg .b64 t, w;\n\t"
        "mov.b64 t, {%1, %2};\n\t"
        "sub.rn.f32x2 t, t, %3;\n\t"
        "mul.rn.f32x2 t, t, %4;\n\t"
        "mov.b64 w, {%5, %6};\n\t"
        "fma.rn.f32x2 %0, t, w, %0;\n\t}"
        : "+l"(acc)
        : "r"(d0), "r"(d1), "l"(c2), "l"(sx2), "f"(sw0), "f"(sw1));
}

}  // namespace e4m3
}  // namespace qmm
