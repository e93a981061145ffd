// qmm_cq4.cuh -- codebook 4-bit (CQ4) weight expansion shared by the kernels.
//
// cactus PR #697 "SME2 acceleration for CQ4 matmul, prefill attention, and
// orthogonal embeddings", Summary: the GEMV leaf expands 4-bit codebook
// indices in-engine through a 16-entry table lookup (the SME2 LUTI4 with the
// table in ZT0), and the codebook scale is folded into the per-row norms so
// that one fp32 rescale remains.
//
// On GB300 the 16 int8 levels live in four registers and a lookup of four
// indices is three byte permutes: prmt picks a byte out of eight, so the low
// three index bits select within levels 0-7 and within levels 8-15, and a
// third prmt chooses between the two per byte from index bit 3. The blob is
// the symmetric variant's tile layout with the raw indices as nibbles and a
// 32-byte trailer after the chunks: the 16 levels (int8), cb_scale (fp32),
// 12 zero bytes.
#pragma once

#include <stdint.h>

namespace qmm {

constexpr int kCq4TrailerBytes = 32;

// The codebook of one matrix: byte j of t[q] is level 4q + j.
struct Cq4Book {
    uint32_t t0, t1, t2, t3;
    float scale;   // cb_scale
};

__host__ __device__ inline size_t cq4_trailer_offset(int N, int K, int group)
{
    return (size_t)((N + 127) / 128) * (size_t)(K / group) * (size_t)(64 * group + 256);
}

// `xor_bytes` is applied to every level (0x80808080 turns int8 levels c into
// the unsigned bytes c + 128 that the fp16 expansion of the tensor-core path
// wants; 0 keeps them signed for dp4a).
__device__ __forceinline__ Cq4Book cq4_load(const uint8_t* trailer, uint32_t xor_bytes = 0u)
{
    const uint4 v = *reinterpret_cast<const uint4*>(trailer);
    Cq4Book b;
    b.t0 = v.x ^ xor_bytes;
    b.t1 = v.y ^ xor_bytes;
    b.t2 = v.z ^ xor_bytes;
    b.t3 = v.w ^ xor_bytes;
    b.scale = *reinterpret_cast<const float*>(trailer + 16);
    return b;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Levels of the 8 indices of one packed word. Slots 0-3 (bits 0-15) hold the
// indices of k = 0, 2, 4, 6 of the word's 8-block, slots 4-7 those of
// k = 1, 3, 5, 7: lo4 = levels of k = 0, 2, 4, 6 (byte e <- slot e), hi4 = of
// k = 1, 3, 5, 7. prmt reads selector bits 0-15 only; a selector nibble with
// bit 3 set would replicate a sign, so the first lookups use the low three
// index bits and the final prmt takes byte e from the upper table (bytes 4-7)
// when bit 3 of index e is set.
__device__ __forceinline__ void cq4_expand(const Cq4Book& b, uint32_t w, uint32_t& lo4, uint32_t& hi4)
{
    const uint32_t m = w & 0x77777777u;
    const uint32_t s = ((w >> 1) & 0x44444444u) | 0x32103210u;
    lo4 = prmt(prmt(b.t0, b.t1, m), prmt(b.t2, b.t3, m), s);
    const uint32_t mh = m >> 16, sh = s >> 16;
    hi4 = prmt(prmt(b.t0, b.t1, mh), prmt(b.t2, b.t3, mh), sh);
}

}  // namespace qmm
