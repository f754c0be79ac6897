// q4a_block.cuh -- the dot product of four asymmetric 4-bit weight blocks
// with one staged q8_0 activation chunk.
//
// A weight block holds 32 values d * nib - m (f16 d, f16 m, unsigned 4-bit
// nib): the q4_K value form d*s*nib - dmin*m of "12 - r5-r6 re-ranking +
// structural rewrite spec" (sec. 3) with its two-level scales folded into one
// scale and one min per 32 elements.  Against a q8_0 activation block the min
// term needs no second dot product: m * d_a * sum_e q_e, and sum_e q_e is the
// int16 ssum that the plane carries for exactly this purpose ("54 - r51 -
// producer-fused A-quantize mode 1", sec. 2.1).
//
// Layout: a block is 20 bytes -- d at +0, m at +2, then byte j (j < 16) holds
// element j in its low nibble and element j + 16 in its high nibble -- so four
// blocks are 80 bytes = five 16-byte words, and every block is five whole
// 32-bit words.  One nibble word gives two dp4a operands: w & 0x0f0f0f0f
// (elements 4i..4i+3) and w & 0xf0f0f0f0, the high nibbles in place, read as
// unsigned bytes 16*nib (elements 16+4i..16+4i+3).  The second sum is 16 times
// the integer it stands for, so an arithmetic shift by 4 recovers it exactly;
// no shift per word is needed.
#pragma once

#include "q8_common.cuh"

namespace q8 {

constexpr int kA4ChunkWords = 20;   // 4 blocks x 5 words (80 bytes)
constexpr int kA4ChunkBytes = 80;

// dp4a of unsigned bytes (a) with signed bytes (b)
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Four blocks of one row (20 words) against a staged activation chunk: 128 B
// of codes, then the four blocks' d|ssum words.
__device__ __forceinline__ float a4_chunk(const uint32_t (&wv)[kA4ChunkWords], const uint8_t *ac, float acc)
{
    const uint4 dsv = *reinterpret_cast<const uint4 *>(ac + 128);
    const uint32_t dsw[4] = {dsv.x, dsv.y, dsv.z, dsv.w};
#pragma unroll
    for (int bb = 0; bb < 4; ++bb) {
        const uint4 a0 = *reinterpret_cast<const uint4 *>(ac + 32 * bb);
        const uint4 a1 = *reinterpret_cast<const uint4 *>(ac + 32 * bb + 16);
        const uint32_t aq[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        int lo = 0, hi16 = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t nw = wv[5 * bb + 1 + i];
            lo = dp4a_us(nw & 0x0f0f0f0fu, aq[i], lo);          // elements 4i .. 4i+3
            hi16 = dp4a_us(nw & 0xf0f0f0f0u, aq[4 + i], hi16);  // 16 x (elements 16+4i .. 16+4i+3)
        }
        const int isum = lo + (hi16 >> 4);  // |hi16| <= 16*16*15*127: exact
        const uint32_t dm = wv[5 * bb];
        const float dw = __half2float(__ushort_as_half(static_cast<unsigned short>(dm & 0xffffu)));
        const float mw = __half2float(__ushort_as_half(static_cast<unsigned short>(dm >> 16)));
        const float da = __half2float(__ushort_as_half(static_cast<unsigned short>(dsw[bb] & 0xffffu)));
        const int ssum = static_cast<int16_t>(static_cast<uint16_t>(dsw[bb] >> 16));
        // d*d_a and m*d_a are exact in f32 (11 + 11 significant bits)
        acc = __fmaf_rn(__fmul_rn(dw, da), static_cast<float>(isum), acc);
        acc = __fmaf_rn(-__fmul_rn(mw, da), static_cast<float>(ssum), acc);
    }
    return acc;
}

} // namespace q8
