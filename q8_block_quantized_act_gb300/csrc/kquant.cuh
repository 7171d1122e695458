// kquant.cuh -- the GGUF K-quant superblocks (256 weights each) that memra-engine 0.81.0
// f16_ffi.rs names beside Q8_0 and Q4_0: Q6_K (210 bytes), Q4_K (144 bytes), Q5_K (176 bytes),
// and the pieces of their layouts that the fp16 mirror, the dp4a GEMV and the tensor-core GEMV
// share.  Superblock layouts (the GGUF formats'), weight e = 0..255:
//   Q6_K: ql[128] | qh[64] | int8 scales[16] | fp16 d.  e = 128h + 32g + l: code = low 4 bits
//         from ql[64h + 32(g&1) + l] (low nibble for g < 2, high for g >= 2) + 16 * 2 bits
//         (qh[32h + l] >> 2g); value = d * scales[e/16] * (code - 32).
//   Q4_K: fp16 d | fp16 dmin | 12 scale bytes | qs[128].  Sub-block j = e/32 has a 6-bit scale
//         and min (j < 4: s[j] & 63, s[j+4] & 63; j >= 4: (s[j+4] & 15) | (s[j-4] >> 6) << 4,
//         (s[j+4] >> 4) | (s[j] >> 6) << 4); e = 64g + 32u + l: code = nibble u of qs[32g + l];
//         value = d * sc_j * code - dmin * m_j.
//   Q5_K: as Q4_K with qh[32] before qs; the code gains bit j of qh[l] as its fifth bit.
#pragma once

#include "common.cuh"

namespace q8 {

constexpr int QK_K = 256;

struct KQ6 {
    static constexpr int BYTES = 210;
    static constexpr int WORDS = 53;   // 212 bytes cover the superblock from any 2-byte offset
};
struct KQ4 {
    static constexpr int BYTES = 144;
    static constexpr int WORDS = 36;
};
struct KQ5 {
    static constexpr int BYTES = 176;
    static constexpr int WORDS = 44;
};

// The 6-bit scales and mins of all 8 sub-blocks of a Q4_K / Q5_K superblock, four to a word
// (byte j & 3 of the word for sub-block j; scales of sub-blocks 0..3 in sc_lo, 4..7 in sc_hi),
// unpacked from the 12 scale bytes (words w1..w3) with word-wide masks.
__device__ __forceinline__ void k4_scales_mins(uint32_t w1, uint32_t w2, uint32_t w3, uint32_t &sc_lo, uint32_t &mn_lo,
                                               uint32_t &sc_hi, uint32_t &mn_hi)
{
    sc_lo = w1 & 0x3F3F3F3Fu;
    mn_lo = w2 & 0x3F3F3F3Fu;
    sc_hi = (w3 & 0x0F0F0F0Fu) | ((w1 >> 2) & 0x30303030u);
    mn_hi = ((w3 >> 4) & 0x0F0F0F0Fu) | ((w2 >> 2) & 0x30303030u);
}

// Byte b (0..3) of w as the f32 value 2^23 + byte: the byte placed under the exponent of 2^23.
__device__ __forceinline__ float byte_magic(uint32_t w, int b)
{
    return __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7650u + (uint32_t)b));
}

// Four 6-bit Q6_K codes (one per byte) as the signed bytes code - 32: flip bit 5; where it is
// now set (code < 32) the byte is code + 32 and must become code + 32 - 64, i.e. gain bits 6
// and 7.
__device__ __forceinline__ uint32_t q6_signed_bytes(uint32_t code)
{
    const uint32_t t = code ^ 0x20202020u;
    const uint32_t s = t & 0x20202020u;
    return t | (s << 1) | (s << 2);
}

}  // namespace q8
