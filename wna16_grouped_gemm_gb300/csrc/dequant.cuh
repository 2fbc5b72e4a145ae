// Exact WNA16 dequantisation helpers shared by the grouped GEMM kernels:
// packed INT32 words of 2- or 4-bit codes -> BF16 pairs for the TMEM A operand,
// plus the clamped SwiGLU and the interleaved K orders.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

namespace wna16 {

// ------------------------------------------------------------------ dequant
//
// (a & b) | c in one LOP3.  Written out because with both b and c constant the
// compiler otherwise emits two logic instructions (one immediate per LOP3),
// which nearly doubles the integer-pipe work of the dequantisation.
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// 2-bit fields: in BF16, 0x4300 is 128.0
// with a unit last place, so OR-ing a field q into mantissa bits 2i..2i+1
// reads 128 + 4^i q.  One bf16x2 add of -(128 + 2*4^i) gives 4^i * code exactly,
// and one bf16x2 multiply by bf16(scale) / 4^i gives code * bf16(scale), which
// for 2-bit codes (0 or +-2^j) IS bf16_rne(code * scale).  A register pairs
// field c (low half) with field c+8 (high half) of a word, so within every
// 16-k block the A operand's K order is (0, 8, 1, 9, ..., 7, 15); the token
// operand is stored in that order too (gather kernel, w13 epilogue).
__device__ __forceinline__ uint32_t bf2_add(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t bf2_mul(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
constexpr uint32_t kBf2Magic = 0x43004300u;    // (128.0, 128.0)
constexpr uint32_t kBf2Neg130 = 0xC302C302u;   // -(128 + 2)
constexpr uint32_t kBf2Neg136 = 0xC308C308u;   // -(128 + 8)
constexpr uint32_t kBf2Neg160 = 0xC320C320u;   // -(128 + 32)

struct Scale2 {  // bf16(s) / 4^i as bf16x2, i = 0, 1, 2
    uint32_t s0, s1, s2;
    __device__ __forceinline__ explicit Scale2(float s) {
        const float sb = __bfloat162float(__float2bfloat16_rn(s));
        s0 = pack_bf16x2(sb, sb);
        s1 = pack_bf16x2(sb * 0.25f, sb * 0.25f);
        s2 = pack_bf16x2(sb * 0.0625f, sb * 0.0625f);
    }
};

__device__ __forceinline__ void dequant_word2_pairs(uint32_t w, const Scale2& c, uint32_t* o) {
    const uint32_t w6 = w >> 6, w12 = w >> 12;
    o[0] = bf2_mul(bf2_add(and_or(w, 0x00030003u, kBf2Magic), kBf2Neg130), c.s0);    // fields 0, 8
    o[1] = bf2_mul(bf2_add(and_or(w, 0x000C000Cu, kBf2Magic), kBf2Neg136), c.s1);    // fields 1, 9
    o[2] = bf2_mul(bf2_add(and_or(w, 0x00300030u, kBf2Magic), kBf2Neg160), c.s2);    // fields 2, 10
    o[3] = bf2_mul(bf2_add(and_or(w6, 0x00030003u, kBf2Magic), kBf2Neg130), c.s0);   // fields 3, 11
    o[4] = bf2_mul(bf2_add(and_or(w6, 0x000C000Cu, kBf2Magic), kBf2Neg136), c.s1);   // fields 4, 12
    o[5] = bf2_mul(bf2_add(and_or(w6, 0x00300030u, kBf2Magic), kBf2Neg160), c.s2);   // fields 5, 13
    o[6] = bf2_mul(bf2_add(and_or(w12, 0x00030003u, kBf2Magic), kBf2Neg130), c.s0);  // fields 6, 14
    o[7] = bf2_mul(bf2_add(and_or(w12, 0x000C000Cu, kBf2Magic), kBf2Neg136), c.s1);  // fields 7, 15
}

// Group-accumulate mode (2-bit codes, scales applied per group after the MMA):
// the A operand is the plain code.  A field q OR-ed into mantissa bits 2i..2i+1
// of 128.0 reads 128 + 4^i q; one bf16x2 FMA by 4^-i with addend
// -(128 * 4^-i + 2) gives q - 2 = code exactly (the product is exact and the
// exact sum is a small integer, so the single rounding has nothing to round).
__device__ __forceinline__ uint32_t bf2_fma(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
constexpr uint32_t kBf2One = 0x3F803F80u;       // 1
constexpr uint32_t kBf2Quarter = 0x3E803E80u;   // 1/4
constexpr uint32_t kBf2Sixteenth = 0x3D803D80u; // 1/16
constexpr uint32_t kBf2Neg34 = 0xC208C208u;     // -(32 + 2)
constexpr uint32_t kBf2Neg10 = 0xC120C120u;     // -(8 + 2)

__device__ __forceinline__ void dequant_word2_codes(uint32_t w, uint32_t* o) {
    const uint32_t w6 = w >> 6, w12 = w >> 12;
    o[0] = bf2_fma(and_or(w, 0x00030003u, kBf2Magic), kBf2One, kBf2Neg130);        // fields 0, 8
    o[1] = bf2_fma(and_or(w, 0x000C000Cu, kBf2Magic), kBf2Quarter, kBf2Neg34);     // fields 1, 9
    o[2] = bf2_fma(and_or(w, 0x00300030u, kBf2Magic), kBf2Sixteenth, kBf2Neg10);   // fields 2, 10
    o[3] = bf2_fma(and_or(w6, 0x00030003u, kBf2Magic), kBf2One, kBf2Neg130);       // fields 3, 11
    o[4] = bf2_fma(and_or(w6, 0x000C000Cu, kBf2Magic), kBf2Quarter, kBf2Neg34);    // fields 4, 12
    o[5] = bf2_fma(and_or(w6, 0x00300030u, kBf2Magic), kBf2Sixteenth, kBf2Neg10);  // fields 5, 13
    o[6] = bf2_fma(and_or(w12, 0x00030003u, kBf2Magic), kBf2One, kBf2Neg130);      // fields 6, 14
    o[7] = bf2_fma(and_or(w12, 0x000C000Cu, kBf2Magic), kBf2Quarter, kBf2Neg34);   // fields 7, 15
}

// Offset codes (group-accumulate mode with a per-token correction): the field
// is OR-ed into a magic number whose exponent makes its weight 1, so the BF16
// reads off + q with off = 128, 32 or 8 for mantissa bits 0-1, 2-3 or 4-5,
// one LOP3 per pair and no arithmetic.  With code = q - 2 the MMA sums
// sum_k (code_k + off_k + 2) x_k; the epilogue subtracts the token's
// sum_k (off_k + 2) x_k over the group, computed where the token operand is
// written.  By k mod 8 the weight off + 2 is 130, 34, 10, 130, 34, 10, 130, 34.
constexpr uint32_t kBf2Magic32 = 0x42004200u;   // (32.0, 32.0)
constexpr uint32_t kBf2Magic8 = 0x41004100u;    // (8.0, 8.0)
__device__ __forceinline__ void offset_word2_codes(uint32_t w, uint32_t* o) {
    const uint32_t w6 = w >> 6, w12 = w >> 12;
    o[0] = and_or(w, 0x00030003u, kBf2Magic);      // fields 0, 8:  128 + q
    o[1] = and_or(w, 0x000C000Cu, kBf2Magic32);    // fields 1, 9:  32 + q
    o[2] = and_or(w, 0x00300030u, kBf2Magic8);     // fields 2, 10: 8 + q
    o[3] = and_or(w6, 0x00030003u, kBf2Magic);     // fields 3, 11
    o[4] = and_or(w6, 0x000C000Cu, kBf2Magic32);   // fields 4, 12
    o[5] = and_or(w6, 0x00300030u, kBf2Magic8);    // fields 5, 13
    o[6] = and_or(w12, 0x00030003u, kBf2Magic);    // fields 6, 14
    o[7] = and_or(w12, 0x000C000Cu, kBf2Magic32);  // fields 7, 15
}

// 64 consecutive k of one row -> 32 bf16x2 plain 2-bit codes, or offset codes
// with OFFSET (same layout as dequant_chunk<2>).
template <bool OFFSET>
__device__ __forceinline__ void codes_chunk2(const uint8_t* row, uint32_t xr, int chunk, uint32_t (&o)[32]) {
    const uint4 v = *reinterpret_cast<const uint4*>(row + ((static_cast<uint32_t>(chunk) ^ xr) << 4));
    if constexpr (OFFSET) {
        offset_word2_codes(v.x, o + 0);
        offset_word2_codes(v.y, o + 8);
        offset_word2_codes(v.z, o + 16);
        offset_word2_codes(v.w, o + 24);
    } else {
        dequant_word2_codes(v.x, o + 0);
        dequant_word2_codes(v.y, o + 8);
        dequant_word2_codes(v.z, o + 16);
        dequant_word2_codes(v.w, o + 24);
    }
}

// 4-bit fields, exact: bf16_rne(code * s) for an fp16 scale s.  With
// s_hi = bf16(s) and s_lo = s - s_hi (exact: an fp16 significand has 11 bits,
// so s_lo is a multiple of s's fp16 ulp of magnitude at most 4 of them, at
// most 2 significant bits), code * s = code * s_hi + code * s_lo exactly;
// t = code * s_lo has at most 3 + 2 significant bits and is exact in BF16, and
// one bf16x2 FMA code * s_hi + t rounds the exact sum once.  The code is read
// exactly: a field q OR-ed into the low mantissa bits of 128.0 reads 128 + q,
// and adding -136 gives q - 8.  Pair c of a word holds fields c and c + 4, so
// within every 8-k word the A operand's K order is (0, 4, 1, 5, 2, 6, 3, 7);
// the token operand is stored in that order too (gather kernel, w13
// epilogue).  Checked against the fp32 product rounded once for every finite
// fp16 scale and every code.
struct Scale4 {  // (s_hi, s_hi) and (s_lo, s_lo) as bf16x2
    uint32_t hi2, lo2;
    __device__ __forceinline__ explicit Scale4(float s) {
        const float hi = __bfloat162float(__float2bfloat16_rn(s));
        const float lo = s - hi;
        hi2 = pack_bf16x2(hi, hi);
        lo2 = pack_bf16x2(lo, lo);
    }
};

__device__ __forceinline__ uint32_t dequant_pair4(uint32_t fields, const Scale4& c) {
    const uint32_t q = bf2_add(and_or(fields, 0x000F000Fu, kBf2Magic), kBf2Neg136);   // codes, exact
    return bf2_fma(q, c.hi2, bf2_mul(q, c.lo2));
}

// One 4-bit word (8 consecutive k) -> 4 bf16x2 (fields (c, c + 4) in pair c).
__device__ __forceinline__ void dequant_word4(uint32_t w, const Scale4& c, uint32_t* o) {
    o[0] = dequant_pair4(w, c);
    o[1] = dequant_pair4(w >> 4, c);
    o[2] = dequant_pair4(w >> 8, c);
    o[3] = dequant_pair4(w >> 12, c);
}

// 64 consecutive k of one row (one TMEM A buffer row) -> 32 bf16x2.
// `row` = this row's packed bytes in the stage, `xr` = its swizzle XOR,
// `chunk` = which 64-k chunk of the stage.
template <int BITS>
__device__ __forceinline__ void dequant_chunk(const uint8_t* row, uint32_t xr, int chunk, float s,
                                              uint32_t (&o)[32]) {
    if constexpr (BITS == 2) {
        const uint4 v = *reinterpret_cast<const uint4*>(row + ((static_cast<uint32_t>(chunk) ^ xr) << 4));
        const Scale2 c(s);
        dequant_word2_pairs(v.x, c, o + 0);
        dequant_word2_pairs(v.y, c, o + 8);
        dequant_word2_pairs(v.z, c, o + 16);
        dequant_word2_pairs(v.w, c, o + 24);
    } else {
        const uint32_t j0 = static_cast<uint32_t>(2 * chunk);
        const uint4 v0 = *reinterpret_cast<const uint4*>(row + ((j0 ^ xr) << 4));
        const uint4 v1 = *reinterpret_cast<const uint4*>(row + (((j0 + 1) ^ xr) << 4));
        const Scale4 c(s);
        dequant_word4(v0.x, c, o + 0);
        dequant_word4(v0.y, c, o + 4);
        dequant_word4(v0.z, c, o + 8);
        dequant_word4(v0.w, c, o + 12);
        dequant_word4(v1.x, c, o + 16);
        dequant_word4(v1.y, c, o + 20);
        dequant_word4(v1.z, c, o + 24);
        dequant_word4(v1.w, c, o + 28);
    }
}

// Group 32: the first 32 k of a 64-k half take scale s_a, the second s_b
// (same layout and exact rounding as dequant_chunk).
template <int BITS>
__device__ __forceinline__ void dequant_chunk_g32(const uint8_t* row, uint32_t xr, int chunk, float s_a, float s_b,
                                                  uint32_t (&o)[32]) {
    if constexpr (BITS == 2) {
        // words of 16 k: x, y in the first 32 k, z, w in the second
        const uint4 v = *reinterpret_cast<const uint4*>(row + ((static_cast<uint32_t>(chunk) ^ xr) << 4));
        const Scale2 ca(s_a), cb(s_b);
        dequant_word2_pairs(v.x, ca, o + 0);
        dequant_word2_pairs(v.y, ca, o + 8);
        dequant_word2_pairs(v.z, cb, o + 16);
        dequant_word2_pairs(v.w, cb, o + 24);
    } else {
        // 16-byte vectors of 32 k: v0 the first 32 k, v1 the second
        const uint32_t j0 = static_cast<uint32_t>(2 * chunk);
        const uint4 v0 = *reinterpret_cast<const uint4*>(row + ((j0 ^ xr) << 4));
        const uint4 v1 = *reinterpret_cast<const uint4*>(row + (((j0 + 1) ^ xr) << 4));
        const Scale4 ca(s_a), cb(s_b);
        dequant_word4(v0.x, ca, o + 0);
        dequant_word4(v0.y, ca, o + 4);
        dequant_word4(v0.z, ca, o + 8);
        dequant_word4(v0.w, ca, o + 12);
        dequant_word4(v1.x, cb, o + 16);
        dequant_word4(v1.y, cb, o + 20);
        dequant_word4(v1.z, cb, o + 24);
        dequant_word4(v1.w, cb, o + 28);
    }
}

__device__ __forceinline__ float swiglu(float g, float u, float L) {
    g = fminf(g, L);
    u = fminf(fmaxf(u, -L), L);
    // fast exp / divide: their fp32 errors (a few ulp) are far below the BF16
    // rounding of h; for very negative g the divisor overflows and the
    // quotient is 0, as silu's is
    return __fdividef(g, 1.0f + __expf(-g)) * u;
}

// Position of element k in the interleaved K order of the A operand: mode 1
// (2-bit) (0, 8, 1, 9, ..., 7, 15) within each 16-k block, mode 2 (4-bit)
// (0, 4, 1, 5, 2, 6, 3, 7) within each 8-k block, mode 0 the natural order.
__device__ __forceinline__ int interleave_pos(int k, int mode) {
    if (mode == 1) {
        const int e = k & 15;
        return (k & ~15) | (e < 8 ? 2 * e : 2 * (e - 8) + 1);
    }
    if (mode == 2) {
        const int e = k & 7;
        return (k & ~7) | (e < 4 ? 2 * e : 2 * (e - 4) + 1);
    }
    return k;
}

}  // namespace wna16
