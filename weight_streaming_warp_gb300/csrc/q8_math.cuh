// q8_math.cuh -- the per-block arithmetic of the activation quantizer, shared by the
// standalone quantizer and the mat-vec that quantizes its own activation, so that the
// two produce the same bytes.
//
// Source: "QuantizeQ8KK is thread-per-superblock: 95.5us/call ..." (vllm.cpp issue),
// sections Cause and The donor: a per-element decomposition with a warp reduction for
// the block scale.  A lane owns 8 consecutive values; a block of BLOCK values is
// BLOCK / 8 adjacent lanes.
//
// Per block: amax = max |x|; d = amax / 127 (IEEE fp32 division);
// q = round-half-away(x / d) (IEEE fp32 division by the fp32 d, then roundf),
// clamped to [-127, 127]; a block whose d is +0 (all zero, or an amax of at most
// 63.5 subnormal steps, so that amax / 127 rounds to +0) has q = 0.
#pragma once

#include "common.cuh"

namespace wsw {
namespace q8m {

// amax over the block of this lane's 8 values; every lane of the warp must call it.
template <int BLOCK>
__device__ __forceinline__ float block_amax(const float (&v)[8]) {
    constexpr int LPB = BLOCK / 8;  // lanes per block
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
    for (int off = LPB / 2; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(WSW_FULL_MASK, amax, off));
    return amax;
}

__device__ __forceinline__ float scale(float amax) { return __fdiv_rn(amax, 127.0f); }

// The exact code of one value: clamp(round-half-away(fl(v / d)), -127, 127).
__device__ __forceinline__ int code_exact(float v, float d) {
    const float t = fminf(fmaxf(roundf(__fdiv_rn(v, d)), -127.0f), 127.0f);
    return static_cast<int>(t);
}

// The 8 codes of this lane, packed little-endian into two words.
//
// Division by d is replaced by a product with r = fl(1 / d).  With the standard model
// fl(a op b) = (a op b)(1 + e), |e| <= 2^-24, and |v| <= amax, so that
// |v / d| <= 127 (1 + 2^-23): t = fl(v * r) = (v / d)(1 + e1)(1 + e2) lies within
// |v / d| (2^-23 + 2^-48) < 1.6e-5 of v / d, and fl(v / d) within half an ulp at 128
// (3.9e-6) of it, so t and fl(v / d) differ by less than 2.0e-5 < 2^-14.
// Rounding to the nearest integer can then only differ when a half-integer lies within
// 2^-14 of t; if any of the lane's 8 values is that close, all 8 take the exact
// quotient (rare).  Away from half-integers round-half-even equals round-half-away, and
// round-half-even of |t| < 2^22 is the integer in the low bits of fl(t + 1.5 * 2^23):
// its low byte is the code's two's-complement byte (|t| < 127.5, so no clamp is
// reached).  A scale outside [1e-37, 1e37] takes the exact path for every value.
__device__ __forceinline__ void codes(const float (&v)[8], float amax, float d, uint32_t (&packed)[2]) {
    (void)amax;
    packed[0] = packed[1] = 0u;
    if (d == 0.0f) return;  // x / d undefined: the block is stored as zero
    constexpr float kRound = 12582912.0f;  // 1.5 * 2^23
    const float r = __frcp_rn(d);
    uint32_t u[8];
    float worst = 0.0f;  // largest |t - round(t)| of the lane
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float t = __fmul_rn(v[i], r);
        const float s = __fadd_rn(t, kRound);
        u[i] = __float_as_uint(s);
        worst = fmaxf(worst, fabsf(__fsub_rn(t, __fsub_rn(s, kRound))));
    }
    if (d >= 1.0e-37f && d <= 1.0e37f && worst < 0.5f - 6.103515625e-05f) {  // 2^-14 from a tie
        packed[0] = __byte_perm(__byte_perm(u[0], u[1], 0x0040), __byte_perm(u[2], u[3], 0x0040), 0x5410);
        packed[1] = __byte_perm(__byte_perm(u[4], u[5], 0x0040), __byte_perm(u[6], u[7], 0x0040), 0x5410);
        return;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
        packed[i >> 2] |= (static_cast<uint32_t>(code_exact(v[i], d)) & 0xffu) << (8 * (i & 3));
}

}  // namespace q8m
}  // namespace wsw
