// q8_dot.cuh -- the canonical arithmetic of one q8_0 block product, shared by every
// CUDA-core q8_0 mat-vec (dense, fused with the quantizer, grouped over experts), so
// that they agree bit for bit.
//
// Source: "QuantizeQ8KK is thread-per-superblock: 95.5us/call ..." (vllm.cpp issue),
// section Scope: q8_0 blocks of 32 int8 values with one binary16 scale.
//
//   block contribution = fp32(Wd) * fp32(xd) * isum,  isum = sum of 32 int8 products
//
// isum is exact in int32 (|isum| <= 32 * 127^2) and in fp32 (< 2^24); Wd * xd is exact
// in fp32 (11 x 11 significant bits); one fused multiply-add adds the block.
#pragma once

#include <cuda_fp16.h>

#include "common.cuh"

namespace wsw {
namespace q8d {

__device__ __forceinline__ int dot32(const uint32_t (&w)[8], const uint4 &x0, const uint4 &x1) {
    int s0 = 0, s1 = 0;
    s0 = __dp4a(static_cast<int>(w[0]), static_cast<int>(x0.x), s0);
    s1 = __dp4a(static_cast<int>(w[4]), static_cast<int>(x1.x), s1);
    s0 = __dp4a(static_cast<int>(w[1]), static_cast<int>(x0.y), s0);
    s1 = __dp4a(static_cast<int>(w[5]), static_cast<int>(x1.y), s1);
    s0 = __dp4a(static_cast<int>(w[2]), static_cast<int>(x0.z), s0);
    s1 = __dp4a(static_cast<int>(w[6]), static_cast<int>(x1.z), s1);
    s0 = __dp4a(static_cast<int>(w[3]), static_cast<int>(x0.w), s0);
    s1 = __dp4a(static_cast<int>(w[7]), static_cast<int>(x1.w), s1);
    return s0 + s1;
}

__device__ __forceinline__ float half_bits(uint32_t h) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
}

__device__ __forceinline__ float accumulate(float acc, int isum, uint32_t wd_bits, uint32_t xd_bits) {
    return fmaf(half_bits(wd_bits) * half_bits(xd_bits), static_cast<float>(isum), acc);
}

// The lane order of the row reduction: a xor-butterfly over the 32 lanes.
__device__ __forceinline__ float warp_sum(float s) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(WSW_FULL_MASK, s, off);
    return s;
}

}  // namespace q8d
}  // namespace wsw
