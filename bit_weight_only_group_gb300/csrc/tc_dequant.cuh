// Dequantization helpers shared by the tensor-core kernels (4-bit codes to
// the fp16 operand they stage in shared memory).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "gemv_impl.cuh"

namespace qg {
namespace tc {

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// 8 consecutive 4-bit codes (one 32-bit word, code i at bits 4i) -> 4 fp16
// pairs (q - zp) * s in the order (c0, c4, c1, c5, c2, c6, c3, c7): masks
// pick two codes 16 bits apart straight into fp16 1024 + 2^p q (p = 0 or 4),
// one packed FMA makes them the exact integers q - zp and one packed multiply
// applies the scale.  x is staged with its K positions permuted the same way
// inside each block of 8 (the product does not depend on the order of k as
// long as both operands agree).
__device__ __forceinline__ uint4 deq8_u4(uint32_t v, uint32_t add_lo, uint32_t add_hi, uint32_t s2, uint32_t magic)
{
    constexpr uint32_t one = 0x3C003C00u, sixteenth = 0x2C002C00u;   // 1, 1/16
    const uint32_t v8 = v >> 8;
    const uint32_t r0 = gemv::and_or<0x000F000Fu>(v, magic);
    const uint32_t r1 = gemv::and_or<0x00F000F0u>(v, magic);
    const uint32_t r2 = gemv::and_or<0x000F000Fu>(v8, magic);
    const uint32_t r3 = gemv::and_or<0x00F000F0u>(v8, magic);
    return make_uint4(hmul2_u32(gemv::hfma2_u32(r0, one, add_lo), s2), hmul2_u32(gemv::hfma2_u32(r1, sixteenth, add_hi), s2),
                      hmul2_u32(gemv::hfma2_u32(r2, one, add_lo), s2), hmul2_u32(gemv::hfma2_u32(r3, sixteenth, add_hi), s2));
}

// position of k (mod 8) inside a permuted block of 8: inverse of (0,4,1,5,2,6,3,7)
__device__ __forceinline__ int perm8_pos(int k) { return ((k & 3) << 1) | ((k >> 2) & 1); }

}  // namespace tc
}  // namespace qg
