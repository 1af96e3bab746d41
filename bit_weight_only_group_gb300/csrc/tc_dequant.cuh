// Dequantization helpers shared by the tensor-core kernels: packed codes to
// the fp16 operand they stage in shared memory, and the per-row power-of-two
// exponent that keeps that operand finite.
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

// Named barrier over the 512 threads of the dequantization warps (warps
// 0 .. 15) of the tensor-core kernels; the producer and MMA warps do not take
// part.
__device__ __forceinline__ void deq_sync() { asm volatile("bar.sync 1, 512;" ::: "memory"); }

// Position of code c (0..31) of a thread's 32-code chunk in the fp16 operand
// the tensor-core kernels write: pair plan entry e puts its codes lo and hi at
// positions 2e and 2e + 1 (the x operand is permuted the same way).
template <int BITS>
__device__ __forceinline__ int chunk_pos(int c)
{
    int p = 0;
#pragma unroll
    for (int e = 0; e < 16; e++) {
        constexpr int NC = 32;
        const gemv::PairE q = gemv::plan_entry(BITS, NC, e);
        p = q.lo == c ? 2 * e : q.hi == c ? 2 * e + 1 : p;
    }
    return p;
}

// Exponent e >= 0 of one weight row such that every operand value of the
// row, (q - zp) * scale * 2^-e, stays inside fp16's finite range: |q - zp|
// is at most 2^bits - 1, so the bound is the row's largest scale times that.
// (A 4-bit group over [0, 65504] has scale 4368, and 15 * 4368 = 65520
// rounds to infinity in fp16.)  The operand is built with the scale times
// 2^-e (exact) and the row's accumulator is multiplied by 2^e (exact) when
// it is stored.  The two threads of a row (lanes 2i and 2i + 1 of a warp
// whose lanes all call this) each scan half of the row's groups.
template <int BITS>
__device__ __forceinline__ int row_exponent_of_max(uint32_t m)
{
    m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
    float b = __half2float(__ushort_as_half((uint16_t)m)) * (float)((1 << BITS) - 1);
    int e = 0;
    while (b > 65504.0f && e < 30) {
        b *= 0.5f;
        ++e;
    }
    return e;
}

template <int BITS>
__device__ __forceinline__ int row_exponent(const uint16_t* srow, int ng, int hk)
{
    uint32_t m = 0;
    if (ng % 8 == 0 && (reinterpret_cast<uintptr_t>(srow) & 15u) == 0) {
        for (int c = hk; c < ng / 8; c += 2) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(srow) + c);
            m = __vmaxu2(m, v.x & 0x7FFF7FFFu);
            m = __vmaxu2(m, v.y & 0x7FFF7FFFu);
            m = __vmaxu2(m, v.z & 0x7FFF7FFFu);
            m = __vmaxu2(m, v.w & 0x7FFF7FFFu);
        }
    } else {
        for (int g = hk; g < ng; g += 2) m = max(m, (uint32_t)(__ldg(srow + g) & 0x7FFFu));
    }
    m = max(m & 0xFFFFu, m >> 16);
    return row_exponent_of_max<BITS>(m);
}

// The same for a row with 8-bit scales: the largest stored scale is the
// largest normal code's (the fp16 value grows with the code) or one of the
// row's fallback scales.
template <int BITS>
__device__ __forceinline__ int row_exponent_8(const ScaleSrc& sc, int E, int n, int ng, int hk)
{
    const uint8_t* crow = sc.scale8 + (size_t)n * ng;
    uint32_t c = 0;
    for (int g = hk; g < ng; g += 2) {
        const uint32_t v = __ldg(crow + g);
        if (v != kScale8Fallback) c = max(c, v);
    }
    uint32_t m = c ? e4m3_scale_bits(c, E) : 0u;
    const int p1 = min(__ldg(sc.fb_row_ptr + n + 1), sc.fb_cap);
    for (int p = min(__ldg(sc.fb_row_ptr + n), sc.fb_cap) + hk; p < p1; p += 2) m = max(m, (uint32_t)__ldg(sc.fb_val + p));
    return row_exponent_of_max<BITS>(m);
}

// fp16 value h times 2^-e (exact while the result stays a normal number).
__device__ __forceinline__ uint32_t f16_times_pow2(uint32_t h, int e)
{
    if (!e) return h & 0xFFFFu;
    const float v = __half2float(__ushort_as_half((uint16_t)h)) * __int_as_float((127 - e) << 23);
    return __half_as_ushort(__float2half_rn(v));
}

// fp16 value of a + b, with a result beyond fp16's range held at +-65504
// (the 2-bit operand at an outlier: codebook entry plus stored residual,
// whose exact sum is the weight, at most half an fp16 step past 65504).
__device__ __forceinline__ uint16_t f16_add_sat(uint16_t a, uint16_t b, int e)
{
    float v = (__half2float(__ushort_as_half(a)) + __half2float(__ushort_as_half(b))) * __int_as_float((127 - e) << 23);
    v = fminf(fmaxf(v, -65504.0f), 65504.0f);
    return __half_as_ushort(__float2half_rn(v));
}

// 2-bit codebook lookup of the operand pair of plan entry 2s + H (H = 0: the
// codes in bytes 0 and 1 of f, H = 1: bytes 2 and 3), f = four 2-bit codes,
// one per byte; L / H hold the low / high bytes of the group's 4 entries.
template <int HALF>
__device__ __forceinline__ uint32_t cb_pair(uint32_t f, uint32_t lo, uint32_t hi)
{
    const uint32_t sel = HALF ? __umulhi(f, 0x00110000u) + 0x4040u : f * 0x11u + 0x4040u;
    return __byte_perm(lo, hi, sel);
}

}  // namespace tc
}  // namespace qg
