// Group scales stored as 8-bit floats (E4M3) with an fp16 fallback
// ("Mixed-width quantization" page, section 2.3: the scale itself stored in
// 8 bits, the groups whose scale the 8-bit format cannot hold kept at fp16).
//
// A group's stored scale is the E4M3 value of its code times 2^E (E one
// exponent per matrix), always a normal fp16 number, or -- code 0x7F -- the
// fp16 scale kept in the row's fallback list (CSR: fb_row_ptr, fb_col =
// group index, fb_val = fp16 scale).  Every reader turns a group's storage
// into fp16 scale bits, so the products keep working on fp16 scales.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "qgemm.h"

namespace qg {

constexpr uint32_t kScale8Fallback = 0x7Fu;

struct ScaleSrc {
    const uint16_t* scale;    // fp16 [N, ng] (when scale8 is null)
    const uint8_t* scale8;    // E4M3 [N, ng], kScale8Fallback = in the fallback list
    const int* exp;           // the matrix exponent E
    const int* fb_row_ptr;    // [N + 1]
    const int* fb_col;        // [fb_cap] group index, ascending within a row
    const uint16_t* fb_val;   // [fb_cap] fp16 scale
    int fb_cap;
};

inline ScaleSrc scale_src(const qg_qweight& w)
{
    return ScaleSrc{w.scale, w.scale8, w.scale8_exp, w.fb_row_ptr, w.fb_col, w.fb_val, w.fb_cap};
}

// fp16 bits of (E4M3 value of the positive normal code c) * 2^E: exponent
// field (c >> 3) - 7 + E + 15, fraction the code's 3 bits on top.
__device__ __forceinline__ uint32_t e4m3_scale_bits(uint32_t c, int E)
{
    return ((uint32_t)((int)((c >> 3) & 15u) + 8 + E) << 10) | ((c & 7u) << 7);
}

// fp16 scale bits of fallback group j of row n (0 if the list lacks it: a
// list that overflowed its capacity is searched only within the capacity).
// Not inlined: the path is rare, and its loop would weigh on the registers
// of the loops that convert scales as they use them.
static __device__ __noinline__ uint32_t fallback_scale_bits(const ScaleSrc& s, int n, int j)
{
    int lo = min(__ldg(s.fb_row_ptr + n), s.fb_cap);
    const int end = min(__ldg(s.fb_row_ptr + n + 1), s.fb_cap);
    int hi = end;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(s.fb_col + mid) < j) lo = mid + 1;
        else hi = mid;
    }
    return (lo < end && __ldg(s.fb_col + lo) == j) ? (uint32_t)__ldg(s.fb_val + lo) : 0u;
}

__device__ __forceinline__ int scale_exp(const ScaleSrc& s) { return s.scale8 ? __ldg(s.exp) : 0; }

// fp16 scale bits of a group whose 8-bit code c was already loaded.
__device__ __forceinline__ uint32_t scale8_bits(const ScaleSrc& s, int E, int n, int j, uint32_t c)
{
    return c == kScale8Fallback ? fallback_scale_bits(s, n, j) : e4m3_scale_bits(c, E);
}

// fp16 scale bits of group j of row n, from either storage.
__device__ __forceinline__ uint32_t scale_bits(const ScaleSrc& s, int E, int n, int ng, int j)
{
    if (!s.scale8) return __ldg(s.scale + (size_t)n * ng + j);
    return scale8_bits(s, E, n, j, __ldg(s.scale8 + (size_t)n * ng + j));
}

}  // namespace qg
