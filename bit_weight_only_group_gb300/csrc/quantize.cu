// Quantize-and-pack of a weight matrix on the GPU (offline step of the
// method).  Bit-exact and deterministic: every floating-point step is an
// explicit IEEE round-to-nearest-even intrinsic (this file is also built with
// -fmad=false), evaluated in the same order as the method's definition.
//
// Method ("70B on one GPU" page, section 2, "group-wise outlier-aware
// quantization"): the largest-magnitude fraction of weights is kept apart in
// FP16; each group of consecutive weights gets its own scale/zero-point from
// the min/max of its remaining weights ("Inference acceleration guide" page, section 1.1
// formula); 2-bit groups use a 4-entry k-means codebook ("Mixed-width quantization" page,
// sections 2.1 and 4.1); codes are packed LSB-first ("Mixed-width quantization" page, section 3).
//
// Launch sequence (all on the caller's stream, no host sync):
//   1. k_hist        per-block shared-memory histogram of the 15-bit |w|
//                    keys, merged into a global histogram;
//   2. k_threshold   one block finds the threshold key T: every key > T is
//                    an outlier, and the first r keys == T in linear order;
//   3. k_row_counts  one warp per row counts keys > T and keys == T;
//   4. k_row_scan    one block: exclusive scans over rows -> CSR row_ptr and
//                    the number of threshold ties each row takes;
//   5. k_compact     one warp per row writes CSR columns/values in k order;
//   6. k_quant_*     one thread per (row, group): group statistics, scale /
//                    zero-point or codebook, codes, packing.
// With 8-bit (E4M3) scales ("Mixed-width quantization" page, section 2.3),
// step 6 is bracketed by:
//   k_fp8_hist       one thread per group: its fp16 scale, a histogram of
//                    floor(log2 scale) over the matrix;
//   k_fp8_exp        one thread: E = the histogram's lower median;
//   k_quant_affine   stores the E4M3 code (or the fallback mark) and codes
//                    the group with the stored scale;
//   k_fb_count       one warp per row counts its fallback groups;
//   k_fb_scan        one block: exclusive scan -> fallback CSR row pointer;
//   k_fb_fill        one warp per row lists its fallback groups and their
//                    fp16 scales.
#include <atomic>
#include <cuda_fp16.h>

#include "qg_internal.h"
#include "scale8.cuh"

namespace qg {
namespace {

constexpr int kBins = 32768;   // |w| as the 15 low bits of an fp16 pattern
constexpr int kLloydIters = 16;

struct SelParams {
    unsigned T;      // threshold key; kBins means "no outliers"
    unsigned c_gt;   // number of keys > T
    unsigned r;      // number of keys == T taken (lowest linear indices)
    unsigned pad;
};

// 8-bit scales: 40 bins of floor(log2 scale) in [-24, 15], then E
constexpr int kF8Bins = 40;
constexpr int kF8Words = 64;

struct QuantWs {
    unsigned* hist;
    SelParams* sel;
    unsigned* cnt_gt;
    unsigned* cnt_eq;
    unsigned* take_eq;
    unsigned* f8;   // [kF8Words]: histogram, then E at kF8Bins
};

size_t ws_layout(int N, QuantWs* p, void* base)
{
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off = align_up(off + bytes, 256);
        return o;
    };
    size_t o_hist = take(sizeof(unsigned) * kBins);
    size_t o_sel = take(sizeof(SelParams));
    size_t o_gt = take(sizeof(unsigned) * (size_t)N);
    size_t o_eq = take(sizeof(unsigned) * (size_t)N);
    size_t o_take = take(sizeof(unsigned) * (size_t)N);
    size_t o_f8 = take(sizeof(unsigned) * kF8Words);
    if (p && base) {
        char* b = static_cast<char*>(base);
        p->hist = reinterpret_cast<unsigned*>(b + o_hist);
        p->sel = reinterpret_cast<SelParams*>(b + o_sel);
        p->cnt_gt = reinterpret_cast<unsigned*>(b + o_gt);
        p->cnt_eq = reinterpret_cast<unsigned*>(b + o_eq);
        p->take_eq = reinterpret_cast<unsigned*>(b + o_take);
        p->f8 = reinterpret_cast<unsigned*>(b + o_f8);
    }
    return off;
}

__device__ __forceinline__ unsigned mag_key(unsigned short h) { return h & 0x7FFFu; }

// ---------------------------------------------------------------- 1. histogram
__global__ void k_hist(const unsigned short* __restrict__ W, long long total,
                       unsigned* __restrict__ hist)
{
    extern __shared__ unsigned sh[];
    for (int i = threadIdx.x; i < kBins; i += blockDim.x) sh[i] = 0;
    __syncthreads();
    const long long nvec = total / 8;
    const uint4* W4 = reinterpret_cast<const uint4*>(W);
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += stride) {
        uint4 v = __ldg(W4 + i);
        unsigned w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; q++) {
            atomicAdd(&sh[w[q] & 0x7FFFu], 1u);
            atomicAdd(&sh[(w[q] >> 16) & 0x7FFFu], 1u);
        }
    }
    for (long long i = nvec * 8 + (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride)
        atomicAdd(&sh[mag_key(W[i])], 1u);
    __syncthreads();
    for (int i = threadIdx.x; i < kBins; i += blockDim.x)
        if (sh[i]) atomicAdd(&hist[i], sh[i]);
}

// Block-wide inclusive scan (blockDim.x == 1024) of unsigned long long values.
__device__ unsigned long long block_incl_scan(unsigned long long v, unsigned long long* tmp32,
                                              unsigned long long* total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        unsigned long long n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    if (lane == 31) tmp32[warp] = v;
    __syncthreads();
    if (warp == 0) {
        unsigned long long s = tmp32[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            unsigned long long n = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += n;
        }
        tmp32[lane] = s;
    }
    __syncthreads();
    if (warp > 0) v += tmp32[warp - 1];
    *total = tmp32[31];
    __syncthreads();
    return v;
}

// ---------------------------------------------------------------- 2. threshold
// Thread i owns bins [32*i, 32*i + 32).  "above" = keys in higher bins.
__global__ void __launch_bounds__(1024) k_threshold(const unsigned* __restrict__ hist, unsigned nnz,
                                                    SelParams* __restrict__ out)
{
    __shared__ unsigned long long tmp[32];
    const int t = threadIdx.x;
    unsigned long long mine = 0;
    for (int b = 0; b < 32; b++) mine += hist[32 * t + b];
    // suffix sum: scan over reversed thread order
    const int rt = 1023 - t;
    unsigned long long tot;
    __shared__ unsigned long long val_by_rt[1024];
    val_by_rt[rt] = mine;
    __syncthreads();
    unsigned long long incl = block_incl_scan(val_by_rt[t], tmp, &tot);
    // incl for reversed index t == sum of bins owned by threads 1023-t .. 1023
    __shared__ unsigned long long incl_by_rt[1024];
    incl_by_rt[t] = incl;
    __syncthreads();
    const unsigned long long above = incl_by_rt[rt] - mine;   // bins above thread t's range
    if (nnz == 0) {
        if (t == 0) *out = SelParams{(unsigned)kBins, 0u, 0u, 0u};
        return;
    }
    if (above < nnz && above + mine >= nnz) {
        unsigned long long cum = above;
        for (int b = 32 * t + 31; b >= 32 * t; b--) {
            unsigned h = hist[b];
            if (cum + h >= nnz) {
                *out = SelParams{(unsigned)b, (unsigned)cum, (unsigned)(nnz - cum), 0u};
                break;
            }
            cum += h;
        }
    }
}

// ---------------------------------------------------------------- 3. per-row counts
__global__ void k_row_counts(const unsigned short* __restrict__ W, int N, int K,
                             const SelParams* __restrict__ sel, unsigned* __restrict__ cnt_gt,
                             unsigned* __restrict__ cnt_eq)
{
    const int lane = threadIdx.x & 31;
    const int n = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (n >= N) return;
    const unsigned T = sel->T;
    unsigned gt = 0, eq = 0;
    const uint4* row = reinterpret_cast<const uint4*>(W + (size_t)n * K);
    for (int i = lane; i < K / 8; i += 32) {
        uint4 v = __ldg(row + i);
        unsigned w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; q++) {
            unsigned a = w[q] & 0x7FFFu, b = (w[q] >> 16) & 0x7FFFu;
            gt += (a > T) + (b > T);
            eq += (a == T) + (b == T);
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        gt += __shfl_xor_sync(0xffffffffu, gt, o);
        eq += __shfl_xor_sync(0xffffffffu, eq, o);
    }
    if (lane == 0) {
        cnt_gt[n] = gt;
        cnt_eq[n] = eq;
    }
}

// ---------------------------------------------------------------- 4. row scans
__global__ void __launch_bounds__(1024) k_row_scan(int N, const SelParams* __restrict__ sel,
                                                   const unsigned* __restrict__ cnt_gt,
                                                   const unsigned* __restrict__ cnt_eq,
                                                   unsigned* __restrict__ take_eq,
                                                   int* __restrict__ row_ptr)
{
    __shared__ unsigned long long tmp[32];
    const long long r = sel->r;
    unsigned long long carry_eq = 0, carry_nz = 0;
    for (int base = 0; base < N; base += 1024) {
        const int n = base + threadIdx.x;
        const unsigned eq = n < N ? cnt_eq[n] : 0u;
        const unsigned gt = n < N ? cnt_gt[n] : 0u;
        unsigned long long tot_eq, tot_nz;
        const unsigned long long eq_before = block_incl_scan(eq, tmp, &tot_eq) - eq + carry_eq;
        long long tk = r - (long long)eq_before;
        if (tk < 0) tk = 0;
        if (tk > (long long)eq) tk = eq;
        const unsigned nz = gt + (unsigned)tk;
        const unsigned long long nz_before = block_incl_scan(nz, tmp, &tot_nz) - nz + carry_nz;
        if (n < N) {
            row_ptr[n] = (int)nz_before;
            take_eq[n] = (unsigned)tk;
        }
        carry_eq += tot_eq;
        carry_nz += tot_nz;
    }
    if (threadIdx.x == 0) row_ptr[N] = (int)carry_nz;
}

// ---------------------------------------------------------------- 5. compaction
__global__ void k_compact(const unsigned short* __restrict__ W, int N, int K,
                          const SelParams* __restrict__ sel, const unsigned* __restrict__ take_eq,
                          const int* __restrict__ row_ptr, int* __restrict__ col,
                          unsigned short* __restrict__ val)
{
    const int lane = threadIdx.x & 31;
    const int n = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (n >= N) return;
    int p = row_ptr[n];
    if (row_ptr[n + 1] == p) return;
    const unsigned T = sel->T, take = take_eq[n];
    const unsigned lt_mask = (1u << lane) - 1u;
    unsigned ties = 0;
    const unsigned short* row = W + (size_t)n * K;
    for (int k0 = 0; k0 < K; k0 += 32) {
        const unsigned short h = row[k0 + lane];
        const unsigned key = mag_key(h);
        const bool is_eq = key == T;
        const unsigned eq_mask = __ballot_sync(0xffffffffu, is_eq);
        const unsigned rank = ties + __popc(eq_mask & lt_mask);
        const bool is_out = key > T || (is_eq && rank < take);
        const unsigned out_mask = __ballot_sync(0xffffffffu, is_out);
        if (is_out) {
            const int pos = p + __popc(out_mask & lt_mask);
            col[pos] = k0 + lane;
            val[pos] = h;
        }
        p += __popc(out_mask);
        ties += __popc(eq_mask);
    }
}

// ---------------------------------------------------------------- 6. groups
// Outlier mask of one group from the row's CSR (columns ascending).
template <int G>
__device__ __forceinline__ int group_outliers(const int* __restrict__ row_ptr,
                                              const int* __restrict__ col, int n, int k0,
                                              unsigned (&om)[G / 32], int* first)
{
#pragma unroll
    for (int i = 0; i < G / 32; i++) om[i] = 0u;
    *first = 0;
    if (!row_ptr) return 0;
    int lo = row_ptr[n], hi = row_ptr[n + 1];
    while (lo < hi) {   // first entry with col >= k0
        int mid = (lo + hi) >> 1;
        if (col[mid] < k0) lo = mid + 1;
        else hi = mid;
    }
    *first = lo;
    int cnt = 0;
    const int end = row_ptr[n + 1];
    for (int p = lo; p < end; p++) {
        const int c = col[p] - k0;
        if (c >= G) break;
        om[c >> 5] |= 1u << (c & 31);
        cnt++;
    }
    return cnt;
}

__device__ __forceinline__ float h2f(unsigned short h) { return __half2float(__ushort_as_half(h)); }

// Calls f(i, fp16 bits) for the G values of a group, in ascending k, with
// 16-byte loads (the group is re-read from L1 on later passes).
template <int G, typename F>
__device__ __forceinline__ void for_group(const unsigned short* __restrict__ src, F&& f)
{
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    for (int c = 0; c < G / 8; c++) {
        const uint4 q = __ldg(s4 + c);
        const unsigned w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int j = 0; j < 4; j++) {
            f(8 * c + 2 * j, (unsigned short)(w[j] & 0xFFFFu));
            f(8 * c + 2 * j + 1, (unsigned short)(w[j] >> 16));
        }
    }
}

// LSB-first packer writing whole 32-bit words.
struct BitWriter {
    unsigned* dst;
    unsigned long long acc;
    int nb;
    __device__ void put(unsigned code, int bits)
    {
        acc |= (unsigned long long)code << nb;
        nb += bits;
        if (nb >= 32) {
            *dst++ = (unsigned)acc;
            acc >>= 32;
            nb -= 32;
        }
    }
};

template <int G>
__device__ __forceinline__ bool is_out(const unsigned (&om)[G / 32], int i)
{
    return (om[i >> 5] >> (i & 31)) & 1u;
}

// Affine parameters of a group (range widened to contain 0): fp16 scale
// rounded up from (max - min) / qmax (1.0 when max == min), zero point
// clamp(-round(min / scale), 0, qmax).
template <int G>
__device__ __forceinline__ void affine_params(const unsigned short* __restrict__ src, const unsigned (&om)[G / 32],
                                              int qmax, unsigned short* s16_out, int* zp_out, float* mn_out = nullptr)
{
    float mn = 0.0f, mx = 0.0f;
    for_group<G>(src, [&](int i, unsigned short h) {
        if (is_out<G>(om, i)) return;
        const float f = h2f(h);
        if (f < mn) mn = f;
        if (f > mx) mx = f;
    });
    unsigned short s16;
    if (mx == mn) {
        s16 = 0x3C00;
    } else {
        const float range = __fsub_rn(mx, mn);
        const float s32 = __fdiv_rn(range, (float)qmax);
        s16 = __half_as_ushort(__float2half_ru(s32));
    }
    const float r = rintf(__fdiv_rn(mn, h2f(s16)));
    int zp = -(int)r;
    *zp_out = zp < 0 ? 0 : (zp > qmax ? qmax : zp);
    *s16_out = s16;
    if (mn_out) *mn_out = mn;
}

// fp16 scale of an affine (sym == 0) or symmetric (sym == 1) group, as the
// quantizer below finds it.
template <int G>
__device__ __forceinline__ unsigned short group_scale16(const unsigned short* __restrict__ src,
                                                        const unsigned (&om)[G / 32], int bits, int sym);

// floor(log2 h) of a positive finite fp16 number h.
__device__ __forceinline__ int f16_floor_log2(unsigned h)
{
    const int e5 = (h >> 10) & 31;
    if (e5) return e5 - 15;
    return (31 - __clz(h & 1023u)) - 24;
}

// E4M3 storage of the fp16 scale s16 under the matrix exponent E: the least
// normal E4M3 value >= s16 * 2^-E (code returned, *eff = fp16 bits of that
// value times 2^E), or kScale8Fallback with *eff = s16 when s16 * 2^-E is
// below 2^-6, the rounded value above 448, or value * 2^E off fp16's normal
// range.  Integer arithmetic on the fp16 fields: s16 = (mant / 1024) *
// 2^lg with mant in [1024, 2048), rounded up to 3 fraction bits.
__device__ __forceinline__ unsigned e4m3_store(unsigned s16, int E, unsigned* eff)
{
    const int e5 = (s16 >> 10) & 31;
    const unsigned m10 = s16 & 1023u;
    int lg;
    unsigned mant;
    if (e5) {
        lg = e5 - 15;
        mant = 1024u + m10;
    } else {
        const int hb = 31 - __clz(m10);
        lg = hb - 24;
        mant = m10 << (10 - hb);
    }
    int ex = lg - E;
    *eff = s16;
    if (ex < -6) return kScale8Fallback;
    unsigned m3 = (mant - 1024u + 127u) >> 7;   // ceil of the fraction in eighths
    if (m3 == 8u) {
        m3 = 0u;
        ++ex;
    }
    if (ex > 8 || (ex == 8 && m3 == 7u)) return kScale8Fallback;
    const int fe = ex + E;
    if (fe < -14 || fe > 15) return kScale8Fallback;
    *eff = ((unsigned)(fe + 15) << 10) | (m3 << 7);
    return ((unsigned)(ex + 7) << 3) | m3;
}

// Largest |w| over the group's non-outliers.
template <int G>
__device__ __forceinline__ float group_amax(const unsigned short* __restrict__ src, const unsigned (&om)[G / 32])
{
    float amax = 0.0f;
    for_group<G>(src, [&](int i, unsigned short h) {
        if (!is_out<G>(om, i)) amax = fmaxf(amax, fabsf(h2f(h)));
    });
    return amax;
}

// Widths 3..6.  sym == 0: asymmetric (scale and zero point from the group's
// range); sym == 1: symmetric, integer range [-qs, qs] with qs = 2^(b-1) - 1,
// scale rounded up from amax / qs (1.0 if amax is 0), codes q + 2^(b-1) with
// the zero point fixed at 2^(b-1).  Outliers take the zero point's code.
// With scale8 set, the group's scale is stored as 8 bits (e4m3_store under
// the exponent *f8_exp) and the codes use the stored scale.
template <int G>
__global__ void k_quant_affine(const unsigned short* __restrict__ W, int N, int K, int bits, int sym,
                               const int* __restrict__ row_ptr, const int* __restrict__ col,
                               unsigned char* __restrict__ packed, unsigned short* __restrict__ scale,
                               unsigned char* __restrict__ zp_out, const unsigned* __restrict__ f8_exp,
                               unsigned char* __restrict__ scale8)
{
    const int ng = K / G;
    const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (gid >= (long long)N * ng) return;
    const int n = (int)(gid / ng), j = (int)(gid % ng);
    const int k0 = j * G;
    unsigned om[G / 32];
    int first;
    group_outliers<G>(row_ptr, col, n, k0, om, &first);
    const unsigned short* src = W + (size_t)n * K + k0;
    const int qmax = (1 << bits) - 1;
    unsigned short s16;
    int zp, qlo, qhi;
    if (sym) {
        const int qs = (1 << (bits - 1)) - 1;
        const float amax = group_amax<G>(src, om);
        s16 = amax == 0.0f ? (unsigned short)0x3C00 : __half_as_ushort(__float2half_ru(__fdiv_rn(amax, (float)qs)));
        zp = 1 << (bits - 1);
        qlo = zp - qs;
        qhi = zp + qs;
    } else {
        float mn;
        affine_params<G>(src, om, qmax, &s16, &zp, &mn);
        qlo = 0;
        qhi = qmax;
        if (scale8) {   // zero point of the stored scale
            unsigned eff;
            e4m3_store(s16, (int)__ldg(f8_exp), &eff);
            const float r = rintf(__fdiv_rn(mn, h2f((unsigned short)eff)));
            zp = -(int)r;
            zp = zp < 0 ? 0 : (zp > qmax ? qmax : zp);
        }
    }
    if (scale8) {
        unsigned eff;
        scale8[gid] = (unsigned char)e4m3_store(s16, (int)__ldg(f8_exp), &eff);
        s16 = (unsigned short)eff;
    }
    const float s = h2f(s16);
    BitWriter bw{reinterpret_cast<unsigned*>(packed + ((size_t)n * K + k0) * bits / 8), 0ull, 0};
    for_group<G>(src, [&](int i, unsigned short h) {
        int q;
        if (is_out<G>(om, i)) {
            q = zp;
        } else {
            q = (int)rintf(__fdiv_rn(h2f(h), s)) + zp;
            q = q < qlo ? qlo : (q > qhi ? qhi : q);
        }
        bw.put((unsigned)q, bits);
    });
    if (!scale8) scale[gid] = s16;
    zp_out[gid] = (unsigned char)zp;
}

template <int G>
__device__ __forceinline__ unsigned short group_scale16(const unsigned short* __restrict__ src,
                                                        const unsigned (&om)[G / 32], int bits, int sym)
{
    if (sym) {
        const int qs = (1 << (bits - 1)) - 1;
        const float amax = group_amax<G>(src, om);
        return amax == 0.0f ? (unsigned short)0x3C00 : __half_as_ushort(__float2half_ru(__fdiv_rn(amax, (float)qs)));
    }
    unsigned short s16;
    int zp;
    affine_params<G>(src, om, (1 << bits) - 1, &s16, &zp);
    return s16;
}

// ---------------------------------------------------------------- 8-bit scales
// Histogram of floor(log2 s16) over every group's fp16 scale (bins -24..15).
template <int G>
__global__ void k_fp8_hist(const unsigned short* __restrict__ W, int N, int K, int bits, int sym,
                           const int* __restrict__ row_ptr, const int* __restrict__ col, unsigned* __restrict__ hist)
{
    __shared__ unsigned sh[kF8Bins];
    for (int i = threadIdx.x; i < kF8Bins; i += blockDim.x) sh[i] = 0u;
    __syncthreads();
    const int ng = K / G;
    const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (gid < (long long)N * ng) {
        const int n = (int)(gid / ng), j = (int)(gid % ng);
        unsigned om[G / 32];
        int first;
        group_outliers<G>(row_ptr, col, n, j * G, om, &first);
        const unsigned short s16 = group_scale16<G>(W + (size_t)n * K + j * G, om, bits, sym);
        atomicAdd(&sh[f16_floor_log2(s16) + 24], 1u);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kF8Bins; i += blockDim.x)
        if (sh[i]) atomicAdd(&hist[i], sh[i]);
}

// E = the lower median (element (count - 1) / 2 in ascending order).
__global__ void k_fp8_exp(unsigned* __restrict__ f8, unsigned long long count, int* __restrict__ exp_out)
{
    const unsigned long long want = (count - 1) / 2;
    unsigned long long seen = 0;
    int E = 0;
    for (int b = 0; b < kF8Bins; b++) {
        seen += f8[b];
        if (seen > want) {
            E = b - 24;
            break;
        }
    }
    f8[kF8Bins] = (unsigned)E;
    *exp_out = E;
}

// Number of fallback groups of every row (one warp per row).
__global__ void k_fb_count(const unsigned char* __restrict__ scale8, int N, int ng, unsigned* __restrict__ cnt)
{
    const int warp = (int)((blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5), lane = threadIdx.x & 31;
    if (warp >= N) return;
    const unsigned char* r = scale8 + (size_t)warp * ng;
    unsigned c = 0;
    for (int j = lane; j < ng; j += 32) c += r[j] == kScale8Fallback;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    if (lane == 0) cnt[warp] = c;
}

// Exclusive scan of the row counts into the fallback CSR row pointer (one
// block); more groups than the list holds sets the status word.
__global__ void __launch_bounds__(1024) k_fb_scan(const unsigned* __restrict__ cnt, int N, int* __restrict__ fb_row_ptr,
                                                  int cap, int* status)
{
    __shared__ unsigned long long part[1024];
    const int t = threadIdx.x;
    const long long per = (N + 1023) / 1024;
    const long long b0 = (long long)t * per, b1 = min((long long)N, b0 + per);
    unsigned long long sum = 0;
    for (long long i = b0; i < b1; i++) sum += cnt[i];
    part[t] = sum;
    __syncthreads();
    for (int o = 1; o < 1024; o <<= 1) {   // inclusive scan of the per-thread sums
        const unsigned long long v = t >= o ? part[t - o] : 0ull;
        __syncthreads();
        part[t] += v;
        __syncthreads();
    }
    unsigned long long run = part[t] - sum;
    for (long long i = b0; i < b1; i++) {
        fb_row_ptr[i] = (int)run;
        run += cnt[i];
    }
    if (t == 1023) {
        fb_row_ptr[N] = (int)part[1023];
        if (part[1023] > (unsigned long long)cap && status) atomicExch(status, (int)QG_ERR_WORKSPACE);
    }
}

// The fallback list of every row (one warp per row): group index and fp16
// scale of each group stored as kScale8Fallback, in ascending order; entries
// beyond the capacity are not written.
template <int G>
__global__ void k_fb_fill(const unsigned short* __restrict__ W, int N, int K, int bits, int sym,
                          const int* __restrict__ row_ptr, const int* __restrict__ col,
                          const unsigned char* __restrict__ scale8, const int* __restrict__ fb_row_ptr,
                          int* __restrict__ fb_col, unsigned short* __restrict__ fb_val, int cap)
{
    const int warp = (int)((blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5), lane = threadIdx.x & 31;
    if (warp >= N) return;
    const int n = warp, ng = K / G;
    int base = fb_row_ptr[n];
    for (int j0 = 0; j0 < ng; j0 += 32) {
        const int j = j0 + lane;
        const bool fb = j < ng && scale8[(size_t)n * ng + j] == kScale8Fallback;
        const unsigned m = __ballot_sync(0xffffffffu, fb);
        if (fb) {
            const int at = base + __popc(m & ((1u << lane) - 1u));
            if (at < cap) {
                unsigned om[G / 32];
                int first;
                group_outliers<G>(row_ptr, col, n, j * G, om, &first);
                fb_col[at] = j;
                fb_val[at] = group_scale16<G>(W + (size_t)n * K + j * G, om, bits, sym);
            }
        }
        base += __popc(m);
    }
}

// 2-bit groups on a uniform grid, stored as the four constants a code
// selects.  mode 1 (symmetric): levels -s, 0, s with s = amax rounded up to
// fp16 (1.0 if 0), codes round(w / s) clamped to [-1, 1], plus 1; constants
// (-s, 0, s, s).  mode 2 (linear): the affine grid at 2 bits, constants
// fp16((i - zp) * scale).  The zero code's constant is exactly 0: outliers
// take it and keep their own value as the stored residual.
template <int G>
__global__ void k_quant_uniform2(const unsigned short* __restrict__ W, int N, int K, int mode,
                                 const int* __restrict__ row_ptr, const int* __restrict__ col,
                                 unsigned char* __restrict__ packed, unsigned short* __restrict__ cb,
                                 unsigned short* __restrict__ val)
{
    const int ng = K / G;
    const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (gid >= (long long)N * ng) return;
    const int n = (int)(gid / ng), j = (int)(gid % ng);
    const int k0 = j * G;
    unsigned om[G / 32];
    int first;
    group_outliers<G>(row_ptr, col, n, k0, om, &first);
    const unsigned short* src = W + (size_t)n * K + k0;
    unsigned short s16;
    int zp, qlo, qhi;
    unsigned short e[4];
    if (mode == 1) {
        const float amax = group_amax<G>(src, om);
        s16 = amax == 0.0f ? (unsigned short)0x3C00 : __half_as_ushort(__float2half_ru(amax));
        zp = 1;
        qlo = 0;
        qhi = 2;
        e[0] = (unsigned short)(s16 | 0x8000u);
        e[1] = 0;
        e[2] = s16;
        e[3] = s16;
    } else {
        affine_params<G>(src, om, 3, &s16, &zp);
        qlo = 0;
        qhi = 3;
        const float sf = h2f(s16);
#pragma unroll
        for (int i = 0; i < 4; i++) e[i] = __half_as_ushort(__float2half_rn(__fmul_rn((float)(i - zp), sf)));
    }
    const float s = h2f(s16);
    BitWriter bw{reinterpret_cast<unsigned*>(packed + ((size_t)n * K + k0) * 2 / 8), 0ull, 0};
    int p = first;
    for_group<G>(src, [&](int i, unsigned short h) {
        int q;
        if (is_out<G>(om, i)) {
            q = zp;
            val[p++] = h;
        } else {
            q = (int)rintf(__fdiv_rn(h2f(h), s)) + zp;
            q = q < qlo ? qlo : (q > qhi ? qhi : q);
        }
        bw.put((unsigned)q, 2);
    });
    uint2 packed_cb;
    packed_cb.x = (unsigned)e[0] | ((unsigned)e[1] << 16);
    packed_cb.y = (unsigned)e[2] | ((unsigned)e[3] << 16);
    reinterpret_cast<uint2*>(cb)[gid] = packed_cb;
}

__device__ __forceinline__ int nearest4(float v, float c0, float c1, float c2, float c3)
{
    int best = 0;
    float bd = fabsf(__fsub_rn(v, c0));
    float d = fabsf(__fsub_rn(v, c1));
    if (d < bd) { bd = d; best = 1; }
    d = fabsf(__fsub_rn(v, c2));
    if (d < bd) { bd = d; best = 2; }
    d = fabsf(__fsub_rn(v, c3));
    if (d < bd) { bd = d; best = 3; }
    return best;
}

template <int G>
__global__ void k_quant_codebook(const unsigned short* __restrict__ W, int N, int K,
                                 const int* __restrict__ row_ptr, const int* __restrict__ col,
                                 unsigned char* __restrict__ packed, unsigned short* __restrict__ cb,
                                 unsigned short* __restrict__ val)
{
    const int ng = K / G;
    const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (gid >= (long long)N * ng) return;
    const int n = (int)(gid / ng), j = (int)(gid % ng);
    const int k0 = j * G;
    unsigned om[G / 32];
    int first;
    group_outliers<G>(row_ptr, col, n, k0, om, &first);
    const unsigned short* src = W + (size_t)n * K + k0;

    // the group stays in L1; it is re-read on every pass
    float mn = 0.0f, mx = 0.0f;
    for (int i = 0; i < G; i++) {
        if (is_out<G>(om, i)) continue;
        const float f = h2f(__ldg(src + i));
        if (f < mn) mn = f;
        if (f > mx) mx = f;
    }
    const float step = __fdiv_rn(__fsub_rn(mx, mn), 3.0f);
    float c0 = __fadd_rn(mn, __fmul_rn(0.0f, step));
    float c1 = __fadd_rn(mn, __fmul_rn(1.0f, step));
    float c2 = __fadd_rn(mn, __fmul_rn(2.0f, step));
    float c3 = __fadd_rn(mn, __fmul_rn(3.0f, step));
    for (int it = 0; it < kLloydIters; it++) {
        float s0 = 0.0f, s1 = 0.0f, s2 = 0.0f, s3 = 0.0f;
        int n0 = 0, n1 = 0, n2 = 0, n3 = 0;
        for (int i = 0; i < G; i++) {   // ascending k
            if (is_out<G>(om, i)) continue;
            const float f = h2f(__ldg(src + i));
            switch (nearest4(f, c0, c1, c2, c3)) {
                case 0: s0 = __fadd_rn(s0, f); n0++; break;
                case 1: s1 = __fadd_rn(s1, f); n1++; break;
                case 2: s2 = __fadd_rn(s2, f); n2++; break;
                default: s3 = __fadd_rn(s3, f); n3++; break;
            }
        }
        if (n0) c0 = __fdiv_rn(s0, (float)n0);
        if (n1) c1 = __fdiv_rn(s1, (float)n1);
        if (n2) c2 = __fdiv_rn(s2, (float)n2);
        if (n3) c3 = __fdiv_rn(s3, (float)n3);
    }
    unsigned short e[4] = {__half_as_ushort(__float2half_rn(c0)), __half_as_ushort(__float2half_rn(c1)),
                           __half_as_ushort(__float2half_rn(c2)), __half_as_ushort(__float2half_rn(c3))};
    // stable insertion sort by value
    for (int i = 1; i < 4; i++) {
        const unsigned short x = e[i];
        const float xv = h2f(x);
        int q = i - 1;
        while (q >= 0 && h2f(e[q]) > xv) {
            e[q + 1] = e[q];
            q--;
        }
        e[q + 1] = x;
    }
    const float f0 = h2f(e[0]), f1 = h2f(e[1]), f2 = h2f(e[2]), f3 = h2f(e[3]);
    const int zc = nearest4(0.0f, f0, f1, f2, f3);
    const float fz = zc == 0 ? f0 : zc == 1 ? f1 : zc == 2 ? f2 : f3;

    BitWriter bw{reinterpret_cast<unsigned*>(packed + ((size_t)n * K + k0) * 2 / 8), 0ull, 0};
    int p = first;
    for (int i = 0; i < G; i++) {
        const float f = h2f(__ldg(src + i));
        int q;
        if (is_out<G>(om, i)) {
            q = zc;
            val[p++] = __half_as_ushort(__float2half_rn(__fsub_rn(f, fz)));
        } else {
            q = nearest4(f, f0, f1, f2, f3);
        }
        bw.put((unsigned)q, 2);
    }
    uint2 packed_cb;
    packed_cb.x = (unsigned)e[0] | ((unsigned)e[1] << 16);
    packed_cb.y = (unsigned)e[2] | ((unsigned)e[3] << 16);
    reinterpret_cast<uint2*>(cb)[gid] = packed_cb;
}

}  // namespace

size_t quantize_workspace_bytes(int N, int /*K*/) { return ws_layout(N, nullptr, nullptr); }

// Launched after the quantizer's kernels: a decode product that reads these
// weights next on the stream may start its weight loads before the kernel
// preceding it has finished (programmatic dependent launch), so that kernel
// must not be one that wrote the weights.
__global__ void k_quant_done() {}

qg_status launch_quantize(const uint16_t* W, float /*frac*/, const qg_qweight& w, void* ws,
                          cudaStream_t s, int mode)
{
    QuantWs p{};
    ws_layout(w.N, &p, ws);
    const long long total = (long long)w.N * w.K;
    const int sms = num_sms();
    cudaError_t e;
    const bool has_out = w.nnz > 0;
    if (has_out) {
        e = cudaMemsetAsync(p.hist, 0, sizeof(unsigned) * kBins, s);
        if (e != cudaSuccess) return cuda_fail(e, "memset histogram");
        static std::atomic<bool> attr_set[64];   // per device (setting it twice is harmless)
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) dev = 0;
        if (dev >= 64 || !attr_set[dev].load(std::memory_order_acquire)) {
            e = cudaFuncSetAttribute(k_hist, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)(sizeof(unsigned) * kBins));
            if (e != cudaSuccess) return cuda_fail(e, "k_hist smem attribute");
            if (dev < 64) attr_set[dev].store(true, std::memory_order_release);
        }
        long long blocks = ceil_div(total / 8 + 1, 1024);
        if (blocks > sms) blocks = sms;
        k_hist<<<(int)blocks, 1024, sizeof(unsigned) * kBins, s>>>(
            reinterpret_cast<const unsigned short*>(W), total, p.hist);
        k_threshold<<<1, 1024, 0, s>>>(p.hist, (unsigned)w.nnz, p.sel);
        const int rows_per_block = 8;
        const int nb = (int)ceil_div(w.N, rows_per_block);
        k_row_counts<<<nb, 32 * rows_per_block, 0, s>>>(reinterpret_cast<const unsigned short*>(W), w.N,
                                                         w.K, p.sel, p.cnt_gt, p.cnt_eq);
        k_row_scan<<<1, 1024, 0, s>>>(w.N, p.sel, p.cnt_gt, p.cnt_eq, p.take_eq, w.out_row_ptr);
        k_compact<<<nb, 32 * rows_per_block, 0, s>>>(reinterpret_cast<const unsigned short*>(W), w.N, w.K,
                                                      p.sel, p.take_eq, w.out_row_ptr, w.out_col,
                                                      w.out_val);
    } else if (w.out_row_ptr) {
        e = cudaMemsetAsync(w.out_row_ptr, 0, sizeof(int) * ((size_t)w.N + 1), s);
        if (e != cudaSuccess) return cuda_fail(e, "memset row_ptr");
    }
    const int* rp = has_out ? w.out_row_ptr : nullptr;
    const long long groups = (long long)w.N * (w.K / w.group);
    const int threads = 128;
    const int blocks = (int)ceil_div(groups, threads);
    const unsigned short* Wh = reinterpret_cast<const unsigned short*>(W);
    if (w.bits == 2 && mode != 0) {
        auto run = [&](auto kern) {
            kern<<<blocks, threads, 0, s>>>(Wh, w.N, w.K, mode, rp, w.out_col, w.packed, w.codebook, w.out_val);
        };
        if (w.group == 32) run(k_quant_uniform2<32>);
        else if (w.group == 64) run(k_quant_uniform2<64>);
        else run(k_quant_uniform2<128>);
    } else if (w.bits == 2) {
        auto run = [&](auto kern) {
            kern<<<blocks, threads, 0, s>>>(Wh, w.N, w.K, rp, w.out_col, w.packed, w.codebook, w.out_val);
        };
        if (w.group == 32) run(k_quant_codebook<32>);
        else if (w.group == 64) run(k_quant_codebook<64>);
        else run(k_quant_codebook<128>);
    } else if (!w.scale8) {
        auto run = [&](auto kern) {
            kern<<<blocks, threads, 0, s>>>(Wh, w.N, w.K, w.bits, mode, rp, w.out_col, w.packed, w.scale, w.zp,
                                            nullptr, nullptr);
        };
        if (w.group == 32) run(k_quant_affine<32>);
        else if (w.group == 64) run(k_quant_affine<64>);
        else run(k_quant_affine<128>);
    } else {
        // 8-bit scales: histogram -> E -> quantize -> fallback list
        e = cudaMemsetAsync(p.f8, 0, sizeof(unsigned) * kF8Words, s);
        if (e != cudaSuccess) return cuda_fail(e, "memset scale histogram");
        auto hist = [&](auto kern) { kern<<<blocks, threads, 0, s>>>(Wh, w.N, w.K, w.bits, mode, rp, w.out_col, p.f8); };
        if (w.group == 32) hist(k_fp8_hist<32>);
        else if (w.group == 64) hist(k_fp8_hist<64>);
        else hist(k_fp8_hist<128>);
        k_fp8_exp<<<1, 1, 0, s>>>(p.f8, (unsigned long long)groups, w.scale8_exp);
        auto run = [&](auto kern) {
            kern<<<blocks, threads, 0, s>>>(Wh, w.N, w.K, w.bits, mode, rp, w.out_col, w.packed, w.scale, w.zp,
                                            p.f8 + kF8Bins, w.scale8);
        };
        if (w.group == 32) run(k_quant_affine<32>);
        else if (w.group == 64) run(k_quant_affine<64>);
        else run(k_quant_affine<128>);
        const int row_blocks = (int)ceil_div(w.N, 8);
        k_fb_count<<<row_blocks, 256, 0, s>>>(w.scale8, w.N, w.K / w.group, p.cnt_gt);
        k_fb_scan<<<1, 1024, 0, s>>>(p.cnt_gt, w.N, w.fb_row_ptr, w.fb_cap, device_status_ptr());
        auto fill = [&](auto kern) {
            kern<<<row_blocks, 256, 0, s>>>(Wh, w.N, w.K, w.bits, mode, rp, w.out_col, w.scale8, w.fb_row_ptr,
                                            w.fb_col, w.fb_val, w.fb_cap);
        };
        if (w.group == 32) fill(k_fb_fill<32>);
        else if (w.group == 64) fill(k_fb_fill<64>);
        else fill(k_fb_fill<128>);
    }
    k_quant_done<<<1, 32, 0, s>>>();
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
    return QG_OK;
}

}  // namespace qg
