// Per-layer quantization diagnostics on the device ("Mixed-width quantization"
// page, section 6.1: unpack the quantized layer and compare it element by
// element with the original fp16 weights -- maximum absolute error, root mean
// square error, cosine similarity; section 6.2: the dynamic-range ratio of
// each block, its largest magnitude over its second largest).
//
// One thread per group (the group's W values, codes, parameters and FP16
// outliers), fp32 sums inside a group, fp64 across groups: k_diag writes one
// partial per CTA, k_diag_final reduces them in a fixed order (the result is
// deterministic) into the caller's qg_diag.  Memory-bound: it reads W (2
// bytes per weight) and the quantized layer once.
#include <cuda_fp16.h>

#include <cmath>

#include "qg_internal.h"
#include "scale8.cuh"

namespace qg {
namespace diag {

constexpr int kThreads = 128;

struct Partial {
    double se, sww, svv, swv, emax, rmax, over;
};

__device__ __forceinline__ float h2f(uint32_t h) { return __half2float(__ushort_as_half((uint16_t)h)); }

template <int BITS, int G>
__global__ void __launch_bounds__(kThreads) k_diag(const uint16_t* __restrict__ W, int N, int K,
                                                    const uint8_t* __restrict__ packed,
                                                    const ScaleSrc sc, const uint8_t* __restrict__ zp,
                                                    const uint2* __restrict__ cb, const int* __restrict__ row_ptr,
                                                    const int* __restrict__ col, const uint16_t* __restrict__ val,
                                                    int nnz, float threshold, float* __restrict__ ratio,
                                                    Partial* __restrict__ part)
{
    constexpr int NW = G * BITS / 32;   // 32-bit words of codes per group
    const int ng = K / G;
    const long long gid = (long long)blockIdx.x * kThreads + threadIdx.x;
    double se = 0.0, sww = 0.0, svv = 0.0, swv = 0.0;
    float emax = 0.0f, rmax = 0.0f, over = 0.0f;
    if (gid < (long long)N * ng) {
        const int n = (int)(gid / ng), j = (int)(gid % ng);
        const int k0 = j * G;
        // codes of the group: 8-byte loads where G * BITS / 8 is a multiple
        // of 8, else 4-byte ones (group 32 at odd widths)
        uint32_t w[NW + 1];
        const uint8_t* pg = packed + (size_t)n * ((size_t)K * BITS / 8) + (size_t)k0 * BITS / 8;
        if constexpr (NW % 2 == 0) {
            const uint2* pc = reinterpret_cast<const uint2*>(pg);
#pragma unroll
            for (int i = 0; i < NW / 2; i++) {
                const uint2 v = __ldg(pc + i);
                w[2 * i] = v.x;
                w[2 * i + 1] = v.y;
            }
        } else {
            const uint32_t* pc = reinterpret_cast<const uint32_t*>(pg);
#pragma unroll
            for (int i = 0; i < NW; i++) w[i] = __ldg(pc + i);
        }
        w[NW] = 0u;
        float s = 0.0f, z = 0.0f;
        float e4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        if constexpr (BITS == 2) {
            const uint2 c = __ldg(cb + (size_t)n * ng + j);
            e4[0] = h2f(c.x & 0xFFFFu); e4[1] = h2f(c.x >> 16); e4[2] = h2f(c.y & 0xFFFFu); e4[3] = h2f(c.y >> 16);
        } else {
            s = h2f(scale_bits(sc, scale_exp(sc), n, ng, j));
            z = (float)__ldg(zp + (size_t)n * ng + j);
        }
        // first outlier of the row at or after column k0 (columns ascend)
        int p = 0, pe = 0, oc = 0x7FFFFFFF;
        if (nnz > 0) {
            int lo = __ldg(row_ptr + n), hi = __ldg(row_ptr + n + 1);
            pe = hi;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (__ldg(col + mid) < k0) lo = mid + 1;
                else hi = mid;
            }
            p = lo;
            oc = p < pe ? __ldg(col + p) : 0x7FFFFFFF;
        }
        float fse = 0.0f, fww = 0.0f, fvv = 0.0f, fwv = 0.0f, m1 = 0.0f, m2 = 0.0f;
        const uint4* wg = reinterpret_cast<const uint4*>(W + (size_t)n * K + k0);
#pragma unroll
        for (int c8 = 0; c8 < G / 8; c8++) {
            const uint4 wv = __ldg(wg + c8);
            const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
            for (int e = 0; e < 8; e++) {
                const int i = 8 * c8 + e;
                constexpr uint32_t mask = (1u << BITS) - 1u;
                const int bit = BITS * i, wi = bit >> 5, off = bit & 31;
                uint32_t code = w[wi] >> off;
                if (off + BITS > 32) code |= w[wi + 1] << (32 - off);
                code &= mask;
                const float x = h2f(ww[e >> 1] >> (16 * (e & 1)));
                float v;
                if constexpr (BITS == 2) v = e4[code];
                else v = ((float)code - z) * s;   // exact: |q - zp| < 64 times an fp16 scale
                if (k0 + i == oc) {                 // FP16 outlier added back
                    v += h2f(__ldg(val + p));
                    ++p;
                    oc = p < pe ? __ldg(col + p) : 0x7FFFFFFF;
                }
                const float d = x - v;
                fse = fmaf(d, d, fse);
                fww = fmaf(x, x, fww);
                fvv = fmaf(v, v, fvv);
                fwv = fmaf(x, v, fwv);
                emax = fmaxf(emax, fabsf(d));
                const float a = fabsf(x);
                if (a > m1) { m2 = m1; m1 = a; }
                else if (a > m2) { m2 = a; }
            }
        }
        const float r = m1 == 0.0f ? 1.0f : (m2 == 0.0f ? INFINITY : m1 / m2);
        if (ratio) ratio[gid] = r;
        rmax = r;
        over = r > threshold ? 1.0f : 0.0f;
        se = fse; sww = fww; svv = fvv; swv = fwv;
    }
    // CTA reduction in a fixed order: warps by shuffles, then warp 0
    __shared__ double red[kThreads / 32][7];
    double v7[7] = {se, sww, svv, swv, (double)emax, (double)rmax, (double)over};
#pragma unroll
    for (int q = 0; q < 7; q++) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const double t = __shfl_xor_sync(0xffffffffu, v7[q], o);
            v7[q] = (q == 4 || q == 5) ? fmax(v7[q], t) : v7[q] + t;
        }
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0)
#pragma unroll
        for (int q = 0; q < 7; q++) red[warp][q] = v7[q];
    __syncthreads();
    if (threadIdx.x == 0) {
        double t[7];
#pragma unroll
        for (int q = 0; q < 7; q++) t[q] = red[0][q];
        for (int wv = 1; wv < kThreads / 32; wv++)
#pragma unroll
            for (int q = 0; q < 7; q++) t[q] = (q == 4 || q == 5) ? fmax(t[q], red[wv][q]) : t[q] + red[wv][q];
        part[blockIdx.x] = Partial{t[0], t[1], t[2], t[3], t[4], t[5], t[6]};
    }
}

// One CTA: the partials, each thread a fixed stride of them, then a fixed tree.
__global__ void __launch_bounds__(256) k_diag_final(const Partial* __restrict__ part, int P, long long count,
                                                      qg_diag* __restrict__ out)
{
    __shared__ double red[256][7];
    double t[7] = {0.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0};
    for (int i = threadIdx.x; i < P; i += 256) {
        const Partial p = part[i];
        t[0] += p.se; t[1] += p.sww; t[2] += p.svv; t[3] += p.swv;
        t[4] = fmax(t[4], p.emax); t[5] = fmax(t[5], p.rmax); t[6] += p.over;
    }
#pragma unroll
    for (int q = 0; q < 7; q++) red[threadIdx.x][q] = t[q];
    __syncthreads();
    for (int h = 128; h > 0; h >>= 1) {
        if ((int)threadIdx.x < h)
#pragma unroll
            for (int q = 0; q < 7; q++)
                red[threadIdx.x][q] = (q == 4 || q == 5) ? fmax(red[threadIdx.x][q], red[threadIdx.x + h][q])
                                                         : red[threadIdx.x][q] + red[threadIdx.x + h][q];
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        const double se = red[0][0], sww = red[0][1], svv = red[0][2], swv = red[0][3];
        qg_diag d;
        d.max_abs_err = red[0][4];
        d.rmse = sqrt(se / (double)count);
        d.cosine = (sww == 0.0 && svv == 0.0) ? 1.0 : (sww == 0.0 || svv == 0.0) ? 0.0 : swv / (sqrt(sww) * sqrt(svv));
        d.max_range_ratio = red[0][5];
        d.groups_over = (int64_t)red[0][6];
        *out = d;
    }
}

inline int blocks_for(int N, int K, int G) { return (int)ceil_div((long long)N * (K / G), kThreads); }

template <int BITS, int G>
qg_status run(const uint16_t* W, const qg_qweight& w, float threshold, float* ratio, qg_diag* out, void* ws,
              cudaStream_t s)
{
    const int P = blocks_for(w.N, w.K, G);
    Partial* part = static_cast<Partial*>(ws);
    k_diag<BITS, G><<<P, kThreads, 0, s>>>(W, w.N, w.K, w.packed, scale_src(w), w.zp,
                                           reinterpret_cast<const uint2*>(w.codebook), w.out_row_ptr, w.out_col,
                                           w.out_val, w.nnz, threshold, ratio, part);
    k_diag_final<<<1, 256, 0, s>>>(part, P, (long long)w.N * w.K, out);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "diagnostics launch");
    return QG_OK;
}

template <int BITS>
qg_status run_bits(const uint16_t* W, const qg_qweight& w, float threshold, float* ratio, qg_diag* out, void* ws,
                   cudaStream_t s)
{
    return w.group == 32   ? run<BITS, 32>(W, w, threshold, ratio, out, ws, s)
           : w.group == 64 ? run<BITS, 64>(W, w, threshold, ratio, out, ws, s)
                           : run<BITS, 128>(W, w, threshold, ratio, out, ws, s);
}

}  // namespace diag

size_t diag_workspace_bytes(int N, int K, int group)
{
    return align_up(sizeof(diag::Partial) * (size_t)diag::blocks_for(N, K, group), 256);
}

qg_status launch_diag(const uint16_t* W, const qg_qweight& w, float threshold, float* ratio, qg_diag* out, void* ws,
                      cudaStream_t s)
{
    switch (w.bits) {
        case 2: return diag::run_bits<2>(W, w, threshold, ratio, out, ws, s);
        case 3: return diag::run_bits<3>(W, w, threshold, ratio, out, ws, s);
        case 4: return diag::run_bits<4>(W, w, threshold, ratio, out, ws, s);
        case 5: return diag::run_bits<5>(W, w, threshold, ratio, out, ws, s);
        case 6: return diag::run_bits<6>(W, w, threshold, ratio, out, ws, s);
        default: return diag::run_bits<8>(W, w, threshold, ratio, out, ws, s);
    }
}

}  // namespace qg
