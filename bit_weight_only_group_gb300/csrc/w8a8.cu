// W8A8 decode product: int8 weights (the 8-bit affine or symmetric format)
// and int8 activations quantized dynamically per token ("Inference
// acceleration guide" page, section 1.2: W8A8 quantizes weights and
// activations to INT8, the activations per token; section 1.1: the
// symmetric INT8 range [-127, 127]):
//     y[m, n] = s_m * ( sum_g scale[n,g] * sum_{k in g} q_x[m,k] (q_w[n,k] - zp[n,g])
//                       + sum_{outliers (n,k,v)} q_x[m,k] * v )
// The integer sums are exact (dp4a, 32-bit), scales and outliers are
// applied in fp32.  GB300's int8 tensor-core rate is far below its fp16 rate,
// so the products run on the CUDA cores' four-way int8 dot product; at
// M <= 16 the product is bound by the weight stream either way.
//   k_quant_act  one CTA per token: max |x|, s = max / 127, q = round(x / s)
//   k_w8a8<MT>   one warp per weight row, lanes over K in 16-byte runs
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gemv_impl.cuh"
#include "qg_internal.h"

namespace qg {
namespace w8a8 {

constexpr int kActThreads = 256;
constexpr int kWarpsPerCta = 8;

__global__ void __launch_bounds__(kActThreads) k_quant_act(const __nv_bfloat16* __restrict__ x, int K, int ldx,
                                                            int8_t* __restrict__ q, float* __restrict__ s)
{
    const int m = blockIdx.x;
    const __nv_bfloat16* xr = x + (size_t)m * ldx;
    float a = 0.0f;
    for (int k = threadIdx.x; k < K; k += kActThreads) a = fmaxf(a, fabsf(__bfloat162float(xr[k])));
    __shared__ float red[kActThreads / 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
    __syncthreads();
    float amax = 0.0f;
#pragma unroll
    for (int w = 0; w < kActThreads / 32; w++) amax = fmaxf(amax, red[w]);
    const float sm = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 127.0f);
    for (int k = threadIdx.x; k < K; k += kActThreads) {
        const float v = fminf(fmaxf(rintf(__fdiv_rn(__bfloat162float(xr[k]), sm)), -127.0f), 127.0f);
        q[(size_t)m * K + k] = (int8_t)v;
    }
    if (threadIdx.x == 0) s[m] = sm;
}

// sum of a_i * b_i over the four bytes: a unsigned, b signed
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

template <int MT>
__global__ void __launch_bounds__(kWarpsPerCta * 32)
    k_w8a8(const int8_t* __restrict__ xq, const float* __restrict__ sx, int M, int N, int K, int G,
           const uint8_t* __restrict__ packed, const ScaleSrc sc, const uint8_t* __restrict__ zp,
           const int* __restrict__ row_ptr, const int* __restrict__ col, const uint16_t* __restrict__ val, int nnz,
           void* __restrict__ y, int ldy, int y_bf16)
{
    const int lane = threadIdx.x & 31;
    const int n = blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
    if (n >= N) return;   // whole warp
    const int ng = K / G;
    const int E8 = scale_exp(sc);
    const uint8_t* wr = packed + (size_t)n * K;
    float acc[MT];
#pragma unroll
    for (int m = 0; m < MT; m++) acc[m] = 0.0f;
#pragma unroll 4
    for (int k = lane * 16; k < K; k += 512) {
        const uint4 wv = gemv::ldg_stream128(wr + k);
        const int g = k / G;   // a 16-code run lies in one group (G is a multiple of 16)
        const float sw = __half2float(__ushort_as_half((uint16_t)scale_bits(sc, E8, n, ng, g)));
        const int z = __ldg(zp + (size_t)n * ng + g);
#pragma unroll
        for (int m = 0; m < MT; m++) {
            if (m < M) {
                const uint4 xv = __ldg(reinterpret_cast<const uint4*>(xq + (size_t)m * K + k));
                int d = dp4a_us(wv.x, xv.x, 0);
                d = dp4a_us(wv.y, xv.y, d);
                d = dp4a_us(wv.z, xv.z, d);
                d = dp4a_us(wv.w, xv.w, d);
                int sq = dp4a_ss(0x01010101u, xv.x, 0);   // sum of the 16 activation codes
                sq = dp4a_ss(0x01010101u, xv.y, sq);
                sq = dp4a_ss(0x01010101u, xv.z, sq);
                sq = dp4a_ss(0x01010101u, xv.w, sq);
                acc[m] = fmaf(sw, (float)(d - z * sq), acc[m]);   // exact integer, then one scale
            }
        }
    }
#pragma unroll
    for (int m = 0; m < MT; m++)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc[m] += __shfl_xor_sync(0xffffffffu, acc[m], o);
    if (lane < MT && lane < M) {
        const int m = lane;
        float v = 0.0f;
#pragma unroll
        for (int i = 0; i < MT; i++) v = i == m ? acc[i] : v;
        if (nnz > 0)
            for (int p = __ldg(row_ptr + n); p < __ldg(row_ptr + n + 1); p++)
                v = fmaf((float)xq[(size_t)m * K + __ldg(col + p)], __half2float(__ushort_as_half(__ldg(val + p))), v);
        v *= sx[m];
        if (y_bf16) reinterpret_cast<__nv_bfloat16*>(y)[(size_t)m * ldy + n] = __float2bfloat16_rn(v);
        else reinterpret_cast<float*>(y)[(size_t)m * ldy + n] = v;
    }
}

struct Ws {
    int8_t* q;
    float* s;
};

size_t ws_layout(int M, int K, Ws* w, void* base)
{
    const size_t oq = 0, os = align_up((size_t)M * K, 256);
    const size_t total = os + align_up(sizeof(float) * (size_t)M, 256);
    if (w && base) {
        w->q = reinterpret_cast<int8_t*>(static_cast<char*>(base) + oq);
        w->s = reinterpret_cast<float*>(static_cast<char*>(base) + os);
    }
    return total;
}

template <int MT>
qg_status run(const Ws& p, int M, const qg_qweight& w, void* y, int ldy, qg_ydtype yt, cudaStream_t s)
{
    const int blocks = (int)ceil_div(w.N, kWarpsPerCta);
    k_w8a8<MT><<<blocks, kWarpsPerCta * 32, 0, s>>>(p.q, p.s, M, w.N, w.K, w.group, w.packed, scale_src(w), w.zp,
                                                    w.out_row_ptr, w.out_col, w.out_val, w.nnz, y, ldy,
                                                    yt == QG_Y_BF16);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "W8A8 kernel launch");
    return QG_OK;
}

}  // namespace w8a8

size_t w8a8_workspace_bytes(int M, int K) { return w8a8::ws_layout(M, K, nullptr, nullptr); }

qg_status launch_w8a8(const uint16_t* x, int M, int ldx, const qg_qweight& w, void* y, int ldy, qg_ydtype yt,
                      void* ws, cudaStream_t s)
{
    w8a8::Ws p{};
    w8a8::ws_layout(M, w.K, &p, ws);
    w8a8::k_quant_act<<<M, w8a8::kActThreads, 0, s>>>(reinterpret_cast<const __nv_bfloat16*>(x), w.K, ldx, p.q, p.s);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "activation quantizer launch");
    if (M <= 1) return w8a8::run<1>(p, M, w, y, ldy, yt, s);
    if (M <= 2) return w8a8::run<2>(p, M, w, y, ldy, yt, s);
    if (M <= 4) return w8a8::run<4>(p, M, w, y, ldy, yt, s);
    if (M <= 8) return w8a8::run<8>(p, M, w, y, ldy, yt, s);
    return w8a8::run<16>(p, M, w, y, ldy, yt, s);
}

}  // namespace qg
