// Prefill-side fused dequantization product on the 5th-generation tensor
// cores (tcgen05 + TMEM), for M above the decode range:
//     y[m, n] = sum_k x[m, k] * (w_hat[n, k] + S[n, k])
//
// The pages' fused kernel dequantizes INT4 tiles into shared memory and runs
// the tensor cores on them (bjdmk.com.cn 5414039 page, section 3); this is
// that structure written for sm_103a:
//  * one CTA computes a 128 x 256 tile of y (128 tokens x 256 weight rows)
//    with its fp32 accumulator in tensor memory (256 TMEM columns);
//  * warp 8 (one lane) streams, per K block of 64, the fp16 x tile (TMA,
//    128-byte swizzle) and the packed 4-bit weight tile (TMA, 256 rows x
//    32 bytes) into a 3-stage shared-memory ring;
//  * warps 0-7 (one weight row per thread) unpack the codes with byte
//    permutes and masks into fp16 1024 + 2^p q, turn them into the exact
//    integers q - zp with one packed FMA and multiply by the fp16 group scale
//    (one rounding), patch the FP16 outliers of the block in place, and
//    store the 256 x 64 fp16 tile in the K-major 128-byte-swizzled layout the
//    tensor core reads;
//  * warp 9 (one lane) issues four tcgen05.mma (M=128, N=256, K=16) per
//    stage and commits them to the stage's "empty" barrier;
//  * warps 0-7 then read the accumulator with tcgen05.ld and store y.
// Every mbarrier wait is bounded (a wait that gives up writes QG_ERR_TIMEOUT
// into the workspace status word).  x is first converted bf16 -> fp16 into
// the workspace (exact in fp16's normal range).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "gemv_impl.cuh"
#include "ptx.cuh"
#include "qg_internal.h"

namespace qg {

qg_status launch_gemv_chunked(const uint16_t* x, int M, int ldx, const qg_qweight& w, void* y, int ldy,
                              qg_ydtype yt, cudaStream_t s);

namespace tc {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 3;
constexpr int kDeqWarps = 8, kThreads = (kDeqWarps + 2) * 32;
constexpr int A_BYTES = BM * BK * 2;   // 16 KB fp16
constexpr int B_BYTES = BN * BK * 2;   // 32 KB fp16

template <int BITS>
struct Cfg {
    static constexpr int P_BYTES = BN * BK * BITS / 8;    // packed tile
    static constexpr int P_ALIGNED = (P_BYTES + 1023) / 1024 * 1024;
    static constexpr int STAGE = A_BYTES + B_BYTES + P_ALIGNED;
    static constexpr int SMEM = STAGES * STAGE + 1024 /* barriers */ + 1024 /* alignment */;
};

struct Args {
    int M, N, K, ng;
    const uint16_t* scale;
    const uint8_t* zp;
    const int* row_ptr;
    const int* col;
    const uint16_t* val;
    int nnz;
    void* y;
    int ldy;
    int y_bf16;
    int* status;
};

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// 8 consecutive 4-bit codes (one 32-bit word, code i at bits 4i) ->
// 4 fp16 pairs ((q_2j - zp) * s, (q_2j+1 - zp) * s) in k order.
__device__ __forceinline__ uint4 deq8_u4(uint32_t v, uint32_t zp_add, uint32_t s2)
{
    constexpr uint32_t mul = 0x3C00u | (0x2C00u << 16);   // (1, 1/16)
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; j++) {
        // byte j into bytes 0 and 2: low nibble -> low half, high nibble -> high half (<< 4)
        const uint32_t u = __byte_perm(v, 0u, 0x4040u | (uint32_t)j | ((uint32_t)j << 8));
        const uint32_t raw = (u & 0x00F0000Fu) | 0x64006400u;
        o[j] = hmul2_u32(gemv::hfma2_u32(raw, mul, zp_add), s2);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

template <int G>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_tc_u4(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
                 const __grid_constant__ Args a)
{
    constexpr int BITS = 4;
    using C = Cfg<BITS>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = ptx::smem_u32(smem);
    const uint32_t bars = sbase + STAGES * C::STAGE;
    auto full_a = [&](int s) { return bars + 8 * s; };
    auto full_b = [&](int s) { return bars + 8 * (STAGES + s); };
    auto empty = [&](int s) { return bars + 8 * (2 * STAGES + s); };
    const uint32_t acc_full = bars + 8 * (3 * STAGES);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + STAGES * C::STAGE + 8 * (3 * STAGES + 1));
    auto a_tile = [&](int s) { return sbase + s * C::STAGE; };
    auto b_tile = [&](int s) { return sbase + s * C::STAGE + A_BYTES; };
    auto p_tile = [&](int s) { return smem + s * C::STAGE + A_BYTES + B_BYTES; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * BM, n0 = blockIdx.y * BN;
    const int KB = a.K / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; s++) {
            ptx::mbar_init(full_a(s), 1);
            ptx::mbar_init(full_b(s), kDeqWarps);
            ptx::mbar_init(empty(s), 1);
        }
        ptx::mbar_init(acc_full, 1);
        ptx::fence_mbar_init();
    }
    if (warp == kDeqWarps + 1) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), 256);
        ptx::tmem_relinquish();
    }
    if (warp == kDeqWarps && lane == 0) {
        ptx::prefetch_tensormap(&xmap);
        ptx::prefetch_tensormap(&wmap);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    if (warp == kDeqWarps) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            for (int kb = 0; kb < KB; kb++) {
                const int s = kb % STAGES;
                const uint32_t ph = (uint32_t)(kb / STAGES) & 1u;
                if (!ptx::mbar_wait(empty(s), ph ^ 1u)) { ok = false; break; }
                ptx::mbar_expect_tx(full_a(s), A_BYTES + C::P_BYTES);
                ptx::tma_load_2d(a_tile(s), &xmap, kb * BK, m0, full_a(s));
                ptx::tma_load_2d(ptx::smem_u32(p_tile(s)), &wmap, kb * (BK * BITS / 8), n0, full_a(s));
            }
        }
    } else if (warp == kDeqWarps + 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = ptx::idesc_f16_f32(BM, BN);
            for (int kb = 0; kb < KB; kb++) {
                const int s = kb % STAGES;
                const uint32_t ph = (uint32_t)(kb / STAGES) & 1u;
                if (!ptx::mbar_wait(full_a(s), ph) || !ptx::mbar_wait(full_b(s), ph)) { ok = false; break; }
                ptx::tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < BK / 16; kk++)
                    ptx::mma_f16(tmem, ptx::sw128_desc(a_tile(s) + 32 * kk), ptx::sw128_desc(b_tile(s) + 32 * kk), idesc,
                                 (kb | kk) != 0);
                ptx::tc_commit(empty(s));
            }
            ptx::tc_commit(acc_full);
        }
    } else {
        // ------------------------------------------------ dequantization (one row per thread)
        const int r = threadIdx.x;                      // 0..255
        const int nr = n0 + r;
        const int n = min(nr, a.N - 1);
        const size_t pbase = (size_t)n * a.ng;
        // per-group parameters, fetched two groups ahead
        constexpr int KB_PER_G = G / BK;                // 1 or 2
        const int ng = a.ng;
        uint32_t sc[3], zq[3];
        auto fetch = [&](int gi, int slot) {
            if (gi < ng) {
                sc[slot] = __ldg(a.scale + pbase + gi);
                zq[slot] = __ldg(a.zp + pbase + gi);
            }
        };
        fetch(0, 0);
        fetch(1, 1);
        // outlier cursor of this row
        int op = 0, oe = 0, ocol = 0x7FFFFFFF;
        uint16_t oval = 0;
        if (a.nnz > 0 && nr < a.N) {
            op = a.row_ptr[n];
            oe = a.row_ptr[n + 1];
            if (op < oe) {
                ocol = a.col[op];
                oval = a.val[op];
            }
        }
        const uint32_t brow = r * 128, bsw = r & 7;
        for (int kb = 0; kb < KB; kb++) {
            const int s = kb % STAGES;
            const uint32_t ph = (uint32_t)(kb / STAGES) & 1u;
            const int gi = kb / KB_PER_G;
            const int slot = gi % 3;
            if (kb % KB_PER_G == 0) fetch(gi + 2, (gi + 2) % 3);
            const uint32_t zp = zq[slot];
            const uint32_t zp_add = zp * (1u | (16u << 16)) + (0xE400u | (0xD400u << 16));
            const uint32_t s1 = sc[slot] & 0xFFFFu;
            const uint32_t s2 = s1 | (s1 << 16);
            if (!ptx::mbar_wait(full_a(s), ph)) { ok = false; break; }
            const uint4* prow = reinterpret_cast<const uint4*>(p_tile(s) + r * 32);
            const uint4 w01 = prow[0], w23 = prow[1];
            const uint32_t wv[8] = {w01.x, w01.y, w01.z, w01.w, w23.x, w23.y, w23.z, w23.w};
            unsigned char* bt = smem + s * C::STAGE + A_BYTES;
#pragma unroll
            for (int c = 0; c < 8; c++) {
                const uint4 h = deq8_u4(wv[c], zp_add, s2);
                *reinterpret_cast<uint4*>(bt + brow + ((c ^ bsw) << 4)) = h;
            }
            // FP16 outliers of this block: the dense value there is exactly 0
            const int k0 = kb * BK;
            while (ocol < k0 + BK) {
                const int kk = ocol - k0;
                *reinterpret_cast<uint16_t*>(bt + brow + (((kk >> 3) ^ bsw) << 4) + ((kk & 7) << 1)) = oval;
                if (++op < oe) {
                    ocol = a.col[op];
                    oval = a.val[op];
                } else {
                    ocol = 0x7FFFFFFF;
                }
            }
            ptx::fence_proxy_async();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(full_b(s));
        }
        // ------------------------------------------------ epilogue: TMEM -> y
        if (ok && ptx::mbar_wait(acc_full, 0)) {
            ptx::tc_fence_after();
            const int q = warp & 3, half = warp >> 2;
            const int m = m0 + 32 * q + lane;
#pragma unroll 1
            for (int i = 0; i < 8; i++) {
                const int cb = 128 * half + 16 * i;
                uint32_t v[16];
                ptx::tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)cb, v);
                ptx::tmem_ld_wait();
                if (m < a.M) {
                    const int nb = n0 + cb;
                    if (a.y_bf16) {
                        __nv_bfloat16* yr = reinterpret_cast<__nv_bfloat16*>(a.y) + (size_t)m * a.ldy;
#pragma unroll
                        for (int j = 0; j < 16; j++)
                            if (nb + j < a.N) yr[nb + j] = __float2bfloat16_rn(__uint_as_float(v[j]));
                    } else {
                        float* yr = reinterpret_cast<float*>(a.y) + (size_t)m * a.ldy;
                        if (nb + 16 <= a.N && ((reinterpret_cast<uintptr_t>(yr + nb) & 15u) == 0)) {
#pragma unroll
                            for (int j = 0; j < 16; j += 4)
                                *reinterpret_cast<float4*>(yr + nb + j) =
                                    make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                                                __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]));
                        } else {
#pragma unroll
                            for (int j = 0; j < 16; j++)
                                if (nb + j < a.N) yr[nb + j] = __uint_as_float(v[j]);
                        }
                    }
                }
            }
        } else {
            ok = false;
        }
    }
    if (!ok) atomicExch(a.status, (int)QG_ERR_TIMEOUT);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == kDeqWarps + 1) ptx::tmem_dealloc(tmem, 256);
}

// bf16 [M, ldx] -> fp16 [M, K] (exact for |x| in fp16's normal range)
__global__ void k_x_to_f16(const __nv_bfloat16* __restrict__ x, int M, int K, int ldx, __half* __restrict__ out)
{
    const long long total8 = (long long)M * K / 8;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total8;
         i += (long long)gridDim.x * blockDim.x) {
        const long long e = i * 8;
        const int m = (int)(e / K), k = (int)(e % K);
        const __nv_bfloat16* src = x + (size_t)m * ldx + k;
        __half h[8];
#pragma unroll
        for (int j = 0; j < 8; j++) h[j] = __float2half_rn(__bfloat162float(src[j]));
        *reinterpret_cast<uint4*>(out + e) = *reinterpret_cast<const uint4*>(h);
    }
}

qg_status encode_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                    uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw)
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !f)
            return fail(QG_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
        fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1u, 1u};
    CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(QG_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return QG_OK;
}

struct Ws {
    int* status;
    __half* x16;
};

size_t ws_layout(int M, int K, Ws* w, void* base)
{
    const size_t o_x = 256;
    const size_t total = align_up(o_x + (size_t)M * K * 2, 256);
    if (w && base) {
        w->status = reinterpret_cast<int*>(base);
        w->x16 = reinterpret_cast<__half*>(static_cast<char*>(base) + o_x);
    }
    return total;
}

bool eligible(const qg_qweight& w) { return w.bits == 4 && (w.K % BK) == 0; }

template <int G>
qg_status run(const uint16_t* x, int M, int ldx, const qg_qweight& w, void* y, int ldy, qg_ydtype yt, void* ws,
              cudaStream_t s)
{
    using C = Cfg<4>;
    Ws p;
    ws_layout(M, w.K, &p, ws);
    {
        const long long total8 = (long long)M * w.K / 8;
        const int blocks = (int)std::min<long long>(ceil_div(total8, 256), (long long)num_sms() * 8);
        k_x_to_f16<<<blocks, 256, 0, s>>>(reinterpret_cast<const __nv_bfloat16*>(x), M, w.K, ldx, p.x16);
    }
    CUtensorMap xmap, wmap;
    qg_status st = encode_2d(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, p.x16, (uint64_t)w.K, (uint64_t)M,
                             (uint64_t)w.K * 2, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != QG_OK) return st;
    st = encode_2d(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, w.packed, (uint64_t)w.K / 2, (uint64_t)w.N,
                   (uint64_t)w.K / 2, BK / 2, BN, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st != QG_OK) return st;
    Args a;
    a.M = M; a.N = w.N; a.K = w.K; a.ng = w.K / G;
    a.scale = w.scale; a.zp = w.zp;
    a.row_ptr = w.out_row_ptr; a.col = w.out_col; a.val = w.out_val; a.nnz = w.nnz;
    a.y = y; a.ldy = ldy; a.y_bf16 = yt == QG_Y_BF16;
    a.status = p.status;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(k_gemm_tc_u4<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return cuda_fail(e, "tensor-core kernel: shared memory attribute");
        attr = true;
    }
    dim3 grid((unsigned)ceil_div(M, BM), (unsigned)ceil_div(w.N, BN), 1);
    k_gemm_tc_u4<G><<<grid, kThreads, C::SMEM, s>>>(xmap, wmap, a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "tensor-core kernel launch");
    return QG_OK;
}

}  // namespace tc

size_t gemm_workspace_bytes(int M, const qg_qweight& w)
{
    return tc::eligible(w) ? tc::ws_layout(M, w.K, nullptr, nullptr) : 0;
}

qg_status launch_gemm(const uint16_t* x, int M, int ldx, const qg_qweight& w, void* y, int ldy, qg_ydtype yt,
                      void* ws, size_t, cudaStream_t s)
{
    if (tc::eligible(w))
        return w.group == 64 ? tc::run<64>(x, M, ldx, w, y, ldy, yt, ws, s) : tc::run<128>(x, M, ldx, w, y, ldy, yt, ws, s);
    return launch_gemv_chunked(x, M, ldx, w, y, ldy, yt, s);
}

}  // namespace qg
