// Grouped (MoE) fused dequantization product on the 5th-generation tensor
// cores with the roles of the operands swapped: the dequantized weights are
// the MMA's M side (128 weight rows per CTA) and an expert's tokens are the N
// side (N = 16 * ceil(tokens / 16), at most 256), so an expert that receives
// a few dozen tokens costs no padding on the tensor core and its weights are
// read from HBM once (per 256 of its tokens).
//     y[pair, n] = sum_k x[token(pair), k] * (w_hat_e[n, k] + S_e[n, k])
//
// Routing (a stable counting sort of the (token, slot) pairs by expert,
// bjdmk.com.cn 5648983 page, sections 1-2) is done by the routing kernel;
// k_gather_x16 then writes x in that order as fp16 with the K positions of
// every block of 8 permuted (0,4,1,5,2,6,3,7) like the weight operand, and
// one CTA of k_gemm_swap_u4 computes a 128-row x (up to 256)-token tile:
//  * warp 8 (one lane) streams the token tile (TMA, 16-row boxes, 128-byte
//    swizzle) into a 3-deep ring, warp 9 the packed 4-bit weight tile of the
//    expert (TMA, 128 rows x 128 bytes = 4 K blocks) into a 4-deep ring;
//  * warps 0-7 (two threads per weight row) dequantize exactly as the prefill
//    kernel does (masks -> fp16 1024 + 2^p q, one packed FMA -> q - zp, one
//    packed multiply by the fp16 scale, FP16 outliers patched in) into a
//    3-deep ring of 128 x 64 fp16 tiles;
//  * warp 10 (one lane) issues four tcgen05.mma (M=128, N=tokens, K=16) per K
//    block into a TMEM accumulator of 128 lanes x 256 columns;
//  * warps 0-7 read the accumulator (lane = weight row, column = token) and
//    store y rows in pair order.
// Every mbarrier wait is bounded; a wait that gives up writes QG_ERR_TIMEOUT
// into the device status word.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>

#include "gemv_impl.cuh"
#include "ptx.cuh"
#include "qg_internal.h"
#include "tc_dequant.cuh"

namespace qg {

qg_status encode_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                    uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw);

namespace swap {

constexpr int BW = 128;        // weight rows per CTA (MMA M)
constexpr int NBMAX = 256;     // tokens per CTA (MMA N, a multiple of 16)
constexpr int BK = 64;         // K block (one 128-byte fp16 row of an operand tile)
constexpr int PK = 4;          // K blocks per packed tile (128-byte rows at 4 bits)
constexpr int SX = 3, SP = 4, SA = 3;
constexpr int kDeqWarps = 8;
constexpr int kWarpX = kDeqWarps, kWarpP = kDeqWarps + 1, kWarpMma = kDeqWarps + 2;
constexpr int kThreads = (kDeqWarps + 3) * 32;
constexpr int X_BYTES = NBMAX * BK * 2;      // 32 KB
constexpr int P_BYTES = BW * PK * BK / 2;    // 16 KB
constexpr int A_BYTES = BW * BK * 2;         // 16 KB
constexpr int OFF_P = SX * X_BYTES;
constexpr int OFF_A = OFF_P + SP * P_BYTES;
constexpr int OFF_BAR = OFF_A + SA * A_BYTES;
constexpr int SMEM = OFF_BAR + 1024 /* barriers */ + 1024 /* alignment */;
constexpr int TMEM_COLS = NBMAX;
constexpr int kMaxExperts = 32;              // tensor maps travel as kernel parameters

struct Maps {
    CUtensorMap w[kMaxExperts];   // packed codes of each expert, box 128 bytes x 128 rows
};

struct Args {
    int N, K, ng, chunk;
    const int* offsets;   // [E + 1] pair offsets of each expert in routed order
    const int* perm;      // routed order -> pair id (token * topk + slot)
    const int2* items;    // (expert, chunk)
    const int* n_items;
    const uint16_t* scale[kMaxExperts];
    const uint8_t* zp[kMaxExperts];
    const int* row_ptr[kMaxExperts];
    const int* col[kMaxExperts];
    const uint16_t* val[kMaxExperts];
    int nnz[kMaxExperts];
    void* y;              // [pairs, N]
    int y_bf16;
    int* status;
    uint32_t magic;       // gemv::kF16Magic, a run-time value (one logic op per code pair)
};

// x rows in routed order, bf16 -> fp16 with the K positions of every block of
// 8 in the order (0,4,1,5,2,6,3,7) of the weight operand.  Only the first
// *n_routed entries of perm are routed pairs (pairs with an id outside
// [0, E) are never placed); the rows after them are written as zeros.
__global__ void k_gather_x16(const __nv_bfloat16* __restrict__ x, int ldx, int K, const int* __restrict__ perm,
                             const int* __restrict__ n_routed, int P, int topk, __half* __restrict__ out)
{
    const int nr = *n_routed;
    const long long total8 = (long long)P * K / 8;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total8;
         i += (long long)gridDim.x * blockDim.x) {
        const long long e = i * 8;
        const int q = (int)(e / K), k = (int)(e % K);
        if (q >= nr) {
            *reinterpret_cast<uint4*>(out + e) = make_uint4(0u, 0u, 0u, 0u);
            continue;
        }
        const __nv_bfloat16* src = x + (size_t)(perm[q] / topk) * ldx + k;
        constexpr int pm[8] = {0, 4, 1, 5, 2, 6, 3, 7};
        __half h[8];
#pragma unroll
        for (int j = 0; j < 8; j++) h[j] = __float2half_rn(__bfloat162float(src[pm[j]]));
        *reinterpret_cast<uint4*>(out + e) = *reinterpret_cast<const uint4*>(h);
    }
}

template <int G>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_swap_u4(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ Maps maps,
                   const __grid_constant__ Args a)
{
    // work item of this CTA row (uniform over the CTA: nothing is set up yet)
    if ((int)blockIdx.y >= *a.n_items) return;
    const int2 item = a.items[blockIdx.y];
    const int e = item.x;
    const int m0 = a.offsets[e] + item.y * a.chunk;
    const int ntok = min(a.chunk, a.offsets[e + 1] - m0);
    const int NB = (ntok + 15) & ~15;   // MMA N: tokens rounded up to 16
    const int n0 = blockIdx.x * BW;
    const int KB = a.K / BK;

    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = ptx::smem_u32(smem);
    const uint32_t bars = sbase + OFF_BAR;
    auto full_x = [&](int s) { return bars + 8 * s; };
    auto empty_x = [&](int s) { return bars + 8 * (SX + s); };
    auto full_p = [&](int s) { return bars + 8 * (2 * SX + s); };
    auto empty_p = [&](int s) { return bars + 8 * (2 * SX + SP + s); };
    auto full_a = [&](int s) { return bars + 8 * (2 * SX + 2 * SP + s); };
    auto empty_a = [&](int s) { return bars + 8 * (2 * SX + 2 * SP + SA + s); };
    const uint32_t acc_full = bars + 8 * (2 * SX + 2 * SP + 2 * SA);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_BAR + 8 * (2 * SX + 2 * SP + 2 * SA + 1));
    auto x_tile = [&](int s) { return sbase + s * X_BYTES; };
    auto p_tile = [&](int s) { return smem + OFF_P + s * P_BYTES; };
    auto a_tile = [&](int s) { return sbase + OFF_A + s * A_BYTES; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < SX; s++) { ptx::mbar_init(full_x(s), 1); ptx::mbar_init(empty_x(s), 1); }
        for (int s = 0; s < SP; s++) { ptx::mbar_init(full_p(s), 1); ptx::mbar_init(empty_p(s), kDeqWarps); }
        for (int s = 0; s < SA; s++) { ptx::mbar_init(full_a(s), kDeqWarps); ptx::mbar_init(empty_a(s), 1); }
        ptx::mbar_init(acc_full, 1);
        ptx::fence_mbar_init();
    }
    if (warp == kWarpMma) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), TMEM_COLS);
        ptx::tmem_relinquish();
    }
    if (warp == kWarpX && lane == 0) {
        ptx::prefetch_tensormap(&xmap);
        ptx::prefetch_tensormap(&maps.w[e]);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    if (warp == kWarpX) {
        // ------------------------------------------------ token tiles (TMA, 16-row boxes)
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            for (int kb = 0; kb < KB; kb++) {
                if (!ptx::mbar_wait(empty_x(s), ph ^ 1u)) { ok = false; break; }
                ptx::mbar_expect_tx(full_x(s), (uint32_t)NB * BK * 2);
                for (int j = 0; j < NB / 16; j++)
                    ptx::tma_load_2d(x_tile(s) + j * 16 * BK * 2, &xmap, kb * BK, m0 + 16 * j, full_x(s));
                if (++s == SX) { s = 0; ph ^= 1u; }
            }
        }
    } else if (warp == kWarpP) {
        // ------------------------------------------------ packed weight tiles of expert e (TMA)
        if (lane == 0) {
            const int KP = (KB + PK - 1) / PK;
            int s = 0;
            uint32_t ph = 0;
            for (int kp = 0; kp < KP; kp++) {
                if (!ptx::mbar_wait(empty_p(s), ph ^ 1u)) { ok = false; break; }
                ptx::mbar_expect_tx(full_p(s), P_BYTES);
                ptx::tma_load_2d(ptx::smem_u32(p_tile(s)), &maps.w[e], kp * (PK * BK / 2), n0, full_p(s));
                if (++s == SP) { s = 0; ph ^= 1u; }
            }
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------ MMA issuer: D[w rows, tokens] += W * X^T
        if (lane == 0) {
            const uint32_t idesc = ptx::idesc_f16_f32(BW, NB);
            int sx = 0, sa = 0;
            uint32_t px = 0, pa = 0;
            for (int kb = 0; kb < KB; kb++) {
                if (!ptx::mbar_wait(full_x(sx), px) || !ptx::mbar_wait(full_a(sa), pa)) { ok = false; break; }
                ptx::tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < BK / 16; kk++)
                    ptx::mma_f16(tmem, ptx::sw128_desc(a_tile(sa) + 32 * kk), ptx::sw128_desc(x_tile(sx) + 32 * kk),
                                 idesc, (kb | kk) != 0);
                ptx::tc_commit(empty_x(sx));
                ptx::tc_commit(empty_a(sa));
                if (++sx == SX) { sx = 0; px ^= 1u; }
                if (++sa == SA) { sa = 0; pa ^= 1u; }
            }
            ptx::tc_commit(acc_full);
        }
    } else {
        // ------------------------------------------------ dequantization (two threads per weight row)
        const uint32_t magic = a.magic;
        const int r = threadIdx.x >> 1;                 // 0..127
        const int hk = threadIdx.x & 1;                 // which 32 k of the block
        const int nr = n0 + r;
        const int n = min(nr, a.N - 1);
        const uint16_t* sp_row = a.scale[e] + (size_t)n * a.ng;
        const uint8_t* zp_row = a.zp[e] + (size_t)n * a.ng;
        constexpr int KB_PER_G = G / BK;                // 1 or 2
        const int ng = a.ng;
        // parameters of the current group and of the next two (loads in flight)
        uint32_t sc_cur = __ldg(sp_row), zq_cur = __ldg(zp_row);
        uint32_t sc_n1 = ng > 1 ? __ldg(sp_row + 1) : 0u, zq_n1 = ng > 1 ? __ldg(zp_row + 1) : 0u;
        uint32_t sc_n2 = ng > 2 ? __ldg(sp_row + 2) : 0u, zq_n2 = ng > 2 ? __ldg(zp_row + 2) : 0u;
        // outlier cursor of this row: the next entry and the one after it
        const int* ocolp = a.col[e];
        const uint16_t* ovalp = a.val[e];
        int op = 0, oe = 0, ocol = 0x7FFFFFFF, ncol = 0x7FFFFFFF;
        uint16_t oval = 0, nval = 0;
        if (a.nnz[e] > 0 && nr < a.N) {
            op = a.row_ptr[e][n];
            oe = a.row_ptr[e][n + 1];
            if (op < oe) {
                ocol = ocolp[op];
                oval = ovalp[op];
            }
            if (op + 1 < oe) {
                ncol = ocolp[op + 1];
                nval = ovalp[op + 1];
            }
        }
        // swizzled offsets, fixed per thread: source chunk (2*sub + hk) of the
        // packed row, destination chunks (4*hk + j) of the fp16 row
        const uint32_t rsw = r & 7;
        uint32_t src_off[PK], dst_off[4];
#pragma unroll
        for (int sub = 0; sub < PK; sub++) src_off[sub] = r * 128 + (((2 * sub + hk) ^ rsw) << 4);
#pragma unroll
        for (int j = 0; j < 4; j++) dst_off[j] = r * 128 + (((4 * hk + j) ^ rsw) << 4);
        unsigned char* const atile0 = smem + OFF_A;
        const int KP = (KB + PK - 1) / PK;
        int sp = 0, sa = 0;
        uint32_t pp = 0, pa = 1;   // parities: full_p to wait for, empty_a to wait for
        for (int kp = 0; kp < KP && ok; kp++) {
            const unsigned char* pt = p_tile(sp);
            ok = __all_sync(0xffffffffu, ptx::mbar_wait(full_p(sp), pp));
            if (!ok) break;
#pragma unroll
            for (int sub = 0; sub < PK; sub++) {
                const int kb = kp * PK + sub;
                if (kb >= KB) break;
                if (kb > 0 && kb % KB_PER_G == 0) {      // next group
                    const int gi = kb / KB_PER_G;
                    sc_cur = sc_n1;
                    zq_cur = zq_n1;
                    sc_n1 = sc_n2;
                    zq_n1 = zq_n2;
                    if (gi + 2 < ng) {
                        sc_n2 = __ldg(sp_row + gi + 2);
                        zq_n2 = __ldg(zp_row + gi + 2);
                    }
                }
                const uint32_t add_lo = zq_cur * 0x00010001u + 0xE400E400u;   // -(1024 + zp)
                const uint32_t add_hi = zq_cur * 0x00100010u + 0xD400D400u;   // -(64 + zp)
                const uint32_t s2 = __byte_perm(sc_cur, 0u, 0x1010u);
                const uint4 w = *reinterpret_cast<const uint4*>(pt + src_off[sub]);
                ok = __all_sync(0xffffffffu, ptx::mbar_wait(empty_a(sa), pa));
                if (!ok) break;
                unsigned char* at = atile0 + sa * A_BYTES;
                *reinterpret_cast<uint4*>(at + dst_off[0]) = tc::deq8_u4(w.x, add_lo, add_hi, s2, magic);
                *reinterpret_cast<uint4*>(at + dst_off[1]) = tc::deq8_u4(w.y, add_lo, add_hi, s2, magic);
                *reinterpret_cast<uint4*>(at + dst_off[2]) = tc::deq8_u4(w.z, add_lo, add_hi, s2, magic);
                *reinterpret_cast<uint4*>(at + dst_off[3]) = tc::deq8_u4(w.w, add_lo, add_hi, s2, magic);
                // FP16 outliers in this thread's 32 k: the dense value there is exactly 0
                const int k0 = kb * BK + 32 * hk;
                while (ocol < k0 + 32) {
                    if (ocol >= k0) {
                        const int kk = ocol - kb * BK;
                        *reinterpret_cast<uint16_t*>(at + r * 128 + (((kk >> 3) ^ rsw) << 4) + (tc::perm8_pos(kk) << 1)) =
                            oval;
                    }
                    ocol = ncol;
                    oval = nval;
                    if (++op + 1 < oe) {
                        ncol = ocolp[op + 1];
                        nval = ovalp[op + 1];
                    } else {
                        ncol = 0x7FFFFFFF;
                    }
                }
                ptx::fence_proxy_async();
                __syncwarp();
                if (lane == 0) {
                    ptx::mbar_arrive(full_a(sa));
                    // the packed slot goes back to its producer only after the
                    // stores that consumed its codes
                    if (sub == PK - 1 || kb == KB - 1) ptx::mbar_arrive(empty_p(sp));
                }
                if (++sa == SA) { sa = 0; pa ^= 1u; }
            }
            if (++sp == SP) { sp = 0; pp ^= 1u; }
        }
        // ------------------------------------------------ epilogue: TMEM (lane = weight row, column = token) -> y
        if (ok) ok = __all_sync(0xffffffffu, ptx::mbar_wait(acc_full, 0));
        if (ok) {
            ptx::tc_fence_after();
            const int q = warp & 3, half = warp >> 2;   // TMEM lanes 32q.., column chunks of parity `half`
            const int nrow = n0 + 32 * q + lane;
            for (int c = half; 16 * c < NB; c += 2) {
                uint32_t v[16];
                ptx::tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(16 * c), v);
                ptx::tmem_ld_wait();
                if (nrow < a.N) {
#pragma unroll
                    for (int j = 0; j < 16; j++) {
                        const int col = 16 * c + j;
                        if (col < ntok) {
                            const size_t yo = (size_t)a.perm[m0 + col] * a.N + nrow;
                            if (a.y_bf16)
                                reinterpret_cast<__nv_bfloat16*>(a.y)[yo] = __float2bfloat16_rn(__uint_as_float(v[j]));
                            else
                                reinterpret_cast<float*>(a.y)[yo] = __uint_as_float(v[j]);
                        }
                    }
                }
            }
        }
    }
    if (!ok && a.status) atomicExch(a.status, (int)QG_ERR_TIMEOUT);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == kWarpMma) ptx::tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace swap

bool moe_tc_eligible(const qg_qweight* experts, int E)
{
    return E <= swap::kMaxExperts && experts[0].bits == 4 && experts[0].K % swap::BK == 0;
}

size_t moe_tc_x16_bytes(int P, int K) { return align_up((size_t)P * K * 2, 256); }

template <int G>
static qg_status moe_tc_run(const uint16_t* x, int T, int k, const qg_qweight* experts, int E, void* y, qg_ydtype yt,
                            const int* offsets, const int* perm, const int2* items, const int* n_items, int max_items,
                            void* x16p, cudaStream_t s)
{
    using namespace swap;
    const int P = T * k, N = experts[0].N, K = experts[0].K;
    {
        const long long total8 = (long long)P * K / 8;
        const int blocks = (int)std::min<long long>(ceil_div(total8, 256), (long long)num_sms() * 8);
        k_gather_x16<<<blocks, 256, 0, s>>>(reinterpret_cast<const __nv_bfloat16*>(x), K, K, perm, offsets + E, P, k,
                                            static_cast<__half*>(x16p));
    }
    CUtensorMap xmap;
    qg_status st = encode_2d(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, x16p, (uint64_t)K, (uint64_t)P, (uint64_t)K * 2,
                             BK, 16, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != QG_OK) return st;
    Maps maps;
    memset(&maps, 0, sizeof(maps));
    Args a;
    memset(&a, 0, sizeof(a));
    for (int e = 0; e < E; e++) {
        st = encode_2d(&maps.w[e], CU_TENSOR_MAP_DATA_TYPE_UINT8, experts[e].packed, (uint64_t)K / 2, (uint64_t)N,
                       (uint64_t)K / 2, PK * BK / 2, BW, CU_TENSOR_MAP_SWIZZLE_128B);
        if (st != QG_OK) return st;
        a.scale[e] = experts[e].scale;
        a.zp[e] = experts[e].zp;
        a.row_ptr[e] = experts[e].out_row_ptr;
        a.col[e] = experts[e].out_col;
        a.val[e] = experts[e].out_val;
        a.nnz[e] = experts[e].nnz;
    }
    a.N = N; a.K = K; a.ng = K / G; a.chunk = NBMAX;
    a.offsets = offsets; a.perm = perm; a.items = items; a.n_items = n_items;
    a.y = y; a.y_bf16 = yt == QG_Y_BF16;
    a.status = device_status_ptr();
    a.magic = gemv::kF16Magic;
    st = gemv::allow_smem(k_gemm_swap_u4<G>, SMEM);
    if (st != QG_OK) return st;
    dim3 grid((unsigned)ceil_div(N, BW), (unsigned)max_items, 1);
    k_gemm_swap_u4<G><<<grid, kThreads, SMEM, s>>>(xmap, maps, a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "grouped tensor-core kernel launch");
    return QG_OK;
}

qg_status launch_moe_tc(const uint16_t* x, int T, int k, const qg_qweight* experts, int E, void* y, qg_ydtype yt,
                        const int* offsets, const int* perm, const int2* items, const int* n_items, int max_items,
                        void* x16p, cudaStream_t s)
{
    return experts[0].group == 64
               ? moe_tc_run<64>(x, T, k, experts, E, y, yt, offsets, perm, items, n_items, max_items, x16p, s)
               : moe_tc_run<128>(x, T, k, experts, E, y, yt, offsets, perm, items, n_items, max_items, x16p, s);
}

}  // namespace qg
