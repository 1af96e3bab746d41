// Prefill-side fused dequantization product on the 5th-generation tensor
// cores (tcgen05 + TMEM), for M above the decode range:
//     y[m, n] = sum_k x[m, k] * (w_hat[n, k] + S[n, k])
//
// The pages' fused kernel dequantizes INT4 tiles into shared memory and runs
// the tensor cores on them ("70B on one GPU" page, section 3); this is
// that structure written for sm_103a:
//  * one CTA computes a 256 x 256 tile of y (256 tokens x 256 weight rows)
//    as two fp32 accumulators of 128 tokens in tensor memory (all 512 TMEM
//    columns), so every dequantized weight tile feeds 256 tokens;
//  * warp 16 (one lane) streams the fp16 x tiles (TMA, 128-byte swizzle,
//    256 x 64) into a 2-deep ring and warp 17 the packed 4-bit weight tiles
//    (TMA, 256 rows x 128 bytes = 4 K blocks, 128-byte swizzle) into a 2-deep
//    ring; each ring has its own full/empty mbarriers, so loads run ahead of
//    the consumers;
//  * warps 0-15 (two threads per weight row, 32 k each) unpack the codes with
//    masks into fp16 1024 + 2^p q, turn them into the exact integers q - zp
//    with one packed FMA and multiply by the fp16 group scale (one
//    rounding), patch the FP16 outliers of the block in place, and store the
//    256 x 64 fp16 tile in the K-major 128-byte-swizzled layout the tensor
//    core reads (K order permuted inside blocks of 8, matching x);
//    the fp16 tiles go to a 3-deep ring (the packed slot is released once
//    the stores that consumed its codes are issued);
//  * warp 18 (one lane) issues eight tcgen05.mma (M=128, N=256, K=16) per K
//    block, four per accumulator, and commits them to the x and fp16
//    rings' "empty" barriers;
//  * warps 0-15 then read the accumulator with tcgen05.ld and store y.
// Every mbarrier wait is bounded (a wait that gives up writes QG_ERR_TIMEOUT
// into the device status word read by qgemm_device_status).  x is first
// converted bf16 -> fp16 into the workspace (exact in fp16's normal range).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "gemv_impl.cuh"
#include "ptx.cuh"
#include "tc_dequant.cuh"
#include "qg_internal.h"

namespace qg {

qg_status launch_gemv_chunked(const uint16_t* x, int M, int ldx, const qg_qweight& w, void* y, int ldy,
                              qg_ydtype yt, cudaStream_t s);

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


namespace tc {

constexpr int BM = 256, BN = 256, BK = 64;
constexpr int MH = 128;                 // tokens per accumulator (one tcgen05.mma covers M = 128)
constexpr int SA = 2, SP = 2, SB = 3;   // ring depths: x tiles, packed tiles, fp16 weight tiles
constexpr int TMEM_COLS = 2 * BN;       // two fp32 accumulators of 128 x 256
constexpr int PK = 4;                   // K blocks per packed tile (128-byte rows at 4 bits)
constexpr int kDeqWarps = 16;
constexpr int kWarpA = kDeqWarps, kWarpP = kDeqWarps + 1, kWarpMma = kDeqWarps + 2;
constexpr int kThreads = (kDeqWarps + 3) * 32;
constexpr int A_BYTES = BM * BK * 2;   // 32 KB fp16
constexpr int B_BYTES = BN * BK * 2;   // 32 KB fp16

template <int BITS>
struct Cfg {
    static constexpr int P_BYTES = BN * PK * BK * BITS / 8;   // packed tile: 256 rows x 128 bytes
    static constexpr int P_ALIGNED = (P_BYTES + 1023) / 1024 * 1024;
    static constexpr int OFF_B = SA * A_BYTES;
    static constexpr int OFF_P = OFF_B + SB * B_BYTES;
    static constexpr int OFF_BAR = OFF_P + SP * P_ALIGNED;
    static constexpr int SMEM = OFF_BAR + 1024 /* barriers */ + 1024 /* alignment */;
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
    uint32_t magic;   // gemv::kF16Magic, a run-time value (one logic op per code pair)
};

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
    const uint32_t bars = sbase + C::OFF_BAR;
    // barriers: full/empty per ring slot, then the accumulator-ready barrier
    auto full_a = [&](int s) { return bars + 8 * s; };
    auto empty_a = [&](int s) { return bars + 8 * (SA + s); };
    auto full_p = [&](int s) { return bars + 8 * (2 * SA + s); };
    auto empty_p = [&](int s) { return bars + 8 * (2 * SA + SP + s); };
    auto full_b = [&](int s) { return bars + 8 * (2 * SA + 2 * SP + s); };
    auto empty_b = [&](int s) { return bars + 8 * (2 * SA + 2 * SP + SB + s); };
    const uint32_t acc_full = bars + 8 * (2 * SA + 2 * SP + 2 * SB);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 8 * (2 * SA + 2 * SP + 2 * SB + 1));
    auto a_tile = [&](int s) { return sbase + s * A_BYTES; };
    auto b_tile = [&](int s) { return sbase + C::OFF_B + s * B_BYTES; };
    auto p_tile = [&](int s) { return smem + C::OFF_P + s * C::P_ALIGNED; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * BM, n0 = blockIdx.y * BN;
    const int KB = a.K / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < SA; s++) { ptx::mbar_init(full_a(s), 1); ptx::mbar_init(empty_a(s), 1); }
        for (int s = 0; s < SP; s++) { ptx::mbar_init(full_p(s), 1); ptx::mbar_init(empty_p(s), kDeqWarps); }
        for (int s = 0; s < SB; s++) { ptx::mbar_init(full_b(s), kDeqWarps); ptx::mbar_init(empty_b(s), 1); }
        ptx::mbar_init(acc_full, 1);
        ptx::fence_mbar_init();
    }
    if (warp == kWarpMma) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), TMEM_COLS);
        ptx::tmem_relinquish();
    }
    if (warp == kWarpA && lane == 0) {
        ptx::prefetch_tensormap(&xmap);
        ptx::prefetch_tensormap(&wmap);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    if (warp == kWarpA) {
        // ------------------------------------------------ x tiles (TMA)
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            for (int kb = 0; kb < KB; kb++) {
                if (!ptx::mbar_wait(empty_a(s), ph ^ 1u)) { ok = false; break; }
                ptx::mbar_expect_tx(full_a(s), A_BYTES);
                ptx::tma_load_2d(a_tile(s), &xmap, kb * BK, m0, full_a(s));
                if (++s == SA) { s = 0; ph ^= 1u; }
            }
        }
    } else if (warp == kWarpP) {
        // ------------------------------------------------ packed weight tiles (TMA, PK K blocks each)
        if (lane == 0) {
            const int KP = (KB + PK - 1) / PK;
            int s = 0;
            uint32_t ph = 0;
            for (int kp = 0; kp < KP; kp++) {
                if (!ptx::mbar_wait(empty_p(s), ph ^ 1u)) { ok = false; break; }
                ptx::mbar_expect_tx(full_p(s), C::P_BYTES);
                ptx::tma_load_2d(ptx::smem_u32(p_tile(s)), &wmap, kp * (PK * BK * BITS / 8), n0, full_p(s));
                if (++s == SP) { s = 0; ph ^= 1u; }
            }
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------ MMA issuer (the whole warp runs the loop; one elected lane issues)
        constexpr uint32_t idesc = ptx::idesc_f16_f32(MH, BN);
        const uint64_t adesc0 = ptx::sw128_desc(a_tile(0)), bdesc0 = ptx::sw128_desc(b_tile(0));
        int sa = 0, sb = 0;
        uint32_t pa = 0, pb = 0;
        for (int kb = 0; kb < KB; kb++) {
            ok = __all_sync(0xffffffffu, ptx::mbar_wait(full_a(sa), pa) && ptx::mbar_wait(full_b(sb), pb));
            if (!ok) break;
            ptx::tc_fence_after();
            // descriptors advance by (byte offset >> 4) in their address field; tokens
            // [0, 128) into columns [0, 256), tokens [128, 256) into [256, 512): the fp16
            // weight tile is read by both
            const uint64_t ad = adesc0 + (uint64_t)((sa * A_BYTES) >> 4);
            const uint64_t bd = bdesc0 + (uint64_t)((sb * B_BYTES) >> 4);
#pragma unroll
            for (int kk = 0; kk < BK / 16; kk++) {
                ptx::mma_f16_elect(tmem, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
                ptx::mma_f16_elect(tmem + BN, ad + ((MH * 128) >> 4) + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
            }
            ptx::tc_commit_elect(empty_a(sa));
            ptx::tc_commit_elect(empty_b(sb));
            if (++sa == SA) { sa = 0; pa ^= 1u; }
            if (++sb == SB) { sb = 0; pb ^= 1u; }
        }
        ptx::tc_commit_elect(acc_full);
    } else {
        // ------------------------------------------------ dequantization (two threads per row)
        const uint32_t magic = a.magic;
        const int r = threadIdx.x >> 1;                 // 0..255
        const int hk = threadIdx.x & 1;                 // which 32 k of the block
        const int nr = n0 + r;
        const int n = min(nr, a.N - 1);
        const uint16_t* sp_row = a.scale + (size_t)n * a.ng;
        const uint8_t* zp_row = a.zp + (size_t)n * a.ng;
        constexpr int KB_PER_G = G / BK;                // 1 or 2
        const int ng = a.ng;
        // parameters of the current group and of the next two (loads in flight)
        uint32_t sc_cur = __ldg(sp_row), zq_cur = __ldg(zp_row);
        uint32_t sc_n1 = ng > 1 ? __ldg(sp_row + 1) : 0u, zq_n1 = ng > 1 ? __ldg(zp_row + 1) : 0u;
        uint32_t sc_n2 = ng > 2 ? __ldg(sp_row + 2) : 0u, zq_n2 = ng > 2 ? __ldg(zp_row + 2) : 0u;
        // outlier cursor of this row: the next entry (ocol, oval) and the one
        // after it (ncol, nval), so that consuming an entry never waits for a load
        int op = 0, oe = 0, ocol = 0x7FFFFFFF, ncol = 0x7FFFFFFF;
        uint16_t oval = 0, nval = 0;
        if (a.nnz > 0 && nr < a.N) {
            op = a.row_ptr[n];
            oe = a.row_ptr[n + 1];
            if (op < oe) {
                ocol = a.col[op];
                oval = a.val[op];
            }
            if (op + 1 < oe) {
                ncol = a.col[op + 1];
                nval = a.val[op + 1];
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
        unsigned char* const btile0 = smem + C::OFF_B;
        const int KP = (KB + PK - 1) / PK;
        int sp = 0, sb = 0;
        uint32_t pp = 0, pb = 1;   // parities: full_p to wait for, empty_b to wait for
        for (int kp = 0; kp < KP && ok; kp++) {
            const unsigned char* pt = p_tile(sp);
            if (!ptx::mbar_wait(full_p(sp), pp)) { ok = false; break; }
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
                if (!ptx::mbar_wait(empty_b(sb), pb)) { ok = false; break; }
                unsigned char* bt = btile0 + sb * B_BYTES;
                *reinterpret_cast<uint4*>(bt + dst_off[0]) = deq8_u4(w.x, add_lo, add_hi, s2, magic);
                *reinterpret_cast<uint4*>(bt + dst_off[1]) = deq8_u4(w.y, add_lo, add_hi, s2, magic);
                *reinterpret_cast<uint4*>(bt + dst_off[2]) = deq8_u4(w.z, add_lo, add_hi, s2, magic);
                *reinterpret_cast<uint4*>(bt + dst_off[3]) = deq8_u4(w.w, add_lo, add_hi, s2, magic);
                // FP16 outliers in this thread's 32 k: the dense value there is exactly 0
                const int k0 = kb * BK + 32 * hk;
                while (ocol < k0 + 32) {
                    if (ocol >= k0) {
                        const int kk = ocol - kb * BK;
                        *reinterpret_cast<uint16_t*>(bt + r * 128 + (((kk >> 3) ^ rsw) << 4) + (perm8_pos(kk) << 1)) = oval;
                    }
                    ocol = ncol;
                    oval = nval;
                    if (++op + 1 < oe) {
                        ncol = a.col[op + 1];
                        nval = a.val[op + 1];
                    } else {
                        ncol = 0x7FFFFFFF;
                    }
                }
                ptx::fence_proxy_async();
                __syncwarp();
                if (lane == 0) {
                    ptx::mbar_arrive(full_b(sb));
                    // the packed slot goes back to its producer only after the
                    // stores that consumed its codes: a shared load of the
                    // whole warp completes in several wavefronts, and a
                    // release right after issuing it let the next TMA tile
                    // overwrite rows that the later lanes had not read yet
                    if (sub == PK - 1 || kb == KB - 1) ptx::mbar_arrive(empty_p(sp));
                }
                if (++sb == SB) { sb = 0; pb ^= 1u; }
            }
            if (++sp == SP) { sp = 0; pp ^= 1u; }
        }
        // ------------------------------------------------ epilogue: TMEM -> y
        if (ok && ptx::mbar_wait(acc_full, 0)) {
            ptx::tc_fence_after();
            // warp w reads TMEM lanes 32 (w % 4) .. (the lanes a warp may
            // access) and a quarter of the 512 columns
            const int q = warp & 3, quarter = warp >> 2;
#pragma unroll 1
            for (int i = 0; i < 8; i++) {
                const int col = 128 * quarter + 16 * i;       // 0..511
                const int half = col / BN, cb = col % BN;
                const int m = m0 + MH * half + 32 * q + lane;
                uint32_t v[16];
                ptx::tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)col, v);
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
    if (!ok && a.status) atomicExch(a.status, (int)QG_ERR_TIMEOUT);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == kWarpMma) ptx::tmem_dealloc(tmem, TMEM_COLS);
}

// bf16 [M, ldx] -> fp16 [M, K] (exact for |x| in fp16's normal range), with
// the K positions of every block of 8 in the order (0,4,1,5,2,6,3,7) the
// weight operand uses.
__global__ void k_x_to_f16(const __nv_bfloat16* __restrict__ x, int M, int K, int ldx, __half* __restrict__ out)
{
    const long long total8 = (long long)M * K / 8;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total8;
         i += (long long)gridDim.x * blockDim.x) {
        const long long e = i * 8;
        const int m = (int)(e / K), k = (int)(e % K);
        const __nv_bfloat16* src = x + (size_t)m * ldx + k;
        constexpr int perm[8] = {0, 4, 1, 5, 2, 6, 3, 7};
        __half h[8];
#pragma unroll
        for (int j = 0; j < 8; j++) h[j] = __float2half_rn(__bfloat162float(src[perm[j]]));
        *reinterpret_cast<uint4*>(out + e) = *reinterpret_cast<const uint4*>(h);
    }
}

// Workspace: x converted to fp16 (K order permuted), M x K.
struct Ws {
    __half* x16;
};

size_t ws_layout(int M, int K, Ws* w, void* base)
{
    const size_t total = align_up((size_t)M * K * 2, 256);
    if (w && base) w->x16 = reinterpret_cast<__half*>(base);
    return total;
}

bool eligible(const qg_qweight& w) { return w.bits == 4 && (w.K % BK) == 0; }

template <int G>
qg_status run(const uint16_t* x, int M, int ldx, const qg_qweight& w, void* y, int ldy, qg_ydtype yt, void* ws,
              cudaStream_t s)
{
    using C = Cfg<4>;
    Ws p{};
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
                   (uint64_t)w.K / 2, PK * BK / 2, BN, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != QG_OK) return st;
    Args a;
    a.M = M; a.N = w.N; a.K = w.K; a.ng = w.K / G;
    a.scale = w.scale; a.zp = w.zp;
    a.row_ptr = w.out_row_ptr; a.col = w.out_col; a.val = w.out_val; a.nnz = w.nnz;
    a.y = y; a.ldy = ldy; a.y_bf16 = yt == QG_Y_BF16;
    a.status = device_status_ptr();
    a.magic = gemv::kF16Magic;
    {
        qg_status st2 = gemv::allow_smem(k_gemm_tc_u4<G>, C::SMEM);
        if (st2 != QG_OK) return st2;
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
