// Prefill-side fused dequantization product on the 5th-generation tensor
// cores (tcgen05 + TMEM), for M above the decode range, at every width:
//     y[m, n] = sum_k x[m, k] * (w_hat[n, k] + S[n, k])
//
// The pages' fused kernel dequantizes INT4 tiles into shared memory and runs
// the tensor cores on them ("70B on one GPU" page, section 3); this is
// that structure written for sm_103a and extended to the 2/3/5/6-bit widths
// of the "Mixed-width quantization" page (sections 2-3):
//  * one CTA computes a 256 x 256 tile of y (256 tokens x 256 weight rows)
//    as two fp32 accumulators of 128 tokens in tensor memory (all 512 TMEM
//    columns), so every dequantized weight tile feeds 256 tokens;
//  * warp 16 (one lane) streams the fp16 x tiles (TMA, 128-byte swizzle,
//    256 x 64) into a 2-deep ring; at 4 bits warp 17 streams the packed
//    weight tiles (TMA, 256 rows x 128 bytes = 4 K blocks, 128-byte swizzle)
//    into a 2-deep ring; at the other widths, whose K blocks are not 128-byte
//    multiples, each dequantization thread loads its own codes from global
//    memory (a register ring four K blocks deep);
//  * warps 0-15 (two threads per weight row, 32 k each) unpack the codes
//    into fp16 pairs -- masks into fp16 1024 + 2^p q and one packed FMA give
//    the exact integers q - zp (per-width pair plans, the decode kernel's),
//    one packed multiply applies the fp16 group scale (one rounding); 2-bit
//    codes look their fp16 codebook entries up with byte permutes -- patch
//    the FP16 outliers of the block in, and store the 256 x 64 fp16 tile in
//    the K-major 128-byte-swizzled layout the tensor core reads (K order
//    permuted inside every 32 as the pair plan orders the codes, matching
//    x) into a ring of 3 (4 bits) or 4 stages;
//  * warp 18 (one lane) issues eight tcgen05.mma (M=128, N=256, K=16) per K
//    block, four per accumulator, and commits them to the x and fp16
//    rings' "empty" barriers;
//  * warps 0-15 then read the accumulator with tcgen05.ld and store y.
// Rows whose largest scale times 2^bits - 1 exceeds fp16's range (groups
// near +-65504) are built at scale * 2^-e and their outputs multiplied by
// 2^e, so the operand never overflows.  Every mbarrier wait is bounded (a
// wait that gives up writes QG_ERR_TIMEOUT into the device status word read
// by qgemm_device_status; TMA loads or MMAs the CTA issued may then still be
// in flight when it exits, and that call's output is not valid).  x is first
// converted bf16 -> fp16 into the workspace (exact in fp16's range).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <utility>

#include "gemv_impl.cuh"
#include "ptx.cuh"
#include "tc_dequant.cuh"
#include "qg_internal.h"

namespace qg {

// Tiled 2-D tensor map (defined in gemm_tc.cu; the grouped kernel uses it too).
qg_status encode_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                    uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw);

namespace tc {

constexpr int BM = 256, BN = 256, BK = 64;
constexpr int MH = 128;                 // tokens per accumulator (one tcgen05.mma covers M = 128)
constexpr int SA = 2, SP = 2;           // ring depths: x tiles, packed tiles (4 bits)
constexpr int TMEM_COLS = 2 * BN;       // two fp32 accumulators of 128 x 256
constexpr int PK = 4;                   // K blocks per packed tile (128-byte rows at 4 bits)
constexpr int DG = 4;                   // K blocks of codes in flight per thread (other widths)
constexpr int kDeqWarps = 16;
constexpr int kWarpA = kDeqWarps, kWarpP = kDeqWarps + 1, kWarpMma = kDeqWarps + 2;
constexpr int kThreads = (kDeqWarps + 3) * 32;
// Split K applies to products of at most kSplitMaxM tokens (one token tile,
// whose grid of 256-row tiles is too small to fill the GPU); at most
// kMaxSplit CTAs share a tile, and at most kSplitSlabRows / M (the partial
// slabs of a split take S x M rows of workspace).
constexpr int kSplitMaxM = 256, kMaxSplit = 8, kSplitSlabRows = 1024;
constexpr int A_BYTES = BM * BK * 2;   // 32 KB fp16
constexpr int B_BYTES = BN * BK * 2;   // 32 KB fp16

// TILES: the codes and group parameters come from the tile-ordered copy
// (one contiguous block per 256 rows x 64 k, staged by one bulk copy).
template <int BITS, int G, bool TILES>
struct Cfg {
    static constexpr bool TMA_CODES = BITS == 4 && !TILES;
    static constexpr int SB = TILES || TMA_CODES ? 3 : 4;               // fp16 weight tiles
    static constexpr int BLOCK = (int)tile_block_bytes(BITS, G);         // one tile-ordered block
    static constexpr int P_BYTES = TMA_CODES ? BN * PK * BK * BITS / 8 : TILES ? BLOCK : 0;
    static constexpr int P_ALIGNED = TMA_CODES ? (P_BYTES + 1023) / 1024 * 1024 : (P_BYTES + 127) / 128 * 128;
    static constexpr int OFF_B = SA * A_BYTES;
    static constexpr int OFF_P = OFF_B + SB * B_BYTES;
    static constexpr int SP_FIT = TILES ? (227 * 1024 - 2048 - OFF_P) / P_ALIGNED : 0;
    static constexpr int SPN = TMA_CODES ? SP : TILES ? (SP_FIT < 6 ? SP_FIT : 6) : 1;   // packed ring depth
    static_assert(!TILES || SPN >= 2, "tile ring of at least two blocks");
    static constexpr int OFF_BAR = OFF_P + (TMA_CODES || TILES ? SPN : 0) * P_ALIGNED;
    static constexpr int OFF_EROW = OFF_BAR + 512;                      // per-row exponents (256 bytes)
    static constexpr int SMEM = OFF_BAR + 1024 /* barriers, exponents */ + 1024 /* alignment */;
};

struct Args {
    int M, N, K, ng;
    const uint8_t* packed;   // codes (read directly at widths other than 4)
    const uint8_t* tiles;    // tile-ordered copy (TILES kernels)
    const uint16_t* scale;
    const uint8_t* zp;
    const uint2* cb;         // 2-bit codebooks: 4 fp16 entries per group
    const int* row_ptr;
    const int* col;
    const uint16_t* val;
    int nnz;
    void* y;
    int ldy;
    int y_bf16;
    int* status;
    uint32_t magic;   // gemv::kF16Magic, a run-time value (one logic op per code pair)
    ScaleSrc sc;      // 8-bit scales when sc.scale8 is set (planar kernels; the tile copy holds fp16)
    // split K (gridDim.z > 1): CTA z takes K blocks [z * kbs, (z + 1) * kbs)
    // and writes its fp32 partial tile to part (z-th slab of M x ldp);
    // k_split_sum then adds the slabs in z order into y
    int kbs;
    float* part;
    int ldp;
    // bytes of one x tile load: the TMA box holds min(256, M rounded up to 8)
    // token rows, so that few tokens do not fill the tile with zeros (rows
    // past the box keep stale values; they feed only accumulator rows of
    // tokens >= M, which are never stored)
    uint32_t x_bytes;
};

static_assert(kDeqWarps * 32 == 512, "deq_sync counts 512 dequantization threads");

// y from the partial slabs of a split-K launch: every thread sums one float4
// column of one token over the S slabs in z order (fixed: the result is
// repeatable bit for bit) and stores it, fp32 or bf16, nothing at or past N.
static __global__ void __launch_bounds__(256) k_split_sum(const float* __restrict__ part, int S, int M, int N, int ldp,
                                                   void* __restrict__ y, int ldy, int y_bf16)
{
    gemv::pdl_release();
    gemv::pdl_wait();   // the slabs come from the kernel just before
    const int cols = (N + 3) / 4;
    const long long items = (long long)M * cols;
    const size_t zs = (size_t)M * ldp;
    for (long long it = (long long)blockIdx.x * blockDim.x + threadIdx.x; it < items;
         it += (long long)gridDim.x * blockDim.x) {
        const int m = (int)(it / cols), nb = 4 * (int)(it % cols);
        const float* pr = part + (size_t)m * ldp + nb;
        float4 t[kMaxSplit];
#pragma unroll
        for (int z = 0; z < kMaxSplit; z++)
            if (z < S) t[z] = __ldcg(reinterpret_cast<const float4*>(pr + z * zs));
        float v[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int z = 0; z < kMaxSplit; z++)
            if (z < S) {
                v[0] += t[z].x; v[1] += t[z].y; v[2] += t[z].z; v[3] += t[z].w;
            }
        if (y_bf16) {
            __nv_bfloat16* yr = reinterpret_cast<__nv_bfloat16*>(y) + (size_t)m * ldy;
#pragma unroll
            for (int j = 0; j < 4; j++)
                if (nb + j < N) yr[nb + j] = __float2bfloat16_rn(v[j]);
        } else {
            float* yr = reinterpret_cast<float*>(y) + (size_t)m * ldy;
            if (nb + 4 <= N && ((reinterpret_cast<uintptr_t>(yr + nb) & 15u) == 0)) {
                *reinterpret_cast<float4*>(yr + nb) = make_float4(v[0], v[1], v[2], v[3]);
            } else {
#pragma unroll
                for (int j = 0; j < 4; j++)
                    if (nb + j < N) yr[nb + j] = v[j];
            }
        }
    }
}

// 16 consecutive y values of token m from column nb (fp32 or bf16 per a.y_bf16;
// nothing at or past N).
__device__ __forceinline__ void store_y16(const Args& a, int m, int nb, const uint32_t (&v)[16])
{
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
                *reinterpret_cast<float4*>(yr + nb + j) = make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                                                                      __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]));
        } else {
#pragma unroll
            for (int j = 0; j < 16; j++)
                if (nb + j < a.N) yr[nb + j] = __uint_as_float(v[j]);
        }
    }
}

template <int BITS, int G, bool TILES, bool S8>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
              const __grid_constant__ Args a)
{
    using C = Cfg<BITS, G, TILES>;
    constexpr int SB = C::SB;
    constexpr int SP = C::SPN;
    extern __shared__ unsigned char smem_raw[];
    // 1024-byte aligned base, derived from the shared array by pointer arithmetic (an
    // integer round trip would leave the compiler a generic pointer)
    unsigned char* smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
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
    uint8_t* e_row = smem + C::OFF_EROW;
    auto a_tile = [&](int s) { return sbase + s * A_BYTES; };
    auto b_tile = [&](int s) { return sbase + C::OFF_B + s * B_BYTES; };
    auto p_tile = [&](int s) { return smem + C::OFF_P + s * C::P_ALIGNED; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * BM, n0 = blockIdx.y * BN;
    // this CTA's K blocks [kb0, kb1); kbs is a multiple of the packed tile's PK blocks
    const int kb0 = (int)blockIdx.z * a.kbs, kb1 = min(a.K / BK, kb0 + a.kbs);
    const int KB = kb1;   // loops run kb0 .. KB - 1
    // tokens m0 + 128 .. m0 + 255 exist: both accumulators; else only the first
    const bool two = a.M - m0 > MH;

    if (threadIdx.x == 0) {
        for (int s = 0; s < SA; s++) { ptx::mbar_init(full_a(s), 1); ptx::mbar_init(empty_a(s), 1); }
        if constexpr (C::TMA_CODES || TILES)
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
        if constexpr (C::TMA_CODES) ptx::prefetch_tensormap(&wmap);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;
    // programmatic dependent launch: the next kernel on the stream may start
    // once every CTA got here (it waits for this grid before touching what
    // this grid writes); x, y and the slabs are touched only after pdl_wait
    gemv::pdl_release();

    if (warp == kWarpA) {
        // ------------------------------------------------ x tiles (TMA)
        gemv::pdl_wait();   // x in fp16 comes from the kernel just before
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            for (int kb = kb0; kb < KB; kb++) {
                if (!ptx::mbar_wait(empty_a(s), ph ^ 1u)) { ok = false; break; }
                ptx::mbar_expect_tx(full_a(s), a.x_bytes);
                ptx::tma_load_2d(a_tile(s), &xmap, kb * BK, m0, full_a(s));
                if (++s == SA) { s = 0; ph ^= 1u; }
            }
        }
    } else if (warp == kWarpP) {
        // ------------------------------------------------ packed weight tiles (TMA, PK K blocks each; 4 bits)
        if constexpr (C::TMA_CODES) {
            if (lane == 0) {
                const int KP = (KB + PK - 1) / PK;
                int s = 0;
                uint32_t ph = 0;
                for (int kp = kb0 / PK; kp < KP; kp++) {
                    if (!ptx::mbar_wait(empty_p(s), ph ^ 1u)) { ok = false; break; }
                    ptx::mbar_expect_tx(full_p(s), C::P_BYTES);
                    ptx::tma_load_2d(ptx::smem_u32(p_tile(s)), &wmap, kp * (PK * BK * BITS / 8), n0, full_p(s));
                    if (++s == SP) { s = 0; ph ^= 1u; }
                }
            }
        } else if constexpr (TILES) {
            // one bulk copy per K block: the block of this CTA's 256-row tile
            if (lane == 0) {
                const uint8_t* base = a.tiles + (size_t)blockIdx.y * (a.K / BK) * C::BLOCK;
                int s = 0;
                uint32_t ph = 0;
                for (int kb = kb0; kb < KB; kb++) {
                    if (!ptx::mbar_wait(empty_p(s), ph ^ 1u)) { ok = false; break; }
                    ptx::mbar_expect_tx(full_p(s), C::BLOCK);
                    ptx::bulk_load(ptx::smem_u32(p_tile(s)), base + (size_t)kb * C::BLOCK, C::BLOCK, full_p(s));
                    if (++s == SP) { s = 0; ph ^= 1u; }
                }
            }
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------ MMA issuer (the whole warp runs the loop; one elected lane issues)
        constexpr uint32_t idesc = ptx::idesc_f16_f32(MH, BN);
        const uint64_t adesc0 = ptx::sw128_desc(a_tile(0)), bdesc0 = ptx::sw128_desc(b_tile(0));
        int sa = 0, sb = 0;
        uint32_t pa = 0, pb = 0;
        for (int kb = kb0; kb < KB; kb++) {
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
                const bool acc = ((kb - kb0) | kk) != 0;
                ptx::mma_f16_elect(tmem, ad + 2 * kk, bd + 2 * kk, idesc, acc);
                if (two) ptx::mma_f16_elect(tmem + BN, ad + ((MH * 128) >> 4) + 2 * kk, bd + 2 * kk, idesc, acc);
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
        const int ng = a.ng;
        // this thread's group in block kb: kb / KB_PER_G (groups of 64 and
        // 128 span one or two blocks), or 2 kb + hk at group 32 (each half of
        // a block is a group of its own); GSTEP apart from one block's to the next
        constexpr int KB_PER_G = G >= BK ? G / BK : 1;
        constexpr int GSTEP = G >= BK ? 1 : BK / G;
        const int g0 = G >= BK ? 0 : hk;
        // power-of-two headroom of this row (affine widths; codebook entries are fp16 already)
        int ex = 0;
        // 8-bit scales: the planar kernels convert each code where it is used
        // (the tile-ordered copy already holds fp16 scales); both find the
        // row exponent from the codes
        const bool has8 = a.sc.scale8 != nullptr;
        constexpr bool s8 = !TILES && S8;   // a compile-time choice: no branch in the loops without it
        const int E8 = has8 ? __ldg(a.sc.exp) : 0;
        if constexpr (BITS != 2) {
            if (has8) ex = row_exponent_8<BITS>(a.sc, E8, n, ng, hk);
            else ex = row_exponent<BITS>(a.scale + (size_t)n * ng, ng, hk);
        }
        if (hk == 0) e_row[r] = (uint8_t)ex;
        // group parameters of the current group and of the next two (loads in
        // flight: kept raw until the group is used, the row exponent applied
        // then): affine (scale bits, zero-point); codebook (two words of 4 fp16)
        const uint16_t* sp_row = a.scale + (size_t)n * ng;
        const uint8_t* s8_row = a.sc.scale8 + (size_t)n * ng;
        const uint8_t* zp_row = a.zp + (size_t)n * ng;
        const uint2* cb_row = a.cb + (size_t)n * ng;
        uint2 prm[3];
        auto load_prm = [&](int gi) -> uint2 {
            if constexpr (BITS == 2) return __ldg(cb_row + gi);
            else return make_uint2(s8 ? (uint32_t)__ldg(s8_row + gi) : (uint32_t)__ldg(sp_row + gi),
                                   (uint32_t)__ldg(zp_row + gi));
        };
        const int gs = g0 + (kb0 / KB_PER_G) * GSTEP;   // group of block kb0
        if constexpr (!TILES) {
            prm[0] = load_prm(gs);
            prm[1] = gs + GSTEP < ng ? load_prm(gs + GSTEP) : make_uint2(0u, 0u);
            prm[2] = gs + 2 * GSTEP < ng ? load_prm(gs + 2 * GSTEP) : make_uint2(0u, 0u);
        }
        // outlier cursor of this row: the next entry (ocol, oval) and the one
        // after it (ncol, nval), so that consuming an entry never waits for a load
        int op = 0, oe = 0, ocol = 0x7FFFFFFF, ncol = 0x7FFFFFFF;
        uint16_t oval = 0, nval = 0;
        if (a.nnz > 0 && nr < a.N) {
            op = a.row_ptr[n];
            oe = a.row_ptr[n + 1];
            if (kb0 > 0) {   // first entry at or after column kb0 * BK
                int hi = oe;
                while (op < hi) {
                    const int mid = (op + hi) >> 1;
                    if (a.col[mid] < kb0 * BK) op = mid + 1;
                    else hi = mid;
                }
            }
            if (op < oe) {
                ocol = a.col[op];
                oval = a.val[op];
            }
            if (op + 1 < oe) {
                ncol = a.col[op + 1];
                nval = a.val[op + 1];
            }
        }
        // swizzled destination chunks (4*hk + j) of the fp16 row, fixed per thread
        const uint32_t rsw = r & 7;
        uint32_t dst_off[4];
#pragma unroll
        for (int j = 0; j < 4; j++) dst_off[j] = r * 128 + (((4 * hk + j) ^ rsw) << 4);
        unsigned char* const btile0 = smem + C::OFF_B;

        // the fp16 ring: wait for a free slot (acquire), write the block's
        // operand, then finish (outliers patched in, handed to the MMA warp)
        int sb = 0;
        uint32_t pb = 1;   // parity of empty_b to wait for
        auto acquire = [&]() -> unsigned char* {
            return ptx::mbar_wait(empty_b(sb), pb) ? btile0 + sb * B_BYTES : nullptr;
        };
        auto finish = [&](int kb, unsigned char* bt) {
            // FP16 outliers in this thread's 32 k; the dense value there is
            // exactly 0 (affine), or the codebook entry nearest 0 (2 bits,
            // whose stored value is the residual)
            const int k0 = kb * BK + 32 * hk;
            while (ocol < k0 + 32) {
                if (ocol >= k0) {
                    const int pos = chunk_pos<BITS>(ocol - k0);
                    uint16_t* dst = reinterpret_cast<uint16_t*>(bt + r * 128 + (((4 * hk + (pos >> 3)) ^ rsw) << 4) + ((pos & 7) << 1));
                    if constexpr (BITS == 2) *dst = f16_add_sat(*dst, oval, 0);
                    else *dst = (uint16_t)f16_times_pow2(oval, ex);
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
            if (lane == 0) ptx::mbar_arrive(full_b(sb));
            if (++sb == SB) { sb = 0; pb ^= 1u; }
        };
        // the operand of block kb in registers (16 fp16 pairs) -> the ring;
        // false if the wait for a free slot gave up
        auto emit = [&](int kb, const uint32_t (&pr)[16]) -> bool {
            unsigned char* bt = acquire();
            if (!bt) return false;
#pragma unroll
            for (int j = 0; j < 4; j++)
                *reinterpret_cast<uint4*>(bt + dst_off[j]) = make_uint4(pr[4 * j], pr[4 * j + 1], pr[4 * j + 2], pr[4 * j + 3]);
            finish(kb, bt);
            return true;
        };
        // next group: shift the parameter window
        int gcur = gs;   // group of prm[0]
        auto next_group = [&](int kb) {
            if (kb > kb0 && kb % KB_PER_G == 0) {
                const int gi = g0 + (kb / KB_PER_G) * GSTEP;
                gcur = gi;
                prm[0] = prm[1];
                prm[1] = prm[2];
                if (gi + 2 * GSTEP < ng) prm[2] = load_prm(gi + 2 * GSTEP);
            }
        };
        // fp16 scale bits of the current group (an 8-bit code converted here,
        // where it is used, so that its load stays in flight until then)
        auto cur_scale = [&]() -> uint32_t { return s8 ? scale8_bits(a.sc, E8, n, gcur, prm[0].x) : prm[0].x; };

        if constexpr (TILES) {
            // codes and parameters of block kb from the tile ring: word i of
            // this thread's chunk at word i * 512 + threadIdx.x, the row's
            // parameters after the 512 * BITS code words (NPG sets per row:
            // at group 32 this thread's half of the block has its own)
            constexpr int NPG = tile_groups_per_block(G);
            int sp = 0;
            uint32_t pp = 0;   // parity of full_p to wait for
            for (int kb = kb0; kb < KB && ok; kb++) {
                if (!ptx::mbar_wait(full_p(sp), pp)) { ok = false; break; }
                const uint32_t* pw = reinterpret_cast<const uint32_t*>(p_tile(sp));
                uint32_t w[BITS];
#pragma unroll
                for (int i = 0; i < BITS; i++) w[i] = pw[i * 512 + threadIdx.x];
                uint32_t pr[16];
                if constexpr (BITS == 2) {
                    const uint2 c = reinterpret_cast<const uint2*>(pw + BITS * 512)[r * NPG + (NPG == 2 ? hk : 0)];
                    const uint32_t lo = __byte_perm(c.x, c.y, 0x6420), hi = __byte_perm(c.x, c.y, 0x7531);
#pragma unroll
                    for (int wi = 0; wi < 2; wi++)
#pragma unroll
                        for (int jf = 0; jf < 4; jf++) {
                            const uint32_t f = (w[wi] >> (2 * jf)) & 0x03030303u;
                            pr[2 * (4 * wi + jf)] = cb_pair<0>(f, lo, hi);
                            pr[2 * (4 * wi + jf) + 1] = cb_pair<1>(f, lo, hi);
                        }
                } else {
                    const uint32_t pq = pw[BITS * 512 + r * NPG + (NPG == 2 ? hk : 0)];
                    const uint32_t s2 = __byte_perm(f16_times_pow2(pq & 0xFFFFu, ex), 0u, 0x1010u);
                    const uint32_t zq = pq >> 16;
                    gemv::static_for<0, 16>([&](auto ec) {
                        constexpr int e = decltype(ec)::value;
                        pr[e] = hmul2_u32(gemv::deq_affine<BITS, 32, e>(w, zq, magic), s2);
                    });
                }
                if (!emit(kb, pr)) { ok = false; break; }
                // the block goes back to its producer after the shared loads
                // that read it completed (emit synchronized the warp)
                if (lane == 0) ptx::mbar_arrive(empty_p(sp));
                if (++sp == SP) { sp = 0; pp ^= 1u; }
            }
        } else if constexpr (C::TMA_CODES) {
            // 4 bits: codes come from the TMA ring (source chunk 2*sub + hk of the packed row)
            uint32_t src_off[PK];
#pragma unroll
            for (int sub = 0; sub < PK; sub++) src_off[sub] = r * 128 + (((2 * sub + hk) ^ rsw) << 4);
            const int KP = (KB + PK - 1) / PK;
            int sp = 0;
            uint32_t pp = 0;   // parity of full_p to wait for
            for (int kp = kb0 / PK; kp < KP && ok; kp++) {
                const unsigned char* pt = p_tile(sp);
                if (!ptx::mbar_wait(full_p(sp), pp)) { ok = false; break; }
#pragma unroll
                for (int sub = 0; sub < PK; sub++) {
                    const int kb = kp * PK + sub;
                    if (kb >= KB) break;
                    next_group(kb);
                    const uint32_t zq = prm[0].y;
                    const uint32_t add_lo = zq * 0x00010001u + 0xE400E400u;   // -(1024 + zp)
                    const uint32_t add_hi = zq * 0x00100010u + 0xD400D400u;   // -(64 + zp)
                    const uint32_t s2 = __byte_perm(f16_times_pow2(cur_scale(), ex), 0u, 0x1010u);
                    const uint4 w = *reinterpret_cast<const uint4*>(pt + src_off[sub]);
                    unsigned char* bt = acquire();
                    if (!bt) { ok = false; break; }
                    *reinterpret_cast<uint4*>(bt + dst_off[0]) = deq8_u4(w.x, add_lo, add_hi, s2, magic);
                    *reinterpret_cast<uint4*>(bt + dst_off[1]) = deq8_u4(w.y, add_lo, add_hi, s2, magic);
                    *reinterpret_cast<uint4*>(bt + dst_off[2]) = deq8_u4(w.z, add_lo, add_hi, s2, magic);
                    *reinterpret_cast<uint4*>(bt + dst_off[3]) = deq8_u4(w.w, add_lo, add_hi, s2, magic);
                    finish(kb, bt);
                    // the packed slot goes back to its producer only after the
                    // stores that consumed its codes (emit synchronized the warp):
                    // a shared load of the whole warp completes in several
                    // wavefronts, and a release right after issuing it let the
                    // next TMA tile overwrite rows that later lanes had not read
                    if (lane == 0 && (sub == PK - 1 || kb == KB - 1)) ptx::mbar_arrive(empty_p(sp));
                }
                if (++sp == SP) { sp = 0; pp ^= 1u; }
            }
        } else {
            // other widths: each thread's 32-code chunk of block kb is 4*BITS
            // bytes at byte (2*kb + hk) * 4*BITS of the row, loaded DG blocks ahead
            using Ch = gemv::Chunk<BITS, 128>;
            constexpr int NW = Ch::NW;
            const uint8_t* prow = a.packed + (size_t)n * ((size_t)a.K * BITS / 8) + hk * 4 * BITS;
            const bool odd = Ch::SPLIT && hk;   // the chunk starts 4 bytes past an 8-byte boundary
            uint32_t wr[DG][NW];
            gemv::static_for<0, DG>([&](auto dc) {
                constexpr int d = decltype(dc)::value;
                if (kb0 + d < KB) Ch::load(prow + (kb0 + d) * 8 * BITS, wr[d]);
            });
            for (int kbd = kb0; kbd < KB && ok; kbd += DG) {
                gemv::static_for<0, DG>([&](auto dc) {
                    constexpr int d = decltype(dc)::value;
                    const int kb = kbd + d;
                    if (ok && kb < KB) {
                        next_group(kb);
                        uint32_t w[NW];
                        if constexpr (Ch::SPLIT) Ch::order(wr[d], w, odd);
                        else {
#pragma unroll
                            for (int i = 0; i < NW; i++) w[i] = wr[d][i];
                        }
                        uint32_t pr[16];
                        if constexpr (BITS == 2) {
                            const uint32_t lo = __byte_perm(prm[0].x, prm[0].y, 0x6420);
                            const uint32_t hi = __byte_perm(prm[0].x, prm[0].y, 0x7531);
                            gemv::static_for<0, NW>([&](auto wc) {
                                constexpr int wi = decltype(wc)::value;
#pragma unroll
                                for (int jf = 0; jf < 4; jf++) {
                                    const uint32_t f = (w[wi] >> (2 * jf)) & 0x03030303u;
                                    pr[2 * (4 * wi + jf)] = cb_pair<0>(f, lo, hi);
                                    pr[2 * (4 * wi + jf) + 1] = cb_pair<1>(f, lo, hi);
                                }
                            });
                        } else {
                            const uint32_t s2 = __byte_perm(f16_times_pow2(cur_scale(), ex), 0u, 0x1010u);
                            const uint32_t zq = prm[0].y;
                            gemv::static_for<0, 16>([&](auto ec) {
                                constexpr int e = decltype(ec)::value;
                                pr[e] = hmul2_u32(gemv::deq_affine<BITS, 32, e>(w, zq, magic), s2);
                            });
                        }
                        if (kb + DG < KB) Ch::load(prow + (kb + DG) * 8 * BITS, wr[d]);
                        if (!emit(kb, pr)) ok = false;
                    }
                });
            }
        }
        // ------------------------------------------------ epilogue: TMEM -> y
        gemv::pdl_wait();   // (long done: the x tiles came after it) before y and the slabs are written
        deq_sync();   // every row's exponent is in shared memory
        if (ok && ptx::mbar_wait(acc_full, 0)) {
            ptx::tc_fence_after();
            // warp w reads TMEM lanes 32 (w % 4) .. (the lanes a warp may
            // access) and a quarter of the 512 columns, or, with tokens in the
            // first accumulator only, an eighth: its 256 columns over all 16
            // warps.  Two 16-column loads are in flight per wait.
            const int q = warp & 3, quarter = warp >> 2;
            const bool split = gridDim.z > 1;
            const int span = two ? 128 : 64;   // columns per warp
#pragma unroll 1
            for (int i = 0; i < span / 16; i += 2) {
                uint32_t v[2][16];
                const int col0 = span * quarter + 16 * i;   // 0..511
                ptx::tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)col0, v[0]);
                ptx::tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(col0 + 16), v[1]);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int u = 0; u < 2; u++) {
                    const int col = col0 + 16 * u;
                    const int half = col / BN, cb = col % BN;
                    const int m = m0 + MH * half + 32 * q + lane;
                    // rows built at scale * 2^-e: multiply back by 2^e (exact)
                    const uint4 ew = *reinterpret_cast<const uint4*>(e_row + cb);
                    if (ew.x | ew.y | ew.z | ew.w) {
                        const uint32_t ewa[4] = {ew.x, ew.y, ew.z, ew.w};
#pragma unroll
                        for (int j = 0; j < 16; j++) {
                            const int ej = (ewa[j >> 2] >> (8 * (j & 3))) & 0xFF;
                            v[u][j] = __float_as_uint(__uint_as_float(v[u][j]) * __int_as_float((127 + ej) << 23));
                        }
                    }
                    if (m < a.M) {
                        if (split) {   // the partial tile to this CTA's slab (ldp covers whole tiles)
                            float* pr = a.part + ((size_t)blockIdx.z * a.M + m) * a.ldp + n0 + cb;
#pragma unroll
                            for (int j = 0; j < 16; j += 4)
                                __stcg(reinterpret_cast<float4*>(pr + j),
                                       make_float4(__uint_as_float(v[u][j]), __uint_as_float(v[u][j + 1]),
                                                   __uint_as_float(v[u][j + 2]), __uint_as_float(v[u][j + 3])));
                        } else {
                            store_y16(a, m, n0 + cb, v[u]);
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

// Whether the width's operand order is the same permutation inside every
// block of 8 k positions (as at 4 and 8 bits): then a thread converts 8
// values with the entries of the first block.
template <int BITS>
constexpr bool perm_within_8()
{
    for (int e = 0; e < 16; e++) {
        const gemv::PairE q = gemv::plan_entry(BITS, 32, e), q0 = gemv::plan_entry(BITS, 32, e % 4);
        if (q0.lo >= 8 || q0.hi >= 8 || q.lo != q0.lo + 8 * (e / 4) || q.hi != q0.hi + 8 * (e / 4)) return false;
    }
    return true;
}

// bf16 [M, ldx] -> fp16 [M, K] (exact for |x| in fp16's range), with the K
// positions of every block of 32 in the order the weight operand uses: the
// pair plan of the width puts codes lo and hi of entry e at 2e and 2e + 1.
// A thread converts a block of 8 (when the order keeps blocks of 8 in place,
// as at 4 bits) or of 32.
template <int BITS>
__global__ void k_x_to_f16(const __nv_bfloat16* __restrict__ x, int M, int K, int ldx, __half* __restrict__ out)
{
    gemv::pdl_release();
    gemv::pdl_wait();   // x may come from the kernel just before; out may still be read by it
    constexpr int R = perm_within_8<BITS>() ? 8 : 32;
    const long long total = (long long)M * K / R;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const long long e = i * R;
        const int m = (int)(e / K), k = (int)(e % K);
        const __nv_bfloat16* src = x + (size_t)m * ldx + k;
        uint32_t v[R / 2];   // the R bf16 values, two per word
        if ((reinterpret_cast<uintptr_t>(src) & 15u) == 0) {
#pragma unroll
            for (int j = 0; j < R / 8; j++) {
                const uint4 q = __ldg(reinterpret_cast<const uint4*>(src) + j);
                v[4 * j] = q.x; v[4 * j + 1] = q.y; v[4 * j + 2] = q.z; v[4 * j + 3] = q.w;
            }
        } else {
            const unsigned short* s16 = reinterpret_cast<const unsigned short*>(src);
#pragma unroll
            for (int j = 0; j < R / 2; j++) v[j] = (uint32_t)__ldg(s16 + 2 * j) | ((uint32_t)__ldg(s16 + 2 * j + 1) << 16);
        }
        auto f16 = [&](int c) -> uint32_t {   // bf16 -> fp32 (exact) -> fp16
            const uint32_t b = (c & 1) ? (v[c >> 1] & 0xFFFF0000u) : (v[c >> 1] << 16);
            return __half_as_ushort(__float2half_rn(__uint_as_float(b)));
        };
        uint32_t o[R / 2];
        gemv::static_for<0, R / 2>([&](auto ec) {
            constexpr int pe = decltype(ec)::value;   // pair entry within this thread's block
            constexpr gemv::PairE q = gemv::plan_entry(BITS, 32, pe);
            o[pe] = f16(q.lo) | (f16(q.hi) << 16);
        });
        uint4* dst = reinterpret_cast<uint4*>(out + e);
#pragma unroll
        for (int j = 0; j < R / 8; j++) dst[j] = make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
    }
}

// Workspace: x converted to fp16 (K order permuted), M x K; for small M also
// the partial slabs (S_max x M x ldp fp32).
struct Ws {
    __half* x16;
    float* part;
    int ldp;
};

inline size_t ws_layout(int M, int N, int K, Ws* w, void* base)
{
    const size_t x16 = align_up((size_t)M * K * 2, 256);
    size_t total = x16, o_part = 0;
    const int ldp = (int)ceil_div(N, BN) * BN;
    if (M <= kSplitMaxM) {
        o_part = total;
        total += align_up((size_t)std::min(kMaxSplit, kSplitSlabRows / M) * M * ldp * 4, 256);
    }
    if (w && base) {
        char* b = static_cast<char*>(base);
        w->x16 = reinterpret_cast<__half*>(b);
        w->part = M <= kSplitMaxM ? reinterpret_cast<float*>(b + o_part) : nullptr;
        w->ldp = ldp;
    }
    return total;
}

// K splits of a launch: none above kSplitMaxM tokens; else the count (at
// most min(kMaxSplit, kSplitSlabRows / M), at least 8 K blocks each, a whole
// number of packed tiles)
// whose waves of one-CTA-per-SM grids end soonest.  Returns the split count
// and sets *kbs to the K blocks per split.
inline int choose_ksplit(int M, int tiles, int KB, int* kbs)
{
    *kbs = KB;
    if (M > kSplitMaxM || KB < 16) return 1;
    const int sms = num_sms();
    int best = 1;
    long long best_cost = ceil_div(tiles, sms) * (long long)KB;
    for (int s = 2; s <= std::min(kMaxSplit, kSplitSlabRows / M); s++) {
        const int k = (int)(ceil_div(ceil_div(KB, s), PK) * PK);
        if (k < 8) break;
        const int se = (int)ceil_div(KB, k);
        const long long cost = ceil_div((long long)tiles * se, sms) * (long long)k;
        if (cost < best_cost) {
            best_cost = cost;
            best = se;
            *kbs = k;
        }
    }
    return best;
}

// Launch with programmatic stream serialization when dependent launch is on
// (every kernel launched this way releases its dependents and waits for the
// kernel before it on its own).
template <typename... KArgs, typename... Act>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, int threads, size_t smem, cudaStream_t s,
                              Act&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3((unsigned)threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = dependent_launch_enabled() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Act>(args)...);
}

// One product.  convert_x = false: x is already in the workspace in fp16 (a
// fused call's later products, which share the first one's conversion).
template <int BITS, int G, bool TILES, bool S8>
qg_status run(const uint16_t* x, int M, int ldx, const qg_qweight& w, const void* tiles, void* y, int ldy,
              qg_ydtype yt, void* ws, bool convert_x, cudaStream_t s)
{
    using C = Cfg<BITS, G, TILES>;
    Ws p{};
    ws_layout(M, w.N, w.K, &p, ws);
    if (convert_x) {
        const long long total32 = (long long)M * w.K / 32;
        const int blocks = (int)std::min<long long>(ceil_div(total32, 256), (long long)num_sms() * 8);
        const cudaError_t e = launch_pdl(k_x_to_f16<BITS>, dim3((unsigned)blocks), 256, 0, s,
                                         reinterpret_cast<const __nv_bfloat16*>(x), M, w.K, ldx, p.x16);
        if (e != cudaSuccess) return cuda_fail(e, "x conversion launch");
    }
    CUtensorMap xmap, wmap;
    const int x_rows = std::min(BM, (M + 7) & ~7);   // a whole number of 8-row swizzle atoms
    qg_status st = encode_2d(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, p.x16, (uint64_t)w.K, (uint64_t)M,
                             (uint64_t)w.K * 2, BK, (uint32_t)x_rows, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != QG_OK) return st;
    if constexpr (C::TMA_CODES) {
        st = encode_2d(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, w.packed, (uint64_t)w.K * BITS / 8, (uint64_t)w.N,
                       (uint64_t)w.K * BITS / 8, PK * BK * BITS / 8, BN, CU_TENSOR_MAP_SWIZZLE_128B);
        if (st != QG_OK) return st;
    } else {
        wmap = xmap;   // unused: the codes are read directly
    }
    Args a;
    a.M = M; a.N = w.N; a.K = w.K; a.ng = w.K / G;
    a.packed = w.packed;
    a.tiles = static_cast<const uint8_t*>(tiles);
    a.scale = w.scale; a.zp = w.zp; a.cb = reinterpret_cast<const uint2*>(w.codebook);
    a.row_ptr = w.out_row_ptr; a.col = w.out_col; a.val = w.out_val; a.nnz = w.nnz;
    a.y = y; a.ldy = ldy; a.y_bf16 = yt == QG_Y_BF16;
    a.status = device_status_ptr();
    a.magic = gemv::kF16Magic;
    a.sc = scale_src(w);
    a.x_bytes = (uint32_t)x_rows * BK * 2;
    {
        qg_status st2 = gemv::allow_smem(k_gemm_tc<BITS, G, TILES, S8>, C::SMEM);
        if (st2 != QG_OK) return st2;
    }
    const int tm = (int)ceil_div(M, BM), tn = (int)ceil_div(w.N, BN);
    const int splits = choose_ksplit(M, tm * tn, w.K / BK, &a.kbs);
    a.part = p.part;
    a.ldp = p.ldp;
    dim3 grid((unsigned)tm, (unsigned)tn, (unsigned)splits);
    cudaError_t e = launch_pdl(k_gemm_tc<BITS, G, TILES, S8>, grid, kThreads, C::SMEM, s, xmap, wmap, a);
    if (e != cudaSuccess) return cuda_fail(e, "tensor-core kernel launch");
    if (splits > 1) {
        const long long items = (long long)M * ceil_div(w.N, 4);
        const int blocks = (int)std::min<long long>(ceil_div(items, 256), 4LL * num_sms());
        e = launch_pdl(k_split_sum, dim3((unsigned)blocks), 256, 0, s, (const float*)p.part, splits, M, w.N, p.ldp, y,
                       ldy, (int)(yt == QG_Y_BF16));
        if (e != cudaSuccess) return cuda_fail(e, "split-K sum launch");
    }
    return QG_OK;
}

template <int BITS, bool TILES>
qg_status run_bits(const uint16_t* x, int M, int ldx, const qg_qweight& w, const void* tiles, void* y, int ldy,
                   qg_ydtype yt, void* ws, bool convert_x, cudaStream_t s)
{
    // planar kernels with 8-bit scales convert them as they use them (their own
    // instantiation); the tile-ordered copy always holds fp16 scales
    if (!TILES && w.scale8)
        return w.group == 32   ? run<BITS, 32, TILES, !TILES>(x, M, ldx, w, tiles, y, ldy, yt, ws, convert_x, s)
               : w.group == 64 ? run<BITS, 64, TILES, !TILES>(x, M, ldx, w, tiles, y, ldy, yt, ws, convert_x, s)
                               : run<BITS, 128, TILES, !TILES>(x, M, ldx, w, tiles, y, ldy, yt, ws, convert_x, s);
    return w.group == 32   ? run<BITS, 32, TILES, false>(x, M, ldx, w, tiles, y, ldy, yt, ws, convert_x, s)
           : w.group == 64 ? run<BITS, 64, TILES, false>(x, M, ldx, w, tiles, y, ldy, yt, ws, convert_x, s)
                           : run<BITS, 128, TILES, false>(x, M, ldx, w, tiles, y, ldy, yt, ws, convert_x, s);
}

}  // namespace tc

}  // namespace qg
