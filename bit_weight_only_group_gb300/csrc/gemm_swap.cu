// Grouped (MoE) fused dequantization product on the 5th-generation tensor
// cores with the roles of the operands swapped: the dequantized weights are
// the MMA's M side (128 weight rows per CTA) and an expert's tokens are the N
// side (N = 16 * ceil(tokens / 16), at most one routing chunk of 64), so an
// expert that receives a few dozen tokens costs no padding on the tensor
// core; an expert with more tokens has several chunks, whose CTAs read the
// same weight tiles at about the same time (HBM once, L2 after).
//     y[pair, n] = sum_k x[token(pair), k] * (w_hat_e[n, k] + S_e[n, k])
//
// Routing (a stable counting sort of the (token, slot) pairs by expert,
// "On-device MoE" page, sections 1-2) is done by the routing kernel;
// k_gather_x16 then writes x in that order as fp16 with the K positions of
// every block of 8 permuted (0,4,1,5,2,6,3,7) like the weight operand, and
// one CTA of k_gemm_swap_u4 computes a 128-row x (up to 64)-token tile:
//  * warp 16 (one lane) streams the token tile (TMA, 16-row boxes, 128-byte
//    swizzle) into a ring of up to 16 stages (as many as the token count
//    allows), warp 17 the packed 4-bit weight tile of the expert (TMA, 128
//    rows x 128 bytes = 4 K blocks) into a 3-deep ring;
//  * warps 0-15, in two groups taking alternate K blocks (two threads per
//    weight row), dequantize as the prefill kernel does (masks -> fp16
//    1024 + 2^p q, one packed FMA -> q - zp, one packed multiply by the fp16
//    scale, FP16 outliers patched in) into a 6-deep ring of 128 x 64 fp16
//    tiles;
//  * warps 18 and 19, one per dequantization group, each issue four
//    tcgen05.mma (M=128, N=tokens, K=16) per K block of their parity from one
//    elected lane into their own TMEM accumulator of 128 lanes x 128 columns;
//  * warps 0-15 add the two accumulators (lane = weight row, column = token)
//    and store y rows in pair order.
// One launch may cover several products over the same routing (an MoE
// layer's gate and up): blockIdx.x runs over every product's row tiles.
// Rows whose largest scale times 15 exceeds fp16's range are built at
// scale * 2^-e and their outputs multiplied by 2^e (see row_exponent).
// Every mbarrier wait is bounded; a wait that gives up writes QG_ERR_TIMEOUT
// into the device status word (TMA loads or MMAs the CTA issued may then
// still be in flight when it exits, and that call's output is not valid).
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
constexpr int NBMAX = 128;     // tokens per CTA (MMA N, a multiple of 16)
constexpr int BK = 64;         // K block (one 128-byte fp16 row of an operand tile)
constexpr int PK = 4;          // K blocks per packed tile (128-byte rows at 4 bits)
constexpr int SXMAX = 16, SP = 3, SA = 6;   // token ring: up to 16 stages in X_RING bytes
// Two groups of 8 dequantization warps take alternate K blocks (group g the
// blocks 4p + g and 4p + g + 2 of packed tile p, both at once: eight
// independent unpack chains per thread and one proxy fence per tile), so the
// per-block latencies overlap; group g writes the fp16 slots of parity g and
// holds up to three of them ahead of the MMA.
constexpr int kGroups = 2, kGroupWarps = 8;
constexpr int kDeqWarps = kGroups * kGroupWarps;
static_assert(SA % kGroups == 0, "a group's K blocks map to its own fp16 slots");
// one MMA issuer warp per group (K blocks of parity g into accumulator g)
constexpr int kWarpX = kDeqWarps, kWarpP = kDeqWarps + 1, kWarpMma = kDeqWarps + 2;
constexpr int kThreads = (kDeqWarps + 2 + kGroups) * 32;
constexpr int X_RING = 80 * 1024;           // split into stages of NB x 64 fp16
constexpr int P_BYTES = BW * PK * BK / 2;    // 16 KB
constexpr int A_BYTES = BW * BK * 2;         // 16 KB
constexpr int OFF_P = X_RING;
constexpr int OFF_A = OFF_P + SP * P_BYTES;
constexpr int OFF_BAR = OFF_A + SA * A_BYTES;
constexpr int OFF_EROW = OFF_BAR + 512;     // per-row exponents (128 bytes)
constexpr int SMEM = OFF_BAR + 1024 /* barriers, exponents */ + 1024 /* alignment */;
constexpr int TMEM_COLS = kGroups * NBMAX;   // one accumulator per group
constexpr int kMaxExperts = 32;              // tensor maps travel as kernel parameters (all products' experts)
constexpr int kMaxProducts = 2;              // products sharing the routing in one launch (gate and up)

struct Maps {
    CUtensorMap w[kMaxExperts];   // packed codes of each expert, box 128 bytes x 128 rows
};

struct Args {
    int N, K, ng, chunk;
    int E, tiles;         // experts per product, row tiles per product
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
    void* y[kMaxProducts];   // per product: [pairs, N]
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
    // blockIdx.x: row tile of product blockIdx.x / tiles; ep indexes that product's expert e
    const int prod = (int)blockIdx.x / a.tiles;
    const int ep = prod * a.E + e;
    const int m0 = a.offsets[e] + item.y * a.chunk;
    const int ntok = min(a.chunk, a.offsets[e + 1] - m0);
    const int NB = (ntok + 15) & ~15;   // MMA N: tokens rounded up to 16
    const int n0 = ((int)blockIdx.x % a.tiles) * BW;
    const int KB = a.K / BK;

    extern __shared__ unsigned char smem_raw[];
    // 1024-byte aligned base, derived from the shared array by pointer arithmetic (an
    // integer round trip would leave the compiler a generic pointer)
    unsigned char* smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = ptx::smem_u32(smem);
    const uint32_t bars = sbase + OFF_BAR;
    // token ring: stages of NB rows x 128 bytes (a multiple of 2 KB, so every
    // stage starts on a 1024-byte boundary), as many as fit X_RING (at most
    // SXMAX): small experts get a deep ring that covers the L2 latency
    const int x_stage = NB * BK * 2;
    const int SX = min(SXMAX, X_RING / x_stage) & ~(kGroups - 1);   // even: slot parity = block parity
    auto full_x = [&](int s) { return bars + 8 * s; };
    auto empty_x = [&](int s) { return bars + 8 * (SXMAX + s); };
    auto full_p = [&](int s) { return bars + 8 * (2 * SXMAX + s); };
    auto empty_p = [&](int s) { return bars + 8 * (2 * SXMAX + SP + s); };
    auto full_a = [&](int s) { return bars + 8 * (2 * SXMAX + 2 * SP + s); };
    auto empty_a = [&](int s) { return bars + 8 * (2 * SXMAX + 2 * SP + SA + s); };
    const uint32_t acc_full = bars + 8 * (2 * SXMAX + 2 * SP + 2 * SA);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_BAR + 8 * (2 * SXMAX + 2 * SP + 2 * SA + 1));
    uint8_t* e_row = smem + OFF_EROW;
    auto x_tile = [&](int s) { return sbase + s * x_stage; };
    auto p_tile = [&](int s) { return smem + OFF_P + s * P_BYTES; };
    auto a_tile = [&](int s) { return sbase + OFF_A + s * A_BYTES; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < SX; s++) { ptx::mbar_init(full_x(s), 1); ptx::mbar_init(empty_x(s), 1); }
        for (int s = 0; s < SP; s++) { ptx::mbar_init(full_p(s), 1); ptx::mbar_init(empty_p(s), kDeqWarps); }
        for (int s = 0; s < SA; s++) { ptx::mbar_init(full_a(s), kGroupWarps); ptx::mbar_init(empty_a(s), 1); }
        ptx::mbar_init(acc_full, kGroups);
        ptx::fence_mbar_init();
    }
    if (warp == kWarpMma) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), TMEM_COLS);
        ptx::tmem_relinquish();
    }
    if (warp == kWarpX && lane == 0) {
        ptx::prefetch_tensormap(&xmap);
        ptx::prefetch_tensormap(&maps.w[ep]);
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
                ptx::tma_load_2d(ptx::smem_u32(p_tile(s)), &maps.w[ep], kp * (PK * BK / 2), n0, full_p(s));
                if (++s == SP) { s = 0; ph ^= 1u; }
            }
        }
    } else if (warp >= kWarpMma) {
        // ------------------------------------------------ MMA issuers: D_g[w rows, tokens] += W * X^T over
        // the K blocks of parity g (the whole warp runs the loop; one elected lane issues)
        const int g = warp - kWarpMma;
        const uint32_t acc = tmem + (uint32_t)(g * NBMAX);
        const uint32_t idesc = ptx::idesc_f16_f32(BW, NB);
        const uint64_t adesc0 = ptx::sw128_desc(a_tile(0)), xdesc0 = ptx::sw128_desc(x_tile(0));
        // ring slots and phases of block kb, advanced by kGroups blocks per
        // iteration (SX and SA are even, so a slot keeps its block parity)
        int sx = g, sa = g;
        uint32_t px = 0, pa = 0;
        for (int kb = g; kb < KB; kb += kGroups) {
            ok = __all_sync(0xffffffffu, ptx::mbar_wait(full_x(sx), px) && ptx::mbar_wait(full_a(sa), pa));
            if (!ok) break;
            ptx::tc_fence_after();
            // descriptors advance by (byte offset >> 4) in their address field
            const uint64_t ad = adesc0 + (uint64_t)((sa * A_BYTES) >> 4);
            const uint64_t xd = xdesc0 + (uint64_t)((sx * x_stage) >> 4);
#pragma unroll
            for (int kk = 0; kk < BK / 16; kk++)
                ptx::mma_f16_elect(acc, ad + 2 * kk, xd + 2 * kk, idesc, (kb >= kGroups || kk > 0) ? 1u : 0u);
            ptx::tc_commit_elect(empty_x(sx));
            ptx::tc_commit_elect(empty_a(sa));
            if ((sx += kGroups) >= SX) { sx -= SX; px ^= 1u; }
            if ((sa += kGroups) >= SA) { sa -= SA; pa ^= 1u; }
        }
        ptx::tc_commit_elect(acc_full);
    } else {
        // ------------------------------------------------ dequantization (two threads per weight row)
        const uint32_t magic = a.magic;
        const int grp = threadIdx.x / (kGroupWarps * 32);   // K blocks kb with kb % kGroups == grp
        const int tg = threadIdx.x % (kGroupWarps * 32);
        const int r = tg >> 1;                          // 0..127
        const int hk = tg & 1;                          // which 32 k of the block
        const int nr = n0 + r;
        const int n = min(nr, a.N - 1);
        const uint16_t* sp_row = a.scale[ep] + (size_t)n * a.ng;
        const uint8_t* zp_row = a.zp[ep] + (size_t)n * a.ng;
        constexpr int KB_PER_G = G / BK;                // 1 or 2
        const int ng = a.ng;
        // the row's group parameters are read per K block through L1; warm
        // their lines now
        for (int off = 0; off < ng * 2; off += 128) asm volatile("prefetch.global.L1 [%0];" ::"l"(sp_row + off / 2));
        for (int off = 0; off < ng; off += 128) asm volatile("prefetch.global.L1 [%0];" ::"l"(zp_row + off));
        // power-of-two headroom of this row, published for the epilogue
        const int ex = tc::row_exponent<4>(sp_row, ng, hk);
        if (grp == 0 && hk == 0) e_row[r] = (uint8_t)ex;
        // outlier cursor of this row: the next entry and the one after it
        const int* ocolp = a.col[ep];
        const uint16_t* ovalp = a.val[ep];
        int op = 0, oe = 0, ocol = 0x7FFFFFFF, ncol = 0x7FFFFFFF;
        uint16_t oval = 0, nval = 0;
        if (a.nnz[ep] > 0 && nr < a.N) {
            op = a.row_ptr[ep][n];
            oe = a.row_ptr[ep][n + 1];
            if (op < oe) {
                ocol = ocolp[op];
                oval = ovalp[op];
            }
            if (op + 1 < oe) {
                ncol = ocolp[op + 1];
                nval = ovalp[op + 1];
            }
        }
        // swizzled offsets, fixed per thread: source chunks (2*sub + hk) of the
        // packed row for this group's two blocks, destination chunks (4*hk + j)
        const uint32_t rsw = r & 7;
        const uint32_t src0 = r * 128 + (((2 * grp + hk) ^ rsw) << 4);
        const uint32_t src1 = r * 128 + (((2 * (grp + 2) + hk) ^ rsw) << 4);
        uint32_t dst_off[4];
#pragma unroll
        for (int j = 0; j < 4; j++) dst_off[j] = r * 128 + (((4 * hk + j) ^ rsw) << 4);
        unsigned char* const atile0 = smem + OFF_A;
        // group parameters of this thread's two K blocks of packed tile kp
        // (scale | zp << 16 each), loaded one packed tile ahead of their use
        auto load_prm = [&](int kp, uint32_t (&pq)[2]) {
#pragma unroll
            for (int b = 0; b < 2; b++) {
                const int kb = kp * PK + grp + b * kGroups;
                const int gi = min(kb, KB - 1) / KB_PER_G;
                pq[b] = (uint32_t)__ldg(sp_row + gi) | ((uint32_t)__ldg(zp_row + gi) << 16);   // raw: loads stay in flight
            }
        };
        auto deq_block = [&](const uint4& w, uint32_t pq, unsigned char* at) {
            const uint32_t sc = tc::f16_times_pow2(pq & 0xFFFFu, ex), zq = pq >> 16;
            const uint32_t add_lo = zq * 0x00010001u + 0xE400E400u;   // -(1024 + zp)
            const uint32_t add_hi = zq * 0x00100010u + 0xD400D400u;   // -(64 + zp)
            const uint32_t s2 = __byte_perm(sc, 0u, 0x1010u);
            *reinterpret_cast<uint4*>(at + dst_off[0]) = tc::deq8_u4(w.x, add_lo, add_hi, s2, magic);
            *reinterpret_cast<uint4*>(at + dst_off[1]) = tc::deq8_u4(w.y, add_lo, add_hi, s2, magic);
            *reinterpret_cast<uint4*>(at + dst_off[2]) = tc::deq8_u4(w.z, add_lo, add_hi, s2, magic);
            *reinterpret_cast<uint4*>(at + dst_off[3]) = tc::deq8_u4(w.w, add_lo, add_hi, s2, magic);
        };
        auto patch = [&](int kb, unsigned char* at) {
            // FP16 outliers in this thread's 32 k of block kb: the dense value there is exactly 0
            const int k0 = kb * BK + 32 * hk;
            while (ocol < k0 + 32) {
                if (ocol >= k0) {
                    const int kk = ocol - kb * BK;
                    const int pos = tc::chunk_pos<4>(kk & 31);
                    *reinterpret_cast<uint16_t*>(at + r * 128 + (((4 * (kk >> 5) + (pos >> 3)) ^ rsw) << 4) + ((pos & 7) << 1)) =
                        (uint16_t)tc::f16_times_pow2(oval, ex);
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
        };
        const int KP = (KB + PK - 1) / PK;
        int sp = 0;
        uint32_t pp = 0;   // parity of full_p to wait for
        uint32_t pcur[2], pnext[2];
        load_prm(0, pcur);
        // fp16 slots and phases of this group's blocks kb0 = 4 kp + grp and
        // kb1 = kb0 + 2, advanced by PK blocks per packed tile
        int sa0 = grp, sa1 = grp + kGroups;
        uint32_t pa0 = 0, pa1 = 0;
        static_assert(SA > PK && SA > 2 * kGroups, "one wrap per advance");
        for (int kp = 0; kp < KP && ok; kp++) {
            if (kp + 1 < KP) load_prm(kp + 1, pnext);
            const unsigned char* pt = p_tile(sp);
            ok = __all_sync(0xffffffffu, ptx::mbar_wait(full_p(sp), pp));
            if (!ok) break;
            const int kb0 = kp * PK + grp, kb1 = kb0 + kGroups;
            const bool v0 = kb0 < KB, v1 = kb1 < KB;   // uniform over the CTA
            uint4 w0 = make_uint4(0u, 0u, 0u, 0u), w1 = w0;
            if (v0) w0 = *reinterpret_cast<const uint4*>(pt + src0);
            if (v1) w1 = *reinterpret_cast<const uint4*>(pt + src1);
            bool free_ok = true;
            if (v0) free_ok = ptx::mbar_wait(empty_a(sa0), pa0 ^ 1u);
            if (v1 && free_ok) free_ok = ptx::mbar_wait(empty_a(sa1), pa1 ^ 1u);
            ok = __all_sync(0xffffffffu, free_ok);
            if (!ok) break;
            unsigned char* at0 = atile0 + sa0 * A_BYTES;
            unsigned char* at1 = atile0 + sa1 * A_BYTES;
            if (v0) deq_block(w0, pcur[0], at0);
            if (v1) deq_block(w1, pcur[1], at1);
            if (v0) patch(kb0, at0);
            if (v1) patch(kb1, at1);
            ptx::fence_proxy_async();
            __syncwarp();
            if (lane == 0) {
                if (v0) ptx::mbar_arrive(full_a(sa0));
                if (v1) ptx::mbar_arrive(full_a(sa1));
                // the packed slot goes back to its producer once per warp, after
                // the stores that consumed its codes
                ptx::mbar_arrive(empty_p(sp));
            }
            if (++sp == SP) { sp = 0; pp ^= 1u; }
            if ((sa0 += PK) >= SA) { sa0 -= SA; pa0 ^= 1u; }
            if ((sa1 += PK) >= SA) { sa1 -= SA; pa1 ^= 1u; }
            pcur[0] = pnext[0];
            pcur[1] = pnext[1];
        }
        // ------------------------------------------------ epilogue: TMEM (lane = weight row, column = token) -> y
        tc::deq_sync();   // every row's exponent is in shared memory
        if (ok) ok = __all_sync(0xffffffffu, ptx::mbar_wait(acc_full, 0));
        if (ok) {
            ptx::tc_fence_after();
            // warp w reads TMEM lanes 32 (w % 4).. and every 4th 16-column chunk from w / 4
            const int q = warp & 3, c0 = warp >> 2;
            const int nrow = n0 + 32 * q + lane;
            const float rescale = __int_as_float((127 + e_row[32 * q + lane]) << 23);   // 2^e of the row
            for (int c = c0; 16 * c < NB; c += kDeqWarps / 4) {
                uint32_t v[16], v1[16];
                ptx::tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(16 * c), v);
                ptx::tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(NBMAX + 16 * c), v1);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; j++) {   // accumulator 1 holds blocks 1, 3, ... (none when K = 64)
                    if (KB > 1) v[j] = __float_as_uint(__uint_as_float(v[j]) + __uint_as_float(v1[j]));
                    v[j] = __float_as_uint(__uint_as_float(v[j]) * rescale);
                }
                if (nrow < a.N) {
#pragma unroll
                    for (int j = 0; j < 16; j++) {
                        const int col = 16 * c + j;
                        if (col < ntok) {
                            const size_t yo = (size_t)a.perm[m0 + col] * a.N + nrow;
                            if (a.y_bf16)
                                reinterpret_cast<__nv_bfloat16*>(a.y[prod])[yo] = __float2bfloat16_rn(__uint_as_float(v[j]));
                            else
                                reinterpret_cast<float*>(a.y[prod])[yo] = __uint_as_float(v[j]);
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

bool moe_tc_eligible(const qg_qweight* experts, int E, int n)
{
    if (!(n >= 1 && n <= swap::kMaxProducts && E * n <= swap::kMaxExperts && experts[0].bits == 4 &&
          experts[0].group != 32 && experts[0].K % swap::BK == 0))
        return false;
    for (int i = 0; i < E * n; i++)   // 8-bit scales take the grouped decode kernel
        if (experts[i].scale8) return false;
    return true;
}

size_t moe_tc_x16_bytes(int P, int K) { return align_up((size_t)P * K * 2, 256); }

// n products (experts[p * E + e] is expert e of product p) over one routing:
// x is gathered once, and one launch covers every product's row tiles.
template <int G>
static qg_status moe_tc_run(const uint16_t* x, int T, int k, const qg_qweight* experts, int E, int n,
                            void* const* ys, qg_ydtype yt, const int* offsets, const int* perm, const int2* items,
                            const int* n_items, int max_items, void* x16p, cudaStream_t s)
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
    for (int i = 0; i < n * E; i++) {
        st = encode_2d(&maps.w[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, experts[i].packed, (uint64_t)K / 2, (uint64_t)N,
                       (uint64_t)K / 2, PK * BK / 2, BW, CU_TENSOR_MAP_SWIZZLE_128B);
        if (st != QG_OK) return st;
        a.scale[i] = experts[i].scale;
        a.zp[i] = experts[i].zp;
        a.row_ptr[i] = experts[i].out_row_ptr;
        a.col[i] = experts[i].out_col;
        a.val[i] = experts[i].out_val;
        a.nnz[i] = experts[i].nnz;
    }
    static_assert(kMoeTcChunk <= NBMAX && kMoeTcChunk % 16 == 0, "routing chunk fits one CTA's token tile");
    a.N = N; a.K = K; a.ng = K / G; a.chunk = kMoeTcChunk;
    a.E = E; a.tiles = (int)ceil_div(N, BW);
    a.offsets = offsets; a.perm = perm; a.items = items; a.n_items = n_items;
    for (int p = 0; p < n; p++) a.y[p] = ys[p];
    a.y_bf16 = yt == QG_Y_BF16;
    a.status = device_status_ptr();
    a.magic = gemv::kF16Magic;
    st = gemv::allow_smem(k_gemm_swap_u4<G>, SMEM);
    if (st != QG_OK) return st;
    dim3 grid((unsigned)(a.tiles * n), (unsigned)max_items, 1);
    k_gemm_swap_u4<G><<<grid, kThreads, SMEM, s>>>(xmap, maps, a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "grouped tensor-core kernel launch");
    return QG_OK;
}

qg_status launch_moe_tc(const uint16_t* x, int T, int k, const qg_qweight* experts, int E, int n, void* const* ys,
                        qg_ydtype yt, const int* offsets, const int* perm, const int2* items, const int* n_items,
                        int max_items, void* x16p, cudaStream_t s)
{
    return experts[0].group == 64
               ? moe_tc_run<64>(x, T, k, experts, E, n, ys, yt, offsets, perm, items, n_items, max_items, x16p, s)
               : moe_tc_run<128>(x, T, k, experts, E, n, ys, yt, offsets, perm, items, n_items, max_items, x16p, s);
}

}  // namespace qg
