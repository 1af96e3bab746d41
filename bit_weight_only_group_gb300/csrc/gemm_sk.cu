// Persistent stream-K form of the tensor-core product over the tile-ordered
// copy (qrepack_tiles), for prefill:
//     y[m, n] = sum_k x[m, k] * (w_hat[n, k] + S[n, k])
//
// The 256 x 256 output tiles times the K blocks of 64 form one list of work
// units (tile-major, the M tiles of one weight tile consecutive so that the
// weight blocks are reused from L2); each of at most one CTA per SM takes an
// equal, contiguous share of it.  A CTA therefore runs whole tiles plus at
// most one partial tile at each end of its share, so every SM does the same
// amount of work whatever the number of tiles (a grid of whole tiles leaves
// up to one wave partly idle: 256 tiles on 148 SMs fill 1.73 waves).  A tile
// whose K range is split between CTAs is finished without any CTA waiting
// on another: each participant stores its fp32 partial accumulator to the
// workspace and counts itself in on the tile's counter; the participant
// that arrives last adds all partials (in participant order, so the result
// does not depend on timing) and stores y.
//
// Roles per CTA (as in the one-tile kernel): warp 16 streams the fp16 x
// tiles (TMA), warp 17 the tile-ordered weight blocks (one bulk copy per K
// block), warps 0-15 dequantize into the fp16 ring and, after each of the
// CTA's tile segments, drain the TMEM accumulator; warp 18 issues the
// tcgen05.mma and waits for the accumulator to be drained before starting
// the next segment.  Every mbarrier wait is bounded (QG_ERR_TIMEOUT in the
// status word on give-up; TMA loads or MMAs in flight may then outlive the
// CTA and that call's output is not valid).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "gemv_impl.cuh"
#include "ptx.cuh"
#include "qg_internal.h"
#include "tc_dequant.cuh"

namespace qg {

qg_status encode_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                    uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw);
size_t gemm_workspace_bytes(int M, const qg_qweight& w);
qg_status launch_x_to_f16(const uint16_t* x, int M, int K, int ldx, int bits, void* x16, cudaStream_t s);

namespace sk {

constexpr int BM = 256, BN = 256, BK = 64, MH = 128;
constexpr int SA = 2, SB = 3;
constexpr int TMEM_COLS = 2 * BN;
constexpr int kDeqWarps = 16;
constexpr int kWarpA = kDeqWarps, kWarpP = kDeqWarps + 1, kWarpMma = kDeqWarps + 2;
constexpr int kThreads = (kDeqWarps + 3) * 32;
constexpr int A_BYTES = BM * BK * 2, B_BYTES = BN * BK * 2;
constexpr int SLOT_FLOATS = BM * 2 * BN / 2;   // one 256 x 256 fp32 partial tile

template <int BITS>
struct Cfg {
    static constexpr int BLOCK = 2048 * BITS + (BITS == 2 ? 2048 : 1024);
    static constexpr int P_ALIGNED = (BLOCK + 127) / 128 * 128;
    static constexpr int OFF_B = SA * A_BYTES;
    static constexpr int OFF_P = OFF_B + SB * B_BYTES;
    static constexpr int SP_FIT = (227 * 1024 - 2048 - OFF_P) / P_ALIGNED;
    static constexpr int SP = SP_FIT < 6 ? SP_FIT : 6;
    static_assert(SP >= 2, "tile ring of at least two blocks");
    static constexpr int OFF_BAR = OFF_P + SP * P_ALIGNED;
    static constexpr int OFF_EROW = OFF_BAR + 512;   // two 256-byte halves (segment parity)
    static constexpr int SMEM = OFF_BAR + 1024 + 1024;
};

struct Args {
    int M, N, K, ng, MT, KB;
    long long U;   // work units: tiles x K blocks
    int P;         // CTAs
    const uint8_t* tiles;
    const uint16_t* scale;
    const int* row_ptr;
    const int* col;
    const uint16_t* val;
    int nnz;
    void* y;
    int ldy;
    int y_bf16;
    int* status;
    uint32_t magic;
    float* partial;   // [P][2][SLOT_FLOATS]: a CTA's first and last segment
    int* count;       // [tiles] participants counted in (zeroed per call)
};

// Share of CTA c: units [lo(c), lo(c + 1)).
__host__ __device__ __forceinline__ long long unit_lo(long long U, int P, int c) { return U * c / P; }

// Segment iterator over a CTA's units: tile t, K blocks [kb0, kb1).  Unit
// indices fit in 31 bits (checked on the host).
struct Seg {
    int u, u1;
    int KB;
    int t, kb0, kb1;
    __device__ __forceinline__ bool next()
    {
        if (u >= u1) return false;
        t = u / KB;
        kb0 = u - t * KB;
        kb1 = min(KB, kb0 + (u1 - u));
        u += kb1 - kb0;
        return true;
    }
};

// The CTAs that hold part of tile t: [first, last].
__device__ __forceinline__ void participants(long long U, int P, int KB, int t, int& first, int& last)
{
    const long long a = (long long)t * KB, b = a + KB;   // units of the tile
    // first: the CTA whose share holds unit a; last: the one holding unit b - 1
    int lo = 0, hi = P - 1;
    while (lo < hi) {   // largest c with unit_lo(c) <= a
        const int mid = (lo + hi + 1) >> 1;
        if (unit_lo(U, P, mid) <= a) lo = mid;
        else hi = mid - 1;
    }
    first = lo;
    lo = first;
    hi = P - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (unit_lo(U, P, mid) <= b - 1) lo = mid;
        else hi = mid - 1;
    }
    last = lo;
}

// Store 16 consecutive outputs of token m from column nb: float4 stores
// when the run is whole and aligned, else one by one within N.
__device__ __forceinline__ void store16(const Args& a, int m, int nb, const float (&f)[16])
{
    if (a.y_bf16) {
        __nv_bfloat16* yr = reinterpret_cast<__nv_bfloat16*>(a.y) + (size_t)m * a.ldy;
#pragma unroll
        for (int q = 0; q < 16; q++)
            if (nb + q < a.N) yr[nb + q] = __float2bfloat16_rn(f[q]);
        return;
    }
    float* yr = reinterpret_cast<float*>(a.y) + (size_t)m * a.ldy;
    if (nb + 16 <= a.N && (reinterpret_cast<uintptr_t>(yr + nb) & 15u) == 0) {
#pragma unroll
        for (int q = 0; q < 16; q += 4) *reinterpret_cast<float4*>(yr + nb + q) = make_float4(f[q], f[q + 1], f[q + 2], f[q + 3]);
    } else {
#pragma unroll
        for (int q = 0; q < 16; q++)
            if (nb + q < a.N) yr[nb + q] = f[q];
    }
}

template <int BITS, int G>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_sk(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ Args a)
{
    using C = Cfg<BITS>;
    constexpr int SP = C::SP;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = ptx::smem_u32(smem);
    const uint32_t bars = sbase + C::OFF_BAR;
    auto full_a = [&](int s) { return bars + 8 * s; };
    auto empty_a = [&](int s) { return bars + 8 * (SA + s); };
    auto full_p = [&](int s) { return bars + 8 * (2 * SA + s); };
    auto empty_p = [&](int s) { return bars + 8 * (2 * SA + SP + s); };
    auto full_b = [&](int s) { return bars + 8 * (2 * SA + 2 * SP + s); };
    auto empty_b = [&](int s) { return bars + 8 * (2 * SA + 2 * SP + SB + s); };
    const uint32_t acc_full = bars + 8 * (2 * SA + 2 * SP + 2 * SB);
    const uint32_t acc_empty = acc_full + 8;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 8 * (2 * SA + 2 * SP + 2 * SB + 2));
    int* bcast = reinterpret_cast<int*>(smem + C::OFF_BAR + 8 * (2 * SA + 2 * SP + 2 * SB + 3));   // 3 ints
    auto a_tile = [&](int s) { return sbase + s * A_BYTES; };
    auto b_tile = [&](int s) { return sbase + C::OFF_B + s * B_BYTES; };
    auto p_tile = [&](int s) { return smem + C::OFF_P + s * C::P_ALIGNED; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x;
    const int KB = a.KB;
    const Seg seg0{(int)unit_lo(a.U, a.P, c), (int)unit_lo(a.U, a.P, c + 1), KB, 0, 0, 0};

    if (threadIdx.x == 0) {
        for (int s = 0; s < SA; s++) { ptx::mbar_init(full_a(s), 1); ptx::mbar_init(empty_a(s), 1); }
        for (int s = 0; s < SP; s++) { ptx::mbar_init(full_p(s), 1); ptx::mbar_init(empty_p(s), kDeqWarps); }
        for (int s = 0; s < SB; s++) { ptx::mbar_init(full_b(s), kDeqWarps); ptx::mbar_init(empty_b(s), 1); }
        ptx::mbar_init(acc_full, 1);
        ptx::mbar_init(acc_empty, kDeqWarps);
        ptx::fence_mbar_init();
    }
    if (warp == kWarpMma) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), TMEM_COLS);
        ptx::tmem_relinquish();
    }
    if (warp == kWarpA && lane == 0) ptx::prefetch_tensormap(&xmap);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    if (warp == kWarpA) {
        // ------------------------------------------------ x tiles (TMA) of every segment
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            Seg g = seg0;
            while (ok && g.next()) {
                const int mt = g.t % a.MT;
                for (int kb = g.kb0; kb < g.kb1; kb++) {
                    if (!ptx::mbar_wait(empty_a(s), ph ^ 1u)) { ok = false; break; }
                    ptx::mbar_expect_tx(full_a(s), A_BYTES);
                    ptx::tma_load_2d(a_tile(s), &xmap, kb * BK, mt * BM, full_a(s));
                    if (++s == SA) { s = 0; ph ^= 1u; }
                }
            }
        }
    } else if (warp == kWarpP) {
        // ------------------------------------------------ tile-ordered weight blocks (one bulk copy each)
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            Seg g = seg0;
            while (ok && g.next()) {
                const int nt = g.t / a.MT;
                const uint8_t* base = a.tiles + (size_t)nt * KB * C::BLOCK;
                for (int kb = g.kb0; kb < g.kb1; kb++) {
                    if (!ptx::mbar_wait(empty_p(s), ph ^ 1u)) { ok = false; break; }
                    ptx::mbar_expect_tx(full_p(s), C::BLOCK);
                    ptx::bulk_load(ptx::smem_u32(p_tile(s)), base + (size_t)kb * C::BLOCK, C::BLOCK, full_p(s));
                    if (++s == SP) { s = 0; ph ^= 1u; }
                }
            }
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------ MMA issuer: one accumulation per segment
        constexpr uint32_t idesc = ptx::idesc_f16_f32(MH, BN);
        const uint64_t adesc0 = ptx::sw128_desc(a_tile(0)), bdesc0 = ptx::sw128_desc(b_tile(0));
        int sa = 0, sb = 0;
        uint32_t pa = 0, pb = 0;
        int j = 0;
        Seg g = seg0;
        while (ok && g.next()) {
            if (j > 0) {   // the previous segment's accumulator has been drained
                ok = __all_sync(0xffffffffu, ptx::mbar_wait(acc_empty, (uint32_t)((j - 1) & 1)));
                if (!ok) break;
                ptx::tc_fence_after();
            }
            for (int kb = g.kb0; kb < g.kb1; kb++) {
                ok = __all_sync(0xffffffffu, ptx::mbar_wait(full_a(sa), pa) && ptx::mbar_wait(full_b(sb), pb));
                if (!ok) break;
                ptx::tc_fence_after();
                const uint64_t ad = adesc0 + (uint64_t)((sa * A_BYTES) >> 4);
                const uint64_t bd = bdesc0 + (uint64_t)((sb * B_BYTES) >> 4);
                const uint32_t acc0 = kb > g.kb0 ? 1u : 0u;
#pragma unroll
                for (int kk = 0; kk < BK / 16; kk++) {
                    ptx::mma_f16_elect(tmem, ad + 2 * kk, bd + 2 * kk, idesc, acc0 | (kk > 0));
                    ptx::mma_f16_elect(tmem + BN, ad + ((MH * 128) >> 4) + 2 * kk, bd + 2 * kk, idesc, acc0 | (kk > 0));
                }
                ptx::tc_commit_elect(empty_a(sa));
                ptx::tc_commit_elect(empty_b(sb));
                if (++sa == SA) { sa = 0; pa ^= 1u; }
                if (++sb == SB) { sb = 0; pb ^= 1u; }
            }
            if (!ok) break;
            ptx::tc_commit_elect(acc_full);
            ++j;
        }
    } else {
        // ------------------------------------------------ dequantization + epilogue (two threads per row)
        const uint32_t magic = a.magic;
        const int r = threadIdx.x >> 1, hk = threadIdx.x & 1;
        const uint32_t rsw = r & 7;
        uint32_t dst_off[4];
#pragma unroll
        for (int q = 0; q < 4; q++) dst_off[q] = r * 128 + (((4 * hk + q) ^ rsw) << 4);
        unsigned char* const btile0 = smem + C::OFF_B;
        int sb = 0, sp = 0;
        uint32_t pb = 1, pp = 0;   // parities: empty_b, full_p to wait for
        int j = 0;
        Seg g = seg0;
        while (g.next()) {   // every dequant warp runs every segment (the named barriers below)
            const int nt = g.t / a.MT, mt = g.t % a.MT;
            const int n0 = nt * BN, m0 = mt * BM;
            const int nr = n0 + r, n = min(nr, a.N - 1);
            uint8_t* e_row = smem + C::OFF_EROW + (j & 1) * 256;
            int ex = 0;
            if constexpr (BITS != 2) ex = tc::row_exponent<BITS>(a.scale + (size_t)n * a.ng, a.ng, hk);
            if (hk == 0) e_row[r] = (uint8_t)ex;
            // outlier cursor from the segment's first column
            int op = 0, oe = 0, ocol = 0x7FFFFFFF, ncol = 0x7FFFFFFF;
            uint16_t oval = 0, nval = 0;
            if (a.nnz > 0 && nr < a.N) {
                int lo = __ldg(a.row_ptr + n), hi = __ldg(a.row_ptr + n + 1);
                oe = hi;
                const int c0 = g.kb0 * BK;
                while (lo < hi) {
                    const int mid = (lo + hi) >> 1;
                    if (__ldg(a.col + mid) < c0) lo = mid + 1;
                    else hi = mid;
                }
                op = lo;
                if (op < oe) { ocol = __ldg(a.col + op); oval = __ldg(a.val + op); }
                if (op + 1 < oe) { ncol = __ldg(a.col + op + 1); nval = __ldg(a.val + op + 1); }
            }
            for (int kb = g.kb0; kb < g.kb1 && ok; kb++) {
                ok = __all_sync(0xffffffffu, ptx::mbar_wait(full_p(sp), pp));
                if (!ok) break;
                const uint32_t* pw = reinterpret_cast<const uint32_t*>(p_tile(sp));
                uint32_t w[BITS];
#pragma unroll
                for (int i = 0; i < BITS; i++) w[i] = pw[i * 512 + threadIdx.x];
                uint32_t pr[16];
                if constexpr (BITS == 2) {
                    const uint2 cbv = reinterpret_cast<const uint2*>(pw + BITS * 512)[r];
                    const uint32_t lo = __byte_perm(cbv.x, cbv.y, 0x6420), hi = __byte_perm(cbv.x, cbv.y, 0x7531);
#pragma unroll
                    for (int wi = 0; wi < 2; wi++)
#pragma unroll
                        for (int jf = 0; jf < 4; jf++) {
                            const uint32_t f = (w[wi] >> (2 * jf)) & 0x03030303u;
                            pr[2 * (4 * wi + jf)] = tc::cb_pair<0>(f, lo, hi);
                            pr[2 * (4 * wi + jf) + 1] = tc::cb_pair<1>(f, lo, hi);
                        }
                } else {
                    const uint32_t pq = pw[BITS * 512 + r];
                    const uint32_t s2 = __byte_perm(tc::f16_times_pow2(pq & 0xFFFFu, ex), 0u, 0x1010u);
                    const uint32_t zq = pq >> 16;
                    gemv::static_for<0, 16>([&](auto ec) {
                        constexpr int e = decltype(ec)::value;
                        pr[e] = tc::hmul2_u32(gemv::deq_affine<BITS, 32, e>(w, zq, magic), s2);
                    });
                }
                ok = __all_sync(0xffffffffu, ptx::mbar_wait(empty_b(sb), pb));
                if (!ok) break;
                unsigned char* bt = btile0 + sb * B_BYTES;
#pragma unroll
                for (int q = 0; q < 4; q++)
                    *reinterpret_cast<uint4*>(bt + dst_off[q]) = make_uint4(pr[4 * q], pr[4 * q + 1], pr[4 * q + 2], pr[4 * q + 3]);
                const int k0 = kb * BK + 32 * hk;
                while (ocol < k0 + 32) {
                    if (ocol >= k0) {
                        const int pos = tc::chunk_pos<BITS>(ocol - k0);
                        uint16_t* dst = reinterpret_cast<uint16_t*>(bt + r * 128 + (((4 * hk + (pos >> 3)) ^ rsw) << 4) + ((pos & 7) << 1));
                        if constexpr (BITS == 2) *dst = tc::f16_add_sat(*dst, oval, 0);
                        else *dst = (uint16_t)tc::f16_times_pow2(oval, ex);
                    }
                    ocol = ncol;
                    oval = nval;
                    if (++op + 1 < oe) { ncol = __ldg(a.col + op + 1); nval = __ldg(a.val + op + 1); }
                    else ncol = 0x7FFFFFFF;
                }
                ptx::fence_proxy_async();
                __syncwarp();
                if (lane == 0) {
                    ptx::mbar_arrive(full_b(sb));
                    ptx::mbar_arrive(empty_p(sp));   // after the warp's shared loads of the block completed
                }
                if (++sb == SB) { sb = 0; pb ^= 1u; }
                if (++sp == SP) { sp = 0; pp ^= 1u; }
            }
            // ------------------------------------------ epilogue of the segment
            tc::deq_sync();   // e_row complete
            const bool whole = g.kb0 == 0 && g.kb1 == KB;
            if (ok) ok = __all_sync(0xffffffffu, ptx::mbar_wait(acc_full, (uint32_t)(j & 1)));
            ptx::tc_fence_after();
            const int q4 = warp & 3, quarter = warp >> 2;
            if (whole) {
                // TMEM -> y (rows built at scale * 2^-e multiplied back by 2^e)
#pragma unroll 1
                for (int i = 0; i < 8; i++) {
                    const int colx = 128 * quarter + 16 * i;
                    const int half = colx / BN, cb = colx % BN;
                    const int m = m0 + MH * half + 32 * q4 + lane;
                    uint32_t v[16];
                    if (ok) {
                        ptx::tmem_ld16(tmem + ((uint32_t)(32 * q4) << 16) + (uint32_t)colx, v);
                        ptx::tmem_ld_wait();
                    }
                    const uint4 ew = *reinterpret_cast<const uint4*>(e_row + cb);
                    if (ok && m < a.M) {
                        const uint32_t ewa[4] = {ew.x, ew.y, ew.z, ew.w};
                        float f[16];
#pragma unroll
                        for (int q = 0; q < 16; q++) {
                            const int ej = (ewa[q >> 2] >> (8 * (q & 3))) & 0xFF;
                            f[q] = __uint_as_float(v[q]) * __int_as_float((127 + ej) << 23);
                        }
                        store16(a, m, n0 + cb, f);
                    }
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(acc_empty);
            } else {
                // split tile: store this CTA's partial, count in; the last participant sums and stores
                // slot 1: the segment that starts the tile (this CTA's last one);
                // slot 0: a segment that starts inside the tile (this CTA's first)
                const int which = g.kb0 == 0 ? 1 : 0;
                float* mine = a.partial + ((size_t)c * 2 + which) * SLOT_FLOATS;
#pragma unroll 1
                for (int i = 0; i < 8; i++) {
                    const int colx = 128 * quarter + 16 * i;
                    uint32_t v[16];
                    if (ok) {
                        ptx::tmem_ld16(tmem + ((uint32_t)(32 * q4) << 16) + (uint32_t)colx, v);
                        ptx::tmem_ld_wait();
                        float4* dst = reinterpret_cast<float4*>(mine + ((size_t)(warp * 8 + i) * 32 + lane) * 16);
#pragma unroll
                        for (int q = 0; q < 4; q++)
                            dst[q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                                 __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
                    }
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(acc_empty);   // TMEM drained: the next segment may start
                __threadfence();
                tc::deq_sync();
                if (threadIdx.x == 0) {
                    int first, last;
                    participants(a.U, a.P, KB, g.t, first, last);
                    bcast[0] = atomicAdd(a.count + g.t, 1);
                    bcast[1] = first;
                    bcast[2] = last;
                }
                tc::deq_sync();
                const int first = bcast[1], last = bcast[2];
                if (bcast[0] == last - first) {   // every other participant has stored and counted in
                    __threadfence();
#pragma unroll 1
                    for (int i = 0; i < 8; i++) {
                        const int colx = 128 * quarter + 16 * i;
                        const int half = colx / BN, cb = colx % BN;
                        const int m = m0 + MH * half + 32 * q4 + lane;
                        float s16v[16];
#pragma unroll
                        for (int q = 0; q < 16; q++) s16v[q] = 0.0f;
                        for (int pc = first; pc <= last; pc++) {   // participant order: deterministic
                            const int pw = pc == first ? 1 : 0;
                            const float4* src = reinterpret_cast<const float4*>(
                                a.partial + ((size_t)pc * 2 + pw) * SLOT_FLOATS + ((size_t)(warp * 8 + i) * 32 + lane) * 16);
#pragma unroll
                            for (int q = 0; q < 4; q++) {
                                const float4 f = __ldcg(src + q);
                                s16v[4 * q] += f.x; s16v[4 * q + 1] += f.y; s16v[4 * q + 2] += f.z; s16v[4 * q + 3] += f.w;
                            }
                        }
                        const uint4 ew = *reinterpret_cast<const uint4*>(e_row + cb);
                        if (ok && m < a.M) {
                            const uint32_t ewa[4] = {ew.x, ew.y, ew.z, ew.w};
#pragma unroll
                            for (int q = 0; q < 16; q++) {
                                const int ej = (ewa[q >> 2] >> (8 * (q & 3))) & 0xFF;
                                s16v[q] *= __int_as_float((127 + ej) << 23);
                            }
                            store16(a, m, n0 + cb, s16v);
                        }
                    }
                }
            }
            tc::deq_sync();   // e_row of this segment no longer read before the next one is written
            ++j;
        }
    }
    if (!ok && a.status) atomicExch(a.status, (int)QG_ERR_TIMEOUT);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == kWarpMma) ptx::tmem_dealloc(tmem, TMEM_COLS);
}

// Workspace after the fp16 copy of x: the partial slots and the tile counters.
struct Ws {
    void* x16;
    float* partial;
    int* count;
};

size_t ws_layout(int M, const qg_qweight& w, int P, Ws* p, void* base)
{
    const size_t ox = 0;
    const size_t op = align_up(gemm_workspace_bytes(M, w), 256);
    const size_t oc = op + (size_t)P * 2 * SLOT_FLOATS * sizeof(float);
    const long long tiles = ceil_div(M, BM) * ceil_div(w.N, BN);
    const size_t total = align_up(oc + sizeof(int) * (size_t)tiles, 256);
    if (p && base) {
        char* b = static_cast<char*>(base);
        p->x16 = b + ox;
        p->partial = reinterpret_cast<float*>(b + op);
        p->count = reinterpret_cast<int*>(b + oc);
    }
    return total;
}

template <int BITS, int G>
qg_status run(const uint16_t* x, int M, int ldx, const qg_qweight& w, const void* tiles, void* y, int ldy,
              qg_ydtype yt, void* ws, cudaStream_t s)
{
    using C = Cfg<BITS>;
    const int MT = (int)ceil_div(M, BM), NT = (int)ceil_div(w.N, BN), KB = w.K / BK;
    const long long U = (long long)MT * NT * KB;
    if (U >= (1LL << 31)) return fail(QG_ERR_UNSUPPORTED, "qgemm_forward_tiles: %lld work units (above 2^31)", U);
    const int P = (int)std::min<long long>(num_sms(), U);
    Ws p{};
    ws_layout(M, w, P, &p, ws);
    qg_status st = launch_x_to_f16(x, M, w.K, ldx, BITS, p.x16, s);
    if (st != QG_OK) return st;
    cudaError_t e = cudaMemsetAsync(p.count, 0, sizeof(int) * (size_t)MT * NT, s);
    if (e != cudaSuccess) return cuda_fail(e, "stream-K counters");
    CUtensorMap xmap;
    st = encode_2d(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, p.x16, (uint64_t)w.K, (uint64_t)M, (uint64_t)w.K * 2, BK, BM,
                   CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != QG_OK) return st;
    Args a;
    a.M = M; a.N = w.N; a.K = w.K; a.ng = w.K / G; a.MT = MT; a.KB = KB; a.U = U; a.P = P;
    a.tiles = static_cast<const uint8_t*>(tiles);
    a.scale = w.scale;
    a.row_ptr = w.out_row_ptr; a.col = w.out_col; a.val = w.out_val; a.nnz = w.nnz;
    a.y = y; a.ldy = ldy; a.y_bf16 = yt == QG_Y_BF16;
    a.status = device_status_ptr();
    a.magic = gemv::kF16Magic;
    a.partial = p.partial;
    a.count = p.count;
    st = gemv::allow_smem(k_gemm_sk<BITS, G>, C::SMEM);
    if (st != QG_OK) return st;
    k_gemm_sk<BITS, G><<<P, kThreads, C::SMEM, s>>>(xmap, a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "stream-K tensor-core kernel launch");
    return QG_OK;
}

template <int BITS>
qg_status run_bits(const uint16_t* x, int M, int ldx, const qg_qweight& w, const void* tiles, void* y, int ldy,
                   qg_ydtype yt, void* ws, cudaStream_t s)
{
    return w.group == 64 ? run<BITS, 64>(x, M, ldx, w, tiles, y, ldy, yt, ws, s)
                         : run<BITS, 128>(x, M, ldx, w, tiles, y, ldy, yt, ws, s);
}

}  // namespace sk

size_t gemm_tiles_workspace_bytes(int M, const qg_qweight& w)
{
    const int MT = (int)ceil_div(M, sk::BM), NT = (int)ceil_div(w.N, sk::BN), KB = w.K / sk::BK;
    const int P = (int)std::min<long long>(num_sms(), (long long)MT * NT * KB);
    return sk::ws_layout(M, w, P, nullptr, nullptr);
}

qg_status launch_gemm_tiles(const uint16_t* x, int M, int ldx, const qg_qweight& w, const void* tiles, void* y,
                            int ldy, qg_ydtype yt, void* ws, cudaStream_t s)
{
    switch (w.bits) {
        case 2: return sk::run_bits<2>(x, M, ldx, w, tiles, y, ldy, yt, ws, s);
        case 3: return sk::run_bits<3>(x, M, ldx, w, tiles, y, ldy, yt, ws, s);
        case 4: return sk::run_bits<4>(x, M, ldx, w, tiles, y, ldy, yt, ws, s);
        case 5: return sk::run_bits<5>(x, M, ldx, w, tiles, y, ldy, yt, ws, s);
        case 6: return sk::run_bits<6>(x, M, ldx, w, tiles, y, ldy, yt, ws, s);
        default: return sk::run_bits<8>(x, M, ldx, w, tiles, y, ldy, yt, ws, s);
    }
}

}  // namespace qg
