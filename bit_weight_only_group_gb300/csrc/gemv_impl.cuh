// Decode-side fused dequantization product for small M (M <= 64):
//     y[m, n] = sum_k x[m, k] * (w_hat[n, k] + S[n, k])
// Memory-bound: every packed weight byte is read from HBM once, unpacked in
// registers (never written back as fp16 -- "Mixed-width quantization" page, section 4.1: unpack
// and multiply-accumulate in one loop, the value lives only in registers),
// and consumed by warp-level tensor-core MMAs with fp32 accumulation
// (section 4.2 requires fp32 accumulation).
//
// Layout of the work (GB300, 152 SMs):
//  * a CTA = 4 warps = 64 consecutive weight rows; a warp owns 16 rows and
//    issues mma.sync.m16n8k16 with the weights as the A operand (rows = W
//    rows, "swap AB") and up to 8 tokens per n8 tile as B;
//  * K is split across the CTAs of a thread-block cluster (1, S, 1); their
//    fp32 partials are summed in rank order through distributed shared
//    memory -- deterministic, no global workspace, no spin-waits;
//  * each thread owns, per group and row, one contiguous quarter of the
//    group's codes ("chunk").  Inside an MMA the 16 k positions may be
//    permuted freely as long as A and B agree, so each thread turns its chunk
//    into fp16 pairs with one AND+OR (LOP3) per pair: a b-bit code placed at
//    mantissa bits [p, p+b) of the fp16 value 1024 reads as 1024 + 2^p * q;
//    one packed FMA (HFMA2) by (2^-p, -1024*2^-p - zp) turns the pair into the
//    exact integers q - zp.  The MMA sums (q - zp) * x exactly per product in
//    fp32, and the group's fp16 scale is applied to that fp32 partial.
//    (Magic-number int->fp16 conversion after Kim et al. 2022, "Who Says
//    Elephants Can't Run"; the per-width pair plans are this library's own.)
//  * 2-bit groups hold 4 fp16 codebook entries; two byte-permutes (PRMT)
//    look up a pair of entries at once from a 2-register table.
//  * the FP16 outliers ("70B on one GPU" page, section 2, step 3: added
//    back after the product) are applied in the cluster epilogue from CSR.
#pragma once

#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>
#include <mutex>
#include <type_traits>

#include "ptx.cuh"
#include "qg_internal.h"
#include "scale8.cuh"

namespace cg = cooperative_groups;

namespace qg {

namespace gemv {

constexpr int kWarps = 4;
constexpr int kRowsPerCta = 16 * kWarps;

// ---------------------------------------------------------------- pair plans
// Entry e of a thread chunk with NC codes: codes `lo` and `hi` of the chunk
// go to the low and high fp16 half; in the 32-bit window that starts at
// chunk bit S, code lo sits at bit plo and code hi at bit 16 + phi
// (plo, phi <= 10 - bits, so 1024 + 2^p * q stays an exact fp16 integer).
// For bits == 2 the entry only names the two codes of a PRMT lookup.
struct PairE {
    int lo, hi, plo, phi, S;
};

__host__ __device__ constexpr PairE plan_entry(int bits, int nc, int e)
{
    if (bits == 4) {   // (i, i+4) within each 8-code word; windows at 0, 8
        const int j = e / 4, q = e % 4;
        return PairE{8 * j + q, 8 * j + q + 4, (q & 1) * 4, (q & 1) * 4, 32 * j + (q / 2) * 8};
    }
    if (bits == 2) {
        if (nc == 8) {   // PRMT pairs of an 8-code chunk: (s, s+4) and (s+2, s+6) in step s
            const int st = e / 2, h = e % 2;
            return PairE{st + 2 * h, st + 2 * h + 4, 0, 0, 0};
        }
        // PRMT pairs: (j, j+4) and (j+8, j+12) within each 16-code word
        const int w = e / 8, j = (e % 8) / 2, h = e % 2;
        const int lo = 16 * w + (h ? 8 : 0) + j;
        return PairE{lo, lo + 4, 0, 0, 0};
    }
    if (bits == 8) {   // bytes (4j + h, 4j + h + 2) of word j: windows at 32j and 32j + 8
        const int j = e / 2, h = e % 2;
        return PairE{4 * j + h, 4 * j + h + 2, 0, 0, 32 * j + 8 * h};
    }
    if (bits == 6) {   // (i, i+2) within each 4-code unit (3 bytes)
        const int m = e / 2, q = e % 2;
        const int lo = 4 * m + q;
        return PairE{lo, lo + 2, 4, 0, 6 * lo - 4};
    }
    if (bits == 3) {   // four pairs per 8-code unit (3 bytes), two windows
        const int u = e / 4, q = e % 4;
        const int lo = 8 * u + q;
        return PairE{lo, lo + 4, (q & 1) ? 7 : 4, (q & 1) ? 3 : 0, 24 * u + (q < 2 ? -4 : 2)};
    }
    // bits == 5: one pair per window
    if (nc == 8) {     // (i, i+4): code i at bit 0 and code i+4 at bit 20 of the window at 5i
        return PairE{e, e + 4, 0, 4, 5 * e};
    }
    // found by an exhaustive search
    if (nc == 16) {
        constexpr PairE t[8] = {{0, 3, 5, 4, -5},  {1, 4, 5, 4, 0},   {2, 6, 1, 5, 9},
                                {5, 8, 5, 4, 20},  {7, 10, 5, 4, 30}, {9, 13, 1, 5, 44},
                                {11, 14, 5, 4, 50}, {12, 15, 5, 4, 55}};
        return t[e];
    }
    constexpr PairE t[16] = {{0, 3, 5, 4, -5},    {1, 4, 5, 4, 0},     {2, 5, 5, 4, 5},
                             {6, 9, 5, 4, 25},    {7, 10, 5, 4, 30},   {8, 11, 5, 4, 35},
                             {12, 15, 5, 4, 55},  {13, 16, 5, 4, 60},  {14, 17, 5, 4, 65},
                             {18, 21, 5, 4, 85},  {19, 22, 5, 4, 90},  {20, 23, 5, 4, 95},
                             {24, 27, 5, 4, 115}, {25, 29, 1, 5, 124}, {26, 30, 1, 5, 129},
                             {28, 31, 5, 4, 135}};
    return t[e];
}

template <int I, int N, typename F>
__device__ __forceinline__ void static_for(F&& f)
{
    if constexpr (I < N) {
        f(std::integral_constant<int, I>{});
        static_for<I + 1, N>(f);
    }
}

// 32 bits of the chunk stream starting at bit S (S may be negative).
template <int S, int NW>
__device__ __forceinline__ uint32_t window(const uint32_t (&w)[NW])
{
    if constexpr (S < 0) {
        return w[0] << (-S);
    } else {
        constexpr int q = S / 32, r = S % 32;
        if constexpr (r == 0) {
            return w[q];
        } else if constexpr (q + 1 < NW) {
            return __funnelshift_r(w[q], w[q + 1], r);
        } else {
            return w[q] >> r;
        }
    }
}

__device__ __forceinline__ float pow2f(int e) { return __int_as_float((127 + e) << 23); }

__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// fp16 pair (q_lo - zp, q_hi - zp) of entry E, exact: the LOP3 gives
// (1024 + 2^plo q_lo, 1024 + 2^phi q_hi); the HFMA2 scales by 2^-p (exact)
// and adds -(1024*2^-p + zp).  Because zp < 2^bits <= 1024*2^-p, the value
// 1024*2^-p + zp stays in the binade of 1024*2^-p, where one fp16 step is
// 2^-p: its bit pattern is bits(1024*2^-p) + zp*2^p, so the addend is one
// integer multiply-add on zp.
template <int BITS, int NC, int E>
__device__ __forceinline__ uint32_t zp_addend(uint32_t zp)
{
    constexpr PairE p = plan_entry(BITS, NC, E);
    constexpr uint32_t base = (uint32_t)(0xE400 - 0x400 * p.plo) | ((uint32_t)(0xE400 - 0x400 * p.phi) << 16);
    constexpr uint32_t mul = (1u << p.plo) | ((1u << p.phi) << 16);
    return zp * mul + base;
}

// Exponent pattern of fp16 1024 in both halves.  The kernels receive it as a
// run-time value (Problem::magic, Args::magic) so that it stays in a register:
// (v & mask) | magic is then one three-input logic op, where two compile-time
// 32-bit constants would not fit one instruction and cost two.
constexpr uint32_t kF16Magic = 0x64006400u;

// (a & MASK) | c in one lop3 (truth table 0xEA = (A & B) | C).
template <uint32_t MASK>
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t c)
{
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "n"(MASK), "r"(c));
    return d;
}

template <int BITS, int NC, int E, int NW>
__device__ __forceinline__ uint32_t deq_affine(const uint32_t (&w)[NW], uint32_t zp, uint32_t magic)
{
    constexpr PairE p = plan_entry(BITS, NC, E);
    constexpr uint32_t cm = (1u << BITS) - 1u;
    constexpr uint32_t mask = (cm << p.plo) | (cm << (16 + p.phi));
    const uint32_t raw = and_or<mask>(window<p.S, NW>(w), magic);
    constexpr uint32_t mul = (uint32_t)(0x3C00 - 0x400 * p.plo) | ((uint32_t)(0x3C00 - 0x400 * p.phi) << 16);
    return hfma2_u32(raw, mul, zp_addend<BITS, NC, E>(zp));
}

// ---------------------------------------------------------------- loads
__device__ __forceinline__ uint4 ldg_stream128(const void* p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ldg_stream64(const void* p)
{
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ldg_stream32(const void* p)
{
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// Load the CB = NC*BITS/8 bytes of one chunk into NW little-endian words.
template <int BITS, int G>
struct Chunk {
    static constexpr int NC = G / 4;
    static constexpr int CB = NC * BITS / 8;
    static constexpr int NW = (NC * BITS + 31) / 32;
    // CB = 12 or 20 (3-bit and 5-bit g128, 6-bit g64): rows and groups are
    // 8-byte aligned and CB = 4 (mod 8), so a chunk starts 8-byte aligned on
    // even lanes t and 4 bytes past that on odd ones.  It is read as one
    // 4-byte and (CB - 4) / 8 8-byte loads -- the 4-byte one at the end of
    // the chunk on even lanes, at its start on odd ones -- instead of CB / 4
    // 4-byte loads, which filled the load queue.  The words stay in load
    // order R = (8-byte words..., 4-byte word) in the ring; order() puts them
    // in stream order when the group is used (odd lanes: the 4-byte word
    // first).
    static constexpr bool SPLIT = CB % 8 == 4 && CB > 4;
    // Group 32 with chunks off word boundaries (2, 3, 5, 6 bits): the group
    // is BITS whole words per row, and lane t of a row's 4 lanes loads its
    // words t and t + 4; each thread gathers the (at most two) words holding
    // its chunk from those lanes with shuffles when the group is used
    // (assemble).  Loading each chunk's own words instead read most bytes
    // two or three times through L2 (2.1x the L2 sectors of group 128).
    static constexpr bool SHUF = G == 32 && CB % 4 != 0;
    __device__ __forceinline__ static void order(const uint32_t (&r)[NW], uint32_t (&w)[NW], bool odd)
    {
#pragma unroll
        for (int i = 0; i < NW; i++) w[i] = odd ? r[(i + NW - 1) % NW] : r[i];
    }
    // SHUF: the lane's words t and t + 4 of the group (p is the chunk at byte
    // t * CB of the group; the words of a group lie inside it)
    __device__ __forceinline__ static void load_words(const uint8_t* p, int t, uint32_t (&r)[NW])
    {
        const uint32_t* g = reinterpret_cast<const uint32_t*>(p - t * CB);
        r[0] = t < BITS ? ldg_stream32(g + t) : 0u;
        if constexpr (NW > 1) r[1] = t + 4 < BITS ? ldg_stream32(g + t + 4) : 0u;
    }
    // SHUF: this thread's chunk words from the loaded words of its row's lanes
    // (every lane of the warp calls it)
    __device__ __forceinline__ static void assemble(const uint32_t (&r)[NW], uint32_t (&w)[NW], int lane)
    {
        const int t = lane & 3, byte0 = t * CB, wa = byte0 >> 2, sh = (byte0 & 3) * 8;
        const int srcA = (lane & ~3) | (wa & 3), srcB = (lane & ~3) | ((wa + 1) & 3);
        uint32_t a = __shfl_sync(0xffffffffu, r[0], srcA);
        uint32_t b = __shfl_sync(0xffffffffu, r[0], srcB);
        if constexpr (NW > 1) {
            const uint32_t a1 = __shfl_sync(0xffffffffu, r[1], srcA);
            const uint32_t b1 = __shfl_sync(0xffffffffu, r[1], srcB);
            a = wa < 4 ? a : a1;
            b = wa + 1 < 4 ? b : b1;
        }
        w[0] = __funnelshift_r(a, b, sh);
        if constexpr (NW > 1) w[1] = sh ? b >> sh : b;
    }
    __device__ __forceinline__ static void load(const uint8_t* p, uint32_t (&w)[NW])
    {
        if constexpr (SPLIT) {
            const bool odd = (reinterpret_cast<uintptr_t>(p) & 4u) != 0;
            const uint8_t* p8 = p + (odd ? 4 : 0);
#pragma unroll
            for (int i = 0; i < (CB - 4) / 8; i++) {
                const uint2 v = ldg_stream64(p8 + 8 * i);
                w[2 * i] = v.x; w[2 * i + 1] = v.y;
            }
            w[NW - 1] = ldg_stream32(p + (odd ? 0 : CB - 4));
        } else if constexpr (CB % 16 == 0) {
#pragma unroll
            for (int i = 0; i < CB / 16; i++) {
                const uint4 v = ldg_stream128(p + 16 * i);
                w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
            }
        } else if constexpr (CB % 8 == 0) {
#pragma unroll
            for (int i = 0; i < CB / 8; i++) {
                const uint2 v = ldg_stream64(p + 8 * i);
                w[2 * i] = v.x; w[2 * i + 1] = v.y;
            }
        } else if constexpr (CB % 4 == 0) {
#pragma unroll
            for (int i = 0; i < CB / 4; i++) w[i] = ldg_stream32(p + 4 * i);
        } else {
            // chunk at any byte offset (group 64 odd widths: 2-byte aligned;
            // group 32 at 3 and 5 bits: byte aligned): the aligned words that
            // hold its bytes, then a funnel shift by the chunk's offset in
            // the first word.  Groups start 4-byte aligned and span a whole
            // number of words, so every word read lies inside this group.
            constexpr int NWL = (CB + 3 + 3) / 4;
            const uintptr_t a = reinterpret_cast<uintptr_t>(p);
            const uint8_t* base = reinterpret_cast<const uint8_t*>(a & ~uintptr_t(3));
            const int off = (int)(a & 3u);
            uint32_t raw[NWL + 1];
#pragma unroll
            for (int i = 0; i < NWL; i++) raw[i] = (4 * i < off + CB) ? ldg_stream32(base + 4 * i) : 0u;
            raw[NWL] = 0u;
            const int sh = off * 8;
#pragma unroll
            for (int i = 0; i < NW; i++) w[i] = __funnelshift_r(raw[i], raw[i + 1], sh);
        }
    }
};

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint16_t x_f16(__nv_bfloat16 v)
{
    return __half_as_ushort(__float2half_rn(__bfloat162float(v)));
}

__device__ __forceinline__ float h2f(uint16_t h) { return __half2float(__ushort_as_half(h)); }

// One product on one weight matrix.  Token m reads x row
// (rowmap ? rowmap[m] / xdiv : m) and writes y row (rowmap ? rowmap[m] : m).
struct Problem {
    const __nv_bfloat16* x;
    int ldx, M, N, K;
    const int* rowmap;
    int xdiv;
    const uint8_t* packed;
    const uint16_t* scale;
    const uint8_t* zp;
    const uint2* cb;
    const int* row_ptr;
    const int* col;
    const uint16_t* val;
    int nnz;
    void* y;
    int ldy;
    int y_bf16;
    uint32_t magic;   // kF16Magic
    // 8-bit scales (scale8 non-null): E4M3 codes, the matrix exponent and
    // the fp16 fallback list
    const uint8_t* scale8;
    const int* scale8_exp;
    const int* fb_row_ptr;
    const int* fb_col;
    const uint16_t* fb_val;
    int fb_cap;
    // x already in fp16 B-fragment order (k_x_frag, once per call; null: each
    // CTA converts its own x blocks), and the device status word
    const unsigned char* xfrag;
    int* status;
    // shared-memory layout with xfrag (host-computed, xpre_layout): two x
    // buffers of xg groups each, then the parameters of all the split's
    // groups at xp_off, the split-K slots at xslot_off, two mbarriers at xbar_off
    int xg, xp_off, xslot_off, xbar_off;
};

__device__ __forceinline__ int x_row(const Problem& p, int m) { return p.rowmap ? p.rowmap[m] / p.xdiv : m; }
__device__ __forceinline__ int y_row(const Problem& p, int m) { return p.rowmap ? p.rowmap[m] : m; }

// MP = padded token count (1, 2, 4, 8, 16, 32 or 64): the staged-x layout
// [group][step][token < MP][t < 4] (8 bytes each) has compile-time strides.
template <int BITS, int G, int MP>
struct Cfg {
    static constexpr int NC = G / 4;
    static constexpr int NW = Chunk<BITS, G>::NW;
    static constexpr int STEPS = G / 16;
    static constexpr int NT = (MP + 7) / 8;                       // n8 token tiles
    static constexpr int NTOK = 8 * NT;
    // prefetch depth (groups) of the register ring: 8-word chunks (8 bits,
    // group 128) take 2; a group of 32 is a quarter of a 128-group's bytes,
    // so its ring is deeper (16 one-word chunks, 8 two-word chunks or 2-bit
    // groups, whose codebooks ride the ring) to keep as many bytes in flight
    static constexpr int D_CLAMP = G == 32 ? (MP <= 16 ? (BITS == 2 || NW > 1 ? 8 : 16) : 4)
                                           : ((MP <= 16 && NW < 8) ? 4 : 2);
    static constexpr int TSTRIDE = 32;                            // bytes per token per step
    static constexpr int SSTRIDE = MP * TSTRIDE;                  // bytes per step
    static constexpr int GSTRIDE = STEPS * SSTRIDE;               // bytes per group
    static constexpr int RED_BYTES = kRowsPerCta * NTOK * 4;     // this CTA's partial sums [64 rows][NTOK]
    // split-K slots: rank r receives [S][ceil(64/S)][NTOK] partials of its rows (S <= 8)
    static constexpr int SLOT_BYTES = (kRowsPerCta + 8) * NTOK * 4;
    static constexpr int XS_BUDGET = 49152 - SLOT_BYTES;
    // affine widths stage the tile's group parameters beside x: one 32-bit
    // word (fp16 scale | zero-point << 16) per row and group
    static constexpr int PSTRIDE = BITS == 2 ? 0 : kRowsPerCta * 4;
    static constexpr int BSTRIDE = GSTRIDE + PSTRIDE;             // block bytes per group
    static constexpr int D = D_CLAMP < XS_BUDGET / BSTRIDE ? D_CLAMP : XS_BUDGET / BSTRIDE;
    static constexpr int XG = (XS_BUDGET / BSTRIDE) / D * D;      // groups per x block
    static_assert(XG >= D, "x block smaller than the prefetch ring");
    // dynamic shared memory for a split of gpsplit groups: the x block, the
    // parameter block (both reused for the partial sums after the main loop),
    // then the split-K slots, which other ranks may write while this CTA
    // still reads x
    __host__ __device__ static int prm_offset(int gpsplit) { return (gpsplit < XG ? gpsplit : XG) * GSTRIDE; }
    __host__ __device__ static int slot_offset(int gpsplit)
    {
        const int xs = (gpsplit < XG ? gpsplit : XG) * BSTRIDE;
        return ((xs > RED_BYTES ? xs : RED_BYTES) + 15) / 16 * 16;
    }
    // the mbarrier of the x-block bulk copies, after the slots
    __host__ __device__ static int mbar_offset(int gpsplit, int S) { return slot_offset(gpsplit) + (S > 1 ? SLOT_BYTES : 0); }
    static int smem(int gpsplit, int S) { return mbar_offset(gpsplit, S) + 16; }
};

// One x item (token m, thread slot t of one group): the thread's NC
// contiguous bf16 values at xr, converted to fp16 and stored as STEPS 8-byte
// entries at dst + s * SSTRIDE, each holding the 4 values whose k positions
// match the A-fragment codes of thread t in step s.  16-byte loads when xr
// is 16-byte aligned.
template <int BITS, int G, int MP, typename Dst>
__device__ __forceinline__ void x_frag_item(const __nv_bfloat16* xr, Dst* dst)
{
    using C = Cfg<BITS, G, MP>;
    constexpr int NV = C::NC / 2;
    uint32_t v[NV];
    if ((reinterpret_cast<uintptr_t>(xr) & 15u) == 0) {
#pragma unroll
        for (int i = 0; i < C::NC / 8; i++) {
            const uint4 q = __ldg(reinterpret_cast<const uint4*>(xr) + i);
            v[4 * i] = q.x; v[4 * i + 1] = q.y; v[4 * i + 2] = q.z; v[4 * i + 3] = q.w;
        }
    } else {
        const unsigned short* x16 = reinterpret_cast<const unsigned short*>(xr);
#pragma unroll
        for (int i = 0; i < NV; i++)
            v[i] = (uint32_t)__ldg(x16 + 2 * i) | ((uint32_t)__ldg(x16 + 2 * i + 1) << 16);
    }
    auto f16 = [&](int c) -> uint32_t {   // bf16 -> fp32 (exact) -> fp16
        const uint32_t bits = (c & 1) ? (v[c >> 1] & 0xFFFF0000u) : (v[c >> 1] << 16);
        return __half_as_ushort(__float2half_rn(__uint_as_float(bits)));
    };
    static_for<0, C::STEPS>([&](auto sc) {
        constexpr int s = decltype(sc)::value;
        constexpr PairE e0 = plan_entry(BITS, C::NC, 2 * s);
        constexpr PairE e1 = plan_entry(BITS, C::NC, 2 * s + 1);
        *reinterpret_cast<uint2*>(reinterpret_cast<unsigned char*>(dst) + s * C::SSTRIDE) =
            make_uint2(f16(e0.lo) | (f16(e0.hi) << 16), f16(e1.lo) | (f16(e1.hi) << 16));
    });
}

// Stage x[:, kbase : kbase + ngr*G] as fp16 in MMA B-fragment order: the
// 8-byte entry (group, step, token m, t) holds the 4 values of token m whose k
// positions match the A-fragment codes of thread t in that step.  One item
// = (group, token, t).  Tokens M..MP-1 are not written: the MMA columns that
// read them are never stored.
template <int BITS, int G, int MP>
__device__ void stage_x(const Problem& a, int kbase, int ngr, unsigned char* xs, int nthr)
{
    using C = Cfg<BITS, G, MP>;
    const int M = a.M;
    const int items = ngr * M * 4;
    for (int it = threadIdx.x; it < items; it += nthr) {
        const int t = it & 3, m = (it >> 2) % M, gi = (it >> 2) / M;
        const __nv_bfloat16* xr = a.x + (size_t)x_row(a, m) * a.ldx + kbase + gi * G + t * C::NC;
        x_frag_item<BITS, G, MP>(xr, xs + (size_t)gi * C::GSTRIDE + m * C::TSTRIDE + t * 8);
    }
}

// An x block from the fragment-order copy of x (a.xfrag, written once per
// call by k_x_frag in exactly the staged layout, group after group): one
// bulk copy by thread 0 into buffer xs, completing on mbarrier bar.
template <int BITS, int G, int MP>
__device__ __forceinline__ void x_bulk_issue(const Problem& a, int g0, int ngr, unsigned char* xs, uint32_t bar)
{
    using C = Cfg<BITS, G, MP>;
    const uint32_t bytes = (uint32_t)ngr * C::GSTRIDE;
    ptx::fence_proxy_async();   // the buffer's earlier generic accesses before the async write
    ptx::mbar_expect_tx(bar, bytes);
    ptx::bulk_load(ptx::smem_u32(xs), a.xfrag + (size_t)g0 * C::GSTRIDE, bytes, bar);
}

// Every thread waits for the copy on bar (bounded; a wait that gives up sets
// the status word and the kernel carries on, so that no thread leaves a
// barrier the others reach).
__device__ __forceinline__ void x_bulk_wait(const Problem& a, uint32_t bar, uint32_t& phase)
{
    if (!ptx::mbar_wait(bar, phase) && a.status) atomicExch(a.status, (int)QG_ERR_TIMEOUT);
    phase ^= 1u;
}

// Programmatic dependent launch.  The dense decode kernels are launched with
// programmatic stream serialization, so that the next one can be resident and
// have its first weight groups in registers while this one drains: a kernel
// reads only weight data (codes, group parameters, outlier CSR) before
// griddepcontrol.wait, which returns once the grids it depends on have
// completed and their writes are visible; x and y are touched only after it.
// The kernel immediately preceding a decode product on its stream therefore
// must not write that product's weights (the quantizer ends with an empty
// kernel for this reason).  Dependents are released when the main loop starts.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_release() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// x [M, K] to fp16 B-fragment order for every group, tokens padded to MP
// with zeros: entry (group, step, token, t) at group * GSTRIDE + step *
// SSTRIDE + token * TSTRIDE + t * 8, the layout a decode CTA stages.  It lets
// dependents launch at once (their weight loads overlap this kernel) and
// waits for the kernel that wrote x before reading it.
template <int BITS, int G, int MP>
__global__ void __launch_bounds__(256) k_x_frag(const __nv_bfloat16* __restrict__ x, int ldx, int M, int K,
                                                unsigned char* __restrict__ out)
{
    using C = Cfg<BITS, G, MP>;
    pdl_release();
    pdl_wait();
    const long long items = (long long)(K / G) * MP * 4;
    for (long long it = (long long)blockIdx.x * blockDim.x + threadIdx.x; it < items;
         it += (long long)gridDim.x * blockDim.x) {
        const int t = (int)(it & 3), m = (int)((it >> 2) % MP), gi = (int)((it >> 2) / MP);
        unsigned char* dst = out + (size_t)gi * C::GSTRIDE + m * C::TSTRIDE + t * 8;
        if (m < M) {
            x_frag_item<BITS, G, MP>(x + (size_t)m * ldx + gi * G + t * C::NC, dst);
        } else {
#pragma unroll
            for (int s = 0; s < C::STEPS; s++) *reinterpret_cast<uint2*>(dst + s * C::SSTRIDE) = make_uint2(0u, 0u);
        }
    }
}

// Stage the scale and zero-point of the tile's 64 rows for the ngr groups
// starting at matrix group g0, one 32-bit word per (group, row): fp16 scale
// bits | zero-point << 16, at word (gi * kWarps + row / 16) * 16 + (row % 8) * 2
// + (row / 8) % 2.  The rows r and r + 8 of a thread are adjacent (one 8-byte
// shared load per group), and a warp reads 32 contiguous bytes.  Read from
// global memory as 16-byte runs of 8 groups of a row where the layout allows,
// else one group at a time.  (Loading the parameters per group inside the
// streaming loop touched 8 rows' sectors per load and kept the L1 data path
// busy; staged, they cost a few wavefronts per CTA and group.)
template <int BITS, int G>
__device__ void stage_prm(const Problem& a, int tile, int g0, int ngr, uint32_t* ps, int nthr)
{
    const int ng = a.K / G;
    auto word = [](int gi, int rl) { return (gi * kWarps + rl / 16) * 16 + (rl % 8) * 2 + (rl / 8) % 2; };
    if (a.scale8) {   // 8-bit scales: each group's fp16 scale bits from its code
        const ScaleSrc sc{a.scale, a.scale8, a.scale8_exp, a.fb_row_ptr, a.fb_col, a.fb_val, a.fb_cap};
        const int E = __ldg(a.scale8_exp);
        for (int it = threadIdx.x; it < kRowsPerCta * ngr; it += nthr) {
            const int rl = it % kRowsPerCta, gi = it / kRowsPerCta;
            const int n = min(tile * kRowsPerCta + rl, a.N - 1);
            const size_t idx = (size_t)n * ng + g0 + gi;
            const uint32_t c = __ldg(a.scale8 + idx);
            ps[word(gi, rl)] = scale8_bits(sc, E, n, g0 + gi, c) | ((uint32_t)__ldg(a.zp + idx) << 16);
        }
        return;
    }
    const bool vec = ng % 8 == 0 && g0 % 8 == 0 && (reinterpret_cast<uintptr_t>(a.scale) & 15u) == 0 &&
                     (reinterpret_cast<uintptr_t>(a.zp) & 7u) == 0;
    if (vec) {
        const int nch = (ngr + 7) / 8;
        for (int it = threadIdx.x; it < kRowsPerCta * nch; it += nthr) {
            const int rl = it % kRowsPerCta, c = it / kRowsPerCta;
            const int n = min(tile * kRowsPerCta + rl, a.N - 1);
            const size_t base = (size_t)n * ng + g0 + 8 * c;   // a multiple of 8, and base + 8 <= (n + 1) * ng
            const uint4 sv = __ldg(reinterpret_cast<const uint4*>(a.scale + base));
            const uint2 zv = __ldg(reinterpret_cast<const uint2*>(a.zp + base));
            const uint32_t sw[4] = {sv.x, sv.y, sv.z, sv.w};
            const uint32_t zw[2] = {zv.x, zv.y};
#pragma unroll
            for (int j = 0; j < 8; j++) {
                if (8 * c + j < ngr)
                    ps[word(8 * c + j, rl)] = ((sw[j / 2] >> (16 * (j & 1))) & 0xFFFFu) |
                                              (((zw[j / 4] >> (8 * (j & 3))) & 0xFFu) << 16);
            }
        }
    } else {
        for (int it = threadIdx.x; it < kRowsPerCta * ngr; it += nthr) {
            const int rl = it % kRowsPerCta, gi = it / kRowsPerCta;
            const int n = min(tile * kRowsPerCta + rl, a.N - 1);
            const size_t idx = (size_t)n * ng + g0 + gi;
            ps[word(gi, rl)] = (uint32_t)__ldg(a.scale + idx) | ((uint32_t)__ldg(a.zp + idx) << 16);
        }
    }
}

// One group of two weight rows (w0: row r0, w1: row r1 of the thread's
// A-fragment rows, NW words each) against the staged x block of that group:
// dequantize to fp16 MMA operands and accumulate into yacc.  pr holds the
// rows' parameters: affine (scale bits, zero-point), codebook (two words of
// four fp16 entries).
template <int BITS, int G, int MP>
__device__ __forceinline__ void mma_group(const uint32_t (&w0)[Chunk<BITS, G>::NW], const uint32_t (&w1)[Chunk<BITS, G>::NW],
                                          const uint32_t (&pr)[2][2],
                                          const unsigned char* const (&xg)[Cfg<BITS, G, MP>::NT],
                                          float (&yacc)[Cfg<BITS, G, MP>::NT][4], uint32_t magic)
{
    using C = Cfg<BITS, G, MP>;
    constexpr int NW = C::NW, NT = C::NT;
    if constexpr (BITS == 2) {
        // per-row lookup tables: low bytes and high bytes of the 4 entries
        const uint32_t L0 = __byte_perm(pr[0][0], pr[0][1], 0x6420);
        const uint32_t H0 = __byte_perm(pr[0][0], pr[0][1], 0x7531);
        const uint32_t L1 = __byte_perm(pr[1][0], pr[1][1], 0x6420);
        const uint32_t H1 = __byte_perm(pr[1][0], pr[1][1], 0x7531);
        if constexpr (C::NC == 8) {
            // an 8-code chunk (group 32) fills two bytes: step s takes codes
            // (s, s+4) from bit 2s of bytes 0 and 1 and (s+2, s+6) from bit
            // 2s + 4, moved into bytes 2 and 3
            static_for<0, 2>([&](auto sc) {
                constexpr int s = decltype(sc)::value;
                const uint32_t f0 = ((w0[0] >> (2 * s)) & 0x0303u) | ((w0[0] << (12 - 2 * s)) & 0x03030000u);
                const uint32_t f1 = ((w1[0] >> (2 * s)) & 0x0303u) | ((w1[0] << (12 - 2 * s)) & 0x03030000u);
                const uint32_t s0l = f0 * 0x11u + 0x4040u, s0h = __umulhi(f0, 0x00110000u) + 0x4040u;
                const uint32_t s1l = f1 * 0x11u + 0x4040u, s1h = __umulhi(f1, 0x00110000u) + 0x4040u;
                const uint32_t a0 = __byte_perm(L0, H0, s0l), a2 = __byte_perm(L0, H0, s0h);
                const uint32_t a1 = __byte_perm(L1, H1, s1l), a3 = __byte_perm(L1, H1, s1h);
#pragma unroll
                for (int nt = 0; nt < NT; nt++) {
                    const uint2 b = *reinterpret_cast<const uint2*>(xg[nt] + s * C::SSTRIDE);
                    mma16816(yacc[nt], a0, a1, a2, a3, b.x, b.y);
                }
            });
            return;
        }
        static_for<0, NW>([&](auto wc) {
            constexpr int wi = decltype(wc)::value;
            static_for<0, 4>([&](auto jc) {
                constexpr int jf = decltype(jc)::value;
                const uint32_t f0 = (w0[wi] >> (2 * jf)) & 0x03030303u;
                const uint32_t f1 = (w1[wi] >> (2 * jf)) & 0x03030303u;
                const uint32_t s0l = f0 * 0x11u + 0x4040u, s0h = __umulhi(f0, 0x00110000u) + 0x4040u;
                const uint32_t s1l = f1 * 0x11u + 0x4040u, s1h = __umulhi(f1, 0x00110000u) + 0x4040u;
                const uint32_t a0 = __byte_perm(L0, H0, s0l), a2 = __byte_perm(L0, H0, s0h);
                const uint32_t a1 = __byte_perm(L1, H1, s1l), a3 = __byte_perm(L1, H1, s1h);
                constexpr int s = 4 * wi + jf;   // entries 2s (lo) and 2s+1 (hi)
#pragma unroll
                for (int nt = 0; nt < NT; nt++) {
                    const uint2 b = *reinterpret_cast<const uint2*>(xg[nt] + s * C::SSTRIDE);
                    mma16816(yacc[nt], a0, a1, a2, a3, b.x, b.y);
                }
            });
        });
    } else {
        float acc[NT][4];
#pragma unroll
        for (int i = 0; i < NT; i++) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;
        const uint32_t z0 = pr[0][1], z1 = pr[1][1];
        static_for<0, C::STEPS>([&](auto sc) {
            constexpr int s = decltype(sc)::value;
            const uint32_t a0 = deq_affine<BITS, C::NC, 2 * s>(w0, z0, magic);
            const uint32_t a1 = deq_affine<BITS, C::NC, 2 * s>(w1, z1, magic);
            const uint32_t a2 = deq_affine<BITS, C::NC, 2 * s + 1>(w0, z0, magic);
            const uint32_t a3 = deq_affine<BITS, C::NC, 2 * s + 1>(w1, z1, magic);
#pragma unroll
            for (int nt = 0; nt < NT; nt++) {
                const uint2 b = *reinterpret_cast<const uint2*>(xg[nt] + s * C::SSTRIDE);
                mma16816(acc[nt], a0, a1, a2, a3, b.x, b.y);
            }
        });
        const float s0 = h2f((uint16_t)pr[0][0]), s1 = h2f((uint16_t)pr[1][0]);
#pragma unroll
        for (int nt = 0; nt < NT; nt++) {
            yacc[nt][0] = fmaf(s0, acc[nt][0], yacc[nt][0]);
            yacc[nt][1] = fmaf(s0, acc[nt][1], yacc[nt][1]);
            yacc[nt][2] = fmaf(s1, acc[nt][2], yacc[nt][2]);
            yacc[nt][3] = fmaf(s1, acc[nt][3], yacc[nt][3]);
        }
    }
}


// Cluster barrier in two halves, and an fp32 add into another CTA's shared
// memory (distributed shared memory of the thread-block cluster).
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void st_cluster_v4(const void* local_addr, int rank, float4 v)
{
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local_addr));
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(r), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
                 : "memory");
}

// Cursor over the FP16 outliers a thread adds back: two threads per tile row
// (threads 2r, 2r+1 take row r; threads beyond the 64 rows take none), and
// the S CTAs of a cluster take every S-th pair of the row's CSR entries, so
// the add-back is spread over every thread of the cluster.  init() reads the
// CSR bounds, fetch() the first OU entries; only the x values they multiply
// are read after the main loop.
struct OutCursor {
    static constexpr int OU = 4;
    int p, end, row, stride;
    int col[OU];
    uint32_t val[OU];
    __device__ __forceinline__ void init(const Problem& a, int splits, int tile)
    {
        row = (int)(threadIdx.x >> 1);
        stride = 2 * splits;
        p = 0;
        end = 0;
#pragma unroll
        for (int u = 0; u < OU; u++) {
            col[u] = -1;
            val[u] = 0u;
        }
        const int n = tile * kRowsPerCta + row;
        if (a.nnz > 0 && threadIdx.x < 2 * kRowsPerCta && n < a.N) {
            p = __ldg(a.row_ptr + n) + 2 * (int)blockIdx.y + (int)(threadIdx.x & 1);
            end = __ldg(a.row_ptr + n + 1);
        }
    }
    __device__ __forceinline__ void fetch(const Problem& a)
    {
#pragma unroll
        for (int u = 0; u < OU; u++) {
            const int q = p + u * stride;
            col[u] = q < end ? __ldg(a.col + q) : -1;
            val[u] = q < end ? __ldg(a.val + q) : 0u;
        }
    }
};

// Split-K reduction, outlier add-back and store of one 64-row tile; every
// thread of the CTA calls it (threads of warps >= kWarps contribute no
// partial sums).  yacc holds the thread's MMA accumulators of the tile; the
// x block at the start of shared memory is reused for the partial sums, and
// the split-K slots start at byte slot_off.
template <int BITS, int G, int MP>
__device__ __forceinline__ void tile_epilogue(const Problem& a, int splits, int slot_off, int tile,
                                              const float (&yacc)[Cfg<BITS, G, MP>::NT][4], OutCursor& oc)
{
    using C = Cfg<BITS, G, MP>;
    constexpr int NT = C::NT;
    extern __shared__ __align__(16) unsigned char smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = lane & 3, gq = lane >> 2;
    const int S = splits;
    // ------------------------------------------------ split-K reduction + epilogue
    // Partial sums of the tile go to shared memory (the x block is dead now)
    // and the CTA's share of the outliers is added to them.  With a K split,
    // rank r owns rows [r*64/S, (r+1)*64/S): every rank writes its partials of
    // those rows into its own slot in rank r's shared memory (plain 16-byte
    // remote stores), and after one cluster barrier the owner adds the S
    // slots and stores its rows.
    const int Mv = min(a.M, MP);
    __syncthreads();
    float* const yp = reinterpret_cast<float*>(smem);   // [64 rows][NTOK]
    const int rl0 = warp * 16 + gq;
#pragma unroll
    for (int nt = 0; nt < NT; nt++) {
        if (warp >= kWarps) break;   // a producer warp holds no partial sums
        const int c = nt * 8 + 2 * t;
        yp[rl0 * C::NTOK + c] = yacc[nt][0];
        yp[rl0 * C::NTOK + c + 1] = yacc[nt][1];
        yp[(rl0 + 8) * C::NTOK + c] = yacc[nt][2];
        yp[(rl0 + 8) * C::NTOK + c + 1] = yacc[nt][3];
    }
    __syncthreads();
    for (int p = oc.p;;) {
        if (oc.col[0] < 0) break;   // entries fill the slots in order
        // tokens four at a time, so that all the x loads of a round are in flight together
        constexpr int OM = MP < 4 ? MP : 4;
        for (int mb = 0; mb < Mv; mb += OM) {
            float xv[OM][OutCursor::OU];
#pragma unroll
            for (int i = 0; i < OM; i++) {
                const int m = mb + i;
                const __nv_bfloat16* xm = a.x + (size_t)x_row(a, min(m, Mv - 1)) * a.ldx;
#pragma unroll
                for (int u = 0; u < OutCursor::OU; u++) xv[i][u] = (m < Mv && oc.col[u] >= 0) ? __bfloat162float(xm[oc.col[u]]) : 0.0f;
            }
#pragma unroll
            for (int i = 0; i < OM; i++) {
                float sum = 0.0f;
#pragma unroll
                for (int u = 0; u < OutCursor::OU; u++) sum = fmaf(xv[i][u], h2f((uint16_t)oc.val[u]), sum);
                if (mb + i < Mv) atomicAdd(&yp[oc.row * C::NTOK + mb + i], sum);
            }
        }
        p += OutCursor::OU * oc.stride;
        if (p >= oc.end) break;
#pragma unroll
        for (int u = 0; u < OutCursor::OU; u++) {
            const int q = p + u * oc.stride;
            oc.col[u] = q < oc.end ? __ldg(a.col + q) : -1;
            oc.val[u] = q < oc.end ? __ldg(a.val + q) : 0u;
        }
    }
    __syncthreads();
    const int rows_cap = (kRowsPerCta + S - 1) / S;
    const float* slots = reinterpret_cast<const float*>(smem + slot_off);   // [S][rows_cap][NTOK]
    if (S > 1) {
        const int me = (int)cluster_rank();
        constexpr int Q = C::NTOK / 4;   // float4 per row
        for (int j = threadIdx.x; j < kRowsPerCta * Q; j += blockDim.x) {
            const int rl = j / Q, c4 = j % Q;
            const int owner = (S * (rl + 1) - 1) / kRowsPerCta;
            const int lr = rl - owner * kRowsPerCta / S;
            const float4 v = *reinterpret_cast<const float4*>(yp + rl * C::NTOK + 4 * c4);
            st_cluster_v4(slots + ((size_t)(me * rows_cap + lr) * C::NTOK + 4 * c4), owner, v);
        }
        cluster_arrive();
        cluster_wait();
    }
    const int rank = S > 1 ? (int)cluster_rank() : 0;
    const int row_lo = rank * kRowsPerCta / S, rows_per = (rank + 1) * kRowsPerCta / S - row_lo;
    for (int it = threadIdx.x; it < rows_per * Mv; it += blockDim.x) {
        const int m = it / rows_per, lr = it % rows_per, rl = row_lo + lr;
        const int n = tile * kRowsPerCta + rl;
        if (n < a.N) {
            float v;
            if (S > 1) {
                v = 0.0f;
                for (int r = 0; r < S; r++) v += slots[(size_t)(r * rows_cap + lr) * C::NTOK + m];
            } else {
                v = yp[rl * C::NTOK + m];
            }
            const size_t yo = (size_t)y_row(a, m) * a.ldy + n;
            if (a.y_bf16)
                reinterpret_cast<__nv_bfloat16*>(a.y)[yo] = __float2bfloat16_rn(v);
            else
                reinterpret_cast<float*>(a.y)[yo] = v;
        }
    }
}

template <int BITS, int G, int MP>
__device__ __forceinline__ void gemv_body(const Problem& a, int splits, int gpsplit, int tile)
{
    using C = Cfg<BITS, G, MP>;
    constexpr int NW = C::NW, D = C::D, NT = C::NT;
    constexpr int GB = G * BITS / 8;   // packed bytes per group
    constexpr int CB = Chunk<BITS, G>::CB;
    extern __shared__ __align__(16) unsigned char smem[];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = lane & 3, gq = lane >> 2;
    const uint32_t magic = a.magic;
    const int row_base = tile * kRowsPerCta + warp * 16 + gq;
    const int r0 = min(row_base, a.N - 1), r1 = min(row_base + 8, a.N - 1);
    const int ng = a.K / G;
    const int g_begin = blockIdx.y * gpsplit;
    const int ngrp = max(0, min(ng, g_begin + gpsplit) - g_begin);

    // streaming pointers of this thread, advanced by D groups per iteration
    const size_t rowbytes = (size_t)a.K * BITS / 8;
    const uint8_t* p0 = a.packed + (size_t)r0 * rowbytes + (size_t)g_begin * GB + t * CB;
    const uint8_t* p1 = a.packed + (size_t)r1 * rowbytes + (size_t)g_begin * GB + t * CB;
    const size_t pidx0 = (size_t)r0 * ng + g_begin, pidx1 = (size_t)r1 * ng + g_begin;
    const uint2* cq0 = a.cb + pidx0;
    const uint2* cq1 = a.cb + pidx1;
    // x from the fragment-order copy (xpre): double-buffered x blocks of a.xg
    // groups and every group's parameters staged once; else x blocks of XG
    // groups converted by the CTA, parameters staged per block
    const bool xpre = a.xfrag != nullptr;
    const int XGB = xpre ? a.xg : C::XG;
    const int poff = xpre ? a.xp_off : C::prm_offset(gpsplit);
    // affine: the staged group parameters, this thread's words of block group 0
    const uint32_t* const ps = reinterpret_cast<const uint32_t*>(smem + poff) + warp * 16 + gq * 2;

    const bool odd_chunk = ((t * CB) & 4) != 0;   // the chunk starts 4 bytes past an 8-byte boundary
    // this lane's B-fragment slot (token clamped to MP-1; its column is discarded)
    uint32_t xlo[NT];
#pragma unroll
    for (int nt = 0; nt < NT; nt++) xlo[nt] = min(nt * 8 + gq, MP - 1) * C::TSTRIDE + t * 8;

    float yacc[NT][4];
#pragma unroll
    for (int i = 0; i < NT; i++) yacc[i][0] = yacc[i][1] = yacc[i][2] = yacc[i][3] = 0.0f;

    uint32_t wr[D][2][NW];
    uint32_t prm[D][2][2];   // group parameters: affine scale bits, zp; codebook two words of 4 fp16

    // load group (current base + REL) into ring slot SLOT (codebooks ride the
    // ring with the codes; affine parameters are staged per x block)
    auto issue = [&](auto slot_c, auto rel_c) {
        constexpr int SLOT = decltype(slot_c)::value, REL = decltype(rel_c)::value;
        if constexpr (Chunk<BITS, G>::SHUF) {
            Chunk<BITS, G>::load_words(p0 + REL * GB, t, wr[SLOT][0]);
            Chunk<BITS, G>::load_words(p1 + REL * GB, t, wr[SLOT][1]);
        } else {
            Chunk<BITS, G>::load(p0 + REL * GB, wr[SLOT][0]);
            Chunk<BITS, G>::load(p1 + REL * GB, wr[SLOT][1]);
        }
        if constexpr (BITS == 2) {
            const uint2 c0 = __ldg(cq0 + REL), c1 = __ldg(cq1 + REL);
            prm[SLOT][0][0] = c0.x; prm[SLOT][0][1] = c0.y;
            prm[SLOT][1][0] = c1.x; prm[SLOT][1][1] = c1.y;
        }
    };
    auto advance = [&]() {
        p0 += D * GB; p1 += D * GB;
        if constexpr (BITS == 2) { cq0 += D; cq1 += D; }
    };

    static_for<0, D>([&](auto dc) {
        constexpr int d = decltype(dc)::value;
        if (d < ngrp) issue(dc, dc);
    });

    OutCursor oc;
    oc.init(a, splits, tile);

    // xpre: mbarriers of the two x buffers
    const uint32_t xbar0 = ptx::smem_u32(smem + (xpre ? a.xbar_off : 0));
    uint32_t xph[2] = {0u, 0u};
    int xcur = 0;   // buffer of the current x block
    auto xbuf = [&](int b) { return smem + (size_t)b * XGB * C::GSTRIDE; };
    if (xpre) {
        if (threadIdx.x == 0) {
            ptx::mbar_init(xbar0, 1);
            ptx::mbar_init(xbar0 + 8, 1);
            ptx::fence_mbar_init();
        }
        __syncthreads();
    }

    uint32_t* const pblock = reinterpret_cast<uint32_t*>(smem + poff);
    if constexpr (BITS != 2)   // weight data: staged before the dependency wait
        if (ngrp > 0) stage_prm<BITS, G>(a, tile, g_begin, xpre ? ngrp : min(C::XG, ngrp), pblock, blockDim.x);

    pdl_wait();   // weight loads are in flight; x may come from the preceding kernel
    if (ngrp > 0) {
        if (xpre) {
            if (threadIdx.x == 0) {
                x_bulk_issue<BITS, G, MP>(a, g_begin, min(XGB, ngrp), xbuf(0), xbar0);
                if (ngrp > XGB) x_bulk_issue<BITS, G, MP>(a, g_begin + XGB, min(XGB, ngrp - XGB), xbuf(1), xbar0 + 8);
            }
            x_bulk_wait(a, xbar0, xph[0]);
        } else {
            stage_x<BITS, G, MP>(a, g_begin * G, min(C::XG, ngrp), smem, blockDim.x);
        }
    }
    __syncthreads();
    oc.fetch(a);

    // dependents may launch now: every CTA of this grid has started, and a
    // dependent CTA cannot pass its own dependency wait (so cannot release the
    // grid after it) before this grid has finished; its weight loads overlap
    // this grid's main loop and tail (about 2 % on the 70B stack against
    // releasing after the main loop)
    pdl_release();

    int xnext = XGB;        // group index (relative) at which the next x block starts
    uint32_t xoff = 0;      // byte offset of group jj inside the shared memory of x
    int pw = 0;             // word offset of group jj inside the parameter block
    for (int jj = 0; jj < ngrp; jj += D) {
        if (jj == xnext) {
            __syncthreads();
            if (xpre) {
                // the finished buffer takes the block after next; the next one
                // was copied during the previous block
                if (threadIdx.x == 0 && jj + XGB < ngrp)
                    x_bulk_issue<BITS, G, MP>(a, g_begin + jj + XGB, min(XGB, ngrp - jj - XGB), xbuf(xcur),
                                              xbar0 + 8 * xcur);
                xcur ^= 1;
                x_bulk_wait(a, xbar0 + 8 * xcur, xph[xcur]);
                xoff = (uint32_t)(xcur * XGB * C::GSTRIDE);
            } else {
                stage_x<BITS, G, MP>(a, (g_begin + jj) * G, min(C::XG, ngrp - jj), smem, blockDim.x);
                if constexpr (BITS != 2) stage_prm<BITS, G>(a, tile, g_begin + jj, min(C::XG, ngrp - jj), pblock, blockDim.x);
                __syncthreads();
                xoff = 0;
                pw = 0;
            }
            xnext += XGB;
        }
        const unsigned char* xb[NT];
#pragma unroll
        for (int nt = 0; nt < NT; nt++) xb[nt] = smem + xoff + xlo[nt];
        if constexpr (BITS != 2 && G != 32) {
            static_for<0, D>([&](auto dc) {
                constexpr int d = decltype(dc)::value;
                if (jj + d < ngrp) {   // only staged groups lie inside the block
                    const uint2 v = *reinterpret_cast<const uint2*>(ps + pw + d * kWarps * 16);
                    prm[d][0][0] = v.x; prm[d][0][1] = v.x >> 16;
                    prm[d][1][0] = v.y; prm[d][1][1] = v.y >> 16;
                }
            });
        }

        static_for<0, D>([&](auto dc) {
            constexpr int d = decltype(dc)::value;
            if (jj + d < ngrp) {
                {
                    const unsigned char* xg[NT];
#pragma unroll
                    for (int nt = 0; nt < NT; nt++) xg[nt] = xb[nt] + d * C::GSTRIDE;
                    if constexpr (BITS != 2 && G == 32) {
                        // group 32: the group's parameters straight from the
                        // staged block (a ring of them would not fit in registers)
                        const uint2 v = *reinterpret_cast<const uint2*>(ps + pw + d * kWarps * 16);
                        const uint32_t pg[2][2] = {{v.x, v.x >> 16}, {v.y, v.y >> 16}};
                        if constexpr (Chunk<BITS, G>::SHUF) {
                            uint32_t s0[NW], s1[NW];
                            Chunk<BITS, G>::assemble(wr[d][0], s0, lane);
                            Chunk<BITS, G>::assemble(wr[d][1], s1, lane);
                            mma_group<BITS, G, MP>(s0, s1, pg, xg, yacc, magic);
                        } else {
                            mma_group<BITS, G, MP>(wr[d][0], wr[d][1], pg, xg, yacc, magic);
                        }
                    } else if constexpr (BITS == 2 && Chunk<BITS, G>::SHUF) {
                        uint32_t s0[NW], s1[NW];
                        Chunk<BITS, G>::assemble(wr[d][0], s0, lane);
                        Chunk<BITS, G>::assemble(wr[d][1], s1, lane);
                        mma_group<BITS, G, MP>(s0, s1, prm[d], xg, yacc, magic);
                    } else if constexpr (Chunk<BITS, G>::SPLIT) {
                        uint32_t s0[NW], s1[NW];
                        Chunk<BITS, G>::order(wr[d][0], s0, odd_chunk);
                        Chunk<BITS, G>::order(wr[d][1], s1, odd_chunk);
                        mma_group<BITS, G, MP>(s0, s1, prm[d], xg, yacc, magic);
                    } else {
                        mma_group<BITS, G, MP>(wr[d][0], wr[d][1], prm[d], xg, yacc, magic);
                    }
                }
                if (jj + d + D < ngrp) issue(dc, std::integral_constant<int, D + d>{});
            }
        });
        advance();
        xoff += D * C::GSTRIDE;
        pw += D * kWarps * 16;
    }

    tile_epilogue<BITS, G, MP>(a, splits, xpre ? a.xslot_off : C::slot_offset(gpsplit), tile, yacc, oc);
}

template <int BITS, int G, int MP>
__global__ void __launch_bounds__(kWarps * 32) k_gemv(const Problem p, int splits, int gpsplit)
{
    gemv_body<BITS, G, MP>(p, splits, gpsplit, blockIdx.x);
}

// Several products that share x, M and K (and bits and group) in one launch:
// the row tiles of product q are blocks [tile_start[q], tile_start[q + 1])
// of the grid's x dimension; every tile runs the decode body on its product.
constexpr int kMultiMax = 4;
struct MultiTable {
    Problem p[kMultiMax];
    int tile_start[kMultiMax + 1];
    int n;
};

template <int BITS, int G, int MP>
__global__ void __launch_bounds__(kWarps * 32) k_gemv_multi(const __grid_constant__ MultiTable t, int splits,
                                                            int gpsplit)
{
    int q = 0;
    while (q + 1 < t.n && (int)blockIdx.x >= t.tile_start[q + 1]) q++;
    gemv_body<BITS, G, MP>(t.p[q], splits, gpsplit, (int)blockIdx.x - t.tile_start[q]);
}

// Grouped product over routed experts.  Pairs (token, slot) are sorted by
// expert on the device (offsets[e] .. offsets[e+1] index `perm`, which holds
// pair ids t*k + j).  The routing kernel also lists the work items
// (expert, chunk of `chunk` pairs); blockIdx.z picks one item.
struct MoeTable {
    const __nv_bfloat16* x;
    int ldx, N, K, topk;
    int chunk;
    const int* offsets;
    const int* perm;
    const int2* items;
    const int* n_items;
    void* y;
    int y_bf16;
    uint32_t magic;   // kF16Magic
    const uint8_t* packed[kMoeMaxExperts];
    const uint16_t* scale[kMoeMaxExperts];
    const uint8_t* zp[kMoeMaxExperts];
    const uint2* cb[kMoeMaxExperts];
    const int* row_ptr[kMoeMaxExperts];
    const int* col[kMoeMaxExperts];
    const uint16_t* val[kMoeMaxExperts];
    int nnz[kMoeMaxExperts];
    // 8-bit scales (all experts alike: scale8 null for none)
    const uint8_t* scale8[kMoeMaxExperts];
    const int* scale8_exp[kMoeMaxExperts];
    const int* fb_row_ptr[kMoeMaxExperts];
    const int* fb_col[kMoeMaxExperts];
    const uint16_t* fb_val[kMoeMaxExperts];
    int fb_cap[kMoeMaxExperts];
};

template <int BITS, int G, int MP>
__global__ void __launch_bounds__(kWarps * 32) k_gemv_moe(const __grid_constant__ MoeTable t, int splits,
                                                          int gpsplit)
{
    if ((int)blockIdx.z >= *t.n_items) return;   // uniform across the cluster (same blockIdx.z)
    const int2 item = t.items[blockIdx.z];
    const int e = item.x;
    const int end = t.offsets[e + 1];
    const int m0 = t.offsets[e] + item.y * t.chunk;
    Problem p;
    p.x = t.x; p.ldx = t.ldx; p.M = min(t.chunk, end - m0); p.N = t.N; p.K = t.K;
    p.rowmap = t.perm + m0; p.xdiv = t.topk;
    p.packed = t.packed[e]; p.scale = t.scale[e]; p.zp = t.zp[e]; p.cb = t.cb[e];
    p.row_ptr = t.row_ptr[e]; p.col = t.col[e]; p.val = t.val[e]; p.nnz = t.nnz[e];
    p.y = t.y; p.ldy = t.N; p.y_bf16 = t.y_bf16;
    p.magic = t.magic;
    p.scale8 = t.scale8[e]; p.scale8_exp = t.scale8_exp[e];
    p.fb_row_ptr = t.fb_row_ptr[e]; p.fb_col = t.fb_col[e]; p.fb_val = t.fb_val[e]; p.fb_cap = t.fb_cap[e];
    p.xfrag = nullptr;   // routed rows: each CTA gathers and converts its x blocks
    p.status = nullptr;
    gemv_body<BITS, G, MP>(p, splits, gpsplit, blockIdx.x);
}

// K split: the largest cluster size S (1..8) whose grid still runs as one
// wave at four CTAs per SM (the cap of clustered launches), keeping at least
// two groups per split; unsplit when even S = 2 does not fit.  The wide
// products of the 70B stack come out as before (gate/up unsplit at about
// three CTAs per SM, o and down 4-way, q/k/v 3-way); a small matrix gets the
// most splits that fit (4096 x 4096: 8 splits of 4 groups, where the earlier
// rule of about three CTAs per SM gave 7 uneven splits of up to 5 groups and
// measured 5 to 10 % slower).
inline int choose_splits(long long ctas_per_split, int ng)
{
    const long long fit = 4LL * num_sms();
    int S = 1;
    for (int s = 2; s <= 8; s++)
        if (ctas_per_split * s <= fit && ng / s >= 2) S = s;
    return S;
}

// Padded token count of a launch.
inline int mp_for(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : M <= 8 ? 8 : M <= 16 ? 16 : M <= 32 ? 32 : 64; }

// Opt a kernel in to `bytes` of dynamic shared memory on the current device
// (once per kernel and device).
template <typename K>
qg_status allow_smem(K kernel, int bytes)
{
    static std::mutex mu;
    static const void* done[64][8] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
    const void* key = reinterpret_cast<const void*>(kernel);
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < 8; i++) {
        if (done[dev][i] == key) return QG_OK;
        if (!done[dev][i]) {
            cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
            if (e != cudaSuccess) return cuda_fail(e, "kernel shared memory attribute");
            done[dev][i] = key;
            return QG_OK;
        }
    }
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    return e == cudaSuccess ? QG_OK : cuda_fail(e, "kernel shared memory attribute");
}

template <typename K, typename... A>
qg_status launch_cluster(K kernel, dim3 grid, int S, unsigned threads, size_t smem_bytes, bool pdl, cudaStream_t s,
                         A... args)
{
    if (smem_bytes > 48 * 1024) {
        qg_status st = allow_smem(kernel, 227 * 1024);
        if (st != QG_OK) return st;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem_bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)S;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl && dependent_launch_enabled() ? 2 : 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
    if (e != cudaSuccess) return cuda_fail(e, "decode kernel launch");
    return QG_OK;
}

// Dynamic shared memory of a decode launch, which also caps the CTAs an SM
// runs.  Clustered (K-split) launches are held to at most four CTAs per SM:
// cluster placement otherwise packed five CTAs onto some SMs while others ran
// two or three, and the crowded SMs set the launch's time.  Unsplit launches
// (about three CTAs per SM of their own) are held to three, so that the
// CTAs of a dependent launch, started early by programmatic dependent launch,
// take only the SMs this launch is leaving.
template <int BITS, int G, int MP>
size_t decode_smem(int gps, int S)
{
    const int need = Cfg<BITS, G, MP>::smem(gps, S);
    return (size_t)std::max(need, smem_for_cap(S > 1 ? 4 : 3));
}

// The fragment-order copy of x for products launched next (one per call,
// shared by the products of a fused call): k_x_frag with programmatic
// serialization, so that it overlaps the tail of the preceding product.
template <int BITS, int G, int MP>
qg_status launch_x_frag(const Problem& p, cudaStream_t s)
{
    const long long items = (long long)(p.K / G) * MP * 4;
    const int blocks = (int)std::max<long long>(1, std::min<long long>(ceil_div(items, 256), 2LL * num_sms()));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = dependent_launch_enabled() ? 1 : 0;
    cudaError_t e = cudaLaunchKernelEx(&cfg, k_x_frag<BITS, G, MP>, p.x, p.ldx, p.M, p.K,
                                       const_cast<unsigned char*>(p.xfrag));
    if (e != cudaSuccess) return cuda_fail(e, "x conversion kernel launch");
    return QG_OK;
}

// Shared-memory layout of a launch with the fragment-order copy of x, inside
// the per-SM cap's share: two x buffers of xg groups, the parameters of all
// gps groups, the split-K slots, two mbarriers.  Sets p's layout fields and
// returns the dynamic shared memory, or 0 if two buffers of D groups do not fit.
template <int BITS, int G, int MP>
size_t xpre_layout(int gps, int S, Problem& p)
{
    using C = Cfg<BITS, G, MP>;
    const int cap = smem_for_cap(S > 1 ? 4 : 3);
    const int pbytes = gps * C::PSTRIDE;
    const int slots = S > 1 ? C::SLOT_BYTES : 0;
    const int avail = cap - pbytes - slots - 32;
    int xg = avail > 0 ? avail / (2 * C::GSTRIDE) / C::D * C::D : 0;
    if (xg < C::D) return 0;
    xg = std::min(xg, (int)ceil_div(gps, C::D) * C::D);
    p.xg = xg;
    p.xp_off = 2 * xg * C::GSTRIDE;
    p.xslot_off = (std::max(p.xp_off + pbytes, C::RED_BYTES) + 15) / 16 * 16;
    p.xbar_off = p.xslot_off + slots;
    return (size_t)std::max(p.xbar_off + 16, cap);
}

template <int BITS, int G, int MP>
qg_status dense_mp(const Problem& p0, cudaStream_t s)
{
    Problem p = p0;
    const int ng = p.K / G;
    const int tiles = (int)ceil_div(p.N, kRowsPerCta);
    const int S = choose_splits(tiles, ng);
    const dim3 grid((unsigned)tiles, (unsigned)S, 1);
    const int gps = (int)ceil_div(ng, S);
    size_t smem = decode_smem<BITS, G, MP>(gps, S);
    if (p.xfrag) {
        const size_t sx = xpre_layout<BITS, G, MP>(gps, S, p);
        if (sx) {
            smem = sx;
            qg_status st = launch_x_frag<BITS, G, MP>(p, s);
            if (st != QG_OK) return st;
        } else {
            p.xfrag = nullptr;   // no room for two x buffers: the CTAs convert x
        }
    }
    // programmatic dependent launch: the next product's CTAs start their weight
    // loads while this one drains (the per-SM caps of decode_smem keep them
    // from crowding the SMs this launch still uses)
    return launch_cluster(k_gemv<BITS, G, MP>, grid, S, kWarps * 32, smem, true, s, p, S, gps);
}

template <int BITS, int G, int MP>
qg_status multi_mp(const MultiTable& t0, cudaStream_t s)
{
    MultiTable t = t0;
    const int ng = t.p[0].K / G;
    const int tiles = t.tile_start[t.n];
    const int S = choose_splits(tiles, ng);
    const dim3 grid((unsigned)tiles, (unsigned)S, 1);
    const int gps = (int)ceil_div(ng, S);
    size_t smem = decode_smem<BITS, G, MP>(gps, S);
    if (t.p[0].xfrag) {
        const size_t sx = xpre_layout<BITS, G, MP>(gps, S, t.p[0]);
        for (int q = 1; q < t.n; q++) {   // one launch, one layout
            t.p[q].xg = t.p[0].xg; t.p[q].xp_off = t.p[0].xp_off;
            t.p[q].xslot_off = t.p[0].xslot_off; t.p[q].xbar_off = t.p[0].xbar_off;
        }
        if (sx) {
            smem = sx;
            qg_status st = launch_x_frag<BITS, G, MP>(t.p[0], s);
            if (st != QG_OK) return st;
        } else {
            for (int q = 0; q < t.n; q++) t.p[q].xfrag = nullptr;
        }
    }
    return launch_cluster(k_gemv_multi<BITS, G, MP>, grid, S, kWarps * 32, smem, true, s, t, S, gps);
}

template <int BITS, int G, int MP>
qg_status grouped_mp(const MoeTable& t, int max_items, int expect_items, cudaStream_t s)
{
    const int ng = t.K / G;
    const int tiles = (int)ceil_div(t.N, kRowsPerCta);
    const int S = choose_splits((long long)tiles * std::max(1, expect_items), ng);
    const int gps = (int)ceil_div(ng, S);
    return launch_cluster(k_gemv_moe<BITS, G, MP>, dim3((unsigned)tiles, (unsigned)S, (unsigned)max_items), S,
                          kWarps * 32, decode_smem<BITS, G, MP>(gps, S), false, s, t, S, gps);
}

template <int BITS, int G, template <int, int, int> class F, typename... Args>
qg_status by_mp(int mp, Args&&... args)
{
    switch (mp) {
        case 1: return F<BITS, G, 1>::run(args...);
        case 2: return F<BITS, G, 2>::run(args...);
        case 4: return F<BITS, G, 4>::run(args...);
        case 8: return F<BITS, G, 8>::run(args...);
        case 16: return F<BITS, G, 16>::run(args...);
        case 32: return F<BITS, G, 32>::run(args...);
        default: return F<BITS, G, 64>::run(args...);
    }
}

template <int BITS, int G, int MP>
struct DenseF {
    static qg_status run(const Problem& p, cudaStream_t s) { return dense_mp<BITS, G, MP>(p, s); }
};
template <int BITS, int G, int MP>
struct MultiF {
    static qg_status run(const MultiTable& t, cudaStream_t s) { return multi_mp<BITS, G, MP>(t, s); }
};
template <int BITS, int G, int MP>
struct GroupedF {
    static qg_status run(const MoeTable& t, int mi, int ei, cudaStream_t s) { return grouped_mp<BITS, G, MP>(t, mi, ei, s); }
};

// One (width, group) pair: each is instantiated in a translation unit of its
// own (gemv_w<bits>.cu for groups 64 and 128, gemv_w<bits>_g32.cu for 32) so
// that the heavy template compiles in parallel.
template <int BITS, int G>
qg_status dense_g(const Problem& p, cudaStream_t s)
{
    return by_mp<BITS, G, DenseF>(mp_for(p.M), p, s);
}

template <int BITS, int G>
qg_status multi_g(const MultiTable& t, cudaStream_t s)
{
    return by_mp<BITS, G, MultiF>(mp_for(t.p[0].M), t, s);
}

// t.chunk must equal the padded token count mp.  max_items bounds the
// device-built item count; expect_items is the typical count (for choosing
// the K split).
template <int BITS, int G>
qg_status grouped_g(const MoeTable& t, int max_items, int expect_items, int mp, cudaStream_t s)
{
    return by_mp<BITS, G, GroupedF>(mp, t, max_items, expect_items, s);
}

#define QG_GEMV_EXTERN(B, G)                                                                      \
    extern template qg_status dense_g<B, G>(const Problem&, cudaStream_t);                       \
    extern template qg_status multi_g<B, G>(const MultiTable&, cudaStream_t);                    \
    extern template qg_status grouped_g<B, G>(const MoeTable&, int, int, int, cudaStream_t);
#define QG_GEMV_INSTANTIATE(B, G)                                                                 \
    template qg_status dense_g<B, G>(const Problem&, cudaStream_t);                              \
    template qg_status multi_g<B, G>(const MultiTable&, cudaStream_t);                           \
    template qg_status grouped_g<B, G>(const MoeTable&, int, int, int, cudaStream_t);
#define QG_GEMV_EXTERN_WIDTH(B) QG_GEMV_EXTERN(B, 32) QG_GEMV_EXTERN(B, 64) QG_GEMV_EXTERN(B, 128)
QG_GEMV_EXTERN_WIDTH(2)
QG_GEMV_EXTERN_WIDTH(3)
QG_GEMV_EXTERN_WIDTH(4)
QG_GEMV_EXTERN_WIDTH(5)
QG_GEMV_EXTERN_WIDTH(6)
QG_GEMV_EXTERN_WIDTH(8)

template <int BITS>
qg_status launch_dense(const Problem& p, int G, cudaStream_t s)
{
    return G == 32 ? dense_g<BITS, 32>(p, s) : G == 64 ? dense_g<BITS, 64>(p, s) : dense_g<BITS, 128>(p, s);
}

template <int BITS>
qg_status launch_multi(const MultiTable& t, int G, cudaStream_t s)
{
    return G == 32 ? multi_g<BITS, 32>(t, s) : G == 64 ? multi_g<BITS, 64>(t, s) : multi_g<BITS, 128>(t, s);
}

template <int BITS>
qg_status launch_grouped(const MoeTable& t, int max_items, int expect_items, int G, int mp, cudaStream_t s)
{
    return G == 32   ? grouped_g<BITS, 32>(t, max_items, expect_items, mp, s)
           : G == 64 ? grouped_g<BITS, 64>(t, max_items, expect_items, mp, s)
                     : grouped_g<BITS, 128>(t, max_items, expect_items, mp, s);
}

}  // namespace gemv
}  // namespace qg
