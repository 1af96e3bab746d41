// One-time device repack of a quantized weight into the tile-ordered layout
// the tensor-core kernel streams ("Mixed-width quantization" page, sections
// 3.1 and 3.3: codes laid out for aligned vector access, the scales beside
// the codes they scale; "70B on one GPU" page, section 3: weights repacked
// once, when loaded, for the fused kernel).  Every (256-row tile, 64-wide K
// block) becomes one contiguous block starting on a 128-byte boundary:
//   codes   4 * bits words per row pair ... word i of dequantization thread
//           t = 2 * row + half (codes [32 half, 32 half + 32) of the row in
//           this K block, LSB-first as in the planar stream) at word
//           i * 512 + t: a warp's 32 threads read 32 consecutive words;
//   params  per row, for each group the block touches (two at group 32,
//           else one) a 32-bit word (fp16 scale | zero-point << 16; an
//           8-bit scale is converted to its fp16 value here), or at 2 bits
//           the four fp16 codebook entries (8 bytes);
// rows beyond N are zero.  The FP16 outliers stay in their CSR arrays.
// One CTA of 512 threads per block; a thread moves its chunk's words and
// the parameters of its chunk's group (at group 32; else the even thread
// writes the row's one set).
#include "qg_internal.h"
#include "scale8.cuh"

namespace qg {
namespace {

template <int BITS>
__global__ void __launch_bounds__(512) k_repack(const uint8_t* __restrict__ packed, const ScaleSrc sc,
                                                const uint8_t* __restrict__ zp, const uint2* __restrict__ cb, int N,
                                                int K, int G, uint8_t* __restrict__ tiles)
{
    const int kb = blockIdx.x, nt = blockIdx.y, KB = K / kTileK;
    const int t = threadIdx.x, r = t >> 1, h = t & 1;
    const int n = nt * kTileRows + r;
    uint32_t* blk = reinterpret_cast<uint32_t*>(tiles + ((size_t)nt * KB + kb) * tile_block_bytes(BITS, G));
    const bool live = n < N;
    // the chunk: 4 * BITS bytes at byte (2 kb + h) * 4 * BITS of the row (word aligned)
    const uint32_t* src = reinterpret_cast<const uint32_t*>(packed + (size_t)n * ((size_t)K * BITS / 8) +
                                                            (size_t)(2 * kb + h) * 4 * BITS);
#pragma unroll
    for (int i = 0; i < BITS; i++) blk[i * 512 + t] = live ? __ldg(src + i) : 0u;
    const int npg = tile_groups_per_block(G);
    if (npg == 2 || h == 0) {
        const int g = (kb * kTileK + 32 * h) / G, ng = K / G;
        const int slot = r * npg + (npg == 2 ? h : 0);
        uint32_t* prm = blk + BITS * 512;
        if constexpr (BITS == 2) {
            reinterpret_cast<uint2*>(prm)[slot] = live ? __ldg(cb + (size_t)n * ng + g) : make_uint2(0u, 0u);
        } else {
            prm[slot] = live ? (scale_bits(sc, scale_exp(sc), n, ng, g) | ((uint32_t)__ldg(zp + (size_t)n * ng + g) << 16))
                             : 0u;
        }
    }
}

template <int BITS>
qg_status repack_bits(const qg_qweight& w, void* tiles, cudaStream_t s)
{
    const dim3 grid((unsigned)(w.K / kTileK), (unsigned)ceil_div(w.N, kTileRows));
    k_repack<BITS><<<grid, 512, 0, s>>>(w.packed, scale_src(w), w.zp, reinterpret_cast<const uint2*>(w.codebook), w.N,
                                        w.K, w.group, static_cast<uint8_t*>(tiles));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "repack kernel launch");
    return QG_OK;
}

// Launched after the repack: a product that reads the copy next on the
// stream may start its code loads before the kernel just before it has
// finished (programmatic dependent launch), so that kernel must not be the
// one that wrote the copy.
__global__ void k_repack_done() {}

}  // namespace

qg_status launch_repack(const qg_qweight& w, void* tiles, cudaStream_t s)
{
    qg_status st;
    switch (w.bits) {
        case 2: st = repack_bits<2>(w, tiles, s); break;
        case 3: st = repack_bits<3>(w, tiles, s); break;
        case 4: st = repack_bits<4>(w, tiles, s); break;
        case 5: st = repack_bits<5>(w, tiles, s); break;
        case 6: st = repack_bits<6>(w, tiles, s); break;
        default: st = repack_bits<8>(w, tiles, s); break;
    }
    if (st != QG_OK) return st;
    k_repack_done<<<1, 32, 0, s>>>();
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "repack launch");
    return QG_OK;
}

}  // namespace qg
