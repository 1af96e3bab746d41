// The tensor-core product from the tile-ordered copy (qgemm_forward_tiles),
// instantiated apart from the planar kernels so that both compile in parallel;
// the kernel is in gemm_tc.cuh.
#include "gemm_tc.cuh"

namespace qg {

qg_status launch_gemm_tiles(const uint16_t* x, int M, int ldx, const qg_qweight& w, const void* tiles, void* y,
                            int ldy, qg_ydtype yt, void* ws, cudaStream_t s)
{
    switch (w.bits) {
        case 2: return tc::run_bits<2, true>(x, M, ldx, w, tiles, y, ldy, yt, ws, true, s);
        case 3: return tc::run_bits<3, true>(x, M, ldx, w, tiles, y, ldy, yt, ws, true, s);
        case 4: return tc::run_bits<4, true>(x, M, ldx, w, tiles, y, ldy, yt, ws, true, s);
        case 5: return tc::run_bits<5, true>(x, M, ldx, w, tiles, y, ldy, yt, ws, true, s);
        case 6: return tc::run_bits<6, true>(x, M, ldx, w, tiles, y, ldy, yt, ws, true, s);
        default: return tc::run_bits<8, true>(x, M, ldx, w, tiles, y, ldy, yt, ws, true, s);
    }
}

}  // namespace qg
