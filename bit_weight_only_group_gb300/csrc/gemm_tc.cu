// Products with M above the decode kernel's range.
#include "qg_internal.h"

namespace qg {

qg_status launch_gemv_chunked(const uint16_t* x, int M, int ldx, const qg_qweight& w, void* y, int ldy,
                              qg_ydtype yt, cudaStream_t s);

size_t gemm_workspace_bytes(int, const qg_qweight&) { return 0; }

qg_status launch_gemm(const uint16_t* x, int M, int ldx, const qg_qweight& w, void* y, int ldy, qg_ydtype yt,
                      void*, size_t, cudaStream_t s)
{
    return launch_gemv_chunked(x, M, ldx, w, y, ldy, yt, s);
}

}  // namespace qg
