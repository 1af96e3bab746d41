// The tensor-core product from the planar layout (qgemm_forward above the
// decode range), its workspace, the x conversion of the tile-ordered path, and
// the tensor-map encoder the tensor-core kernels share; the kernel is in
// gemm_tc.cuh.
#include "gemm_tc.cuh"

namespace qg {

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


size_t gemm_workspace_bytes(int M, const qg_qweight& w) { return tc::ws_layout(M, w.N, w.K, nullptr, nullptr); }

qg_status launch_gemm(const uint16_t* x, int M, int ldx, const qg_qweight& w, void* y, int ldy, qg_ydtype yt,
                      void* ws, size_t, bool convert_x, cudaStream_t s)
{
    switch (w.bits) {
        case 2: return tc::run_bits<2, false>(x, M, ldx, w, nullptr, y, ldy, yt, ws, convert_x, s);
        case 3: return tc::run_bits<3, false>(x, M, ldx, w, nullptr, y, ldy, yt, ws, convert_x, s);
        case 4: return tc::run_bits<4, false>(x, M, ldx, w, nullptr, y, ldy, yt, ws, convert_x, s);
        case 5: return tc::run_bits<5, false>(x, M, ldx, w, nullptr, y, ldy, yt, ws, convert_x, s);
        case 6: return tc::run_bits<6, false>(x, M, ldx, w, nullptr, y, ldy, yt, ws, convert_x, s);
        default: return tc::run_bits<8, false>(x, M, ldx, w, nullptr, y, ldy, yt, ws, convert_x, s);
    }
}

}  // namespace qg
