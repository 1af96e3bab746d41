// Instantiation of the decode / grouped kernels for 2-bit weights, groups 64 and 128.
#include "gemv_impl.cuh"

namespace qg {
namespace gemv {
QG_GEMV_INSTANTIATE(2, 64)
QG_GEMV_INSTANTIATE(2, 128)
template qg_status launch_dense<2>(const Problem&, int, cudaStream_t);
template qg_status launch_multi<2>(const MultiTable&, int, cudaStream_t);
template qg_status launch_grouped<2>(const MoeTable&, int, int, int, int, cudaStream_t);
}  // namespace gemv
}  // namespace qg
