// Instantiation of the decode / grouped kernels for 6-bit weights, groups 64 and 128.
#include "gemv_impl.cuh"

namespace qg {
namespace gemv {
QG_GEMV_INSTANTIATE(6, 64)
QG_GEMV_INSTANTIATE(6, 128)
template qg_status launch_dense<6>(const Problem&, int, cudaStream_t);
template qg_status launch_multi<6>(const MultiTable&, int, cudaStream_t);
template qg_status launch_grouped<6>(const MoeTable&, int, int, int, int, cudaStream_t);
}  // namespace gemv
}  // namespace qg
