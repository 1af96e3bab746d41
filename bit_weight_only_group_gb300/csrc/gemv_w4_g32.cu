// Instantiation of the decode / grouped kernels for 4-bit weights, group 32.
#include "gemv_impl.cuh"

namespace qg {
namespace gemv {
QG_GEMV_INSTANTIATE(4, 32)
}  // namespace gemv
}  // namespace qg
