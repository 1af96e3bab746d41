// Instantiation of the decode / grouped kernels for 3-bit weights, group 32.
#include "gemv_impl.cuh"

namespace qg {
namespace gemv {
QG_GEMV_INSTANTIATE(3, 32)
}  // namespace gemv
}  // namespace qg
