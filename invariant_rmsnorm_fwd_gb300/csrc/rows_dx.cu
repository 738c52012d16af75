// Instantiations of the row launcher for: kDx, kAddDx, kDw.
#include "launch.cuh"

namespace rbi {
template int run_rows<kDx>(KParams, const Shape &, const rmsnorm_layout_t *, cudaStream_t);
template int run_rows<kAddDx>(KParams, const Shape &, const rmsnorm_layout_t *, cudaStream_t);
template int run_rows<kDw>(KParams, const Shape &, const rmsnorm_layout_t *, cudaStream_t);
}  // namespace rbi
