// Instantiations of the row launcher for: kDxDw.
#include "launch.cuh"

namespace rbi {
template int run_rows<kDxDw>(KParams, const Shape &, const rmsnorm_layout_t *, cudaStream_t);
}  // namespace rbi
