// Instantiations of the row launcher for: kAddDxDw.
#include "launch.cuh"

namespace rbi {
template int run_rows<kAddDxDw>(KParams, const Shape &, const rmsnorm_layout_t *, cudaStream_t);
}  // namespace rbi
