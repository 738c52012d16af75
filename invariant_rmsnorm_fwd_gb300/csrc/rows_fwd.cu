// Instantiations of the row launcher for: kFwd, kAddFwd.
#include "launch.cuh"

namespace rbi {
template int run_rows<kFwd>(KParams, const Shape &, const rmsnorm_layout_t *, cudaStream_t);
template int run_rows<kAddFwd>(KParams, const Shape &, const rmsnorm_layout_t *, cudaStream_t);
}  // namespace rbi
