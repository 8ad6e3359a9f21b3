// Kernel instantiations of the LL128 protocol's wide variant (four groups
// of lines per warp and pass, for long slices): ring and tree, element types
// 0-3 (int32, float32, bfloat16, float16), every reduction op; the other
// four types are in a translation unit of their own (compile time).
#include "kernels.cuh"

namespace vrccl {
extern const void* const kRingLL128W[4][5];
extern const void* const kTreeLL128W[4][5];
const void* const kRingLL128W[4][5] = VRCCL_KERNEL_ROWS4(kLL128Wide, ringKernel, 0);
const void* const kTreeLL128W[4][5] = VRCCL_KERNEL_ROWS4(kLL128Wide, treeKernel, 0);
}  // namespace vrccl
