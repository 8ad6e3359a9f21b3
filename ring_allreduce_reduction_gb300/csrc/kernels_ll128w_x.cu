// Kernel instantiations of the LL128 protocol's wide variant (four groups
// of lines per warp and pass, for long slices): ring and tree, element types
// 4-7 (int8, uint8, int64, float64), every reduction op.
#include "kernels.cuh"

namespace vrccl {
extern const void* const kRingLL128WX[4][5];
extern const void* const kTreeLL128WX[4][5];
const void* const kRingLL128WX[4][5] = VRCCL_KERNEL_ROWS4(kLL128Wide, ringKernel, 4);
const void* const kTreeLL128WX[4][5] = VRCCL_KERNEL_ROWS4(kLL128Wide, treeKernel, 4);
}  // namespace vrccl
