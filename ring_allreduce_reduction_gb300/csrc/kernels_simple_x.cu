// Kernel instantiations of the Simple protocol: ring and tree, element types
// 4-7 (int8, uint8, int64, float64), every reduction op.
#include "kernels.cuh"

namespace vrccl {
extern const void* const kRingSimpleX[4][5];
extern const void* const kTreeSimpleX[4][5];
const void* const kRingSimpleX[4][5] = VRCCL_KERNEL_ROWS4(kSimple, ringKernel, 4);
const void* const kTreeSimpleX[4][5] = VRCCL_KERNEL_ROWS4(kSimple, treeKernel, 4);
}  // namespace vrccl
