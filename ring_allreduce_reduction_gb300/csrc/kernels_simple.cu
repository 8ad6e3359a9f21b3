// Kernel instantiations of the Simple protocol: ring and tree, element types
// 0-3 (int32, float32, bfloat16, float16), every reduction op; the other
// four types are in a translation unit of their own (compile time).
#include "kernels.cuh"

namespace vrccl {
extern const void* const kRingSimple[4][5];
extern const void* const kTreeSimple[4][5];
const void* const kRingSimple[4][5] = VRCCL_KERNEL_ROWS4(kSimple, ringKernel, 0);
const void* const kTreeSimple[4][5] = VRCCL_KERNEL_ROWS4(kSimple, treeKernel, 0);
}  // namespace vrccl
