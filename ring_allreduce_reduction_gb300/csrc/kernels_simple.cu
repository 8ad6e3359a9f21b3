// Kernel instantiations of the Simple protocol: ring and tree, every element
// type and reduction op.
#include "kernels.cuh"

namespace vrccl {
extern const void* const kRingSimple[4][5];
extern const void* const kTreeSimple[4][5];
const void* const kRingSimple[4][5] = VRCCL_KERNEL_ROW(kSimple, ringKernel);
const void* const kTreeSimple[4][5] = VRCCL_KERNEL_ROW(kSimple, treeKernel);
}  // namespace vrccl
