// Kernel instantiations of the LL protocol: ring and tree, every element
// type and reduction op.
#include "kernels.cuh"

namespace vrccl {
extern const void* const kRingLL[4][5];
extern const void* const kTreeLL[4][5];
const void* const kRingLL[4][5] = VRCCL_KERNEL_ROW(kLL, ringKernel);
const void* const kTreeLL[4][5] = VRCCL_KERNEL_ROW(kLL, treeKernel);
}  // namespace vrccl
