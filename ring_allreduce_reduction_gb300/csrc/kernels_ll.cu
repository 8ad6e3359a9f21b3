// Kernel instantiations of the LL protocol: ring and tree, every element
// type and reduction op.
#include "kernels.cuh"

namespace vrccl {
extern const void* const kRingLL[vrcclNumTypes][5];
extern const void* const kTreeLL[vrcclNumTypes][5];
const void* const kRingLL[vrcclNumTypes][5] = VRCCL_KERNEL_ROWS8(kLL, ringKernel);
const void* const kTreeLL[vrcclNumTypes][5] = VRCCL_KERNEL_ROWS8(kLL, treeKernel);
}  // namespace vrccl
