// Kernel instantiations of the LL128 protocol: ring and tree, every element
// type and reduction op.
#include "kernels.cuh"

namespace vrccl {
extern const void* const kRingLL128[vrcclNumTypes][5];
extern const void* const kTreeLL128[vrcclNumTypes][5];
const void* const kRingLL128[vrcclNumTypes][5] = VRCCL_KERNEL_ROWS8(kLL128, ringKernel);
const void* const kTreeLL128[vrcclNumTypes][5] = VRCCL_KERNEL_ROWS8(kLL128, treeKernel);
}  // namespace vrccl
