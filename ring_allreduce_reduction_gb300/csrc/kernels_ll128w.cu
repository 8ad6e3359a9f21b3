// Kernel instantiations of the LL128 protocol's wide variant (four groups
// of lines per warp and pass, for long slices): ring and tree, every element
// type and reduction op.
#include "kernels.cuh"

namespace vrccl {
extern const void* const kRingLL128W[4][5];
extern const void* const kTreeLL128W[4][5];
const void* const kRingLL128W[4][5] = VRCCL_KERNEL_ROW(kLL128Wide, ringKernel);
const void* const kTreeLL128W[4][5] = VRCCL_KERNEL_ROW(kLL128Wide, treeKernel);
}  // namespace vrccl
