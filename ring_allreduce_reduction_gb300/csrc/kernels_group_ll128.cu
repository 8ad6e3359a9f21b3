// Kernel instantiations of the grouped ring AllReduce, LL128 protocol: every
// element type and reduction op.
#include "group.cuh"

namespace vrccl {
extern const void* const kGroupLL128[vrcclNumTypes][5];
const void* const kGroupLL128[vrcclNumTypes][5] = VRCCL_GROUP_TABLE(kLL128);
}  // namespace vrccl
