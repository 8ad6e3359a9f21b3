// Kernel instantiations of the grouped ring AllReduce, LL protocol: every
// element type and reduction op.
#include "group.cuh"

namespace vrccl {
extern const void* const kGroupLL[vrcclNumTypes][5];
const void* const kGroupLL[vrcclNumTypes][5] = VRCCL_GROUP_TABLE(kLL);
}  // namespace vrccl
