// Kernel instantiations of the grouped ring AllReduce, Simple protocol: every
// element type and reduction op.
#include "group.cuh"

namespace vrccl {
extern const void* const kGroupSimple[vrcclNumTypes][5];
const void* const kGroupSimple[vrcclNumTypes][5] = VRCCL_GROUP_TABLE(kSimple);
}  // namespace vrccl
