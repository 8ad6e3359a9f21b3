// VRCCL_ALGO / VRCCL_PROTO: NCCL_ALGO / NCCL_PROTO's list syntax (parseList,
// "NCCL architecture: topology, channels, algorithms and protocols", §8.5).
// Elements are comma separated; a leading '^' excludes the listed ones
// instead; "function:" restricts a list to one collective; ';' separates
// lists, and the first may have no prefix (it then applies to every
// collective). Names are case-insensitive and must be NCCL's.
#pragma once

namespace vrccl {

// NCCL's orders, which the bit masks follow.
enum ParseFunc { kFnBroadcast = 0, kFnReduce, kFnAllGather, kFnReduceScatter, kFnAllReduce, kNumParseFuncs };
// algorithms: Tree Ring CollNetDirect CollNetChain NVLS NVLSTree PAT (bits 0..6)
// protocols:  LL LL128 Simple (bits 0..2)
constexpr int kParseAlgo = 0, kParseProto = 1;

// Fills masks[f] for every function f (all bits set where the string says
// nothing). Returns 0, or -1 for an unknown function or element name.
int parseList(const char* s, int kind, unsigned masks[kNumParseFuncs]);

}  // namespace vrccl
