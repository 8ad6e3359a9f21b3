// The pages' analytic model of an AllReduce's time, T = latency + S / bw
// (ncclTopoTuneModel and ncclTopoGetAlgoTime, "NCCL architecture: topology,
// channels, algorithms and protocols", §8.1-§8.3). It is not used to choose
// schedules here (the tuner is measured); it is printed beside the measured
// table, with the constants the pages give.
#pragma once

#include <cstddef>

namespace vrccl {

struct ModelGraph {
  int nRanks, nNodes, nChannels;
  double bwIntra, bwInter;  // GB/s per channel inside a node / across nodes
  double latencyInter;      // us added to every inter-node step
  int hwIntra;              // 0 NVLink, 1 PCI
  int arch;                 // 0 Volta, 1 Ampere, 2 Hopper, 3 Blackwell
};

// Latency (us) and algorithm bandwidth (GB/s) of the AllReduce for
// algo (kRing, kTree) x proto (kSimple, kLL, kLL128).
void modelTable(const ModelGraph& g, double lat[2][3], double bw[2][3]);

// Predicted time (us) of one AllReduce of `bytes`, one of `numPipeOps`
// aggregated operations; < 0 if the combination is disabled.
double modelTime(const ModelGraph& g, int algo, int proto, size_t bytes, int numPipeOps);

}  // namespace vrccl
