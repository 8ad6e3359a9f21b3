#include "model.h"

#include <algorithm>
#include <cmath>

#include "vrccl_internal.h"

namespace vrccl {

// Constants as the pages print them ("NCCL architecture ...", §8.1), in the
// pages' protocol order {LL, LL128, Simple}.
static const double kBaseLat[2][3] = {
    {14.0, 14.0, 8.4},  // Ring. The table prints 6.6 for LL; every worked
                        // example on the page (the 8-GPU table row, machines
                        // one and three) uses 14, which is followed here.
    {6.8, 14.0, 8.4},   // Tree
};
static const double kHwLat[3][2][3] = {
    {{0.6, 1.9, 3.4}, {0.6, 1.25, 4.0}},    // NVLink: Ring, Tree
    {{1.0, 2.5, 5.7}, {1.0, 1.9, 4.0}},     // PCI
    {{2.7, 4.0, 14.0}, {5.0, 8.5, 14.0}},   // network
};
// Per architecture, per node-count tier (1 node, 2 nodes, more).
static const double kLLMaxBw[4][3] = {{39.0, 39.0, 20.4}, {87.7, 22.5, 19.0}, {141.0, 45.0, 35.0},
                                      {282.0, 90.0, 70.0}};  // Blackwell: Hopper's doubled
// Per-channel caps. Hopper's are printed; Volta/Ampere's are the values the
// worked examples use (24 for the tree, 20 for ring LL128); Blackwell keeps
// Hopper's.
static const double kPerChRingLL128[4] = {20.0, 20.0, 36.7, 36.7};
static const double kPerChTree[4][3] = {{24.0, 24.0, 24.0}, {24.0, 24.0, 24.0}, {38.7, 41.4, 36.0},
                                        {38.7, 41.4, 36.0}};

// pages' protocol index from ours
static int pp(int proto) { return proto == kLL ? 0 : proto == kLL128 ? 1 : 2; }

void modelTable(const ModelGraph& g, double lat[2][3], double bw[2][3]) {
  const int tier = g.nNodes <= 1 ? 0 : g.nNodes == 2 ? 1 : 2;
  const int arch = std::min(std::max(g.arch, 0), 3);
  const double linkBw = g.nNodes <= 2 ? g.bwIntra : g.bwInter;
  const double bus0 = g.nChannels * linkBw;
  const int nsteps = 2 * (g.nRanks - 1);
  const int nInter = 2 * (g.nNodes - 1);
  const int perNode = g.nRanks / std::max(g.nNodes, 1);
  const double log2Nodes = std::log2((double)std::max(g.nNodes, 1));
  for (int a = 0; a < 2; ++a) {
    for (int p = 0; p < 3; ++p) {
      const int proto = p == 0 ? kSimple : p == 1 ? kLL : kLL128;
      const int q = pp(proto);
      double bus = bus0;
      if (a == kRing) {
        if (proto == kLL) bus = std::min(kLLMaxBw[arch][tier], bus * 0.5);
        if (proto == kLL128) bus = std::min(bus * 0.92, g.nChannels * kPerChRingLL128[arch]);
      } else {
        bus = std::min(bus * 0.92, g.nChannels * kPerChTree[arch][tier]);
        if (proto == kLL) bus = std::min(kLLMaxBw[arch][tier], bus / 3.8);
        if (proto == kLL128) bus *= g.nNodes == 1 ? 7.0 / 9.0 : 120.0 / 128.0;
        if (arch >= 2) bus *= 0.85;  // the tree pattern on Hopper and later
      }
      bw[a][proto] = a == kRing ? bus * g.nRanks / nsteps : bus * 0.5;
      const double intra = kHwLat[g.hwIntra == 1 ? 1 : 0][a][q];
      const double inter = kHwLat[2][a][q] + g.latencyInter;
      lat[a][proto] = a == kRing ? kBaseLat[a][q] + (nsteps - nInter) * intra + nInter * inter
                                 : kBaseLat[a][q] + 2.0 * ((perNode - 1) * intra + log2Nodes * inter);
    }
  }
}

double modelTime(const ModelGraph& g, int algo, int proto, size_t bytes, int numPipeOps) {
  double lat[2][3], bw[2][3];
  modelTable(g, lat, bw);
  double b = bw[algo][proto], l = lat[algo][proto];
  if (b <= 0) return -1.0;
  // the ring's plateau across nodes (ncclTopoGetAlgoTime)
  if (algo == kRing && proto == kSimple && g.nNodes > 1 && bytes / (size_t(g.nChannels) * g.nRanks) >= 64)
    l *= g.arch == 0 ? 1.9 : 1.4;
  // every ring operation pays its latency; a tree pipeline pays it once
  const int latCount = algo == kRing ? std::max(numPipeOps, 1) : 1;
  return l * latCount + double(bytes) / (1000.0 * b);
}

}  // namespace vrccl
