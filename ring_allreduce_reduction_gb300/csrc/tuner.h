// Schedule choice for algo = auto / proto = auto / channels = auto.
//
// NCCL predicts a time per (algorithm, protocol) with T = latency +
// bytes / bandwidth from constants of its tuning tables and takes the
// minimum ("NCCL architecture: topology, channels, algorithms and
// protocols", §8.2, ncclTopoGetAlgoTime). Here the table holds times
// measured on this GPU for this communicator's rank count: per (element
// size, algo, proto, channels, slice size) and per power-of-two message
// size, and the choice is the measured minimum at the nearest size among
// the rows of the call's element size (or, if the table has none, of the
// nearest measured element size). Without a table the rule below stands
// in: LL up to 64 KiB, LL128 up to 2 MiB, Simple beyond (the nearest
// allowed protocol in that order of preference), the ring if allowed, and
// NCCL's channel shrink (§6.4 of the same page).
#pragma once

#include <cstddef>
#include <cstdint>
#include <mutex>
#include <string>
#include <unordered_map>
#include <vector>

namespace vrccl {

struct Choice {
  int algo;
  int proto;
  int channels;       // 0 = use defaultChannels()
  size_t sliceBytes;  // 0 = protocol default
  size_t chunkBytes;  // 0 = VRCCL_STEPS/2 slices
  bool measured;      // from a table entry (else the size rule)
  int esize;          // element size of the rows it came from (0 = rows for any size)
  int log2bytes;      // size of the entry it came from
};

// NCCL's rule: start from the maximum and drop channels while each would
// get less than threads x threadThreshold bytes (thresholds 64 B for
// Simple, 8 B for LL128, 8 B x n for ring LL).
int defaultChannels(int proto, size_t bytes, int nranks, int maxChannels);

class Tuner {
 public:
  struct Entry {
    int nranks, algo, proto, channels;
    int log2bytes;
    size_t sliceBytes;
    double us;
    int esize;  // bytes per element the row was measured with; 0 = any
  };
  // Only entries whose algorithm is in algoMask (bit kRing, bit kTree) and
  // whose protocol is in protoMask (bits kSimple, kLL, kLL128) are eligible;
  // a mask with one bit forces that choice. Masks must not be empty.
  // esize: the call's element size in bytes.
  Choice choose(int nranks, size_t bytes, int esize, int maxChannels, unsigned algoMask = 3u,
                unsigned protoMask = 7u) const;
  // Reads VRCCL_TUNE_FILE if set, else the table shipped next to the
  // library (tuning/gb300_n<nranks>.txt) if there is one. Format: one entry
  // per line, "nranks algo proto channels log2bytes sliceBytes
  // microseconds [elementBytes]"; '#' starts a comment; a line without
  // the element size applies to every element type.
  void loadEnvFile(int nranks);
  int load(const char* path, int nranks);  // entries read, -1 on error
  void add(const Entry& e) {
    table_.push_back(e);
    forget();
  }
  void clear() {
    table_.clear();
    forget();
  }
  size_t size() const { return table_.size(); }
  Tuner() = default;
  Tuner(const Tuner& o) : table_(o.table_) {}
  Tuner& operator=(const Tuner& o) {
    table_ = o.table_;
    forget();
    return *this;
  }

 private:
  Choice scan(int nranks, size_t bytes, int esize, int maxChannels, unsigned algoMask, unsigned protoMask) const;
  void forget() {
    std::lock_guard<std::mutex> lk(mu_);
    memo_.clear();
  }
  std::vector<Entry> table_;
  // A call's choice depends only on (rank count, power-of-two size bucket,
  // element size, channel budget, masks); it is found by a scan of the
  // table once and kept, so a call does no search (the tables hold
  // thousands of rows).
  mutable std::mutex mu_;
  mutable std::unordered_map<uint64_t, Choice> memo_;
};

}  // namespace vrccl
