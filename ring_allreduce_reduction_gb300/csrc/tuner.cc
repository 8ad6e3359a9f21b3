#include "tuner.h"

#include <dlfcn.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>

#include "vrccl_internal.h"

namespace vrccl {

int defaultChannels(int proto, size_t bytes, int nranks, int maxChannels) {
  const size_t threads = proto == kSimple ? 512 : 256;
  const size_t perThread = proto == kSimple ? 64 : proto == kLL128 ? 8 : size_t(8) * nranks;
  int nc = maxChannels;
  while (nc > 1 && bytes < size_t(nc) * threads * perThread) --nc;
  return nc;
}

static int log2Bucket(size_t bytes) {
  int b = 0;
  while ((size_t(1) << (b + 1)) <= bytes && b < 62) ++b;
  // round to the nearer power of two
  if (b < 62 && bytes - (size_t(1) << b) > (size_t(1) << (b + 1)) - bytes) ++b;
  return b;
}

Choice Tuner::choose(int nranks, size_t bytes, int esize, int maxChannels, unsigned algoMask,
                     unsigned protoMask) const {
  // the choice depends on the size only through its bucket (nearest power
  // of two) and the size rule's thresholds; key on both
  const int bucket = log2Bucket(bytes);
  const int rule = bytes <= 65536 ? 0 : bytes <= (size_t(2) << 20) ? 1 : 2;
  const uint64_t key = (uint64_t(nranks) << 48) ^ (uint64_t(bucket) << 40) ^ (uint64_t(rule) << 38) ^
                       (uint64_t(esize & 15) << 34) ^ (uint64_t(maxChannels & 127) << 24) ^
                       (uint64_t(algoMask & 255) << 8) ^ uint64_t(protoMask & 255);
  {
    std::lock_guard<std::mutex> lk(mu_);
    auto it = memo_.find(key);
    if (it != memo_.end()) return it->second;
  }
  const Choice c = scan(nranks, bytes, esize, maxChannels, algoMask, protoMask);
  std::lock_guard<std::mutex> lk(mu_);
  memo_.emplace(key, c);
  return c;
}

Choice Tuner::scan(int nranks, size_t bytes, int esize, int maxChannels, unsigned algoMask,
                   unsigned protoMask) const {
  // the size rule's preference order, first allowed protocol wins
  static const int kSmall[3] = {kLL, kLL128, kSimple}, kMid[3] = {kLL128, kSimple, kLL},
                   kLarge[3] = {kSimple, kLL128, kLL};
  const int* pref = bytes <= 65536 ? kSmall : bytes <= (size_t(2) << 20) ? kMid : kLarge;
  int proto = pref[0];
  for (int i = 2; i >= 0; --i)
    if (protoMask & (1u << pref[i])) proto = pref[i];
  Choice c{(algoMask & (1u << kRing)) ? kRing : kTree, proto, 0, 0, 0, false, 0, 0};
  auto eligible = [&](const Entry& e) {
    return e.nranks == nranks && e.channels <= maxChannels && (algoMask & (1u << e.algo)) &&
           (protoMask & (1u << e.proto));
  };
  // The rows to use: those of the call's element size; else the rows that
  // apply to any size; else those of the nearest measured element size
  // (ties: the larger).
  auto dist = [&](int s) { return std::abs(std::log2(double(s)) - std::log2(double(esize))); };
  int group = -1;
  for (const Entry& e : table_) {
    if (!eligible(e)) continue;
    if (e.esize == esize) {
      group = esize;
      break;
    }
    if (e.esize == 0) {
      group = 0;
    } else if (group != 0 && (group < 0 || dist(e.esize) < dist(group) ||
                              (dist(e.esize) == dist(group) && e.esize > group))) {
      group = e.esize;
    }
  }
  if (group < 0) return c;
  const int want = log2Bucket(bytes);
  int bestDist = 1 << 30;
  for (const Entry& e : table_)
    if (eligible(e) && e.esize == group) bestDist = std::min(bestDist, std::abs(e.log2bytes - want));
  double best = 1e300;
  for (const Entry& e : table_) {
    // the nearest measured size; the fastest entry there (ties keep the first)
    if (!eligible(e) || e.esize != group || std::abs(e.log2bytes - want) != bestDist) continue;
    if (e.us < best) {
      best = e.us;
      c.algo = e.algo;
      c.proto = e.proto;
      c.channels = e.channels;
      c.sliceBytes = e.sliceBytes;
      c.measured = true;
      c.esize = e.esize;
      c.log2bytes = e.log2bytes;
    }
  }
  return c;
}

int Tuner::load(const char* path, int nranks) {
  FILE* f = fopen(path, "r");
  if (!f) return -1;
  char line[512];
  int count = 0;
  while (fgets(line, sizeof(line), f)) {
    char* hash = strchr(line, '#');
    if (hash) *hash = 0;
    Entry e;
    unsigned long long slice = 0;
    int esize = 0;
    const int got = sscanf(line, "%d %d %d %d %d %llu %lf %d", &e.nranks, &e.algo, &e.proto, &e.channels,
                           &e.log2bytes, &slice, &e.us, &esize);
    if (got == 7 || got == 8) {
      e.sliceBytes = slice;
      e.esize = got == 8 ? esize : 0;
      if (e.nranks == nranks && e.algo >= 0 && e.algo <= 1 && e.proto >= 0 && e.proto <= 2 && e.channels >= 1 &&
          e.us > 0 && (e.esize == 0 || e.esize == 1 || e.esize == 2 || e.esize == 4 || e.esize == 8)) {
        table_.push_back(e);
        ++count;
      }
    }
  }
  fclose(f);
  forget();
  return count;
}

void Tuner::loadEnvFile(int nranks) {
  const char* p = getenv("VRCCL_TUNE_FILE");
  if (p && *p) {
    load(p, nranks);
    return;
  }
  Dl_info info;
  if (dladdr(reinterpret_cast<const void*>(&defaultChannels), &info) == 0 || !info.dli_fname) return;
  std::string dir(info.dli_fname);
  const size_t slash = dir.rfind('/');
  dir = slash == std::string::npos ? std::string(".") : dir.substr(0, slash);
  load((dir + "/tuning/gb300_n" + std::to_string(nranks) + ".txt").c_str(), nranks);
}

}  // namespace vrccl
