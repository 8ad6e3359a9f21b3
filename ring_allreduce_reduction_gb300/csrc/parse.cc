#include "parse.h"

#include <cctype>
#include <cstring>
#include <string>
#include <vector>

namespace vrccl {

static const char* const kFuncNames[kNumParseFuncs] = {"broadcast", "reduce", "allgather", "reducescatter",
                                                       "allreduce"};
static const char* const kAlgoNames[] = {"tree", "ring", "collnetdirect", "collnetchain", "nvls", "nvlstree", "pat"};
static const char* const kProtoNames[] = {"ll", "ll128", "simple"};

static std::string lower(std::string s) {
  for (auto& c : s) c = (char)std::tolower((unsigned char)c);
  return s;
}

static std::string trim(const std::string& s) {
  size_t a = 0, b = s.size();
  while (a < b && std::isspace((unsigned char)s[a])) ++a;
  while (b > a && std::isspace((unsigned char)s[b - 1])) --b;
  return s.substr(a, b - a);
}

static std::vector<std::string> split(const std::string& s, char sep) {
  std::vector<std::string> out;
  size_t a = 0;
  while (true) {
    const size_t b = s.find(sep, a);
    out.push_back(s.substr(a, b == std::string::npos ? std::string::npos : b - a));
    if (b == std::string::npos) break;
    a = b + 1;
  }
  return out;
}

// One list ("a,b" or "^a,b") -> mask, or -1.
static long long listMask(const std::string& list, int kind) {
  const char* const* names = kind == kParseAlgo ? kAlgoNames : kProtoNames;
  const int count = kind == kParseAlgo ? 7 : 3;
  const unsigned all = (1u << count) - 1;
  std::string body = trim(list);
  bool invert = false;
  if (!body.empty() && body[0] == '^') {
    invert = true;
    body = body.substr(1);
  }
  unsigned mask = 0;
  for (const std::string& raw : split(body, ',')) {
    const std::string tok = lower(trim(raw));
    if (tok.empty()) continue;
    int found = -1;
    for (int i = 0; i < count; ++i)
      if (tok == names[i]) found = i;
    if (found < 0) return -1;  // "Unrecognized element token"
    mask |= 1u << found;
  }
  return invert ? (all & ~mask) : mask;
}

int parseList(const char* s, int kind, unsigned masks[kNumParseFuncs]) {
  const unsigned all = kind == kParseAlgo ? 0x7Fu : 0x7u;
  for (int f = 0; f < kNumParseFuncs; ++f) masks[f] = all;
  if (!s) return 0;
  const std::vector<std::string> groups = split(s, ';');
  for (size_t g = 0; g < groups.size(); ++g) {
    const std::string grp = trim(groups[g]);
    if (grp.empty()) continue;
    const size_t colon = grp.find(':');
    int func = -1;  // -1: every function
    std::string list = grp;
    if (colon != std::string::npos) {
      const std::string fn = lower(trim(grp.substr(0, colon)));
      for (int f = 0; f < kNumParseFuncs; ++f)
        if (fn == kFuncNames[f]) func = f;
      if (func < 0) return -1;
      list = grp.substr(colon + 1);
    }
    const long long m = listMask(list, kind);
    if (m < 0) return -1;
    for (int f = 0; f < kNumParseFuncs; ++f)
      if (func < 0 || f == func) masks[f] = (unsigned)m;
  }
  return 0;
}

}  // namespace vrccl
