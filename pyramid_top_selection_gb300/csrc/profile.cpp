// Per-kernel CUDA-event timing for the C ABI's profiling calls. Single host thread: the
// calls are meant for a benchmark loop, not for concurrent use.
#include "profile.h"

#include <cstring>
#include <string>
#include <vector>

#include "internal.h"

namespace pisa {
namespace {

constexpr int kPairs = 1 << 14;

struct Rec {
  const char* name;
  cudaEvent_t b, e;
};

struct Prof {
  bool on = false;
  bool overflow = false;
  std::vector<Rec> recs;
  int used = 0;
} g_prof;

}  // namespace

ProfScope::ProfScope(cudaStream_t st, const char* name) : st_(st), slot_(-1) {
  if (!g_prof.on) return;
  if (g_prof.used >= static_cast<int>(g_prof.recs.size())) {
    g_prof.overflow = true;
    return;
  }
  slot_ = g_prof.used++;
  g_prof.recs[slot_].name = name;
  cudaEventRecord(g_prof.recs[slot_].b, st_);
}

ProfScope::~ProfScope() {
  if (slot_ >= 0) cudaEventRecord(g_prof.recs[slot_].e, st_);
}

}  // namespace pisa

extern "C" {

int pisa_profile_start(void) {
  using pisa::g_prof;
  if (g_prof.recs.empty()) {
    g_prof.recs.resize(pisa::kPairs);
    for (auto& r : g_prof.recs) {
      if (cudaEventCreate(&r.b) != cudaSuccess || cudaEventCreate(&r.e) != cudaSuccess) {
        g_prof.recs.clear();
        return PISA_ECUDA;
      }
    }
  }
  g_prof.used = 0;
  g_prof.overflow = false;
  g_prof.on = true;
  return PISA_OK;
}

int pisa_profile_stop(void) {
  pisa::g_prof.on = false;
  return PISA_OK;
}

int pisa_profile_read(pisa_profile_entry_t* out, int32_t max_entries, int32_t* n_entries) {
  using pisa::g_prof;
  if (!out || !n_entries || max_entries < 0) return PISA_EINVAL;
  int n = 0;
  for (int k = 0; k < g_prof.used; ++k) {
    const auto& r = g_prof.recs[k];
    if (cudaEventSynchronize(r.e) != cudaSuccess) return PISA_ECUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, r.b, r.e) != cudaSuccess) return PISA_ECUDA;
    int j = 0;
    while (j < n && std::strncmp(out[j].name, r.name, sizeof(out[j].name)) != 0) ++j;
    if (j == n) {
      if (n >= max_entries) continue;
      std::memset(&out[n], 0, sizeof(out[n]));
      std::strncpy(out[n].name, r.name, sizeof(out[n].name) - 1);
      ++n;
    }
    out[j].launches += 1;
    out[j].total_ms += ms;
  }
  *n_entries = n;
  g_prof.used = 0;
  return g_prof.overflow ? PISA_EWORKSPACE : PISA_OK;
}

}  // extern "C"
