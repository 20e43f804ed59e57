// Event-based per-kernel timing (see prof.h) and its C entry points.
#include <string.h>

#include <atomic>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/csa.h"
#include "prof.h"

namespace csa {
namespace {

struct Rec {
  cudaEvent_t a = nullptr, b = nullptr;
  const char* name = nullptr;
};

constexpr int kMaxRecs = 1 << 15;
std::atomic<bool> g_on{false};
std::mutex g_mu;
std::vector<Rec> g_pool;  // events, created once when profiling is first enabled
int g_used = 0;

}  // namespace

bool prof_enabled() { return g_on.load(std::memory_order_relaxed); }

int prof_begin(cudaStream_t stream, const char* name) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_used >= (int)g_pool.size()) return -1;
  Rec& r = g_pool[g_used];
  r.name = name;
  if (cudaEventRecord(r.a, stream) != cudaSuccess) return -1;
  return g_used++;
}

void prof_end(cudaStream_t stream, int slot) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (slot >= 0 && slot < (int)g_pool.size()) cudaEventRecord(g_pool[slot].b, stream);
}

}  // namespace csa

using namespace csa;

extern "C" {

csa_status csa_profiler_enable(int on) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (on && g_pool.empty()) {
    g_pool.resize(kMaxRecs);
    for (Rec& r : g_pool) {
      if (cudaEventCreate(&r.a) != cudaSuccess || cudaEventCreate(&r.b) != cudaSuccess)
        return CSA_ERR_CUDA;
    }
  }
  g_on.store(on != 0);
  return CSA_OK;
}

csa_status csa_profiler_collect(csa_kernel_time* out, int max_entries, int* n_entries, int reset) {
  if (!n_entries || (max_entries > 0 && !out)) return CSA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  std::vector<std::string> names;
  std::vector<double> ms;
  std::vector<int> cnt;
  for (int i = 0; i < g_used; ++i) {
    Rec& r = g_pool[i];
    if (cudaEventSynchronize(r.b) != cudaSuccess) return CSA_ERR_CUDA;
    float t = 0.f;
    if (cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) return CSA_ERR_CUDA;
    size_t j = 0;
    while (j < names.size() && names[j] != r.name) ++j;
    if (j == names.size()) {
      names.emplace_back(r.name);
      ms.push_back(0.0);
      cnt.push_back(0);
    }
    ms[j] += t;
    cnt[j] += 1;
  }
  const int n = (int)names.size();
  for (int j = 0; j < n && j < max_entries; ++j) {
    memset(&out[j], 0, sizeof(out[j]));
    strncpy(out[j].name, names[j].c_str(), sizeof(out[j].name) - 1);
    out[j].launches = cnt[j];
    out[j].total_ms = ms[j];
  }
  *n_entries = n;
  if (reset) g_used = 0;
  return CSA_OK;
}

}  // extern "C"
