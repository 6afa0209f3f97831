// ssd_profile.cu -- optional per-kernel timing of libssd's launches with CUDA
// events recorded on the launching stream (a measurement aid: while enabled,
// each kernel of ssd_fwd/ssd_bwd is bracketed by two events).
#include <mutex>
#include <string.h>
#include <vector>

#include "ssd_internal.cuh"

namespace ssd {

namespace {

constexpr int kPoolEvents = 65536;  // two per launch

struct Rec {
  const char* name;
  cudaEvent_t a, b;
};

std::mutex g_mu;
bool g_on = false;
int g_dev = -1;
std::vector<cudaEvent_t> g_pool;
std::vector<Rec> g_recs;
size_t g_next = 0;
long long g_dropped = 0;

struct Stat {
  const char* name;
  int launches;
  double ms;
};
std::vector<Stat> g_stats;

thread_local const char* t_name = nullptr;
thread_local cudaEvent_t t_start = nullptr;

}  // namespace

void set_kernel_name(const char* name) { t_name = name; }

void prof_before(cudaStream_t s) {
  t_start = nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_on || g_next + 2 > g_pool.size()) {
    if (g_on) ++g_dropped;
    return;
  }
  t_start = g_pool[g_next++];
  cudaEventRecord(t_start, s);
}

void prof_after(cudaStream_t s) {
  if (t_start == nullptr) return;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_on || g_next >= g_pool.size()) return;
  cudaEvent_t b = g_pool[g_next++];
  cudaEventRecord(b, s);
  g_recs.push_back(Rec{t_name ? t_name : "?", t_start, b});
  t_start = nullptr;
}

}  // namespace ssd

using namespace ssd;

extern "C" {

int ssd_profile_start(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SSD_ERR_CUDA;
  if (g_pool.empty() || g_dev != dev) {
    for (cudaEvent_t e : g_pool) cudaEventDestroy(e);
    g_pool.clear();
    for (int i = 0; i < kPoolEvents; ++i) {
      cudaEvent_t e;
      if (cudaEventCreate(&e) != cudaSuccess) return SSD_ERR_CUDA;
      g_pool.push_back(e);
    }
    g_dev = dev;
  }
  g_recs.clear();
  g_stats.clear();
  g_next = 0;
  g_dropped = 0;
  g_on = true;
  return SSD_OK;
}

int ssd_profile_stop(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_on = false;
  // fold the records into per-kernel totals (waits for the recorded events)
  for (const Rec& r : g_recs) {
    if (cudaEventSynchronize(r.b) != cudaSuccess) return SSD_ERR_CUDA;
    float ms = 0.0f;
    if (cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) return SSD_ERR_CUDA;
    bool found = false;
    for (Stat& s : g_stats)
      if (strcmp(s.name, r.name) == 0) {
        s.launches += 1;
        s.ms += ms;
        found = true;
      }
    if (!found) g_stats.push_back(Stat{r.name, 1, (double)ms});
  }
  g_recs.clear();
  g_next = 0;
  return g_dropped ? SSD_ERR_WORKSPACE_TOO_SMALL : SSD_OK;
}

int ssd_profile_count(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  return (int)g_stats.size();
}

int ssd_profile_get(int i, const char** name, int* launches, double* total_ms) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (i < 0 || i >= (int)g_stats.size() || !name || !launches || !total_ms)
    return SSD_ERR_INVALID_ARGUMENT;
  *name = g_stats[i].name;
  *launches = g_stats[i].launches;
  *total_ms = g_stats[i].ms;
  return SSD_OK;
}

}  // extern "C"
