// Launch accounting for benchmarks (moe_profile_enable / moe_profile_read).
#include <atomic>
#include <map>
#include <mutex>
#include <string>
#include <string.h>
#include <vector>

#include "common.cuh"

namespace moe {

namespace {

struct Rec {
  const char* name;
  cudaEvent_t a, b;
};

std::mutex g_mu;
std::atomic<bool> g_on{false};
std::vector<Rec> g_recs;
std::vector<cudaEvent_t> g_pool;

cudaEvent_t take_event() {
  if (!g_pool.empty()) {
    cudaEvent_t e = g_pool.back();
    g_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

}  // namespace

void prof_begin(const char* name, cudaStream_t s) {
  if (!g_on.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> lk(g_mu);
  Rec r{name, take_event(), take_event()};
  cudaEventRecord(r.a, s);
  g_recs.push_back(r);
}

void prof_end(cudaStream_t s) {
  if (!g_on.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_recs.empty()) cudaEventRecord(g_recs.back().b, s);
}

}  // namespace moe

extern "C" {

int moe_profile_enable(int on) {
  using namespace moe;
  std::lock_guard<std::mutex> lk(g_mu);
  if (on) {
    for (auto& r : g_recs) {
      g_pool.push_back(r.a);
      g_pool.push_back(r.b);
    }
    g_recs.clear();
  }
  g_on.store(on != 0);
  return MOE_OK;
}

int moe_profile_read(moe_profile_entry* entries, int max_entries) {
  using namespace moe;
  if (!entries || max_entries < 0) return set_error(MOE_EINVAL, "entries is NULL");
  std::lock_guard<std::mutex> lk(g_mu);
  std::map<std::string, std::pair<int, double>> agg;
  std::vector<std::string> order;
  for (auto& r : g_recs) {
    cudaError_t e = cudaEventSynchronize(r.b);
    if (e != cudaSuccess) return set_error(MOE_ECUDA, "profile sync: %s", cudaGetErrorString(e));
    float ms = 0.f;
    cudaEventElapsedTime(&ms, r.a, r.b);
    auto it = agg.find(r.name);
    if (it == agg.end()) {
      order.push_back(r.name);
      agg[r.name] = {1, ms};
    } else {
      it->second.first += 1;
      it->second.second += ms;
    }
  }
  int n = 0;
  for (auto& name : order) {
    if (n >= max_entries) break;
    moe_profile_entry& o = entries[n++];
    memset(o.name, 0, sizeof(o.name));
    strncpy(o.name, name.c_str(), sizeof(o.name) - 1);
    o.launches = agg[name].first;
    o.total_ms = agg[name].second;
  }
  return n;
}

}  // extern "C"
