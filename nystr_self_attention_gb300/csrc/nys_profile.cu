// Launch counter and optional per-kernel CUDA-event timing (nystrom.h:
// nystrom_launch_count, nystrom_profile_enable, nystrom_profile_read).
#include <cuda_runtime.h>

#include <atomic>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "nys_internal.h"

namespace nys {
namespace {

std::atomic<unsigned long long> g_launches{0};
std::atomic<bool> g_profiling{false};

struct Record {
  const char* name;
  cudaEvent_t begin, end;
};
std::mutex g_mu;
std::vector<Record> g_records;
std::vector<cudaEvent_t> g_pool;

cudaEvent_t take_event() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_pool.empty()) {
    cudaEvent_t e = g_pool.back();
    g_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

}  // namespace

KernelScope::KernelScope(const char* name, cudaStream_t stream) : name_(name), stream_(stream) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (g_profiling.load(std::memory_order_relaxed)) {
    begin_ = take_event();
    if (begin_) cudaEventRecord(begin_, stream_);
  }
}

KernelScope::~KernelScope() {
  if (!begin_) return;
  cudaEvent_t end = take_event();
  if (!end) return;
  cudaEventRecord(end, stream_);
  std::lock_guard<std::mutex> lk(g_mu);
  g_records.push_back({name_, begin_, end});
}

}  // namespace nys

extern "C" {

unsigned long long nystrom_launch_count(void) { return nys::g_launches.load(); }

int nystrom_profile_enable(int on) {
  nys::g_profiling.store(on != 0);
  return NYS_OK;
}

int nystrom_profile_read(int max_kernels, char* names, int name_len, double* total_ms,
                         long long* launches) {
  std::vector<nys::Record> recs;
  {
    std::lock_guard<std::mutex> lk(nys::g_mu);
    recs.swap(nys::g_records);
  }
  std::map<std::string, std::pair<double, long long>> agg;
  std::vector<std::string> order;
  int rc = NYS_OK;
  for (auto& r : recs) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.end) != cudaSuccess ||
        cudaEventElapsedTime(&ms, r.begin, r.end) != cudaSuccess)
      rc = NYS_ERR_CUDA;
    auto it = agg.find(r.name);
    if (it == agg.end()) {
      order.push_back(r.name);
      agg[r.name] = {ms, 1};
    } else {
      it->second.first += ms;
      it->second.second += 1;
    }
    std::lock_guard<std::mutex> lk(nys::g_mu);
    nys::g_pool.push_back(r.begin);
    nys::g_pool.push_back(r.end);
  }
  if (rc != NYS_OK) return rc;
  const int count = (int)order.size();
  for (int i = 0; i < count && i < max_kernels; ++i) {
    if (names && name_len > 0) {
      std::strncpy(names + (size_t)i * name_len, order[i].c_str(), name_len - 1);
      names[(size_t)i * name_len + name_len - 1] = '\0';
    }
    if (total_ms) total_ms[i] = agg[order[i]].first;
    if (launches) launches[i] = agg[order[i]].second;
  }
  return count;
}

}  // extern "C"
