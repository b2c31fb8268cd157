// Launch profiler of libsa2: when enabled, every kernel launch of the library is bracketed
// by two CUDA events recorded on its stream, so a caller can read each kernel's device
// time and launch count without an external profiler.  Disabled by default (one relaxed
// atomic load per launch).
#include <atomic>
#include <mutex>
#include <vector>

#include "../../include/sa2.h"
#include "sa2_internal.h"

namespace sa2 {
namespace {

struct Record {
  int id;
  cudaEvent_t start, stop;
};

std::atomic<int> g_enabled{0};
std::mutex g_mu;
std::vector<Record> g_open;         // started, not yet stopped (per id, at most one per stream)
std::vector<Record> g_done;         // stopped, not yet collected
std::vector<cudaEvent_t> g_pool;    // events ready for reuse

const char* kNames[kNumKernelIds] = {"pool", "select", "csc", "to_f16", "attn_fwd",
                                     "bwd_preprocess", "attn_bwd_dkdv", "attn_bwd_dq",
                                     "bwd_pair_union", "vd_loss", "score_tc", "item_order"};

cudaEvent_t take_event() {
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

void prof_start(cudaStream_t st, int id) {
  if (!g_enabled.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> lk(g_mu);
  Record r{id, take_event(), take_event()};
  if (!r.start || !r.stop) return;
  cudaEventRecord(r.start, st);
  g_open.push_back(r);
}

void prof_stop(cudaStream_t st, int id) {
  if (!g_enabled.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> lk(g_mu);
  for (size_t i = g_open.size(); i-- > 0;) {
    if (g_open[i].id == id) {
      cudaEventRecord(g_open[i].stop, st);
      g_done.push_back(g_open[i]);
      g_open.erase(g_open.begin() + (long)i);
      return;
    }
  }
}

}  // namespace sa2

extern "C" {

void sa2_profiler_enable(int on) { sa2::g_enabled.store(on ? 1 : 0); }

int sa2_profiler_collect(sa2_kernel_time* out, int max_entries) {
  using namespace sa2;
  if (!out) return kNumKernelIds;  // size query: records stay for the next call
  std::lock_guard<std::mutex> lk(g_mu);
  double ms[kNumKernelIds] = {0};
  int launches[kNumKernelIds] = {0};
  int status = 0;
  for (const Record& r : g_done) {
    float t = 0.f;
    if (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&t, r.start, r.stop) != cudaSuccess)
      status = -1;
    if (r.id >= 0 && r.id < kNumKernelIds) {
      ms[r.id] += t;
      launches[r.id] += 1;
    }
    g_pool.push_back(r.start);
    g_pool.push_back(r.stop);
  }
  g_done.clear();
  if (status != 0) return -1;
  int n = 0;
  for (int id = 0; id < kNumKernelIds && n < max_entries; ++id) {
    out[n].name = kNames[id];
    out[n].launches = launches[id];
    out[n].total_ms = ms[id];
    ++n;
  }
  return n;
}

}  // extern "C"
