// profile.cu -- optional per-kernel timing.  When enabled, every launch of a
// library kernel is counted and, if its kind is selected (all kinds unless
// jfa_profile_select() narrowed them), bracketed by two CUDA events recorded on
// the launch stream; jfa_profile_read() synchronises on them and returns the
// summed device time and the launch count per kernel kind.  Disabled (the
// default) it costs one branch.
#include <cuda_runtime.h>

#include <mutex>
#include <vector>

#include "../../include/jfa.h"
#include "profile.h"

namespace jfa {
namespace {
struct Pair {
  cudaEvent_t a, b;
};
std::mutex g_mu;
bool g_on = false;
int g_mask = (1 << kNumKernelKinds) - 1;  // kinds whose launches get events
std::vector<Pair> g_pool;
std::vector<Pair> g_used[kNumKernelKinds];
int g_count[kNumKernelKinds] = {};
}  // namespace

ProfileScope::ProfileScope(int kind, cudaStream_t stream) : kind_(kind), stream_(stream) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_on || kind < 0 || kind >= kNumKernelKinds) return;
  ++g_count[kind];
  if (!(g_mask & (1 << kind))) return;
  Pair p;
  if (!g_pool.empty()) {
    p = g_pool.back();
    g_pool.pop_back();
  } else if (cudaEventCreate(&p.a) != cudaSuccess || cudaEventCreate(&p.b) != cudaSuccess) {
    return;
  }
  if (cudaEventRecord(p.a, stream_) != cudaSuccess) {
    g_pool.push_back(p);
    return;
  }
  b_ = p.b;
  a_ = p.a;
  active_ = true;
}

ProfileScope::~ProfileScope() {
  if (!active_) return;
  std::lock_guard<std::mutex> lk(g_mu);
  cudaEventRecord(b_, stream_);
  g_used[kind_].push_back({a_, b_});
}

}  // namespace jfa

using namespace jfa;

extern "C" int jfa_profile_enable(int on) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_on = on != 0;
  for (auto& v : g_used) {
    for (auto& p : v) g_pool.push_back(p);
    v.clear();
  }
  for (int& c : g_count) c = 0;
  return JFA_OK;
}

extern "C" int jfa_profile_select(int kind_mask) {
  if (kind_mask < 0 || kind_mask >= (1 << kNumKernelKinds)) return JFA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  g_mask = kind_mask;
  return JFA_OK;
}

extern "C" int jfa_profile_read(int kind, double* total_ms, int* launches) {
  if (kind < 0 || kind >= kNumKernelKinds || total_ms == nullptr || launches == nullptr) return JFA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  double t = 0.0;
  for (auto& p : g_used[kind]) {
    if (cudaEventSynchronize(p.b) != cudaSuccess) return JFA_ERR_CUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, p.a, p.b) != cudaSuccess) return JFA_ERR_CUDA;
    t += ms;
  }
  *total_ms = t;
  *launches = g_count[kind];
  return JFA_OK;
}
