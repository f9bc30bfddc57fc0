// Opt-in per-kernel timing (mf_timing_* in mf.h): CUDA events around each kernel
// launch on the launching stream, accumulated per kernel id when read.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "../../include/mf.h"
#include "common.cuh"

namespace mf {
namespace {
struct Rec {
  int id;
  cudaEvent_t a, b;
};
std::atomic<bool> g_on{false};
std::mutex g_mu;
std::vector<Rec> g_pending;
std::vector<cudaEvent_t> g_pool;
double g_ms[MF_K_COUNT] = {};
int64_t g_n[MF_K_COUNT] = {};

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

// Fold completed records into the totals (caller holds g_mu).
bool drain_locked() {
  bool ok = true;
  for (const Rec& r : g_pending) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess)
      ok = false;
    g_ms[r.id] += ms;
    g_n[r.id] += 1;
    g_pool.push_back(r.a);
    g_pool.push_back(r.b);
  }
  g_pending.clear();
  return ok;
}
}  // namespace

KernelTimer::KernelTimer(int id, cudaStream_t s) : id_(id), s_(s) {
  if (!g_on.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> lk(g_mu);
  a_ = take_event();
  if (a_ != nullptr && cudaEventRecord(static_cast<cudaEvent_t>(a_), s) != cudaSuccess) a_ = nullptr;
}

KernelTimer::~KernelTimer() {
  if (a_ == nullptr) return;
  std::lock_guard<std::mutex> lk(g_mu);
  cudaEvent_t b = take_event();
  if (b == nullptr || cudaEventRecord(b, s_) != cudaSuccess) return;
  g_pending.push_back(Rec{id_, static_cast<cudaEvent_t>(a_), b});
}

}  // namespace mf

using namespace mf;

extern "C" {

mf_status mf_timing_enable(int32_t on) {
  g_on.store(on != 0);
  return MF_OK;
}

mf_status mf_timing_reset(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  const bool ok = drain_locked();
  for (int i = 0; i < MF_K_COUNT; ++i) {
    g_ms[i] = 0.0;
    g_n[i] = 0;
  }
  return ok ? MF_OK : MF_ERR_CUDA;
}

mf_status mf_timing_read(int32_t id, double* total_ms, int64_t* launches) {
  if (id < 0 || id >= MF_K_COUNT) return MF_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  const bool ok = drain_locked();
  if (total_ms) *total_ms = g_ms[id];
  if (launches) *launches = g_n[id];
  return ok ? MF_OK : MF_ERR_CUDA;
}

}  // extern "C"
