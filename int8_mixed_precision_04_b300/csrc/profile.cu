// Per-kernel CUDA-event timing (see bnb_profile_* in include/bnb_int8.h).
#include <atomic>
#include <mutex>
#include <vector>

#include "kernels.h"

namespace bnb {

static const char *const kKernelNames[kKernelCount] = {
    "memset_status_mask", "outlier_scan", "quantize_rows", "dec_fused",
    "gemm_mma",           "gemm_tc",      "quantize_weight",
    "quantize_blockwise", "dequantize_blockwise"};

namespace {
struct Rec {
  int kid;
  cudaEvent_t a, b;
};
std::mutex g_mu;
bool g_on = false;
std::atomic<int> g_mode{0};
std::vector<Rec> g_recs;
std::vector<cudaEvent_t> g_pool;

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

bool profile_only_main() { return g_mode.load(std::memory_order_relaxed) == 2; }

ProfScope::ProfScope(int kid, cudaStream_t s) : kid_(kid), s_(s), a_(nullptr) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_on) return;
  a_ = take_event();
  if (a_ && cudaEventRecord(a_, s_) != cudaSuccess) {
    g_pool.push_back(a_);
    a_ = nullptr;
  }
}

ProfScope::~ProfScope() {
  if (!a_) return;
  std::lock_guard<std::mutex> lk(g_mu);
  cudaEvent_t b = take_event();
  if (!b || cudaEventRecord(b, s_) != cudaSuccess) {
    g_pool.push_back(a_);
    if (b) g_pool.push_back(b);
    return;
  }
  g_recs.push_back(Rec{kid_, a_, b});
}

}  // namespace bnb

using namespace bnb;

extern "C" {

void bnb_profile_enable(int mode) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_on = mode == 1;
  g_mode.store(mode == 1 || mode == 2 ? mode : 0, std::memory_order_relaxed);
}

bnb_status_t bnb_profile_collect(double *ms, uint64_t *n) {
  std::lock_guard<std::mutex> lk(g_mu);
  bnb_status_t st = BNB_OK;
  for (const Rec &r : g_recs) {
    float t = 0.f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess)
      st = BNB_ERR_CUDA;
    else if (r.kid >= 0 && r.kid < kKernelCount) {
      if (ms) ms[r.kid] += t;
      if (n) n[r.kid] += 1;
    }
    g_pool.push_back(r.a);
    g_pool.push_back(r.b);
  }
  g_recs.clear();
  return st;
}

int bnb_profile_kernel_count(void) { return kKernelCount; }

const char *bnb_profile_kernel_name(int id) {
  return (id >= 0 && id < kKernelCount) ? kKernelNames[id] : nullptr;
}

}  // extern "C"
