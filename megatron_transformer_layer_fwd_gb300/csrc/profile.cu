// Kernel timing and launch counting.
//
// Every kernel launch of the library goes through a LaunchScope. The scope
// always counts launches; when profiling is enabled it also records a CUDA
// event before and after the launch on the launching stream, so elapsed times
// are device times of exactly those kernels. Results are grouped by kernel
// kind and read (after an event synchronisation) by mgb_profile_read.
#include <atomic>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace mgb {

namespace {

struct Pending {
  int kind;
  int launches;
  cudaEvent_t a, b;
};

std::atomic<uint64_t> g_launches{0};
std::atomic<int> g_enabled{0};
std::mutex g_mu;
std::vector<Pending> g_pending;
std::vector<cudaEvent_t> g_free;
double g_total_ms[PROF_KINDS] = {};
int64_t g_count[PROF_KINDS] = {};

cudaEvent_t take_event() {
  if (!g_free.empty()) {
    cudaEvent_t e = g_free.back();
    g_free.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Fold finished event pairs into the totals (caller holds g_mu).
mgb_status drain_locked() {
  for (const Pending& p : g_pending) {
    if (cudaEventSynchronize(p.b) != cudaSuccess) return MGB_ERR_CUDA;
    float ms = 0.0f;
    if (cudaEventElapsedTime(&ms, p.a, p.b) != cudaSuccess) return MGB_ERR_CUDA;
    g_total_ms[p.kind] += ms;
    g_count[p.kind] += p.launches;
    g_free.push_back(p.a);
    g_free.push_back(p.b);
  }
  g_pending.clear();
  return MGB_OK;
}

const char* kKindNames[PROF_KINDS] = {
    "gemm_tc_fwd",  "gemm_tc_dgrad", "gemm_tc_wgrad", "gemm_f32",  "attn_fwd",   "attn_bwd",
    "layernorm_fwd", "layernorm_bwd", "colsum",       "ce_stats", "ce_combine", "ce_grad",
    "gemm_tc_ce_logits", "embedding", "dropout", "gemm_tc_ce_dgrad", "gemm_tc_ce_wgrad",
    "splitk_reduce",
    "stage_attention", "stage_ffn", "stage_backward", "stage_ce_products"};

}  // namespace

LaunchScope::LaunchScope(int kind, cudaStream_t st, int launches, bool count_launches)
    : kind_(kind), launches_(launches), st_(st), a_(nullptr) {
  if (count_launches) g_launches.fetch_add((uint64_t)launches, std::memory_order_relaxed);
  if (g_enabled.load(std::memory_order_relaxed)) {
    std::lock_guard<std::mutex> lock(g_mu);
    a_ = take_event();
    if (a_ && cudaEventRecord(static_cast<cudaEvent_t>(a_), st) != cudaSuccess) a_ = nullptr;
  }
}

LaunchScope::~LaunchScope() {
  if (a_ == nullptr) return;
  std::lock_guard<std::mutex> lock(g_mu);
  cudaEvent_t b = take_event();
  if (b && cudaEventRecord(b, st_) == cudaSuccess)
    g_pending.push_back({kind_, launches_, static_cast<cudaEvent_t>(a_), b});
}

}  // namespace mgb

using namespace mgb;

extern "C" {

uint64_t mgb_launch_count(void) { return g_launches.load(); }

mgb_status mgb_profile_enable(int32_t on) {
  g_enabled.store(on ? 1 : 0);
  return MGB_OK;
}

mgb_status mgb_profile_reset(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  const mgb_status s = drain_locked();
  for (int k = 0; k < PROF_KINDS; ++k) {
    g_total_ms[k] = 0.0;
    g_count[k] = 0;
  }
  return s;
}

int32_t mgb_profile_kinds(void) { return PROF_KINDS; }

const char* mgb_profile_kind_name(int32_t kind) {
  return (kind >= 0 && kind < PROF_KINDS) ? kKindNames[kind] : "";
}

mgb_status mgb_profile_read(int32_t kind, double* total_ms, int64_t* launches) {
  if (kind < 0 || kind >= PROF_KINDS) return MGB_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  const mgb_status s = drain_locked();
  if (total_ms) *total_ms = g_total_ms[kind];
  if (launches) *launches = g_count[kind];
  return s;
}

}  // extern "C"
