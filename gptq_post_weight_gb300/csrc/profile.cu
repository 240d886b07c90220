// Launch accounting and optional per-kernel-kind timing with CUDA events
// recorded on the launching stream (the library's tracing hook).
#include "common.cuh"

#include <atomic>
#include <mutex>
#include <vector>

namespace gq {
namespace {

std::atomic<long long> g_launches{0};
std::mutex g_mu;
bool g_on = false;
int g_cap = 0;
std::vector<cudaEvent_t> g_ev;  // 2 per recorded launch
std::vector<int> g_kind;
int g_used = 0;
int g_open = -1;
unsigned g_mask = ~0u;  // kinds that record events

constexpr unsigned long long kDefaultWaitNs = 2000000000ull;  // 2 s
constexpr unsigned long long kMaxWaitNs = 10000000000ull;     // 10 s
std::atomic<unsigned long long> g_wait_ns{kDefaultWaitNs};
std::atomic<int> g_no_loads{0};

const char* kNames[K_NKINDS] = {"diag", "build", "potrf", "trsm", "fold_gemm", "ladder",
                                "sweep_block", "prep_ut", "sweep_gemm", "group", "copy",
                                "gram_prep", "gram_gemm", "place", "debias",
                                "debias_gemm", "fold_strip"};

}  // namespace

void prof_begin(int kind, cudaStream_t s) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_on || g_used >= g_cap || !((g_mask >> kind) & 1u)) return;
  cudaEventRecord(g_ev[2 * g_used], s);
  g_kind[g_used] = kind;
  g_open = g_used;
}

void prof_end(int kind, cudaStream_t s) {
  (void)kind;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_on || g_open < 0) return;
  cudaEventRecord(g_ev[2 * g_open + 1], s);
  g_used = g_open + 1;
  g_open = -1;
}

WaitCfg wait_cfg() {
  WaitCfg c;
  c.ns = g_wait_ns.load(std::memory_order_relaxed);
  c.no_loads = g_no_loads.load(std::memory_order_relaxed);
  return c;
}

}  // namespace gq

namespace gq {
bool prof_active() {
  std::lock_guard<std::mutex> lk(g_mu);
  return g_on;
}
void prof_add_launches(long long n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
}  // namespace gq

using namespace gq;

extern "C" {

gptq_status gptq_test_set_wait(unsigned long long wait_ns, int no_loads) {
  if (wait_ns > kMaxWaitNs || (no_loads != 0 && no_loads != 1)) return GPTQ_ERR_ARG;
  g_wait_ns.store(wait_ns == 0 ? kDefaultWaitNs : wait_ns);
  g_no_loads.store(no_loads);
  return GPTQ_OK;
}

long long gptq_launch_count(void) { return g_launches.load(); }

const char* gptq_kernel_kind_name(int kind) {
  return (kind >= 0 && kind < K_NKINDS) ? kNames[kind] : "?";
}

int gptq_kernel_kinds(void) { return K_NKINDS; }

void gptq_profile_select(unsigned kind_mask) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_mask = kind_mask;
}

gptq_status gptq_profile_start(int max_launches) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (max_launches <= 0) return GPTQ_ERR_ARG;
  if ((int)g_ev.size() < 2 * max_launches) {
    size_t old = g_ev.size();
    g_ev.resize(2 * (size_t)max_launches);
    for (size_t i = old; i < g_ev.size(); ++i)
      if (cudaEventCreate(&g_ev[i]) != cudaSuccess) return GPTQ_ERR_CUDA;
  }
  g_kind.assign(max_launches, 0);
  g_cap = max_launches;
  g_used = 0;
  g_open = -1;
  g_on = true;
  return GPTQ_OK;
}

int gptq_profile_stop(double* ms_by_kind, long long* launches_by_kind, int nkinds) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_on = false;
  const int nk = nkinds < K_NKINDS ? nkinds : K_NKINDS;
  for (int k = 0; k < nk; ++k) {
    if (ms_by_kind) ms_by_kind[k] = 0.0;
    if (launches_by_kind) launches_by_kind[k] = 0;
  }
  for (int i = 0; i < g_used; ++i) {
    if (cudaEventSynchronize(g_ev[2 * i + 1]) != cudaSuccess) return -1;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, g_ev[2 * i], g_ev[2 * i + 1]) != cudaSuccess) return -1;
    const int k = g_kind[i];
    if (k < nk) {
      if (ms_by_kind) ms_by_kind[k] += ms;
      if (launches_by_kind) launches_by_kind[k] += 1;
    }
  }
  const int used = g_used;
  g_used = 0;
  return used >= g_cap ? -2 : nk;
}

}  // extern "C"
