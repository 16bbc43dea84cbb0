// Status strings and the device error query of the moet C ABI.
#include <atomic>
#include <mutex>
#include <vector>

#include "common.cuh"

namespace moet {
namespace {
constexpr int kMaxTimed = 8192;
std::atomic<bool> g_prof_on{false};
std::mutex g_prof_mu;
struct Rec { int kind; cudaEvent_t a, b; };
std::vector<cudaEvent_t> g_pool;          // created lazily, reused
std::vector<Rec> g_recs;
int g_launches[MOET_KERNEL_KINDS] = {0};
int g_open_kind = -1;
cudaEvent_t g_open_a = nullptr;

cudaEvent_t take_event() {
  const size_t used = 2 * g_recs.size() + (g_open_a ? 1 : 0);
  while (g_pool.size() <= used) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    g_pool.push_back(e);
  }
  return g_pool[used];
}
}  // namespace

void prof_begin(int kind, cudaStream_t st) {
  if (!g_prof_on.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_launches[kind] += 1;
  if ((int)g_recs.size() >= kMaxTimed) return;
  cudaEvent_t a = take_event();
  if (!a) return;
  cudaEventRecord(a, st);
  g_open_kind = kind;
  g_open_a = a;
}

void prof_end(int kind, cudaStream_t st) {
  if (!g_prof_on.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (g_open_a == nullptr || g_open_kind != kind) return;
  const size_t used = 2 * g_recs.size() + 1;
  while (g_pool.size() <= used) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) { g_open_a = nullptr; return; }
    g_pool.push_back(e);
  }
  cudaEvent_t b = g_pool[used];
  cudaEventRecord(b, st);
  g_recs.push_back(Rec{kind, g_open_a, b});
  g_open_a = nullptr;
  g_open_kind = -1;
}
}  // namespace moet

extern "C" moet_status moet_profile_enable(int on) {
  moet::g_prof_on.store(on != 0);
  return MOET_OK;
}

extern "C" moet_status moet_profile_read(int* launches, int* timed, float* total_ms) {
  if (!launches || !timed || !total_ms) return MOET_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(moet::g_prof_mu);
  for (int i = 0; i < MOET_KERNEL_KINDS; ++i) {
    launches[i] = moet::g_launches[i];
    timed[i] = 0;
    total_ms[i] = 0.0f;
    moet::g_launches[i] = 0;
  }
  moet_status st = MOET_OK;
  for (const auto& r : moet::g_recs) {
    float ms = 0.0f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) {
      st = MOET_ERR_CUDA;
      continue;
    }
    timed[r.kind] += 1;
    total_ms[r.kind] += ms;
  }
  moet::g_recs.clear();
  return st;
}

extern "C" __attribute__((visibility("hidden"))) int moet_internal_error_requant(void);
extern "C" __attribute__((visibility("hidden"))) int moet_internal_error_route(void);
extern "C" __attribute__((visibility("hidden"))) int moet_internal_error_moe(void);
extern "C" __attribute__((visibility("hidden"))) int moet_internal_error_moe_tc(void);
extern "C" __attribute__((visibility("hidden"))) int moet_internal_error_moe_pf(void);
extern "C" __attribute__((visibility("hidden"))) int moet_internal_debug_waits_moe_tc(int, int);
extern "C" __attribute__((visibility("hidden"))) int moet_internal_debug_waits_moe_pf(int, int);

extern "C" moet_status moet_debug_wait_expiry(int polls, int withhold) {
  if (polls < 0 || (withhold != 0 && withhold != 1)) return MOET_ERR_INVALID_ARG;
  if (moet_internal_debug_waits_moe_tc(polls, withhold) != 0 ||
      moet_internal_debug_waits_moe_pf(polls, withhold) != 0)
    return MOET_ERR_CUDA;
  return MOET_OK;
}

extern "C" const char* moet_status_string(moet_status s) {
  switch (s) {
    case MOET_OK: return "MOET_OK";
    case MOET_ERR_INVALID_ARG: return "MOET_ERR_INVALID_ARG";
    case MOET_ERR_SHAPE: return "MOET_ERR_SHAPE";
    case MOET_ERR_ALIGN: return "MOET_ERR_ALIGN";
    case MOET_ERR_UNSUPPORTED: return "MOET_ERR_UNSUPPORTED";
    case MOET_ERR_WORKSPACE: return "MOET_ERR_WORKSPACE";
    case MOET_ERR_CUDA: return "MOET_ERR_CUDA";
    case MOET_ERR_TIMEOUT: return "MOET_ERR_TIMEOUT";
    case MOET_ERR_DEVICE_INDEX: return "MOET_ERR_DEVICE_INDEX";
  }
  return "MOET_ERR_UNKNOWN";
}

extern "C" moet_status moet_last_device_error(moet_stream stream) {
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return MOET_ERR_CUDA;
  int first = 0;
  const int codes[5] = {moet_internal_error_requant(), moet_internal_error_route(),
                        moet_internal_error_moe(), moet_internal_error_moe_tc(), moet_internal_error_moe_pf()};
  for (int c : codes) {
    if (c < 0) return MOET_ERR_CUDA;
    if (first == 0 && c != 0) first = c;
  }
  return (moet_status)first;
}
