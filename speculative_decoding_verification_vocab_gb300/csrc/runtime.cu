// runtime.cu -- host-side error reporting, launch accounting and tracing.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "common.cuh"

namespace sv {

static thread_local char g_err[512] = "";

sv_status set_error(sv_status st, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return st;
}

sv_status check_launch(const char *what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return set_error(SV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return SV_OK;
}

sv_status check_launch(const char *what, cudaError_t launched) {
  if (launched != cudaSuccess) {
    cudaGetLastError();  // clear the sticky copy of a launch error
    return set_error(SV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(launched));
  }
  return check_launch(what);
}

sv_status map_ptr(const void **p, const char *what) {
  if (!*p) return SV_OK;
  cudaPointerAttributes a;
  cudaError_t e = cudaPointerGetAttributes(&a, *p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return set_error(SV_ERR_INVALID_ARG, "%s: pointer not usable by CUDA (%s)", what,
                     cudaGetErrorString(e));
  }
  int dev = -1;
  cudaGetDevice(&dev);
  switch (a.type) {
    case cudaMemoryTypeDevice:
      if (a.device != dev)
        return set_error(SV_ERR_INVALID_ARG, "%s: memory of device %d, current device %d", what,
                         a.device, dev);
      return SV_OK;
    case cudaMemoryTypeManaged:
      return SV_OK;
    case cudaMemoryTypeHost:
      if (!a.devicePointer)
        return set_error(SV_ERR_INVALID_ARG, "%s: page-locked host memory with no device mapping",
                         what);
      *p = a.devicePointer;
      return SV_OK;
    default:
      return set_error(SV_ERR_INVALID_ARG,
                       "%s: pageable host memory (page-lock it or copy it to the device)", what);
  }
}

int is_device_memory(const void *p) {
  cudaPointerAttributes a;
  if (!p || cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return a.type == cudaMemoryTypeDevice;
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  return n;
}

// ---------------------------------------------------------------- tracing
namespace {
struct TraceRec {
  const char *name;
  cudaEvent_t beg, end;
};
std::atomic<uint64_t> g_launches{0};
std::atomic<int> g_tracing{0};
std::mutex g_mu;
std::vector<TraceRec> g_recs;    // events recorded so far
std::vector<cudaEvent_t> g_pool; // spare events
constexpr size_t kMaxRecs = 1 << 16;

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

LaunchScope::LaunchScope(const char *name, cudaStream_t s) : slot(-1), stream(s) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (!g_tracing.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_recs.size() >= kMaxRecs) return;
  TraceRec r{name, take_event(), take_event()};
  if (!r.beg || !r.end) return;
  cudaEventRecord(r.beg, s);
  g_recs.push_back(r);
  slot = (int)g_recs.size() - 1;
}

LaunchScope::~LaunchScope() {
  if (slot < 0) return;
  std::lock_guard<std::mutex> lk(g_mu);
  cudaEventRecord(g_recs[slot].end, stream);
}

}  // namespace sv

using namespace sv;

extern "C" const char *sv_last_error(void) { return g_err; }

extern "C" uint64_t sv_launch_count(void) { return g_launches.load(); }

extern "C" sv_status sv_trace_enable(int on) {
  g_tracing.store(on ? 1 : 0);
  return SV_OK;
}

extern "C" int sv_trace_collect(sv_trace_entry *out, int max) {
  std::lock_guard<std::mutex> lk(g_mu);
  std::vector<sv_trace_entry> agg;
  int rc = 0;
  for (auto &r : g_recs) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.end) != cudaSuccess ||
        cudaEventElapsedTime(&ms, r.beg, r.end) != cudaSuccess) {
      set_error(SV_ERR_CUDA, "sv_trace_collect: %s", cudaGetErrorString(cudaGetLastError()));
      rc = -1;
      break;
    }
    size_t i = 0;
    for (; i < agg.size(); ++i)
      if (strncmp(agg[i].name, r.name, sizeof agg[i].name) == 0) break;
    if (i == agg.size()) {
      sv_trace_entry e;
      memset(&e, 0, sizeof e);
      strncpy(e.name, r.name, sizeof e.name - 1);
      agg.push_back(e);
    }
    agg[i].launches += 1;
    agg[i].total_ms += ms;
  }
  for (auto &r : g_recs) {
    g_pool.push_back(r.beg);
    g_pool.push_back(r.end);
  }
  g_recs.clear();
  if (rc < 0) return -1;
  int n = 0;
  for (; n < (int)agg.size() && n < max; ++n) out[n] = agg[n];
  return n;
}
