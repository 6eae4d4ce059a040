// pa_profile.cu -- kernel timing with CUDA events (see pa_profile_enable in
// include/pa.h).  Each bracketed launch takes a pair of pooled events; reading
// synchronises on the end events, sums elapsed time per kernel id and returns
// the pairs to the pool.
#include <mutex>
#include <vector>

#include "pa_internal.h"

namespace pa {
namespace {

struct Record {
  int id;
  cudaEvent_t start, end;
};

std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<Record> g_records;
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

bool capturing(cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  return cudaStreamIsCapturing(st, &cs) == cudaSuccess && cs != cudaStreamCaptureStatusNone;
}

}  // namespace

int prof_begin(int id, cudaStream_t st) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  if (!g_prof_on || capturing(st)) return -1;
  Record r{id, take_event(), take_event()};
  if (!r.start || !r.end || cudaEventRecord(r.start, st) != cudaSuccess) {
    cudaGetLastError();
    if (r.start) g_pool.push_back(r.start);
    if (r.end) g_pool.push_back(r.end);
    return -1;
  }
  g_records.push_back(r);
  return (int)g_records.size() - 1;
}

void prof_end(int slot, cudaStream_t st) {
  if (slot < 0) return;
  std::lock_guard<std::mutex> lock(g_prof_mu);
  if (slot < (int)g_records.size()) cudaEventRecord(g_records[slot].end, st);
}

}  // namespace pa

using namespace pa;

extern "C" {

pa_status pa_profile_enable(int on) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  g_prof_on = on != 0;
  return PA_OK;
}

pa_status pa_profile_read(double *total_ms, int *launches) {
  if (!total_ms || !launches) return PA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_prof_mu);
  for (int i = 0; i < PA_K_COUNT; ++i) {
    total_ms[i] = 0.0;
    launches[i] = 0;
  }
  pa_status st = PA_OK;
  for (const Record &r : g_records) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.end) != cudaSuccess ||
        cudaEventElapsedTime(&ms, r.start, r.end) != cudaSuccess) {
      cudaGetLastError();
      st = PA_ERR_CUDA;
    } else if (r.id >= 0 && r.id < PA_K_COUNT) {
      total_ms[r.id] += ms;
      launches[r.id] += 1;
    }
    g_pool.push_back(r.start);
    g_pool.push_back(r.end);
  }
  g_records.clear();
  return st;
}

const char *pa_kernel_name(int kernel_id) {
  switch (kernel_id) {
    case PA_K_PLAN: return "plan";
    case PA_K_ROW: return "row";
    case PA_K_TILE: return "tile";
    case PA_K_MERGE: return "merge";
    case PA_K_MLA: return "mla";
    case PA_K_MLA_MERGE: return "mla_merge";
    case PA_K_GATHER: return "gather";
    case PA_K_UPPROJ: return "upproj";
    case PA_K_MLA_ROPE: return "mla_rope";
  }
  return "unknown";
}

}  // extern "C"
