// pa_static.cu -- pa_forward_static_scratch: unified paged attention with
// its scratch in a fixed, file-scope device array instead of library-
// allocated workspace (see include/pa.h for who needs this and why).
#include <mutex>

#include "pa_internal.h"

namespace {

// The fixed scratch region.  Host code only ever sees the shadow of this
// symbol; the device address comes from cudaGetSymbolAddress, once per
// device.  The first 256 bytes hold the fallback status word, the rest is
// the planner / partials workspace that pa_forward would otherwise allocate.
__device__ __align__(256) unsigned char g_static_scratch[PA_STATIC_SCRATCH_BYTES];
constexpr size_t kStatusBytes = 256;

struct StaticScratch {
  bool ready = false;
  unsigned char *base = nullptr;
  int num_sms = 0;
};

std::mutex g_static_mu;
StaticScratch g_static_dev[64];

// Device address of the region on the current device (set up on first use).
// The set-up queries the runtime, which may load the module: it is refused
// while `stream` is capturing, so that it can never invalidate a capture.
pa_status static_scratch(cudaStream_t stream, StaticScratch **out) {
  int dev = 0;
  const pa_status ds = pa::current_device_for(stream, &dev);
  if (ds != PA_OK) return ds;
  std::lock_guard<std::mutex> lock(g_static_mu);
  StaticScratch &d = g_static_dev[dev];
  if (!d.ready) {
    if (pa::stream_capturing(stream)) return PA_ERR_WORKSPACE;
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return PA_ERR_CUDA;
    }
    if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return PA_ERR_CUDA;
    }
    d.base = static_cast<unsigned char *>(ptr);
    d.ready = true;
  }
  *out = &d;
  return PA_OK;
}

}  // namespace

extern "C" pa_status pa_forward_static_scratch(
    const void *q, const void *k_cache, const void *v_cache, const int32_t *block_table,
    const int32_t *seq_lens, const int32_t *query_start_loc, int num_heads, int num_kv_heads,
    int head_dim, int block_size, float scale, void *out, void *stream, pa_dtype dtype,
    int num_seqs, int num_tokens, int max_blocks_per_seq, int num_blocks, int max_seq_len,
    int kv_split_tokens, uint32_t *device_status) {
  const pa::FwdCall c{q, k_cache, v_cache, block_table, seq_lens, query_start_loc, num_heads,
                      num_kv_heads, head_dim, block_size, scale, out, dtype, num_seqs,
                      num_tokens, max_blocks_per_seq, num_blocks, max_seq_len, kv_split_tokens};
  pa_status s = pa::fwd_check(c);
  if (s != PA_OK || num_tokens == 0) return s;
  if (pa::fwd_workspace_bytes(c) > PA_STATIC_SCRATCH_BYTES - kStatusBytes)
    return PA_ERR_SCRATCH_LIMIT;
  StaticScratch *d = nullptr;
  s = static_scratch(reinterpret_cast<cudaStream_t>(stream), &d);
  if (s != PA_OK) return s;
  unsigned int *status =
      device_status ? reinterpret_cast<unsigned int *>(device_status)
                    : reinterpret_cast<unsigned int *>(d->base);
  return pa::fwd_launch(c, d->base + kStatusBytes, status, d->num_sms,
                        reinterpret_cast<cudaStream_t>(stream), false);
}
