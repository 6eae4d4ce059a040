// pa_internal.h -- host-side interface between the translation units of
// libpa.so (not part of the public C ABI).
#pragma once

#include <atomic>

#include "pa_common.cuh"

namespace pa {

// A kernel's launch attributes (dynamic shared memory size, carveout) are
// per device: set them on the kernel's first launch on each device only
// (each cudaFuncSetAttribute costs host time on every call otherwise).
template <typename Kernel>
cudaError_t set_smem_attrs_once(Kernel kernel, int smem, std::atomic<unsigned long long> &done) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// Launches `kernel` with programmatic stream serialization: its CTAs may be
// scheduled while the previous kernel of the stream drains.  The kernel must
// call pdl_wait() before it reads anything earlier kernels wrote.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// Kernel timing: prof_begin records a start event when timing is on and the
// stream is not capturing (returns -1 otherwise); prof_end records the end.
int prof_begin(int kernel_id, cudaStream_t stream);
void prof_end(int slot, cudaStream_t stream);

// Row-streaming kernel: decode rows (and, where no tensor-core kernel
// applies, extend/prefill rows), one query token x one GQA group per item.
bool row_kernel_supported(int dtype, int head_dim, int group);
// Resident CTAs per SM of the instantiation (0 if unsupported).
int row_kernel_ctas_per_sm(int dtype, int head_dim, int group);
cudaError_t launch_row_kernel(const FwdParams &p, const CUtensorMap &tm_k,
                              const CUtensorMap &tm_v, int grid, cudaStream_t stream);

// bf16 decode rows on warp-level MMAs (mma.sync m16n8k16); K/V maps are the
// 128-byte-swizzled 64-element boxes the tile kernel also uses.
bool row_mma_supported(int dtype, int head_dim, int group);
int row_mma_ctas_per_sm(int head_dim, int group);
cudaError_t launch_row_mma_kernel(const FwdParams &p, const CUtensorMap &tm_k,
                                  const CUtensorMap &tm_v, int grid, cudaStream_t stream);

// Tensor-core (tcgen05) tile kernel for bf16 extend/prefill rows.
bool tile_kernel_supported(int dtype, int head_dim, int group);
// tm_kr: the shared rotary-key columns when p.k_rope_split (else unused).
cudaError_t launch_tile_kernel(const FwdParams &p, const CUtensorMap &tm_q,
                               const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                               const CUtensorMap &tm_kr, int grid, cudaStream_t stream);

// Up-projection of the non-absorbed MLA prefill (tensor cores): the latent
// rows of every dense row (request s's positions from seg[s] on, 16-aligned
// runs) are read through the block table and multiplied by each head's
// w_kv rows into key and value rows.
struct UpprojArgs {
  const int32_t *block_table;
  int num_seqs, num_heads, block_size, max_blocks_per_seq, num_blocks;
  const long long *total;  // dense rows in use (device)
  const long long *seg;    // [num_seqs] first dense row of each request
  __nv_bfloat16 *k_nope;   // [rows, num_heads, 128]
  __nv_bfloat16 *v;        // [rows, num_heads, 128]
  unsigned int *status;
};
cudaError_t launch_upproj(const UpprojArgs &a, const void *kv_cache, const void *w_kv,
                          int num_sms, cudaStream_t stream);

// One pa_forward call's host-side arguments.
struct FwdCall {
  const void *q, *k_cache, *v_cache;
  const int32_t *block_table, *seq_lens, *qsl;
  int num_heads, num_kv_heads, head_dim, block_size;
  float scale;
  void *out;
  pa_dtype dtype;
  int num_seqs, num_tokens, max_blocks_per_seq, num_blocks, max_seq_len, kv_split_tokens;
  const float *sinks = nullptr;  // [num_heads] device array of sink logits, or null
  int kv_layout = PA_KV_NHD;     // pa_kv_layout of k_cache / v_cache
  int sliding_window = 0;        // 0: none
  const float *alibi_slopes = nullptr;  // [num_heads] device array, or null
  int alibi_sqrt = 0;
  // Non-absorbed MLA prefill: q and k rows of head_dim_qk (0: head_dim)
  // elements, v and out rows of head_dim, every row on the tile kernel.
  int head_dim_qk = 0;
  bool all_tile = false;
  // Keys split in two tensors: k_cache holds the first head_dim_qk - 64
  // columns of every (position, head) key row, k_rope the last 64 columns,
  // shared by all heads: [num_blocks, block_size, 64].  Null: keys whole.
  const void *k_rope = nullptr;
  int max_query_len = 0;  // caller's bound on new tokens per request (0: unknown)
};
// Host-side argument checks of pa_forward (PA_OK also when num_tokens == 0).
pa_status fwd_check(const FwdCall &c);
// Workspace bytes the call needs.
size_t fwd_workspace_bytes(const FwdCall &c);
// The launch sequence (planner, row kernel, tile kernel, merge) on a given
// workspace and device status word; records kernel timing when `timed`.
pa_status fwd_launch(const FwdCall &c, void *workspace, unsigned int *status, int num_sms,
                     cudaStream_t stream, bool timed);

// True while `stream` is capturing a CUDA graph.
bool stream_capturing(cudaStream_t stream);
// The calling thread's current device in *dev; PA_ERR_INVALID_ARG when
// `stream` belongs to another device (kernels would get this device's
// workspace addresses), PA_ERR_CUDA when the device cannot be queried.  A
// capturing stream is not checked.
pa_status current_device_for(cudaStream_t stream, int *dev);

// Library-owned per-device resources for an entry point: workspace of at
// least ws_bytes (grown outside capture), the device status word, SM count.
pa_status device_resources(cudaStream_t stream, size_t ws_bytes, void **ws,
                           unsigned int **status, int *num_sms);

// cuTensorMapEncodeTiled over a bf16/fp32 tensor of `rank` dims (innermost
// first), strides in bytes for dims 1..rank-1, optional 128-byte swizzle.
bool encode_tiled(CUtensorMap *map, const void *base, int dtype, int rank,
                  const unsigned long long *dims, const unsigned long long *strides,
                  const unsigned int *box, bool swizzle128);

}  // namespace pa
