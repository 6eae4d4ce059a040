// pa_internal.h -- host-side interface between the translation units of
// libpa.so (not part of the public C ABI).
#pragma once

#include "pa_common.cuh"

namespace pa {

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

// Tensor-core (tcgen05) tile kernel for bf16 extend/prefill rows.
bool tile_kernel_supported(int dtype, int head_dim, int group);
cudaError_t launch_tile_kernel(const FwdParams &p, const CUtensorMap &tm_q,
                               const CUtensorMap &tm_k, const CUtensorMap &tm_v, int grid,
                               cudaStream_t stream);

// Absorbed-MLA decode.
struct MlaParams {
  const void *q;
  void *out;
  const int32_t *block_table;
  const int32_t *seq_lens;
  int num_seqs, num_heads, kv_lora_rank, rope_dim, block_size;
  int max_blocks_per_seq, num_blocks, max_seq_len, kv_split_tokens;
  float scale_log2;
  int split_len;          // KV positions per split
  int max_splits;         // splits per sequence the workspace holds
  unsigned int *counter;  // work counter (reset by a memset node)
  float *part_o;          // [num_seqs * num_heads * max_splits][kv_lora_rank]
  float *part_lse;        // [num_seqs * num_heads * max_splits]
  unsigned int *status;
};
cudaError_t launch_mla_decode(const MlaParams &p, const CUtensorMap &tm_q,
                              const CUtensorMap &tm_kv, int num_sms, cudaStream_t stream);

}  // namespace pa
