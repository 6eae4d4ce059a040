// pa_cache.cu -- the paged KV-cache write: a step's new K and V rows go to
// their page slots ("vLLM Triton attention backend deep dive", section
// "Technical implementation of paged attention": the cache is a pool of
// fixed-size blocks and a sequence's block table maps its logical block j to
// a physical block).  New token i of request s sits at position
// pos = seq_lens[s] - q_len_s + i, in physical block block_table[s][pos / bs]
// at slot pos % bs.  This is the step that runs before pa_forward, whose
// seq_lens already count the new tokens.
//
// Two launches on the caller's stream:
//  * a one-block check of query_start_loc (starts at 0, non-decreasing, ends
//    at num_tokens), which leaves a flag in the library workspace: a bad
//    query_start_loc writes nothing;
//  * the copy, launched programmatically after the check: min(32, row bytes /
//    16) lanes per (new token, KV head) row, several rows per warp when
//    they are short; the token's request by binary search over
//    query_start_loc, its slot through the block table, then the K and the V
//    row copied with 16-byte vector accesses.  HBM-bound: it reads and writes
//    2 x num_tokens x num_kv_heads x head_dim elements.
// The cache layout (NHD or HND) only changes where a (page, slot, head) row
// lands.
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kCheckThreads = 1024;
constexpr int kCopyThreads = 256;

struct CacheWriteArgs {
  const uint8_t *k_new, *v_new;
  uint8_t *k_cache, *v_cache;
  const int32_t *block_table, *seq_lens, *qsl;
  int num_seqs, num_tokens, num_kv_heads, row_bytes, block_size, max_blocks_per_seq, num_blocks;
  int hnd;      // 1: caches are [num_blocks, num_kv_heads, block_size, head_dim]
  int *qsl_ok;  // workspace flag written by the check
  unsigned int *status;
};

__global__ void __launch_bounds__(kCheckThreads) cache_check_kernel(const CacheWriteArgs a) {
  pdl_wait();  // whatever preceded this call in the stream (it may have written the metadata)
  pdl_trigger();
  const int S = a.num_seqs;
  int bad = 0;
  if (threadIdx.x == 0 && (a.qsl[0] != 0 || a.qsl[S] != a.num_tokens)) bad = 1;
  for (int s = threadIdx.x; s < S; s += kCheckThreads)
    if (a.qsl[s + 1] < a.qsl[s]) bad = 1;
  bad = __syncthreads_or(bad);
  if (threadIdx.x == 0) {
    *a.qsl_ok = bad ? 0 : 1;
    if (bad) atomicOr(a.status, PA_DEV_BAD_QSL);
  }
}

__global__ void __launch_bounds__(kCopyThreads) cache_copy_kernel(const CacheWriteArgs a) {
  pdl_wait();  // the check
  if (!*a.qsl_ok) return;
  // A row takes min(32, row_bytes / 16) lanes; a warp moves 32 / that rows
  // at once (two 256-byte bf16 rows, four 128-byte ones).
  const int lpr = min(32, a.row_bytes / 16);
  const int rpw = 32 / lpr;
  const int lane = (threadIdx.x & 31) % lpr, sub = (threadIdx.x & 31) / lpr;
  if (sub >= rpw) return;  // lanes left over when lpr does not divide 32
  const long long gw = ((long long)blockIdx.x * kCopyThreads + threadIdx.x) >> 5;
  const long long nw = ((long long)gridDim.x * kCopyThreads) >> 5;
  const long long nrows = (long long)a.num_tokens * a.num_kv_heads;
  const int S = a.num_seqs, bs = a.block_size;
  for (long long row = gw * rpw + sub; row < nrows; row += nw * rpw) {
    const int t = (int)(row / a.num_kv_heads), h = (int)(row % a.num_kv_heads);
    // the request: the last s with qsl[s] <= t (qsl checked non-decreasing)
    int lo = 0, hi = S - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(a.qsl + mid) <= t) lo = mid; else hi = mid - 1;
    }
    const int s = lo;
    const int q0 = __ldg(a.qsl + s), q_len = __ldg(a.qsl + s + 1) - q0;
    const int prefix = __ldg(a.seq_lens + s) - q_len;
    if (prefix < 0) {  // q_len > seq_len: the request is skipped
      if (lane == 0) atomicOr(a.status, PA_DEV_BAD_QLEN);
      continue;
    }
    const int pos = prefix + (t - q0);
    const int lp = pos / bs;
    const int page = lp < a.max_blocks_per_seq
                         ? __ldg(a.block_table + (size_t)s * a.max_blocks_per_seq + lp)
                         : -1;
    if (page < 0 || page >= a.num_blocks) {  // no valid slot: the row is skipped
      if (lane == 0) atomicOr(a.status, PA_DEV_BAD_BLOCK);
      continue;
    }
    const size_t src = ((size_t)t * a.num_kv_heads + h) * a.row_bytes;
    const size_t dst =
        (a.hnd ? ((size_t)page * a.num_kv_heads + h) * bs + pos % bs
               : ((size_t)page * bs + pos % bs) * a.num_kv_heads + h) *
        a.row_bytes;
    for (int c = lane * 16; c < a.row_bytes; c += lpr * 16) {
      const uint4 kv = *reinterpret_cast<const uint4 *>(a.k_new + src + c);
      const uint4 vv = *reinterpret_cast<const uint4 *>(a.v_new + src + c);
      *reinterpret_cast<uint4 *>(a.k_cache + dst + c) = kv;
      *reinterpret_cast<uint4 *>(a.v_cache + dst + c) = vv;
    }
  }
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" pa_status pa_cache_write(const void *k_new, const void *v_new, void *k_cache,
                                    void *v_cache, const int32_t *block_table,
                                    const int32_t *seq_lens, const int32_t *query_start_loc,
                                    int num_kv_heads, int head_dim, int block_size, void *stream,
                                    pa_dtype dtype, int num_seqs, int num_tokens,
                                    int max_blocks_per_seq, int num_blocks,
                                    pa_kv_layout kv_layout) {
  if (num_seqs < 0 || num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
      max_blocks_per_seq < 0 || num_blocks < 0 || (dtype != PA_F32 && dtype != PA_BF16) ||
      (kv_layout != PA_KV_NHD && kv_layout != PA_KV_HND))
    return PA_ERR_INVALID_ARG;
  const int es = dtype == PA_F32 ? 4 : 2;
  if ((head_dim * es) % 16 != 0) return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  if (num_seqs == 0 || !k_new || !v_new || !k_cache || !v_cache || !block_table || !seq_lens ||
      !query_start_loc || num_blocks == 0 || max_blocks_per_seq == 0)
    return PA_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  void *ws = nullptr;
  unsigned int *status = nullptr;
  int num_sms = 0;
  pa_status s = device_resources(st, 256, &ws, &status, &num_sms);
  if (s != PA_OK) return s;
  CacheWriteArgs a{};
  a.k_new = static_cast<const uint8_t *>(k_new);
  a.v_new = static_cast<const uint8_t *>(v_new);
  a.k_cache = static_cast<uint8_t *>(k_cache);
  a.v_cache = static_cast<uint8_t *>(v_cache);
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.qsl = query_start_loc;
  a.num_seqs = num_seqs;
  a.num_tokens = num_tokens;
  a.num_kv_heads = num_kv_heads;
  a.row_bytes = head_dim * es;
  a.block_size = block_size;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_blocks = num_blocks;
  a.hnd = kv_layout == PA_KV_HND;
  a.qsl_ok = static_cast<int *>(ws);
  a.status = status;
  if (launch_dependent(cache_check_kernel, dim3(1), dim3(kCheckThreads), 0, st, a) != cudaSuccess)
    return PA_ERR_CUDA;
  // enough warps for every row (many copies in flight), at most 32 blocks per SM
  const int lpr = (head_dim * es / 16) < 32 ? head_dim * es / 16 : 32;
  const long long rows = (long long)num_tokens * num_kv_heads;
  const long long warps = (rows + (32 / lpr) - 1) / (32 / lpr);
  long long blocks = (warps + kCopyThreads / 32 - 1) / (kCopyThreads / 32);
  if (blocks > (long long)num_sms * 32) blocks = (long long)num_sms * 32;
  if (launch_dependent(cache_copy_kernel, dim3((unsigned)blocks), dim3(kCopyThreads), 0, st, a) !=
      cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}
