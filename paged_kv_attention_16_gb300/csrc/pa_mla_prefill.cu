// pa_mla_prefill.cu -- non-absorbed MLA prefill / extend.
//
// "vLLM AMD ROCm attention backend optimisation", section "AITER MLA backend:
// optimised for DeepSeek": prefill and extend compute attention with a
// standard multi-head kernel on the uncompressed representation, while decode
// works directly on the 576-wide latent (pa_mla_decode).  Here the latent
// rows a batch's requests can see are decompressed once per call and then
// attended to by the tensor-core tile kernel of pa_forward:
//
//   1. mla_seg_kernel (one block): each request's rows in dense buffers
//      start at a 16-aligned offset (an exclusive scan of ceil16(seq_len));
//      a dense block table names 16-row "pages" of those buffers, so the
//      attention's page gather runs on them unchanged;
//   2. mla_rope_kernel: every position's rotary key k^R_j (the last 64
//      columns of its cached row) goes to one dense row shared by all heads
//      (a request with a bad block id is unmapped from the dense block
//      table, so its rows come out as zeros);
//   3. upproj_kernel (pa_upproj.cu, tcgen05): K[:, h, :] = C W_K,h^T and
//      V[:, h, :] = C W_V,h^T for every head, the latent rows C read through
//      the block table, bf16 in, fp32 accumulation, bf16 out;
//   4. pa_forward's planner, tile kernel (q rows of 192, keys as 128 columns
//      from K plus the 64 shared rotary columns, v and out rows of 128, every
//      row on the tile kernel) and merge, with the dense buffers as a
//      16-slot paged cache of num_heads KV heads.
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kSegThreads = 1024;
constexpr int kRopeThreads = 256;
constexpr int kL = 512, kR = 64, kNope = 128, kDv = 128, kDqk = kNope + kR;

struct MlaPrefillArgs {
  const __nv_bfloat16 *cache;  // [num_blocks, block_size, 576]
  const int32_t *block_table, *seq_lens;
  int num_seqs, num_heads, block_size, max_blocks_per_seq, num_blocks, max_seq_len;
  long long cap;        // rows of the dense buffers
  int dense_width;      // entries per request of the dense block table
  long long *total;     // rows used (written by the seg kernel)
  long long *seg;       // [num_seqs] first dense row of each request
  int32_t *dense_bt;    // [num_seqs, dense_width]
  __nv_bfloat16 *rope;  // [cap, 64]
  unsigned int *status;
};

__device__ inline long long rows_of(const MlaPrefillArgs &a, int s) {
  const int ctx = __ldg(a.seq_lens + s);
  if (ctx <= 0 || ctx > a.max_seq_len) return 0;  // the planner flags bad lengths
  return (ctx + 15) / 16 * 16;
}

__global__ void __launch_bounds__(kSegThreads) mla_seg_kernel(const MlaPrefillArgs a) {
  __shared__ long long scratch[2 * 33];
  pdl_wait();
  pdl_trigger();
  const int S = a.num_seqs, tid = threadIdx.x;
  long long carry = 0;
  for (int base = 0; base < S; base += kSegThreads) {
    const int s = base + tid;
    long long v[1] = {s < S ? rows_of(a, s) : 0};
    long long tot[1];
    block_scan_multi<1>(v, scratch, tot);  // v becomes the inclusive prefix
    if (s < S) a.seg[s] = carry + v[0] - (s < S ? rows_of(a, s) : 0);
    carry += tot[0];
    __syncthreads();
  }
  const bool overflow = carry > a.cap;
  if (tid == 0) {
    *a.total = overflow ? 0 : carry;
    if (overflow) atomicOr(a.status, PA_DEV_OVERFLOW);
  }
  // dense block table: request s's 16-row pages, -1 past its rows (and
  // everywhere on overflow, which zeroes the batch through the page checks)
  const long long n = (long long)S * a.dense_width;
  for (long long e = tid; e < n; e += kSegThreads) {
    const int s = (int)(e / a.dense_width), j = (int)(e % a.dense_width);
    const long long rows = rows_of(a, s);
    a.dense_bt[e] = (!overflow && (long long)j * 16 < rows) ? (int32_t)(a.seg[s] / 16 + j) : -1;
  }
}

// Eight dense rows per warp-iteration (four lanes a row, 16 bytes each): the
// rotary key of every position to its dense row; rows past a request's
// context are zeros.  A bad block id unmaps the whole request: its attention
// work items then find no valid page and write zeros (as pa_forward's do).
__global__ void __launch_bounds__(kRopeThreads) mla_rope_kernel(const MlaPrefillArgs a) {
  pdl_wait();
  pdl_trigger();
  const long long total = *a.total;
  const int S = a.num_seqs;
  const long long t = (long long)blockIdx.x * kRopeThreads + threadIdx.x;
  const long long nthreads = (long long)gridDim.x * kRopeThreads;
  for (long long e = t; e < total * 8; e += nthreads) {
    const long long r = e >> 3;
    const int x = (int)(e & 7);
    int lo = 0, hi = S - 1;  // the request: the last s with seg[s] <= r
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(a.seg + mid) <= r) lo = mid; else hi = mid - 1;
    }
    const int s = lo;
    const int j = (int)(r - __ldg(a.seg + s));
    const int ctx = __ldg(a.seq_lens + s);
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (j < ctx) {
      const int lp = j / a.block_size;
      const int page = lp < a.max_blocks_per_seq
                           ? __ldg(a.block_table + (size_t)s * a.max_blocks_per_seq + lp)
                           : -1;
      if (page >= 0 && page < a.num_blocks) {
        v = __ldg(reinterpret_cast<const uint4 *>(
                      a.cache + ((size_t)page * a.block_size + j % a.block_size) * (kL + kR) + kL) +
                  x);
      } else if (x == 0) {
        atomicOr(a.status, PA_DEV_BAD_BLOCK);
        for (int w = 0; w < a.dense_width; ++w) a.dense_bt[(size_t)s * a.dense_width + w] = -1;
      }
    }
    reinterpret_cast<uint4 *>(a.rope + (size_t)r * kR)[x] = v;
  }
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

struct MlaPrefillLayout {
  size_t fwd, hdr, seg, dbt, rope, k, v, total;
  long long cap;
  int dense_width;
};

FwdCall dense_call(const void *q, const int32_t *seq_lens, const int32_t *qsl, int num_heads,
                   float scale, void *out, int num_seqs, int num_tokens, int max_seq_len,
                   int kv_split_tokens, long long cap, int dense_width) {
  FwdCall c{q, nullptr, nullptr, nullptr, seq_lens, qsl, num_heads, num_heads, kDv, 16, scale,
            out, PA_BF16, num_seqs, num_tokens, dense_width, (int)(cap / 16), max_seq_len,
            kv_split_tokens};
  c.head_dim_qk = kDqk;
  c.all_tile = true;
  return c;
}

MlaPrefillLayout mla_prefill_layout(int num_seqs, int num_tokens, int num_heads, int max_seq_len,
                                    long long max_total_kv, int kv_split_tokens) {
  MlaPrefillLayout l{};
  l.cap = (max_total_kv + 15ll * num_seqs + 15) / 16 * 16;
  l.dense_width = (max_seq_len + 15) / 16;
  if (l.dense_width < 1) l.dense_width = 1;
  const FwdCall fc = dense_call(nullptr, nullptr, nullptr, num_heads, 1.f, nullptr, num_seqs,
                                num_tokens, max_seq_len, kv_split_tokens, l.cap, l.dense_width);
  size_t off = 0;
  l.fwd = off;
  off = align256(off + fwd_workspace_bytes(fc));
  l.hdr = off;
  off = align256(off + 256);
  l.seg = off;
  off = align256(off + (size_t)num_seqs * sizeof(long long));
  l.dbt = off;
  off = align256(off + (size_t)num_seqs * l.dense_width * sizeof(int32_t));
  l.rope = off;
  off = align256(off + (size_t)l.cap * kR * 2);
  l.k = off;
  off = align256(off + (size_t)l.cap * num_heads * kNope * 2);
  l.v = off;
  off = align256(off + (size_t)l.cap * num_heads * kDv * 2);
  l.total = off;
  return l;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" size_t pa_mla_prefill_workspace_bytes(int num_seqs, int num_tokens, int num_heads,
                                                 int max_seq_len, long long max_total_kv,
                                                 int kv_split_tokens) {
  if (num_seqs < 0 || num_tokens < 0 || num_heads <= 0 || max_seq_len < 0 || max_total_kv < 0 ||
      kv_split_tokens < 0)
    return 0;
  return mla_prefill_layout(num_seqs, num_tokens, num_heads, max_seq_len, max_total_kv,
                            kv_split_tokens)
      .total;
}

extern "C" pa_status pa_mla_prefill(const void *q, const void *kv_cache, const void *w_kv,
                                    const int32_t *block_table, const int32_t *seq_lens,
                                    const int32_t *query_start_loc, int num_heads,
                                    int kv_lora_rank, int qk_nope_dim, int rope_dim,
                                    int v_head_dim, int block_size, float scale, void *out,
                                    void *stream, int num_seqs, int num_tokens,
                                    int max_blocks_per_seq, int num_blocks, int max_seq_len,
                                    long long max_total_kv, int kv_split_tokens) {
  if (num_seqs < 0 || num_tokens < 0 || num_heads <= 0 || block_size <= 0 ||
      max_blocks_per_seq < 0 || num_blocks < 0 || max_seq_len < 0 || max_total_kv < 0 ||
      kv_split_tokens < 0)
    return PA_ERR_INVALID_ARG;
  if (kv_lora_rank != kL || rope_dim != kR || qk_nope_dim != kNope || v_head_dim != kDv ||
      kv_split_tokens % 16 != 0 || block_size % 16 != 0 || block_size > 256)
    return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  if (num_seqs == 0 || !q || !kv_cache || !w_kv || !block_table || !seq_lens ||
      !query_start_loc || !out || num_blocks == 0 || max_blocks_per_seq == 0)
    return PA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv_cache) || !aligned16(w_kv) || !aligned16(out))
    return PA_ERR_INVALID_ARG;
  const MlaPrefillLayout lay = mla_prefill_layout(num_seqs, num_tokens, num_heads, max_seq_len,
                                                  max_total_kv, kv_split_tokens);
  if (lay.cap > (long long)INT32_MAX || (long long)lay.cap * num_heads * kDqk > (1ll << 40) ||
      (long long)num_heads * 256 > (1ll << 31))
    return PA_ERR_UNSUPPORTED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  void *ws_v = nullptr;
  unsigned int *status = nullptr;
  int num_sms = 0;
  pa_status s = device_resources(st, lay.total, &ws_v, &status, &num_sms);
  if (s != PA_OK) return s;
  uint8_t *ws = static_cast<uint8_t *>(ws_v);

  MlaPrefillArgs a{};
  a.cache = static_cast<const __nv_bfloat16 *>(kv_cache);
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.num_seqs = num_seqs;
  a.num_heads = num_heads;
  a.block_size = block_size;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_blocks = num_blocks;
  a.max_seq_len = max_seq_len;
  a.cap = lay.cap;
  a.dense_width = lay.dense_width;
  a.total = reinterpret_cast<long long *>(ws + lay.hdr);
  a.seg = reinterpret_cast<long long *>(ws + lay.seg);
  a.dense_bt = reinterpret_cast<int32_t *>(ws + lay.dbt);
  a.rope = reinterpret_cast<__nv_bfloat16 *>(ws + lay.rope);
  a.status = status;
  __nv_bfloat16 *k = reinterpret_cast<__nv_bfloat16 *>(ws + lay.k);
  __nv_bfloat16 *v = reinterpret_cast<__nv_bfloat16 *>(ws + lay.v);

  if (launch_dependent(mla_seg_kernel, dim3(1), dim3(kSegThreads), 0, st, a) != cudaSuccess)
    return PA_ERR_CUDA;
  int slot = prof_begin(PA_K_MLA_ROPE, st);
  long long gblocks = (lay.cap * 8 + kRopeThreads - 1) / kRopeThreads;
  if (gblocks > (long long)num_sms * 8) gblocks = (long long)num_sms * 8;
  if (gblocks < 1) gblocks = 1;
  cudaError_t err = launch_dependent(mla_rope_kernel, dim3((unsigned)gblocks), dim3(kRopeThreads),
                                     0, st, a);
  prof_end(slot, st);
  if (err != cudaSuccess) return PA_ERR_CUDA;

  UpprojArgs u{};
  u.block_table = block_table;
  u.num_seqs = num_seqs;
  u.num_heads = num_heads;
  u.block_size = block_size;
  u.max_blocks_per_seq = max_blocks_per_seq;
  u.num_blocks = num_blocks;
  u.total = a.total;
  u.seg = a.seg;
  u.k_nope = k;
  u.v = v;
  u.status = status;
  slot = prof_begin(PA_K_UPPROJ, st);
  err = launch_upproj(u, kv_cache, w_kv, num_sms, st);
  prof_end(slot, st);
  if (err != cudaSuccess) return PA_ERR_CUDA;

  FwdCall c = dense_call(q, seq_lens, query_start_loc, num_heads, scale, out, num_seqs,
                         num_tokens, max_seq_len, kv_split_tokens, lay.cap, lay.dense_width);
  c.k_cache = k;
  c.k_rope = a.rope;
  c.v_cache = v;
  c.block_table = a.dense_bt;
  s = fwd_check(c);
  if (s != PA_OK) return s;
  return fwd_launch(c, ws + lay.fwd, status, num_sms, st, true);
}
