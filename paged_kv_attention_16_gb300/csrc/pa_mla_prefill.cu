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
//   2. mla_gather_kernel: every position's latent c_j (512) goes to a dense
//      matrix C, and its rotary key k^R_j (64) to columns 128..191 of every
//      head's key row (a request with a bad block id is unmapped from the
//      dense block table, so its rows come out as zeros);
//   3. two library GEMMs (the up-projection, a plain dense contraction):
//      K[:, h, 0:128] = C W_K,h^T and V[:, h, :] = C W_V,h^T, bf16 in, fp32
//      accumulation, bf16 out;
//   4. pa_forward's planner, tile kernel (q and k rows of 192, v and out rows
//      of 128, every row on the tile kernel) and merge, with the dense
//      buffers as a 16-slot paged cache of num_heads KV heads.
//
// The GEMMs come from cuBLAS, loaded at run time (dlopen): a missing cuBLAS
// makes pa_mla_prefill return PA_ERR_UNSUPPORTED and leaves every other entry
// point working.
#include <cublas_v2.h>
#include <dlfcn.h>

#include <mutex>

#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kSegThreads = 1024;
constexpr int kGatherThreads = 128;
constexpr int kL = 512, kR = 64, kNope = 128, kDv = 128, kDqk = kNope + kR;
constexpr size_t kCublasWs = 32u << 20;

struct MlaPrefillArgs {
  const __nv_bfloat16 *cache;  // [num_blocks, block_size, 576]
  const int32_t *block_table, *seq_lens;
  int num_seqs, num_heads, block_size, max_blocks_per_seq, num_blocks, max_seq_len;
  long long cap;        // rows of the dense buffers
  int dense_width;      // entries per request of the dense block table
  long long *total;     // rows used (written by the seg kernel)
  long long *seg;       // [num_seqs] first dense row of each request
  int32_t *dense_bt;    // [num_seqs, dense_width]
  __nv_bfloat16 *c;     // [cap, 512]
  __nv_bfloat16 *k;     // [cap, num_heads, 192]
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

// One block per dense row at a time: the latent to C, the rotary key to every
// head's key row; rows past a request's context are zeros.
__global__ void __launch_bounds__(kGatherThreads) mla_gather_kernel(const MlaPrefillArgs a) {
  pdl_wait();
  const long long total = *a.total;
  const int S = a.num_seqs, H = a.num_heads, tid = threadIdx.x;
  for (long long r = blockIdx.x; r < total; r += gridDim.x) {
    // the request: the last s with seg[s] <= r
    int lo = 0, hi = S - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(a.seg + mid) <= r) lo = mid; else hi = mid - 1;
    }
    const int s = lo;
    const int j = (int)(r - __ldg(a.seg + s));
    const int ctx = __ldg(a.seq_lens + s);
    const uint4 *src = nullptr;
    if (j < ctx) {
      const int lp = j / a.block_size;
      const int page = lp < a.max_blocks_per_seq
                           ? __ldg(a.block_table + (size_t)s * a.max_blocks_per_seq + lp)
                           : -1;
      if (page >= 0 && page < a.num_blocks) {
        src = reinterpret_cast<const uint4 *>(
            a.cache + ((size_t)page * a.block_size + j % a.block_size) * (kL + kR));
      } else {
        // a bad block id: unmap the whole request, whose attention work items
        // then find no valid page and write zeros (as pa_forward's do)
        if (tid == 0) atomicOr(a.status, PA_DEV_BAD_BLOCK);
        for (int e = tid; e < a.dense_width; e += kGatherThreads)
          a.dense_bt[(size_t)s * a.dense_width + e] = -1;
      }
    }
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    // C row: 512 bf16 = 64 vectors
    if (tid < kL / 8)
      reinterpret_cast<uint4 *>(a.c + (size_t)r * kL)[tid] = src ? __ldg(src + tid) : zero;
    // rope: 64 bf16 = 8 vectors, to columns 128..191 of each head
    const int nv = H * (kR / 8);
    for (int e = tid; e < nv; e += kGatherThreads) {
      const int h = e / (kR / 8), x = e % (kR / 8);
      reinterpret_cast<uint4 *>(a.k + ((size_t)r * H + h) * kDqk + kNope)[x] =
          src ? __ldg(src + kL / 8 + x) : zero;
    }
  }
}

// cuBLAS, resolved at run time (the strided-batched GEMM's C entry point).
typedef cublasStatus_t (*GemmStridedBatchedFn)(cublasHandle_t, cublasOperation_t,
                                               cublasOperation_t, int, int, int, const void *,
                                               const void *, cudaDataType, int, long long,
                                               const void *, cudaDataType, int, long long,
                                               const void *, void *, cudaDataType, int,
                                               long long, int, cublasComputeType_t,
                                               cublasGemmAlgo_t);
struct Cublas {
  decltype(&cublasCreate_v2) create = nullptr;
  decltype(&cublasSetStream_v2) set_stream = nullptr;
  decltype(&cublasSetWorkspace_v2) set_workspace = nullptr;
  GemmStridedBatchedFn gemm_sb = nullptr;
  bool ok = false;
};

const Cublas &cublas() {
  static Cublas cb;
  static std::once_flag once;
  std::call_once(once, [] {
    void *h = dlopen("libcublas.so.13", RTLD_NOW | RTLD_GLOBAL);
    if (!h) h = dlopen("/usr/local/cuda/lib64/libcublas.so.13", RTLD_NOW | RTLD_GLOBAL);
    if (!h) return;
    cb.create = reinterpret_cast<decltype(cb.create)>(dlsym(h, "cublasCreate_v2"));
    cb.set_stream = reinterpret_cast<decltype(cb.set_stream)>(dlsym(h, "cublasSetStream_v2"));
    cb.set_workspace =
        reinterpret_cast<decltype(cb.set_workspace)>(dlsym(h, "cublasSetWorkspace_v2"));
    cb.gemm_sb = reinterpret_cast<decltype(cb.gemm_sb)>(dlsym(h, "cublasGemmStridedBatchedEx"));
    cb.ok = cb.create && cb.set_stream && cb.set_workspace && cb.gemm_sb;
  });
  return cb;
}

// One handle per device, created on first use.
cublasHandle_t cublas_handle() {
  static std::mutex mu;
  static cublasHandle_t handles[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!handles[dev] && cublas().create(&handles[dev]) != CUBLAS_STATUS_SUCCESS)
    handles[dev] = nullptr;
  return handles[dev];
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

struct MlaPrefillLayout {
  size_t fwd, hdr, seg, dbt, c, k, v, cublas_ws, total;
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
  l.c = off;
  off = align256(off + (size_t)l.cap * kL * 2);
  l.k = off;
  off = align256(off + (size_t)l.cap * num_heads * kDqk * 2);
  l.v = off;
  off = align256(off + (size_t)l.cap * num_heads * kDv * 2);
  l.cublas_ws = off;
  off = align256(off + kCublasWs);
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
      kv_split_tokens % 16 != 0)
    return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  if (num_seqs == 0 || !q || !kv_cache || !w_kv || !block_table || !seq_lens ||
      !query_start_loc || !out || num_blocks == 0 || max_blocks_per_seq == 0)
    return PA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv_cache) || !aligned16(w_kv) || !aligned16(out))
    return PA_ERR_INVALID_ARG;
  const Cublas &cb = cublas();
  if (!cb.ok) return PA_ERR_UNSUPPORTED;
  const MlaPrefillLayout lay = mla_prefill_layout(num_seqs, num_tokens, num_heads, max_seq_len,
                                                  max_total_kv, kv_split_tokens);
  if (lay.cap > (long long)INT32_MAX || (long long)lay.cap * num_heads * kDqk > (1ll << 40))
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
  a.c = reinterpret_cast<__nv_bfloat16 *>(ws + lay.c);
  a.k = reinterpret_cast<__nv_bfloat16 *>(ws + lay.k);
  a.status = status;
  __nv_bfloat16 *v = reinterpret_cast<__nv_bfloat16 *>(ws + lay.v);

  if (launch_dependent(mla_seg_kernel, dim3(1), dim3(kSegThreads), 0, st, a) != cudaSuccess)
    return PA_ERR_CUDA;
  long long gblocks = lay.cap < (long long)num_sms * 16 ? lay.cap : (long long)num_sms * 16;
  if (gblocks < 1) gblocks = 1;
  if (launch_dependent(mla_gather_kernel, dim3((unsigned)gblocks), dim3(kGatherThreads), 0, st,
                       a) != cudaSuccess)
    return PA_ERR_CUDA;

  // Up-projection, per head h (column-major view): K_h^T [128 x rows] =
  // W_K,h [128 x 512] . C^T [512 x rows]; W_K,h is rows h*256 .. h*256+127 of
  // w_kv (row-major [H*256, 512]), W_V,h the next 128 rows.  C is shared by
  // every head (stride 0); outputs land in each head's key / value row.
  cublasHandle_t handle = cublas_handle();
  if (!handle) return PA_ERR_CUDA;
  if (cb.set_stream(handle, st) != CUBLAS_STATUS_SUCCESS ||
      cb.set_workspace(handle, ws + lay.cublas_ws, kCublasWs) != CUBLAS_STATUS_SUCCESS)
    return PA_ERR_CUDA;
  const float one = 1.f, zero = 0.f;
  const int rows = (int)lay.cap;
  const __nv_bfloat16 *w = static_cast<const __nv_bfloat16 *>(w_kv);
  if (cb.gemm_sb(handle, CUBLAS_OP_T, CUBLAS_OP_N, kNope, rows, kL, &one, w, CUDA_R_16BF, kL,
                 (long long)(kNope + kDv) * kL, a.c, CUDA_R_16BF, kL, 0, &zero, a.k, CUDA_R_16BF,
                 num_heads * kDqk, kDqk, num_heads, CUBLAS_COMPUTE_32F,
                 CUBLAS_GEMM_DEFAULT) != CUBLAS_STATUS_SUCCESS)
    return PA_ERR_CUDA;
  if (cb.gemm_sb(handle, CUBLAS_OP_T, CUBLAS_OP_N, kDv, rows, kL, &one, w + (size_t)kNope * kL,
                 CUDA_R_16BF, kL, (long long)(kNope + kDv) * kL, a.c, CUDA_R_16BF, kL, 0, &zero,
                 v, CUDA_R_16BF, num_heads * kDv, kDv, num_heads, CUBLAS_COMPUTE_32F,
                 CUBLAS_GEMM_DEFAULT) != CUBLAS_STATUS_SUCCESS)
    return PA_ERR_CUDA;

  FwdCall c = dense_call(q, seq_lens, query_start_loc, num_heads, scale, out, num_seqs,
                         num_tokens, max_seq_len, kv_split_tokens, lay.cap, lay.dense_width);
  c.k_cache = a.k;
  c.v_cache = v;
  c.block_table = a.dense_bt;
  s = fwd_check(c);
  if (s != PA_OK) return s;
  return fwd_launch(c, ws + lay.fwd, status, num_sms, st, true);
}
