/*
 * pa.h -- C ABI of libpa.so: unified paged attention over a continuous batch
 * on one GB300 (sm_103a), plus the absorbed-MLA decode variant.
 *
 * What is computed ("vLLM Triton attention backend deep dive", section
 * "Technical implementation of paged attention"; "vLLM AMD ROCm attention
 * backend optimisation", section "Mixed inference workload challenge"):
 * every query token of every request in one batch -- decode (1 new token),
 * extend (new tokens on a partly built cache) or prefill (no cached prefix)
 * -- attends, per query head, to the K/V rows of its own sequence, which live
 * in fixed-size pages of a shared cache reached through a per-sequence block
 * table:
 *
 *   for request s, query i (0 <= i < q_len_s) at token row r = qsl[s] + i,
 *   head h, kv head k = h / (num_heads / num_kv_heads):
 *     prefix = seq_lens[s] - q_len_s;   visible j = 0 .. prefix + i
 *     K_j = k_cache[block_table[s][j / block_size]][j % block_size][k][:]
 *     out[r][h][:] = sum_j softmax_j(scale * <q[r][h], K_j>) * V_j
 *
 * Conventions shared by every entry point:
 *  - All tensor pointers are device pointers owned by the caller, row-major,
 *    contiguous, 16-byte aligned.  The library keeps no pointer after return.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Calls are asynchronous on it: they never synchronise and never read
 *    device memory on the host, so pa_forward / pa_mla_decode can be captured
 *    in a CUDA graph (reserve the workspace first, see pa_reserve).
 *  - Host-side argument errors return a status and launch nothing.  A stream
 *    that belongs to a device other than the calling thread's current device
 *    is such an error (PA_ERR_INVALID_ARG): the library's per-device state is
 *    that of the current device.  (A stream that is capturing a graph is not
 *    queried for its device: the query would invalidate the capture.)
 *  - Bad *device* metadata never traps: it sets a bit in the device status word
 *    (read with pa_get_device_status) and the affected output rows are written
 *    as zeros:
 *      PA_DEV_BAD_BLOCK   a block id outside [0, num_blocks) on a visible page;
 *                         the rows whose visible range covers that page are 0
 *      PA_DEV_BAD_QLEN    q_len < 0 or q_len > seq_len; the request's rows are 0
 *      PA_DEV_BAD_SEQLEN  seq_len > max_seq_len (or < 0); the request's rows are 0
 *      PA_DEV_BAD_QSL     query_start_loc[0] != 0, decreasing, or
 *                         query_start_loc[num_seqs] != num_tokens; every row is 0
 *      PA_DEV_OVERFLOW    the plan needs more split partials than the workspace
 *                         holds (only if seq_lens exceed max_seq_len); every row is 0
 *      PA_DEV_TIMEOUT     a bounded wait inside a kernel gave up (never expected)
 *      PA_DEV_INTERNAL    a kernel found its launch set-up unusable (its shared
 *                         memory window not 1024-byte aligned) and wrote
 *                         nothing (never expected)
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { PA_F32 = 0, PA_BF16 = 1 } pa_dtype;

/*
 * Memory layout of a paged K or V cache.  "vLLM AMD ROCm attention backend
 * optimisation", section "ROCM_AITER_FA" ("Hardware-Optimized KV Cache
 * Layout"), reports that a cache laid out for the hardware's access pattern
 * speeds decode up; PA_KV_HND is this library's counterpart: one (page, KV
 * head) pair is one contiguous run of block_size x head_dim elements, which
 * one bulk copy moves.
 *   PA_KV_NHD  [num_blocks, block_size, num_kv_heads, head_dim]  (default)
 *   PA_KV_HND  [num_blocks, num_kv_heads, block_size, head_dim]
 */
typedef enum { PA_KV_NHD = 0, PA_KV_HND = 1 } pa_kv_layout;

typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad alignment ...   */
  PA_ERR_UNSUPPORTED = 2, /* a shape or dtype this build has no kernel for     */
  PA_ERR_WORKSPACE = 3,   /* workspace too small while the stream is capturing */
  PA_ERR_CUDA = 4,        /* a CUDA runtime / driver call failed               */
  PA_ERR_SCRATCH_LIMIT = 5 /* the call needs more than the static scratch region */
} pa_status;

/* Device status bits (see above). */
#define PA_DEV_BAD_BLOCK 0x1u
#define PA_DEV_BAD_QLEN 0x2u
#define PA_DEV_BAD_SEQLEN 0x4u
#define PA_DEV_BAD_QSL 0x8u
#define PA_DEV_OVERFLOW 0x10u
#define PA_DEV_TIMEOUT 0x20u
#define PA_DEV_INTERNAL 0x40u

/*
 * pa_forward -- unified paged attention over a mixed batch.
 *
 * Follows "vLLM Triton attention backend deep dive" (sections "Technical
 * implementation of paged attention", "Q-block optimisation", "Parallel tiled
 * softmax (3D kernel)", "Persistent kernels and CUDA graphs") and "vLLM AMD
 * ROCm attention backend optimisation" (sections "Mixed inference workload
 * challenge", "Three-path routing", "Batch reordering", "Chunked context
 * processing").  Internally: a one-block planner classifies the requests,
 * orders the work [decode : extend : prefill] and sizes the KV splits; fixed-
 * grid persistent kernels (grid = a multiple of the SM count) pull work items
 * from device counters; split results are combined by a log-sum-exp merge.
 *
 *  q               [num_tokens, num_heads, head_dim]                 dtype
 *  k_cache,v_cache [num_blocks, block_size, num_kv_heads, head_dim]  dtype
 *                  (pa_forward_ex also takes the PA_KV_HND layout)
 *  block_table     [num_seqs, max_blocks_per_seq] int32; entries past
 *                  ceil(seq_len / block_size) are never read (may hold -1)
 *  seq_lens        [num_seqs] int32: context length INCLUDING this step's
 *                  new tokens, whose K/V must already be in the cache
 *  query_start_loc [num_seqs + 1] int32, qsl[0] = 0, non-decreasing,
 *                  qsl[num_seqs] = num_tokens; q_len_s = qsl[s+1] - qsl[s]
 *  num_heads % num_kv_heads == 0; num_heads / num_kv_heads in {1,2,4,8,16}
 *  head_dim in {64, 128}; block_size a multiple of 16, at most 256
 *  scale           softmax scale (usually 1/sqrt(head_dim))
 *  out             [num_tokens, num_heads, head_dim] dtype, fully overwritten
 *  dtype           PA_F32 (fp32 everywhere, CUDA-core FFMA, no TF32) or
 *                  PA_BF16 (bf16 storage, fp32 accumulation, bf16 output
 *                  rounded to nearest-even)
 *  max_seq_len     host-known upper bound on seq_lens (sizes the workspace)
 *  kv_split_tokens 0 = automatic; otherwise the most KV positions one work
 *                  item covers (e.g. 32768 for chunked long context), a
 *                  multiple of 16; splits are merged by log-sum-exp.
 *                  Extend / prefill rows on the tensor-core path are cut
 *                  into equal splits of whole 64-position tiles, up to twice
 *                  as many as the bound needs when the batch holds too few
 *                  of them to keep every CTA busy (the workspace size allows
 *                  for that)
 *
 * Errors: PA_ERR_INVALID_ARG for null pointers with nonzero sizes, negative
 * sizes, misaligned pointers; PA_ERR_UNSUPPORTED for shapes outside the list
 * above; PA_ERR_WORKSPACE when the stream is capturing and the reserved
 * workspace is too small; PA_ERR_CUDA when a launch fails.
 */
pa_status pa_forward(const void *q, const void *k_cache, const void *v_cache,
                     const int32_t *block_table, const int32_t *seq_lens,
                     const int32_t *query_start_loc, int num_heads,
                     int num_kv_heads, int head_dim, int block_size,
                     float scale, void *out, void *stream, pa_dtype dtype,
                     int num_seqs, int num_tokens, int max_blocks_per_seq,
                     int num_blocks, int max_seq_len, int kv_split_tokens);

/*
 * pa_forward_ex -- pa_forward with per-call options.
 *
 * Arguments: those of pa_forward, plus `options` (host pointer, read during
 * the call only; NULL = pa_forward exactly).  Options:
 *   sinks  device array of num_heads fp32 sink logits in natural-log units,
 *          or NULL.  "vLLM Triton attention backend deep dive", section
 *          "Usage scenarios", lists sink tokens among the model features of
 *          the unified backend: head h's softmax denominator gains
 *          exp(sinks[h]) while the sink adds no value row, so
 *            out = sum_j exp(s_j) v_j / (sum_j exp(s_j) + exp(sinks[h])).
 *          Owned by the caller; must stay valid until the call's kernels
 *          have run; 4-byte aligned (PA_ERR_INVALID_ARG otherwise).  A row
 *          with no visible key returns zeros.  pa_mla_decode takes no sinks.
 *   kv_layout  layout of k_cache and v_cache (PA_KV_NHD when options is
 *          NULL); any other value is PA_ERR_INVALID_ARG.
 *   sliding_window  0 = none; W > 0: the query at position p (p = seq_len -
 *          q_len + i for new token i) sees only the W most recent positions
 *          p - W < j <= p (the local attention of "GPT-OSS behaviour", named
 *          in the same section).  Pages wholly below every window of a
 *          request are never read, so their block-table entries may be -1.
 *          Negative: PA_ERR_INVALID_ARG.
 *   alibi_slopes  device array of num_heads fp32 ALiBi slopes m_h (natural-
 *          log units per position), or NULL; "ALiBi sqrt" is named in the
 *          same section.  Every score of head h gains -m_h * (p - j), or
 *          -m_h * sqrt(p - j) when alibi_sqrt is 1.  Caller-owned, 4-byte
 *          aligned, valid until the call's kernels have run.
 *   alibi_sqrt  0 or 1 (else PA_ERR_INVALID_ARG); ignored without slopes.
 *   max_query_len  0 = unknown; otherwise the caller's host-known bound on
 *          every request's new tokens (a serving scheduler knows it when it
 *          builds the batch).  A request with more new tokens than the
 *          bound is bad metadata: PA_DEV_BAD_QLEN, its rows written as
 *          zeros.  1 declares a decode-only batch, and no tile kernel is
 *          launched.  With bf16 inputs, head_dim 64 or 128, at most 16 query
 *          heads per KV head, num_tokens == num_seqs <= 1024 and max_seq_len
 *          <= 524288, such a call runs as ONE kernel launch -- the row kernel
 *          sizes the KV splits from seq_lens itself (at most 64 a row) and
 *          merges a row's splits in the thread block that finishes last --
 *          instead of planner, row and merge launches.  The
 *          contract is then query_start_loc[s] == s for every s: a request
 *          that breaks it (or whose seq_len is out of range) sets
 *          PA_DEV_BAD_QSL (or PA_DEV_BAD_SEQLEN) and its row s is written as
 *          zeros.  The split counters it uses live in a small library-owned
 *          buffer that is grown outside capture (PA_ERR_WORKSPACE during
 *          capture).  Values must be >= 0 (else PA_ERR_INVALID_ARG).
 * Errors as for pa_forward.
 */
typedef struct {
  const float *sinks;
  pa_kv_layout kv_layout;
  int sliding_window;
  const float *alibi_slopes;
  int alibi_sqrt;
  int max_query_len;
} pa_forward_options;

pa_status pa_forward_ex(const void *q, const void *k_cache, const void *v_cache,
                        const int32_t *block_table, const int32_t *seq_lens,
                        const int32_t *query_start_loc, int num_heads,
                        int num_kv_heads, int head_dim, int block_size,
                        float scale, void *out, void *stream, pa_dtype dtype,
                        int num_seqs, int num_tokens, int max_blocks_per_seq,
                        int num_blocks, int max_seq_len, int kv_split_tokens,
                        const pa_forward_options *options);

/* Workspace bytes pa_forward needs for these host-known extents. */
size_t pa_forward_workspace_bytes(pa_dtype dtype, int num_seqs, int num_tokens,
                                  int num_heads, int num_kv_heads,
                                  int head_dim, int max_seq_len,
                                  int kv_split_tokens);

/*
 * pa_forward_static_scratch -- pa_forward without any device allocation.
 *
 * The pages describe no counterpart of this entry point.  It serves callers
 * that must not allocate device memory while attention runs:
 *   - code running while a CUDA graph is captured in global or thread-local
 *     capture mode, where cudaMalloc / cudaFree are illegal and pa_forward
 *     would otherwise need a pa_reserve call made beforehand;
 *   - serving runtimes that hand all device memory to their own pool up
 *     front and account for every byte, so a library that allocates or grows
 *     its own workspace breaks their budget;
 *   - latency-critical loops that cannot afford pa_forward's on-demand
 *     workspace growth (freeing the old buffer synchronises the device).
 * It computes exactly what pa_forward computes, with the same kernels.  Its
 * scratch (planner tables, work counters, split partials) is one fixed region
 * of PA_STATIC_SCRATCH_BYTES that libpa.so declares as a file-scope
 * __device__ array: every GPU that loads the library holds that region until
 * the process exits.
 *
 * Arguments: those of pa_forward, plus
 *   device_status  optional device pointer to one uint32 owned by the caller;
 *                  the PA_DEV_* bits of this call are OR-ed into it (clearing
 *                  it is the caller's job).  NULL turns error reporting off:
 *                  the bits land in a word inside the static region that no
 *                  call clears or reads, so bad metadata then goes unseen
 *                  (the affected rows are still zeros).  Callers that need
 *                  the PA_DEV_* bits pass a word of their own.
 * Returns PA_ERR_SCRATCH_LIMIT and launches nothing when the call needs more
 * scratch than the region holds, i.e. when pa_forward_workspace_bytes() for
 * the same extents exceeds PA_STATIC_SCRATCH_BYTES - 256 (a decode batch of 64
 * sequences, 32 heads, head_dim 128 and max_seq_len 8192 needs about 34 MB).
 * Otherwise the status codes of pa_forward (PA_ERR_WORKSPACE only as below).
 *
 * The first call on each device looks up the region's device address
 * (cudaGetSymbolAddress, with that device current) and caches it; make that
 * first call outside any stream capture.  A first call made while `stream`
 * is capturing returns PA_ERR_WORKSPACE and launches nothing (the capture is
 * left intact); later calls may be captured.  All calls share the one region,
 * which keeps the last call's contents (each call's planner rewrites, in
 * stream order, every table and counter the call reads): calls that overlap
 * on the GPU -- on different streams, or from host threads without ordering --
 * race on it and must be serialised by the caller.  Kernel timing
 * (pa_profile_*) is not recorded for this entry point.
 */
#define PA_STATIC_SCRATCH_BYTES (64u * 1024u * 1024u)
pa_status pa_forward_static_scratch(
    const void *q, const void *k_cache, const void *v_cache,
    const int32_t *block_table, const int32_t *seq_lens,
    const int32_t *query_start_loc, int num_heads, int num_kv_heads,
    int head_dim, int block_size, float scale, void *out, void *stream,
    pa_dtype dtype, int num_seqs, int num_tokens, int max_blocks_per_seq,
    int num_blocks, int max_seq_len, int kv_split_tokens,
    uint32_t *device_status);

/*
 * pa_mla_decode -- absorbed multi-head latent attention decode ("vLLM AMD ROCm
 * attention backend optimisation", section "AITER MLA backend: optimised for
 * DeepSeek" and its "hybrid processing strategy": decode runs directly on the
 * 576-wide compressed latent).  One query token per sequence; all heads share
 * one cached latent row per position:
 *   score_j = scale * <q[s][h][0:L+R], c_j[0:L+R]>,  out[s][h] = sum_j p_j c_j[0:L]
 *
 *  q         [num_seqs, num_heads, kv_lora_rank + rope_dim] bf16
 *  kv_cache  [num_blocks, block_size, kv_lora_rank + rope_dim] bf16
 *  block_table, seq_lens as for pa_forward (seq_len >= 1)
 *  out       [num_seqs, num_heads, kv_lora_rank] bf16
 *  Supported: num_heads = 128, kv_lora_rank = 512, rope_dim = 64,
 *  block_size a multiple of 32 (at most 256).
 *  kv_split_tokens: 0 = automatic; otherwise the KV positions per work item,
 *  a multiple of 32 (the kernel's tile: a tile never crosses a page).
 *  Errors as for pa_forward; PA_ERR_UNSUPPORTED for other shapes or a
 *  kv_split_tokens that is not a multiple of 32.
 */
pa_status pa_mla_decode(const void *q, const void *kv_cache,
                        const int32_t *block_table, const int32_t *seq_lens,
                        int num_heads, int kv_lora_rank, int rope_dim,
                        int block_size, float scale, void *out, void *stream,
                        int num_seqs, int max_blocks_per_seq, int num_blocks,
                        int max_seq_len, int kv_split_tokens);

size_t pa_mla_decode_workspace_bytes(int num_seqs, int num_heads,
                                     int kv_lora_rank, int max_seq_len,
                                     int kv_split_tokens);

/*
 * pa_mla_prefill -- non-absorbed MLA prefill and extend ("vLLM AMD ROCm
 * attention backend optimisation", section "AITER MLA backend: optimised for
 * DeepSeek": prefill and extend run a standard multi-head attention on the
 * uncompressed representation, decode runs absorbed on the latent).  The
 * latent cache is decompressed for every position a request can see,
 *   k_{j,h} = [ W_K,h c_j ; k^R_j ]  (qk_nope_dim + rope_dim),
 *   v_{j,h} = W_V,h c_j              (v_head_dim),
 * and query i of request s, at position p = seq_len - q_len + i, attends
 * causally (j <= p) with softmax(scale q_{i,h} . k_{j,h}).
 *
 *  q          [num_tokens, num_heads, qk_nope_dim + rope_dim] bf16: each
 *             head's no-position part, then its rotary part
 *  kv_cache   [num_blocks, block_size, kv_lora_rank + rope_dim] bf16: per
 *             position the latent c_j, then the rotary key k^R_j shared by
 *             all heads (the pa_mla_decode cache)
 *  w_kv       [num_heads, qk_nope_dim + v_head_dim, kv_lora_rank] bf16:
 *             head h's up-projection, key rows first, then value rows
 *  block_table, seq_lens, query_start_loc: as for pa_forward (seq_lens
 *             include the new tokens, whose latents are already cached)
 *  out        [num_tokens, num_heads, v_head_dim] bf16, fully overwritten
 *  A bad block id in a request's context sets PA_DEV_BAD_BLOCK and zeroes
 *  that request's rows.
 *  Supported: kv_lora_rank 512, rope_dim 64, qk_nope_dim 128, v_head_dim
 *  128, any num_heads, block_size a multiple of 16 (at most 256: a run of
 *  16 positions never crosses a page); kv_split_tokens as for pa_forward.
 *  max_seq_len    host-known bound on seq_lens
 *  max_total_kv   host-known bound on the sum of seq_lens (sizes the
 *                 decompressed keys and values: about 81 KB per position at
 *                 128 heads); a batch beyond it sets PA_DEV_OVERFLOW and
 *                 writes zeros
 * The up-projection is this library's tensor-core GEMM (bf16 in, fp32
 * accumulation, bf16 keys and values), whose A operand is read from the
 * pages the block table names; the 64 rotary columns are stored once per
 * position, not per head.  The attention is pa_forward's tensor-core tile
 * kernel with q and k rows of 192 and v rows of 128.  Status bits and errors
 * as for pa_forward; PA_ERR_UNSUPPORTED for other dimensions.
 */
pa_status pa_mla_prefill(const void *q, const void *kv_cache, const void *w_kv,
                         const int32_t *block_table, const int32_t *seq_lens,
                         const int32_t *query_start_loc, int num_heads,
                         int kv_lora_rank, int qk_nope_dim, int rope_dim,
                         int v_head_dim, int block_size, float scale, void *out,
                         void *stream, int num_seqs, int num_tokens,
                         int max_blocks_per_seq, int num_blocks, int max_seq_len,
                         long long max_total_kv, int kv_split_tokens);

/* Workspace bytes pa_mla_prefill needs for these host-known extents. */
size_t pa_mla_prefill_workspace_bytes(int num_seqs, int num_tokens,
                                      int num_heads, int max_seq_len,
                                      long long max_total_kv,
                                      int kv_split_tokens);

/*
 * pa_reserve -- make sure the calling thread's current device has at least
 * `bytes` of library-owned workspace (split partials, planner tables, work
 * counters).  Call it before capturing a graph: during capture the library
 * never allocates and returns PA_ERR_WORKSPACE instead.  Outside capture,
 * pa_forward / pa_mla_decode grow the workspace on demand; growing frees the
 * old buffer, so graphs captured before a growth must be re-captured.
 * Returns PA_ERR_CUDA if the allocation fails.
 */
pa_status pa_reserve(size_t bytes);

/* Synchronises `stream`, copies the device status word of the current device
 * into *host_flags and clears it.  Not capturable (it synchronises). */
pa_status pa_get_device_status(void *stream, uint32_t *host_flags);

/* Static, human-readable name of a status code. */
const char *pa_status_string(pa_status status);

/* Number of SMs of the current device, as the library sizes its grids. */
int pa_num_sms(void);

/*
 * pa_cache_write -- the paged KV-cache write that precedes pa_forward ("vLLM
 * Triton attention backend deep dive", section "Technical implementation of
 * paged attention": the cache is a pool of fixed-size blocks and a sequence's
 * block table maps its logical block j to a physical block).  New token i of
 * request s (q_len_s = qsl[s+1] - qsl[s] new tokens, seq_lens[s] positions
 * including them) sits at position pos = seq_lens[s] - q_len_s + i; its K and
 * V rows are copied, bit for bit, to slot pos % block_size of physical block
 * block_table[s][pos / block_size]:
 *
 *  k_new, v_new     [num_tokens, num_kv_heads, head_dim]            dtype
 *  k_cache, v_cache [num_blocks, block_size, num_kv_heads, head_dim] dtype
 *                   (PA_KV_NHD) or [num_blocks, num_kv_heads, block_size,
 *                   head_dim] (PA_KV_HND), written in place; every other slot
 *                   is left untouched
 *  block_table, seq_lens, query_start_loc: as for pa_forward (seq_lens are
 *                   the lengths after this write)
 *  head_dim x element size a multiple of 16 bytes; any block_size >= 1
 *
 * Asynchronous on `stream`, allocation-free after the first call on a device
 * (it uses 256 bytes of the library workspace), graph-capturable.  Bad device
 * metadata never traps (status bits as for pa_forward):
 *   PA_DEV_BAD_QSL    query_start_loc[0] != 0, decreasing, or
 *                     query_start_loc[num_seqs] != num_tokens: nothing written
 *   PA_DEV_BAD_QLEN   q_len > seq_len: that request's rows are not written
 *   PA_DEV_BAD_BLOCK  a block id outside [0, num_blocks) (or past
 *                     max_blocks_per_seq): that token's rows are not written
 * Errors: PA_ERR_INVALID_ARG for null pointers with num_tokens > 0, negative
 * sizes, num_seqs == 0 with num_tokens > 0, or tensors not 16-byte aligned;
 * PA_ERR_UNSUPPORTED when a row is not a multiple of 16 bytes; PA_ERR_CUDA
 * when a launch fails; PA_ERR_INVALID_ARG for an unknown kv_layout.
 * num_tokens == 0 launches nothing.
 */
pa_status pa_cache_write(const void *k_new, const void *v_new, void *k_cache,
                         void *v_cache, const int32_t *block_table,
                         const int32_t *seq_lens, const int32_t *query_start_loc,
                         int num_kv_heads, int head_dim, int block_size,
                         void *stream, pa_dtype dtype, int num_seqs,
                         int num_tokens, int max_blocks_per_seq, int num_blocks,
                         pa_kv_layout kv_layout);

/*
 * pa_debug_gather -- the page-gather indexing alone (PA_KV_NHD), for
 * bit-exact tests:
 *   dense_out[s][j][:] = k_cache[block_table[s][j / bs]][j % bs][0:row_elems]
 * for j < seq_lens[s] (raw element bits copied, elem_bytes 2 or 4); positions
 * j >= seq_lens[s] are left untouched.  dense_out is
 * [num_seqs, max_seq_len, row_elems].  Bad block ids set PA_DEV_BAD_BLOCK and
 * leave their rows untouched.
 */
pa_status pa_debug_gather(const void *k_cache, const int32_t *block_table,
                          const int32_t *seq_lens, int num_seqs,
                          int max_blocks_per_seq, int num_blocks,
                          int block_size, int row_elems, int elem_bytes,
                          int max_seq_len, void *dense_out, void *stream);

/*
 * pa_debug_wait_timeout -- test-only check of the kernels' failure path: one
 * kernel waits, with the bounded wait every kernel of this library uses, on
 * an mbarrier that nothing arrives on.  After limit_ns nanoseconds of wall
 * clock (1 <= limit_ns <= 1e9, the kernels' own limit) the wait gives up,
 * sets PA_DEV_TIMEOUT in the device status word and the kernel returns, so
 * the context stays usable: nothing traps, no copy is left in flight.
 *   done  device pointer to one int owned by the caller; set to 2 when the
 *         kernel has returned (its timed-out wait and a second wait that
 *         returns at once).
 * Asynchronous on `stream`; read the bit with pa_get_device_status.
 */
pa_status pa_debug_wait_timeout(uint64_t limit_ns, int *done, void *stream);

/*
 * Kernel timing.  While enabled, every kernel that pa_forward, pa_mla_decode
 * and pa_debug_gather launch is bracketed by a pair of CUDA events recorded
 * on the caller's stream (nothing is recorded for a stream that is being
 * captured).  pa_profile_read synchronises on those events, writes for each
 * kernel id below the summed milliseconds and the launch count (arrays of
 * PA_K_COUNT entries), and clears the record.  Recording costs two event
 * records per launch and no synchronisation.
 */
enum {
  PA_K_PLAN = 0,      /* one-block planner                          */
  PA_K_ROW = 1,       /* row-streaming kernel (decode path)         */
  PA_K_TILE = 2,      /* tensor-core extend/prefill tile kernel     */
  PA_K_MERGE = 3,     /* log-sum-exp merge of split partials        */
  PA_K_MLA = 4,       /* absorbed-MLA decode kernel                 */
  PA_K_MLA_MERGE = 5, /* MLA log-sum-exp merge                      */
  PA_K_GATHER = 6,    /* debug gather                               */
  PA_K_UPPROJ = 7,    /* MLA prefill up-projection (tensor cores)   */
  PA_K_MLA_ROPE = 8,  /* MLA prefill rotary-key copy                */
  PA_K_COUNT = 10
};
pa_status pa_profile_enable(int on);
pa_status pa_profile_read(double *total_ms, int *launches);
const char *pa_kernel_name(int kernel_id);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
