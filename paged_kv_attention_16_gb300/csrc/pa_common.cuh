// pa_common.cuh -- device-side building blocks shared by the kernels of
// libpa.so: plan structures written by the planner, inline-PTX wrappers for
// mbarriers, TMA tensor copies and proxy fences, bounded waits, warp scans.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa.h"

namespace pa {

// ---------------------------------------------------------------------------
// Plan: what the one-block planner writes for the consumer kernels.
// ---------------------------------------------------------------------------

enum ReqClass : int { kDecode = 0, kExtend = 1, kPrefill = 2 };

enum ReqFlags : int {
  kFlagValid = 1 << 4,   // metadata checks passed
  kFlagRowPath = 1 << 5, // rows go through the row-streaming kernel
};

// Per request (original index s).
struct ReqInfo {
  int q_start;        // query_start_loc[s]
  int q_len;          // new tokens
  int ctx;            // seq_lens[s]: KV positions including the new tokens
  int flags;          // ReqClass in bits 0..3, ReqFlags above
  int nsplit;         // KV splits per row (>= 1)
  int split_len;      // KV positions per split
  int kv_base;        // first KV position of split 0 (16-aligned; > 0 only
                      // with a sliding window, below which no row looks)
  long long partial_base;  // first partial row of this request (nsplit > 1)
};

// Work lists are never materialised: every list is a virtual index space
// [0, n) laid over the requests in [decode : extend : prefill] order, with
// end[k] = inclusive prefix of the per-request counts.  A consumer maps an
// index to its request with a binary search over end[].
// kListMergeLong: the merge rows with more than kWarpMergeSplits non-empty
// splits (a suffix of each request's rows), merged by a whole block each.
enum ListId : int {
  kListRow = 0,
  kListTile = 1,
  kListMerge = 2,
  kListZero = 3,
  kListMergeLong = 4,
  kNumLists = 5
};

// Rows with at most this many non-empty splits are merged by one warp.
constexpr int kWarpMergeSplits = 32;

struct PlanHeader {
  long long n[kNumLists];       // total entries per list
  unsigned long long counter[8];  // dynamic work counters, reset by the planner
  int qsl_bad;                  // query_start_loc failed its checks
  int split_len_decode;         // chosen decode split length
  long long partial_rows;       // partial rows the plan uses
};

// Device pointers into the workspace plus the call's scalars.
struct FwdParams {
  const void *q;
  void *out;
  const int32_t *block_table;
  const int32_t *seq_lens;
  const int32_t *qsl;
  int num_seqs, num_tokens, num_heads, num_kv_heads, head_dim, block_size;
  int max_blocks_per_seq, num_blocks, max_seq_len, kv_split_tokens;
  float scale;
  float scale_log2;   // scale * log2(e): scores kept in the base-2 domain
  int tile_ok;        // extend/prefill rows go to the tensor-core tile kernel
  int row_ctas;       // resident CTAs of the row kernel (split sizing)
  int tile_ctas;      // CTAs of the tile kernel's grid (split sizing)
  int dtype;          // pa_dtype
  // workspace
  PlanHeader *plan;
  ReqInfo *req;
  int *ord;                 // [num_seqs] request index at each reordered position
  long long *list_end;      // [kNumLists][num_seqs]
  float *part_o;            // [part_cap][head_dim]
  float *part_lse;          // [part_cap] (base-2 log-sum-exp; NaN marks a bad split)
  long long part_cap;
  unsigned int *status;
  const float *sinks;       // [num_heads] sink logits (natural-log units) or null
  int window;               // sliding window in positions (0: none)
  int head_dim_qk;          // width of q / k rows when it differs from head_dim
                            // (the value / output width); 0: the same
  int all_tile;             // 1: every row, decode included, on the tile kernel
  int tile_page_boxes;      // 1: every 64-position tile of the tile kernel lies in
                            // one page (block_size % 64 == 0, 64-aligned tiles):
                            // K and V load as one 64-slot box per tile
  const float *alibi;       // [num_heads] ALiBi slopes (natural-log units) or null
  int alibi_sqrt;           // 1: the bias grows with the square root of the distance
  int k_rope_split;         // 1: the last 64 key columns come from a separate
                            // [pages, slots, 1, 64] tensor shared by all heads
  int max_qlen;             // the caller's bound on q_len (0: none); a request
                            // above it is bad metadata (PA_DEV_BAD_QLEN)
  // Decode-only batches declared by the caller (one launch, no planner): the
  // row kernel sizes the splits itself from seq_lens (at most fast_nsmax a
  // row); partial rows (s * H + head) * fast_nsmax + split; fast_work: [0]
  // item counter, [1] CTAs done taking items; fast_cnt: [num_seqs *
  // kv_heads] splits finished per row group (zero between calls).
  int fast;
  int fast_nsmax;
  unsigned long long *fast_work;
  unsigned int *fast_cnt;
};

// First KV position the query at position `pos` sees: with a sliding window
// W the W most recent positions pos - W < j <= pos ("vLLM Triton attention
// backend deep dive", section "Usage scenarios": GPT-OSS behaviour).
__host__ __device__ inline int window_lo(int pos, int window) {
  return window > 0 && pos - window + 1 > 0 ? pos - window + 1 : 0;
}

// ALiBi bias of a key `dist` = pos - j positions back, in the base-2 score
// domain (slope2 = slope * log2 e): -slope2 * dist, or -slope2 * sqrt(dist).
// dist < 0 (a masked future key) is clamped so that sqrt stays defined.  The
// square root is the single-instruction approximate one (relative error of
// a few ulp): the bias feeds a softmax whose inputs are rounded far more
// coarsely, and the exact root costs several instructions per score.
__device__ inline float alibi_bias(float slope2, float dist, int use_sqrt) {
  if (!use_sqrt) return -slope2 * dist;
  float r;
  asm("sqrt.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(fmaxf(dist, 0.f)));
  return -slope2 * r;
}

constexpr float kLog2eF = 1.4426950408889634f;

// Attention sinks ("vLLM Triton attention backend deep dive", section "Usage
// scenarios": sink tokens): head h's softmax denominator gains exp(sink_h),
// and the sink carries no value.  With a row's keys reduced to (m, l) in the
// base-2 domain (l = sum 2^(s - m)), the reciprocal of the full denominator.
__device__ inline float sink_inv(const float *sinks, int head, float m, float l) {
  const float den = sinks ? l + exp2f(__ldg(sinks + head) * kLog2eF - m) : l;
  return den > 0.f ? 1.f / den : 0.f;
}

// Largest split length of the row kernel (bounds its per-item page list).
constexpr int kRowMaxSplit = 8192;
constexpr int kRowMinSplit = 256;
// Decode-only batches run as one row-kernel launch up to this many requests
// (the kernel keeps one prefix entry per request in shared memory).
constexpr int kFastMaxSeqs = 1024;
constexpr int kFastMinSplit = 64;  // their shortest split: one row-kernel stage
// Rows per tensor-core tile of the extend/prefill kernel.
constexpr int kTileRows = 128;

__host__ __device__ inline long long ceil_div_ll(long long a, long long b) {
  return (a + b - 1) / b;
}

// Index of the list entry: first k with end[k] > idx (end is non-decreasing).
__device__ inline int list_find(const long long *end, int n, long long idx) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    int mid = (lo + hi) >> 1;
    if (__ldg(end + mid) > idx) hi = mid; else lo = mid + 1;
  }
  return lo;
}

// list_find over a copy in shared memory (plain loads: __ldg is global-only).
__device__ inline int list_find_shared(const long long *end, int n, long long idx) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    int mid = (lo + hi) >> 1;
    if (end[mid] > idx) hi = mid; else lo = mid + 1;
  }
  return lo;
}

// Rolling cache of block-table entries for a producer warp: lane i holds
// entry base + i of the current chunk and base + 32 + i of the next, so a
// stream of page look-ups that only moves forward costs one coalesced load
// per 32 pages, issued a chunk ahead, instead of a dependent load per tile.
struct PageCache {
  const int32_t *bt;
  int limit;  // entries at or beyond `limit` read as -1
  int base, cur, nxt;

  __device__ void start(const int32_t *table, int lim, int first, int lane) {
    bt = table;
    limit = lim;
    base = first;
    cur = first + lane < lim ? __ldg(table + first + lane) : -1;
    nxt = first + 32 + lane < lim ? __ldg(table + first + 32 + lane) : -1;
  }

  // All 32 lanes call; lp < 0 means this lane needs no page.  Needed pages
  // must not move backwards between calls.
  __device__ int get(int lp, int lane) {
    int lo = __reduce_min_sync(0xffffffffu, lp < 0 ? 0x7fffffff : lp);
    while (lo != 0x7fffffff && lo >= base + 32) {
      base += 32;
      cur = nxt;
      const int n = base + 32 + lane;
      nxt = n < limit ? __ldg(bt + n) : -1;
    }
    const int off = lp - base;
    const int a = __shfl_sync(0xffffffffu, cur, off & 31);
    const int b = __shfl_sync(0xffffffffu, nxt, off & 31);
    if (lp < 0) return -1;
    if (off >= 0 && off < 32) return a;
    if (off >= 32 && off < 64) return b;
    return lp < limit ? __ldg(bt + lp) : -1;  // far jump: read directly
  }
};

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------

__device__ inline uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ inline void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ inline void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ inline void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ inline void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ inline void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ inline bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ inline uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Wall-clock limit of one bounded wait.  A wait that runs out sets
// PA_DEV_TIMEOUT and the caller carries on (results are then flagged as
// garbage by the status word); `dead` makes every later wait of the same
// thread return at once so a kernel whose copies never land still ends.
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s

// Bounded wait with an explicit limit (the kernels use kWaitLimitNs).
__device__ inline void mbar_wait_limit(uint64_t *bar, uint32_t parity, bool &dead,
                                       unsigned int *status, uint64_t limit_ns) {
  if (dead) return;
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return;
    if ((i & 63u) == 0 && global_timer_ns() - t0 > limit_ns) {
      atomicOr(status, PA_DEV_TIMEOUT);
      dead = true;
      return;
    }
  }
}

__device__ inline void mbar_wait(uint64_t *bar, uint32_t parity, bool &dead,
                                 unsigned int *status) {
  mbar_wait_limit(bar, parity, dead, status, kWaitLimitNs);
}

// 4-D tiled TMA load global -> shared, completion counted on `bar`.
__device__ inline void tma_load_4d(void *dst, const CUtensorMap *map, int c0, int c1, int c2,
                                   int c3, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "r"(smem_u32(bar))
      : "memory");
}

// 5-D tiled TMA load global -> shared, completion counted on `bar`.
__device__ inline void tma_load_5d(void *dst, const CUtensorMap *map, int c0, int c1, int c2,
                                   int c3, int c4, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4),
      "r"(smem_u32(bar))
      : "memory");
}

__device__ inline void tma_load_2d(void *dst, const CUtensorMap *map, int c0, int c1,
                                   uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

__device__ inline void tma_load_3d(void *dst, const CUtensorMap *map, int c0, int c1, int c2,
                                   uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// Bring a 4-D / 3-D TMA box into L2 without touching shared memory (deepens
// the load pipeline beyond what the shared-memory ring can hold).
__device__ inline void tma_prefetch_4d(const CUtensorMap *map, int c0, int c1, int c2, int c3) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}

__device__ inline void tma_prefetch_3d(const CUtensorMap *map, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}

__device__ inline void prefetch_tensor_map(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Hardware base-2 exponential (MUFU), used for softmax weights.
__device__ inline float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed two-lane fp32 FMA (one instruction, two IEEE fma results):
// returns {a0 * b0 + c0, a1 * b1 + c1}.
// Three-input maximum (one instruction on sm_100 and later).
__device__ inline float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ inline void ffma2(float &c0, float &c1, float a0, float a1, float b0, float b1) {
  asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%0, %1};\n\t"
      "fma.rn.f32x2 rc, ra, rb, rc;\n\t"
      "mov.b64 {%0, %1}, rc;\n\t}"
      : "+f"(c0), "+f"(c1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// bf16x2 packed in a 32-bit word -> two floats (bf16 is the top half of fp32).
__device__ inline float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ inline float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// ---------------------------------------------------------------------------
// Block-wide inclusive scan of 64-bit counts (blockDim.x a multiple of 32,
// at most 1024).  `scratch` holds 33 long longs.  Returns the inclusive
// prefix of `v`; *total receives the block total.  All threads must call.
// ---------------------------------------------------------------------------
__device__ inline long long block_inclusive_scan(long long v, long long *scratch,
                                                 long long *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    long long w = lane < nwarps ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      long long y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < nwarps) scratch[lane] = w;
    if (lane == nwarps - 1) scratch[32] = w;
  }
  __syncthreads();
  if (warp > 0) x += scratch[warp - 1];
  *total = scratch[32];
  __syncthreads();
  return x;
}

// Block-wide inclusive scan of N 64-bit counts at once (one pair of
// barriers for all N).  `scratch` holds N * 33 long longs; tot[i] receives
// the block total of v[i].  All threads must call.
template <int N>
__device__ inline void block_scan_multi(long long (&v)[N], long long *scratch,
                                        long long (&tot)[N]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
#pragma unroll
  for (int i = 0; i < N; ++i) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, v[i], o);
      if (lane >= o) v[i] += y;
    }
    if (lane == 31) scratch[i * 33 + warp] = v[i];
  }
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
      long long w = lane < nwarps ? scratch[i * 33 + lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      if (lane < nwarps) scratch[i * 33 + lane] = w;
      if (lane == nwarps - 1) scratch[i * 33 + 32] = w;
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < N; ++i) {
    if (warp > 0) v[i] += scratch[i * 33 + warp - 1];
    tot[i] = scratch[i * 33 + 32];
  }
  __syncthreads();
}

}  // namespace pa

namespace pa {

// ---------------------------------------------------------------------------
// tcgen05 (5th-generation tensor core) wrappers: TMEM allocation, MMA issue,
// commit to an mbarrier, TMEM <-> register moves, and the ordering fences.
// ---------------------------------------------------------------------------

// Shared-memory matrix descriptor for a 128-byte-swizzled operand tile
// (start address, leading / stride byte offsets, descriptor version 1,
// layout SWIZZLE_128B).  The tile's base must be 1024-byte aligned.
__device__ inline uint64_t umma_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;  // SWIZZLE_128B
  return d;
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 accumulator, M x N,
// A K-major; B K-major (b_mn_major = 0) or MN-major (1).
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N, int b_mn_major) {
  return (1u << 4)                      // D format: f32
         | (1u << 7)                    // A format: bf16
         | (1u << 10)                   // B format: bf16
         | ((uint32_t)b_mn_major << 16) // B major-ness
         | ((uint32_t)(N >> 3) << 17)   // N / 8
         | ((uint32_t)(M >> 4) << 24);  // M / 16
}

__device__ inline void tc_mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                   uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Same MMA with the A operand (M x K, K-major, bf16 pairs packed in 32-bit
// columns, row i in lane i) read from tensor memory at `tmem_a`.
__device__ inline void tc_mma_bf16_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc,
                                      uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
      "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 op issued so far by this thread is done.
__device__ inline void tc_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ inline void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ inline void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Warp-wide TMEM allocation of `ncols` columns; the base address lands in *dst.
__device__ inline void tc_alloc(uint32_t *dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ inline void tc_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// 32 consecutive 32-bit TMEM columns of this thread's lane (warp-wide).
__device__ inline void tc_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ inline void tc_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// 16 consecutive 32-bit TMEM columns of this thread's lane (warp-wide).
__device__ inline void tc_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

__device__ inline void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ inline void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Named barrier over `count` threads (ids 1..15; 0 is __syncthreads).
// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialization may start (and run its prologue) while the kernel before it
// in the stream is still finishing; pdl_wait() blocks until that kernel has
// completed and its writes are visible, so it must precede every access to
// data the earlier kernels produce.  pdl_trigger() lets the next kernel start
// launching early; the next kernel still waits for this one to complete.
__device__ inline void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ inline void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ inline void named_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

}  // namespace pa

namespace pa {

// ---------------------------------------------------------------------------
// Thread-block-cluster wrappers (distributed shared memory)
// ---------------------------------------------------------------------------

__device__ inline uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of the same shared-memory offset in CTA `rank` of this cluster.
__device__ inline uint32_t cluster_map(uint32_t local_saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_saddr), "r"(rank));
  return r;
}

__device__ inline void st_cluster_v4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b),
               "f"(c), "f"(d)
               : "memory");
}

// Arrive on an mbarrier of another CTA of the cluster, releasing this
// thread's prior writes at cluster scope.
__device__ inline void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// Remote arrive without release semantics: for signalling "my reads of a
// buffer are done" after a CTA barrier that already orders those reads (a
// cluster-scope release costs on the order of two thousand cycles here).
__device__ inline void mbar_arrive_remote_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

__device__ inline bool mbar_try_wait_cluster(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait with cluster-scope acquire (for barriers other CTAs arrive on).
__device__ inline void mbar_wait_cluster(uint64_t *bar, uint32_t parity, bool &dead,
                                         unsigned int *status) {
  if (dead) return;
  if (mbar_try_wait_cluster(bar, parity)) return;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait_cluster(bar, parity)) return;
    if ((i & 63u) == 0 && global_timer_ns() - t0 > kWaitLimitNs) {
      atomicOr(status, PA_DEV_TIMEOUT);
      dead = true;
      return;
    }
  }
}

// Bulk copy of `bytes` (multiple of 16) from this CTA's shared memory to
// another CTA of the cluster; completion is counted as transaction bytes on
// the destination CTA's mbarrier.
__device__ inline void bulk_copy_to_peer(uint32_t dst_cluster, const void *src, uint32_t bytes,
                                         uint32_t mbar_cluster) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst_cluster),
      "r"(smem_u32(src)), "r"(bytes), "r"(mbar_cluster)
      : "memory");
}

__device__ inline void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

}  // namespace pa
