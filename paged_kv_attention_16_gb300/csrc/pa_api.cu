// pa_api.cu -- the C ABI of libpa.so (include/pa.h): argument checks,
// library-owned workspace, TMA tensor maps, and the three small kernels around
// the attention kernels: the one-block planner, the log-sum-exp merge and the
// debug gather.
//
// Planner ("vLLM AMD ROCm attention backend optimisation", sections "Mixed
// inference workload challenge" and "Batch reordering"; "vLLM Triton
// attention backend deep dive", section "Persistent kernels and CUDA graphs"):
// reads seq_lens / query_start_loc on the device, classifies each request as
// decode (1 new token), prefill (no cached prefix) or extend, stably orders
// the requests [decode : extend : prefill], sizes the KV splits, and lays the
// work lists over that order as prefix sums.  The host never reads device
// metadata, so the whole call is capturable in a CUDA graph and the grids
// are fixed (a multiple of the SM count).
//
// Merge ("vLLM Triton attention backend deep dive", section "Parallel tiled
// softmax (3D kernel)": a second launch reduces the partial results;
// "vLLM AMD ROCm attention backend optimisation", section "Chunked context
// processing": LSE-based merge): out = sum_p w_p O_p with
// w_p = 2^(lse_p - M) / sum_q 2^(lse_q - M), M = max_p lse_p (base 2).
#include <algorithm>
#include <mutex>

#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kPlanThreads = 1024;
constexpr int kMergeThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------------------
// planner
// ---------------------------------------------------------------------------

struct ReqScalars {
  int q_start, q_len, ctx, cls;
  bool valid;
};

__device__ inline ReqScalars classify(const FwdParams &p, int q_start, int q_end, int ctx,
                                      bool qsl_bad) {
  ReqScalars r;
  r.q_start = q_start;
  r.q_len = q_end - q_start;
  r.ctx = ctx;
  r.valid = !qsl_bad && r.q_len >= 0 && r.ctx >= 0 && r.q_len <= r.ctx &&
            (p.max_qlen <= 0 || r.q_len <= p.max_qlen) && r.ctx <= p.max_seq_len &&
            ceil_div_ll(r.ctx, p.block_size) <= (long long)p.max_blocks_per_seq;
  if (r.q_len == 1) r.cls = kDecode;
  else if (r.q_len == r.ctx) r.cls = kPrefill;
  else r.cls = kExtend;
  if (!r.valid || r.q_len <= 0) r.cls = kDecode;  // no work; position is irrelevant
  return r;
}

// Requests handled from shared memory in one pass per step; larger batches
// loop over chunks of kPlanThreads and re-read the metadata.
constexpr int kPlanCache = kPlanThreads;

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const FwdParams p) {
  __shared__ long long scratch[(kNumLists + 1) * 33];
  __shared__ int4 s_req[kPlanCache];  // q_start, q_end, ctx, -
  __shared__ int s_ord[kPlanCache];
  const int S = p.num_seqs, T = p.num_tokens, tid = threadIdx.x, nthr = blockDim.x;
  const int Hk = p.num_kv_heads, G = p.num_heads / p.num_kv_heads, H = p.num_heads;
  const bool cached = S <= kPlanCache;
  // Launched programmatically after whatever preceded this call in the
  // stream: wait for it (it may have written the metadata, or still read
  // this workspace) before touching memory.
  pdl_wait();
  pdl_trigger();  // the row kernel may start its prologue meanwhile
  auto raw = [&](int s) -> int4 {
    if (cached) return s_req[s];
    return make_int4(p.qsl[s], p.qsl[s + 1], p.seq_lens[s], 0);
  };

  // -- one read of the metadata, and the global query_start_loc checks -------
  int bad = 0;
  if (cached && tid < S) s_req[tid] = make_int4(p.qsl[tid], p.qsl[tid + 1], p.seq_lens[tid], 0);
  if (tid == 0 && (p.qsl[0] != 0 || p.qsl[S] != T)) bad = 1;
  for (int s = tid; s < S; s += nthr)
    if (p.qsl[s + 1] < p.qsl[s]) bad = 1;
  const bool qsl_bad = __syncthreads_or(bad) != 0;

  // -- pass 1: class counts, decode KV work, tile work (split sizing) --------
  // v1: packed class counts (21 bits each), decode KV positions, and the
  // tile kernel's work in KV positions x query tiles (per KV head)
  long long v1[3] = {0, 0, 0};
  const int TQ = p.tile_ok && G <= kTileRows ? kTileRows / G : 0;  // tokens per query tile
  int metabad = 0;
  for (int s = tid; s < S; s += nthr) {
    const int4 q = raw(s);
    const ReqScalars r = classify(p, q.x, q.y, q.z, qsl_bad);
    v1[0] += 1ll << (21 * r.cls);
    if (r.valid && r.q_len == 1) v1[1] += p.window > 0 ? min(r.ctx, p.window) : r.ctx;
    if (TQ > 0 && r.valid && r.q_len > 0 && (r.cls != kDecode || p.all_tile)) {
      // tile t sees prefix + min((t + 1) TQ, q_len) positions
      const int nt = (r.q_len + TQ - 1) / TQ;
      long long w = (long long)nt * (r.ctx - r.q_len) + (((long long)TQ * (nt - 1) * nt) >> 1) + r.q_len;
      if (p.window > 0) w = min(w, (long long)nt * (p.window + TQ));
      v1[2] += w;
    }
    if (!qsl_bad && !r.valid) {
      if (r.q_len < 0 || r.q_len > r.ctx || (p.max_qlen > 0 && r.q_len > p.max_qlen))
        metabad |= PA_DEV_BAD_QLEN;
      if (r.ctx < 0 || r.ctx > p.max_seq_len ||
          ceil_div_ll(r.ctx, p.block_size) > (long long)p.max_blocks_per_seq)
        metabad |= PA_DEV_BAD_SEQLEN;
    }
  }
  if (metabad) atomicOr(p.status, (unsigned)metabad);
  if (tid == 0 && qsl_bad) atomicOr(p.status, PA_DEV_BAD_QSL);
  long long t1[3];
  block_scan_multi<3>(v1, scratch, t1);
  const long long class_tot = t1[0], work_tot = t1[1], tile_tot = t1[2];
  const long long mask21 = (1ll << 21) - 1;
  const long long n_dec = class_tot & mask21, n_ext = (class_tot >> 21) & mask21;

  // Decode split: the multiple of 64 positions that makes the item count
  // about 8 items per resident CTA (4 per CTA from G = 8 on: their items
  // carry more work per KV byte), within [kRowMinSplit, kRowMaxSplit].  Not
  // rounded to a power of two: that could leave the last wave of items
  // covering only part of the grid.
  const long long target = (G >= 8 ? 4ll : 8ll) * (p.row_ctas > 0 ? p.row_ctas : 1);
  const long long kv_work = work_tot * Hk;
  const long long Lw = ceil_div_ll(ceil_div_ll(kv_work, target), 64) * 64;
  int L = (int)(Lw < kRowMinSplit ? kRowMinSplit : (Lw > kRowMaxSplit ? kRowMaxSplit : Lw));
  if (p.kv_split_tokens > 0 && p.kv_split_tokens < L) L = p.kv_split_tokens;
  // Tile rows under a kv_split_tokens bound: equal splits of whole 64-position
  // tiles, twice as many as the bound needs when the tile work would give each
  // tile CTA fewer than about 4 bound-long items (the dynamic deal then ends
  // with a long tail of single items).
  const bool tile_fine = p.kv_split_tokens > 0 && p.tile_ctas > 0 &&
                         tile_tot * Hk < 4ll * p.kv_split_tokens * p.tile_ctas;
  // Extend/prefill rows on the row path: at most ~4 splits per row.
  int Lr = (int)ceil_div_ll(ceil_div_ll(p.max_seq_len, 4), 16) * 16;
  if (Lr < L) Lr = L;
  if (Lr > kRowMaxSplit) Lr = kRowMaxSplit;
  if (p.kv_split_tokens > 0 && p.kv_split_tokens < Lr) Lr = p.kv_split_tokens;

  // -- pass 2: stable partition into [decode : extend : prefill] -------------
  long long carry = 0;
  for (int base = 0; base < S; base += nthr) {
    const int s = base + tid;
    long long v[1] = {0};
    int cls = 0;
    if (s < S) {
      const int4 q = raw(s);
      cls = classify(p, q.x, q.y, q.z, qsl_bad).cls;
      v[0] = 1ll << (21 * cls);
    }
    long long ct[1];
    block_scan_multi<1>(v, scratch, ct);
    const long long incl = v[0] + carry;
    if (s < S) {
      const long long before = ((incl >> (21 * cls)) & mask21) - 1;
      const long long off = cls == kDecode ? 0 : cls == kExtend ? n_dec : n_dec + n_ext;
      p.ord[off + before] = s;
      if (cached) s_ord[off + before] = s;
    }
    carry += ct[0];
  }
  __syncthreads();

  // -- pass 3: per-request plan and list prefix sums in reordered order ------
  long long run[kNumLists + 1] = {};  // lists, then partial rows
  for (int base = 0; base < S; base += nthr) {
    const int k = base + tid;
    long long cnt[kNumLists + 1] = {};
    int s = -1;
    ReqInfo info{};
    if (k < S) {
      s = cached ? s_ord[k] : p.ord[k];
      const int4 q = raw(s);
      const ReqScalars r = classify(p, q.x, q.y, q.z, qsl_bad);
      // Decode rows stream through the row kernel (warp MMAs for bf16, at
      // most 16 query rows per KV head); extend and prefill rows fill
      // 128-row tiles of the tcgen05 tile kernel when it applies.
      const bool row_path = !p.tile_ok || (r.cls == kDecode && !p.all_tile);
      // With a sliding window no row looks below the first row's window:
      // splits start there (16-aligned, so that no copy box crosses a page).
      const int kv_base = window_lo(r.ctx - r.q_len, p.window) & ~15;
      int len;
      if (r.cls == kDecode) {
        len = L;
        if (p.kv_split_tokens > 0 && p.kv_split_tokens < len) len = p.kv_split_tokens;
      } else if (row_path) {
        len = Lr;
      } else if (p.kv_split_tokens > 0) {
        const int range = r.ctx - kv_base > 0 ? r.ctx - kv_base : 1;
        const int ns = (int)ceil_div_ll(range, p.kv_split_tokens) * (tile_fine ? 2 : 1);
        len = (int)ceil_div_ll(ceil_div_ll(range, ns), 64) * 64;
        if (len > p.kv_split_tokens) len = p.kv_split_tokens;
      } else {
        len = r.ctx > 0 ? r.ctx : 1;
      }
      int nsplit = (int)ceil_div_ll(r.ctx - kv_base > 0 ? r.ctx - kv_base : 1, len);
      if (nsplit < 1) nsplit = 1;
      info.q_start = r.q_start;
      info.q_len = r.q_len;
      info.ctx = r.ctx;
      info.flags = r.cls | (r.valid ? kFlagValid : 0) | (row_path ? kFlagRowPath : 0);
      info.nsplit = nsplit;
      info.split_len = len;
      info.kv_base = kv_base;
      if (r.valid && r.q_len > 0) {
        if (row_path) cnt[kListRow] = (long long)Hk * r.q_len * nsplit;
        else cnt[kListTile] = (long long)Hk * ceil_div_ll((long long)r.q_len * G, kTileRows) * nsplit;
        if (nsplit > 1) {
          // row i reaches split ceil((ctx - q_len + i + 1 - kv_base) / len)
          // - 1: more than kWarpMergeSplits splits from
          // i = W * len - (ctx - q_len - kv_base) on (a sliding window can
          // leave fewer non-empty ones; the long pass skips those rows)
          const long long i_long =
              max(0ll, (long long)kWarpMergeSplits * len - (r.ctx - r.q_len - kv_base));
          if (i_long < r.q_len) cnt[kListMergeLong] = (r.q_len - i_long) * H;
          cnt[kListMerge] = (long long)r.q_len * H;
          cnt[kNumLists] = (long long)r.q_len * H * nsplit;
        }
      } else if (!qsl_bad && r.q_len > 0) {
        cnt[kListZero] = (long long)r.q_len * H;
      }
    }
    const long long part = cnt[kNumLists];
    long long tot[kNumLists + 1];
    block_scan_multi<kNumLists + 1>(cnt, scratch, tot);
    info.partial_base = cnt[kNumLists] + run[kNumLists] - part;
#pragma unroll
    for (int x = 0; x < kNumLists; ++x)
      if (k < S) p.list_end[(size_t)x * S + k] = cnt[x] + run[x];
#pragma unroll
    for (int x = 0; x <= kNumLists; ++x) run[x] += tot[x];
    if (k < S) p.req[s] = info;
  }
  if (tid == 0) {
    const long long run_part = run[kNumLists];
    const bool overflow = run_part > p.part_cap;
    if (overflow) atomicOr(p.status, PA_DEV_OVERFLOW);
    const bool zero_all = qsl_bad || overflow;
    for (int x = 0; x < kNumLists; ++x) p.plan->n[x] = zero_all ? 0 : run[x];
    for (int x = 0; x < 8; ++x) p.plan->counter[x] = 0;
    p.plan->qsl_bad = zero_all ? 1 : 0;
    p.plan->split_len_decode = L;
    p.plan->partial_rows = run_part;
  }
}

// ---------------------------------------------------------------------------
// log-sum-exp merge of split partials (one CTA per row)
// ---------------------------------------------------------------------------

template <typename T>
__device__ inline void store_out(T *dst, float v);
template <>
__device__ inline void store_out<float>(float *dst, float v) { *dst = v; }
template <>
__device__ inline void store_out<__nv_bfloat16>(__nv_bfloat16 *dst, float v) {
  *dst = __float2bfloat16_rn(v);
}

// Rows with at most kWarpMergeSplits non-empty splits are merged by one warp
// (lane q holds split q's log-sum-exp; lanes over head_dim for the sums);
// longer rows (their own list) by a whole block (warps over splits).
// Merge-list prefix sums kept in shared memory for batches up to this size.
constexpr int kMergeCache = 1024;

struct MergeRow {
  long long tok, base;
  int h, nn;
};

// Row i, head h of request r: its non-empty splits are first .. last, the
// splits holding its first and its last visible position.
__device__ inline MergeRow merge_row_of(const FwdParams &p, const ReqInfo &r, int i, int h) {
  const int pos = r.ctx - r.q_len + i;
  const int first = (window_lo(pos, p.window) - r.kv_base) / r.split_len;
  const int last = (pos - r.kv_base) / r.split_len;
  MergeRow m;
  m.h = h;
  m.tok = r.q_start + i;
  m.nn = last - first + 1;
  m.base = r.partial_base + ((long long)i * p.num_heads + h) * r.nsplit + first;
  return m;
}

// mend / ord: the merge list's ends and the request order, in global memory
// or (shared = true) as shared-memory copies.
__device__ inline MergeRow merge_row(const FwdParams &p, const long long *mend, const int *ord,
                                     bool shared, long long row) {
  const int S = p.num_seqs, H = p.num_heads;
  const int k = shared ? list_find_shared(mend, S, row) : list_find(mend, S, row);
  const long long local = row - (k ? mend[k - 1] : 0);
  const ReqInfo r = p.req[ord[k]];
  return merge_row_of(p, r, (int)(local / H), (int)(local % H));
}

// Entry `row` of the long-row list: request k's rows i >= i_long (those that
// reach past split kWarpMergeSplits - 1), H heads each.
__device__ inline MergeRow merge_row_long(const FwdParams &p, const long long *lend,
                                          long long row) {
  const int S = p.num_seqs, H = p.num_heads;
  const int k = list_find(lend, S, row);
  const long long local = row - (k ? lend[k - 1] : 0);
  const ReqInfo r = p.req[p.ord[k]];
  const long long i_long =
      max(0ll, (long long)kWarpMergeSplits * r.split_len - (r.ctx - r.q_len - r.kv_base));
  return merge_row_of(p, r, (int)(i_long + local / H), (int)(local % H));
}

template <typename T>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const FwdParams p) {
  __shared__ float s_red[kMergeThreads / 32][128];
  __shared__ float s_wl[kMergeThreads / 32];
  __shared__ float s_m[kMergeThreads / 32];
  __shared__ int s_bad[kMergeThreads / 32];
  const int S = p.num_seqs, H = p.num_heads, D = p.head_dim;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int NW = kMergeThreads / 32;
  pdl_trigger();  // the next call's planner may get its CTA in place
  pdl_wait();
  T *out = reinterpret_cast<T *>(p.out);
  const long long gw = ((long long)blockIdx.x * blockDim.x + tid) >> 5;
  const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;

  if (p.plan->qsl_bad) {
    const size_t n = (size_t)p.num_tokens * H * D;
    for (size_t e = (size_t)blockIdx.x * blockDim.x + tid; e < n; e += (size_t)gridDim.x * blockDim.x)
      store_out<T>(out + e, 0.f);
    return;
  }

  // rows of requests whose metadata failed: zeros
  {
    const long long *zend = p.list_end + (size_t)kListZero * S;
    const long long nz = p.plan->n[kListZero];
    for (long long row = gw; row < nz; row += nw) {
      const int k = list_find(zend, S, row);
      const long long local = row - (k ? zend[k - 1] : 0);
      const ReqInfo r = p.req[p.ord[k]];
      const long long tok = r.q_start + local / H;
      const int h = (int)(local % H);
      for (int d = lane; d < D; d += 32) store_out<T>(out + ((size_t)tok * H + h) * D + d, 0.f);
    }
  }

  const long long nm = p.plan->n[kListMerge];
  if (nm == 0) return;
  // the merge list's per-request ends (searched once per row) and the
  // request order, copied to shared memory for batches up to kMergeCache
  __shared__ long long s_mend[kMergeCache];
  __shared__ int s_ordc[kMergeCache];
  const long long *mend = p.list_end + (size_t)kListMerge * S;
  const int *ord = p.ord;
  const bool mend_shared = S <= kMergeCache;
  if (mend_shared) {
    for (int k = tid; k < S; k += kMergeThreads) {
      s_mend[k] = mend[k];
      s_ordc[k] = ord[k];
    }
    __syncthreads();
    mend = s_mend;
    ord = s_ordc;
  }
  const int dpl = D / 32;  // dims per lane: 2 or 4

  // ---- short rows: one warp each ---------------------------------------------
  for (long long row = gw; row < nm; row += nw) {
    const MergeRow mr = merge_row(p, mend, ord, mend_shared, row);
    if (mr.nn <= 1 || mr.nn > kWarpMergeSplits) continue;
    const float lse = lane < mr.nn ? p.part_lse[mr.base + lane] : -INFINITY;
    int bad = isnan(lse) ? 1 : 0;
    float M = bad ? -INFINITY : lse;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      bad |= __shfl_xor_sync(0xffffffffu, bad, o);
    }
    // a sink joins the max and the denominator once, with no value
    const float sink2 = p.sinks ? __ldg(p.sinks + mr.h) * kLog2eF : -INFINITY;
    M = fmaxf(M, sink2);
    const float w_own = (lane < mr.nn && !bad) ? fast_exp2(lse - M) : 0.f;
    float L = w_own;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    if (p.sinks) L += fast_exp2(sink2 - M);
    // partial rows in groups of 8: the loads of a group are independent
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    const float *src0 = p.part_o + (size_t)mr.base * D + lane * dpl;
    for (int q0 = 0; q0 < mr.nn; q0 += 8) {
      if (dpl == 4) {
        float4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (q0 + u < mr.nn) v[u] = __ldg(reinterpret_cast<const float4 *>(src0 + (size_t)(q0 + u) * D));
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (q0 + u >= mr.nn) break;
          const float w = __shfl_sync(0xffffffffu, w_own, q0 + u);
          acc[0] = fmaf(w, v[u].x, acc[0]);
          acc[1] = fmaf(w, v[u].y, acc[1]);
          acc[2] = fmaf(w, v[u].z, acc[2]);
          acc[3] = fmaf(w, v[u].w, acc[3]);
        }
      } else {
        float2 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (q0 + u < mr.nn) v[u] = __ldg(reinterpret_cast<const float2 *>(src0 + (size_t)(q0 + u) * D));
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (q0 + u >= mr.nn) break;
          const float w = __shfl_sync(0xffffffffu, w_own, q0 + u);
          acc[0] = fmaf(w, v[u].x, acc[0]);
          acc[1] = fmaf(w, v[u].y, acc[1]);
        }
      }
    }
    const float inv = (bad || !(L > 0.f)) ? 0.f : 1.f / L;
    T *dst = out + ((size_t)mr.tok * H + mr.h) * D + lane * dpl;
    for (int x = 0; x < dpl; ++x) store_out<T>(dst + x, acc[x] * inv);
  }

  // ---- long rows: one block each, warps over splits ---------------------------
  const long long nl = p.plan->n[kListMergeLong];
  const long long *lend = p.list_end + (size_t)kListMergeLong * S;
  for (long long row = blockIdx.x; row < nl; row += gridDim.x) {
    const MergeRow mr = merge_row_long(p, lend, row);
    if (mr.nn <= kWarpMergeSplits) continue;  // a windowed row: the warp pass has it
    float M = -INFINITY;
    int bad = 0;
    for (int q = tid; q < mr.nn; q += kMergeThreads) {
      const float v = p.part_lse[mr.base + q];
      if (isnan(v)) bad = 1; else M = fmaxf(M, v);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      bad |= __shfl_xor_sync(0xffffffffu, bad, o);
    }
    if (lane == 0) {
      s_m[warp] = M;
      s_bad[warp] = bad;
    }
    __syncthreads();
    M = s_m[0];
    bad = s_bad[0];
    for (int w = 1; w < NW; ++w) {
      M = fmaxf(M, s_m[w]);
      bad |= s_bad[w];
    }
    // a sink joins the max and the denominator once, with no value
    const float sink2 = p.sinks ? __ldg(p.sinks + mr.h) * kLog2eF : -INFINITY;
    M = fmaxf(M, sink2);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float wl = 0.f;
    if (!bad && M != -INFINITY) {
#pragma unroll 8
      for (int q = warp; q < mr.nn; q += NW) {
        const float w = fast_exp2(p.part_lse[mr.base + q] - M);
        wl += w;
        const float *src = p.part_o + (size_t)(mr.base + q) * D + lane * dpl;
        if (dpl == 4) {
          const float4 v = *reinterpret_cast<const float4 *>(src);
          acc[0] = fmaf(w, v.x, acc[0]);
          acc[1] = fmaf(w, v.y, acc[1]);
          acc[2] = fmaf(w, v.z, acc[2]);
          acc[3] = fmaf(w, v.w, acc[3]);
        } else {
          const float2 v = *reinterpret_cast<const float2 *>(src);
          acc[0] = fmaf(w, v.x, acc[0]);
          acc[1] = fmaf(w, v.y, acc[1]);
        }
      }
    }
    for (int x = 0; x < dpl; ++x) s_red[warp][lane * dpl + x] = acc[x];
    if (lane == 0) s_wl[warp] = wl;
    __syncthreads();
    if (tid < D) {
      float a = 0.f, L = 0.f;
      for (int w = 0; w < NW; ++w) {
        a += s_red[w][tid];
        L += s_wl[w];
      }
      if (p.sinks) L += fast_exp2(sink2 - M);
      const float v = (bad || !(L > 0.f)) ? 0.f : a / L;
      store_out<T>(out + ((size_t)mr.tok * H + mr.h) * D + tid, v);
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// debug gather: dense[s][j][:] = cache row (block_table[s][j / bs], j % bs)
// ---------------------------------------------------------------------------

__global__ void gather_kernel(const uint8_t *cache, const int32_t *bt, const int32_t *seq_lens,
                              int num_seqs, int mbps, int num_blocks, int bs, int row_bytes,
                              int max_seq_len, uint8_t *dense, unsigned int *status) {
  const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
  const int lane = threadIdx.x & 31;
  const long long n = (long long)num_seqs * max_seq_len;
  for (long long w = gw; w < n; w += nw) {
    const int s = (int)(w / max_seq_len), j = (int)(w % max_seq_len);
    if (j >= seq_lens[s]) continue;
    const int lp = j / bs;
    const int page = lp < mbps ? bt[(size_t)s * mbps + lp] : -1;
    if (page < 0 || page >= num_blocks) {
      if (lane == 0) atomicOr(status, PA_DEV_BAD_BLOCK);
      continue;
    }
    const uint8_t *src = cache + ((size_t)page * bs + (j % bs)) * row_bytes;
    uint8_t *dst = dense + ((size_t)s * max_seq_len + j) * row_bytes;
    if ((row_bytes & 15) == 0) {
      for (int b = lane * 16; b < row_bytes; b += 32 * 16)
        *reinterpret_cast<uint4 *>(dst + b) = *reinterpret_cast<const uint4 *>(src + b);
    } else {
      for (int b = lane * 2; b < row_bytes; b += 64)
        *reinterpret_cast<uint16_t *>(dst + b) = *reinterpret_cast<const uint16_t *>(src + b);
    }
  }
}

// ---------------------------------------------------------------------------
// debug wait: one bounded mbarrier wait that nothing ever completes
// ---------------------------------------------------------------------------

// One warp: lane 0 initialises an mbarrier expecting one arrival that never
// comes and waits on it through the kernels' bounded wait; the wait gives up
// after limit_ns, sets PA_DEV_TIMEOUT and the kernel returns.  A second wait
// of the same thread returns at once (the `dead` latch every kernel relies
// on to end after a timeout).  No copy is issued, so nothing is in flight
// when the kernel ends.  *done receives 2 when the first wait ran out and the
// second returned.
__global__ void wait_timeout_kernel(uint64_t limit_ns, unsigned int *status, int *done) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_mbar_init();
  bool dead = false;
  mbar_wait_limit(&bar, 0, dead, status, limit_ns);  // runs out: dead
  const int timed_out = dead ? 1 : 0;
  mbar_wait_limit(&bar, 0, dead, status, limit_ns);  // returns at once
  *done = timed_out + 1;
}

// ---------------------------------------------------------------------------
// host state
// ---------------------------------------------------------------------------

struct DeviceState {
  bool init = false;
  int num_sms = 0;
  unsigned int *status = nullptr;
  void *ws = nullptr;
  size_t ws_bytes = 0;
  // decode-only batches: [0] item counter, [1] blocks done taking items,
  // then one split count per (request, kv head); all zero between calls
  unsigned long long *fast_ctr = nullptr;
  size_t fast_groups = 0;
  // the row kernel's K / V tensor maps of the last decode-only call (a
  // serving loop calls with the same caches: encoding them is host time)
  bool maps_valid = false;
  const void *maps_k = nullptr, *maps_v = nullptr;
  int maps_key[6] = {0, 0, 0, 0, 0, 0};
  CUtensorMap map_k, map_v;
};

std::mutex g_mu;
DeviceState g_dev[64];

}  // namespace

bool stream_capturing(cudaStream_t stream) {
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &st) != cudaSuccess) return false;
  return st != cudaStreamCaptureStatusNone;
}

pa_status current_device_for(cudaStream_t stream, int *dev) {
  if (cudaGetDevice(dev) != cudaSuccess || *dev < 0 || *dev >= 64) {
    cudaGetLastError();
    return PA_ERR_CUDA;
  }
  // A stream that is capturing is not queried (the query would invalidate a
  // global-mode capture); the check applies to calls made outside capture.
  if (stream_capturing(stream)) return PA_OK;
  int sdev = *dev;
  if (cudaStreamGetDevice(stream, &sdev) != cudaSuccess) {
    cudaGetLastError();
    return PA_ERR_INVALID_ARG;
  }
  return sdev == *dev ? PA_OK : PA_ERR_INVALID_ARG;
}

namespace {

// Device state of the current device; initialises it outside capture.
pa_status device_state(cudaStream_t stream, DeviceState **out) {
  int dev = 0;
  const pa_status ds = current_device_for(stream, &dev);
  if (ds != PA_OK) return ds;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState &d = g_dev[dev];
  if (!d.init) {
    if (stream_capturing(stream)) return PA_ERR_WORKSPACE;
    if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return PA_ERR_CUDA;
    }
    if (cudaMalloc(&d.status, 256) != cudaSuccess) {
      cudaGetLastError();
      return PA_ERR_CUDA;
    }
    if (cudaMemset(d.status, 0, 256) != cudaSuccess) return PA_ERR_CUDA;
    d.init = true;
  }
  *out = &d;
  return PA_OK;
}

pa_status ensure_workspace(DeviceState *d, size_t bytes, cudaStream_t stream) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (d->ws_bytes >= bytes) return PA_OK;
  if (stream_capturing(stream)) return PA_ERR_WORKSPACE;
  if (d->ws) {
    cudaFree(d->ws);  // synchronises the device: no call still uses the old buffer
    d->ws = nullptr;
    d->ws_bytes = 0;
  }
  size_t want = bytes + bytes / 4;
  if (cudaMalloc(&d->ws, want) != cudaSuccess) {
    cudaGetLastError();
    if (cudaMalloc(&d->ws, bytes) != cudaSuccess) {
      cudaGetLastError();
      return PA_ERR_CUDA;
    }
    want = bytes;
  }
  d->ws_bytes = want;
  return PA_OK;
}

// The decode-only path's counters for `groups` row groups, zeroed when
// (re)allocated; they return to zero at the end of every call.
pa_status ensure_fast_counters(DeviceState *d, size_t groups, cudaStream_t stream) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (d->fast_ctr && d->fast_groups >= groups) return PA_OK;
  if (stream_capturing(stream)) return PA_ERR_WORKSPACE;
  if (d->fast_ctr) {
    cudaFree(d->fast_ctr);  // synchronises the device: no call still uses it
    d->fast_ctr = nullptr;
    d->fast_groups = 0;
  }
  const size_t want = groups + groups / 4 + 64;
  const size_t bytes = 2 * sizeof(unsigned long long) + want * sizeof(unsigned int);
  if (cudaMalloc(&d->fast_ctr, bytes) != cudaSuccess) {
    cudaGetLastError();
    d->fast_ctr = nullptr;
    return PA_ERR_CUDA;
  }
  if (cudaMemset(d->fast_ctr, 0, bytes) != cudaSuccess) return PA_ERR_CUDA;
  d->fast_groups = want;
  return PA_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct FwdLayout {
  size_t plan, req, ord, list_end, part_o, part_lse, total;
  long long part_cap;
};

long long ceil_div_h(long long a, long long b) { return (a + b - 1) / b; }

// Upper bound on the split partial rows pa_forward may need; mirrors the
// planner's split rules using only host-known extents.
long long partial_capacity(int num_seqs, int num_tokens, int num_heads, int max_seq_len,
                           int kvs, bool tile_ok) {
  const long long msl = max_seq_len > 0 ? max_seq_len : 1;
  const long long kvs_or_inf = kvs > 0 ? kvs : (1ll << 40);
  // decode rows: at most min(S, T) requests with one row each
  const long long l_dec = kRowMinSplit < kvs_or_inf ? kRowMinSplit : kvs_or_inf;
  const long long n_dec = ceil_div_h(msl, l_dec);
  const long long dec_rows = (long long)(num_seqs < num_tokens ? num_seqs : num_tokens);
  long long cap = n_dec > 1 ? dec_rows * num_heads * n_dec : 0;
  long long n_other;
  if (tile_ok) {
    // tile rows: up to twice the splits kv_split_tokens needs (equal splits,
    // doubled when the tile work is coarse)
    n_other = kvs > 0 ? 2 * ceil_div_h(msl, kvs) : 1;
  } else {
    long long lr = ceil_div_h(ceil_div_h(msl, 4), 16) * 16;
    if (lr < kRowMinSplit) lr = kRowMinSplit;
    if (lr > kRowMaxSplit) lr = kRowMaxSplit;
    if (kvs_or_inf < lr) lr = kvs_or_inf;
    n_other = ceil_div_h(msl, lr);
  }
  if (n_other > 1) cap += (long long)num_tokens * num_heads * n_other;
  return cap;
}

FwdLayout fwd_layout(int num_seqs, int num_tokens, int num_heads, int head_dim,
                     int max_seq_len, int kvs, bool tile_ok) {
  FwdLayout l{};
  const size_t S = num_seqs > 0 ? num_seqs : 1;
  size_t off = 0;
  l.plan = off;
  off = align256(off + sizeof(PlanHeader));
  l.req = off;
  off = align256(off + S * sizeof(ReqInfo));
  l.ord = off;
  off = align256(off + S * sizeof(int));
  l.list_end = off;
  off = align256(off + S * kNumLists * sizeof(long long));
  l.part_cap = partial_capacity(num_seqs, num_tokens, num_heads, max_seq_len, kvs, tile_ok);
  l.part_o = off;
  off = align256(off + (size_t)l.part_cap * head_dim * sizeof(float));
  l.part_lse = off;
  off = align256(off + (size_t)l.part_cap * sizeof(float));
  l.total = off;
  return l;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// Tensor map over a paged cache with coordinates (dim, kv head, slot, page)
// and a box of {box_dim0, 1, box_slots, 1}: one (page, kv head) run of slots
// per copy.  The layout only changes the strides: [num_blocks, block_size,
// heads, dim] (PA_KV_NHD) or [num_blocks, heads, block_size, dim] (PA_KV_HND).
bool encode_cache_map(CUtensorMap *map, const void *base, int dtype, int kv_layout,
                      int num_blocks, int block_size, int heads, int dim, int box_dim0,
                      int box_slots, CUtensorMapSwizzle swz) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const size_t es = dtype == PA_F32 ? 4 : 2;
  const bool hnd = kv_layout == PA_KV_HND;
  cuuint64_t dims[4] = {(cuuint64_t)dim, (cuuint64_t)heads, (cuuint64_t)block_size,
                        (cuuint64_t)num_blocks};
  const cuuint64_t row = dim * es;  // one (slot, head) row
  cuuint64_t strides[3] = {hnd ? (cuuint64_t)block_size * row : row,
                           hnd ? row : (cuuint64_t)heads * row,
                           (cuuint64_t)block_size * heads * row};
  cuuint32_t box[4] = {(cuuint32_t)box_dim0, 1, (cuuint32_t)box_slots, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType t =
      dtype == PA_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  return fn(map, t, 4, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

bool group_ok(int g) { return g == 1 || g == 2 || g == 4 || g == 8 || g == 16; }

// Resident CTAs per SM of the row kernel, cached per (device, dtype, dim, group).
int row_ctas_per_sm_cached(int dtype, int head_dim, int group) {
  static std::mutex mu;
  static int cache[64][2][2][5];
  static bool have[64][2][2][5];
  int dev = 0;
  cudaGetDevice(&dev);
  const int a = dtype == PA_BF16 ? 1 : 0, b = head_dim == 128 ? 1 : 0;
  const int c = group == 1 ? 0 : group == 2 ? 1 : group == 4 ? 2 : group == 8 ? 3 : 4;
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 0 || dev >= 64) return 1;
  if (!have[dev][a][b][c]) {
    cache[dev][a][b][c] = row_mma_supported(dtype, head_dim, group)
                              ? row_mma_ctas_per_sm(head_dim, group)
                              : row_kernel_ctas_per_sm(dtype, head_dim, group);
    have[dev][a][b][c] = true;
  }
  return cache[dev][a][b][c] > 0 ? cache[dev][a][b][c] : 1;
}

bool tile_path_ok(int dtype, int head_dim, int group) {
  return tile_kernel_supported(dtype, head_dim, group);
}

// Decode-only batches (the caller declares max_query_len == 1): one row-kernel
// launch, no planner.  The kernel sizes the splits from seq_lens itself; the
// host only bounds the splits per row (so the partial rows fit a workspace
// sized from max_seq_len) at fast_nsmax <= 64, the most a row's in-kernel
// merge takes.
struct FastPlan {
  int nsmax = 0;
  long long part_rows = 0;
  size_t part_o = 0, part_lse = 0, ws_bytes = 0;
};

bool fast_decode_plan(const FwdCall &c, int num_sms, FastPlan *f) {
  (void)num_sms;
  if (c.max_query_len != 1 || c.dtype != PA_BF16 || c.all_tile || c.num_seqs <= 0 ||
      c.num_tokens != c.num_seqs || c.num_seqs > kFastMaxSeqs)
    return false;
  const int group = c.num_heads / c.num_kv_heads;
  if (!row_mma_supported(c.dtype, c.head_dim, group)) return false;
  const long long msl = c.max_seq_len > 0 ? c.max_seq_len : 1;
  if (msl > 64ll * kRowMaxSplit) return false;
  // splits are at least kFastMinSplit long (or kv_split_tokens, if shorter)
  long long nsmax = ceil_div_h(msl, kFastMinSplit);
  if (c.kv_split_tokens > 0) nsmax = std::max(nsmax, ceil_div_h(msl, c.kv_split_tokens));
  if (nsmax > 64) {
    if (c.kv_split_tokens > 0) return false;  // the requested splits are too short
    nsmax = 64;
  }
  f->nsmax = (int)nsmax;
  f->part_rows = (long long)c.num_seqs * c.num_heads * nsmax;
  f->part_o = 0;
  f->part_lse = align256((size_t)f->part_rows * c.head_dim * sizeof(float));
  f->ws_bytes = f->part_lse + align256((size_t)f->part_rows * sizeof(float));
  return true;
}

// The row kernel's K / V tensor maps: bf16 boxes of 16 slots x both 64-dim
// halves of one KV head, dims {64 dims, slots, halves, kv heads, pages} (the
// slot stride is larger than the half stride; TMA takes strides in any
// order).  In the HND layout a box is one contiguous run of 16 x head_dim.
bool encode_row_maps(const FwdCall &c, CUtensorMap *tm_k, CUtensorMap *tm_v) {
  const unsigned long long es = 2, row = (unsigned long long)c.head_dim * es;
  const bool hnd = c.kv_layout == PA_KV_HND;
  const unsigned long long dims[5] = {64, (unsigned long long)c.block_size,
                                      (unsigned long long)(c.head_dim / 64),
                                      (unsigned long long)c.num_kv_heads,
                                      (unsigned long long)c.num_blocks};
  const unsigned long long strides[4] = {
      hnd ? row : (unsigned long long)c.num_kv_heads * row, 64 * es,
      hnd ? (unsigned long long)c.block_size * row : row,
      (unsigned long long)c.block_size * c.num_kv_heads * row};
  const unsigned int box[5] = {64, 16, (unsigned int)(c.head_dim / 64), 1, 1};
  return (!tm_k || encode_tiled(tm_k, c.k_cache, c.dtype, 5, dims, strides, box, true)) &&
         encode_tiled(tm_v, c.v_cache, c.dtype, 5, dims, strides, box, true);
}

pa_status fast_decode_launch(const FwdCall &c, const FastPlan &f, DeviceState *d,
                             cudaStream_t st) {
  void *workspace = d->ws;
  unsigned int *status = d->status;
  unsigned long long *fast_ctr = d->fast_ctr;
  const int num_sms = d->num_sms;
  const int group = c.num_heads / c.num_kv_heads;
  uint8_t *ws = reinterpret_cast<uint8_t *>(workspace);
  FwdParams p{};
  p.q = c.q;
  p.out = c.out;
  p.block_table = c.block_table;
  p.seq_lens = c.seq_lens;
  p.qsl = c.qsl;
  p.num_seqs = c.num_seqs;
  p.num_tokens = c.num_tokens;
  p.num_heads = c.num_heads;
  p.num_kv_heads = c.num_kv_heads;
  p.head_dim = c.head_dim;
  p.block_size = c.block_size;
  p.max_blocks_per_seq = c.max_blocks_per_seq;
  p.num_blocks = c.num_blocks;
  p.max_seq_len = c.max_seq_len;
  p.kv_split_tokens = c.kv_split_tokens;
  p.scale = c.scale;
  p.scale_log2 = c.scale * kLog2e;
  p.dtype = c.dtype;
  p.part_o = reinterpret_cast<float *>(ws + f.part_o);
  p.part_lse = reinterpret_cast<float *>(ws + f.part_lse);
  p.part_cap = f.part_rows;
  p.status = status;
  p.sinks = c.sinks;
  p.window = c.sliding_window;
  p.alibi = c.alibi_slopes;
  p.alibi_sqrt = c.alibi_sqrt;
  p.head_dim_qk = c.head_dim;
  p.fast = 1;
  p.fast_nsmax = f.nsmax;
  p.fast_work = fast_ctr;
  p.fast_cnt = reinterpret_cast<unsigned int *>(fast_ctr + 2);
  CUtensorMap tm_k, tm_v;
  {
    const int key[6] = {c.dtype, c.kv_layout, c.num_blocks, c.block_size, c.num_kv_heads,
                        c.head_dim};
    std::lock_guard<std::mutex> lock(g_mu);
    if (d->maps_valid && d->maps_k == c.k_cache && d->maps_v == c.v_cache &&
        std::equal(key, key + 6, d->maps_key)) {
      tm_k = d->map_k;
      tm_v = d->map_v;
    } else {
      if (!encode_row_maps(c, &tm_k, &tm_v)) return PA_ERR_CUDA;
      d->map_k = tm_k;
      d->map_v = tm_v;
      d->maps_k = c.k_cache;
      d->maps_v = c.v_cache;
      std::copy(key, key + 6, d->maps_key);
      d->maps_valid = true;
    }
  }
  const int row_ctas = row_ctas_per_sm_cached(c.dtype, c.head_dim, group) * num_sms;
  p.row_ctas = row_ctas;
  const int slot = prof_begin(PA_K_ROW, st);
  const cudaError_t err = launch_row_mma_kernel(p, tm_k, tm_v, row_ctas, st);
  prof_end(slot, st);
  return err == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace

pa_status fwd_check(const FwdCall &c) {
  if (c.num_seqs < 0 || c.num_tokens < 0 || c.max_seq_len < 0 || c.kv_split_tokens < 0 ||
      c.num_heads <= 0 || c.num_kv_heads <= 0 || c.head_dim <= 0 || c.block_size <= 0)
    return PA_ERR_INVALID_ARG;
  if (c.dtype != PA_F32 && c.dtype != PA_BF16) return PA_ERR_INVALID_ARG;
  if (c.num_heads % c.num_kv_heads != 0) return PA_ERR_INVALID_ARG;
  const int group = c.num_heads / c.num_kv_heads;
  if (!group_ok(group) || (c.head_dim != 64 && c.head_dim != 128) || c.block_size % 16 != 0 ||
      c.block_size > 256 || c.kv_split_tokens % 16 != 0)
    return PA_ERR_UNSUPPORTED;
  if (c.num_tokens == 0) return PA_OK;  // no output rows
  if (!c.q || !c.out || !c.qsl || (c.num_seqs > 0 && (!c.seq_lens || !c.block_table)))
    return PA_ERR_INVALID_ARG;
  if (c.num_seqs > 0 &&
      (!c.k_cache || !c.v_cache || c.num_blocks <= 0 || c.max_blocks_per_seq <= 0))
    return PA_ERR_INVALID_ARG;
  if (!aligned16(c.q) || !aligned16(c.out) ||
      (c.num_seqs > 0 && (!aligned16(c.k_cache) || !aligned16(c.v_cache))))
    return PA_ERR_INVALID_ARG;
  if ((long long)c.num_tokens * c.num_heads * c.head_dim > (1ll << 40)) return PA_ERR_UNSUPPORTED;
  return PA_OK;
}

size_t fwd_workspace_bytes(const FwdCall &c) {
  const bool tile_ok = tile_path_ok(c.dtype, c.head_dim, c.num_heads / c.num_kv_heads);
  return fwd_layout(c.num_seqs, c.num_tokens, c.num_heads, c.head_dim, c.max_seq_len,
                    c.kv_split_tokens, tile_ok)
      .total;
}

pa_status fwd_launch(const FwdCall &c, void *workspace, unsigned int *status, int num_sms,
                     cudaStream_t st, bool timed) {
  const int group = c.num_heads / c.num_kv_heads;
  const int dqk = c.head_dim_qk > 0 ? c.head_dim_qk : c.head_dim;
  const bool tile_ok = c.all_tile || tile_path_ok(c.dtype, c.head_dim, group);
  const FwdLayout lay = fwd_layout(c.num_seqs, c.num_tokens, c.num_heads, c.head_dim,
                                   c.max_seq_len, c.kv_split_tokens, tile_ok);
  const int row_ctas = row_ctas_per_sm_cached(c.dtype, c.head_dim, group) * num_sms;
  uint8_t *ws = reinterpret_cast<uint8_t *>(workspace);
  FwdParams p{};
  p.q = c.q;
  p.out = c.out;
  p.block_table = c.block_table;
  p.seq_lens = c.seq_lens;
  p.qsl = c.qsl;
  p.num_seqs = c.num_seqs;
  p.num_tokens = c.num_tokens;
  p.num_heads = c.num_heads;
  p.num_kv_heads = c.num_kv_heads;
  p.head_dim = c.head_dim;
  p.block_size = c.block_size;
  p.max_blocks_per_seq = c.max_blocks_per_seq;
  p.num_blocks = c.num_blocks;
  p.max_seq_len = c.max_seq_len;
  p.kv_split_tokens = c.kv_split_tokens;
  p.scale = c.scale;
  p.scale_log2 = c.scale * kLog2e;
  p.tile_ok = tile_ok ? 1 : 0;
  p.row_ctas = row_ctas;
  p.tile_ctas = 2 * num_sms;  // the tile kernel's grid
  p.dtype = c.dtype;
  p.plan = reinterpret_cast<PlanHeader *>(ws + lay.plan);
  p.req = reinterpret_cast<ReqInfo *>(ws + lay.req);
  p.ord = reinterpret_cast<int *>(ws + lay.ord);
  p.list_end = reinterpret_cast<long long *>(ws + lay.list_end);
  p.part_o = reinterpret_cast<float *>(ws + lay.part_o);
  p.part_lse = reinterpret_cast<float *>(ws + lay.part_lse);
  p.part_cap = lay.part_cap;
  p.status = status;
  p.sinks = c.sinks;
  p.window = c.sliding_window;
  p.alibi = c.alibi_slopes;
  p.alibi_sqrt = c.alibi_sqrt;
  p.head_dim_qk = dqk;
  p.all_tile = c.all_tile ? 1 : 0;
  p.max_qlen = c.max_query_len;

  int slot = timed ? prof_begin(PA_K_PLAN, st) : -1;
  // One thread per request, whole warps, at most kPlanThreads: small batches
  // get a small block and cheap barriers.  (The shared-memory copy of the
  // metadata needs a thread per request whenever S <= kPlanCache.)
  int plan_threads = ((c.num_seqs > 0 ? c.num_seqs : 1) + 31) / 32 * 32;
  if (plan_threads > kPlanThreads) plan_threads = kPlanThreads;
  const cudaError_t plan_err =
      launch_dependent(plan_kernel, dim3(1), dim3(plan_threads), 0, st, p);
  prof_end(slot, st);
  if (plan_err != cudaSuccess) return PA_ERR_CUDA;

  if (c.num_seqs > 0) {
    const bool mma_rows = row_mma_supported(c.dtype, c.head_dim, group);
    // bf16 K/V boxes of 16 slots x both 64-dim halves of one KV head:
    // dims {64 dims, slots, halves, kv heads, pages} (the slot stride is
    // larger than the half stride; TMA takes strides in any order).  The row
    // kernel reads K and V through them, the tile kernel V.  In the HND
    // layout a box is one contiguous run of 16 x head_dim elements.
    CUtensorMap tm_kr, tm_vr;
    // (all-tile calls have no row items: their K rows may be wider than V's)
    if (c.dtype == PA_BF16 && !encode_row_maps(c, c.all_tile ? nullptr : &tm_kr, &tm_vr))
      return PA_ERR_CUDA;
    // The tile kernel's K: one 64-element (128-byte) swizzled box per half
    // and 16 slots, so the S product sees a uniform row stride.
    // When every 64-position tile lies in one page (block_size a multiple of
    // 64; tiles start at multiples of 64: no window, splits of a multiple of
    // 64), the tile kernel loads a whole tile's K chunk or V rows as one box.
    const bool page_boxes = tile_ok && c.dtype == PA_BF16 && c.block_size % 64 == 0 &&
                            c.sliding_window == 0 && c.kv_split_tokens % 64 == 0;
    p.tile_page_boxes = page_boxes ? 1 : 0;
    // Split keys (MLA prefill): the key tensor holds dqk - 64 columns per
    // (position, head) and the last 64 come from one row per position.
    CUtensorMap tm_kt, tm_vt, tm_krope;
    p.k_rope_split = c.k_rope ? 1 : 0;
    if (tile_ok && !encode_cache_map(&tm_kt, c.k_cache, c.dtype, c.kv_layout, c.num_blocks,
                                     c.block_size, c.num_kv_heads, c.k_rope ? dqk - 64 : dqk, 64,
                                     page_boxes ? 64 : 16, CU_TENSOR_MAP_SWIZZLE_128B))
      return PA_ERR_CUDA;
    if (c.k_rope && !encode_cache_map(&tm_krope, c.k_rope, c.dtype, PA_KV_NHD, c.num_blocks,
                                      c.block_size, 1, 64, 64, page_boxes ? 64 : 16,
                                      CU_TENSOR_MAP_SWIZZLE_128B))
      return PA_ERR_CUDA;
    if (!c.k_rope) tm_krope = tm_kt;
    if (page_boxes) {
      const unsigned long long es = 2, row = (unsigned long long)c.head_dim * es;
      const bool hnd = c.kv_layout == PA_KV_HND;
      const unsigned long long dims[5] = {64, (unsigned long long)c.block_size,
                                          (unsigned long long)(c.head_dim / 64),
                                          (unsigned long long)c.num_kv_heads,
                                          (unsigned long long)c.num_blocks};
      const unsigned long long strides[4] = {
          hnd ? row : (unsigned long long)c.num_kv_heads * row, 64 * es,
          hnd ? (unsigned long long)c.block_size * row : row,
          (unsigned long long)c.block_size * c.num_kv_heads * row};
      const unsigned int box[5] = {64, 64, (unsigned int)(c.head_dim / 64), 1, 1};
      if (!encode_tiled(&tm_vt, c.v_cache, c.dtype, 5, dims, strides, box, true))
        return PA_ERR_CUDA;
    }
    cudaError_t row_err = cudaSuccess;
    slot = timed ? prof_begin(PA_K_ROW, st) : -1;
    if (c.all_tile) {
      // no row items: the row kernel is not launched
    } else if (mma_rows) {
      row_err = launch_row_mma_kernel(p, tm_kr, tm_vr, row_ctas, st);
    } else {
      // fp32: whole rows of head_dim elements, no swizzle (CUDA-core kernel)
      CUtensorMap tm_k, tm_v;
      if (!encode_cache_map(&tm_k, c.k_cache, c.dtype, c.kv_layout, c.num_blocks, c.block_size,
                            c.num_kv_heads, c.head_dim, c.head_dim, 16,
                            CU_TENSOR_MAP_SWIZZLE_NONE) ||
          !encode_cache_map(&tm_v, c.v_cache, c.dtype, c.kv_layout, c.num_blocks, c.block_size,
                            c.num_kv_heads, c.head_dim, c.head_dim, 16,
                            CU_TENSOR_MAP_SWIZZLE_NONE))
        return PA_ERR_CUDA;
      row_err = launch_row_kernel(p, tm_k, tm_v, row_ctas, st);
    }
    prof_end(slot, st);
    if (row_err != cudaSuccess) return PA_ERR_CUDA;
    // A decode-only batch (the caller's bound max_query_len == 1; a request
    // above it is zeroed as bad metadata) has no tile items: no launch.
    if (tile_ok && c.max_query_len != 1) {
      // Q as [tokens, heads, dim] with 64-element (128-byte) swizzled boxes of
      // G heads x (128 / G) tokens.
      CUtensorMap tm_q;
      EncodeTiledFn fn = encode_fn();
      cuuint64_t qd[3] = {(cuuint64_t)dqk, (cuuint64_t)c.num_heads, (cuuint64_t)c.num_tokens};
      cuuint64_t qs[2] = {(cuuint64_t)dqk * 2, (cuuint64_t)c.num_heads * dqk * 2};
      cuuint32_t qb[3] = {64, (cuuint32_t)group, (cuuint32_t)(kTileRows / group)};
      cuuint32_t qe[3] = {1, 1, 1};
      if (!fn ||
          fn(&tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(c.q), qd, qs, qb, qe,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return PA_ERR_CUDA;
      slot = timed ? prof_begin(PA_K_TILE, st) : -1;
      const cudaError_t tile_err =
          launch_tile_kernel(p, tm_q, tm_kt, page_boxes ? tm_vt : tm_vr, tm_krope, num_sms, st);
      prof_end(slot, st);
      if (tile_err != cudaSuccess) return PA_ERR_CUDA;
    }
  }
  slot = timed ? prof_begin(PA_K_MERGE, st) : -1;
  const cudaError_t merge_err =
      c.dtype == PA_BF16
          ? launch_dependent(merge_kernel<__nv_bfloat16>, dim3(num_sms * 4), dim3(kMergeThreads),
                             0, st, p)
          : launch_dependent(merge_kernel<float>, dim3(num_sms * 4), dim3(kMergeThreads), 0, st,
                             p);
  prof_end(slot, st);
  if (merge_err != cudaSuccess) return PA_ERR_CUDA;
  return PA_OK;
}

pa_status device_resources(cudaStream_t stream, size_t ws_bytes, void **ws,
                           unsigned int **status, int *num_sms) {
  DeviceState *d = nullptr;
  pa_status s = device_state(stream, &d);
  if (s != PA_OK) return s;
  s = ensure_workspace(d, ws_bytes, stream);
  if (s != PA_OK) return s;
  *ws = d->ws;
  *status = d->status;
  *num_sms = d->num_sms;
  return PA_OK;
}

bool encode_tiled(CUtensorMap *map, const void *base, int dtype, int rank,
                  const unsigned long long *dims, const unsigned long long *strides,
                  const unsigned int *box, bool swizzle128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || rank < 1 || rank > 5) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t b[5], e[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    e[i] = 1;
  }
  for (int i = 0; i + 1 < rank; ++i) st[i] = strides[i];
  const CUtensorMapDataType t =
      dtype == PA_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  return fn(map, t, rank, const_cast<void *>(base), d, st, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace pa

using namespace pa;

extern "C" {

const char *pa_status_string(pa_status status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case PA_ERR_WORKSPACE: return "workspace too small during stream capture";
    case PA_ERR_CUDA: return "CUDA error";
    case PA_ERR_SCRATCH_LIMIT: return "call exceeds the static scratch region";
  }
  return "unknown status";
}

int pa_num_sms(void) {
  DeviceState *d = nullptr;
  if (device_state(nullptr, &d) != PA_OK) return 0;
  return d->num_sms;
}

size_t pa_forward_workspace_bytes(pa_dtype dtype, int num_seqs, int num_tokens, int num_heads,
                                  int num_kv_heads, int head_dim, int max_seq_len,
                                  int kv_split_tokens) {
  if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads) return 0;
  const bool tile_ok = tile_path_ok(dtype, head_dim, num_heads / num_kv_heads);
  return fwd_layout(num_seqs, num_tokens, num_heads, head_dim, max_seq_len, kv_split_tokens,
                    tile_ok)
      .total;
}

pa_status pa_reserve(size_t bytes) {
  DeviceState *d = nullptr;
  pa_status st = device_state(nullptr, &d);
  if (st != PA_OK) return st;
  return ensure_workspace(d, bytes, nullptr);
}

pa_status pa_get_device_status(void *stream, uint32_t *host_flags) {
  if (!host_flags) return PA_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  DeviceState *d = nullptr;
  pa_status s = device_state(st, &d);
  if (s != PA_OK) return s;
  if (cudaStreamSynchronize(st) != cudaSuccess) return PA_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpy(&v, d->status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
    return PA_ERR_CUDA;
  if (cudaMemset(d->status, 0, sizeof(v)) != cudaSuccess) return PA_ERR_CUDA;
  *host_flags = v;
  return PA_OK;
}

pa_status pa_forward(const void *q, const void *k_cache, const void *v_cache,
                     const int32_t *block_table, const int32_t *seq_lens,
                     const int32_t *query_start_loc, int num_heads, int num_kv_heads,
                     int head_dim, int block_size, float scale, void *out, void *stream,
                     pa_dtype dtype, int num_seqs, int num_tokens, int max_blocks_per_seq,
                     int num_blocks, int max_seq_len, int kv_split_tokens) {
  return pa_forward_ex(q, k_cache, v_cache, block_table, seq_lens, query_start_loc, num_heads,
                       num_kv_heads, head_dim, block_size, scale, out, stream, dtype, num_seqs,
                       num_tokens, max_blocks_per_seq, num_blocks, max_seq_len, kv_split_tokens,
                       nullptr);
}

pa_status pa_forward_ex(const void *q, const void *k_cache, const void *v_cache,
                        const int32_t *block_table, const int32_t *seq_lens,
                        const int32_t *query_start_loc, int num_heads, int num_kv_heads,
                        int head_dim, int block_size, float scale, void *out, void *stream,
                        pa_dtype dtype, int num_seqs, int num_tokens, int max_blocks_per_seq,
                        int num_blocks, int max_seq_len, int kv_split_tokens,
                        const pa_forward_options *options) {
  FwdCall c{q, k_cache, v_cache, block_table, seq_lens, query_start_loc, num_heads,
            num_kv_heads, head_dim, block_size, scale, out, dtype, num_seqs, num_tokens,
            max_blocks_per_seq, num_blocks, max_seq_len, kv_split_tokens};
  if (options) {
    if (options->sinks && (reinterpret_cast<uintptr_t>(options->sinks) & 3))
      return PA_ERR_INVALID_ARG;
    if (options->kv_layout != PA_KV_NHD && options->kv_layout != PA_KV_HND)
      return PA_ERR_INVALID_ARG;
    if (options->sliding_window < 0 || (options->alibi_sqrt != 0 && options->alibi_sqrt != 1))
      return PA_ERR_INVALID_ARG;
    if (options->alibi_slopes && (reinterpret_cast<uintptr_t>(options->alibi_slopes) & 3))
      return PA_ERR_INVALID_ARG;
    c.sinks = options->sinks;
    c.kv_layout = options->kv_layout;
    c.sliding_window = options->sliding_window;
    c.alibi_slopes = options->alibi_slopes;
    c.alibi_sqrt = options->alibi_sqrt;
    if (options->max_query_len < 0) return PA_ERR_INVALID_ARG;
    c.max_query_len = options->max_query_len;
  }
  pa_status s = fwd_check(c);
  if (s != PA_OK || num_tokens == 0) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  DeviceState *d = nullptr;
  s = device_state(st, &d);
  if (s != PA_OK) return s;
  FastPlan fp;
  if (fast_decode_plan(c, d->num_sms, &fp)) {
    s = ensure_workspace(d, fp.ws_bytes, st);
    if (s != PA_OK) return s;
    s = ensure_fast_counters(d, (size_t)c.num_seqs * c.num_kv_heads, st);
    if (s != PA_OK) return s;
    return fast_decode_launch(c, fp, d, st);
  }
  s = ensure_workspace(d, fwd_workspace_bytes(c), st);
  if (s != PA_OK) return s;
  return fwd_launch(c, d->ws, d->status, d->num_sms, st, true);
}

pa_status pa_debug_gather(const void *k_cache, const int32_t *block_table,
                          const int32_t *seq_lens, int num_seqs, int max_blocks_per_seq,
                          int num_blocks, int block_size, int row_elems, int elem_bytes,
                          int max_seq_len, void *dense_out, void *stream) {
  if (num_seqs < 0 || max_seq_len < 0 || row_elems <= 0 || block_size <= 0 ||
      (elem_bytes != 2 && elem_bytes != 4))
    return PA_ERR_INVALID_ARG;
  if (num_seqs == 0 || max_seq_len == 0) return PA_OK;
  if (!k_cache || !block_table || !seq_lens || !dense_out || num_blocks <= 0 ||
      max_blocks_per_seq <= 0)
    return PA_ERR_INVALID_ARG;
  const int row_bytes = row_elems * elem_bytes;
  if ((row_bytes & 15) == 0 && (!aligned16(k_cache) || !aligned16(dense_out)))
    return PA_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  DeviceState *d = nullptr;
  pa_status s = device_state(st, &d);
  if (s != PA_OK) return s;
  const int slot = prof_begin(PA_K_GATHER, st);
  gather_kernel<<<d->num_sms * 8, 256, 0, st>>>(
      reinterpret_cast<const uint8_t *>(k_cache), block_table, seq_lens, num_seqs,
      max_blocks_per_seq, num_blocks, block_size, row_bytes, max_seq_len,
      reinterpret_cast<uint8_t *>(dense_out), d->status);
  prof_end(slot, st);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_debug_wait_timeout(uint64_t limit_ns, int *done, void *stream) {
  if (!done || limit_ns == 0 || limit_ns > kWaitLimitNs) return PA_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  DeviceState *d = nullptr;
  pa_status s = device_state(st, &d);
  if (s != PA_OK) return s;
  wait_timeout_kernel<<<1, 32, 0, st>>>(limit_ns, d->status, done);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // extern "C"
