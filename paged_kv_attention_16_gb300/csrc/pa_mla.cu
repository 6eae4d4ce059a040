// pa_mla.cu -- absorbed multi-head latent attention decode.
//
// "vLLM AMD ROCm attention backend optimisation", section "AITER MLA backend:
// optimised for DeepSeek": the KV cache holds one 576-wide compressed latent
// row per position (512 latent + 64 rope); the "hybrid processing strategy"
// runs decode absorbed, directly on that latent.  Every query head scores
// against the whole 576-wide row; the value of a row is its 512 latent
// entries.  128 heads share each row, so this is a dense contraction
// (M = 128 heads) and runs on the tensor cores.
//
// GB300 design: a 128 x 512 fp32 output accumulator fills all of one SM's
// TMEM, so one work item -- a KV split of one sequence -- runs on a CLUSTER
// OF TWO CTAs that split the contraction dimensions between them:
//   CTA 0 owns latent columns 0..255 plus the 64 rope columns,
//   CTA 1 owns latent columns 256..511.
// Each CTA loads only its own columns of every cached row (TMA, 128-byte
// swizzled boxes of 64 columns x 32 slots), so the cache is read from HBM
// exactly once and no FLOP is duplicated.  Per 32-position tile each CTA
// forms its partial scores S_c = Q[:, own] K[:, own]^T in TMEM, stages them in
// its own shared memory and pushes them to its peer with one bulk DSMEM copy
// (completion counted on the peer's mbarrier), adds the peer's partial, runs
// the same online softmax (base 2, lazy rescaling), stores P as packed bf16
// in TMEM and accumulates O[:, own] += P V[:, own] (N = 256, P read from TMEM,
// V read MN-major from the staged rows).
// Splits of a long context are merged by log-sum-exp in a second kernel.
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kMlaL = 512, kMlaR = 64, kMlaW = 576, kMlaH = 128;
constexpr int kMN = 32;             // KV positions per tile
constexpr int kMlaThreads = 192;    // 4 softmax warps, producer warp, MMA warp
constexpr int kMlaStages = 4;
constexpr int kChunkQ = 128 * 128;  // Q: 128 heads x 64 columns, bf16
constexpr int kChunkKV = kMN * 128; // KV: 32 rows x 64 columns, bf16
constexpr int kMaxChunks = 5;
constexpr int kVHalf = 256;         // value columns per CTA
constexpr float kTau = 8.0f;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;      // O: columns [0, 256)
constexpr uint32_t kTmemS = 256;    // S: two buffers of 32 columns
constexpr uint32_t kTmemP = 320;    // P: two buffers of 16 columns (32 bf16 per row)
constexpr int kMinSplit = 512;

constexpr int OFF_Q = 0;
constexpr int OFF_KV = OFF_Q + kMaxChunks * kChunkQ;
constexpr int STAGE_BYTES = kMaxChunks * kChunkKV;
constexpr int X_BYTES = 128 * kMN * 4;               // one tile of partial scores
constexpr int OFF_X = OFF_KV + kMlaStages * STAGE_BYTES;  // peer's partials, 2 buffers
constexpr int OFF_XS = OFF_X + 2 * X_BYTES;               // own partials staged, 2 buffers
constexpr int OFF_BAR = OFF_XS + 2 * X_BYTES;

enum MBar {
  kQFull = 0, kQFree, kKVFull0, kKVFree0 = kKVFull0 + kMlaStages, kSFull0 = kKVFree0 + kMlaStages,
  kSFree0 = kSFull0 + 2, kXFull0 = kSFree0 + 2, kXFree0 = kXFull0 + 2, kPFull0 = kXFree0 + 2,
  kODone0 = kPFull0 + 2, kOFree = kODone0 + 2, kNumMBars
};
constexpr int OFF_MISC = OFF_BAR + kNumMBars * 8;
constexpr int MLA_SMEM = OFF_MISC + 64 + 1024;

constexpr uint32_t IDESC_S = umma_idesc_bf16(128, kMN, 0);
constexpr uint32_t IDESC_PV = umma_idesc_bf16(128, kVHalf, 1);

struct MlaArgs {
  const void *q;
  void *out;
  const int32_t *block_table;
  const int32_t *seq_lens;
  int num_seqs, block_size, max_blocks_per_seq, num_blocks, max_seq_len, kv_split_tokens;
  float scale_log2;
  int max_splits, num_clusters;
  long long *plan;      // [0] work items, [1] split length
  long long *item_end;  // [num_seqs] inclusive prefix of splits
  int *nsplit;          // [num_seqs]; 0 marks a sequence whose metadata failed
  float *part_o;        // [(s * 128 + h) * max_splits + split][512]
  float *part_lse;      // same rows; base-2 log-sum-exp, NaN = bad split
  unsigned int *status;
};

// Column chunk (of 64) that local chunk i of CTA `rank` holds.
__device__ inline int chunk_of(uint32_t rank, int i) {
  return rank == 0 ? (i < 4 ? i : 8) : 4 + i;
}

// ---------------------------------------------------------------------------
// planner: validity, split length, prefix sums of splits (one block)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) mla_plan_kernel(const MlaArgs a) {
  __shared__ long long scratch[33];
  const int S = a.num_seqs, tid = threadIdx.x;
  pdl_wait();     // whatever preceded this call in the stream
  pdl_trigger();  // the decode kernel may start its prologue meanwhile
  long long tot = 0;
  int bad = 0;
  for (int s = tid; s < S; s += 1024) {
    const int ctx = a.seq_lens[s];
    const bool ok = ctx >= 1 && ctx <= a.max_seq_len &&
                    ceil_div_ll(ctx, a.block_size) <= (long long)a.max_blocks_per_seq;
    if (ok) tot += ctx; else bad = 1;
  }
  if (bad) atomicOr(a.status, PA_DEV_BAD_SEQLEN);
  long long total;
  block_inclusive_scan(tot, scratch, &total);
  long long L;
  if (a.kv_split_tokens > 0) {
    L = a.kv_split_tokens;
  } else {
    L = kMinSplit;
    while (L < 8192 && total > L * 6ll * a.num_clusters) L <<= 1;
  }
  long long run = 0;
  for (int base = 0; base < S; base += 1024) {
    const int s = base + tid;
    int ns = 0;
    if (s < S) {
      const int ctx = a.seq_lens[s];
      const bool ok = ctx >= 1 && ctx <= a.max_seq_len &&
                      ceil_div_ll(ctx, a.block_size) <= (long long)a.max_blocks_per_seq;
      ns = ok ? (int)ceil_div_ll(ctx, L) : 0;
      if (ns > a.max_splits) ns = 0;  // cannot happen when seq_lens <= max_seq_len
    }
    long long ctot;
    const long long incl = block_inclusive_scan(ns, scratch, &ctot) + run;
    if (s < S) {
      a.item_end[s] = incl;
      a.nsplit[s] = ns;
    }
    run += ctot;
  }
  if (tid == 0) {
    a.plan[0] = run;
    a.plan[1] = L;
  }
}

// ---------------------------------------------------------------------------
// the cluster kernel
// ---------------------------------------------------------------------------
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kMlaThreads, 1)
    mla_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kv,
               const MlaArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t *sQ = smem + OFF_Q;
  uint8_t *sKV = smem + OFF_KV;
  uint8_t *sX = smem + OFF_X;
  uint8_t *sXS = smem + OFF_XS;
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
  uint32_t *s_tmem = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
  int *s_bad = reinterpret_cast<int *>(smem + OFF_MISC + 16);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank(), peer = rank ^ 1u;
  const int nch = rank == 0 ? 5 : 4;
  const long long cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
  pdl_trigger();
  pdl_wait();  // the plan
  const long long n_items = a.plan[0];
  const int L = (int)a.plan[1];
  const int S = a.num_seqs, bs = a.block_size;

  if (tid == 0) {
    prefetch_tensor_map(&tm_q);
    prefetch_tensor_map(&tm_kv);
    for (int b = 0; b < kNumMBars; ++b) {
      const bool per_warp = b == kSFree0 || b == kSFree0 + 1 || b == kPFull0 ||
                            b == kPFull0 + 1 || b == kOFree;
      mbar_init(&bar[b], per_warp ? 4u : 1u);
    }
    fence_mbar_init();
  }
  if (warp == 5) tc_alloc(s_tmem, kTmemCols);
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // the peer's barriers exist before anyone arrives remotely
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  bool dead = false;

  auto decode = [&](long long item, int &s, int &split, int &kv_lo, int &kv_hi) {
    s = list_find(a.item_end, S, item);
    split = (int)(item - (s ? a.item_end[s - 1] : 0));
    kv_lo = split * L;
    kv_hi = min(kv_lo + L, a.seq_lens[s]);
  };

  if (warp == 4) {
    // ------------------------------------------------------------- producer
    // The whole warp walks the items (the page cache is warp-wide); lane 0
    // waits on the barriers and issues the copies.
    uint32_t tiles = 0, items = 0;
    for (long long item = cluster; item < n_items; item += nclusters) {
      int s, split, kv_lo, kv_hi;
      decode(item, s, split, kv_lo, kv_hi);
      const int nt = (kv_hi - kv_lo + kMN - 1) / kMN;
      if (lane == 0) {
        if (items > 0) mbar_wait(&bar[kQFree], (items - 1) & 1, dead, a.status);
        mbar_arrive_expect_tx(&bar[kQFull], nch * kChunkQ);
        for (int i = 0; i < nch; ++i)
          tma_load_3d(sQ + i * kChunkQ, &tm_q, chunk_of(rank, i) * 64, 0, s, &bar[kQFull]);
      }
      const int32_t *bt = a.block_table + (size_t)s * a.max_blocks_per_seq;
      PageCache pc;
      pc.start(bt, a.max_blocks_per_seq, kv_lo / bs, lane);
      for (int j = 0; j < nt; ++j) {
        const uint32_t g = tiles + j;
        const int st = g % kMlaStages;
        const int pos = kv_lo + j * kMN;
        const int page = pc.get(pos / bs, lane);
        const bool ok = page >= 0 && page < a.num_blocks;
        if (lane == 0) {
          if (!ok) atomicOr(a.status, PA_DEV_BAD_BLOCK);
          if (g >= kMlaStages)
            mbar_wait(&bar[kKVFree0 + st], ((g / kMlaStages) - 1) & 1, dead, a.status);
          mbar_arrive_expect_tx(&bar[kKVFull0 + st], ok ? nch * kChunkKV : 0);
          if (ok)
            for (int i = 0; i < nch; ++i)
              tma_load_3d(sKV + st * STAGE_BYTES + i * kChunkKV, &tm_kv, chunk_of(rank, i) * 64,
                          pos % bs, page, &bar[kKVFull0 + st]);
        }
        __syncwarp();
      }
      tiles += nt;
      ++items;
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t tiles = 0, items = 0;
      const uint32_t sq = smem_u32(sQ), skv = smem_u32(sKV);
      auto issue_s = [&](uint32_t g) {
        const int st = g % kMlaStages, b = g & 1;
        mbar_wait(&bar[kKVFull0 + st], (g / kMlaStages) & 1, dead, a.status);
        if (g >= 2) mbar_wait(&bar[kSFree0 + b], ((g >> 1) - 1) & 1, dead, a.status);
        tc_fence_after();
        const uint32_t kb = skv + st * STAGE_BYTES;
        for (int i = 0; i < nch; ++i)
#pragma unroll
          for (int sub = 0; sub < 4; ++sub) {
            const uint64_t ad = umma_desc_sw128(sq + i * kChunkQ + sub * 32, 16, 1024);
            const uint64_t bd = umma_desc_sw128(kb + i * kChunkKV + sub * 32, 16, 1024);
            tc_mma_bf16(tmem + kTmemS + b * kMN, ad, bd, IDESC_S, (i > 0 || sub > 0) ? 1u : 0u);
          }
        tc_commit(&bar[kSFull0 + b]);
      };
      for (long long item = cluster; item < n_items; item += nclusters) {
        int s, split, kv_lo, kv_hi;
        decode(item, s, split, kv_lo, kv_hi);
        const int nt = (kv_hi - kv_lo + kMN - 1) / kMN;
        mbar_wait(&bar[kQFull], items & 1, dead, a.status);
        issue_s(tiles);
        for (int j = 0; j < nt; ++j) {
          const uint32_t g = tiles + j;
          if (j + 1 < nt) issue_s(g + 1);
          const int pb = g & 1;
          mbar_wait(&bar[kPFull0 + pb], (g >> 1) & 1, dead, a.status);
          if (j == 0 && items > 0) mbar_wait(&bar[kOFree], (items - 1) & 1, dead, a.status);
          tc_fence_after();
          const uint32_t vb = skv + (g % kMlaStages) * STAGE_BYTES;
#pragma unroll
          for (int kk = 0; kk < kMN / 16; ++kk) {
            const uint64_t bd = umma_desc_sw128(vb + kk * 16 * 128, kChunkKV, 1024);
            tc_mma_bf16_ts(tmem + kTmemO, tmem + kTmemP + pb * 16 + kk * 8, bd, IDESC_PV,
                           (j > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(&bar[kKVFree0 + g % kMlaStages]);
          tc_commit(&bar[kODone0 + pb]);
        }
        tc_commit(&bar[kQFree]);
        tiles += nt;
        ++items;
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------- softmax
    const int r = tid;  // head == TMEM lane
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    uint32_t x_peer[2], xfull_peer[2], xfree_peer[2];
    for (int b = 0; b < 2; ++b) {
      x_peer[b] = cluster_map(smem_u32(sX + b * X_BYTES), peer);
      xfull_peer[b] = cluster_map(smem_u32(&bar[kXFull0 + b]), peer);
      xfree_peer[b] = cluster_map(smem_u32(&bar[kXFree0 + b]), peer);
    }
    uint32_t tiles = 0, items = 0;
    for (long long item = cluster; item < n_items; item += nclusters) {
      int s, split, kv_lo, kv_hi;
      decode(item, s, split, kv_lo, kv_hi);
      const int nt = (kv_hi - kv_lo + kMN - 1) / kMN;
      {
        const int pfirst = kv_lo / bs, plast = (kv_hi - 1) / bs;
        const int32_t *bt = a.block_table + (size_t)s * a.max_blocks_per_seq;
        int bad = 0;
        for (int lp = pfirst + r; lp <= plast; lp += 128) {
          const int pg = lp < a.max_blocks_per_seq ? __ldg(bt + lp) : -1;
          if (pg < 0 || pg >= a.num_blocks) bad = 1;
        }
        bad = __any_sync(0xffffffffu, bad);
        if (r == 0) s_bad[items & 1] = 0;
        named_sync(1, 128);
        if (bad && lane == 0) atomicOr(&s_bad[items & 1], 1);
        named_sync(1, 128);
      }
      const bool item_bad = s_bad[items & 1] != 0;
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < nt; ++j) {
        const uint32_t g = tiles + j;
        const int b = g & 1;
        const int base = kv_lo + j * kMN;
        mbar_wait(&bar[kSFull0 + b], (g >> 1) & 1, dead, a.status);
        tc_fence_after();
        uint32_t raw[32];
        tc_ld32(tmem + lane_off + kTmemS + b * kMN, raw);
        tc_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[kSFree0 + b]);
        // stage the partial scores, then one bulk copy to the peer: the staging
        // and the peer's buffer b are free once the peer has consumed tile g - 2
        if (g >= 2) mbar_wait_cluster(&bar[kXFree0 + b], ((g >> 1) - 1) & 1, dead, a.status);
        // Row r of the partial scores is 8 float4s; float4 v sits in slot
        // v ^ (r % 8), so the 8 rows a quarter-warp touches hit 8 different
        // bank groups (plain rows of 128 bytes all start in the same banks).
        float4 *st4 = reinterpret_cast<float4 *>(sXS + b * X_BYTES + r * kMN * 4);
#pragma unroll
        for (int v = 0; v < kMN / 4; ++v)
          st4[v ^ (r & 7)] = make_float4(__uint_as_float(raw[4 * v]), __uint_as_float(raw[4 * v + 1]),
                                         __uint_as_float(raw[4 * v + 2]), __uint_as_float(raw[4 * v + 3]));
        fence_proxy_async();
        named_sync(1, 128);
        if (r == 0) {
          mbar_arrive_expect_tx(&bar[kXFull0 + b], X_BYTES);  // the peer's tile g lands here
          bulk_copy_to_peer(x_peer[b], sXS + b * X_BYTES, X_BYTES, xfull_peer[b]);
        }
        mbar_wait_cluster(&bar[kXFull0 + b], (g >> 1) & 1, dead, a.status);
        float sc[kMN];
        const float4 *xr = reinterpret_cast<const float4 *>(sX + b * X_BYTES + r * kMN * 4);
#pragma unroll
        for (int v = 0; v < kMN / 4; ++v) {
          const float4 o4 = xr[v ^ (r & 7)];
          sc[4 * v] = __uint_as_float(raw[4 * v]) + o4.x;
          sc[4 * v + 1] = __uint_as_float(raw[4 * v + 1]) + o4.y;
          sc[4 * v + 2] = __uint_as_float(raw[4 * v + 2]) + o4.z;
          sc[4 * v + 3] = __uint_as_float(raw[4 * v + 3]) + o4.w;
        }
        named_sync(1, 128);
        // Hand our buffer b back to the peer.  Every thread's reads of it have
        // returned (their sums are in registers) and the CTA barrier above
        // orders them before this arrive, so a relaxed arrive suffices; a
        // cluster-scope release arrive cost about 1.8k cycles a tile.
        if (r == 0) mbar_arrive_remote_relaxed(xfree_peer[b]);
        float mxa[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < kMN; ++c) {
          sc[c] = (base + c < kv_hi) ? sc[c] * a.scale_log2 : -INFINITY;
          mxa[c & 3] = fmaxf(mxa[c & 3], sc[c]);
        }
        const float mx = fmaxf(fmaxf(mxa[0], mxa[1]), fmaxf(mxa[2], mxa[3]));
        // P buffer b was last read by the PV product of tile g - 2
        if (g >= 2) mbar_wait(&bar[kODone0 + b], ((g >> 1) - 1) & 1, dead, a.status);
        tc_fence_after();
        float alpha = 1.f;
        bool rescale = false;
        if (mx > m + kTau) {
          alpha = fast_exp2(m - mx);
          l *= alpha;
          m = mx;
          rescale = j > 0;
        }
        if (__any_sync(0xffffffffu, rescale)) {
          mbar_wait(&bar[kODone0 + (b ^ 1)], ((g - 1) >> 1) & 1, dead, a.status);
          tc_fence_after();
          const float al = rescale ? alpha : 1.f;
          for (int c0 = 0; c0 < kVHalf; c0 += 32) {
            uint32_t o[32];
            tc_ld32(tmem + lane_off + kTmemO + c0, o);
            tc_wait_ld();
#pragma unroll
            for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * al);
            tc_st32(tmem + lane_off + kTmemO + c0, o);
          }
          tc_wait_st();
        }
        const float mu = m == -INFINITY ? 0.f : m;
        float suma[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t pw[kMN / 2];
#pragma unroll
        for (int x = 0; x < kMN / 2; ++x) {
          const float p0 = fast_exp2(sc[2 * x] - mu);
          const float p1 = fast_exp2(sc[2 * x + 1] - mu);
          suma[x & 3] += p0 + p1;
          const __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
          pw[x] = *reinterpret_cast<const uint32_t *>(&h2);
        }
        tc_st16(tmem + lane_off + kTmemP + b * 16, pw);
        tc_wait_st();
        l += (suma[0] + suma[1]) + (suma[2] + suma[3]);
        if (j == nt - 1 && kv_hi - base < kMN) {
          // slots past the sequence end may hold anything; 0 * NaN is NaN
          mbar_wait(&bar[kKVFull0 + g % kMlaStages], (g / kMlaStages) & 1, dead, a.status);
          const int first = kv_hi - base;
          uint8_t *vb = sKV + (g % kMlaStages) * STAGE_BYTES;
          const int per_chunk = (kMN - first) * 8;
          for (int e = r; e < 4 * per_chunk; e += 128) {
            const int ci = e / per_chunk, rem = e % per_chunk;
            *reinterpret_cast<uint4 *>(vb + ci * kChunkKV + (first + rem / 8) * 128 + (rem % 8) * 16) =
                make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[kPFull0 + b]);
      }
      // ---- epilogue
      const uint32_t glast = tiles + nt - 1;
      mbar_wait(&bar[kODone0 + (glast & 1)], (glast >> 1) & 1, dead, a.status);
      tc_fence_after();
      const int ns = a.nsplit[s];
      const bool direct = ns == 1;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const uint32_t keep = item_bad ? 0u : 0xffffffffu;
      const long long prow = ((long long)s * kMlaH + r) * a.max_splits + split;
      for (int c0 = 0; c0 < kVHalf; c0 += 32) {
        uint32_t o[32];
        tc_ld32(tmem + lane_off + kTmemO + c0, o);
        tc_wait_ld();
#pragma unroll
        for (int x = 0; x < 32; ++x) o[x] &= keep;
        const int col = (int)rank * kVHalf + c0;
        if (direct) {
          uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(a.out) +
                                                 ((size_t)s * kMlaH + r) * kMlaL + col);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint32_t w[4];
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              const __nv_bfloat162 h2 =
                  __floats2bfloat162_rn(__uint_as_float(o[v * 8 + 2 * x]) * inv,
                                        __uint_as_float(o[v * 8 + 2 * x + 1]) * inv);
              w[x] = *reinterpret_cast<const uint32_t *>(&h2);
            }
            dst[v] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        } else {
          float4 *dst = reinterpret_cast<float4 *>(a.part_o + prow * kMlaL + col);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            dst[v] = make_float4(__uint_as_float(o[4 * v]) * inv, __uint_as_float(o[4 * v + 1]) * inv,
                                 __uint_as_float(o[4 * v + 2]) * inv,
                                 __uint_as_float(o[4 * v + 3]) * inv);
        }
      }
      if (!direct && rank == 0)
        a.part_lse[prow] = item_bad ? __int_as_float(0x7fc00000) : (l > 0.f ? m + log2f(l) : -INFINITY);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[kOFree]);
      tiles += nt;
      ++items;
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no remote access to this CTA's shared memory remains
  tc_fence_after();
  if (warp == 5) tc_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------
// merge of split partials: one block per (sequence, head) row
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) mla_merge_kernel(const MlaArgs a) {
  const int tid = threadIdx.x;
  const long long rows = (long long)a.num_seqs * kMlaH;
  pdl_trigger();
  pdl_wait();  // the split partials
  __nv_bfloat16 *out = reinterpret_cast<__nv_bfloat16 *>(a.out);
  for (long long row = blockIdx.x; row < rows; row += gridDim.x) {
    const int s = (int)(row / kMlaH);
    const int ns = a.nsplit[s];
    if (ns == 1) continue;
    __nv_bfloat162 *dst = reinterpret_cast<__nv_bfloat162 *>(out + row * kMlaL) + tid;
    if (ns == 0) {
      *dst = __floats2bfloat162_rn(0.f, 0.f);
      continue;
    }
    const long long base = row * a.max_splits;
    float M = -INFINITY;
    bool bad = false;
    for (int q = 0; q < ns; ++q) {
      const float v = a.part_lse[base + q];
      if (isnan(v)) bad = true; else M = fmaxf(M, v);
    }
    float L = 0.f, x = 0.f, y = 0.f;
    if (!bad && M != -INFINITY) {
      for (int q = 0; q < ns; ++q) {
        const float w = fast_exp2(a.part_lse[base + q] - M);
        const float2 v = reinterpret_cast<const float2 *>(a.part_o + (base + q) * kMlaL)[tid];
        L += w;
        x = fmaf(w, v.x, x);
        y = fmaf(w, v.y, y);
      }
    }
    const float inv = (bad || !(L > 0.f)) ? 0.f : 1.f / L;
    *dst = __floats2bfloat162_rn(x * inv, y * inv);
  }
}

struct MlaLayout {
  size_t plan, item_end, nsplit, part_o, part_lse, total;
  int max_splits;
};

size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

MlaLayout mla_layout(int num_seqs, int max_seq_len, int kvs) {
  MlaLayout l{};
  const long long lmin = kvs > 0 ? kvs : kMinSplit;
  l.max_splits = (int)ceil_div_ll(max_seq_len > 0 ? max_seq_len : 1, lmin);
  const size_t S = num_seqs > 0 ? num_seqs : 1;
  const size_t rows = (size_t)S * kMlaH * l.max_splits;
  size_t off = 0;
  l.plan = off;
  off = al256(off + 64);
  l.item_end = off;
  off = al256(off + S * sizeof(long long));
  l.nsplit = off;
  off = al256(off + S * sizeof(int));
  l.part_o = off;
  off = al256(off + rows * kMlaL * sizeof(float));
  l.part_lse = off;
  off = al256(off + rows * sizeof(float));
  l.total = off;
  return l;
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" {

size_t pa_mla_decode_workspace_bytes(int num_seqs, int num_heads, int kv_lora_rank,
                                     int max_seq_len, int kv_split_tokens) {
  if (num_heads != kMlaH || kv_lora_rank != kMlaL || num_seqs < 0 || max_seq_len < 0 ||
      kv_split_tokens < 0)
    return 0;
  return mla_layout(num_seqs, max_seq_len, kv_split_tokens).total;
}

pa_status pa_mla_decode(const void *q, const void *kv_cache, const int32_t *block_table,
                        const int32_t *seq_lens, int num_heads, int kv_lora_rank, int rope_dim,
                        int block_size, float scale, void *out, void *stream, int num_seqs,
                        int max_blocks_per_seq, int num_blocks, int max_seq_len,
                        int kv_split_tokens) {
  if (num_seqs < 0 || max_seq_len < 0 || kv_split_tokens < 0 || block_size <= 0 ||
      num_heads <= 0 || kv_lora_rank <= 0 || rope_dim < 0)
    return PA_ERR_INVALID_ARG;
  if (num_heads != kMlaH || kv_lora_rank != kMlaL || rope_dim != kMlaR || block_size % 32 != 0 ||
      block_size > 256 || kv_split_tokens % 32 != 0)
    return PA_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PA_OK;
  if (!q || !kv_cache || !block_table || !seq_lens || !out || num_blocks <= 0 ||
      max_blocks_per_seq <= 0)
    return PA_ERR_INVALID_ARG;
  if (((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(kv_cache) |
        reinterpret_cast<uintptr_t>(out)) & 15) != 0)
    return PA_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const MlaLayout lay = mla_layout(num_seqs, max_seq_len, kv_split_tokens);
  void *ws = nullptr;
  unsigned int *status = nullptr;
  int num_sms = 0;
  pa_status s = device_resources(st, lay.total, &ws, &status, &num_sms);
  if (s != PA_OK) return s;
  uint8_t *w = reinterpret_cast<uint8_t *>(ws);

  static bool attr_done[64] = {};
  static int max_clusters[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return PA_ERR_CUDA;
  if (!attr_done[dev]) {
    if (cudaFuncSetAttribute(mla_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, MLA_SMEM) !=
            cudaSuccess ||
        cudaFuncSetAttribute(mla_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess)
      return PA_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (num_sms / 2));
    cfg.blockDim = dim3(kMlaThreads);
    cfg.dynamicSmemBytes = MLA_SMEM;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, mla_kernel, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = num_sms / 2;
    }
    max_clusters[dev] = n < num_sms / 2 ? n : num_sms / 2;
    attr_done[dev] = true;
  }

  MlaArgs a{};
  a.q = q;
  a.out = out;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.num_seqs = num_seqs;
  a.block_size = block_size;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_blocks = num_blocks;
  a.max_seq_len = max_seq_len;
  a.kv_split_tokens = kv_split_tokens;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.max_splits = lay.max_splits;
  a.num_clusters = max_clusters[dev];
  a.plan = reinterpret_cast<long long *>(w + lay.plan);
  a.item_end = reinterpret_cast<long long *>(w + lay.item_end);
  a.nsplit = reinterpret_cast<int *>(w + lay.nsplit);
  a.part_o = reinterpret_cast<float *>(w + lay.part_o);
  a.part_lse = reinterpret_cast<float *>(w + lay.part_lse);
  a.status = status;

  CUtensorMap tm_q, tm_kv;
  const unsigned long long qd[3] = {kMlaW, kMlaH, (unsigned long long)num_seqs};
  const unsigned long long qs[2] = {kMlaW * 2, (unsigned long long)kMlaH * kMlaW * 2};
  const unsigned int qb[3] = {64, 128, 1};
  const unsigned long long kd[3] = {kMlaW, (unsigned long long)block_size,
                                    (unsigned long long)num_blocks};
  const unsigned long long ks[2] = {kMlaW * 2, (unsigned long long)block_size * kMlaW * 2};
  const unsigned int kb[3] = {64, kMN, 1};
  if (!encode_tiled(&tm_q, q, PA_BF16, 3, qd, qs, qb, true) ||
      !encode_tiled(&tm_kv, kv_cache, PA_BF16, 3, kd, ks, kb, true))
    return PA_ERR_CUDA;

  int slot = prof_begin(PA_K_PLAN, st);
  cudaError_t err = launch_dependent(mla_plan_kernel, dim3(1), dim3(1024), 0, st, a);
  prof_end(slot, st);
  if (err != cudaSuccess) return PA_ERR_CUDA;
  slot = prof_begin(PA_K_MLA, st);
  err = launch_dependent(mla_kernel, dim3(2 * a.num_clusters), dim3(kMlaThreads),
                                     MLA_SMEM, st, tm_q, tm_kv, a);
  prof_end(slot, st);
  if (err != cudaSuccess) return PA_ERR_CUDA;
  slot = prof_begin(PA_K_MLA_MERGE, st);
  err = launch_dependent(mla_merge_kernel, dim3(num_sms * 4), dim3(256), 0, st, a);
  prof_end(slot, st);
  if (err != cudaSuccess) return PA_ERR_CUDA;
  return PA_OK;
}

}  // extern "C"
