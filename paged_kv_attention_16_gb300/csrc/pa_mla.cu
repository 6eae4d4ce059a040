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
// swizzled boxes of 64 columns x 32 slots into a 4-stage ring of 64-position
// tiles), so the cache is read from HBM exactly once and no FLOP is
// duplicated.  Tensor memory per CTA: O (128 x 256 fp32), the item's query
// columns (bf16 pairs, the A operand of the score product), one S tile
// (128 x 64 fp32) and P (128 x 64 bf16).  Per tile each CTA forms its partial
// scores S_c = Q[:, own] K[:, own]^T, and its softmax warps push them from
// registers straight into the peer's shared memory with asynchronous remote
// stores that complete on the peer's mbarrier -- for tile j + 1 while tile j
// is being finished, so the exchange latency hides behind a softmax.  Each
// CTA adds the peer's partial to its own (the same sum in both), runs the
// same online softmax (base 2, lazy rescaling), stores P as packed bf16 in
// TMEM and accumulates O[:, own] += P V[:, own] (N = 256, P read from TMEM,
// V read MN-major from the staged rows).  The score product runs two tiles
// ahead of the value product.
// Splits of a long context are merged by log-sum-exp in a second kernel.
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kMlaL = 512, kMlaR = 64, kMlaW = 576, kMlaH = 128;
constexpr int kMN = 64;             // KV positions per tile
constexpr int kMHalf = 32;          // slots per TMA box (a box never crosses a page)
constexpr int kSoftWarps = 8;       // two per TMEM lane quarter: each thread half a row
constexpr int kSoftThreads = 32 * kSoftWarps;
constexpr int kProducerWarp = kSoftWarps, kMmaWarp = kSoftWarps + 1;
constexpr int kMlaThreads = 32 * (kSoftWarps + 2);
constexpr int kMlaStages = 4;
constexpr int kChunkKV = kMN * 128; // one 64-column chunk of a tile: 64 rows x 128 B
constexpr int kMaxChunks = 5;
constexpr int kVHalf = 256;         // value columns per CTA
constexpr float kTau = 8.0f;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;      // O: columns [0, 256)
constexpr uint32_t kTmemQ = 256;    // query columns: 160 (CTA 0) or 128 (CTA 1)
constexpr uint32_t kTmemS = 416;    // S: 64 columns
constexpr uint32_t kTmemP = 480;    // P: 32 columns (64 bf16 per row)
constexpr int kMinSplit = 512;

constexpr int STAGE_BYTES = kMaxChunks * kChunkKV;
constexpr int X_BYTES = 128 * kMN * 4;               // one tile of partial scores
constexpr int OFF_KV = 0;
constexpr int OFF_X = OFF_KV + kMlaStages * STAGE_BYTES;  // the peer's partials of a tile
constexpr int OFF_XS = OFF_X + X_BYTES;                   // own partials staged for the copy
constexpr int OFF_BAR = OFF_XS + X_BYTES;

enum MBar {
  kQFull = 0, kQFree, kKVFull0, kKVFree0 = kKVFull0 + kMlaStages, kSFull = kKVFree0 + kMlaStages,
  kSFree, kPFull, kODone, kOFree, kXFull, kXFree, kNumMBars
};
constexpr int OFF_RED = OFF_BAR + kNumMBars * 8;          // 256 floats: row halves' maxima
constexpr int OFF_MISC = OFF_RED + kSoftThreads * 4;
constexpr int MLA_SMEM = OFF_MISC + 64 + 1024;
static_assert(MLA_SMEM <= 232448, "shared memory budget");

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
  int page_tiles;       // 1: every 64-position tile lies in one page (block_size % 64 == 0
                        // and tiles start at multiples of 64): one box per 4 chunks
  // plan[2] = 0 (fixed split length): [0] work items, [1] split length,
  //   item_end = inclusive prefix of each sequence's splits;
  // plan[2] = 1 (balanced): [0] 64-position tiles in all, [1] tiles per
  //   cluster, item_end = inclusive prefix of each sequence's tiles
  long long *plan;
  long long *item_end;  // [num_seqs]
  int *nsplit;          // [num_seqs] pieces (partials); 0 marks a sequence whose metadata failed
  float *part_o;        // [(s * 128 + h) * max_splits + split][512]
  float *part_lse;      // same rows; base-2 log-sum-exp, NaN = bad split
  unsigned int *status;
};

// Column chunk (of 64) that local chunk i of CTA `rank` holds.
__device__ inline int chunk_of(uint32_t rank, int i) {
  return rank == 0 ? (i < 4 ? i : 8) : 4 + i;
}

// ---------------------------------------------------------------------------
// planner: validity, work split, prefix sums (one block)
//
// Automatic split (kv_split_tokens == 0): the batch's 64-position tiles, in
// sequence order, are cut into one contiguous run per cluster of
// ceil(tiles / clusters) tiles (at least kMinSplit / 64): every cluster gets
// the same work whatever the mix of lengths, and a sequence is split only
// where a run boundary falls inside it, so at most one partial per cluster
// boundary is written.  A fixed kv_split_tokens cuts every sequence into
// splits of that length, dealt to the clusters in turn.
// ---------------------------------------------------------------------------
constexpr int kMinRunTiles = kMinSplit / kMN;

__device__ inline bool mla_seq_ok(const MlaArgs &a, int ctx) {
  return ctx >= 1 && ctx <= a.max_seq_len &&
         ceil_div_ll(ctx, a.block_size) <= (long long)a.max_blocks_per_seq;
}

__global__ void __launch_bounds__(1024) mla_plan_kernel(const MlaArgs a) {
  __shared__ long long scratch[33];
  const int S = a.num_seqs, tid = threadIdx.x;
  pdl_wait();     // whatever preceded this call in the stream
  pdl_trigger();  // the decode kernel may start its prologue meanwhile
  const bool fixed = a.kv_split_tokens > 0;
  const long long L = fixed ? a.kv_split_tokens : kMN;
  // per sequence: splits (fixed) or tiles (balanced)
  long long run = 0;
  int bad = 0;
  for (int base = 0; base < S; base += 1024) {
    const int s = base + tid;
    long long n = 0;
    if (s < S) {
      const int ctx = a.seq_lens[s];
      if (mla_seq_ok(a, ctx)) n = ceil_div_ll(ctx, L); else bad = 1;
    }
    long long ctot;
    const long long incl = block_inclusive_scan(n, scratch, &ctot) + run;
    if (s < S) a.item_end[s] = incl;
    run += ctot;
  }
  if (bad) atomicOr(a.status, PA_DEV_BAD_SEQLEN);
  __syncthreads();
  long long per = L;
  if (!fixed) {
    per = ceil_div_ll(run, a.num_clusters > 0 ? a.num_clusters : 1);
    if (per < kMinRunTiles) per = kMinRunTiles;
  }
  for (int s = tid; s < S; s += 1024) {
    const long long t1 = a.item_end[s], t0 = s ? a.item_end[s - 1] : 0;
    int ns = (int)(t1 - t0);
    if (!fixed && t1 > t0) ns = (int)((t1 - 1) / per - t0 / per + 1);  // run boundaries inside
    if (ns > a.max_splits) ns = 0;  // cannot happen when seq_lens <= max_seq_len
    a.nsplit[s] = ns;
  }
  if (tid == 0) {
    a.plan[0] = run;
    a.plan[1] = per;
    a.plan[2] = fixed ? 0 : 1;
  }
}

// One work piece: positions [kv_lo, kv_hi) of sequence s, its split `split`.
struct MlaPiece {
  int s, split, kv_lo, kv_hi;
};

// Walks a cluster's pieces in order; every warp role keeps its own walker.
struct PieceWalk {
  long long pos, end, step;
  bool balanced;

  __device__ void start(const MlaArgs &a, long long cluster, long long nclusters) {
    balanced = a.plan[2] != 0;
    if (balanced) {
      pos = cluster * a.plan[1];
      end = min(pos + a.plan[1], a.plan[0]);
      step = 0;
    } else {
      pos = cluster;
      end = a.plan[0];
      step = nclusters;
    }
  }

  __device__ bool next(const MlaArgs &a, MlaPiece &p) {
    if (pos >= end) return false;
    const int s = list_find(a.item_end, a.num_seqs, pos);
    const long long first = s ? a.item_end[s - 1] : 0;
    const int ctx = a.seq_lens[s];
    p.s = s;
    if (balanced) {
      const long long per = a.plan[1];
      const long long stop = min(end, a.item_end[s]);
      p.split = (int)(pos / per - first / per);
      p.kv_lo = (int)((pos - first) * kMN);
      p.kv_hi = (int)min((stop - first) * kMN, (long long)ctx);
      pos = stop;
    } else {
      const int L = (int)a.plan[1];
      p.split = (int)(pos - first);
      p.kv_lo = p.split * L;
      p.kv_hi = min(p.kv_lo + L, ctx);
      pos += step;
    }
    return true;
  }
};

// ---------------------------------------------------------------------------
// the cluster kernel
// ---------------------------------------------------------------------------
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kMlaThreads, 1)
    mla_kernel(const __grid_constant__ CUtensorMap tm_kv, const __grid_constant__ CUtensorMap tm_kv4,
               const MlaArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t *sKV = smem + OFF_KV;
  uint8_t *sX = smem + OFF_X;
  uint8_t *sXS = smem + OFF_XS;
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
  float *s_red = reinterpret_cast<float *>(smem + OFF_RED);
  uint32_t *s_tmem = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
  int *s_bad = reinterpret_cast<int *>(smem + OFF_MISC + 16);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank(), peer = rank ^ 1u;
  const int nch = rank == 0 ? 5 : 4;
  const long long cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
  pdl_trigger();
  pdl_wait();  // the plan
  const int bs = a.block_size;

  if (tid == 0) {
    prefetch_tensor_map(&tm_kv);
    prefetch_tensor_map(&tm_kv4);
    for (int b = 0; b < kNumMBars; ++b) {
      const bool per_warp =
          b == kQFull || b == kSFree || b == kPFull || b == kOFree || b == kXFree;
      mbar_init(&bar[b], per_warp ? (uint32_t)kSoftWarps : 1u);
    }
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tc_alloc(s_tmem, kTmemCols);
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // the peer's barriers exist before anyone arrives remotely
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  bool dead = false;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------- producer
    // The whole warp walks the pieces (the page caches are warp-wide); lanes
    // 0 and 1 handle the two 32-slot halves of each tile, lane 0 waits.  (An
    // L2 prefetch of the tile four ahead measured 1.5 % slower: the
    // prefetch copies take this warp's issue time too.)
    uint32_t tiles = 0;
    PieceWalk walk;
    walk.start(a, cluster, nclusters);
    MlaPiece pc_;
    while (walk.next(a, pc_)) {
      const int s = pc_.s, kv_lo = pc_.kv_lo, kv_hi = pc_.kv_hi;
      const int nt = (kv_hi - kv_lo + kMN - 1) / kMN;
      const int32_t *bt = a.block_table + (size_t)s * a.max_blocks_per_seq;
      PageCache pc;
      pc.start(bt, a.max_blocks_per_seq, kv_lo / bs, lane);
      // A tile's rows: with page_tiles, one box of 4 latent chunks x 64 slots
      // (whole 512-byte row spans, so the copy engine moves few large pieces)
      // plus, on CTA 0, one box for the rope chunk; otherwise one 64-column x
      // 32-slot box per chunk and half tile (lanes 0 and 1).
      const bool big = a.page_tiles != 0;
      const int c4 = rank == 0 ? 0 : 4;  // first latent chunk of this CTA
      for (int j = 0; j < nt; ++j) {
        const uint32_t g = tiles + j;
        const int st = g % kMlaStages;
        const int pos = kv_lo + j * kMN + lane * kMHalf;
        const bool need = (big ? lane == 0 : lane < 2) && pos < kv_hi;
        const int page = pc.get(need ? pos / bs : -1, lane);
        const bool ok = need && page >= 0 && page < a.num_blocks;
        if (need && !ok) atomicOr(a.status, PA_DEV_BAD_BLOCK);
        const unsigned mask = __ballot_sync(0xffffffffu, ok);
        if (lane == 0) {
          if (g >= kMlaStages)
            mbar_wait(&bar[kKVFree0 + st], ((g / kMlaStages) - 1) & 1, dead, a.status);
          mbar_arrive_expect_tx(&bar[kKVFull0 + st],
                                __popc(mask) * nch * (big ? kMN : kMHalf) * 128);
        }
        __syncwarp();
        if (ok) {
          uint8_t *dst = sKV + st * STAGE_BYTES;
          if (big) {
            tma_load_4d(dst, &tm_kv4, 0, pos % bs, c4, page, &bar[kKVFull0 + st]);
            if (rank == 0)
              tma_load_3d(dst + 4 * kChunkKV, &tm_kv, 8 * 64, pos % bs, page, &bar[kKVFull0 + st]);
          } else {
            for (int i = 0; i < nch; ++i)
              tma_load_3d(dst + i * kChunkKV + lane * kMHalf * 128, &tm_kv, chunk_of(rank, i) * 64,
                          pos % bs, page, &bar[kKVFull0 + st]);
          }
        }
        __syncwarp();
      }
      tiles += nt;
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t g = 0, items = 0;
      const uint32_t skv = smem_u32(sKV);
      // S of tile t (global count) once its K rows have landed and the
      // softmax has read S of tile t - 1 out of the single S buffer.
      auto issue_s = [&](uint32_t t) {
        const int st = t % kMlaStages;
        mbar_wait(&bar[kKVFull0 + st], (t / kMlaStages) & 1, dead, a.status);
        if (t > 0) mbar_wait(&bar[kSFree], (t - 1) & 1, dead, a.status);
        tc_fence_after();
        const uint32_t kb = skv + st * STAGE_BYTES;
        for (int kk = 0; kk < nch * 4; ++kk) {
          const uint64_t bd = umma_desc_sw128(kb + (kk >> 2) * kChunkKV + (kk & 3) * 32, 16, 1024);
          tc_mma_bf16_ts(tmem + kTmemS, tmem + kTmemQ + kk * 8, bd, IDESC_S, kk > 0 ? 1u : 0u);
        }
        tc_commit(&bar[kSFull]);
      };
      PieceWalk walk;
      walk.start(a, cluster, nclusters);
      MlaPiece pc_;
      while (walk.next(a, pc_)) {
        const int nt = (pc_.kv_hi - pc_.kv_lo + kMN - 1) / kMN;
        mbar_wait(&bar[kQFull], items & 1, dead, a.status);
        tc_fence_after();
        issue_s(g);
        if (nt == 1) tc_commit(&bar[kQFree]);
        if (nt > 1) {
          issue_s(g + 1);
          if (nt == 2) tc_commit(&bar[kQFree]);
        }
        for (int j = 0; j < nt; ++j) {
          const uint32_t t = g + j;
          if (j + 2 < nt) {
            issue_s(t + 2);
            if (j + 2 == nt - 1) tc_commit(&bar[kQFree]);
          }
          mbar_wait(&bar[kPFull], t & 1, dead, a.status);
          if (j == 0 && items > 0) mbar_wait(&bar[kOFree], (items - 1) & 1, dead, a.status);
          tc_fence_after();
          const uint32_t vb = skv + (t % kMlaStages) * STAGE_BYTES;
#pragma unroll
          for (int kk = 0; kk < kMN / 16; ++kk) {
            const uint64_t bd = umma_desc_sw128(vb + kk * 16 * 128, kChunkKV, 1024);
            tc_mma_bf16_ts(tmem + kTmemO, tmem + kTmemP + kk * 8, bd, IDESC_PV,
                           (j > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(&bar[kKVFree0 + t % kMlaStages]);
          tc_commit(&bar[kODone]);
        }
        g += nt;
        ++items;
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------- softmax
    // Thread = (head r = TMEM lane, half h): positions 32h .. 32h + 31 of each
    // tile, value columns 128h .. 128h + 127 of O.
    constexpr int kHalfN = kMN / 2;
    const int r = (warp & 3) * 32 + lane;
    const int h = warp >> 2;
    const int partner = tid ^ 128;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t x_peer = cluster_map(smem_u32(sX), peer);
    const uint32_t xfull_peer = cluster_map(smem_u32(&bar[kXFull]), peer);
    const uint32_t xfree_peer = cluster_map(smem_u32(&bar[kXFree]), peer);
    // This CTA's query columns of sequence s into TMEM (bf16 pairs, the A
    // operand of the score product): 64-column chunks in contraction order,
    // the two halves of a row taking alternate chunks.
    auto load_q = [&](int s) {
      const uint4 *qrow = reinterpret_cast<const uint4 *>(a.q) + ((size_t)s * kMlaH + r) * (kMlaW / 8);
#pragma unroll 1
      for (int i = h; i < nch; i += 2) {  // one chunk at a time (the rows are in L2)
        uint4 qv[8];
#pragma unroll
        for (int x = 0; x < 8; ++x) qv[x] = __ldg(qrow + chunk_of(rank, i) * 8 + x);
        tc_st32(tmem + lane_off + kTmemQ + i * 32, *reinterpret_cast<const uint32_t(*)[32]>(qv));
      }
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[kQFull]);
    };
    // Exchange buffers (the peer's, and this CTA's staging copy) hold one
    // tile as [half][head][8 float4]: each warp's 32 rows x 128 B are one
    // contiguous 4 KB block, which the warp copies to the peer by itself.
    // Slot x of row r is stored at x ^ (r % 8), so the rows a quarter-warp
    // touches fall in different banks.
    const uint32_t xrow = (uint32_t)(h * 128 + r) * 128;
    const uint32_t xwarp = (uint32_t)(h * 128 + (warp & 3) * 32) * 128;
    // Read this thread's 32 scores of tile t out of TMEM, free the buffer,
    // stage them and push the warp's block into the peer's exchange buffer
    // with one bulk copy (completion counted on the peer's mbarrier).  The
    // staging block is reused once the warp's previous copy has read it, the
    // peer's buffer once every peer warp has consumed tile t - 1.
    auto fetch_send = [&](uint32_t t, float (&v)[kHalfN]) {
      mbar_wait(&bar[kSFull], t & 1, dead, a.status);
      tc_fence_after();
      uint32_t raw[kHalfN];
      tc_ld32(tmem + lane_off + kTmemS + h * kHalfN, raw);
      tc_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[kSFree]);
#pragma unroll
      for (int x = 0; x < kHalfN; ++x) v[x] = __uint_as_float(raw[x]);
      if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
      __syncwarp();
      float4 *st4 = reinterpret_cast<float4 *>(sXS + xrow);
#pragma unroll
      for (int x = 0; x < kHalfN / 4; ++x)
        st4[x ^ (r & 7)] = make_float4(v[4 * x], v[4 * x + 1], v[4 * x + 2], v[4 * x + 3]);
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) {
        if (t >= 1) mbar_wait_cluster(&bar[kXFree], (t - 1) & 1, dead, a.status);
        bulk_copy_to_peer(x_peer + xwarp, sXS + xwarp, 32 * 128, xfull_peer);
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      }
    };

    uint32_t g = 0, items = 0;
    PieceWalk walk;
    walk.start(a, cluster, nclusters);
    MlaPiece piece, next_piece;
    bool have = walk.next(a, piece);
    if (have) load_q(piece.s);
    while (have) {
      const bool have_next = walk.next(a, next_piece);
      const int s = piece.s, split = piece.split, kv_lo = piece.kv_lo, kv_hi = piece.kv_hi;
      const int nt = (kv_hi - kv_lo + kMN - 1) / kMN;
      {
        const int pfirst = kv_lo / bs, plast = (kv_hi - 1) / bs;
        const int32_t *bt = a.block_table + (size_t)s * a.max_blocks_per_seq;
        int bad = 0;
        for (int lp = pfirst + tid; lp <= plast; lp += kSoftThreads) {
          const int pg = lp < a.max_blocks_per_seq ? __ldg(bt + lp) : -1;
          if (pg < 0 || pg >= a.num_blocks) bad = 1;
        }
        bad = __any_sync(0xffffffffu, bad);
        if (tid == 0) s_bad[items & 1] = 0;
        named_sync(1, kSoftThreads);
        if (bad && lane == 0) atomicOr(&s_bad[items & 1], 1);
        named_sync(1, kSoftThreads);
      }
      const bool item_bad = s_bad[items & 1] != 0;
      // the next piece's queries reach L2 while this one runs
      if (have_next) {
        const char *qn =
            reinterpret_cast<const char *>(a.q) + ((size_t)next_piece.s * kMlaH + r) * kMlaW * 2;
        for (int i = h; i < nch; i += 2)
          asm volatile("prefetch.global.L2 [%0];" ::"l"(qn + chunk_of(rank, i) * 128) : "memory");
      }
      float cur[kHalfN], nxt[kHalfN];
      fetch_send(g, cur);
      float m = -INFINITY, l = 0.f;  // l: this half's share of the row sum
      for (int j = 0; j < nt; ++j) {
        const uint32_t t = g + j;
        const int base = kv_lo + j * kMN + h * kHalfN;
        // the peer's partial scores of tile t
        if (tid == 0) mbar_arrive_expect_tx(&bar[kXFull], X_BYTES);
        mbar_wait_cluster(&bar[kXFull], t & 1, dead, a.status);
        const float4 *xr = reinterpret_cast<const float4 *>(sX + xrow);
        float mxa[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int x = 0; x < kHalfN / 4; ++x) {
          const float4 o4 = xr[x ^ (r & 7)];
          const float e[4] = {o4.x, o4.y, o4.z, o4.w};
#pragma unroll
          for (int y = 0; y < 4; ++y) {
            const int c = 4 * x + y;
            cur[c] = (base + c < kv_hi) ? (cur[c] + e[y]) * a.scale_log2 : -INFINITY;
            mxa[y] = fmaxf(mxa[y], cur[c]);
          }
        }
        // this warp is done with the peer's buffer
        __syncwarp();
        if (lane == 0) mbar_arrive_remote_relaxed(xfree_peer);
        // the two halves of a row meet through shared memory (the first pair
        // barrier keeps this write clear of the partner's previous read)
        named_sync(2 + (warp & 3), 64);
        s_red[tid] = fmaxf(fmaxf(mxa[0], mxa[1]), fmaxf(mxa[2], mxa[3]));
        named_sync(2 + (warp & 3), 64);
        const float mx = fmaxf(s_red[tid], s_red[partner]);
        // then this CTA's partial scores of the next tile go to the peer
        if (j + 1 < nt) fetch_send(t + 1, nxt);
        // P and O were last touched by the value product of tile t - 1
        if (t > 0) mbar_wait(&bar[kODone], (t - 1) & 1, dead, a.status);
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
          const float al = rescale ? alpha : 1.f;
          for (int c0 = 0; c0 < kVHalf / 2; c0 += 32) {
            uint32_t o[32];
            tc_ld32(tmem + lane_off + kTmemO + h * (kVHalf / 2) + c0, o);
            tc_wait_ld();
#pragma unroll
            for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * al);
            tc_st32(tmem + lane_off + kTmemO + h * (kVHalf / 2) + c0, o);
          }
          tc_wait_st();
        }
        const float mu = m == -INFINITY ? 0.f : m;
        float suma[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t pw[kHalfN / 2];
#pragma unroll
        for (int x = 0; x < kHalfN / 2; ++x) {
          const float p0 = fast_exp2(cur[2 * x] - mu);
          const float p1 = fast_exp2(cur[2 * x + 1] - mu);
          suma[x & 3] += p0 + p1;
          const __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
          pw[x] = *reinterpret_cast<const uint32_t *>(&h2);
        }
        tc_st16(tmem + lane_off + kTmemP + h * (kHalfN / 2), pw);
        tc_wait_st();
        l += (suma[0] + suma[1]) + (suma[2] + suma[3]);
        const int tile0 = kv_lo + j * kMN;
        if (j == nt - 1 && kv_hi - tile0 < kMN) {
          // slots past the sequence end may hold anything; 0 * NaN is NaN.
          // S of this tile is done, so its K rows may be overwritten too.
          mbar_wait(&bar[kKVFull0 + t % kMlaStages], (t / kMlaStages) & 1, dead, a.status);
          const int first = kv_hi - tile0;
          uint8_t *vb = sKV + (t % kMlaStages) * STAGE_BYTES;
          const int per_chunk = (kMN - first) * 8;
          for (int e = tid; e < 4 * per_chunk; e += kSoftThreads) {
            const int ci = e / per_chunk, rem = e % per_chunk;
            *reinterpret_cast<uint4 *>(vb + ci * kChunkKV + (first + rem / 8) * 128 + (rem % 8) * 16) =
                make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[kPFull]);
        if (j + 1 < nt) {
#pragma unroll
          for (int x = 0; x < kHalfN; ++x) cur[x] = nxt[x];
        }
      }
      // the next piece's queries, once the last score product of this one is done
      if (have_next) {
        mbar_wait(&bar[kQFree], items & 1, dead, a.status);
        tc_fence_after();
        load_q(next_piece.s);
      }
      // ---- epilogue: the row sum is the two halves' shares
      named_sync(2 + (warp & 3), 64);
      s_red[tid] = l;
      named_sync(2 + (warp & 3), 64);
      l = s_red[tid] + s_red[partner];
      const uint32_t glast = g + nt - 1;
      mbar_wait(&bar[kODone], glast & 1, dead, a.status);
      tc_fence_after();
      const int ns = a.nsplit[s];
      const bool direct = ns == 1;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const uint32_t keep = item_bad ? 0u : 0xffffffffu;
      const long long prow = ((long long)s * kMlaH + r) * a.max_splits + split;
      for (int c0 = 0; c0 < kVHalf / 2; c0 += 32) {
        uint32_t o[32];
        tc_ld32(tmem + lane_off + kTmemO + h * (kVHalf / 2) + c0, o);
        tc_wait_ld();
#pragma unroll
        for (int x = 0; x < 32; ++x) o[x] &= keep;
        const int col = (int)rank * kVHalf + h * (kVHalf / 2) + c0;
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
      if (!direct && rank == 0 && h == 0)
        a.part_lse[prow] = item_bad ? __int_as_float(0x7fc00000) : (l > 0.f ? m + log2f(l) : -INFINITY);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[kOFree]);
      g += nt;
      ++items;
      piece = next_piece;
      have = have_next;
    }
    if (tid == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no remote access to this CTA's shared memory remains
  tc_fence_after();
  if (warp == kMmaWarp) tc_dealloc(tmem, kTmemCols);
}

// One warp per (sequence, head) row: lane q < 32 holds split q's
// log-sum-exp (more splits loop), every lane 16 of the 512 columns.
constexpr int kMergeWarps = 8;
__global__ void __launch_bounds__(32 * kMergeWarps) mla_merge_kernel(const MlaArgs a) {
  const int lane = threadIdx.x & 31;
  const long long rows = (long long)a.num_seqs * kMlaH;
  const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
  pdl_trigger();
  pdl_wait();  // the split partials
  __nv_bfloat16 *out = reinterpret_cast<__nv_bfloat16 *>(a.out);
  for (long long row = gw; row < rows; row += nw) {
    const int s = (int)(row / kMlaH);
    const int ns = a.nsplit[s];
    if (ns == 1) continue;
    uint4 *dst = reinterpret_cast<uint4 *>(out + row * kMlaL) + lane * 2;
    if (ns == 0) {
      dst[0] = make_uint4(0u, 0u, 0u, 0u);
      dst[1] = make_uint4(0u, 0u, 0u, 0u);
      continue;
    }
    const long long base = row * a.max_splits;
    float M = -INFINITY;
    int bad = 0;
    for (int q = lane; q < ns; q += 32) {
      const float v = a.part_lse[base + q];
      if (isnan(v)) bad = 1; else M = fmaxf(M, v);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      bad |= __shfl_xor_sync(0xffffffffu, bad, o);
    }
    float acc[16];
#pragma unroll
    for (int x = 0; x < 16; ++x) acc[x] = 0.f;
    float L = 0.f;
    if (!bad && M != -INFINITY) {
      for (int q = 0; q < ns; ++q) {
        const float w = fast_exp2(a.part_lse[base + q] - M);
        const float4 *src = reinterpret_cast<const float4 *>(a.part_o + (base + q) * kMlaL) + lane * 4;
        L += w;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const float4 x4 = __ldg(src + v);
          acc[4 * v] = fmaf(w, x4.x, acc[4 * v]);
          acc[4 * v + 1] = fmaf(w, x4.y, acc[4 * v + 1]);
          acc[4 * v + 2] = fmaf(w, x4.z, acc[4 * v + 2]);
          acc[4 * v + 3] = fmaf(w, x4.w, acc[4 * v + 3]);
        }
      }
    }
    const float inv = (bad || !(L > 0.f)) ? 0.f : 1.f / L;
    uint32_t w[8];
#pragma unroll
    for (int x = 0; x < 8; ++x) {
      const __nv_bfloat162 h2 = __floats2bfloat162_rn(acc[2 * x] * inv, acc[2 * x + 1] * inv);
      w[x] = *reinterpret_cast<const uint32_t *>(&h2);
    }
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

struct MlaLayout {
  size_t plan, item_end, nsplit, part_o, part_lse, total;
  int max_splits;
};

size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

MlaLayout mla_layout(int num_seqs, int max_seq_len, int kvs) {
  MlaLayout l{};
  // fixed splits: ceil(len / kvs); automatic runs of at least kMinSplit
  // positions: a sequence meets at most ceil(len / kMinSplit) + 1 of them
  l.max_splits = kvs > 0 ? (int)ceil_div_ll(max_seq_len > 0 ? max_seq_len : 1, kvs)
                         : (int)ceil_div_ll(max_seq_len > 0 ? max_seq_len : 1, kMinSplit) + 1;
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

  // page_tiles: every 64-position tile is 64 slots of one page (automatic
  // splits are whole tiles; a fixed split must be a multiple of 64 too)
  a.page_tiles = (block_size % 64 == 0 && kv_split_tokens % 64 == 0) ? 1 : 0;
  const unsigned box_slots = a.page_tiles ? kMN : kMHalf;
  CUtensorMap tm_kv, tm_kv4;
  const unsigned long long kd[3] = {kMlaW, (unsigned long long)block_size,
                                    (unsigned long long)num_blocks};
  const unsigned long long ks[2] = {kMlaW * 2, (unsigned long long)block_size * kMlaW * 2};
  const unsigned int kb[3] = {64, box_slots, 1};
  // the same rows as {64 columns, slots, 9 chunks of 64 columns, pages}: one
  // box of 4 chunks x 64 slots lands as [chunk][slot][128 B]
  const unsigned long long k4d[4] = {64, (unsigned long long)block_size, kMlaW / 64,
                                     (unsigned long long)num_blocks};
  const unsigned long long k4s[3] = {kMlaW * 2, 128, (unsigned long long)block_size * kMlaW * 2};
  const unsigned int k4b[4] = {64, kMN, 4, 1};
  if (!encode_tiled(&tm_kv, kv_cache, PA_BF16, 3, kd, ks, kb, true) ||
      !encode_tiled(&tm_kv4, kv_cache, PA_BF16, 4, k4d, k4s, k4b, true))
    return PA_ERR_CUDA;

  int slot = prof_begin(PA_K_PLAN, st);
  cudaError_t err = launch_dependent(mla_plan_kernel, dim3(1), dim3(1024), 0, st, a);
  prof_end(slot, st);
  if (err != cudaSuccess) return PA_ERR_CUDA;
  slot = prof_begin(PA_K_MLA, st);
  err = launch_dependent(mla_kernel, dim3(2 * a.num_clusters), dim3(kMlaThreads), MLA_SMEM, st,
                         tm_kv, tm_kv4, a);
  prof_end(slot, st);
  if (err != cudaSuccess) return PA_ERR_CUDA;
  slot = prof_begin(PA_K_MLA_MERGE, st);
  long long mblocks = ((long long)num_seqs * kMlaH + kMergeWarps - 1) / kMergeWarps;
  if (mblocks > (long long)num_sms * 16) mblocks = (long long)num_sms * 16;
  err = launch_dependent(mla_merge_kernel, dim3((unsigned)mblocks), dim3(32 * kMergeWarps), 0, st,
                         a);
  prof_end(slot, st);
  if (err != cudaSuccess) return PA_ERR_CUDA;
  return PA_OK;
}

}  // extern "C"
