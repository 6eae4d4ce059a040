// pa_tile.cu -- tensor-core tile kernel for bf16 extend / prefill rows.
//
// "vLLM Triton attention backend deep dive", section "Q-block optimisation":
// several query tokens and heads are packed into one work item so the matrix
// unit is fed and, under GQA, every KV page is read once for the whole group.
// "vLLM AMD ROCm attention backend optimisation", section "Mixed inference
// workload challenge": prefill is compute-bound, extend is hybrid; section
// "Chunked context processing": long KV is walked in fixed chunks whose
// partial results are merged by log-sum-exp.
//
// GB300 design.  One work item = 128 query rows (128/G tokens x the G heads of
// one KV head, GQA-packed so the M = 128 MMA is full and the causal diagonal of
// a tile is only 128/G positions wide) x one KV split.  Per CTA (2 per SM):
//   warps 4, 6  TMA producers: the Q tile (128-byte swizzled boxes of G
//            heads x 128/G tokens), then per 64-position KV tile the K page
//            boxes {64 dims x 16 slots} (warp 4) and the V page boxes
//            {16 slots x all dims} (warp 6) named by the block table, into
//            rings of three K and two V tiles.  A TMA copy holds its issuing
//            warp for about as long as the data takes to land (measured: some
//            20 bytes per clock per warp, whatever the depth of the ring), so
//            one warp could not load both for two CTAs' products.  (The
//            192-wide keys fit only one K stage beside Q: there warp 4 alone
//            loads K of tile j, then V of tile j - 1.)
//   warps 7, 5  tcgen05 issue (one thread each; warp 5 owns TMEM): warp 7
//            S = Q K^T (M=128, N=64, K=head_dim, bf16 in, fp32 in TMEM) into
//            one of two S buffers, running a tile ahead of the softmax; warp
//            5 O += P V with P read from TMEM (N=head_dim, K=64, V read
//            MN-major straight from its page layout).  Issuing a tcgen05.mma
//            holds the thread some 70 clocks, so one thread issuing both
//            kinds held each PV product behind the next S.  (With one
//            producer, warp 5 issues both.)
//   warps 0-3  softmax: thread r owns row r (TMEM lane r): reads its S row
//            (twice -- for the maximum, then for the weights -- where 128
//            registers a thread leave no room to hold 64 scores),
//            masks by select (causal bound, split bound), keeps a base-2
//            online softmax with lazy rescaling of O in TMEM (only when the
//            running max grows by more than 8), stores P as packed bf16 over
//            the first half of the tile's own S buffer (so S of tile j+1 is
//            computed while the softmax works on tile j, and the softmax of
//            tile j+1 overlaps the PV product of tile j), and finally
//            normalises O and stores the row (or a split partial with its
//            log-sum-exp).
// Work items are taken from a device counter (block b's first item is b), so a
// CTA that drew short items takes more of them: the splits of a long request
// are much longer than its causal tail, and a fixed deal by block index gave
// every CTA the same split position.  The lead producer thread takes the next
// item when it needs one and posts it in a small shared-memory ring that the
// other roles read in order.
// Tiles of a split that lie past every row's causal bound are never loaded.
#include "pa_internal.h"

namespace pa {
namespace {

// KV positions per tile.  64: two CTAs per SM with 256 TMEM columns each.
// 128 also works: one CTA per SM then holds two S buffers and O in 512
// columns, but with one softmax pipeline per SM instead of two it measured
// slower (mixed batch 2.00 ms against 1.62 ms).
constexpr int kBN = 64;
constexpr int kBox = 16;           // slots per TMA box
constexpr int kKWarp0 = 4, kMmaWarp = 5, kVWarp = 6, kSWarp = 7;
constexpr int kKStages = 3;        // K tiles in flight per CTA (at most; see TileCfg::KST)
constexpr int kVStages = 2;        // V tiles in flight per CTA
constexpr float kTau = 8.0f;       // lazy-rescale headroom (base 2)
constexpr int kItemRing = 8;       // work items posted ahead by the lead producer
// Dynamic shared memory one CTA may take with `ctas` CTAs per SM (228 KB
// per SM, 1 KB of it reserved per CTA).
constexpr int tile_smem_budget(int ctas) { return 233472 / ctas - 1024; }
constexpr uint32_t kTmemCols = kBN == 64 ? 256 : 512;
// Tensor memory: two S buffers of kBN fp32 columns; P (kBN bf16 per row =
// kBN / 2 columns) is written over the first half of its own S buffer; O after
// them.
constexpr uint32_t kTmemS = 0;        // S buffer b: columns [kBN b, kBN b + kBN)
constexpr uint32_t kTmemO = 2 * kBN;  // O: columns [2 kBN, 2 kBN + head_dim)
constexpr uint32_t kSBufsCols = kTmemO;

// S buffer b = tile & 1: kSFull0 + b (S product done), kPFull0 + b (P
// written over it), kODone0 + b (the PV product that read P is done: the
// buffer is free for S of tile + 2, and V stage b for V of tile + 2).  With
// two or more K stages, kKFree0 + tile % KST (K stage free) also stands for
// "S of the tile is done", so one commit serves both: tcgen05.commit holds
// the issuing thread for some 60 clocks, and one thread issues every product.
// (A barrier can stand for an event of tile t only while no later event on it
// can complete before its waiters have seen it; with one K stage, S of tile
// t + 1 may complete before the softmax has seen S of tile t.)
enum Bar { kQFull = 0, kQFree, kSFull0, kSFull1, kPFull0, kPFull1, kODone0, kODone1, kOFree, kKFull0 };
constexpr int kKFree0 = kKFull0 + kKStages;
constexpr int kVFull0 = kKFree0 + kKStages;
// item ring slot x: kItemFull0 + x (posted), kItemFree0 + x (read by every role)
constexpr int kItemFull0 = kVFull0 + kVStages;
constexpr int kItemFree0 = kItemFull0 + kItemRing;
constexpr int kNumBars = kItemFree0 + kItemRing;

// DQK: width of the query / key rows (the S product's K dimension); DV:
// width of the value / output rows.  They differ for the non-absorbed MLA
// prefill (192 = 128 + 64 rotary, and 128).
template <int DQK, int DV>
struct TileCfg {
  static constexpr int NHQ = DQK / 64;              // 128-byte chunks of a Q / K row
  static constexpr int NHV = DV / 64;               // 128-byte chunks of a V / O row
  static constexpr int Q_BYTES = NHQ * 128 * 128;   // 128 rows x 128 B per chunk
  static constexpr int KV_HALF = kBN * 128;         // one 64-wide chunk of a K tile
  static constexpr int K_BYTES = NHQ * KV_HALF;
  static constexpr int V_BYTES = NHV * KV_HALF;
  static constexpr int V_BOX = NHV * kBox * 128;    // one V box: [chunks][16 rows][128 B]
  // Two CTAs per SM (two softmax pipelines share the tensor pipe), two V
  // stages, and as many K stages, up to three, as fit beside Q.  Where two or
  // more fit, the loads come from three producer warps and the softmax
  // (128 registers a thread) reads S from TMEM twice; where only one fits
  // (the 192-wide keys), a single producer warp interleaves K and V, and the
  // softmax (168 registers) reads S once and holds it.  (A one-stage V ring
  // gave wrong results on the 192-wide keys and is not used.)
  static constexpr int TAIL = kNumBars * 8 + 64 + kItemRing * 8;
  static constexpr bool fits(int k, int v) {
    return Q_BYTES + k * K_BYTES + v * V_BYTES + TAIL <= tile_smem_budget(2);
  }
  static constexpr bool SPLIT = fits(2, kVStages);
  static constexpr int KST = fits(3, kVStages) ? 3 : SPLIT ? 2 : 1;
  static constexpr int VST = kVStages;
  static_assert(VST == 2, "V stage g & 1 is freed by the PV product's kODone0 + (g & 1)");
  static constexpr int THREADS = SPLIT ? 256 : 192;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + KST * K_BYTES;
  static constexpr int OFF_BAR = OFF_V + VST * V_BYTES;
  static constexpr int OFF_MISC = OFF_BAR + kNumBars * 8;
  static constexpr int OFF_ITEMS = OFF_MISC + 64;
  // no alignment slack: the dynamic window is declared 1024-aligned (and
  // the kernel checks that it is)
  static constexpr int SMEM = OFF_ITEMS + kItemRing * 8;
  static_assert(SMEM == OFF_BAR + TAIL, "shared memory layout");
  // roles that read each posted item besides the lead producer: the V warp,
  // the S-issuing and PV-issuing threads and the softmax group; with one
  // producer, one issuing thread and the softmax group
  static constexpr int ITEM_READERS = SPLIT ? 4 : 2;
  static_assert(fits(KST, VST), "shared memory budget");
  static constexpr uint32_t IDESC_S = umma_idesc_bf16(128, kBN, 0);
  static constexpr uint32_t IDESC_PV = umma_idesc_bf16(128, DV, 1);
  static_assert(DQK % 64 == 0 && DQK <= 256 && (DV == 64 || DV == 128), "tile widths");
  static_assert(kSBufsCols + DV <= kTmemCols, "TMEM budget");
};

struct TileItem {
  int s, kvh, split, t0;
  int q_start, q_len, prefix, nsplit, split_len, kv_base;
  long long partial_base;
  int split_lo;           // first position of the split
  int kv_lo, kv_hi, nt;   // loaded range (kv_lo on a 16-slot bound) and its tiles
};

__device__ inline bool decode_tile_item(const FwdParams &p, long long item, int G, TileItem &it) {
  const int S = p.num_seqs;
  const long long *end = p.list_end + (size_t)kListTile * S;
  const int k = list_find(end, S, item);
  const long long local = item - (k ? end[k - 1] : 0);
  it.s = p.ord[k];
  const ReqInfo r = p.req[it.s];
  const int TQ = kTileRows / G;
  const int ntiles = (r.q_len + TQ - 1) / TQ;
  const long long per_kvh = (long long)ntiles * r.nsplit;
  it.kvh = (int)(local / per_kvh);
  const int rem = (int)(local % per_kvh);
  const int qt = ntiles - 1 - rem / r.nsplit;  // tiles nearer the end see more KV: first
  it.split = rem % r.nsplit;
  it.t0 = qt * TQ;
  it.q_start = r.q_start;
  it.q_len = r.q_len;
  it.prefix = r.ctx - r.q_len;
  it.nsplit = r.nsplit;
  it.split_len = r.split_len;
  it.kv_base = r.kv_base;
  it.partial_base = r.partial_base;
  const int t_last = min(it.t0 + TQ, r.q_len) - 1;
  // the first row of the tile sees the lowest positions (sliding window)
  const int lo0 = window_lo(it.prefix + it.t0, p.window);
  it.split_lo = r.kv_base + it.split * r.split_len;
  it.kv_hi = min(it.split_lo + r.split_len, it.prefix + t_last + 1);
  if (max(it.split_lo, lo0) >= it.kv_hi) return false;  // nothing visible in this split
  it.kv_lo = max(it.split_lo, lo0 & ~15);
  it.nt = (it.kv_hi - it.kv_lo + kBN - 1) / kBN;
  return true;
}

// PB64: every 64-position tile is one page's 64 slots (one box per tile).
template <int DQK, int DV, bool PB64>
__global__ void __launch_bounds__((TileCfg<DQK, DV>::THREADS), 2)
    tile_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_kr,
                const FwdParams p) {
  using C = TileCfg<DQK, DV>;
  // 128-byte swizzled operand tiles need 1024-byte alignment.
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw;
  uint8_t *sQ = smem + C::OFF_Q;
  uint8_t *sK = smem + C::OFF_K;
  uint8_t *sV = smem + C::OFF_V;
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
  uint32_t *s_tmem = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  int *s_bad = reinterpret_cast<int *>(smem + C::OFF_MISC + 16);
  volatile long long *s_cur = reinterpret_cast<long long *>(smem + C::OFF_MISC + 32);
  volatile long long *s_items = reinterpret_cast<long long *>(smem + C::OFF_ITEMS);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.num_heads / p.num_kv_heads;
  constexpr bool pb64 = PB64;
  const int H = p.num_heads, bs = p.block_size;
  pdl_trigger();
  pdl_wait();  // the plan, and the row kernel before us in the stream
  const long long n_items = p.plan->n[kListTile];
  if (n_items == 0) return;  // no extend / prefill rows in this batch
  if (smem_u32(smem_raw) & 1023) {  // the same for every thread: all leave together
    if (tid == 0) atomicOr(p.status, PA_DEV_INTERNAL);
    return;
  }

  if (tid == 0) {
    prefetch_tensor_map(&tm_q);
    prefetch_tensor_map(&tm_k);
    prefetch_tensor_map(&tm_v);
    if (p.k_rope_split) prefetch_tensor_map(&tm_kr);
    for (int b = 0; b < kNumBars; ++b) {
      const bool per_warp = b == kPFull0 || b == kPFull1 || b == kOFree;
      const bool item_free = b >= kItemFree0 && b < kItemFree0 + kItemRing;
      mbar_init(&bar[b], per_warp ? 4 : item_free ? C::ITEM_READERS : 1);
    }
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tc_alloc(s_tmem, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  bool dead = false;

  // The item ring.  Entry k is the k-th item index this CTA handles (or
  // n_items: no more); every role walks the entries in order and skips the
  // same empty items, so their counts of items and tiles stay in step.
  unsigned long long *counter = &p.plan->counter[kListTile];
  auto ring_post = [&](uint32_t k) -> long long {  // lead producer, one thread
    const int x = k % kItemRing;
    if (k >= kItemRing) mbar_wait(&bar[kItemFree0 + x], ((k / kItemRing) - 1) & 1, dead, p.status);
    long long v = k == 0 ? (long long)blockIdx.x
                  : n_items <= (long long)gridDim.x ? n_items
                                                    : (long long)gridDim.x + (long long)atomicAdd(counter, 1ull);
    if (dead || v > n_items) v = n_items;  // a timed-out kernel stops taking items
    s_items[x] = v;
    mbar_arrive(&bar[kItemFull0 + x]);
    return v;
  };
  auto ring_take = [&](uint32_t k) -> long long {  // a reading role, one thread
    const int x = k % kItemRing;
    mbar_wait(&bar[kItemFull0 + x], (k / kItemRing) & 1, dead, p.status);
    const long long v = dead ? n_items : s_items[x];
    mbar_arrive(&bar[kItemFree0 + x]);
    return v;
  };

  if (warp == kKWarp0 || (C::SPLIT && warp == kVWarp)) {
    if constexpr (C::SPLIT) {
      // ------------------------------------------------------------- producers
      // A TMA copy holds up the warp that issues it for about as long as its
      // data takes to arrive (some 20 bytes per clock per warp), so the loads
      // come from two warps: Q and K (kKWarp0, which also posts each K tile's
      // byte count) and V (kVWarp).  Each walks the same items and tiles.
      const bool is_v = warp == kVWarp, lead = warp == kKWarp0;
      const int h_lo = 0, h_hi = C::NHQ;
      uint32_t tiles = 0, items = 0;
      for (uint32_t k = 0; is_v || h_lo < h_hi; ++k) {
        long long item = 0;
        if (lane == 0) item = lead ? ring_post(k) : ring_take(k);
        item = __shfl_sync(0xffffffffu, item, 0);
        if (item >= n_items) break;
        TileItem it;
        if (!decode_tile_item(p, item, G, it)) continue;
        const int32_t *bt = p.block_table + (size_t)it.s * p.max_blocks_per_seq;
        PageCache pc;  // the pages of this warp's stream: only moves forward
        pc.start(bt, p.max_blocks_per_seq, it.kv_lo / bs, lane);
        if (lead && lane == 0) {
          if (items > 0) mbar_wait(&bar[kQFree], (items - 1) & 1, dead, p.status);
          mbar_arrive_expect_tx(&bar[kQFull], C::Q_BYTES);
          for (int h = 0; h < C::NHQ; ++h)
            tma_load_3d(sQ + h * 128 * 128, &tm_q, h * 64, it.kvh * G, it.q_start + it.t0,
                        &bar[kQFull]);
        }
        for (int j = 0; j < it.nt; ++j) {
          const uint32_t g = tiles + j;
          // 16-slot boxes, one per lane; or, when a tile is one page's 64
          // slots, a single 64-slot box from lane 0
          const int pos = it.kv_lo + j * kBN + (pb64 ? 0 : lane * kBox);
          const bool need = (pb64 ? lane == 0 : lane < kBN / kBox) && pos < it.kv_hi;
          const int page = pc.get(need ? pos / bs : -1, lane);
          const bool ok = need && page >= 0 && page < p.num_blocks;
          if (need && !ok && !is_v) atomicOr(p.status, PA_DEV_BAD_BLOCK);
          const unsigned mask = __ballot_sync(0xffffffffu, ok);
          if (is_v) {
            const int st = g % C::VST;
            if (lane == 0) {
              if (g >= C::VST)
                mbar_wait(&bar[kODone0 + st], ((g / C::VST) - 1) & 1, dead, p.status);
              mbar_arrive_expect_tx(&bar[kVFull0 + st],
                                    __popc(mask) * C::NHV * (pb64 ? kBN : kBox) * 128);
            }
            __syncwarp();
            // V: [16-slot boxes][chunks][16 rows], or [chunks][64 rows] (each
            // K = 16 step of the PV product is one box)
            if (ok)
              tma_load_5d(sV + st * C::V_BYTES + (pb64 ? 0 : lane * C::V_BOX), &tm_v, 0, pos % bs,
                          0, it.kvh, page, &bar[kVFull0 + st]);
          } else {
            const int st = g % C::KST;
            if (lane == 0) {
              if (g >= C::KST)
                mbar_wait(&bar[kKFree0 + st], ((g / C::KST) - 1) & 1, dead, p.status);
              if (lead)
                mbar_arrive_expect_tx(&bar[kKFull0 + st],
                                      __popc(mask) * C::NHQ * (pb64 ? kBN : kBox) * 128);
            }
            __syncwarp();
            // K: one box per 64-dim chunk ([chunks][64 rows] for the S
            // product's uniform row stride)
            if (ok) {
              for (int h = h_lo; h < h_hi; ++h) {
                // split keys: the last 64 columns are the shared rotary key
                const bool rope = p.k_rope_split && h == C::NHQ - 1;
                tma_load_4d(sK + st * C::K_BYTES + h * C::KV_HALF + (pb64 ? 0 : lane * kBox * 128),
                            rope ? &tm_kr : &tm_k, rope ? 0 : h * 64, rope ? 0 : it.kvh, pos % bs,
                            page, &bar[kKFull0 + st]);
              }
            }
          }
          __syncwarp();
        }
        tiles += it.nt;
        ++items;
      }
    } else {
      // One producer warp (warp 4): Q, then K of tile j and V of tile j - 1
      // (V is consumed a softmax later).
      uint32_t tiles = 0, items = 0;
      for (uint32_t k = 0;; ++k) {
        long long item = 0;
        if (lane == 0) item = ring_post(k);
        item = __shfl_sync(0xffffffffu, item, 0);
        if (item >= n_items) break;
        TileItem it;
        if (!decode_tile_item(p, item, G, it)) continue;
        const int32_t *bt = p.block_table + (size_t)it.s * p.max_blocks_per_seq;
        PageCache kc, vc;  // one per stream: each only moves forward
        kc.start(bt, p.max_blocks_per_seq, it.kv_lo / bs, lane);
        vc.start(bt, p.max_blocks_per_seq, it.kv_lo / bs, lane);
        if (lane == 0) {
          if (items > 0) mbar_wait(&bar[kQFree], (items - 1) & 1, dead, p.status);
          mbar_arrive_expect_tx(&bar[kQFull], C::Q_BYTES);
          for (int h = 0; h < C::NHQ; ++h)
            tma_load_3d(sQ + h * 128 * 128, &tm_q, h * 64, it.kvh * G, it.q_start + it.t0,
                        &bar[kQFull]);
        }
        for (int j = 0; j <= it.nt; ++j) {
#pragma unroll
          for (int which = 0; which < 2; ++which) {
            const int jj = which == 0 ? j : j - 1;
            if (jj < 0 || jj >= it.nt) continue;
            const uint32_t g = tiles + jj;
            const int pos = it.kv_lo + jj * kBN + (pb64 ? 0 : lane * kBox);
            const bool need = (pb64 ? lane == 0 : lane < kBN / kBox) && pos < it.kv_hi;
            // (each cache by name: a reference chosen at run time would move
            // both caches to local memory, a slow round trip per look-up)
            const int page = which == 0 ? kc.get(need ? pos / bs : -1, lane)
                                        : vc.get(need ? pos / bs : -1, lane);
            const bool ok = need && page >= 0 && page < p.num_blocks;
            if (need && !ok) atomicOr(p.status, PA_DEV_BAD_BLOCK);
            const unsigned mask = __ballot_sync(0xffffffffu, ok);
            if (which == 0) {
              const int st = g % C::KST;
              if (lane == 0) {
                if (g >= C::KST)
                  mbar_wait(&bar[kKFree0 + st], ((g / C::KST) - 1) & 1, dead, p.status);
                mbar_arrive_expect_tx(&bar[kKFull0 + st],
                                      __popc(mask) * C::NHQ * (pb64 ? kBN : kBox) * 128);
              }
              __syncwarp();
              if (ok) {
                for (int h = 0; h < C::NHQ; ++h) {
                  const bool rope = p.k_rope_split && h == C::NHQ - 1;
                  tma_load_4d(sK + st * C::K_BYTES + h * C::KV_HALF +
                                  (pb64 ? 0 : lane * kBox * 128),
                              rope ? &tm_kr : &tm_k, rope ? 0 : h * 64, rope ? 0 : it.kvh,
                              pos % bs, page, &bar[kKFull0 + st]);
                }
              }
            } else {
              const int st = g % C::VST;
              if (lane == 0) {
                if (g >= C::VST)
                  mbar_wait(&bar[kODone0 + st], ((g / C::VST) - 1) & 1, dead, p.status);
                mbar_arrive_expect_tx(&bar[kVFull0 + st],
                                      __popc(mask) * C::NHV * (pb64 ? kBN : kBox) * 128);
              }
              __syncwarp();
              if (ok)
                tma_load_5d(sV + st * C::V_BYTES + (pb64 ? 0 : lane * C::V_BOX), &tm_v, 0,
                            pos % bs, 0, it.kvh, page, &bar[kVFull0 + st]);
            }
            __syncwarp();
          }
        }
        tiles += it.nt;
        ++items;
      }
    }
  } else if (warp == kMmaWarp || (C::SPLIT && warp == kSWarp)) {
    // ------------------------------------------------------------- MMA issuers
    // With two producer warps the S products come from their own warp
    // (kSWarp) and the MMA warp issues the PV products: a thread issuing a
    // tcgen05.mma is held some 70 clocks per product, so one thread issuing
    // both kinds made each PV product wait behind the next S and S(j + 2)
    // behind the completion of PV(j).
    const bool s_role = !C::SPLIT || warp == kSWarp, pv_role = !C::SPLIT || warp == kMmaWarp;
    if (lane == 0) {
      uint32_t tiles = 0, items = 0;
      const uint32_t sq = smem_u32(sQ), sk = smem_u32(sK), sv = smem_u32(sV);
      // S of tile g into buffer g & 1, once the PV product of tile g - 2
      // (which read P from that buffer) is done.
      auto issue_s = [&](uint32_t g) {
        const int st = g % C::KST, sb = g & 1;
        mbar_wait(&bar[kKFull0 + st], (g / C::KST) & 1, dead, p.status);
        if (g >= 2) mbar_wait(&bar[kODone0 + sb], ((g - 2) >> 1) & 1, dead, p.status);
        tc_fence_after();
        const uint32_t kb = sk + st * C::K_BYTES;
#pragma unroll
        for (int kk = 0; kk < DQK / 16; ++kk) {
          const int h = kk / 4, sub = kk % 4;
          const uint64_t a = umma_desc_sw128(sq + h * 128 * 128 + sub * 32, 16, 1024);
          const uint64_t b = umma_desc_sw128(kb + h * C::KV_HALF + sub * 32, 16, 1024);
          tc_mma_bf16(tmem + kTmemS + sb * kBN, a, b, C::IDESC_S, kk > 0);
        }
        tc_commit(&bar[kKFree0 + st]);
        if constexpr (C::KST < 2) tc_commit(&bar[kSFull0 + sb]);
      };
      for (uint32_t k = 0;; ++k) {
        const long long item = ring_take(k);
        if (item >= n_items) break;
        TileItem it;
        if (!decode_tile_item(p, item, G, it)) continue;
        if (s_role) {
          mbar_wait(&bar[kQFull], items & 1, dead, p.status);
          issue_s(tiles);
          if (it.nt > 1) issue_s(tiles + 1);
        }
        for (int j = 0; j < it.nt; ++j) {
          const uint32_t g = tiles + j;
          const int pb = g & 1, vs = g % C::VST;
          if (pv_role) {
            mbar_wait(&bar[kPFull0 + pb], (g >> 1) & 1, dead, p.status);
            mbar_wait(&bar[kVFull0 + vs], (g / C::VST) & 1, dead, p.status);
            if (j == 0 && items > 0) mbar_wait(&bar[kOFree], (items - 1) & 1, dead, p.status);
            tc_fence_after();
            const uint32_t vb = sv + vs * C::V_BYTES;
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk) {
              // 16 V rows (K = 16 of the PV product); the leading byte offset
              // steps to the next 64-wide chunk of the row
              const uint64_t b = pb64 ? umma_desc_sw128(vb + kk * 16 * 128, kBN * 128, 1024)
                                      : umma_desc_sw128(vb + kk * C::V_BOX, kBox * 128, 1024);
              tc_mma_bf16_ts(tmem + kTmemO, tmem + kTmemS + pb * kBN + kk * 8, b, C::IDESC_PV,
                             (j > 0 || kk > 0) ? 1u : 0u);
            }
            tc_commit(&bar[kODone0 + pb]);  // also frees V stage vs == pb
          }
          if (s_role && j + 2 < it.nt) issue_s(g + 2);
        }
        if (s_role) tc_commit(&bar[kQFree]);
        tiles += it.nt;
        ++items;
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------- softmax
    const int r = tid;  // row of the tile == TMEM lane
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    uint32_t tiles = 0, items = 0;
    for (uint32_t k = 0;; ++k) {
      // thread 0 reads the ring for the group (all four warps then take the
      // same items, whatever each thread's wait did): slot k & 1 is rewritten
      // only after every thread has passed entry k + 1's barrier
      if (r == 0) s_cur[k & 1] = ring_take(k);
      named_sync(1, 128);
      const long long item = s_cur[k & 1];
      if (item >= n_items) break;
      TileItem it;
      if (!decode_tile_item(p, item, G, it)) continue;
      // Any invalid page in the item's KV range zeroes the item's rows.
      {
        const int pfirst = it.kv_lo / bs, plast = (it.kv_hi - 1) / bs;
        const int32_t *bt = p.block_table + (size_t)it.s * p.max_blocks_per_seq;
        int bad = 0;
        for (int lp = pfirst + r; lp <= plast; lp += 128) {
          const int pg = lp < p.max_blocks_per_seq ? __ldg(bt + lp) : -1;
          if (pg < 0 || pg >= p.num_blocks) bad = 1;
        }
        bad = __any_sync(0xffffffffu, bad);
        if (r == 0) s_bad[items & 1] = 0;
        named_sync(1, 128);
        if (bad && lane == 0) atomicOr(&s_bad[items & 1], 1);
        named_sync(1, 128);
      }
      const bool item_bad = s_bad[items & 1] != 0;
      const int i = it.t0 + r / G;
      const int head = it.kvh * G + r % G;
      const bool row_valid = i < it.q_len;
      const int qpos = it.prefix + i;
      const int row_hi_full = qpos + 1;
      const int row_lo = window_lo(qpos, p.window);
      const int row_hi = row_valid ? min(row_hi_full, it.split_lo + it.split_len) : it.kv_lo;
      // this row has visible positions in the split
      const bool row_in = row_valid && max(row_lo, it.split_lo) < row_hi;
      const float al = p.alibi ? __ldg(p.alibi + head) * kLog2eF : 0.f;  // base-2 slope
      // Warps whose 32 rows are all padding (a decode tile holds G rows) keep
      // the barrier protocol but skip the TMEM traffic and the exponentials.
      const bool warp_active = __any_sync(0xffffffffu, row_in);
      // exp2(s * c - m) as one FFMA needs c > 0 and no bias; otherwise scale
      // (and bias) first, then mask, so that the mask wins whatever c's sign.
      const float c2 = p.scale_log2;
      const bool fold = c2 > 0.f && !p.alibi;
      float m = -INFINITY, l = 0.f;
      // With registers to spare (one producer warp) a tile's 64 scores are
      // read from TMEM once and held; with three producer warps (128
      // registers a thread) S is read twice, once for the row maximum, once
      // for the weights.
      constexpr bool kOnePass = !C::SPLIT;
      for (int j = 0; j < it.nt; ++j) {
        const uint32_t g = tiles + j;
        const int base = it.kv_lo + j * kBN;
        const int pb = g & 1;  // S buffer of this tile; P goes over its first half
        if constexpr (C::KST >= 2)
          mbar_wait(&bar[kKFree0 + g % C::KST], (g / C::KST) & 1, dead, p.status);
        else
          mbar_wait(&bar[kSFull0 + pb], (g >> 1) & 1, dead, p.status);
        tc_fence_after();
        if (warp_active) {
          // raw S of this tile -> scaled (and biased) scores, masked to the
          // row's visible range; column c is position base + c
          const bool cross = __any_sync(0xffffffffu, base + kBN > row_hi || base < row_lo);
          auto scores = [&](float (&x)[kBN], bool transformed) {
            {
              uint32_t raw[kBN];
#pragma unroll
              for (int c0 = 0; c0 < kBN; c0 += 32)
                tc_ld32(tmem + lane_off + kTmemS + pb * kBN + c0,
                        *reinterpret_cast<uint32_t(*)[32]>(raw + c0));
              tc_wait_ld();
#pragma unroll
              for (int c = 0; c < kBN; ++c) x[c] = __uint_as_float(raw[c]);
            }
            if (transformed) return;  // S already holds the biased, masked scores
            if (!fold) {
              if (p.alibi) {
                const float dist0 = (float)(qpos - base);
#pragma unroll
                for (int c = 0; c < kBN; ++c)
                  x[c] = fmaf(x[c], c2, alibi_bias(al, dist0 - (float)c, p.alibi_sqrt));
              } else {
#pragma unroll
                for (int c = 0; c < kBN; ++c) x[c] *= c2;
              }
            }
            if (cross) {
#pragma unroll
              for (int c = 0; c < kBN; ++c) {
                const int pos = base + c;
                x[c] = (pos < row_hi && pos >= row_lo) ? x[c] : -INFINITY;
              }
            }
          };
          // row max with 8 independent chains (a single chain is 64 deep)
          float mxa[8];
          auto row_max = [&](const float (&x)[kBN]) {
#pragma unroll
            for (int c = 0; c < 8; ++c) mxa[c] = x[c];
#pragma unroll
            for (int c = 8; c < kBN; c += 2) mxa[(c >> 1) & 7] = fmax3(mxa[(c >> 1) & 7], x[c], x[c + 1]);
          };
          float sv[kOnePass ? kBN : 1];  // the scores, held in one-pass mode
          if constexpr (kOnePass) {
            scores(*reinterpret_cast<float(*)[kBN]>(sv), false);
            row_max(*reinterpret_cast<float(*)[kBN]>(sv));
          } else {
            float x[kBN];
            scores(x, false);
            row_max(x);
            if (!fold) {
              // a bias (or a scale that cannot fold) costs per score: store
              // the finished scores over S so the second read skips it
#pragma unroll
              for (int c0 = 0; c0 < kBN; c0 += 32)
                tc_st32(tmem + lane_off + kTmemS + pb * kBN + c0,
                        *reinterpret_cast<const uint32_t(*)[32]>(x + c0));
              tc_wait_st();
            }
          }
          float mx = fmax3(fmax3(mxa[0], mxa[1], mxa[2]), fmax3(mxa[3], mxa[4], mxa[5]),
                           fmaxf(mxa[6], mxa[7]));
          if (fold && mx != -INFINITY) mx *= c2;
          float alpha = 1.f;
          bool rescale = false;
          if (mx > m + kTau) {
            alpha = fast_exp2(m - mx);
            l *= alpha;
            m = mx;
            rescale = j > 0;
          }
          if (__any_sync(0xffffffffu, rescale)) {
            // O must hold the product of tile g - 1 before it is rescaled.
            mbar_wait(&bar[kODone0 + (pb ^ 1)], ((g - 1) >> 1) & 1, dead, p.status);
            tc_fence_after();
            const float a = rescale ? alpha : 1.f;
#pragma unroll
            for (int c0 = 0; c0 < DV; c0 += 32) {
              uint32_t raw[32];
              tc_ld32(tmem + lane_off + kTmemO + c0, raw);
              tc_wait_ld();
#pragma unroll
              for (int x = 0; x < 32; ++x) raw[x] = __float_as_uint(__uint_as_float(raw[x]) * a);
              tc_st32(tmem + lane_off + kTmemO + c0, raw);
            }
            tc_wait_st();
          }
          const float mu = m == -INFINITY ? 0.f : m;
          const float cs = fold ? c2 : 1.f;
          float suma[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
          // P of columns [c0, c0 + 32) (16 packed words) goes over S columns
          // [c0 / 2, c0 / 2 + 16), already read.
          auto weights = [&](const float (&x)[kBN]) {
#pragma unroll
            for (int c0 = 0; c0 < kBN; c0 += 32) {
              uint32_t pw[16];
#pragma unroll
              for (int w = 0; w < 16; ++w) {
                // packed (f32x2) multiply-adds: half the issue slots of the
                // scalar ones, on a loop that is issue-bound
                float a0 = -mu, a1 = -mu;
                ffma2(a0, a1, x[c0 + 2 * w], x[c0 + 2 * w + 1], cs, cs);
                const float p0 = fast_exp2(a0), p1 = fast_exp2(a1);
                ffma2(suma[2 * (w & 3)], suma[2 * (w & 3) + 1], p0, p1, 1.f, 1.f);
                const __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
                pw[w] = *reinterpret_cast<const uint32_t *>(&h2);
              }
              tc_st16(tmem + lane_off + kTmemS + pb * kBN + c0 / 2, pw);
            }
          };
          if constexpr (kOnePass) {
            weights(*reinterpret_cast<const float(*)[kBN]>(sv));
          } else {
            float x[kBN];
            scores(x, !fold);
            weights(x);
          }
          tc_wait_st();
          l += ((suma[0] + suma[1]) + (suma[2] + suma[3])) + ((suma[4] + suma[5]) + (suma[6] + suma[7]));
        }
        if (j == it.nt - 1 && it.kv_hi - base < kBN) {
          // Rows past the tile's KV end may hold anything (NaN tails, stale
          // data); P is 0 there but 0 * NaN is NaN, so zero those V rows.
          const int vst = g % C::VST;
          mbar_wait(&bar[kVFull0 + vst], (g / C::VST) & 1, dead, p.status);
          const int first = it.kv_hi - base;
          const int nchunks = (kBN - first) * 8 * C::NHV;
          uint8_t *vs = sV + vst * C::V_BYTES;
          for (int e = r; e < nchunks; e += 128) {
            const int h = e / ((kBN - first) * 8);
            const int rem = e % ((kBN - first) * 8);
            const int row = first + rem / 8;
            const int off = pb64 ? h * (kBN * 128) + row * 128
                                 : (row / kBox) * C::V_BOX + h * (kBox * 128) + (row % kBox) * 128;
            *reinterpret_cast<uint4 *>(vs + off + (rem % 8) * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[kPFull0 + pb]);
      }
      // ---- epilogue: O / l -> output row or split partial
      const uint32_t glast = tiles + it.nt - 1;
      mbar_wait(&bar[kODone0 + (glast & 1)], (glast >> 1) & 1, dead, p.status);
      tc_fence_after();
      const bool write = row_in;
      const bool direct =
          (row_lo - it.kv_base) / it.split_len == (qpos - it.kv_base) / it.split_len;
      // partials are normalised by their own l; a row's own output also
      // counts its head's sink
      const float inv = direct ? sink_inv(p.sinks, head, m, l) : (l > 0.f ? 1.f / l : 0.f);
      const uint32_t keep = item_bad ? 0u : 0xffffffffu;  // bad items write exact zeros
      const size_t tok = (size_t)it.q_start + i;
      const long long prow = it.partial_base + ((long long)i * H + head) * it.nsplit + it.split;
#pragma unroll
      for (int c0 = 0; c0 < DV; c0 += 32) {
        if (!warp_active) break;
        uint32_t raw[32];
        tc_ld32(tmem + lane_off + kTmemO + c0, raw);
        tc_wait_ld();
#pragma unroll
        for (int x = 0; x < 32; ++x) raw[x] &= keep;
        if (write) {
          if (direct) {
            uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(p.out) +
                                                   (tok * H + head) * DV + c0);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint32_t w[4];
#pragma unroll
              for (int x = 0; x < 4; ++x) {
                const __nv_bfloat162 h2 =
                    __floats2bfloat162_rn(__uint_as_float(raw[v * 8 + 2 * x]) * inv,
                                          __uint_as_float(raw[v * 8 + 2 * x + 1]) * inv);
                w[x] = *reinterpret_cast<const uint32_t *>(&h2);
              }
              dst[v] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          } else {
            float4 *dst = reinterpret_cast<float4 *>(p.part_o + prow * DV + c0);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              dst[v] = make_float4(__uint_as_float(raw[4 * v]) * inv,
                                   __uint_as_float(raw[4 * v + 1]) * inv,
                                   __uint_as_float(raw[4 * v + 2]) * inv,
                                   __uint_as_float(raw[4 * v + 3]) * inv);
          }
        }
      }
      if (write && !direct)
        p.part_lse[prow] = item_bad ? __int_as_float(0x7fc00000) : (l > 0.f ? m + log2f(l) : -INFINITY);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[kOFree]);
      tiles += it.nt;
      ++items;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tc_dealloc(tmem, kTmemCols);
}

template <int DQK, int DV, bool PB64>
cudaError_t launch_v(const FwdParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                     const CUtensorMap &tv, const CUtensorMap &tkr, int num_sms,
                     cudaStream_t stream) {
  using C = TileCfg<DQK, DV>;
  auto kern = tile_kernel<DQK, DV, PB64>;
  static std::atomic<unsigned long long> done{0};
  const cudaError_t e = set_smem_attrs_once(kern, C::SMEM, done);
  if (e != cudaSuccess) return e;
  return launch_dependent(kern, dim3(num_sms * 2), dim3(C::THREADS), C::SMEM,
                          stream, tq, tk, tv, tkr, p);
}

template <int DQK, int DV>
cudaError_t launch_d(const FwdParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                     const CUtensorMap &tv, const CUtensorMap &tkr, int num_sms,
                     cudaStream_t stream) {
  return p.tile_page_boxes ? launch_v<DQK, DV, true>(p, tq, tk, tv, tkr, num_sms, stream)
                           : launch_v<DQK, DV, false>(p, tq, tk, tv, tkr, num_sms, stream);
}

}  // namespace

bool tile_kernel_supported(int dtype, int head_dim, int group) {
  return dtype == PA_BF16 && (head_dim == 64 || head_dim == 128) &&
         (group == 1 || group == 2 || group == 4 || group == 8 || group == 16);
}

cudaError_t launch_tile_kernel(const FwdParams &p, const CUtensorMap &tm_q,
                               const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                               const CUtensorMap &tm_kr, int num_sms, cudaStream_t stream) {
  const int dqk = p.head_dim_qk > 0 ? p.head_dim_qk : p.head_dim;
  if (dqk == 128 && p.head_dim == 128)
    return launch_d<128, 128>(p, tm_q, tm_k, tm_v, tm_kr, num_sms, stream);
  if (dqk == 64 && p.head_dim == 64)
    return launch_d<64, 64>(p, tm_q, tm_k, tm_v, tm_kr, num_sms, stream);
  if (dqk == 192 && p.head_dim == 128)
    return launch_d<192, 128>(p, tm_q, tm_k, tm_v, tm_kr, num_sms, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pa
