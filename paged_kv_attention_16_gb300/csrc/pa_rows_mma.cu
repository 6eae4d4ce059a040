// pa_rows_mma.cu -- the bf16 decode row kernel on warp-level tensor-core MMAs.
//
// A decode row is one query token of one request against that request's KV
// pages ("vLLM Triton attention backend deep dive", sections "Technical
// implementation of paged attention" and "Parallel tiled softmax (3D
// kernel)"); it is bound by HBM bandwidth ("vLLM AMD ROCm attention backend
// optimisation", section "Mixed inference workload challenge").  One work
// item is one token x one KV head (its G query heads) x one KV split, as in
// the CUDA-core row kernel (pa_rows.cu), which keeps the fp32 path.
//
// Why warp MMAs here: on CUDA cores a bf16 decode row costs ~50 warp
// instructions per KV position (conversions, 2*G*D FMAs, shuffle
// reductions), which caps the kernel below HBM speed at two resident CTAs
// per SM.  The row's contraction is a dense (G x D) . (D x N) product, so it
// is run as mma.sync m16n8k16 (bf16 in, fp32 accumulate) with the G heads
// padded to 16 rows: ~6 instructions per KV position.  tcgen05 needs at
// least 64 rows per MMA and a round trip through tensor memory for the
// softmax; with G <= 16 real rows the warp-level form keeps S and P in
// registers and needs no tensor-memory traffic.
//
// Layout and flow:
//  * Producer warp: per item, the split's page ids; per stage (64 KV
//    positions), one TMA box per 16 slots of a page and per K / V:
//    {64 dims x 16 slots x D/64 halves} of one KV head, 128-byte swizzled,
//    straight from the page into a ring of shared-memory stages.  A box
//    covers whole 256-byte KV rows (both 64-dim halves): TMA throughput on
//    these gathers is set by the number of boxes, so one box per 16 slots
//    (not one per half) matters.  Stage = [K | V], each [4 boxes][D/64
//    halves][16 rows][128 B].
//  * Compute warp w owns rows 16w..16w+15 of every stage (one TMA box).
//    S = Q K^T: Q fragments stay in registers for the item; K fragments by
//    ldmatrix (conflict-free thanks to the swizzle).  Online softmax in base
//    2 on the accumulator fragment (row max over the 4 lanes of a quad),
//    lazy rescale (the max moves only when it grows by more than 8).  P is
//    packed to bf16 in place as the A operand of O += P V (V by ldmatrix.trans).
//  * KV positions past the split's end: their scores are masked by select;
//    their V rows (which may hold anything, including NaN) are zeroed in
//    shared memory before the PV product, since 0 * NaN is NaN.
//  * End of item: the four warps' (m, l, O) are merged through shared memory
//    and written to the output (single split) or as a split partial.
#include "pa_internal.h"

namespace pa {
namespace {

constexpr float kLazyRescale = 8.0f;

template <int D, int G>
struct MmaRowCfg {
  static constexpr int NWARP = 4;                    // compute warps
  static constexpr int NTHREADS = 32 * (NWARP + 1);  // + producer warp
  static constexpr int ROWS_W = 16;                  // KV rows per warp per stage
  static constexpr int ST = NWARP * ROWS_W;          // KV rows per stage (64)
  static constexpr int BOX = 16;                     // slots per TMA box
  static constexpr int HALVES = D / 64;              // 128-byte swizzle atoms per row
  static constexpr int BOX_BYTES = BOX * 128 * HALVES;  // one box: [halves][16 rows][128 B]
  static constexpr int KV_BYTES = NWARP * BOX_BYTES;     // K (or V) of a stage
  static constexpr int STAGE_BYTES = 2 * KV_BYTES;
  static constexpr int KS = D / 16;                  // k-steps of S = Q K^T
  static constexpr int NT = D / 8;                   // n-tiles of O
  static constexpr int NSLOT = 2;                    // merge scratch slots
  static constexpr int SCR_BYTES = NSLOT * G * D * 4;
  static constexpr int MAX_PAGES = kRowMaxSplit / BOX + 2;
  static constexpr int FPREF_BYTES = (kFastMaxSeqs + 1) * 4;  // decode-only item prefix
  // everything but the ring and the scratch (barriers for up to 6 stages)
  static constexpr int MISC_BYTES = 2 * NSLOT * G * 4 + MAX_PAGES * 4 + 2 * 64 + FPREF_BYTES + 16 * 8 + 16;
  // two resident CTAs per SM: 228 KB less 1 KB reserved each, less the
  // 1024-byte alignment slack
  static constexpr int NSTAGE0 = (233472 / 2 - 1024 - 1024 - 64 - SCR_BYTES - MISC_BYTES) / STAGE_BYTES;
  static constexpr int NSTAGE = NSTAGE0 < 2 ? 2 : (NSTAGE0 > 6 ? 6 : NSTAGE0);
  static constexpr int OFF_RING = 0;  // 1024-byte aligned (swizzle atoms)
  static constexpr int OFF_SCR = OFF_RING + NSTAGE * STAGE_BYTES;
  static constexpr int OFF_ML = OFF_SCR + SCR_BYTES;
  static constexpr int OFF_PAGES = OFF_ML + 2 * NSLOT * G * 4;
  static constexpr int OFF_DESC = OFF_PAGES + MAX_PAGES * 4;
  static constexpr int OFF_FPREF = OFF_DESC + 2 * 64;
  static constexpr int OFF_BAR = (OFF_FPREF + FPREF_BYTES + 15) / 16 * 16;
  static constexpr int NBAR = 2 * NSTAGE + 4;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 1024;  // + alignment slack
  static_assert(2 * (SMEM + 64 + 1024) <= 233472, "two CTAs per SM");
  static constexpr int OPT = (G * D + 127) / 128;         // merge outputs per thread
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
  static_assert(G >= 1 && G <= 16, "at most 16 query heads per KV head");
};

struct MmaRowDesc {
  int done, bad;
  int tok, kvh, i, split, kv_lo, kv_hi, direct, nsplit;
  int mask_lo;      // first visible position (kv_lo is rounded down to a box)
  int qpos;         // the query's position
  long long prow0;  // partial row of head 0 of the group (split partials)
  int nmerge;       // decode-only batches: the row group's splits (merged in-kernel)
};
static_assert(sizeof(MmaRowDesc) <= 64, "descriptor slot is 64 bytes");

__device__ inline void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

__device__ inline void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

// c += a (16x16, row) * b (16x8, col); bf16 inputs, fp32 accumulators.
__device__ inline void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                 uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two floats to a bf16 pair (round to nearest even): `lo` in bits 0..15.
__device__ inline uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&v);
}

// Shared-memory address of 16-byte chunk `c` (0 .. D/8-1) of stage row `r`:
// box r / 16, half c / 8, row r % 16, under the 128-byte swizzle the TMA
// copies apply (chunk index XOR row % 8 inside each 1024-byte atom).
template <int D>
__device__ inline uint32_t swz_addr(uint32_t base, int r, int c) {
  return base + (r >> 4) * (16 * 128 * (D / 64)) + (c >> 3) * (16 * 128) + (r & 15) * 128 +
         (((c & 7) ^ (r & 7)) << 4);
}


// Decode-only batches: the KV positions row s reads (from its window's first
// 16-slot boundary to its end), or -1 when its metadata is bad.
__device__ inline int fast_work(const FwdParams &p, int s) {
  const int ctx = __ldg(p.seq_lens + s);
  const bool qok = __ldg(p.qsl + s) == s && __ldg(p.qsl + s + 1) == s + 1;
  const bool cok = ctx >= 1 && ctx <= p.max_seq_len &&
                   ceil_div_ll(ctx, p.block_size) <= (long long)p.max_blocks_per_seq;
  if (!qok || !cok) return -1;
  return ctx - (window_lo(ctx - 1, p.window) & ~15);
}

__device__ inline unsigned fast_bad_bits(const FwdParams &p, int s) {
  const bool qok = __ldg(p.qsl + s) == s && __ldg(p.qsl + s + 1) == s + 1;
  return qok ? PA_DEV_BAD_SEQLEN : PA_DEV_BAD_QSL;
}

template <int D, int G>
__global__ void __maxnreg__(168) row_mma_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                const __grid_constant__ CUtensorMap tm_v,
                                                const FwdParams p) {
  using C = MmaRowCfg<D, G>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t *ring = smem + C::OFF_RING;
  float *s_o = reinterpret_cast<float *>(smem + C::OFF_SCR);
  float *s_m = reinterpret_cast<float *>(smem + C::OFF_ML);
  float *s_l = s_m + C::NSLOT * G;
  int *s_pages = reinterpret_cast<int *>(smem + C::OFF_PAGES);
  MmaRowDesc *s_desc = reinterpret_cast<MmaRowDesc *>(smem + C::OFF_DESC);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
  uint64_t *empty = full + C::NSTAGE;
  uint64_t *item_full = empty + C::NSTAGE;  // [2]
  uint64_t *item_free = item_full + 2;      // [2]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int S = p.num_seqs, H = p.num_heads, bs = p.block_size;
  __shared__ int s_last;  // this block finished a row group's last split

  if (tid == 0) {
    prefetch_tensor_map(&tm_k);
    prefetch_tensor_map(&tm_v);
    for (int i = 0; i < C::NSTAGE; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], C::NWARP);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&item_full[i], 1);
      mbar_init(&item_free[i], C::NWARP);
    }
    fence_mbar_init();
  }
  __syncthreads();
  pdl_trigger();
  pdl_wait();  // the plan
  bool dead = false;

  if (warp == C::NWARP) {
    // ===================================================== producer warp
    const int Hk = p.num_kv_heads;
    // Decode-only batches: this warp sizes the splits from seq_lens -- the
    // split length spreads the whole KV work over about (8 or, from G = 8,
    // 4) items per resident block, at most fast_nsmax splits a row -- and
    // lays the items out request by request, KV head by KV head (a row
    // group's splits consecutive, so that they finish close together):
    // s_fpref[s] = items before request s (a request with bad metadata has
    // one item per KV head, which writes its row as zeros).
    int *s_fpref = reinterpret_cast<int *>(smem + C::OFF_FPREF);
    int fL = 0;
    if (p.fast) {
      long long wsum = 0;
      int wmax = 0;
      for (int s = lane; s < S; s += 32) {
        const int w = fast_work(p, s);
        s_fpref[s + 1] = w;
        if (w > 0) {
          wsum += w;
          wmax = max(wmax, w);
        }
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
        wmax = max(wmax, __shfl_xor_sync(0xffffffffu, wmax, o));
      }
      const long long target = (G >= 8 ? 4ll : 8ll) * gridDim.x;
      // (down to one 64-position stage: on a small batch one block streams
      // only some tens of GB/s, so a short row still gains from its splits)
      long long L = ceil_div_ll(ceil_div_ll(wsum * Hk, target), 64) * 64;
      L = max(L, (long long)kFastMinSplit);
      L = max(L, ceil_div_ll(ceil_div_ll(wmax, p.fast_nsmax), 64) * 64);
      L = min(L, (long long)kRowMaxSplit);
      if (p.kv_split_tokens > 0 && p.kv_split_tokens < L) L = p.kv_split_tokens;
      fL = (int)L;
      // item counts: lane l takes a contiguous run of requests, an exclusive
      // scan over the lanes, then each lane writes its run's inclusive ends
      // over the works it alone has read
      const int chunk = (S + 31) / 32, s0 = min(S, lane * chunk), s1 = min(S, s0 + chunk);
      int cnt = 0;
      for (int s = s0; s < s1; ++s) {
        const int w = s_fpref[s + 1];
        cnt += w < 0 ? Hk : (int)ceil_div_ll(w, fL) * Hk;
      }
      int run = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, run, o);
        if (lane >= o) run += t;
      }
      run -= cnt;
      for (int s = s0; s < s1; ++s) {
        const int w = s_fpref[s + 1];
        run += w < 0 ? Hk : (int)ceil_div_ll(w, fL) * Hk;
        s_fpref[s + 1] = run;
      }
      if (lane == 0) s_fpref[0] = 0;
      __syncwarp();
    }
    const long long n_items = p.fast ? (long long)s_fpref[S] : p.plan->n[kListRow];
    const long long *row_end = p.list_end + (size_t)kListRow * S;
    unsigned long long *counter = p.fast ? p.fast_work : &p.plan->counter[kListRow];
    uint32_t g = 0, seq = 0;  // stages issued, descriptors written
    // Block b's first item is b (no round trip to the counter); the counter
    // hands out the rest, from gridDim.x on.
    bool first = true;
    for (;;) {
      long long item = 0;
      // (when the items fit the grid, every item is some block's first and
      // the counter is never touched)
      if (lane == 0)
        item = first ? (long long)blockIdx.x
               : n_items <= (long long)gridDim.x ? n_items
                                                 : (long long)gridDim.x + (long long)atomicAdd(counter, 1ull);
      item = __shfl_sync(0xffffffffu, item, 0);
      first = false;
      MmaRowDesc d{};
      int npages = 0, pfirst = 0, s = 0, inval = 0;
      if (item >= n_items) {
        d.done = 1;
      } else if (p.fast) {
        // decode-only batch, no planner: item -> (request, kv head, split)
        int lo = 0, hi = S - 1;
        while (lo < hi) {  // the request whose items include `item`
          const int mid = (lo + hi + 1) >> 1;
          if (s_fpref[mid] <= item) lo = mid; else hi = mid - 1;
        }
        s = lo;
        const int local = (int)(item - s_fpref[s]);
        const int w = fast_work(p, s);
        d.tok = s;
        d.i = 0;
        if (w < 0) {
          // bad metadata: one item per KV head zeroes its heads of row s
          d.kvh = local;
          d.split = 0;
          if (local == 0 && lane == 0) atomicOr(p.status, fast_bad_bits(p, s));
          inval = 1;
          d.direct = 1;
        } else {
          const int ctx = __ldg(p.seq_lens + s);
          const int nsplit = (int)ceil_div_ll(w, fL);
          d.kvh = local / nsplit;
          d.split = local % nsplit;
          d.qpos = ctx - 1;
          d.mask_lo = window_lo(d.qpos, p.window);
          const int s_lo = (d.mask_lo & ~15) + d.split * fL;
          d.kv_hi = min(d.qpos + 1, s_lo + fL);
          d.kv_lo = max(s_lo, d.mask_lo & ~15);
          d.direct = nsplit == 1;
          d.nsplit = p.fast_nsmax;  // the stride between a head's partial rows
          d.nmerge = nsplit;
          d.prow0 = ((long long)s * H + d.kvh * G) * p.fast_nsmax + d.split;
          pfirst = d.kv_lo / bs;
          npages = (d.kv_hi - 1) / bs - pfirst + 1;
        }
      } else {
        const int k = list_find(row_end, S, item);
        const long long start = k ? row_end[k - 1] : 0;
        s = p.ord[k];
        const ReqInfo r = p.req[s];
        const long long local = item - start;
        const long long per_kvh = (long long)r.nsplit * r.q_len;
        d.kvh = (int)(local / per_kvh);
        const int rem = (int)(local % per_kvh);
        d.split = rem / r.q_len;
        d.i = rem % r.q_len;
        d.tok = r.q_start + d.i;
        d.qpos = r.ctx - r.q_len + d.i;  // causal: positions up to qpos
        d.mask_lo = window_lo(d.qpos, p.window);
        const int s_lo = r.kv_base + d.split * r.split_len;
        d.kv_hi = min(d.qpos + 1, s_lo + r.split_len);
        if (max(s_lo, d.mask_lo) >= d.kv_hi) continue;  // no visible position in this split
        d.kv_lo = max(s_lo, d.mask_lo & ~15);  // copy boxes start on 16-slot bounds
        d.direct = (d.mask_lo - r.kv_base) / r.split_len == (d.qpos - r.kv_base) / r.split_len;
        d.nsplit = r.nsplit;
        d.prow0 = r.partial_base + ((long long)d.i * H + d.kvh * G) * r.nsplit + d.split;
        pfirst = d.kv_lo / bs;
        npages = (d.kv_hi - 1) / bs - pfirst + 1;
      }
      // the page list is private to this warp; its earlier readers (TMA
      // issues below) are synchronous, so it is free to overwrite
      const int32_t *bt = p.block_table + (size_t)s * p.max_blocks_per_seq;
      int bad = 0;
      for (int j = lane; j < npages; j += 32) {
        const int lp = pfirst + j;
        const int pid = lp < p.max_blocks_per_seq ? __ldg(bt + lp) : -1;
        if (pid < 0 || pid >= p.num_blocks) bad = 1;
        s_pages[j] = pid;
      }
      d.bad = __any_sync(0xffffffffu, bad);
      if (d.bad && lane == 0) atomicOr(p.status, PA_DEV_BAD_BLOCK);
      d.bad |= inval;
      __syncwarp();
      const int slot = seq & 1;
      if (lane == 0) {
        if (seq >= 2) mbar_wait(&item_free[slot], ((seq >> 1) - 1) & 1, dead, p.status);
        s_desc[slot] = d;
        mbar_arrive(&item_full[slot]);
      }
      ++seq;
      if (d.done) {
        if (p.fast && lane == 0 && n_items > (long long)gridDim.x) {
          // the last block to stop taking items resets the counters
          __threadfence();
          if (atomicAdd(p.fast_work + 1, 1ull) == (unsigned long long)gridDim.x - 1) {
            __threadfence();
            atomicExch(p.fast_work, 0ull);
            atomicExch(p.fast_work + 1, 0ull);
          }
        }
        break;
      }
      if (d.bad) continue;
      // stream the split: per stage, lane -> (box, K|V)
      const int nst = (d.kv_hi - d.kv_lo + C::ST - 1) / C::ST;
      const int bx = lane >> 1, kv = lane & 1;
      for (int j = 0; j < nst; ++j, ++g) {
        const int b = g % C::NSTAGE;
        const int pos0 = d.kv_lo + j * C::ST;
        const int pos = pos0 + bx * C::BOX;
        const bool issue = bx < C::NWARP && pos < d.kv_hi;
        const int nbox = min(C::NWARP, (d.kv_hi - pos0 + C::BOX - 1) / C::BOX);
        if (lane == 0) {
          if (g >= C::NSTAGE) mbar_wait(&empty[b], ((g / C::NSTAGE) - 1) & 1, dead, p.status);
          mbar_arrive_expect_tx(&full[b], nbox * 2 * C::BOX_BYTES);
        }
        __syncwarp();
        if (issue) {
          const int page = s_pages[pos / bs - pfirst];
          uint8_t *dst = ring + b * C::STAGE_BYTES + kv * C::KV_BYTES + bx * C::BOX_BYTES;
          tma_load_5d(dst, kv ? &tm_v : &tm_k, 0, pos % bs, 0, d.kvh, page, &full[b]);
        }
      }
    }
    return;
  }

  // ======================================================= compute warps
  const int gq = lane >> 2, tq = lane & 3;  // fragment row group, column pair
  const int r0 = warp * C::ROWS_W;          // this warp's rows in every stage
  const uint32_t ring_s = smem_u32(ring);
  uint32_t g = 0, seq = 0;
  // Descriptor of item `sq` from the producer's two-slot hand-off.
  auto take = [&](uint32_t sq) {
    const int islot = sq & 1;
    mbar_wait(&item_full[islot], (sq >> 1) & 1, dead, p.status);
    const MmaRowDesc x = s_desc[islot];
    __syncwarp();
    if (lane == 0) mbar_arrive(&item_free[islot]);
    return x;
  };
  // Q of the G heads as A fragments (rows >= G are zero): a0/a2 row gq,
  // a1/a3 row gq + 8; columns 16 ks + 2 tq (+8 for a2/a3).
  uint32_t qa[C::KS][4];
  // ALiBi slopes of rows gq and gq + 8 (base 2; zero without ALiBi)
  float al_lo = 0.f, al_hi = 0.f;
  auto load_q = [&](const MmaRowDesc &x) {
    if (p.alibi) {
      al_lo = gq < G ? __ldg(p.alibi + x.kvh * G + gq) * kLog2eF : 0.f;
      al_hi = gq + 8 < G ? __ldg(p.alibi + x.kvh * G + gq + 8) * kLog2eF : 0.f;
    }
    const uint32_t *qrow = reinterpret_cast<const uint32_t *>(
        reinterpret_cast<const __nv_bfloat16 *>(p.q) + ((size_t)x.tok * H + x.kvh * G) * D);
#pragma unroll
    for (int ks = 0; ks < C::KS; ++ks) {
      const int c = (ks * 16 + 2 * tq) >> 1;  // in bf16 pairs
      qa[ks][0] = gq < G ? __ldg(qrow + gq * (D / 2) + c) : 0u;
      qa[ks][1] = gq + 8 < G ? __ldg(qrow + (gq + 8) * (D / 2) + c) : 0u;
      qa[ks][2] = gq < G ? __ldg(qrow + gq * (D / 2) + c + 4) : 0u;
      qa[ks][3] = gq + 8 < G ? __ldg(qrow + (gq + 8) * (D / 2) + c + 4) : 0u;
    }
  };
  // Decode-only batches: after a split's partial rows are written, the block
  // that finishes a row group's last split merges its splits (log-sum-exp,
  // the sink joining the denominator) into the output and clears the count.
  auto fast_finish = [&](const MmaRowDesc &x) {
    named_sync(1, 128);  // every partial row of this block written
    const size_t grp = (size_t)x.tok * p.num_kv_heads + x.kvh;
    if (tid == 0) {
      // One acquire-release count at GPU scope: it publishes this block's
      // partial rows (ordered before it by the barrier) and, for the block
      // that counts last, makes every other block's rows visible to the merge
      // below (the barrier after it passes that on to the other threads).
      unsigned old;
      asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;"
                   : "=r"(old)
                   : "l"(p.fast_cnt + grp)
                   : "memory");
      s_last = old == (unsigned)x.nmerge - 1 ? 1 : 0;
    }
    named_sync(1, 128);
    if (!s_last) return;
    float *s_wt = s_o;             // [G][64] merge weights of the splits
    float *s_iv = s_o + G * 64;    // [G] reciprocal denominators (0: the row is zero)
    const long long row0 = ((long long)x.tok * H + x.kvh * G) * p.fast_nsmax;
    // The first eight splits' partial values of this thread's elements,
    // loaded now: their latency overlaps the weights' (a short row is one
    // round trip, not two).
    constexpr int EPT = (G * D + 127) / 128;  // elements per thread
    constexpr bool kPre = EPT <= 4;
    float pre[kPre ? EPT : 1][8];
    if constexpr (kPre) {
#pragma unroll
      for (int k = 0; k < EPT; ++k) {
        const int e = tid + 128 * k;
        const bool in = e < G * D;
        const float *src = p.part_o + (row0 + (long long)(e / D) * p.fast_nsmax) * D + e % D;
#pragma unroll
        for (int u = 0; u < 8; ++u) pre[k][u] = in && u < x.nmerge ? __ldcg(src + (size_t)u * D) : 0.f;
      }
    }
    // one warp per head: lane q holds split q's log-sum-exp (two when a row
    // has more than 32 splits)
    for (int hh = warp; hh < G; hh += C::NWARP) {
      const long long r = row0 + (long long)hh * p.fast_nsmax;
      const float v0 = lane < x.nmerge ? __ldcg(p.part_lse + r + lane) : -INFINITY;
      const float v1 = lane + 32 < x.nmerge ? __ldcg(p.part_lse + r + lane + 32) : -INFINITY;
      int badp = (isnan(v0) || isnan(v1)) ? 1 : 0;
      float M = fmaxf(isnan(v0) ? -INFINITY : v0, isnan(v1) ? -INFINITY : v1);
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        badp |= __shfl_xor_sync(0xffffffffu, badp, o);
      }
      const float sink2 = p.sinks ? __ldg(p.sinks + x.kvh * G + hh) * kLog2eF : -INFINITY;
      M = fmaxf(M, sink2);
      const bool any = !badp && M != -INFINITY;
      const float w0 = (any && v0 != -INFINITY) ? fast_exp2(v0 - M) : 0.f;
      const float w1 = (any && v1 != -INFINITY) ? fast_exp2(v1 - M) : 0.f;
      if (lane < x.nmerge) s_wt[hh * 64 + lane] = w0;
      if (lane + 32 < x.nmerge) s_wt[hh * 64 + lane + 32] = w1;
      float L = w0 + w1;
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
      if (any && p.sinks) L += fast_exp2(sink2 - M);
      if (lane == 0) s_iv[hh] = (!any || !(L > 0.f)) ? 0.f : 1.f / L;
    }
    named_sync(1, 128);
    // the partial rows, eight splits at a time (independent loads)
    __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(p.out) + ((size_t)x.tok * H + x.kvh * G) * D;
#pragma unroll
    for (int k = 0; k < EPT; ++k) {
      const int e = tid + 128 * k;
      if (e >= G * D) break;
      const int h = e / D, dd = e % D;
      const float *src = p.part_o + (row0 + (long long)h * p.fast_nsmax) * D + dd;
      float acc = 0.f;
      for (int q0 = 0; q0 < x.nmerge; q0 += 8) {
        float pv[8];
        if (kPre && q0 == 0) {
#pragma unroll
          for (int u = 0; u < 8; ++u) pv[u] = pre[kPre ? k : 0][u];
        } else {
#pragma unroll
          for (int u = 0; u < 8; ++u) pv[u] = q0 + u < x.nmerge ? __ldcg(src + (size_t)(q0 + u) * D) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (q0 + u < x.nmerge) acc = fmaf(s_wt[h * 64 + q0 + u], pv[u], acc);
      }
      dst[e] = __float2bfloat16_rn(acc * s_iv[h]);
    }
    if (tid == 0) p.fast_cnt[grp] = 0u;
  };
  MmaRowDesc nd = take(seq);
  if (!nd.done && !nd.bad) load_q(nd);
  for (;;) {
    const MmaRowDesc d = nd;
    if (d.done) break;
    const int kvh = d.kvh;
    if (d.bad) {
      for (int e = tid; e < G * D; e += 128) {
        const int h = e / D, dd = e % D;
        if (d.direct) {
          reinterpret_cast<__nv_bfloat16 *>(p.out)[((size_t)d.tok * H + kvh * G + h) * D + dd] =
              __float2bfloat16_rn(0.f);
        } else {
          const long long prow = d.prow0 + (long long)h * d.nsplit;
          p.part_o[prow * D + dd] = 0.f;
          if (dd == 0) p.part_lse[prow] = __int_as_float(0x7fc00000);  // NaN: bad split
        }
      }
      if (p.fast && !d.direct) fast_finish(d);
      nd = take(++seq);
      if (!nd.done && !nd.bad) load_q(nd);
      continue;
    }

    float o[C::NT][4];
#pragma unroll
    for (int n = 0; n < C::NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;
    const float sl2 = p.scale_log2;

    const int nst = (d.kv_hi - d.kv_lo + C::ST - 1) / C::ST;
    for (int j = 0; j < nst; ++j, ++g) {
      const int b = g % C::NSTAGE;
      mbar_wait(&full[b], (g / C::NSTAGE) & 1, dead, p.status);
      const int box0 = d.kv_lo + j * C::ST + r0;  // position of this warp's first row
      const int nv = min(C::ROWS_W, d.kv_hi - box0);
      const int hv = d.mask_lo - box0;  // rows below it are outside the window
      const uint32_t kbase = ring_s + b * C::STAGE_BYTES;
      const uint32_t vbase = kbase + C::KV_BYTES;
      if (nv > 0) {
        if (nv < C::ROWS_W) {
          // zero the V rows past the split's end (this warp's box only)
          uint8_t *vb = ring + b * C::STAGE_BYTES + C::KV_BYTES + warp * C::BOX_BYTES;
          for (int e = lane; e < (C::ROWS_W - nv) * C::HALVES * 8; e += 32) {
            const int r = nv + e / (C::HALVES * 8);  // row inside the box
            const int c = e % (C::HALVES * 8);
            *reinterpret_cast<uint4 *>(vb + (c >> 3) * (16 * 128) + r * 128 + (c & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          __syncwarp();
        }
        // ---- S = Q K^T for this warp's 16 rows (two n-tiles of 8)
        float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        {
          const int mi = lane >> 3, rr = lane & 7;
          const int kr = r0 + (mi >> 1) * 8 + rr;  // K row this lane addresses
#pragma unroll
          for (int ks = 0; ks < C::KS; ++ks) {
            uint32_t kb[4];
            ldsm_x4(swz_addr<D>(kbase, kr, ks * 2 + (mi & 1)), kb);
            mma_16816(s[0], qa[ks], kb[0], kb[1]);
            mma_16816(s[1], qa[ks], kb[2], kb[3]);
          }
        }
        // ---- scale, bias, mask, online softmax (rows gq and gq + 8)
        float mx_lo = -INFINITY, mx_hi = -INFINITY;
        const float dist0 = (float)(d.qpos - box0);  // distance back to row 0 of the box
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int col = n * 8 + 2 * tq + (e & 1);
            float v = s[n][e] * sl2;
            if (p.alibi) v += alibi_bias(e < 2 ? al_lo : al_hi, dist0 - (float)col, p.alibi_sqrt);
            s[n][e] = (col < nv && col >= hv) ? v : -INFINITY;
            if (e < 2) mx_lo = fmaxf(mx_lo, s[n][e]);
            else mx_hi = fmaxf(mx_hi, s[n][e]);
          }
        mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
        mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
        if (mx_lo > m_lo + kLazyRescale) {
          const float a = fast_exp2(m_lo - mx_lo);
          l_lo *= a;
#pragma unroll
          for (int n = 0; n < C::NT; ++n) {
            o[n][0] *= a;
            o[n][1] *= a;
          }
          m_lo = mx_lo;
        }
        if constexpr (G > 8) {
          mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
          mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
          if (mx_hi > m_hi + kLazyRescale) {
            const float a = fast_exp2(m_hi - mx_hi);
            l_hi *= a;
#pragma unroll
            for (int n = 0; n < C::NT; ++n) {
              o[n][2] *= a;
              o[n][3] *= a;
            }
            m_hi = mx_hi;
          }
        }
        float pr[2][4];
#pragma unroll
        for (int n = 0; n < 2; ++n) {
          pr[n][0] = fast_exp2(s[n][0] - m_lo);
          pr[n][1] = fast_exp2(s[n][1] - m_lo);
          if constexpr (G > 8) {
            pr[n][2] = fast_exp2(s[n][2] - m_hi);
            pr[n][3] = fast_exp2(s[n][3] - m_hi);
          } else {
            pr[n][2] = pr[n][3] = 0.f;
          }
        }
        l_lo += (pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1]);
        if constexpr (G > 8) l_hi += (pr[0][2] + pr[0][3]) + (pr[1][2] + pr[1][3]);
        // P as the A operand (16 rows x 16 KV positions)
        uint32_t pa[4];
        pa[0] = pack_bf16(pr[0][0], pr[0][1]);
        pa[1] = pack_bf16(pr[0][2], pr[0][3]);
        pa[2] = pack_bf16(pr[1][0], pr[1][1]);
        pa[3] = pack_bf16(pr[1][2], pr[1][3]);
        // ---- O += P V (V fragments transposed out of the row-major stage)
        {
          const int mi = lane >> 3, rr = lane & 7;
          const int vr = r0 + (mi & 1) * 8 + rr;  // V row this lane addresses
#pragma unroll
          for (int np = 0; np < C::NT / 2; ++np) {
            uint32_t vb4[4];
            ldsm_x4_trans(swz_addr<D>(vbase, vr, np * 2 + (mi >> 1)), vb4);
            mma_16816(o[2 * np], pa, vb4[0], vb4[1]);
            mma_16816(o[2 * np + 1], pa, vb4[2], vb4[3]);
          }
        }
        if (nv < C::ROWS_W) fence_proxy_async();  // generic zeroing before the next TMA fill
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[b]);
    }

    // The next item's descriptor and Q now: their latency hides under the
    // epilogue below (the Q registers are free after the last S product).
    nd = take(++seq);
    if (!nd.done && !nd.bad) load_q(nd);

    // ---- this warp's (m, l, O) rows to shared memory
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
    if constexpr (G > 8) {
      l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
      l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);
    }
    // Two slots of scratch: warps 2 and 3 hand their rows to warps 0 and 1,
    // which fold them in (log-sum-exp) and hand the result on; the output
    // stage then merges two slots.  (Four slots would cost a ring stage at
    // G = 8.)
    auto put = [&](int slot) {
      if (gq < G) {
#pragma unroll
        for (int n = 0; n < C::NT; ++n)
          *reinterpret_cast<float2 *>(&s_o[(slot * G + gq) * D + n * 8 + 2 * tq]) =
              make_float2(o[n][0], o[n][1]);
        if (tq == 0) {
          s_m[slot * G + gq] = m_lo;
          s_l[slot * G + gq] = l_lo;
        }
      }
      if constexpr (G > 8) {
        if (gq + 8 < G) {
#pragma unroll
          for (int n = 0; n < C::NT; ++n)
            *reinterpret_cast<float2 *>(&s_o[(slot * G + gq + 8) * D + n * 8 + 2 * tq]) =
                make_float2(o[n][2], o[n][3]);
          if (tq == 0) {
            s_m[slot * G + gq + 8] = m_hi;
            s_l[slot * G + gq + 8] = l_hi;
          }
        }
      }
    };
    // fold slot `slot`'s row `row` (fragment columns c0, c0 + 1 of o) into m, l, o
    auto fold = [&](int slot, int row, float &m, float &l, int c0) {
      const float mp = s_m[slot * G + row], lp = s_l[slot * G + row];
      const float mn = fmaxf(m, mp);
      const float a = m == -INFINITY ? 0.f : fast_exp2(m - mn);
      const float b = mp == -INFINITY ? 0.f : fast_exp2(mp - mn);
      l = l * a + lp * b;
      m = mn;
#pragma unroll
      for (int n = 0; n < C::NT; ++n) {
        const float2 po = *reinterpret_cast<const float2 *>(&s_o[(slot * G + row) * D + n * 8 + 2 * tq]);
        o[n][c0] = o[n][c0] * a + po.x * b;
        o[n][c0 + 1] = o[n][c0 + 1] * a + po.y * b;
      }
    };
    named_sync(1, 128);  // the scratch of the previous item has been read
    if (warp >= 2) put(warp - 2);
    named_sync(1, 128);
    if (warp < 2) {
      if (gq < G) fold(warp, gq, m_lo, l_lo, 0);
      if constexpr (G > 8) {
        if (gq + 8 < G) fold(warp, gq + 8, m_hi, l_hi, 2);
      }
    }
    named_sync(1, 128);  // slots read
    if (warp < 2) put(warp);
    named_sync(1, 128);
    // ---- log-sum-exp merge of the two slots, then output or partial
    const int e0 = tid * C::OPT;
    if (e0 < G * D) {
      const int h = e0 / D, d0 = e0 % D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < C::NSLOT; ++w) M = fmaxf(M, s_m[w * G + h]);
      float L = 0.f, acc[C::OPT];
#pragma unroll
      for (int x = 0; x < C::OPT; ++x) acc[x] = 0.f;
#pragma unroll
      for (int w = 0; w < C::NSLOT; ++w) {
        const float ms = s_m[w * G + h];
        if (ms == -INFINITY) continue;
        const float wt = fast_exp2(ms - M);
        L = fmaf(s_l[w * G + h], wt, L);
#pragma unroll
        for (int x = 0; x < C::OPT; ++x) acc[x] = fmaf(s_o[(w * G + h) * D + d0 + x], wt, acc[x]);
      }
      const float inv = L > 0.f ? 1.f / L : 0.f;
      if (d.direct) {
        const float dinv = sink_inv(p.sinks, kvh * G + h, M, L);  // the row's own output
        __nv_bfloat16 *dst =
            reinterpret_cast<__nv_bfloat16 *>(p.out) + ((size_t)d.tok * H + kvh * G + h) * D + d0;
#pragma unroll
        for (int x = 0; x < C::OPT; ++x) dst[x] = __float2bfloat16_rn(acc[x] * dinv);
      } else {
        const long long prow = d.prow0 + (long long)h * d.nsplit;
#pragma unroll
        for (int x = 0; x < C::OPT; ++x) p.part_o[prow * D + d0 + x] = acc[x] * inv;
        if (d0 == 0) p.part_lse[prow] = L > 0.f ? M + log2f(L) : -INFINITY;
      }
    }
    if (p.fast && !d.direct) fast_finish(d);
  }
}

template <int D, int G>
cudaError_t set_attrs() {
  using C = MmaRowCfg<D, G>;
  static std::atomic<unsigned long long> done{0};
  return set_smem_attrs_once(row_mma_kernel<D, G>, C::SMEM, done);
}

template <typename Fn>
bool dispatch_mma(int head_dim, int group, Fn &&fn) {
#define PA_MMA_CASE(D, G) \
  if (head_dim == D && group == G) { fn.template operator()<D, G>(); return true; }
#define PA_MMA_GROUPS(D) \
  PA_MMA_CASE(D, 1) PA_MMA_CASE(D, 2) PA_MMA_CASE(D, 4) PA_MMA_CASE(D, 8) PA_MMA_CASE(D, 16)
  PA_MMA_GROUPS(64)
  PA_MMA_GROUPS(128)
#undef PA_MMA_GROUPS
#undef PA_MMA_CASE
  return false;
}

struct MmaOccFn {
  int n = 0;
  template <int D, int G>
  void operator()() {
    using C = MmaRowCfg<D, G>;
    if (set_attrs<D, G>() != cudaSuccess) return;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, row_mma_kernel<D, G>, C::NTHREADS,
                                                      C::SMEM) != cudaSuccess)
      n = 0;
  }
};

struct MmaLaunchFn {
  const FwdParams &p;
  const CUtensorMap &tk, &tv;
  int grid;
  cudaStream_t stream;
  cudaError_t err;
  template <int D, int G>
  void operator()() {
    using C = MmaRowCfg<D, G>;
    err = set_attrs<D, G>();
    if (err != cudaSuccess) return;
    err = launch_dependent(row_mma_kernel<D, G>, dim3(grid), dim3(C::NTHREADS), C::SMEM, stream,
                           tk, tv, p);
  }
};

}  // namespace

bool row_mma_supported(int dtype, int head_dim, int group) {
  return dtype == PA_BF16 && (head_dim == 64 || head_dim == 128) &&
         (group == 1 || group == 2 || group == 4 || group == 8 || group == 16);
}

int row_mma_ctas_per_sm(int head_dim, int group) {
  MmaOccFn occ;
  dispatch_mma(head_dim, group, occ);
  return occ.n;
}

cudaError_t launch_row_mma_kernel(const FwdParams &p, const CUtensorMap &tm_k,
                                  const CUtensorMap &tm_v, int grid, cudaStream_t stream) {
  MmaLaunchFn l{p, tm_k, tm_v, grid, stream, cudaErrorInvalidValue};
  dispatch_mma(p.head_dim, p.num_heads / p.num_kv_heads, l);
  return l.err;
}

}  // namespace pa
