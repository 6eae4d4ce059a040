// pa_rows.cu -- the fp32 row-streaming kernel on CUDA cores (bf16 rows use
// the warp-MMA kernel of pa_rows_mma.cu): one work item is one query token of
// one request, all G query heads of one KV head (the GQA group), over one KV
// split.  It carries every fp32 row, decode, extend and prefill (fp32 has no
// tensor-core path: no TF32).  Decode rows are bound by HBM bandwidth
// ("vLLM AMD ROCm attention backend optimisation", section "Mixed inference
// workload challenge": decode is memory-bound; "vLLM Triton attention backend
// deep dive", section "Parallel tiled softmax (3D kernel)": the KV walk of a
// single-token query is split across instances that write partial results).
//
// Design (GB300):
//  * Page-gather loader: one thread issues 4-D TMA box copies
//    {head_dim x 1 kv head x 16 slots x 1 page} of K and V straight from the
//    page named by the block table into a ring of shared-memory stages (16-byte
//    aligned rows, fully coalesced HBM reads), completion counted on mbarriers.
//  * GQA packer: the G heads of a KV head live in the same CTA, so every K/V
//    byte fetched from HBM feeds all G heads.
//  * Compute: CUDA-core FFMA in fp32.  Thread (token slot, head group, lane c)
//    holds HPT heads x DPT dims of q and of its output accumulator; the LPT
//    lanes of a token reduce their partial dot products with a transpose-
//    reduce of warp shuffles (HPT-1 + log2(LPT/HPT) shuffles, then HPT
//    broadcasts) instead of HPT full butterflies.
//  * Online softmax per thread over the tokens of its slot, in base 2, with
//    lazy rescaling: the running max moves only when a score exceeds it by
//    more than 8 (weights stay <= 256), so the O(HPT*DPT) rescale is rare.
//  * End of item: the token slots' (m, l, O) are merged through shared memory
//    (a log-sum-exp merge inside the CTA) and written either straight to the
//    output (the row's KV fits one split) or as a split partial.
//  * Persistent fixed grid; items come from a device counter.
#include "pa_internal.h"

namespace pa {
namespace {

constexpr float kLazyRescale = 8.0f;  // base-2 headroom before the max moves

__device__ inline void load_vec(const float *src, float *f) {
  const float4 v = *reinterpret_cast<const float4 *>(src);
  f[0] = v.x;
  f[1] = v.y;
  f[2] = v.z;
  f[3] = v.w;
}

__device__ inline void load_vec(const __nv_bfloat16 *src, float *f) {
  const uint4 v = *reinterpret_cast<const uint4 *>(src);
  f[0] = bf16lo(v.x);
  f[1] = bf16hi(v.x);
  f[2] = bf16lo(v.y);
  f[3] = bf16hi(v.y);
  f[4] = bf16lo(v.z);
  f[5] = bf16hi(v.z);
  f[6] = bf16lo(v.w);
  f[7] = bf16hi(v.w);
}

__device__ inline void store_elem(float *dst, float v) { *dst = v; }
__device__ inline void store_elem(__nv_bfloat16 *dst, float v) { *dst = __float2bfloat16_rn(v); }

template <typename T, int D, int G>
struct RowCfg {
  static constexpr int E = 16 / static_cast<int>(sizeof(T));  // elements per 16-B vector
  static constexpr int HPT = G < 8 ? G : 8;                    // heads per thread
  static constexpr int HG = G / HPT;                           // head groups per token
  static constexpr int DPT0 = (64 / HPT) < (D / 4) ? (64 / HPT) : (D / 4);
  static constexpr int DPT = DPT0 > E ? DPT0 : E;              // dims per thread
  static constexpr int VPT = DPT / E;                          // vectors per thread
  static constexpr int LPT = D / DPT;                          // lanes per (token, head group)
  static constexpr int LANES_TOK = LPT * HG;                   // lanes per token
  static constexpr int TPW = 32 / LANES_TOK;                   // tokens per warp
  static constexpr int NWARP = 4;                              // compute warps
  static constexpr int NTHREADS = 32 * (NWARP + 1);            // + one producer warp
  static constexpr int TPS = TPW * NWARP;                      // tokens per sub-step
  static constexpr int BOX = 16;                               // slots per TMA box
  static constexpr int ST = TPS > 32 ? TPS : 32;               // tokens per stage
  static constexpr int SUB = ST / TPS;                         // sub-steps per stage
  static constexpr int NB0 = HPT >= 8 ? 1 : 8 / HPT;
  static constexpr int NB = SUB < NB0 ? SUB : NB0;             // tokens batched per thread
  static constexpr int NBOX = ST / BOX;
  static constexpr int ROWB = D * static_cast<int>(sizeof(T));
  static constexpr int HALF_STAGE = ST * ROWB;
  static constexpr int STAGE_BYTES = 2 * HALF_STAGE;
  static constexpr int NSTAGE = (64 * 1024 / STAGE_BYTES) < 3 ? 3 : (64 * 1024 / STAGE_BYTES);
  static constexpr int MAX_PAGES = kRowMaxSplit / BOX + 2;
  // shared memory layout
  static constexpr int OFF_RING = 0;
  static constexpr int OFF_SCR = OFF_RING + NSTAGE * STAGE_BYTES;  // per-warp partials
  static constexpr int SCR_BYTES = NWARP * G * D * 4;
  static constexpr int OFF_ML = OFF_SCR + SCR_BYTES;               // per-warp m, l
  static constexpr int OFF_PAGES = OFF_ML + 2 * NWARP * G * 4;
  static constexpr int OFF_DESC = OFF_PAGES + MAX_PAGES * 4;       // two item descriptors
  static constexpr int OFF_BAR = (OFF_DESC + 2 * 64 + 15) / 16 * 16;
  static constexpr int NBAR = 2 * NSTAGE + 4;
  static constexpr int SMEM = OFF_BAR + NBAR * 8;
  static constexpr int OPT = (G * D + 127) / 128;  // outputs per compute thread
  static constexpr int LOG2_HPT = HPT == 1 ? 0 : HPT == 2 ? 1 : HPT == 4 ? 2 : 3;
  static_assert(LPT >= HPT, "transpose-reduce needs at least HPT lanes per token");
  static_assert(32 % LANES_TOK == 0, "token groups must tile a warp");
  static_assert(DPT % E == 0 && D % DPT == 0, "dims must split into 16-byte vectors");
  static_assert(HPT * DPT <= 64, "register budget");
  static_assert(SUB % NB == 0, "batches tile a stage");
  static_assert(D % OPT == 0 || G * D <= 128, "outputs per thread must not straddle heads");
};

// Work item handed from the producer warp to the compute warps.
struct RowDesc {
  int done;       // 1: no more work
  int bad;        // a page of the split is outside the pool
  int tok, kvh, i, split, kv_lo, kv_hi, direct;
  int nsplit;
  int mask_lo;      // first visible position (kv_lo is rounded down to a box)
  int qpos;         // the query's position
  long long prow0;  // partial row of head 0 of the group (split partials)
};

// Sum the HPT partial dot products of the LPT lanes of one (token, head
// group) and hand every lane all HPT totals.
template <int HPT, int LPT, int LOG2_HPT>
__device__ inline void reduce_scores(const float (&part)[HPT], float (&score)[HPT], int lane,
                                     int c) {
  float v[HPT];
#pragma unroll
  for (int h = 0; h < HPT; ++h) v[h] = part[h];
#pragma unroll
  for (int lvl = 0; lvl < LOG2_HPT; ++lvl) {
    const int o = LPT >> (lvl + 1);
    const int n = HPT >> lvl;
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = upper ? v[i] : v[i + n / 2];
      const float keep = upper ? v[i + n / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
#pragma unroll
  for (int o = LPT / HPT / 2; o >= 1; o >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
  // Lane c now holds the total of head c / (LPT / HPT).
  const int base = lane - c;
#pragma unroll
  for (int h = 0; h < HPT; ++h)
    score[h] = __shfl_sync(0xffffffffu, v[0], base + h * (LPT / HPT));
}

template <typename T, int D, int G>
__global__ void __maxnreg__(168) row_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                     const __grid_constant__ CUtensorMap tm_v,
                                                     const FwdParams p) {
  using C = RowCfg<T, D, G>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t *ring = smem + C::OFF_RING;
  float *s_o = reinterpret_cast<float *>(smem + C::OFF_SCR);
  float *s_m = reinterpret_cast<float *>(smem + C::OFF_ML);
  float *s_l = s_m + C::NWARP * G;
  int *s_pages = reinterpret_cast<int *>(smem + C::OFF_PAGES);
  RowDesc *s_desc = reinterpret_cast<RowDesc *>(smem + C::OFF_DESC);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
  uint64_t *empty = full + C::NSTAGE;
  uint64_t *item_full = empty + C::NSTAGE;  // [2]
  uint64_t *item_free = item_full + 2;      // [2]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int S = p.num_seqs, H = p.num_heads, bs = p.block_size;

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
    const long long n_items = p.plan->n[kListRow];
    const long long *row_end = p.list_end + (size_t)kListRow * S;
    uint32_t g = 0, seq = 0;  // stages issued, descriptors written
    for (;;) {
      long long item = 0;
      if (lane == 0) item = (long long)atomicAdd(&p.plan->counter[kListRow], 1ull);
      item = __shfl_sync(0xffffffffu, item, 0);
      RowDesc d{};
      int kvh = 0, npages = 0, pfirst = 0, s = 0;
      if (item >= n_items) {
        d.done = 1;
      } else {
        const int k = list_find(row_end, S, item);
        const long long start = k ? row_end[k - 1] : 0;
        s = p.ord[k];
        const ReqInfo r = p.req[s];
        const long long local = item - start;
        const long long per_kvh = (long long)r.nsplit * r.q_len;
        kvh = (int)(local / per_kvh);
        const int rem = (int)(local % per_kvh);
        d.split = rem / r.q_len;
        d.i = rem % r.q_len;
        d.tok = r.q_start + d.i;
        d.kvh = kvh;
        d.qpos = r.ctx - r.q_len + d.i;  // causal: positions up to qpos
        d.mask_lo = window_lo(d.qpos, p.window);
        const int s_lo = r.kv_base + d.split * r.split_len;
        d.kv_hi = min(d.qpos + 1, s_lo + r.split_len);
        if (max(s_lo, d.mask_lo) >= d.kv_hi) continue;  // no visible position in this split
        d.kv_lo = max(s_lo, d.mask_lo & ~15);  // copy boxes start on 16-slot bounds
        d.direct = (d.mask_lo - r.kv_base) / r.split_len == (d.qpos - r.kv_base) / r.split_len;
        d.nsplit = r.nsplit;
        d.prow0 = r.partial_base + ((long long)d.i * H + kvh * G) * r.nsplit + d.split;
        pfirst = d.kv_lo / bs;
        npages = (d.kv_hi - 1) / bs - pfirst + 1;
      }
      // the page list is private to this warp; reuse it once our earlier TMA
      // issues (which read it) are done -- they are: issue is synchronous
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
      __syncwarp();
      // hand the descriptor over
      const int slot = seq & 1;
      if (lane == 0) {
        if (seq >= 2) mbar_wait(&item_free[slot], ((seq >> 1) - 1) & 1, dead, p.status);
        s_desc[slot] = d;
        mbar_arrive(&item_full[slot]);
      }
      ++seq;
      if (d.done) break;
      if (d.bad) continue;
      // stream the split's K/V stages
      const int nst = (d.kv_hi - d.kv_lo + C::ST - 1) / C::ST;
      for (int j = 0; j < nst; ++j, ++g) {
        const int b = g % C::NSTAGE;
        const int pos0 = d.kv_lo + j * C::ST;
        const int pos = pos0 + lane * C::BOX;
        const bool issue = lane < C::NBOX && pos < d.kv_hi;
        const int nbox = __popc(__ballot_sync(0xffffffffu, issue));
        if (lane == 0) {
          if (g >= C::NSTAGE) mbar_wait(&empty[b], ((g / C::NSTAGE) - 1) & 1, dead, p.status);
          mbar_arrive_expect_tx(&full[b], nbox * 2 * C::BOX * C::ROWB);
        }
        __syncwarp();
        if (issue) {
          const int page = s_pages[pos / bs - pfirst];
          uint8_t *kb = ring + b * C::STAGE_BYTES + lane * C::BOX * C::ROWB;
          tma_load_4d(kb, &tm_k, 0, kvh, pos % bs, page, &full[b]);
          tma_load_4d(kb + C::HALF_STAGE, &tm_v, 0, kvh, pos % bs, page, &full[b]);
        }

      }
    }
    return;
  }

  // ======================================================= compute warps
  const int slot_tok = warp * C::TPW + lane / C::LANES_TOK;  // token slot in a sub-step
  const int hg = (lane % C::LANES_TOK) / C::LPT;
  const int c = lane % C::LPT;
  const int tgrp = lane / C::LANES_TOK;  // token group inside the warp
  uint32_t g = 0;
  for (uint32_t seq = 0;; ++seq) {
    const int islot = seq & 1;
    mbar_wait(&item_full[islot], (seq >> 1) & 1, dead, p.status);
    const RowDesc d = s_desc[islot];
    __syncwarp();
    if (lane == 0) mbar_arrive(&item_free[islot]);
    if (d.done) break;
    const int kvh = d.kvh;
    if (d.bad) {
      for (int e = tid; e < G * D; e += 128) {
        const int h = e / D, dd = e % D;
        if (d.direct) {
          store_elem(reinterpret_cast<T *>(p.out) + ((size_t)d.tok * H + kvh * G + h) * D + dd, 0.f);
        } else {
          const long long prow = d.prow0 + (long long)h * d.nsplit;
          p.part_o[prow * D + dd] = 0.f;
          if (dd == 0) p.part_lse[prow] = __int_as_float(0x7fc00000);  // NaN: bad split
        }
      }
      continue;
    }

    // q of this thread's heads and dims, pre-scaled to base 2
    float qv[C::HPT][C::DPT];
    const T *qrow =
        reinterpret_cast<const T *>(p.q) + ((size_t)d.tok * H + kvh * G + hg * C::HPT) * D;
#pragma unroll
    for (int h = 0; h < C::HPT; ++h)
#pragma unroll
      for (int v = 0; v < C::VPT; ++v) {
        load_vec(qrow + h * D + (c + v * C::LPT) * C::E, &qv[h][v * C::E]);
#pragma unroll
        for (int e = 0; e < C::E; ++e) qv[h][v * C::E + e] *= p.scale_log2;
      }
    // ALiBi slopes of this thread's heads (base 2; zero without ALiBi)
    float al[C::HPT];
#pragma unroll
    for (int h = 0; h < C::HPT; ++h)
      al[h] = p.alibi ? __ldg(p.alibi + kvh * G + hg * C::HPT + h) * kLog2eF : 0.f;
    float m[C::HPT], l[C::HPT], o[C::HPT][C::DPT];
#pragma unroll
    for (int h = 0; h < C::HPT; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.f;
#pragma unroll
      for (int x = 0; x < C::DPT; ++x) o[h][x] = 0.f;
    }

    const int nst = (d.kv_hi - d.kv_lo + C::ST - 1) / C::ST;
    for (int j = 0; j < nst; ++j, ++g) {
      const int b = g % C::NSTAGE;
      mbar_wait(&full[b], (g / C::NSTAGE) & 1, dead, p.status);
      const T *kb = reinterpret_cast<const T *>(ring + b * C::STAGE_BYTES);
      const T *vb = kb + C::ST * D;
#pragma unroll
      for (int sb = 0; sb < C::SUB; sb += C::NB) {
        float sc[C::NB][C::HPT];
        bool valid[C::NB];
        // scores of NB tokens (independent chains)
#pragma unroll
        for (int nb = 0; nb < C::NB; ++nb) {
          const int tl = (sb + nb) * C::TPS + slot_tok;
          const int kpos = d.kv_lo + j * C::ST + tl;
          valid[nb] = kpos < d.kv_hi && kpos >= d.mask_lo;
          float kf[C::DPT];
#pragma unroll
          for (int v = 0; v < C::VPT; ++v)
            load_vec(kb + tl * D + (c + v * C::LPT) * C::E, &kf[v * C::E]);
          float part[C::HPT];
#pragma unroll
          for (int h = 0; h < C::HPT; ++h) {
            float a0 = 0.f, a1 = 0.f;  // even / odd dims, two-lane packed FMA
#pragma unroll
            for (int x = 0; x < C::DPT; x += 2)
              ffma2(a0, a1, qv[h][x], qv[h][x + 1], kf[x], kf[x + 1]);
            part[h] = a0 + a1;
          }
          reduce_scores<C::HPT, C::LPT, C::LOG2_HPT>(part, sc[nb], lane, c);
          if (p.alibi) {
#pragma unroll
            for (int h = 0; h < C::HPT; ++h)
              sc[nb][h] += alibi_bias(al[h], (float)(d.qpos - kpos), p.alibi_sqrt);
          }
        }
        // one max update for the batch (lazy: only when it grows by > 8)
#pragma unroll
        for (int h = 0; h < C::HPT; ++h) {
          float mx = -INFINITY;
#pragma unroll
          for (int nb = 0; nb < C::NB; ++nb)
            if (valid[nb]) mx = fmaxf(mx, sc[nb][h]);
          if (mx > m[h] + kLazyRescale) {
            const float a = fast_exp2(m[h] - mx);
            l[h] *= a;
#pragma unroll
            for (int x = 0; x < C::DPT; ++x) o[h][x] *= a;
            m[h] = mx;
          }
        }
#pragma unroll
        for (int nb = 0; nb < C::NB; ++nb) {
          if (!valid[nb]) continue;
          const int tl = (sb + nb) * C::TPS + slot_tok;
          float vf[C::DPT];
#pragma unroll
          for (int v = 0; v < C::VPT; ++v)
            load_vec(vb + tl * D + (c + v * C::LPT) * C::E, &vf[v * C::E]);
#pragma unroll
          for (int h = 0; h < C::HPT; ++h) {
            const float pr = fast_exp2(sc[nb][h] - m[h]);
            l[h] += pr;
#pragma unroll
            for (int x = 0; x < C::DPT; x += 2) ffma2(o[h][x], o[h][x + 1], pr, pr, vf[x], vf[x + 1]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[b]);
    }

    // ---- merge the token groups of this warp (log-sum-exp via shuffles)
#pragma unroll
    for (int off = C::LANES_TOK; off < 32; off <<= 1) {
#pragma unroll
      for (int h = 0; h < C::HPT; ++h) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m[h], off);
        const float l2 = __shfl_xor_sync(0xffffffffu, l[h], off);
        const float M = fmaxf(m[h], m2);
        const float a1 = m[h] == -INFINITY ? 0.f : fast_exp2(m[h] - M);
        const float a2 = m2 == -INFINITY ? 0.f : fast_exp2(m2 - M);
        l[h] = l[h] * a1 + l2 * a2;
#pragma unroll
        for (int x = 0; x < C::DPT; ++x) {
          const float o2 = __shfl_xor_sync(0xffffffffu, o[h][x], off);
          o[h][x] = o[h][x] * a1 + o2 * a2;
        }
        m[h] = M;
      }
    }
    // ---- across the four warps through shared memory
    named_sync(1, 128);  // the scratch of the previous item has been read
    if (tgrp == 0) {
#pragma unroll
      for (int h = 0; h < C::HPT; ++h) {
        const int head = hg * C::HPT + h;
#pragma unroll
        for (int v = 0; v < C::VPT; ++v)
#pragma unroll
          for (int e = 0; e < C::E; ++e)
            s_o[(warp * G + head) * D + (c + v * C::LPT) * C::E + e] = o[h][v * C::E + e];
        if (c == 0) {
          s_m[warp * G + head] = m[h];
          s_l[warp * G + head] = l[h];
        }
      }
    }
    named_sync(1, 128);
    const int e0 = tid * C::OPT;
    if (e0 < G * D) {
      const int h = e0 / D, d0 = e0 % D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < C::NWARP; ++w) M = fmaxf(M, s_m[w * G + h]);
      float L = 0.f, acc[C::OPT];
#pragma unroll
      for (int x = 0; x < C::OPT; ++x) acc[x] = 0.f;
#pragma unroll
      for (int w = 0; w < C::NWARP; ++w) {
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
        T *dst = reinterpret_cast<T *>(p.out) + ((size_t)d.tok * H + kvh * G + h) * D + d0;
#pragma unroll
        for (int x = 0; x < C::OPT; ++x) store_elem(dst + x, acc[x] * dinv);
      } else {
        const long long prow = d.prow0 + (long long)h * d.nsplit;
#pragma unroll
        for (int x = 0; x < C::OPT; ++x) p.part_o[prow * D + d0 + x] = acc[x] * inv;
        if (d0 == 0) p.part_lse[prow] = L > 0.f ? M + log2f(L) : -INFINITY;
      }
    }
  }
}

template <typename T, int D, int G>
cudaError_t launch_one(const FwdParams &p, const CUtensorMap &tk, const CUtensorMap &tv,
                       int grid, cudaStream_t stream) {
  using C = RowCfg<T, D, G>;
  cudaError_t err = cudaFuncSetAttribute(row_kernel<T, D, G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(row_kernel<T, D, G>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  if (err != cudaSuccess) return err;
  return launch_dependent(row_kernel<T, D, G>, dim3(grid), dim3(C::NTHREADS), C::SMEM, stream,
                          tk, tv, p);
}

template <typename T, int D, int G>
int occupancy_one() {
  using C = RowCfg<T, D, G>;
  if (cudaFuncSetAttribute(row_kernel<T, D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           C::SMEM) != cudaSuccess ||
      cudaFuncSetAttribute(row_kernel<T, D, G>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared) != cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, row_kernel<T, D, G>, C::NTHREADS,
                                                    C::SMEM) != cudaSuccess)
    return 0;
  return n;
}

// Dispatch over (dtype, head_dim, group); Fn is called with the instantiation.
template <typename Fn>
bool dispatch(int dtype, int head_dim, int group, Fn &&fn) {
#define PA_ROW_CASE(T, D, G) \
  if (head_dim == D && group == G) { fn.template operator()<T, D, G>(); return true; }
#define PA_ROW_GROUPS(T, D) \
  PA_ROW_CASE(T, D, 1) PA_ROW_CASE(T, D, 2) PA_ROW_CASE(T, D, 4) PA_ROW_CASE(T, D, 8) \
  PA_ROW_CASE(T, D, 16)
  if (dtype == PA_F32) {
    PA_ROW_GROUPS(float, 64)
    PA_ROW_GROUPS(float, 128)
  }
#undef PA_ROW_GROUPS
#undef PA_ROW_CASE
  return false;
}

struct NopFn {
  template <typename T, int D, int G>
  void operator()() {}
};

struct OccFn {
  int n = 0;
  template <typename T, int D, int G>
  void operator()() { n = occupancy_one<T, D, G>(); }
};

struct LaunchFn {
  const FwdParams &p;
  const CUtensorMap &tk, &tv;
  int grid;
  cudaStream_t stream;
  cudaError_t err;
  template <typename T, int D, int G>
  void operator()() { err = launch_one<T, D, G>(p, tk, tv, grid, stream); }
};

}  // namespace

bool row_kernel_supported(int dtype, int head_dim, int group) {
  NopFn nop;
  return dispatch(dtype, head_dim, group, nop);
}

int row_kernel_ctas_per_sm(int dtype, int head_dim, int group) {
  OccFn occ;
  dispatch(dtype, head_dim, group, occ);
  return occ.n;
}

cudaError_t launch_row_kernel(const FwdParams &p, const CUtensorMap &tm_k,
                              const CUtensorMap &tm_v, int grid, cudaStream_t stream) {
  LaunchFn l{p, tm_k, tm_v, grid, stream, cudaErrorInvalidValue};
  dispatch(p.dtype, p.head_dim, p.num_heads / p.num_kv_heads, l);
  return l.err;
}

}  // namespace pa
