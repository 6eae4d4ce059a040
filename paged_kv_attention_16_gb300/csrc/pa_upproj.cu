// pa_upproj.cu -- the up-projection of the non-absorbed MLA prefill / extend
// on the tensor cores, reading the latent rows straight from the paged cache.
//
// "vLLM AMD ROCm attention backend optimisation", section "AITER MLA backend:
// optimised for DeepSeek": prefill and extend attend over the uncompressed
// representation.  Every visible position's latent row c_j (512 wide, the
// first 512 columns of its 576-wide cached row) is decompressed, per head h,
// into a key part W_K,h c_j and a value W_V,h c_j (128 each).  Over the dense
// rows of a batch that is one GEMM, [rows x 512] . [512 x 256 H], whose
// B operand is w_kv read as [256 H, 512] (K-major: head h's 128 key rows,
// then its 128 value rows).
//
// GB300 design (one CTA per SM, persistent over units of 128 dense rows x a
// group of heads):
//   warp 4   TMA producer: the A tile -- 128 dense rows x 512, held in shared
//            memory for every head of the unit -- as 16-row boxes straight
//            from the pages the block table names (dense rows come in
//            16-aligned runs per request, and a 16-row run of positions lies
//            in one page when block_size is a multiple of 16), one barrier per
//            64-column chunk so the next unit's chunk k loads as soon as the
//            last MMA reading this unit's chunk k is done;
//   warps 6-9  TMA producers of B: per head eight chunks of 256 w_kv rows x
//            64 columns through a 3-stage ring, each warp a quarter (64 rows)
//            of every chunk.  A TMA copy holds up the warp that issues it for
//            about as long as the data takes to arrive, so one warp moves
//            only some 20 bytes per clock; a chunk (32 KB) is consumed in
//            about 500 clocks, so four warps share the loads;
//   warp 5   MMA issuer (one thread): per head, D (M = 128, N = 256, fp32 in
//            TMEM) += A_k B_k^T over the eight chunks, into one of two TMEM
//            accumulators, so the epilogue of head h overlaps the MMAs of
//            head h + 1;
//   warps 0-3  epilogue: thread r owns dense row r (TMEM lane r); its 128 key
//            and 128 value entries, rounded to nearest-even bf16, go to that
//            head's key and value rows, two neighbouring lanes storing each
//            whole 32-byte sector together.
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kUpL = 512;          // latent width: the contraction
constexpr int kUpW = 576;          // cached row width (latent + rotary key)
constexpr int kUpN = 256;          // output columns per head: 128 key + 128 value
constexpr int kUpHalf = 128;       // key (or value) columns per head
constexpr int kUpM = 128;          // dense rows per tile
constexpr int kUpKC = kUpL / 64;   // 64-column chunks of the contraction
constexpr int kUpGroups = kUpM / 16;
constexpr int kUpBStages = 3;
constexpr int kUpWWarps = 4;       // warps loading B, a quarter of each chunk each
constexpr int kUpWarpW0 = 6;       // first of them
constexpr int kUpWRows = kUpN / kUpWWarps;
constexpr int kUpThreads = 32 * (kUpWarpW0 + kUpWWarps);  // + 4 epilogue, A producer, MMA
constexpr int kUpHeadsPerUnit = 8; // heads sharing one resident A tile
constexpr uint32_t kUpTmemCols = 512;  // two N = 256 fp32 accumulators

constexpr int A_CHUNK = kUpM * 128;    // 128 rows x 64 columns, bf16
constexpr int B_STAGE = kUpN * 128;    // 256 rows x 64 columns, bf16
constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + kUpKC * A_CHUNK;
constexpr int OFF_BAR = OFF_B + kUpBStages * B_STAGE;
enum UpBar {
  kAFull0 = 0,
  kAFree0 = kAFull0 + kUpKC,
  kBFull0 = kAFree0 + kUpKC,
  kBFree0 = kBFull0 + kUpBStages,
  kAccFull0 = kBFree0 + kUpBStages,
  kAccFree0 = kAccFull0 + 2,
  kUpNumBars = kAccFree0 + 2
};
constexpr int OFF_MISC = OFF_BAR + kUpNumBars * 8;
constexpr int UP_SMEM = OFF_MISC + 64 + 1024;  // + slack for 1024-byte alignment
static_assert(UP_SMEM <= 232448, "shared memory budget");

constexpr uint32_t IDESC_UP = umma_idesc_bf16(kUpM, kUpN, 0);

// Dense row r0 (16-aligned, < total): the request it belongs to is the last
// s with seg[s] <= r0 (requests with no rows share the next one's offset).
__device__ inline int dense_request(const UpprojArgs &a, long long r0) {
  int lo = 0, hi = a.num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(a.seg + mid) <= r0) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(kUpThreads, 1)
    upproj_kernel(const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_w,
                  const UpprojArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t *sA = smem + OFF_A;
  uint8_t *sB = smem + OFF_B;
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
  uint32_t *s_tmem = reinterpret_cast<uint32_t *>(smem + OFF_MISC);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = a.num_heads;
  const int n_hg = (H + kUpHeadsPerUnit - 1) / kUpHeadsPerUnit;
  pdl_trigger();
  pdl_wait();  // the dense offsets
  const long long total = *a.total;
  const long long n_units = ceil_div_ll(total, kUpM) * n_hg;
  if (n_units == 0) return;

  if (tid == 0) {
    prefetch_tensor_map(&tm_c);
    prefetch_tensor_map(&tm_w);
    for (int b = 0; b < kUpNumBars; ++b)
      mbar_init(&bar[b], (b == kAccFree0 || b == kAccFree0 + 1) ? 4u : 1u);
    fence_mbar_init();
  }
  if (warp == 5) tc_alloc(s_tmem, kUpTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  bool dead = false;

  auto unit_of = [&](long long u, long long &r0, int &h0, int &h1) {
    r0 = (u / n_hg) * kUpM;
    h0 = (int)(u % n_hg) * kUpHeadsPerUnit;
    h1 = min(h0 + kUpHeadsPerUnit, H);
  };

  if (warp == 4) {
    // ------------------------------------------------------------- producer
    uint32_t ucount = 0;
    for (long long u = blockIdx.x; u < n_units; u += gridDim.x) {
      long long r0;
      int h0, h1;
      unit_of(u, r0, h0, h1);
      // lane g < 8: the page and first slot of the tile's 16-row group g
      int page = -1, slot = 0;
      bool ok = false;
      if (lane < kUpGroups) {
        const long long rg = r0 + 16 * lane;
        if (rg < total) {
          const int s = dense_request(a, rg);
          const int j0 = (int)(rg - __ldg(a.seg + s));
          const int lp = j0 / a.block_size;
          page = lp < a.max_blocks_per_seq
                     ? __ldg(a.block_table + (size_t)s * a.max_blocks_per_seq + lp)
                     : -1;
          slot = j0 % a.block_size;
          ok = page >= 0 && page < a.num_blocks;
          // (a bad page unmaps the request elsewhere; its rows are never read)
        }
      }
      const unsigned mask = __ballot_sync(0xffffffffu, ok);
      for (int kc = 0; kc < kUpKC; ++kc) {
        // A chunk kc of this unit, once the previous unit's last MMA on it is done
        if (lane == 0) {
          if (ucount > 0) mbar_wait(&bar[kAFree0 + kc], (ucount - 1) & 1, dead, a.status);
          mbar_arrive_expect_tx(&bar[kAFull0 + kc], __popc(mask) * 16 * 128);
        }
        __syncwarp();
        if (ok)
          tma_load_3d(sA + kc * A_CHUNK + lane * 16 * 128, &tm_c, kc * 64, slot, page,
                      &bar[kAFull0 + kc]);
        __syncwarp();
      }
      ++ucount;
    }
  } else if (warp >= kUpWarpW0) {
    // ------------------------------------------------------------- B producers
    // Warp q loads rows [64 q, 64 q + 64) of every chunk; the first also
    // posts the chunk's byte count (the others' bytes may land before it: the
    // stage cannot complete while that arrival is pending).
    const int q = warp - kUpWarpW0;
    if (lane == 0) {
      uint32_t bcount = 0;
      for (long long u = blockIdx.x; u < n_units; u += gridDim.x) {
        long long r0;
        int h0, h1;
        unit_of(u, r0, h0, h1);
        for (int h = h0; h < h1; ++h) {
          for (int kc = 0; kc < kUpKC; ++kc) {
            const int st = bcount % kUpBStages;
            if (bcount >= kUpBStages)
              mbar_wait(&bar[kBFree0 + st], ((bcount / kUpBStages) - 1) & 1, dead, a.status);
            if (q == 0) mbar_arrive_expect_tx(&bar[kBFull0 + st], B_STAGE);
            tma_load_2d(sB + st * B_STAGE + q * kUpWRows * 128, &tm_w, kc * 64,
                        h * kUpN + q * kUpWRows, &bar[kBFull0 + st]);
            ++bcount;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t bcount = 0, ucount = 0, tcount = 0;
      const uint32_t sa = smem_u32(sA), sb = smem_u32(sB);
      for (long long u = blockIdx.x; u < n_units; u += gridDim.x) {
        long long r0;
        int h0, h1;
        unit_of(u, r0, h0, h1);
        for (int h = h0; h < h1; ++h) {
          const uint32_t acc = tcount & 1;
          if (tcount >= 2) mbar_wait(&bar[kAccFree0 + acc], ((tcount >> 1) - 1) & 1, dead, a.status);
          tc_fence_after();
          for (int kc = 0; kc < kUpKC; ++kc) {
            if (h == h0) mbar_wait(&bar[kAFull0 + kc], ucount & 1, dead, a.status);
            const int st = bcount % kUpBStages;
            mbar_wait(&bar[kBFull0 + st], (bcount / kUpBStages) & 1, dead, a.status);
            tc_fence_after();
#pragma unroll
            for (int sub = 0; sub < 4; ++sub) {
              const uint64_t ad = umma_desc_sw128(sa + kc * A_CHUNK + sub * 32, 16, 1024);
              const uint64_t bd = umma_desc_sw128(sb + st * B_STAGE + sub * 32, 16, 1024);
              tc_mma_bf16(tmem + acc * kUpN, ad, bd, IDESC_UP, (kc > 0 || sub > 0) ? 1u : 0u);
            }
            tc_commit(&bar[kBFree0 + st]);
            if (h == h1 - 1) tc_commit(&bar[kAFree0 + kc]);
            ++bcount;
          }
          tc_commit(&bar[kAccFull0 + acc]);
          ++tcount;
        }
        ++ucount;
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------- epilogue
    const int r = tid;  // tile row == TMEM lane
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    uint32_t tcount = 0;
    for (long long u = blockIdx.x; u < n_units; u += gridDim.x) {
      long long r0;
      int h0, h1;
      unit_of(u, r0, h0, h1);
      // Lanes 2k and 2k + 1 (rows 2k and 2k + 1 of the warp) store together:
      // each store of the pair fills one whole 32-byte sector of one row, so
      // no sector is half written (which would make L2 fetch the other half
      // from DRAM).  rowA / rowB: the pair's even and odd row.
      const bool odd = lane & 1;
      const long long rowA = r0 + (r & ~1), rowB = r0 + (r | 1);
      const bool writeA = rowA < total, writeB = rowB < total;
      for (int h = h0; h < h1; ++h) {
        const uint32_t acc = tcount & 1;
        mbar_wait(&bar[kAccFull0 + acc], (tcount >> 1) & 1, dead, a.status);
        tc_fence_after();
#pragma unroll 1
        for (int c0 = 0; c0 < kUpN; c0 += 32) {
          uint32_t raw[32];
          tc_ld32(tmem + lane_off + acc * kUpN + c0, raw);
          tc_wait_ld();
          uint4 ch[4];  // this row's 64 bytes: four 16-byte chunks
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint32_t w[4];
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              const __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(raw[v * 8 + 2 * x]),
                                                              __uint_as_float(raw[v * 8 + 2 * x + 1]));
              w[x] = *reinterpret_cast<const uint32_t *>(&h2);
            }
            ch[v] = make_uint4(w[0], w[1], w[2], w[3]);
          }
          const bool is_k = c0 < kUpHalf;
          const int cc = is_k ? c0 : c0 - kUpHalf;  // first column in the key / value row
          __nv_bfloat16 *baseA = (is_k ? a.k_nope : a.v) + ((size_t)rowA * H + h) * kUpHalf + cc;
          __nv_bfloat16 *baseB = (is_k ? a.k_nope : a.v) + ((size_t)rowB * H + h) * kUpHalf + cc;
#pragma unroll
          for (int pv = 0; pv < 2; ++pv) {
            const uint4 lo = ch[2 * pv], hi = ch[2 * pv + 1];
            const uint4 send = odd ? lo : hi;
            uint4 got;
            got.x = __shfl_xor_sync(0xffffffffu, send.x, 1);
            got.y = __shfl_xor_sync(0xffffffffu, send.y, 1);
            got.z = __shfl_xor_sync(0xffffffffu, send.z, 1);
            got.w = __shfl_xor_sync(0xffffffffu, send.w, 1);
            const int chunk = 2 * pv + (odd ? 1 : 0);
            if (writeA) reinterpret_cast<uint4 *>(baseA)[chunk] = odd ? got : lo;
            if (writeB) reinterpret_cast<uint4 *>(baseB)[chunk] = odd ? hi : got;
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[kAccFree0 + acc]);
        ++tcount;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tc_dealloc(tmem, kUpTmemCols);
}

}  // namespace

cudaError_t launch_upproj(const UpprojArgs &a, const void *kv_cache, const void *w_kv,
                          int num_sms, cudaStream_t stream) {
  CUtensorMap tm_c, tm_w;
  // latent cache rows: dims {576 columns, block_size slots, num_blocks pages},
  // boxes of 64 columns x 16 slots of one page (128-byte swizzle)
  const unsigned long long cd[3] = {kUpW, (unsigned long long)a.block_size,
                                    (unsigned long long)a.num_blocks};
  const unsigned long long cs[2] = {kUpW * 2, (unsigned long long)a.block_size * kUpW * 2};
  const unsigned int cb[3] = {64, 16, 1};
  // w_kv as [num_heads * 256 rows, 512 columns], boxes of 64 columns x 64 rows
  const unsigned long long wd[2] = {kUpL, (unsigned long long)a.num_heads * kUpN};
  const unsigned long long ws[1] = {kUpL * 2};
  const unsigned int wb[2] = {64, kUpWRows};
  if (!encode_tiled(&tm_c, kv_cache, PA_BF16, 3, cd, cs, cb, true) ||
      !encode_tiled(&tm_w, w_kv, PA_BF16, 2, wd, ws, wb, true))
    return cudaErrorInvalidValue;
  static std::atomic<unsigned long long> done{0};
  const cudaError_t e = set_smem_attrs_once(upproj_kernel, UP_SMEM, done);
  if (e != cudaSuccess) return e;
  return launch_dependent(upproj_kernel, dim3(num_sms), dim3(kUpThreads), UP_SMEM, stream, tm_c,
                          tm_w, a);
}

}  // namespace pa
