// Fused decode step: score a few query rows against every visible block key
// and select each row's top blocks into its mask, in one launch.
//
// The operation is the scorer's and the selector's, unchanged (PR #1160
// "score QSA token-indexer blocks in native CUDA": S[p, b] = sum_h relu(q_h .
// k_b) / sqrt(128) over the row's visible blocks, relu per head before the
// head sum, NaN kept; PR #1178 "select QSA indexer blocks", "Exact semantics":
// the keep = min(budget / 4, blocks) highest scores under (score descending,
// block index ascending, -0.0 == +0.0), their tokens and the row's tail
// visible).  metrale layers/qsa.rs decode_select runs the two back to back
// for each decode step; at one row per step the second launch and the
// selector's single-CTA passes over the row are most of the step's time, so
// here the row's scoring CTAs also do the selection:
//
//  1. each CTA scores a contiguous range of at most 256 of the row's blocks
//     on the tensor cores: warp 0 copies them with TMA (128-byte swizzle), one
//     128-block tile per stage, issued as soon as the launch may read memory;
//     warps 2-3 prepare the row's four query heads ((1 + w) RMSNorm, RoPE at
//     the row's position) as the 16 x 128 operand of the MMA (rows 4..15
//     zero); warp 1 issues tcgen05.mma M128 N16 K16 x 8 per tile (keys on M,
//     heads on N) into its own TMEM accumulator; warps 4-7 first pool the
//     newly complete blocks of the range (writing each into its landed tile
//     as well, since the copy may have read the old key), then read the
//     accumulators (one block per TMEM lane, its four heads in four columns),
//     apply relu, the head sum in order 0..3 and the scale, and keep the
//     scores in shared memory;
//  2. the epilogue warps add each score's top-16-bit order-key bin into the
//     row's histogram in the workspace (one add per distinct bin per warp);
//  3. the row's CTAs meet at a grid barrier (the launch is cooperative, so
//     they are co-resident; the wait is bounded);
//  4. every CTA reads the row's histogram, finds the bin holding the keep-th
//     key (a non-finite score shows up in the 256 outer bins), appends that
//     bin's keys with their block indices to the row's candidate list, takes
//     an atomic ticket, and writes the mask bytes of its other blocks;
//  5. the last CTA of the row to take its ticket zeroes the row's workspace
//     for the next call (its stores drain while it works on), runs the
//     remaining radix rounds (8 and 8 bits) over the candidates, cuts exact
//     ties at the final key by radix rounds on the block index (lowest kept),
//     and writes the candidates' mask bytes.
//
// Workspace per row: the 65536-bin histogram (interleaved over L2 lines, see
// hist_slot; only the bins between the row's lowest and highest are touched),
// a few counters, and room for tokens / 4 candidates (key, block index).  It must be zero before the first call; every call that completes
// leaves it zero.  A call that reports an error may leave it dirty: zero it
// again before the next call.
#include "qsa_device.cuh"
#include "qsa_launch.h"
#include "qsa_select_util.cuh"
#include "qsa_tc_device.cuh"
#include "qsa_tma.h"

namespace qsa {

namespace {

constexpr int kDecThreads = 256;
constexpr int kDecTile = 128;                                 // blocks per key tile: the MMA's M
constexpr int kDecStages = 2;                                 // tiles per CTA, one stage each
constexpr int kDecMaxBpc = kDecStages * kDecTile;             // blocks per CTA
constexpr uint32_t kDecTileBytes = kDecTile * kHeadDim * 2;   // 32 KiB
constexpr uint32_t kDecHalfBytes = kDecTile * 64 * 2;         // one 64-dim box: 16 KiB
constexpr int kDecN = 16;                                     // MMA N: 4 heads, 12 zero rows
constexpr uint32_t kDecTmemCols = 32;                         // one 16-column accumulator per tile
constexpr int kDecCandCache = 4096;  // candidates the last CTA copies into shared memory
constexpr long long kDecSpinLimit = 4000000000LL;  // ~2 s of SM clock
// instruction descriptor, kind::f16: D f32, A and B bf16, both K-major, M = 128, N = 16
constexpr uint32_t kDecIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                               ((uint32_t)(kDecN >> 3) << 17) | ((uint32_t)(kDecTile >> 4) << 24);

constexpr int kDecBinBits = 16;                 // first-level bins: the order key's top 16 bits
constexpr uint32_t kDecBins = 1u << kDecBinBits;
constexpr uint32_t kDecHiBad = 0xFF80u;  // a positive non-finite score's bins start here
constexpr uint32_t kDecLoBad = 0x0080u;  // ... and a negative one's end below this
constexpr uint32_t kDecZeroBin = 0x8000u;  // the bin of a +0.0 score (relu's zero; -0.0 folds in)

struct RowHdr {  // per row, at the start of the row's workspace
  uint32_t hist0[kDecBins];  // bin b's count at hist_slot(b)
  uint32_t arrive;  // CTAs whose histogram is in
  uint32_t binrev;  // kDecBins - 1 minus the lowest bin other than kDecZeroBin any key landed in
  // candidates listed (low 32 bits) and CTAs done writing their blocks (high
  // 32 bits): the last CTA's ticket returns the list's length with it
  unsigned long long tc;
  uint32_t maxbin[8];  // the highest bin any key landed in (CTA y adds to slot y % 8)
  uint32_t lowbad;     // a key landed below kDecLoBad (a negative non-finite score)
  uint32_t pad[51];
};
static_assert(sizeof(RowHdr) == 262400, "qsa_decode_workspace_bytes reports this size");

// A row's scores crowd into a range of neighbouring bins, and every CTA of the
// row adds into them.  Bins go in runs of eight (one 32-byte sector), and run
// r sits in 128-byte line r mod 2048 (sector r / 2048 of it): each line holds
// one run of the crowded range rather than four, while a read of consecutive
// bins still uses whole sectors.
__device__ __forceinline__ uint32_t hist_slot(uint32_t bin) {
  return (((bin >> 3) & 2047u) << 5) | ((bin >> 14) << 3) | (bin & 7u);
}

// Keys of the keep-th largest score and everything above it sit within a few
// hundred bins (two octaves of score) of the row's highest one, so each CTA
// first reads only this many bins below it, and lower ones only if they fall
// short.
constexpr int kDecWindow = 256;
constexpr int kDecChunk = 4096;  // bins per later read

struct DecSmem {  // selection scratch, laid over the key ring once scoring is done
  uint32_t hist0[kDecChunk];
  uint32_t hist1[256];
  uint32_t hist2[256];
  uint32_t warp_tot[kDecThreads / 32];
  int32_t sel_bin;
  uint32_t sel_above;
  uint32_t sel_total;
  uint32_t row_max, row_min;  // the row's highest and lowest bin
  int32_t flag;
  uint32_t rule_prefix;
  uint32_t rule_shift;
  int32_t rule_cut;
  uint32_t nl;         // candidates listed over the row (the last CTA)
  int32_t rsel[4];     // each candidate round's bin ...
  uint32_t rabove[4];  // ... and the keys above it
};
constexpr size_t kDecCandOff = (sizeof(DecSmem) + 127) & ~size_t(127);
static_assert(kDecCandOff + (size_t)kDecCandCache * 8 <= kDecStages * kDecTileBytes,
              "selection scratch overflows the ring");

// Shared memory, from a 1024-byte aligned base: the key ring (the selection's
// scratch once the keys are scored), the query operand, the scores, control.
constexpr uint32_t kDecQOff = kDecStages * kDecTileBytes;
constexpr uint32_t kDecQBytes = kDecN * kHeadDim * 2;  // two 64-dim halves of 2 KiB
constexpr uint32_t kDecScOff = kDecQOff + kDecQBytes;
constexpr uint32_t kDecCtrlOff = kDecScOff + kDecMaxBpc * 4;

struct DecCtrl {
  uint64_t full[kDecStages];
  uint64_t tfull[kDecStages];
  uint64_t qready;
  uint64_t pooled;
  uint64_t drain;
  uint32_t tmem_base;
  int32_t abort;
  int32_t issued;        // key tiles the producer issued
  uint32_t maxbin;       // this CTA's highest bin
  uint32_t minbin;       // ... and lowest
  uint32_t low;          // a key of this CTA landed below bin 8
};
constexpr size_t kDecSmemBytes = kDecCtrlOff + sizeof(DecCtrl) + 1024;  // + alignment slack

__device__ __forceinline__ void red_add_release_gpu(uint32_t *p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// A plain load kept in program order after the loads issued before it (they
// are inline assembly too), so that its use does not delay their issue.
__device__ __forceinline__ int32_t ld_global_s32(const int32_t *p) {
  int32_t v;
  asm volatile("ld.global.s32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__global__ void __launch_bounds__(kDecThreads, 3)
decode_fused_kernel(const __grid_constant__ CUtensorMap kmap, const ScoreArgs a, int32_t keep_max,
                    uint8_t *__restrict__ mask, uint8_t *__restrict__ ws, int64_t row_ws_bytes,
                    int32_t bpc, const PoolArgs pa) {
  extern __shared__ uint8_t dec_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(dec_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *ring = smem;
  DecCtrl &C = *reinterpret_cast<DecCtrl *>(smem + kDecCtrlOff);
  float *sc_s = reinterpret_cast<float *>(smem + kDecScOff);
  DecSmem &D = *reinterpret_cast<DecSmem *>(ring);  // selection scratch, once the keys are scored
  uint32_t *ck_s = reinterpret_cast<uint32_t *>(ring + kDecCandOff);  // cached candidate keys
  uint32_t *ci_s = ck_s + kDecCandCache;                              // ... and block indices
  const uint32_t sRing = sm32(ring), sQ = sm32(smem + kDecQOff);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = blockIdx.x, y = blockIdx.y, ny = gridDim.y;

  // ---- set-up while the previous launch finishes: barriers, the zero rows of
  // the query operand, TMEM; and L2 warmed with this CTA's key tiles and the
  // row's query heads.  A prefetch brings nothing into the CTA and L2 is where
  // every write lands, so the copies issued after the dependency wait still
  // read whatever the previous launch wrote, only sooner.
  if (tid == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&kmap)) : "memory");
    const int32_t np = a.tokens >> 2, cp = y * bpc;
    for (int t = 0; t < (max(0, min(bpc, np - cp)) + kDecTile - 1) / kDecTile; ++t) {
      asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                       reinterpret_cast<uint64_t>(&kmap)),
                   "r"(0), "r"(cp + t * kDecTile)
                   : "memory");
      asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                       reinterpret_cast<uint64_t>(&kmap)),
                   "r"(64), "r"(cp + t * kDecTile)
                   : "memory");
    }
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a.q + (int64_t)row * a.q_stride),
                 "r"((uint32_t)(kHeads * kHeadDim * 2))
                 : "memory");
    for (int s = 0; s < kDecStages; ++s) {
      mbar_init(sm32(&C.full[s]), 1);
      mbar_init(sm32(&C.tfull[s]), 1);
    }
    mbar_init(sm32(&C.qready), 64);  // the query-prep threads
    mbar_init(sm32(&C.pooled), 128);  // the epilogue threads, once they have pooled
    mbar_init(sm32(&C.drain), 1);
    C.abort = 0;
    C.issued = 0;
    C.maxbin = 0u;
    C.minbin = kDecBins - 1u;
    C.low = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  reinterpret_cast<uint4 *>(smem + kDecQOff)[tid] = make_uint4(0u, 0u, 0u, 0u);  // 4 KiB
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     sm32(&C.tmem_base)),
                 "r"(kDecTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  grid_dependency_sync();
  // warps 2-3 issue the loads of the query row and the norm weight before the
  // position's: only the RoPE rows wait for it
  uint4 qv = make_uint4(0u, 0u, 0u, 0u), qw8 = make_uint4(0u, 0u, 0u, 0u);
  if (warp == 2 || warp == 3) {
    const int h = (warp - 2) * 2 + (lane >> 4), g = lane & 15;
    qv = ldg_nc_v4(a.q + (int64_t)row * a.q_stride + h * kHeadDim + 8 * g);
    qw8 = ldg_nc_v4(a.q_norm_w + 8 * g);
  }

  const int32_t n_max = a.tokens >> 2;
  const int c0 = y * bpc;
  if (warp == 0 && lane == 0) {
    // ---- TMA producer: every tile of the range, one stage each, issued before
    // the position is read (a row that sees fewer blocks ignores the rest)
    const int ntiles = (max(0, min(bpc, n_max - c0)) + kDecTile - 1) / kDecTile;
    int issued = 0;
    for (int t = 0; t < ntiles; ++t) {
      const int32_t b0 = c0 + t * kDecTile;
      const uint32_t fb = sm32(&C.full[t]);
      mbar_expect_tx(fb, kDecTileBytes);
      tma_load_2d(sRing + t * kDecTileBytes, &kmap, 0, b0, fb);
      tma_load_2d(sRing + t * kDecTileBytes + kDecHalfBytes, &kmap, 64, b0, fb);
      issued = t + 1;
    }
    C.issued = issued;
  }

  // the position is read by every other role
  const int32_t p = ld_global_s32(a.pos + row);
  const bool valid = p >= 0 && p < a.tokens;
  const int32_t n = valid ? (p + 1) >> 2 : 0;
  const int c1 = min(n, c0 + bpc);
  const int cnt = max(0, c1 - c0);
  const int tiles = (cnt + kDecTile - 1) / kDecTile;
  // the newly complete blocks in this CTA's range (every row's CTAs pool them,
  // writing identical keys, so the range is covered whatever each row sees)
  const int pr0 = max(pa.first, c0);
  const int pr1 = min(pa.first + pa.n, min(c0 + bpc, n_max));
  const int npool = max(0, pr1 - pr0);
  const long long lim = a.wait_limit > 0 ? a.wait_limit : kDecSpinLimit;
  volatile int32_t *abort_flag = &C.abort;
  const uint32_t tmem = C.tmem_base;
  uint8_t *wrow = ws + (int64_t)row * row_ws_bytes;
  RowHdr &W = *reinterpret_cast<RowHdr *>(wrow);

  if (warp == 0) {
    // (the producer issued its copies above)
  } else if (warp == 1) {
    // ---- MMA issuer: tile t into accumulator t
    if (lane == 0 && tiles > 0) {
      bool ok = tc_wait(sm32(&C.qready), 0u, lim, abort_flag);
      if (ok) tc_fence_after();
      bool patched = npool == 0;
      for (int t = 0; t < tiles && ok; ++t) {
        if (!(ok = tc_wait(sm32(&C.full[t]), 0u, lim, abort_flag))) break;
        const int32_t b0 = c0 + t * kDecTile;
        if (!patched && b0 < pr1 && b0 + kDecTile > pr0) {  // the tile holds pooled blocks
          if (!(ok = tc_wait(sm32(&C.pooled), 0u, kDecSpinLimit, abort_flag))) break;
          patched = true;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t kin = (uint32_t)(kk & 3) * 32u;  // K step inside the 128-byte row
          const uint64_t ad =
              sw128_desc(sRing + t * kDecTileBytes + (uint32_t)(kk >> 2) * kDecHalfBytes + kin);
          const uint64_t bd = sw128_desc(sQ + (uint32_t)(kk >> 2) * (kDecQBytes / 2) + kin);
          mma_bf16(tmem + (uint32_t)(t * kDecN), ad, bd, kDecIdesc, kk > 0 ? 1u : 0u);
        }
        mma_commit(sm32(&C.tfull[t]));
      }
      // every MMA this thread issued has finished before TMEM is freed
      mma_commit(sm32(&C.drain));
      tc_wait(sm32(&C.drain), 0u, kDecSpinLimit, nullptr);
    }
  } else if (warp < 4) {
    // ---- warps 2-3: the query operand
    const int h = (warp - 2) * 2 + (lane >> 4);  // head
    const int g = lane & 15;                     // dims 8g .. 8g+7
    const uint4 v = qv, w8 = qw8;
    const int64_t pp = valid ? p : 0;  // (an invalid row's operand is never used)
    uint4 c8 = make_uint4(0u, 0u, 0u, 0u), s8 = make_uint4(0u, 0u, 0u, 0u);
    if (g < 8) {
      c8 = ldg_nc_v4(a.cos_t + pp * kRot + 8 * g);
      s8 = ldg_nc_v4(a.sin_t + pp * kRot + 8 * g);
    }
    float x[8];
    unpack8(v, x);
    const uint4 o = norm_rope_16(x, w8, c8, s8, a.eps, g);
    // row h of the operand, 16-byte chunk g: 128-byte swizzle within its half
    const int half = g >> 3, j = g & 7;
    *reinterpret_cast<uint4 *>(smem + kDecQOff + half * (kDecQBytes / 2) + h * 128 +
                               ((j ^ (h & 7)) << 4)) = o;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the MMAs
    mbar_arrive(sm32(&C.qready));
  } else {
    // ---- warps 4-7, first: pool the newly complete blocks of the range (one per
    // 16 lanes).  Their tile's copy may have read the old key, so a block
    // this CTA scores is also written into its landed tile (the 128-byte
    // swizzled row of the MMA operand) before the MMAs read it.
    const int g = lane & 15;
    for (int j0 = 0; j0 < npool; j0 += 8) {
      const int jj = j0 + (warp - 4) * 2 + (lane >> 4);
      const int b = pr0 + min(jj, npool - 1);
      const uint4 key = pool_block_16(pa.keys + (int64_t)(b - pa.first) * kRatio * pa.key_stride,
                                      pa.key_stride, b, pa.k_norm_w, a.cos_t, a.sin_t, a.eps, g);
      if (jj < npool) {
        *reinterpret_cast<uint4 *>(pa.block_keys + (int64_t)b * kHeadDim + 8 * g) = key;
        const int t = (b - c0) / kDecTile, r = (b - c0) % kDecTile;
        if (t < tiles && tc_wait(sm32(&C.full[t]), 0u, kDecSpinLimit, abort_flag)) {
          const int half = g >> 3, j = g & 7;
          *reinterpret_cast<uint4 *>(ring + t * kDecTileBytes + half * kDecHalfBytes + r * 128 +
                                     ((j ^ (r & 7)) << 4)) = key;
        }
      }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the patches, to the MMAs
    mbar_arrive(sm32(&C.pooled));
    // ---- then one TMEM lane quarter each, one block per lane
    const int q = warp & 3;
    const float inv_sqrt_hd = 0.08838834764831845f;  // 1/sqrt(128)
    float *srow = a.scores + (int64_t)row * a.score_cols;
    const bool selecting = n > keep_max;  // uniform over the row's CTAs
    uint32_t my_max = 0u, my_min = kDecBins - 1u, my_low = 0u;
    for (int t = 0; t < tiles; ++t) {
      if (!tc_warp_wait(sm32(&C.tfull[t]), 0u, lim, abort_flag)) break;
      tc_fence_after();
      uint32_t v[4];
      tmem_ld4(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(t * kDecN), v);
      const float h0 = relu_nan(__uint_as_float(v[0]));
      const float h1 = relu_nan(__uint_as_float(v[1]));
      const float h2 = relu_nan(__uint_as_float(v[2]));
      const float h3 = relu_nan(__uint_as_float(v[3]));
      const float sc = __fmul_rn(__fadd_rn(__fadd_rn(__fadd_rn(h0, h1), h2), h3), inv_sqrt_hd);
      const int bl = t * kDecTile + 32 * q + lane;
      if (bl < cnt) {
        sc_s[bl] = sc;
        srow[c0 + bl] = sc;
      }
      if (selecting) {
        // the score's top-16-bit bin into the row's histogram, one add per
        // distinct bin per warp (every CTA of the row adds into it)
        const uint32_t bin = bl < cnt ? order_key(sc) >> (32 - kDecBinBits) : 0xFFFFFFFFu;
        const uint32_t peers = __match_any_sync(0xffffffffu, bin);
        if (bin != 0xFFFFFFFFu) {
          if (lane == __ffs(peers) - 1) atomicAdd(&W.hist0[hist_slot(bin)], (uint32_t)__popc(peers));
          my_max = max(my_max, bin);
          if (bin != kDecZeroBin) my_min = min(my_min, bin);  // (+0.0 has a bin of its own)
          my_low |= bin < kDecLoBad ? 1u : 0u;
        }
      }
    }
    my_max = __reduce_max_sync(0xffffffffu, my_max);
    my_min = __reduce_min_sync(0xffffffffu, my_min);
    my_low = __reduce_or_sync(0xffffffffu, my_low);
    if (lane == 0) {
      atomicMax(&C.maxbin, my_max);
      atomicMin(&C.minbin, my_min);
      if (my_low) C.low = 1u;
    }
  }

  __syncthreads();  // scoring done or given up; every MMA has drained
  if (tid == 0 && (C.issued > tiles || C.abort)) {
    // let every copy this CTA issued land before its shared memory is reused
    for (int t = 0; t < C.issued; ++t) tc_wait(sm32(&C.full[t]), 0u, kDecSpinLimit, nullptr);
  }
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kDecTmemCols)
                 : "memory");
  }
  __syncthreads();
  if (!valid) {  // uniform over the row's CTAs: nobody waits for them
    if (y == 0 && tid == 0) report_error(a.status, kErrRowRange, row);
    return;
  }
  if (C.abort) {
    if (tid == 0) report_error(a.status, kErrTimeout, row);
    return;  // the row's other CTAs time out at the barrier below
  }
  uint8_t *mrow = mask + (int64_t)row * a.tokens;
  uint32_t *cand_key = reinterpret_cast<uint32_t *>(wrow + sizeof(RowHdr));
  uint32_t *cand_idx = cand_key + (a.tokens >> 2);
  if (n <= keep_max) {  // every block kept: this CTA's share of the visible prefix
    const int64_t span = ((int64_t)a.tokens + ny - 1) / ny;
    const int64_t lo = (int64_t)y * span;
    fill_visible(mrow, lo, min((int64_t)a.tokens, lo + span), p);
    return;
  }
  // ---- 2. grid barrier over the row's CTAs (the histogram adds and C.maxbin
  // were made by the epilogue warps before the barrier after scoring)
  if (tid == 0) {
    asm volatile("red.relaxed.gpu.global.max.u32 [%0], %1;" ::"l"(&W.maxbin[y & 7]), "r"(C.maxbin)
                 : "memory");
    asm volatile("red.relaxed.gpu.global.max.u32 [%0], %1;" ::"l"(&W.binrev),
                 "r"(kDecBins - 1u - C.minbin)
                 : "memory");
    if (C.low) asm volatile("red.relaxed.gpu.global.or.b32 [%0], 1;" ::"l"(&W.lowbad) : "memory");
    // release: the CTA's histogram adds (ordered before it by the barrier
    // above) are visible to whoever sees the count
    red_add_release_gpu(&W.arrive, 1u);
    const long long t0 = clock64();
    const long long limit = a.wait_limit > 0 ? a.wait_limit : kDecSpinLimit;
    int ok = 1;
    while (ld_acquire_gpu(&W.arrive) < (uint32_t)ny) {
      if (clock64() - t0 > limit) {
        ok = 0;
        break;
      }
    }
    D.flag = ok;
  }
  __syncthreads();
  if (!D.flag) {
    if (tid == 0) report_error(a.status, kErrTimeout, row);
    return;
  }

  // ---- 3. the threshold bin, this CTA's mask bytes and candidates
  // A non-finite score lands at or above bin kDecHiBad (positive) or below
  // kDecLoBad (negative); every finite one between.  The row's highest bin is
  // read beside a copy of the 512 bins ending 256 above this CTA's own highest
  // one (a row's highest bin lies within that unless a few CTAs hold scores
  // four times the others'), so the kDecWindow bins ending at the row's
  // highest one are usually in shared memory after one round trip.  Otherwise
  // those bins are loaded in a second one, and, only if they hold fewer than
  // keep keys, the bins below them kDecChunk at a time.
  const uint32_t spec_lo = (uint32_t)min(max((int)C.maxbin + 256 - 511, 0), (int)kDecBins - 512);
  {
    const uint32_t v0 = __ldcg(&W.hist0[hist_slot(spec_lo + tid)]);
    const uint32_t v1 = __ldcg(&W.hist0[hist_slot(spec_lo + 256 + tid)]);
    if (tid == 0) {
      uint32_t mx = 0u;
#pragma unroll
      for (int k = 0; k < 8; ++k) mx = max(mx, __ldcg(&W.maxbin[k]));
      const bool nf = __ldcg(&W.lowbad) != 0u || mx >= kDecHiBad;
      D.rule_prefix = nf ? 1u : 0u;  // (scratch: the non-finite verdict)
      D.rule_shift = (uint32_t)max(0, (int)mx + 1 - kDecWindow);  // the window ends at mx
      D.row_max = mx;
      D.row_min = kDecBins - 1u - __ldcg(&W.binrev);
      D.sel_bin = -1;
    }
    D.hist0[tid] = v0;
    D.hist0[256 + tid] = v1;
  }
  __syncthreads();
  const bool bad = D.rule_prefix != 0u;
  const uint32_t wlo = D.rule_shift;
  auto fetch_hist = [&](uint32_t first, uint32_t nbins) {  // bins [first, first + nbins <= kDecChunk)
    __syncthreads();  // every thread is done with the previous copy
    uint32_t v[kDecChunk / kDecThreads];  // every load in flight before the first store
#pragma unroll
    for (int u = 0; u < kDecChunk / kDecThreads; ++u) {
      const uint32_t b = u * kDecThreads + tid;
      v[u] = b < nbins ? __ldcg(&W.hist0[hist_slot(first + b)]) : 0u;
    }
#pragma unroll
    for (int u = 0; u < kDecChunk / kDecThreads; ++u)
      if (u * kDecThreads + tid < (int)nbins) D.hist0[u * kDecThreads + tid] = v[u];
    if (tid == 0) D.sel_bin = -1;
    __syncthreads();
  };
  uint32_t need = (uint32_t)min(keep_max, n);
  uint32_t hbase = spec_lo;  // D.hist0[i] holds bin hbase + i
  int32_t sel = -1;          // the bin holding the need-th key, relative to hbase
  if (!bad) {
    if (wlo >= spec_lo && wlo + kDecWindow <= spec_lo + 512) {
      find_bin<kDecThreads>(D.hist0 + (wlo - spec_lo), kDecWindow, need, D.warp_tot, &D.sel_bin,
                            &D.sel_above, &D.sel_total);
      sel = D.sel_bin < 0 ? -1 : D.sel_bin + (int32_t)(wlo - spec_lo);
    } else {
      hbase = wlo;
      fetch_hist(wlo, kDecWindow);
      find_bin<kDecThreads>(D.hist0, kDecWindow, need, D.warp_tot, &D.sel_bin, &D.sel_above,
                            &D.sel_total);
      sel = D.sel_bin;
    }
    // the keep-th key lies below the window: the bins below it, a chunk at a
    // time (the histogram holds all n >= need keys, so the scan ends)
    for (uint32_t top = wlo; sel < 0 && top > 0;) {
      need -= D.sel_total;
      const uint32_t lo = top > (uint32_t)kDecChunk ? top - kDecChunk : 0u;
      hbase = lo;
      fetch_hist(lo, top - lo);  // (its first barrier: every thread has read sel_bin, sel_total)
      find_bin<kDecThreads>(D.hist0, (int)(top - lo), need, D.warp_tot, &D.sel_bin, &D.sel_above,
                            &D.sel_total);
      sel = D.sel_bin;
      top = lo;
    }
    if (sel < 0) {  // (only a workspace left dirty by the caller gets here)
      sel = 0;
      hbase = 0;
    }
    __syncthreads();  // every thread has read sel_bin
  }
  uint32_t B0 = 0;
  bool whole = false;  // the bin's keys are all kept
  const uintptr_t rb = reinterpret_cast<uintptr_t>(mrow);
  const bool al16 = (rb & 15u) == 0, al4 = (rb & 3u) == 0;
  // this thread's quad of the CTA's blocks (cnt <= 256: one quad at most)
  const int i = 4 * tid;
  const int mq = i < cnt ? min(4, cnt - i) : 0;
  uint32_t kept = 0, bits = 0;  // kept blocks; blocks of bin B0 (the candidates)
  if (bad) {
    if (y == 0 && tid == 0) report_error(a.status, kErrNonFinite, row);
  } else {
    B0 = hbase + (uint32_t)sel;
    need -= D.sel_above;
    whole = D.hist0[B0 - hbase] == need;
    uint32_t k[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      k[e] = e < mq ? order_key(sc_s[i + e]) : 0u;
      const uint32_t d = k[e] >> (32 - kDecBinBits);
      if (e < mq) {
        kept |= (d > B0 || (whole && d == B0) ? 1u : 0u) << e;
        bits |= (!whole && d == B0 ? 1u : 0u) << e;
      }
    }
    if (bits) {  // listed for the last CTA, which also writes their mask bytes
      uint32_t at = (uint32_t)atomicAdd(&W.tc, (unsigned long long)__popc(bits));
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (bits & (1u << e)) {
          cand_key[at] = k[e];
          cand_idx[at] = (uint32_t)(c0 + i + e);
          ++at;
        }
      }
    }
  }

  // ---- 4. the ticket: the last CTA of the row resolves the candidates
  __syncthreads();
  if (tid == 0) {
    // release this CTA's candidates; the last CTA acquires every CTA's
    unsigned long long t;
    asm volatile("atom.acq_rel.gpu.global.add.u64 %0, [%1], %2;"
                 : "=l"(t)
                 : "l"(&W.tc), "l"(1ull << 32)
                 : "memory");
    D.flag = (uint32_t)(t >> 32) == (uint32_t)(ny - 1);
    D.nl = (uint32_t)t;  // every CTA's candidates are listed by now
  }
  // this CTA's mask bytes other than the candidates' (no other CTA writes
  // them, so they need not precede the ticket)
  if (!bad) {
    if (bits == 0u) {
      if (mq) store_blocks(mrow, (int64_t)c0 + i, mq, kept, al16, al4);
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (e < mq && !(bits & (1u << e)))
          store_blocks(mrow, (int64_t)c0 + i + e, 1, (kept >> e) & 1u, false, al4);
    }
    // tokens past the complete blocks: the tail is visible, the rest zero
    if (y == ny - 1) fill_visible(mrow, 4 * (int64_t)n, a.tokens, p);
  }
  __syncthreads();
  if (!D.flag) return;
  const int32_t nl = (int32_t)D.nl;
  const bool few = !bad && !whole && nl <= 32;
  uint32_t ck = 0u, ci = 0u;  // (few: lane j of warp 0 holds candidate j)
  if (few && warp == 0 && lane < nl) {  // loaded before the clearing stores below
    ck = __ldcg(&cand_key[lane]);
    ci = __ldcg(&cand_idx[lane]);
  }
  // every CTA has read the histogram and taken its ticket: clear the bins the
  // row's keys landed in for the next call now, so that the stores drain
  // while the candidates are resolved (runs of eight bins, one 32-byte sector
  // each, from the row's lowest bin to its highest, and the zero bin)
  for (uint32_t r = (D.row_min >> 3) + tid; r <= (D.row_max >> 3); r += kDecThreads) {
    uint4 *run = reinterpret_cast<uint4 *>(&W.hist0[hist_slot(r << 3)]);
    run[0] = make_uint4(0u, 0u, 0u, 0u);
    run[1] = make_uint4(0u, 0u, 0u, 0u);
  }
  if (tid == 0) W.hist0[hist_slot(kDecZeroBin)] = 0u;
  auto clear_counters = [&]() {
    if (tid == 0) {
      W.arrive = 0u;
      W.binrev = 0u;
      W.tc = 0ull;
#pragma unroll
      for (int k = 0; k < 8; ++k) W.maxbin[k] = 0u;
      W.lowbad = 0u;
    }
  };
  if (bad || whole || few) clear_counters();
  if (few && warp == 0) {
    // a warp ranks the few candidates exactly: candidate j is kept if fewer
    // than `need` others come before it (a higher key, or the same key and a
    // lower block index)
    uint32_t rank = 0;
    for (int j = 0; j < nl; ++j) {
      const uint32_t kj = __shfl_sync(0xffffffffu, ck, j);
      const uint32_t ij = __shfl_sync(0xffffffffu, ci, j);
      rank += (kj > ck || (kj == ck && ij < ci)) ? 1u : 0u;
    }
    if (lane < nl) {
      store_blocks(mrow, (int64_t)ci, 1, rank < need ? 1u : 0u, false, al4);
      cand_key[lane] = 0u;
      cand_idx[lane] = 0u;
    }
  }
  if (!bad && !whole && !few) {
    for (int j0 = 0; j0 < min(nl, kDecCandCache); j0 += 8 * kDecThreads) {
      uint32_t kk[8], ii[8];  // eight entries per thread in flight
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int j = j0 + u * kDecThreads + tid;
        kk[u] = j < nl ? __ldcg(&cand_key[j]) : 0u;
        ii[u] = j < nl ? __ldcg(&cand_idx[j]) : 0u;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int j = j0 + u * kDecThreads + tid;
        if (j < min(nl, kDecCandCache)) {
          ck_s[j] = kk[u];
          ci_s[j] = ii[u];
          cand_key[j] = 0u;  // (the entry lives on in shared memory)
          cand_idx[j] = 0u;
        }
      }
    }
    for (int i = tid; i < 256 + 256; i += kDecThreads) (&D.hist1[0])[i] = 0u;
    __syncthreads();
    clear_counters();
    auto ckey = [&](int32_t j) { return j < kDecCandCache ? ck_s[j] : __ldcg(&cand_key[j]); };
    auto cidx = [&](int32_t j) { return j < kDecCandCache ? ci_s[j] : __ldcg(&cand_idx[j]); };
    uint32_t prefix = B0;
    int shift = 32 - kDecBinBits;
    bool done = false;
    // two rounds of 8 bits on the candidates (each round's result in its own
    // slot: two barriers a round)
    for (int r = 1; r < 3 && !done; ++r) {
      uint32_t *H = r == 1 ? D.hist1 : D.hist2;
      const int nb = 256, sh = r == 1 ? 8 : 0;
      for (int32_t j = tid; j < nl; j += kDecThreads) {
        const uint32_t key = ckey(j);
        if ((key >> shift) == prefix) atomicAdd(&H[(key >> sh) & (uint32_t)(nb - 1)], 1u);
      }
      __syncthreads();
      if (warp == 0) {
        uint32_t B, above;
        warp_find_bin(H, nb, need, lane, B, above);
        if (lane == 0) {
          D.rsel[r] = (int32_t)B;
          D.rabove[r] = above;
        }
      }
      __syncthreads();
      const uint32_t B = (uint32_t)D.rsel[r];
      const uint32_t cB = H[B];
      need -= D.rabove[r];
      prefix = (prefix << (shift - sh)) | B;
      shift = sh;
      done = cB == need;
    }
    if (done) {
      if (tid == 0) {
        D.rule_prefix = prefix;
        D.rule_shift = (uint32_t)shift;
        D.rule_cut = INT32_MAX;
      }
    } else {
      // ties at the full key: the `need` equal keys of lowest block index are
      // kept; radix rounds on the index, 8 bits at a time from the highest bit
      // an index < n can have, find the cut
      const uint32_t top = (uint32_t)n - 1u;
      int ish = top ? ((32 - __clz((int)top) + 7) & ~7) : 8;
      uint32_t iprefix = 0;
      uint32_t *H = D.hist0;  // no longer read
      for (int ir = 0; ir < 4; ++ir) {
        const int sh = ish - 8;
        H[tid] = 0u;  // kDecThreads == 256 bins
        __syncthreads();
        for (int32_t j = tid; j < nl; j += kDecThreads) {
          if (ckey(j) != prefix) continue;
          const uint32_t gi = cidx(j);
          if (ish >= 32 || (gi >> ish) == iprefix)  // ascending: digit d counts in bin 255-d
            atomicAdd(&H[255u - ((gi >> sh) & 255u)], 1u);
        }
        __syncthreads();
        if (warp == 0) {
          uint32_t B, above;
          warp_find_bin(H, 256, need, lane, B, above);
          if (lane == 0) {
            D.sel_bin = (int32_t)B;
            D.sel_above = above;
          }
        }
        __syncthreads();
        const uint32_t cB = H[D.sel_bin];
        need -= D.sel_above;
        iprefix = (iprefix << 8) | (255u - (uint32_t)D.sel_bin);
        ish = sh;
        __syncthreads();  // sel_bin and H are rewritten next round
        if (cB == need || ish == 0) break;  // at ish == 0 a bin holds one index
      }
      if (tid == 0) {
        D.rule_prefix = prefix;
        D.rule_shift = 0;
        D.rule_cut = (int32_t)((((uint64_t)iprefix + 1u) << ish) - 1u);
      }
    }
    __syncthreads();
    // every candidate's mask bytes (their owners wrote none)
    const uint32_t rp = D.rule_prefix, rs = D.rule_shift;
    const int32_t rc = D.rule_cut;
    for (int32_t j = tid; j < nl; j += kDecThreads) {
      const uint32_t kk = ckey(j) >> rs;
      const int32_t gi = (int32_t)cidx(j);
      store_blocks(mrow, gi, 1, (kk > rp || (kk == rp && gi <= rc)) ? 1u : 0u, false, al4);
    }
    // candidates past the shared-memory cache were read from the workspace
    // until now: cleared last
    for (int32_t j = kDecCandCache + tid; j < nl; j += kDecThreads) {
      cand_key[j] = 0u;
      cand_idx[j] = 0u;
    }
  }
}

// Co-resident CTAs of the fused kernel on the current device (0: not usable),
// with its shared-memory attribute set; once per device.
int dec_capacity() {
  static PerDevice cache;
  return cache.get([]() -> int {
    int dev = 0, sms = 0, per = 0;
    if (cudaFuncSetAttribute(decode_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kDecSmemBytes) != cudaSuccess ||
        cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, decode_fused_kernel, kDecThreads,
                                                      kDecSmemBytes) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    return per * sms;
  });
}

}  // namespace

int64_t decode_row_ws_bytes(int32_t tokens) {
  const int64_t b = (int64_t)sizeof(RowHdr) + 8 * (int64_t)(tokens / kRatio);
  return (b + 255) & ~int64_t(255);
}

cudaError_t launch_decode_fused(const ScoreArgs &a, int32_t budget, uint8_t *mask, void *ws,
                                const uint16_t *pool_keys, int64_t pool_key_stride,
                                int32_t pool_first, int32_t pool_n, const uint16_t *k_norm_w,
                                uint16_t *block_keys, cudaStream_t stream, bool *launched) {
  *launched = false;
  const int64_t n_max = (int64_t)a.tokens / kRatio;
  const int cap = dec_capacity();
  if (n_max == 0 || cap <= 0 || a.key_base != nullptr) return cudaSuccess;
  // the fewest blocks per CTA (128 or 256) that keep every CTA co-resident
  int32_t bpc = 0;
  for (int32_t k = kDecTile; k <= kDecMaxBpc; k += kDecTile) {
    if ((int64_t)a.n_rows * ((n_max + k - 1) / k) <= cap && (n_max + k - 1) / k <= 65535) {
      bpc = k;
      break;
    }
  }
  if (bpc == 0) return cudaSuccess;  // too many rows: the caller takes the two-kernel path
  CUtensorMap kmap;
  if (!encode_bf16_sw128(&kmap, a.block_keys, kHeadDim, (uint64_t)n_max, kHeadDim, 64, kDecTile))
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3((unsigned)a.n_rows, (unsigned)((n_max + bpc - 1) / bpc));
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = kDecSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const PoolArgs pa{pool_keys, pool_key_stride, pool_first, pool_n, k_norm_w, block_keys};
  const cudaError_t e =
      cudaLaunchKernelEx(&cfg, decode_fused_kernel, kmap, a, budget / kRatio, mask,
                         static_cast<uint8_t *>(ws), decode_row_ws_bytes(a.tokens), bpc, pa);
  if (e == cudaSuccess) *launched = true;
  return e;
}

}  // namespace qsa
