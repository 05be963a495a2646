// Streaming tensor-core block scorer (decode shape: few rows, each with its
// own long run of block keys; any row set).
//
// PR #1160 "score QSA token-indexer blocks in native CUDA", description: each
// query row's four heads are normed with (1 + q_norm_w) and rotated at the
// row's own position, then score(p, b) = sum_h relu(q_h . k_b) / sqrt(128), relu
// per head before the head sum (a NaN kept), over the row's visible blocks.
// metrale layers/qsa.rs decode_select scores one decode row against every
// complete block; this kernel does that for any rows, keys per row addressed
// through key_base.
//
// Each CTA scores a contiguous range of one row's visible blocks, a 128-block
// tile at a time, the way the fused decode launch scores its tiles:
//  * warp 0 streams the whole tiles into a ring of shared-memory stages with
//    TMA (two 64-dim boxes, 128-byte swizzle), refilling a stage once the MMAs
//    that read it have finished; a partial tile goes first, copied into the
//    same layout by the six warps that do not build the query operand (only
//    the row's own blocks are read, so no copy reaches past the caller's key
//    buffer);
//  * warps 2-3 prepare the row's four query heads as the 16 x 128 B operand
//    (rows 4..15 zero);
//  * one lane of warp 1 issues tcgen05.mma M128 N16 K16 x 8 per tile (keys on
//    M, heads on N) into one of two TMEM accumulators;
//  * warps 4-7 read an accumulator (one block per TMEM lane, its four heads in
//    four columns), apply relu, the head sum in order 0..3 and the scale, and
//    store the scores; the accumulator is released as soon as it is read.
// A block's score is the same MMA and the same epilogue as the fused decode
// launch's, so both give identical scores.  HBM traffic: 256 B of key read and
// 4 B of score written per (row, block).  Every wait is bounded; on a timeout
// the CTA records QSA_ERR_TIMEOUT once its own copies have landed.
#include "qsa_device.cuh"
#include "qsa_launch.h"
#include "qsa_tc_device.cuh"
#include "qsa_tma.h"

namespace qsa {

namespace {

constexpr int kStThreads = 256;
constexpr int kStTile = 128;                                // blocks per key tile: the MMA's M
constexpr int kStStages = 3;                                // key tiles in flight per CTA
constexpr uint32_t kStTileBytes = kStTile * kHeadDim * 2;   // 32 KiB
constexpr uint32_t kStHalfBytes = kStTile * 64 * 2;         // one 64-dim box: 16 KiB
constexpr int kStN = 16;                                    // MMA N: 4 heads, 12 zero rows
constexpr uint32_t kStTmemCols = 32;                        // two 16-column accumulators
constexpr long long kStSpinLimit = 4000000000LL;            // ~2 s of SM clock
// instruction descriptor, kind::f16: D f32, A and B bf16, both K-major, M = 128, N = 16
constexpr uint32_t kStIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kStN >> 3) << 17) |
                              ((uint32_t)(kStTile >> 4) << 24);

// Shared memory, from a 1024-byte aligned base: the key ring, the query
// operand, control.
constexpr uint32_t kStQOff = kStStages * kStTileBytes;
constexpr uint32_t kStQBytes = kStN * kHeadDim * 2;  // two 64-dim halves of 2 KiB
constexpr uint32_t kStCtrlOff = kStQOff + kStQBytes;

struct StCtrl {
  uint64_t full[kStStages];   // a tile has landed in the stage
  uint64_t empty[kStStages];  // the MMAs that read the stage are done
  uint64_t tfull[2];          // an accumulator holds a tile's head sums
  uint64_t tempty[2];         // the four epilogue warps have read it
  uint64_t qready;
  uint64_t drain;
  uint32_t tmem_base;
  int32_t abort;
  int32_t issued;  // tiles the producer started
};
constexpr size_t kStSmemBytes = kStCtrlOff + sizeof(StCtrl) + 1024;  // + alignment slack

__global__ void __launch_bounds__(kStThreads, 2)
score_stream_kernel(const __grid_constant__ CUtensorMap kmap, const ScoreArgs a, int32_t bpc) {
  extern __shared__ uint8_t st_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(st_raw) + 1023) & ~uintptr_t(1023));
  StCtrl &C = *reinterpret_cast<StCtrl *>(smem + kStCtrlOff);
  const uint32_t sRing = sm32(smem), sQ = sm32(smem + kStQOff);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = blockIdx.x, y = blockIdx.y;

  // ---- set-up while the previous launch finishes: barriers, the zero rows
  // of the query operand, TMEM
  if (tid == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&kmap)) : "memory");
    for (int s = 0; s < kStStages; ++s) {
      mbar_init(sm32(&C.full[s]), 1);
      mbar_init(sm32(&C.empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(sm32(&C.tfull[b]), 1);
      mbar_init(sm32(&C.tempty[b]), 4);  // one arrival per epilogue warp
    }
    mbar_init(sm32(&C.qready), 64);  // the query-prep threads
    mbar_init(sm32(&C.drain), 1);
    C.abort = 0;
    C.issued = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  reinterpret_cast<uint4 *>(smem + kStQOff)[tid] = make_uint4(0u, 0u, 0u, 0u);  // 4 KiB
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     sm32(&C.tmem_base)),
                 "r"(kStTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  grid_dependency_sync();

  const int32_t p = a.pos[row];
  const int32_t vis = a.visible_len ? a.visible_len[row] : p + 1;
  const bool valid = !(p < 0 || p >= a.tokens || vis < 0 || vis > p + 1);
  const int32_t n = valid ? vis >> 2 : 0;
  const int c0 = y * bpc;
  const int c1 = min(n, c0 + bpc);
  const int cnt = max(0, c1 - c0);
  const int tiles = (cnt + kStTile - 1) / kStTile;
  const int tail = cnt % kStTile;  // blocks of a partial last tile
  const int64_t kbase = a.key_base ? a.key_base[row] : 0;
  // TMA's row coordinate is a 32-bit int: 2^31 blocks are 512 GiB of keys, so
  // a row past it has an invalid key_base, reported like a bad position
  const bool keys_ok = kbase >= 0 && kbase + c1 <= (int64_t)0x7fffffff;
  const int ntiles = keys_ok ? tiles : 0;
  const long long lim = a.wait_limit > 0 ? a.wait_limit : kStSpinLimit;
  volatile int32_t *abort_flag = &C.abort;
  const uint32_t tmem = C.tmem_base;
  // Tile t of the range: a partial tile, if any, comes first (t = 0), then
  // the whole ones in order.  Its first block relative to c0:
  auto tile_off = [&](int t) {
    return tail ? (t == 0 ? (tiles - 1) * kStTile : (t - 1) * kStTile) : t * kStTile;
  };
  auto issue_tma = [&](int t) {  // a whole tile into stage t % kStStages (one thread)
    const int s = t % kStStages;
    const uint32_t fb = sm32(&C.full[s]);
    const int y0 = (int)(kbase + c0 + tile_off(t));
    mbar_expect_tx(fb, kStTileBytes);
    tma_load_2d(sRing + s * kStTileBytes, &kmap, 0, y0, fb);
    tma_load_2d(sRing + s * kStTileBytes + kStHalfBytes, &kmap, 64, y0, fb);
  };
  // ---- the first stages: the whole tiles by TMA, and the partial tile (only
  // the row's own blocks, so no copy reaches past the caller's key buffer) by
  // the six warps other than the query preparers, which meanwhile build the
  // query operand: 16 bytes a load, each chunk where the swizzled copy would
  // put it (chunk j of a box's row r at 16 * (j ^ (r % 8)))
  const int first = min(kStStages, ntiles);
  if (tid == 0) {
    for (int t = tail ? 1 : 0; t < first; ++t) issue_tma(t);
    C.issued = first;
  }
  if (tail && ntiles > 0 && (warp < 2 || warp >= 4)) {
    constexpr int kCopiers = kStThreads - 64;
    const int ct = (warp < 2 ? warp : warp - 2) * 32 + lane;
    const uint16_t *src = a.block_keys + (kbase + c0 + tile_off(0)) * kHeadDim;
    for (int i0 = 0; i0 < kStTile * 16; i0 += 4 * kCopiers) {
      uint4 v[4];  // four loads in flight a thread
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * kCopiers + ct, r = i >> 4, ch = i & 15;
        v[u] = (i < kStTile * 16 && r < tail) ? ldg_nc_v4(src + (int64_t)r * kHeadDim + 8 * ch)
                                              : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * kCopiers + ct, r = i >> 4, ch = i & 15;
        if (i < kStTile * 16)
          *reinterpret_cast<uint4 *>(smem + (ch >> 3) * kStHalfBytes + r * 128 +
                                     (((ch & 7) ^ (r & 7)) << 4)) = v[u];
      }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the MMAs
    asm volatile("bar.sync 1, %0;" ::"n"(kCopiers) : "memory");
    if (ct == 0) mbar_arrive(sm32(&C.full[0]));
  }

  if (warp == 0) {
    // ---- producer: whole tile t into stage t % kStStages once the MMAs of
    // the stage's previous tile are done
    for (int t = first; t < ntiles; ++t) {
      const int s = t % kStStages;
      if (!tc_warp_wait(sm32(&C.empty[s]), (uint32_t)((t / kStStages) - 1) & 1u, lim, abort_flag))
        break;
      if (lane == 0) {
        issue_tma(t);
        C.issued = t + 1;
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer: tile t into accumulator t % 2
    if (lane == 0 && ntiles > 0) {
      bool ok = tc_wait(sm32(&C.qready), 0u, lim, abort_flag);
      if (ok) tc_fence_after();
      for (int t = 0; t < ntiles && ok; ++t) {
        const int s = t % kStStages, acc = t & 1;
        if (!(ok = tc_wait(sm32(&C.full[s]), (uint32_t)(t / kStStages) & 1u, lim, abort_flag))) break;
        if (t >= 2 &&
            !(ok = tc_wait(sm32(&C.tempty[acc]), (uint32_t)((t >> 1) - 1) & 1u, lim, abort_flag)))
          break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t kin = (uint32_t)(kk & 3) * 32u;  // K step inside the 128-byte row
          const uint64_t ad =
              sw128_desc(sRing + s * kStTileBytes + (uint32_t)(kk >> 2) * kStHalfBytes + kin);
          const uint64_t bd = sw128_desc(sQ + (uint32_t)(kk >> 2) * (kStQBytes / 2) + kin);
          mma_bf16(tmem + (uint32_t)(acc * kStN), ad, bd, kStIdesc, kk > 0 ? 1u : 0u);
        }
        mma_commit(sm32(&C.empty[s]));    // the stage may be refilled once these MMAs are done
        mma_commit(sm32(&C.tfull[acc]));  // ... and the accumulator read
      }
      // every MMA this thread issued has finished before TMEM is freed
      mma_commit(sm32(&C.drain));
      tc_wait(sm32(&C.drain), 0u, kStSpinLimit, nullptr);
    }
  } else if (warp < 4) {
    // ---- warps 2-3: the query operand
    if (ntiles > 0) {
      const int h = (warp - 2) * 2 + (lane >> 4);  // head
      const int g = lane & 15;                     // dims 8g .. 8g+7
      const uint4 v = ldg_nc_v4(a.q + (int64_t)row * a.q_stride + h * kHeadDim + 8 * g);
      const uint4 w8 = ldg_nc_v4(a.q_norm_w + 8 * g);
      uint4 c8 = make_uint4(0u, 0u, 0u, 0u), s8 = make_uint4(0u, 0u, 0u, 0u);
      if (g < 8) {
        c8 = ldg_nc_v4(a.cos_t + (int64_t)p * kRot + 8 * g);
        s8 = ldg_nc_v4(a.sin_t + (int64_t)p * kRot + 8 * g);
      }
      float x[8];
      unpack8(v, x);
      const uint4 o = norm_rope_16(x, w8, c8, s8, a.eps, g);
      // row h of the operand, 16-byte chunk g: 128-byte swizzle within its half
      const int half = g >> 3, j = g & 7;
      *reinterpret_cast<uint4 *>(smem + kStQOff + half * (kStQBytes / 2) + h * 128 +
                                 ((j ^ (h & 7)) << 4)) = o;
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the MMAs
      mbar_arrive(sm32(&C.qready));
    }
  } else {
    // ---- warps 4-7: one TMEM lane quarter each, one block per lane
    const int q = warp & 3;
    const float inv_sqrt_hd = 0.08838834764831845f;  // 1/sqrt(128)
    float *srow = a.scores + (int64_t)row * a.score_cols + c0;
    for (int t = 0; t < ntiles; ++t) {
      const int acc = t & 1;
      if (!tc_warp_wait(sm32(&C.tfull[acc]), (uint32_t)(t >> 1) & 1u, lim, abort_flag)) break;
      tc_fence_after();
      uint32_t v[4];
      tmem_ld4(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * kStN), v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sm32(&C.tempty[acc]));  // the MMA may overwrite it
      const float h0 = relu_nan(__uint_as_float(v[0]));
      const float h1 = relu_nan(__uint_as_float(v[1]));
      const float h2 = relu_nan(__uint_as_float(v[2]));
      const float h3 = relu_nan(__uint_as_float(v[3]));
      const float sc = __fmul_rn(__fadd_rn(__fadd_rn(__fadd_rn(h0, h1), h2), h3), inv_sqrt_hd);
      const int r = 32 * q + lane;  // the block's row in the tile
      if (r < (tail && t == 0 ? tail : kStTile)) srow[tile_off(t) + r] = sc;
    }
  }

  __syncthreads();  // scoring done or given up; every MMA has drained
  if (tid == 0 && C.abort) {
    // let every copy this CTA issued land before its shared memory is released
    const int issued = C.issued;
    for (int t = max(0, issued - kStStages); t < issued; ++t)
      if (!(tail && t == 0))
        tc_wait(sm32(&C.full[t % kStStages]), (uint32_t)(t / kStStages) & 1u, kStSpinLimit, nullptr);
  }
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kStTmemCols)
                 : "memory");
  }
  if (tid == 0) {
    if ((!valid && y == 0) || (valid && !keys_ok)) report_error(a.status, kErrRowRange, row);
    if (C.abort) report_error(a.status, kErrTimeout, row);
  }
}

}  // namespace

cudaError_t launch_score_stream(const ScoreArgs &a, cudaStream_t stream) {
  const int64_t n_max = (int64_t)a.tokens / kRatio;
  if (n_max == 0 || a.n_rows == 0) return cudaSuccess;
  static PerDevice smem_attr;
  const cudaError_t e = set_smem_once(smem_attr, score_stream_kernel, kStSmemBytes);
  if (e != cudaSuccess) return e;
  // every row's keys through one map whose rows reach past any key_base the
  // caller may pass (a tile is only fetched by TMA inside a row's own blocks)
  CUtensorMap kmap;
  if (!encode_bf16_sw128(&kmap, a.block_keys, kHeadDim, 0x7fffffffull, kHeadDim, 64, kStTile))
    return cudaErrorInvalidValue;
  // tiles per CTA: one wave of two CTAs per SM over every row's tiles at most
  // (a CTA's ring fills and drains once, and no second wave runs half full:
  // 32 rows of 131k-262k tokens in 63 us on one wave, 67 us on about two, 71
  // us on four)
  const int64_t row_tiles = (n_max + kStTile - 1) / kStTile;
  int64_t k = ((int64_t)a.n_rows * row_tiles) / (2 * (int64_t)device_sm_count());
  k = k < 2 ? 2 : k;
  if (k > row_tiles) k = row_tiles;  // (one CTA per row)
  while ((row_tiles + k - 1) / k > 65535) ++k;
  const int32_t bpc = (int32_t)(k * kStTile);
  const dim3 grid((unsigned)a.n_rows, (unsigned)((n_max + bpc - 1) / bpc));
  return launch_dependent(score_stream_kernel, grid, dim3(kStThreads), kStSmemBytes, stream, 1u,
                          kmap, a, bpc);
}

}  // namespace qsa
