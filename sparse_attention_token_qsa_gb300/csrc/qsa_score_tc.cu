// Prefill block scorer on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// PR #1160 "score QSA token-indexer blocks in native CUDA", description: for a
// query row at position p and a visible block b,
//     S[p, b] = sum_h relu(q_h . k_b) / sqrt(128),
// relu per head before the head sum (a comparison, so NaN stays NaN); q_h is
// the row's head h after (1 + q_norm_w) RMSNorm and RoPE at p; only blocks
// b < visible_len / 4 are written.  The pages score prefill rows with SIMT
// reductions because an m16n8k16 tile cannot hold 4 rows; atlas
// layers/qsa_select.rs (prefill_select) already moves prefill scoring to
// tensor cores.  On GB300 the prefill contraction
//     D[rows*4, blocks] = Q[rows*4, 128] x K[blocks, 128]^T
// is a dense bf16 GEMM with K = 128, so it runs as tcgen05.mma.
//
// CTA tile: 128 blocks (M, the TMEM lanes) x 64 query rows * 4 heads (N = 256,
// column = 4 * row + head), K = 128 in 8 MMAs of K = 16.  With the heads on N,
// one TMEM lane (one thread of the epilogue) holds a block's dot with all four
// heads of a row in four adjacent columns, so the relu and the head sum are
// register-local and each warp store writes 32 consecutive blocks of one row.
//  * the rows' heads are prepared once per launch by qprep_kernel into a
//    workspace laid out [rows * 4, 128] (the B operand, K-major);
//  * warp 0 (one lane) streams block-key tiles (the A operand) with TMA
//    (128B swizzle) into a 4-stage ring guarded by mbarriers, and at every
//    row-tile switch, once the MMAs reading the old query tile are done, loads
//    the new 64-row query tile (2 x 32 KiB) with TMA;
//  * warp 1 (one lane) issues the MMAs into one of two TMEM accumulators
//    (256 columns each, 512 in all) and commits to mbarriers that free the key
//    stage and publish the accumulator;
//  * warps 4..19 drain the accumulators in two groups of eight, group g
//    taking accumulator g (every other unit), so each SM sub-partition holds
//    warps of two units in different phases: warp w reads TMEM lane quarter
//    w % 4 (32 blocks) and half of the columns (32 rows) in chunks of 16
//    columns, the next chunk loading while the current one is reduced (relu
//    per head, ((h0 + h1) + h2) + h3, scale) and stored with coalesced
//    128-byte stores; units off the causal diagonal store without per-row
//    tests;
//  * every mbarrier wait is bounded: on timeout the kernel records
//    QSA_ERR_TIMEOUT, lets the other roles drop out, drains its own MMAs and
//    frees its TMEM.
#include <cuda.h>  // CUtensorMap and its enums (the encoder comes from the runtime)

#include "qsa_device.cuh"
#include "qsa_launch.h"

namespace qsa {

const bool kTcScorerReady = true;

namespace {

constexpr int kRowsPerCta = 64;
constexpr int kBN = 128;
constexpr int kStages = 4;
constexpr int kThreads = 640;   // 20 warps
constexpr int kEpiWarp0 = 4;
constexpr int kEpiWarps = 16;   // 4 per TMEM lane quarter
constexpr int kQCols = kRowsPerCta * 4;       // N = 256 query-head rows
constexpr uint32_t kQChunk = kQCols * 128;     // 64 dims x 256 rows (32 KiB)
constexpr uint32_t kQBytes = 2 * kQChunk;      // the whole query tile (64 KiB)
constexpr uint32_t kKStage = kBN * 128 * 2;    // one key tile: 128 blocks x 128 dims (32 KiB)
constexpr uint32_t kKChunk = kBN * 128;        // 64 dims x 128 blocks (16 KiB)
constexpr uint32_t kQOff = 0;
constexpr uint32_t kKOff = kQBytes;
constexpr uint32_t kCtrlOff = kKOff + kStages * kKStage;
constexpr uint32_t kTmemCols = 512;
constexpr long long kSpinLimit = 4000000000LL;  // ~2 s of SM clock

constexpr int kMaxRowTiles = 1024;           // per-row-tile balancing up to 65536 rows

struct Ctrl {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint64_t qfree;
  uint64_t qready;
  uint32_t tmem_base;
  int32_t abort;
  int32_t need[kMaxRowTiles];
  int32_t start[kMaxRowTiles + 2];
};

constexpr size_t kSmemBytes = kCtrlOff + sizeof(Ctrl) + 1024;  // + alignment slack

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t a, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(count) : "memory");
}

// One potentially blocking test of a phase: the thread sleeps in hardware for
// up to kSuspendNs (or until the phase completes) instead of spinning.
constexpr uint32_t kSuspendNs = 20000;

__device__ __forceinline__ bool mbar_try(uint32_t a, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(a), "r"(parity), "r"(kSuspendNs)
      : "memory");
  return ok != 0;
}

// Bounded wait by one thread.  Returns false when the limit is hit (and raises
// the CTA's abort flag) or when another role already aborted.
__device__ bool mbar_wait(uint32_t a, uint32_t parity, volatile int32_t *abort_flag) {
  if (mbar_try(a, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try(a, parity)) return true;
    if (abort_flag != nullptr && *abort_flag) return false;
    if (clock64() - t0 > kSpinLimit) {
      if (abort_flag != nullptr) *abort_flag = 1;
      return false;
    }
  }
}

// The same wait made warp-uniform: lane 0 waits, the verdict is broadcast.
__device__ __forceinline__ bool warp_wait(uint32_t a, uint32_t parity, volatile int32_t *abort_flag) {
  uint32_t ok = 0;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(a, parity, abort_flag) ? 1u : 0u;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

__device__ __forceinline__ void mbar_arrive(uint32_t a) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(a) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t a, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(a), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(mbar)
      : "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (stride byte offset), descriptor version 1 (sm_100 family).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)1u << 16;                 // leading byte offset (unused by swizzled K-major)
  d |= (uint64_t)(1024u >> 4) << 32;       // stride byte offset
  d |= (uint64_t)1u << 46;                 // version
  d |= (uint64_t)2u << 61;                 // SWIZZLE_128B
  return d;
}

// Instruction descriptor, kind::f16: D f32, A/B bf16, both K-major, M = 128, N = 256.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kQCols >> 3) << 17) |
                            ((uint32_t)(kBN >> 4) << 24);

__device__ __forceinline__ void mma_bf16(uint32_t dtmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(dtmem),
      "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t mbar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld16_async(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
        "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
}

// Wait for this thread's TMEM loads.  The loaded registers pass through the
// statement, so no use of them can be scheduled before the wait.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&v)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]),
                 "+r"(v[6]), "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]),
                 "+r"(v[12]), "+r"(v[13]), "+r"(v[14]), "+r"(v[15])
               :
               : "memory");
}

// relu that keeps NaN (max.NaN returns NaN when either input is NaN)
__device__ __forceinline__ float relu_nan(float d) {
  float r;
  asm("max.NaN.f32 %0, %1, 0f00000000;" : "=f"(r) : "f"(d));
  return r;
}

// Walks a CTA's contiguous range of (row tile, block tile) work units in
// row-tile-major order; `k` counts row-tile switches (the first unit is one).
struct UnitCursor {
  const int32_t *start;  // exclusive prefix of block tiles per row tile
  int32_t rt, nt, k;
  __device__ void init(const int32_t *st, int32_t w) {
    start = st;
    rt = 0;
    while (start[rt + 1] <= w) ++rt;
    nt = w - start[rt];
    k = 0;
  }
  // advance to w + 1; returns true when the row tile changed
  __device__ bool next() {
    ++nt;
    if (start[rt] + nt < start[rt + 1]) return false;
    do {
      ++rt;
    } while (start[rt + 1] == start[rt]);
    nt = 0;
    ++k;
    return true;
  }
};

__global__ void __launch_bounds__(kThreads, 1)
score_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                const ScoreArgs a, int32_t tiles_total, int32_t row_base) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctrl &C = *reinterpret_cast<Ctrl *>(smem + kCtrlOff);
  const uint32_t sQ = smem_u32(smem + kQOff);
  const uint32_t sK = smem_u32(smem + kKOff);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int32_t row_tiles = (a.n_rows + kRowsPerCta - 1) / kRowsPerCta;

  // ---- set-up: barriers, TMEM, and the work each row tile needs.  It runs
  // while the previous launch in the stream finishes: that launch is always
  // the query preparation or an earlier slab of this kernel, which let this
  // one start only once every launch before them had completed, and neither
  // writes what the set-up reads (positions, visible lengths).  A CTA of an
  // earlier slab still holding TMEM cannot share an SM with this one (each
  // takes most of the shared memory), so the allocation does not wait on it.
  // The wait for the previous launch itself comes before the first copy of
  // the prepared queries.
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&C.full[s]), 1);
      mbar_init(smem_u32(&C.empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&C.tfull[b]), 1);
      mbar_init(smem_u32(&C.tempty[b]), kEpiWarps / 2);  // one group per accumulator
    }
    mbar_init(smem_u32(&C.drain), 1);
    mbar_init(smem_u32(&C.qfree), 1);
    mbar_init(smem_u32(&C.qready), 1);
    C.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 2) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&C.tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  for (int t = tid; t < row_tiles; t += kThreads) C.need[t] = 0;  // row_tiles <= kMaxRowTiles
  __syncthreads();
  // block tiles each row tile needs: its longest visible prefix
  for (int r = tid; r < a.n_rows; r += kThreads) {
    const int32_t p = a.pos[r];
    const int32_t vis = a.visible_len ? a.visible_len[r] : p + 1;
    if (p < 0 || p >= a.tokens || vis < 0 || vis > p + 1) {
      if (blockIdx.x == 0) report_error(a.status, kErrRowRange, row_base + r);
    } else if (vis >= 4) {
      atomicMax(&C.need[r / kRowsPerCta], ((vis >> 2) + kBN - 1) / kBN);
    }
  }
  __syncthreads();
  if (tid == 0) {
    int32_t acc = 0;
    for (int t = 0; t < row_tiles; ++t) {
      C.start[t] = acc;
      acc += C.need[t];
    }
    C.start[row_tiles] = acc;
    C.start[row_tiles + 1] = 0x7fffffff;  // sentinel for the cursor
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  grid_dependency_sync();

  const int64_t W = C.start[row_tiles];
  const int32_t w0 = (int32_t)(W * blockIdx.x / gridDim.x);
  const int32_t w1 = (int32_t)(W * (blockIdx.x + 1) / gridDim.x);
  const int nunits = w1 - w0;
  const uint32_t tmem = C.tmem_base;
  volatile int32_t *abort_flag = &C.abort;

  if (warp == 0) {
    // ---- TMA producer: key tiles, and the query tile at every row-tile switch
    if (lane == 0 && nunits > 0) {
      UnitCursor cur;
      cur.init(C.start, w0);
      int issued = 0;
      for (int i = 0; i < nunits; ++i) {
        const bool sw = (i == 0) || cur.next();
        const int s = i % kStages;
        const uint32_t it = (uint32_t)(i / kStages);
        if (!mbar_wait(smem_u32(&C.empty[s]), (it & 1u) ^ 1u, abort_flag)) break;
        const uint32_t fb = smem_u32(&C.full[s]);
        mbar_expect_tx(fb, kKStage);
        const int n0 = cur.nt * kBN;
        tma_load_2d(sK + s * kKStage, &kmap, 0, n0, fb);
        tma_load_2d(sK + s * kKStage + kKChunk, &kmap, 64, n0, fb);
        issued = i + 1;
        if (sw) {  // the MMAs reading the previous query tile have drained
          if (!mbar_wait(smem_u32(&C.qfree), (uint32_t)(cur.k & 1), abort_flag)) break;
          const uint32_t qb = smem_u32(&C.qready);
          mbar_expect_tx(qb, kQBytes);
          const int qy = (row_base + cur.rt * kRowsPerCta) * kHeads;
          tma_load_2d(sQ, &qmap, 0, qy, qb);
          tma_load_2d(sQ + kQChunk, &qmap, 64, qy, qb);
        }
      }
      if (*abort_flag) {  // let our own copies land before the CTA leaves
        for (int i = issued - kStages < 0 ? 0 : issued - kStages; i < issued; ++i)
          mbar_wait(smem_u32(&C.full[i % kStages]), (uint32_t)(i / kStages) & 1u, nullptr);
        mbar_wait(smem_u32(&C.qready), (uint32_t)(cur.k & 1), nullptr);
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer
    if (lane == 0 && nunits > 0) {
      UnitCursor cur;
      cur.init(C.start, w0);
      int drains = 0;
      bool ok = true;
      for (int i = 0; i < nunits && ok; ++i) {
        const bool sw = (i == 0) || cur.next();
        if (sw) {  // the query tile is rebuilt: every MMA reading it must be done
          if (i > 0) {
            mma_commit(smem_u32(&C.drain));
            ok = mbar_wait(smem_u32(&C.drain), (uint32_t)(drains & 1), abort_flag);
            ++drains;
            if (!ok) break;
          }
          mbar_arrive(smem_u32(&C.qfree));
          if (!mbar_wait(smem_u32(&C.qready), (uint32_t)(cur.k & 1), abort_flag)) break;
          tc_fence_after();
        }
        const int s = i % kStages;
        const uint32_t it = (uint32_t)(i / kStages);
        const int buf = i & 1;
        const uint32_t ja = (uint32_t)(i >> 1);
        if (!mbar_wait(smem_u32(&C.tempty[buf]), (ja & 1u) ^ 1u, abort_flag)) break;
        if (!mbar_wait(smem_u32(&C.full[s]), it & 1u, abort_flag)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t kin = (uint32_t)(kk & 3) * 32u;  // K step inside the 128-byte swizzle row
          const uint64_t ad = sw128_desc(sK + s * kKStage + (uint32_t)(kk >> 2) * kKChunk + kin);
          const uint64_t bd = sw128_desc(sQ + (uint32_t)(kk >> 2) * kQChunk + kin);
          mma_bf16(tmem + (uint32_t)(buf * kQCols), ad, bd, kk > 0 ? 1u : 0u);
        }
        mma_commit(smem_u32(&C.empty[s]));
        mma_commit(smem_u32(&C.tfull[buf]));
      }
      // every MMA this thread issued has finished before TMEM is freed
      mma_commit(smem_u32(&C.drain));
      mbar_wait(smem_u32(&C.drain), (uint32_t)(drains & 1), nullptr);
    }
  } else if (nunits > 0) {
    // ---- warps 4..19: drain TMEM (warps 2 and 3 have no role).  Two groups of
    // eight warps, one per accumulator: group g drains the units i with
    // i % 2 == g, so each SM sub-partition holds warps of two units at once.
    const bool epi = warp >= kEpiWarp0;
    const int grp = (warp - kEpiWarp0) >> 3;       // accumulator / unit parity
    const int quarter = warp & 3;                  // the TMEM lane quarter this warp may read
    const int half = ((warp - kEpiWarp0) >> 2) & 1;  // which 32 rows (128 columns) it drains
    const float inv_sqrt_hd = 0.08838834764831845f;
    const int64_t ld = a.score_cols;
    UnitCursor cur;
    cur.init(C.start, w0);
    int32_t my_n = 0;     // lane j: visible blocks of this warp's row j
    int32_t lim_min = 0;  // the smallest over the warp's 32 rows
    for (int i = 0; i < nunits && epi; ++i) {
      const bool sw = (i == 0) || cur.next();
      if (sw) {  // new row tile: this warp's rows and how far each may be written
        const int r = cur.rt * kRowsPerCta + half * 32 + lane;
        my_n = 0;
        if (r < a.n_rows) {
          const int32_t p = a.pos[r];
          const int32_t vis = a.visible_len ? a.visible_len[r] : p + 1;
          if (!(p < 0 || p >= a.tokens || vis < 0 || vis > p + 1)) my_n = vis >> 2;
        }
        lim_min = my_n;
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1)
          lim_min = min(lim_min, __shfl_xor_sync(0xffffffffu, lim_min, off));
      }
      if ((i & 1) != grp) continue;
      const int buf = grp;
      const uint32_t ja = (uint32_t)(i >> 1);
      if (!warp_wait(smem_u32(&C.tfull[buf]), ja & 1u, abort_flag)) break;
      tc_fence_after();
      const int b = cur.nt * kBN + quarter * 32 + lane;  // this thread's block
      // warp-uniform: all 32 blocks visible to all 32 rows (every unit off the
      // causal diagonal), so the stores need no per-row test
      const bool whole = cur.nt * kBN + quarter * 32 + 32 <= lim_min;
      float *dst = a.scores + (int64_t)(cur.rt * kRowsPerCta + half * 32) * ld + b;
      // eight chunks of 16 columns (4 rows x 4 heads); chunk c + 1 loads while
      // chunk c is reduced and stored
      const uint32_t taddr =
          tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(buf * kQCols + half * 128);
      uint32_t va[16], vb[16];
      tmem_ld16_async(taddr, va);
      tmem_wait_ld(va);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t(&v)[16] = (c & 1) ? vb : va;
        uint32_t(&vn)[16] = (c & 1) ? va : vb;
        if (c < 7) tmem_ld16_async(taddr + (uint32_t)(c + 1) * 16u, vn);
        float sc[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float h0 = relu_nan(__uint_as_float(v[4 * j + 0]));
          const float h1 = relu_nan(__uint_as_float(v[4 * j + 1]));
          const float h2 = relu_nan(__uint_as_float(v[4 * j + 2]));
          const float h3 = relu_nan(__uint_as_float(v[4 * j + 3]));
          sc[j] = __fmul_rn(__fadd_rn(__fadd_rn(__fadd_rn(h0, h1), h2), h3), inv_sqrt_hd);
        }
        if (whole) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            *dst = sc[j];
            dst += ld;
          }
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (b < __shfl_sync(0xffffffffu, my_n, c * 4 + j)) *dst = sc[j];
            dst += ld;
          }
        }
        if (c < 7) tmem_wait_ld(vn);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&C.tempty[buf]));
    }
  }

  __syncthreads();
  if (C.abort && tid == 0) report_error(a.status, kErrTimeout, (int32_t)blockIdx.x);
  if (warp == 2) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder (process-wide; looked up once, thread-safe).
EncodeTiledFn encoder() {
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(p);
    cudaGetLastError();
    return nullptr;
  }();
  return fn;
}

}  // namespace

cudaError_t launch_score_tc(const ScoreArgs &a, uint16_t *qws, cudaStream_t stream,
                            const PoolArgs *pool) {
  const int64_t n_cap = (int64_t)a.tokens / kRatio;  // no row sees more blocks than this
  if (n_cap == 0 || a.n_rows == 0) {
    if (pool == nullptr || pool->n == 0) return cudaSuccess;
    return launch_pool_blocks(pool->keys, pool->key_stride, pool->first, pool->n, pool->k_norm_w,
                              a.cos_t, a.sin_t, a.eps, pool->block_keys, stream);
  }
  if ((int64_t)a.n_rows * kHeads > INT32_MAX) return cudaErrorInvalidValue;
  EncodeTiledFn enc = encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  const cuuint32_t estr[2] = {1, 1};
  // block keys: 2D [n_cap rows, 128 bf16], rows 256 B apart; boxes of 128 rows x 64 dims
  CUtensorMap kmap;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)n_cap};
    const cuuint64_t strides[1] = {(cuuint64_t)kHeadDim * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)kBN};
    if (enc(&kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(a.block_keys),
            dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  // prepared queries: 2D [n_rows * 4, 128 bf16]; boxes of 256 rows (64 query rows) x 64 dims
  CUtensorMap qmap;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)a.n_rows * kHeads};
    const cuuint64_t strides[1] = {(cuuint64_t)kHeadDim * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)kQCols};
    if (enc(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, qws, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  static PerDevice smem_attr;
  cudaError_t e = set_smem_once(smem_attr, score_tc_kernel, kSmemBytes);
  if (e != cudaSuccess) return e;
  e = launch_qprep(a, qws, stream, pool);
  if (e != cudaSuccess) return e;
  // persistent: one CTA per SM, each taking a balanced contiguous range of
  // (row tile, block tile) units; more than kMaxRowTiles row tiles go in slabs,
  // and row tiles x block tiles stays in int32 per slab
  const int32_t tiles_total = (int32_t)((n_cap + kBN - 1) / kBN);
  int64_t slab_tiles = (int64_t)INT32_MAX / tiles_total;
  if (slab_tiles > kMaxRowTiles) slab_tiles = kMaxRowTiles;
  const int32_t slab = (int32_t)slab_tiles * kRowsPerCta;
  for (int32_t r0 = 0; r0 < a.n_rows; r0 += slab) {
    ScoreArgs b = a;
    b.n_rows = a.n_rows - r0 < slab ? a.n_rows - r0 : slab;
    b.q = a.q + (int64_t)r0 * a.q_stride;
    b.pos = a.pos + r0;
    b.visible_len = a.visible_len ? a.visible_len + r0 : nullptr;
    b.scores = a.scores + (int64_t)r0 * a.score_cols;
    const int64_t row_tiles = (b.n_rows + kRowsPerCta - 1) / kRowsPerCta;
    int64_t ctas = device_sm_count();
    if (ctas > row_tiles * tiles_total) ctas = row_tiles * tiles_total;
    e = launch_dependent(score_tc_kernel, dim3((unsigned)ctas), dim3(kThreads), kSmemBytes, stream,
                         1u, kmap, qmap, b, tiles_total, r0);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace qsa
