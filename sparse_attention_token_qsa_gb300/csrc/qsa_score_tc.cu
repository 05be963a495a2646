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
//  * the CTA prepares its 64 rows' heads itself (norm + RoPE, exact sums like
//    the pooling kernel) and writes them into shared memory in the 128-byte
//    swizzled K-major layout the MMA descriptors expect (the B operand);
//  * warp 0 (one lane) streams block-key tiles (the A operand) with TMA
//    (128B swizzle) into a 4-stage ring guarded by mbarriers;
//  * warp 1 (one lane) issues the MMAs into one of two TMEM accumulators
//    (256 columns each, 512 in all) and commits to mbarriers that free the key
//    stage and publish the accumulator;
//  * warps 4..11 drain the accumulator: warp w reads TMEM lane quarter w % 4
//    (32 blocks) and one half of the columns (32 rows), 32 columns per
//    tcgen05.ld, relu per head, ((h0 + h1) + h2) + h3, scale, coalesced stores
//    of the blocks each row can see;
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
constexpr int kThreads = 384;
constexpr int kEpiWarp0 = 4;
constexpr int kEpiWarps = 8;
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

struct Ctrl {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int32_t abort;
  int32_t max_n;
  int32_t row_n[kRowsPerCta];
};

constexpr size_t kSmemBytes = kCtrlOff + sizeof(Ctrl) + 1024;  // + alignment slack

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t a, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t a, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(a), "r"(parity)
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

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
        "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]),
        "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]),
        "=r"(v[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
        "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]),
        "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]),
        "=r"(v[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// relu that keeps NaN (max.NaN returns NaN when either input is NaN)
__device__ __forceinline__ float relu_nan(float d) {
  float r;
  asm("max.NaN.f32 %0, %1, 0f00000000;" : "=f"(r) : "f"(d));
  return r;
}

// Reduce one 32-column chunk (8 rows x 4 heads) held in `cur` to 8 scores and
// store the ones inside each row's visible prefix; before that, start the TMEM
// load of the next chunk into `nxt` (when `prefetch`), and wait for it after.
__device__ __forceinline__ void drain_chunk(const uint32_t (&cur)[32], int c, uint32_t tbase,
                                            uint32_t (&nxt)[32], bool prefetch,
                                            const int32_t *row_n, float *srow0, int64_t ld, int b,
                                            float inv_sqrt_hd) {
  int32_t lim[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) lim[j] = row_n[c * 8 + j];
  if (prefetch) tmem_ld32_async(tbase + (uint32_t)((c + 1) * 32), nxt);
  float out[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float h0 = relu_nan(__uint_as_float(cur[4 * j + 0]));
    const float h1 = relu_nan(__uint_as_float(cur[4 * j + 1]));
    const float h2 = relu_nan(__uint_as_float(cur[4 * j + 2]));
    const float h3 = relu_nan(__uint_as_float(cur[4 * j + 3]));
    out[j] = __fmul_rn(__fadd_rn(__fadd_rn(__fadd_rn(h0, h1), h2), h3), inv_sqrt_hd);
  }
  float *dst = srow0 + (int64_t)(c * 8) * ld + b;
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if (b < lim[j]) dst[(int64_t)j * ld] = out[j];
  if (prefetch) tmem_wait_ld();
}

__global__ void __launch_bounds__(kThreads, 1)
score_tc_kernel(const __grid_constant__ CUtensorMap kmap, const ScoreArgs a, int32_t tiles_total,
                int32_t tiles_per_split) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctrl &C = *reinterpret_cast<Ctrl *>(smem + kCtrlOff);
  const uint32_t sQ = smem_u32(smem + kQOff);
  const uint32_t sK = smem_u32(smem + kKOff);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row0 = blockIdx.x * kRowsPerCta;

  // ---- set-up: barriers, TMEM, per-row visible blocks
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&C.full[s]), 1);
      mbar_init(smem_u32(&C.empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&C.tfull[b]), 1);
      mbar_init(smem_u32(&C.tempty[b]), kEpiWarps);
    }
    mbar_init(smem_u32(&C.drain), 1);
    C.abort = 0;
    C.max_n = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 2) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&C.tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid < kRowsPerCta) {
    const int row = row0 + tid;
    int32_t n = 0;
    if (row < a.n_rows) {
      const int32_t p = a.pos[row];
      const int32_t vis = a.visible_len ? a.visible_len[row] : p + 1;
      if (p < 0 || p >= a.tokens || vis < 0 || vis > p + 1) {
        if (blockIdx.y == 0) report_error(a.status, kErrRowRange, row);
        n = -1;  // invalid row: no query, no writes
      } else {
        n = vis >> 2;
      }
    }
    C.row_n[tid] = n;
    if (n > 0) atomicMax(&C.max_n, n);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // ---- query heads of the 64 rows into the swizzled B (N-side) tile
  for (int pair = warp; pair < kRowsPerCta * kHeads / 2; pair += kThreads / 32) {
    const int vec = pair * 2 + (lane >> 4);
    const int rl = vec >> 2, h = vec & 3, g = lane & 15;
    const int row = row0 + rl;
    const bool valid = C.row_n[rl] >= 0 && row < a.n_rows;
    const int32_t p = valid ? a.pos[row] : 0;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (valid) v = ldg_nc_v4(a.q + (int64_t)row * a.q_stride + h * kHeadDim + 8 * g);
    const uint4 w8 = ldg_nc_v4(a.q_norm_w + 8 * g);
    uint4 c8 = make_uint4(0, 0, 0, 0), s8 = make_uint4(0, 0, 0, 0);
    if (g < 8) {
      c8 = ldg_nc_v4(a.cos_t + (int64_t)p * kRot + 8 * g);
      s8 = ldg_nc_v4(a.sin_t + (int64_t)p * kRot + 8 * g);
    }
    float x[8];
    unpack8(v, x);
    uint4 o = norm_rope_16(x, w8, c8, s8, a.eps, g);
    if (!valid) o = make_uint4(0, 0, 0, 0);
    const int n = 4 * rl + h;
    const int chunk = g >> 3, unit = g & 7;
    uint8_t *dst = smem + kQOff + chunk * kQChunk + n * 128 + ((unit ^ (n & 7)) << 4);
    *reinterpret_cast<uint4 *>(dst) = o;
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // read by the tensor core
  __syncthreads();

  const int32_t max_n = C.max_n;
  const int32_t t_begin = blockIdx.y * tiles_per_split;
  int32_t t_end = t_begin + tiles_per_split;
  if (t_end > tiles_total) t_end = tiles_total;
  const int32_t need = (max_n + kBN - 1) / kBN;
  if (t_end > need) t_end = need;
  const int ntiles = t_end > t_begin ? t_end - t_begin : 0;
  const uint32_t tmem = C.tmem_base;
  volatile int32_t *abort_flag = &C.abort;

  if (warp == 0) {
    // ---- TMA producer
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < ntiles; ++i) {
        const int s = i % kStages;
        const uint32_t it = (uint32_t)(i / kStages);
        if (!mbar_wait(smem_u32(&C.empty[s]), (it & 1u) ^ 1u, abort_flag)) break;
        const uint32_t fb = smem_u32(&C.full[s]);
        mbar_expect_tx(fb, kKStage);
        const int n0 = (t_begin + i) * kBN;
        tma_load_2d(sK + s * kKStage, &kmap, 0, n0, fb);
        tma_load_2d(sK + s * kKStage + kKChunk, &kmap, 64, n0, fb);
        issued = i + 1;
      }
      if (*abort_flag) {  // let our own copies land before the CTA leaves
        for (int i = issued - kStages < 0 ? 0 : issued - kStages; i < issued; ++i)
          mbar_wait(smem_u32(&C.full[i % kStages]), (uint32_t)(i / kStages) & 1u, nullptr);
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer
    if (lane == 0) {
      bool any = false;
      for (int i = 0; i < ntiles; ++i) {
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
        any = true;
      }
      if (any) {  // every MMA this thread issued has finished before TMEM is freed
        mma_commit(smem_u32(&C.drain));
        mbar_wait(smem_u32(&C.drain), 0u, nullptr);
      }
    }
  } else if (warp >= kEpiWarp0) {
    // ---- epilogue: TMEM -> relu -> head sum -> scale -> scores
    const int quarter = warp & 3;               // the TMEM lane quarter this warp may read
    const int chalf = (warp - kEpiWarp0) >> 2;  // which 32 rows (128 columns) it drains
    const float inv_sqrt_hd = 0.08838834764831845f;
    float *const srow0 = a.scores + (int64_t)(row0 + chalf * 32) * a.score_cols;
    const int64_t ld = a.score_cols;
    for (int i = 0; i < ntiles; ++i) {
      const int buf = i & 1;
      const uint32_t ja = (uint32_t)(i >> 1);
      if (!warp_wait(smem_u32(&C.tfull[buf]), ja & 1u, abort_flag)) break;
      tc_fence_after();
      const int b = (t_begin + i) * kBN + quarter * 32 + lane;  // this thread's block
      const uint32_t tbase =
          tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(buf * kQCols + chalf * 128);
      // TMEM loads are pipelined: chunk c+1 is in flight while chunk c is reduced
      uint32_t va[32], vb[32];
      tmem_ld32_async(tbase, va);
      tmem_wait_ld();
      drain_chunk(va, 0, tbase, vb, true, C.row_n + chalf * 32, srow0, ld, b, inv_sqrt_hd);
      drain_chunk(vb, 1, tbase, va, true, C.row_n + chalf * 32, srow0, ld, b, inv_sqrt_hd);
      drain_chunk(va, 2, tbase, vb, true, C.row_n + chalf * 32, srow0, ld, b, inv_sqrt_hd);
      drain_chunk(vb, 3, tbase, va, false, C.row_n + chalf * 32, srow0, ld, b, inv_sqrt_hd);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&C.tempty[buf]));
    }
  }

  __syncthreads();
  if (C.abort && tid == 0) report_error(a.status, kErrTimeout, row0);
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

EncodeTiledFn encoder() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

}  // namespace

cudaError_t launch_score_tc(const ScoreArgs &a, cudaStream_t stream) {
  const int64_t n_cap = (int64_t)a.tokens / kRatio;  // no row sees more blocks than this
  if (n_cap == 0) return cudaSuccess;
  EncodeTiledFn enc = encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  // block keys: 2D [n_cap rows, 128 bf16], rows 256 B apart; boxes of 128 rows x 64 dims
  CUtensorMap map;
  const cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)n_cap};
  const cuuint64_t strides[1] = {(cuuint64_t)kHeadDim * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)kBN};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(a.block_keys),
                   dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;

  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(score_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int32_t row_tiles = (a.n_rows + kRowsPerCta - 1) / kRowsPerCta;
  const int32_t tiles_total = (int32_t)((n_cap + kBN - 1) / kBN);
  // one CTA per SM: pick the split of the N tiles that minimises the critical
  // path, waves x (tiles per CTA + the CTA's fixed cost: query prep, TMEM
  // allocation, pipeline fill ~ 3 tiles), fewer CTAs on a tie
  const int64_t sms = sm_count();
  constexpr int64_t kCtaOverheadTiles = 3;
  int32_t splits = 1;
  int64_t best = -1;
  for (int32_t sp = 1; sp <= tiles_total && sp <= 65535; ++sp) {
    const int64_t waves = ((int64_t)row_tiles * sp + sms - 1) / sms;
    const int64_t cost = waves * ((tiles_total + sp - 1) / sp + kCtaOverheadTiles);
    if (best < 0 || cost < best) {
      best = cost;
      splits = sp;
    }
    if ((int64_t)row_tiles * sp > 64 * sms) break;
  }
  const int32_t per_split = (tiles_total + splits - 1) / splits;
  dim3 grid((unsigned)row_tiles, (unsigned)splits);
  score_tc_kernel<<<grid, kThreads, kSmemBytes, stream>>>(map, a, tiles_total, per_split);
  return cudaGetLastError();
}

}  // namespace qsa
