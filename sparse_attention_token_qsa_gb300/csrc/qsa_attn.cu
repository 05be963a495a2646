// Sparse attention over each row's selected tokens (the prefill consumer of
// the selection).
//
// atlas layers/qsa_select.rs prefill_select: a row at or past the inert bound
// gets its attention context replaced by attention over exactly its selected
// set -- the kept blocks' tokens and the tail -- read from the paged K/V cache
// through the sequence's block table, with nq query heads over nkv KV heads
// and a 1/sqrt(d) scale (metrale layers/qsa.rs module comment: each query
// attends the top budget/ratio blocks plus the incomplete tail).  Here the
// selected set comes as the token lists qsa_mask_tokens writes.
//
// Per (row, KV head, chunk of 8 query heads) one CTA of 4 warps; the warps
// split the row's tokens into 16-token tiles, round robin, and run an online
// softmax each, combined at the end through shared memory.  A tile's K and V
// rows (one 16-byte aligned run of head_dim bf16 per token and KV head) are
// brought by the bulk-copy engine into a per-warp ring of three stages, row
// stride head_dim * 2 + 16 bytes so that the fragment loads below hit 32
// distinct banks.
//
// The contraction per (row, KV head) has only 8 query heads, so it runs on
// warp-level mma.sync m16n8k16 (bf16 in, f32 accumulate):
//   S = Q K^T   M = query heads (8, padded to 16 with zero rows), N = 8 tokens
//               (two tiles per 16 tokens), K = head dims;
//   O^T += V^T P^T   M = head dims, N = the 8 query heads, K = 16 tokens,
// where P^T's operand registers are exactly S's accumulator registers (the
// accumulator of S holds, per lane, head lane/4 at tokens 2(lane%4), +1, which
// is the B operand layout of the second product), so no shuffle moves P.
// Both products are order-free in their K dimension, so head dims and tokens
// are assigned to lanes in whatever order makes each lane's loads 16-byte
// vectors (the same assignment on both operands of a product).
//
// Traffic: head_dim * 2 * 2 bytes of K and V per selected token and KV head,
// plus the query and output rows; the bound is memory (HBM, or L2 for tokens
// that several rows select), not the tensor pipe: 8 * head_dim * 4 flop per
// token and KV head is 8 flop per byte.
#include "qsa_device.cuh"
#include "qsa_launch.h"

namespace qsa {

namespace {

constexpr int kAttnWarps = 4;
constexpr int kAttnStages = 3;
constexpr int kAttnTile = 16;  // tokens per tile
constexpr long long kAttnSpinLimit = 4000000000LL;

template <int HD>
struct AttnGeom {
  static constexpr int kRowBytes = HD * 2;                        // one token's K (or V) row
  static constexpr int kStride = kRowBytes + 16;                  // in shared memory
  static constexpr int kStageBytes = 2 * kAttnTile * kStride;     // K rows then V rows
  static constexpr int kWarpBytes = kAttnStages * kStageBytes;
  static constexpr int kSteps = HD / 16;                          // k-steps of S = Q K^T
  static constexpr int kChunksPerLane = HD / 32;                  // 16-byte K/Q chunks per lane
  static constexpr int kMTiles = HD / 16;                         // m-tiles of O^T
  static constexpr int kVChunks = HD / 64;                        // 16-byte V chunks per lane and token
  static constexpr size_t kSmem = 128 + (size_t)kAttnWarps * kWarpBytes;
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// Bounded wait on an mbarrier phase; false once the limit is reached.
__device__ __forceinline__ bool attn_wait(uint32_t mbar, uint32_t parity) {
  const long long t0 = clock64();
  while (true) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(mbar), "r"(parity), "r"(20000u)
        : "memory");
    if (ok) return true;
    if (clock64() - t0 > kAttnSpinLimit) return false;
  }
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// Two f32 as a bf16x2 word (round to nearest even), lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// The 16-byte chunk of a K row (and of a query head) that lane quad position
// q reads for its j-th chunk: chunks {2q, 2q+1, 2q+8, 2q+9, 2q+16, ...}.  Over
// q = 0..3 they cover every chunk once, and the 8 lanes of a quarter-warp (two
// rows, four q) start on 8 distinct 4-bank groups.
__device__ __forceinline__ int k_chunk(int q, int j) { return 8 * (j >> 1) + 2 * q + (j & 1); }

struct AttnArgs {
  const uint16_t *q;
  int64_t q_stride;
  int32_t nq, nkv, group;  // group = nq / nkv
  const uint16_t *k_pool, *v_pool;
  int32_t pool_pages, page_size;
  const int32_t *table;
  int32_t table_len;
  int64_t table_cols;
  const int32_t *sel;
  int64_t sel_cols;
  const int32_t *n_sel;
  int32_t max_sel;
  float scale_log2;  // scale * log2(e)
  uint16_t *out;
  int64_t out_stride;
  int32_t *status;
  int32_t n_rows;
};

template <int HD>
__global__ void __launch_bounds__(32 * kAttnWarps, 1)
sparse_attn_kernel(const AttnArgs a, int32_t head_chunks) {
  using Geo = AttnGeom<HD>;
  extern __shared__ __align__(128) uint8_t attn_smem[];
  uint64_t *bars = reinterpret_cast<uint64_t *>(attn_smem);  // [warp][stage]
  uint8_t *rings = attn_smem + 128;
  grid_dependency_sync();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, q = lane & 3;
  // KV head slowest: the launch works through one KV head's cache at a time,
  // which a 64k context's K and V for one head (64 MiB) fit in L2
  const int64_t unit = blockIdx.x;
  const int hc = (int)(unit % head_chunks);
  const int32_t row = (int32_t)((unit / head_chunks) % a.n_rows);
  const int kvh = (int)(unit / ((int64_t)head_chunks * a.n_rows));
  const int32_t n = max(0, min(a.n_sel[row], a.max_sel));
  const int32_t *srow = a.sel + (int64_t)row * a.sel_cols;
  const int32_t *trow = a.table + (int64_t)row * a.table_cols;
  const int heads_here = min(8, a.group - hc * 8);
  uint8_t *ring = rings + (size_t)warp * Geo::kWarpBytes;
  uint64_t *wbar = bars + warp * kAttnStages;

  // query head g of this chunk (zero rows past the group), in k_chunk order
  uint32_t qa[Geo::kSteps][2];
  {
    const bool hv = g < heads_here;
    const uint16_t *qh =
        a.q + (int64_t)row * a.q_stride + (int64_t)(kvh * a.group + hc * 8 + (hv ? g : 0)) * HD;
#pragma unroll
    for (int j = 0; j < Geo::kChunksPerLane; ++j) {
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (hv) v = ldg_nc_v4(qh + 8 * k_chunk(q, j));
      qa[2 * j][0] = v.x;
      qa[2 * j][1] = v.y;
      qa[2 * j + 1][0] = v.z;
      qa[2 * j + 1][1] = v.w;
    }
  }
  if (lane == 0) {
    for (int s = 0; s < kAttnStages; ++s)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&wbar[s])) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();

  // this warp's tiles are warp, warp + 4, ...: local tile i is row tokens
  // [16 (warp + 4 i), +16).  Lane x and lane x + 16 handle token x of a tile
  // (its K row and its V row).  The two lookups before a tile's copies (its
  // token, then that token's page entry) are loads whose results the next
  // tile's issue consumes, so their latency overlaps a tile of work.
  const int n_tiles = (n + kAttnTile - 1) / kAttnTile;
  const int my_tiles = n_tiles > warp ? (n_tiles - warp + kAttnWarps - 1) / kAttnWarps : 0;
  constexpr int32_t kNoToken = INT32_MIN;
  auto fetch_tok = [&](int i) -> int32_t {
    const int32_t j = (warp + kAttnWarps * i) * kAttnTile + (lane & 15);
    return (i < my_tiles && j < n) ? srow[j] : kNoToken;
  };
  auto fetch_page = [&](int32_t t) -> int32_t {  // -1: outside the table
    if (t == kNoToken) return kNoToken;
    const int32_t pg = t >= 0 ? t / a.page_size : -1;
    return (t >= 0 && pg < a.table_len) ? trow[pg] : -1;
  };
  uint64_t vbits = 0;  // valid-token bits of the tile in each stage (16 per stage)
  auto start = [&](int i, int32_t t, int32_t phys) {
    const int s = i % kAttnStages;
    const bool ok = t != kNoToken && phys >= 0 && phys < a.pool_pages;
    if (t != kNoToken && !ok && lane < 16) report_error(a.status, kErrTokenRange, row);
    const uint32_t bal = __ballot_sync(0xffffffffu, ok);
    vbits = (vbits & ~(0xFFFFull << (16 * s))) | ((uint64_t)(bal & 0xFFFFu) << (16 * s));
    const uint32_t mb = smem_u32(&wbar[s]);
    if (lane == 0)
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mb),
                   "r"((uint32_t)__popc(bal) * (uint32_t)Geo::kRowBytes)
                   : "memory");
    __syncwarp();
    if (ok) {
      const int32_t pg = t / a.page_size;
      const int64_t src_row = ((int64_t)phys * a.page_size + (t - pg * a.page_size)) * a.nkv + kvh;
      const uint16_t *src = (lane < 16 ? a.k_pool : a.v_pool) + src_row * HD;
      const uint8_t *dst = ring + (size_t)s * Geo::kStageBytes +
                           (lane < 16 ? 0 : kAttnTile * Geo::kStride) + (lane & 15) * Geo::kStride;
      asm volatile(
          "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
              "r"(smem_u32(dst)), "l"(src), "r"((uint32_t)Geo::kRowBytes), "r"(mb)
          : "memory");
    }
  };
  // prologue: the first kAttnStages tiles, their lookups issued side by side
  int32_t tok_pre[kAttnStages + 1], page_pre[kAttnStages];
#pragma unroll
  for (int k = 0; k <= kAttnStages; ++k) tok_pre[k] = fetch_tok(k);
#pragma unroll
  for (int k = 0; k < kAttnStages; ++k) page_pre[k] = fetch_page(tok_pre[k]);
  int issued = 0;
#pragma unroll
  for (int k = 0; k < kAttnStages; ++k)
    if (k < my_tiles) {
      start(k, tok_pre[k], page_pre[k]);
      ++issued;
    }
  int32_t tok_next = tok_pre[kAttnStages];            // tile `issued`
  int32_t page_next = fetch_page(tok_next);           // in flight
  int32_t tok_after = fetch_tok(kAttnStages + 1);     // tile `issued + 1`, in flight

  float m_run = -INFINITY;  // running max of head g's logits (log2 units)
  float l_run = 0.f;        // this lane's part of head g's weight sum
  float acc[Geo::kMTiles][4];
#pragma unroll
  for (int t = 0; t < Geo::kMTiles; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
  bool failed = false;
  int i = 0;
  for (; i < my_tiles; ++i) {
    const int s = i % kAttnStages;
    const bool okw = attn_wait(smem_u32(&wbar[s]), (uint32_t)(i / kAttnStages) & 1u);
    if (!__all_sync(0xffffffffu, okw)) {
      failed = true;
      break;
    }
    const uint8_t *kt = ring + (size_t)s * Geo::kStageBytes;
    const uint8_t *vt = kt + kAttnTile * Geo::kStride;
    const uint32_t vb = (uint32_t)(vbits >> (16 * s)) & 0xFFFFu;

    // ---- S = Q K^T over the tile's two 8-token halves (two chains each)
    float sc[2][2][4];
#pragma unroll
    for (int x = 0; x < 2; ++x)
#pragma unroll
      for (int y = 0; y < 2; ++y) sc[x][y][0] = sc[x][y][1] = sc[x][y][2] = sc[x][y][3] = 0.f;
#pragma unroll
    for (int j = 0; j < Geo::kChunksPerLane; ++j) {
      const int c = k_chunk(q, j);
      const uint4 k0 = *reinterpret_cast<const uint4 *>(kt + g * Geo::kStride + 16 * c);
      const uint4 k1 = *reinterpret_cast<const uint4 *>(kt + (g + 8) * Geo::kStride + 16 * c);
      mma_bf16(sc[0][j & 1], qa[2 * j][0], 0u, qa[2 * j][1], 0u, k0.x, k0.y);
      mma_bf16(sc[1][j & 1], qa[2 * j][0], 0u, qa[2 * j][1], 0u, k1.x, k1.y);
      mma_bf16(sc[0][j & 1], qa[2 * j + 1][0], 0u, qa[2 * j + 1][1], 0u, k0.z, k0.w);
      mma_bf16(sc[1][j & 1], qa[2 * j + 1][0], 0u, qa[2 * j + 1][1], 0u, k1.z, k1.w);
    }
    // this lane's logits: head g at tile tokens 2q, 2q+1, 2q+8, 2q+9
    float sv[4] = {sc[0][0][0] + sc[0][1][0], sc[0][0][1] + sc[0][1][1], sc[1][0][0] + sc[1][1][0],
                   sc[1][0][1] + sc[1][1][1]};
    float tmax = -INFINITY;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int tk = 2 * q + (e & 1) + 8 * (e >> 1);
      sv[e] = ((vb >> tk) & 1u) ? sv[e] * a.scale_log2 : -INFINITY;
      tmax = fmaxf(tmax, sv[e]);
    }
    tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
    tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
    const float m_new = fmaxf(m_run, tmax);
    const float m_use = m_new == -INFINITY ? 0.f : m_new;
    const float alpha = exp2f(m_run - m_use);  // 0 while nothing was seen
    m_run = m_new;
    const uint32_t pb0 = pack_bf16x2(exp2f(sv[0] - m_use), exp2f(sv[1] - m_use));
    const uint32_t pb1 = pack_bf16x2(exp2f(sv[2] - m_use), exp2f(sv[3] - m_use));
    // the weights the product uses are the rounded ones: so is their sum
    l_run = l_run * alpha + ((bf16_lo(pb0) + bf16_hi(pb0)) + (bf16_lo(pb1) + bf16_hi(pb1)));
    // O^T's columns are heads 2q, 2q+1, whose factors lanes 8q and 8q+4 hold
    if (__any_sync(0xffffffffu, alpha != 1.f)) {  // some head's maximum moved
      const float al0 = __shfl_sync(0xffffffffu, alpha, 8 * q);
      const float al1 = __shfl_sync(0xffffffffu, alpha, 8 * q + 4);
#pragma unroll
      for (int t = 0; t < Geo::kMTiles; ++t) {
        acc[t][0] *= al0;
        acc[t][2] *= al0;
        acc[t][1] *= al1;
        acc[t][3] *= al1;
      }
    }

    // ---- O^T += V^T P^T: V rows of tokens 2q, 2q+1, 2q+8, 2q+9 at chunks g + 8c
    // (in a partial tile a token outside the list contributes zeros: its stage
    // row may hold anything)
    auto pv = [&](const uint32_t z0, const uint32_t z1, const uint32_t z2, const uint32_t z3) {
#pragma unroll
      for (int c = 0; c < Geo::kVChunks; ++c) {
        const int off = 16 * (g + 8 * c);
        const uint4 v0 = *reinterpret_cast<const uint4 *>(vt + (2 * q) * Geo::kStride + off);
        const uint4 v1 = *reinterpret_cast<const uint4 *>(vt + (2 * q + 1) * Geo::kStride + off);
        const uint4 v2 = *reinterpret_cast<const uint4 *>(vt + (2 * q + 8) * Geo::kStride + off);
        const uint4 v3 = *reinterpret_cast<const uint4 *>(vt + (2 * q + 9) * Geo::kStride + off);
        const uint32_t w0[4] = {v0.x & z0, v0.y & z0, v0.z & z0, v0.w & z0};
        const uint32_t w1[4] = {v1.x & z1, v1.y & z1, v1.z & z1, v1.w & z1};
        const uint32_t w2[4] = {v2.x & z2, v2.y & z2, v2.z & z2, v2.w & z2};
        const uint32_t w3[4] = {v3.x & z3, v3.y & z3, v3.z & z3, v3.w & z3};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          // m-tile 4c + e: rows g, g+8 are dims 8(g + 8c) + 2e, +1
          mma_bf16(acc[4 * c + e], prmt(w0[e], w1[e], 0x5410u), prmt(w0[e], w1[e], 0x7632u),
                   prmt(w2[e], w3[e], 0x5410u), prmt(w2[e], w3[e], 0x7632u), pb0, pb1);
        }
      }
    };
    if (vb == 0xFFFFu) {  // a whole tile (uniform over the warp): constant masks fold away
      pv(0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu);
    } else {
      pv((vb >> (2 * q)) & 1u ? 0xFFFFFFFFu : 0u, (vb >> (2 * q + 1)) & 1u ? 0xFFFFFFFFu : 0u,
         (vb >> (2 * q + 8)) & 1u ? 0xFFFFFFFFu : 0u, (vb >> (2 * q + 9)) & 1u ? 0xFFFFFFFFu : 0u);
    }
    if (issued < my_tiles) {  // refill this stage once every lane is done reading it
      __syncwarp();
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      start(issued, tok_next, page_next);
      ++issued;
      tok_next = tok_after;
      page_next = fetch_page(tok_next);
      tok_after = fetch_tok(issued + 1);
    }
  }
  if (failed) {
    if (lane == 0) report_error(a.status, kErrTimeout, row);
    // let this warp's own copies land before the ring is reused below
    for (int k = i; k < issued; ++k)
      attn_wait(smem_u32(&wbar[k % kAttnStages]), (uint32_t)(k / kAttnStages) & 1u);
  }

  // ---- combine the warps: head h's output is sum_w 2^(m_w - M) O_w / sum_w 2^(m_w - M) l_w
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
  __syncthreads();  // every warp's copies have landed: the rings are free
  float *mw = reinterpret_cast<float *>(rings);  // [warp][8] running maxima
  float *lw = mw + kAttnWarps * 8;               // [warp][8] weight sums
  float *ow = lw + kAttnWarps * 8;               // [warp][8 heads][HD] unnormalised outputs
  if (q == 0) {
    mw[warp * 8 + g] = m_run;
    lw[warp * 8 + g] = l_run;
  }
#pragma unroll
  for (int t = 0; t < Geo::kMTiles; ++t) {
    const int d0 = 8 * (g + 8 * (t >> 2)) + 2 * (t & 3);
    float *o0 = ow + (size_t)(warp * 8 + 2 * q) * HD + d0;
    float *o1 = ow + (size_t)(warp * 8 + 2 * q + 1) * HD + d0;
    o0[0] = acc[t][0];
    o0[1] = acc[t][2];
    o1[0] = acc[t][1];
    o1[1] = acc[t][3];
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < heads_here * (HD / 8); idx += 32 * kAttnWarps) {
    const int h = idx / (HD / 8), d0 = 8 * (idx % (HD / 8));
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) mx = fmaxf(mx, mw[w * 8 + h]);
    float f[kAttnWarps], den = 0.f;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) {
      f[w] = mx == -INFINITY ? 0.f : exp2f(mw[w * 8 + h] - mx);
      den += f[w] * lw[w * 8 + h];
    }
    float o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) {
      const float4 x0 = *reinterpret_cast<const float4 *>(ow + (size_t)(w * 8 + h) * HD + d0);
      const float4 x1 = *reinterpret_cast<const float4 *>(ow + (size_t)(w * 8 + h) * HD + d0 + 4);
      o[0] += f[w] * x0.x;
      o[1] += f[w] * x0.y;
      o[2] += f[w] * x0.z;
      o[3] += f[w] * x0.w;
      o[4] += f[w] * x1.x;
      o[5] += f[w] * x1.y;
      o[6] += f[w] * x1.z;
      o[7] += f[w] * x1.w;
    }
    const float inv = den == 0.f ? 0.f : 1.f / den;  // no selected token: zeros
    const uint4 r = make_uint4(pack_bf16x2(o[0] * inv, o[1] * inv), pack_bf16x2(o[2] * inv, o[3] * inv),
                               pack_bf16x2(o[4] * inv, o[5] * inv), pack_bf16x2(o[6] * inv, o[7] * inv));
    *reinterpret_cast<uint4 *>(a.out + (int64_t)row * a.out_stride +
                               (int64_t)(kvh * a.group + hc * 8 + h) * HD + d0) = r;
  }
}

template <int HD>
cudaError_t launch_attn_hd(const AttnArgs &a, int32_t n_rows, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(sparse_attn_kernel<HD>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)AttnGeom<HD>::kSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int32_t head_chunks = (a.group + 7) / 8;
  const int64_t units = (int64_t)n_rows * a.nkv * head_chunks;
  return launch_dependent(sparse_attn_kernel<HD>, dim3((unsigned)units), dim3(32 * kAttnWarps),
                          AttnGeom<HD>::kSmem, stream, 1u, a, head_chunks);
}

}  // namespace

cudaError_t launch_sparse_attn(const uint16_t *q, int64_t q_stride, int32_t nq, int32_t nkv,
                               int32_t head_dim, const uint16_t *k_pool, const uint16_t *v_pool,
                               int32_t pool_pages, int32_t page_size, const int32_t *table,
                               int32_t table_len, int64_t table_cols, const int32_t *sel,
                               int64_t sel_cols, const int32_t *n_sel, int32_t n_rows,
                               int32_t max_sel, float scale, uint16_t *out, int64_t out_stride,
                               int32_t *status, cudaStream_t stream) {
  AttnArgs a;
  a.q = q;
  a.q_stride = q_stride;
  a.nq = nq;
  a.nkv = nkv;
  a.group = nq / nkv;
  a.k_pool = k_pool;
  a.v_pool = v_pool;
  a.pool_pages = pool_pages;
  a.page_size = page_size;
  a.table = table;
  a.table_len = table_len;
  a.table_cols = table_cols;
  a.sel = sel;
  a.sel_cols = sel_cols;
  a.n_sel = n_sel;
  a.max_sel = max_sel;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.out = out;
  a.out_stride = out_stride;
  a.status = status;
  a.n_rows = n_rows;
  if (head_dim == 256) return launch_attn_hd<256>(a, n_rows, stream);
  return launch_attn_hd<128>(a, n_rows, stream);
}

}  // namespace qsa
