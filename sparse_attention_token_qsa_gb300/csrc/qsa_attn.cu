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
// Per (row, KV head, chunk of 8 query heads) one CTA of 4 warps, the grid
// ordered KV head first.  The CTA walks the row's tokens in 32-token tiles:
// each warp's lanes bring 8 tokens' K and V rows (one 16-byte aligned run of
// head_dim bf16 per token and KV head) with the bulk-copy engine into a ring
// shared by the CTA (two stages at head_dim 256, three at 128; row stride
// head_dim * 2 + 16 bytes, so the fragment loads below hit 32 distinct
// banks); the four warps split the head dims, each computing its part of the
// logits and of the output.  The partial logits meet once per tile in shared
// memory and every warp sums them in the same order, so every warp holds the
// same softmax state and no final combine is needed.  About 74 KiB of shared
// memory per CTA at head_dim 256: three CTAs (12 warps) per SM.  (16-token
// tiles in a three-stage ring, four CTAs per SM, took 4 % longer: the
// barrier, the exchange and the softmax bookkeeping come once per tile.)
//
// The contraction per (row, KV head) has only 8 query heads, so it runs on
// warp-level mma.sync m16n8k16 (bf16 in, f32 accumulate):
//   S = Q K^T   M = query heads (8, padded to 16 with zero rows), N = 8 tokens
//               (four tiles per 32 tokens), K = head dims;
//   O^T += V^T P^T   M = head dims, N = the 8 query heads, K = 16 tokens (two
//               steps per tile),
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
constexpr int kAttnStagesMax = 3;
constexpr int kAttnTile = 32;  // tokens per tile (each warp brings 8)
constexpr long long kAttnSpinLimit = 4000000000LL;

// Control block at the start of shared memory (one per CTA).
struct AttnCtrl {
  uint64_t full[kAttnStagesMax];               // a tile's K and V rows have landed
  uint32_t vmask[kAttnStagesMax][kAttnWarps];  // which of each warp's 8 tokens are in the list
  int32_t abort;
  alignas(16) float xbuf[2][kAttnWarps * 32 * 8];  // partial logits, double-buffered by tile
};

template <int HD>
struct AttnGeom {
  static constexpr int kStages = HD >= 256 ? 2 : 3;           // three CTAs per SM at HD 256
  static constexpr int kRowBytes = HD * 2;                     // one token's K (or V) row
  static constexpr int kStride = kRowBytes + 16;               // in shared memory
  static constexpr int kStageBytes = 2 * kAttnTile * kStride;  // K rows then V rows
  static constexpr int kJ = HD / 128;  // 16-byte K chunks per lane per warp (S, its head dims)
  static constexpr int kMT = HD / 64;  // m-tiles of O^T per warp (its head dims)
  static constexpr size_t kRingOff = (sizeof(AttnCtrl) + 127) & ~size_t(127);
  static constexpr size_t kSmem = kRingOff + (size_t)kStages * kStageBytes;
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// Bounded wait on an mbarrier phase.  Returns false at once when the CTA has
// aborted, and raises the abort flag when the limit is reached.
__device__ bool attn_wait(uint32_t mbar, uint32_t parity, volatile int32_t *abort_flag) {
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
    if (abort_flag != nullptr && *abort_flag) return false;
    if (clock64() - t0 > kAttnSpinLimit) {
      if (abort_flag != nullptr) *abort_flag = 1;
      return false;
    }
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
  // page of token t >= 0: t / page_size as umulhi(t, pg_mul) >> pg_shift
  // (pg_shift < 0: page_size 1, the page is t)
  uint32_t pg_mul;
  int32_t pg_shift;
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
__global__ void __launch_bounds__(32 * kAttnWarps, 3)
sparse_attn_kernel(const AttnArgs a, int32_t head_chunks) {
  using Geo = AttnGeom<HD>;
  extern __shared__ __align__(128) uint8_t attn_smem[];
  AttnCtrl &C = *reinterpret_cast<AttnCtrl *>(attn_smem);
  uint8_t *ring = attn_smem + Geo::kRingOff;
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
  volatile int32_t *abort_flag = &C.abort;

  // query head g of this chunk (zero rows past the group): this warp's head
  // dims only, in k_chunk order (j = warp * kJ + jj)
  uint32_t qa[2 * Geo::kJ][2];
  {
    const bool hv = g < heads_here;
    const uint16_t *qh =
        a.q + (int64_t)row * a.q_stride + (int64_t)(kvh * a.group + hc * 8 + (hv ? g : 0)) * HD;
#pragma unroll
    for (int jj = 0; jj < Geo::kJ; ++jj) {
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (hv) v = ldg_nc_v4(qh + 8 * k_chunk(q, warp * Geo::kJ + jj));
      qa[2 * jj][0] = v.x;
      qa[2 * jj][1] = v.y;
      qa[2 * jj + 1][0] = v.z;
      qa[2 * jj + 1][1] = v.w;
    }
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < Geo::kStages; ++s)  // one expect_tx arrival per warp
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(&C.full[s])),
                   "r"(kAttnWarps)
                   : "memory");
    C.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  // ---- producers: warp w brings tokens 8w .. 8w+7 of each tile, lanes 0..7
  // their K rows and lanes 8..15 their V rows, into the stage tile i % S.  The
  // two lookups before a tile's copies (its token, then that token's page
  // entry) run ahead in queues: tokens 2L tiles ahead, pages L tiles ahead.
  const int n_tiles = (n + kAttnTile - 1) / kAttnTile;
  const int tok_in_tile = 8 * warp + (lane & 7);  // lanes 0..15 (the rest mirror them)
  constexpr int32_t kNoToken = INT32_MIN;
  auto page_of = [&](int32_t t) -> int32_t {  // t >= 0
    return a.pg_shift < 0 ? t : (int32_t)(__umulhi((uint32_t)t, a.pg_mul) >> a.pg_shift);
  };
  auto fetch_tok = [&](int i) -> int32_t {
    const int32_t j = i * kAttnTile + tok_in_tile;
    return (i < n_tiles && j < n) ? srow[j] : kNoToken;
  };
  auto fetch_page = [&](int32_t t) -> int32_t {  // -1: outside the table
    if (t == kNoToken) return kNoToken;
    const int32_t pg = t >= 0 ? page_of(t) : -1;
    return (t >= 0 && pg < a.table_len) ? trow[pg] : -1;
  };
  auto start = [&](int i, int32_t t, int32_t phys) {  // this warp's part of tile i
    const int s = i % Geo::kStages;
    const bool ok = lane < 16 && t != kNoToken && phys >= 0 && phys < a.pool_pages;
    if (lane < 8 && t != kNoToken && !ok) report_error(a.status, kErrTokenRange, row);
    const uint32_t bal = __ballot_sync(0xffffffffu, ok);
    const uint32_t mb = smem_u32(&C.full[s]);
    if (lane == 0) {
      C.vmask[s][warp] = (bal & 0xFFu) << (8 * warp);
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mb),
                   "r"((uint32_t)__popc(bal) * (uint32_t)Geo::kRowBytes)
                   : "memory");
    }
    __syncwarp();
    if (ok) {
      const int32_t pg = page_of(t);
      const int64_t src_row = ((int64_t)phys * a.page_size + (t - pg * a.page_size)) * a.nkv + kvh;
      const uint16_t *src = (lane < 8 ? a.k_pool : a.v_pool) + src_row * HD;
      const uint8_t *dst = ring + (size_t)s * Geo::kStageBytes +
                           (lane < 8 ? 0 : kAttnTile * Geo::kStride) + tok_in_tile * Geo::kStride;
      asm volatile(
          "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
              "r"(smem_u32(dst)), "l"(src), "r"((uint32_t)Geo::kRowBytes), "r"(mb)
          : "memory");
    }
  };
  constexpr int kLook = 3, kLook2 = 2 * kLook;
  int issued = 0;
  int32_t tokq[kLook2], pageq[kLook];
  {
    int32_t tok_pre[Geo::kStages + kLook2], page_pre[Geo::kStages + kLook];
#pragma unroll
    for (int k = 0; k < Geo::kStages + kLook2; ++k) tok_pre[k] = fetch_tok(k);
#pragma unroll
    for (int k = 0; k < Geo::kStages + kLook; ++k) page_pre[k] = fetch_page(tok_pre[k]);
#pragma unroll
    for (int k = 0; k < Geo::kStages; ++k)
      if (k < n_tiles) {
        start(k, tok_pre[k], page_pre[k]);
        ++issued;
      }
#pragma unroll
    for (int k = 0; k < kLook2; ++k) tokq[k] = tok_pre[Geo::kStages + k];  // tiles S .. S + 2L - 1
#pragma unroll
    for (int k = 0; k < kLook; ++k) pageq[k] = page_pre[Geo::kStages + k];  // tiles S .. S + L - 1
  }

  float m_run = -INFINITY;  // running max of head g's logits (log2 units), same in every warp
  float l_run = 0.f;        // this lane's part of head g's weight sum
  float acc[Geo::kMT][4];
#pragma unroll
  for (int t = 0; t < Geo::kMT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
  for (int i = 0; i < n_tiles; ++i) {
    const int s = i % Geo::kStages;
    // every warp runs every iteration and every barrier; after an abort the
    // waits return at once and the results are discarded
    // (every lane waits: each acquires the bulk copies' writes for itself)
    const bool okw = __all_sync(
        0xffffffffu, attn_wait(smem_u32(&C.full[s]), (uint32_t)(i / Geo::kStages) & 1u, abort_flag));
    const uint8_t *kt = ring + (size_t)s * Geo::kStageBytes;
    const uint8_t *vt = kt + kAttnTile * Geo::kStride;
    uint32_t vb = 0;
    if (okw) {
#pragma unroll
      for (int w = 0; w < kAttnWarps; ++w) vb |= C.vmask[s][w];
    }

    // ---- this warp's part of S = Q K^T: its head dims, four 8-token n-tiles
    float sc[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
    for (int jj = 0; jj < Geo::kJ; ++jj) {
      const int c = k_chunk(q, warp * Geo::kJ + jj);
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const uint4 kv = *reinterpret_cast<const uint4 *>(kt + (g + 8 * nt) * Geo::kStride + 16 * c);
        mma_bf16(sc[nt], qa[2 * jj][0], 0u, qa[2 * jj][1], 0u, kv.x, kv.y);
        mma_bf16(sc[nt], qa[2 * jj + 1][0], 0u, qa[2 * jj + 1][1], 0u, kv.z, kv.w);
      }
    }
    // partial logits of head g at tile tokens 2q + 8nt, +1 (nt = 0..3), summed
    // over the warps in a fixed order so every warp holds the same values
    float4 *xb = reinterpret_cast<float4 *>(C.xbuf[i & 1]);
    xb[2 * (warp * 32 + lane)] = make_float4(sc[0][0], sc[0][1], sc[1][0], sc[1][1]);
    xb[2 * (warp * 32 + lane) + 1] = make_float4(sc[2][0], sc[2][1], sc[3][0], sc[3][1]);
    __syncthreads();
    // every warp is past tile i - 1: its stage takes tile i - 1 + S
    const bool aborted = __shfl_sync(0xffffffffu, *abort_flag, 0) != 0;  // one verdict per warp
    if (i >= 1 && issued < n_tiles && !aborted) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      start(issued, tokq[0], pageq[0]);  // the queues' head is tile `issued`
      ++issued;
#pragma unroll
      for (int k = 0; k + 1 < kLook; ++k) pageq[k] = pageq[k + 1];
      pageq[kLook - 1] = fetch_page(tokq[kLook]);  // token loaded kLook tiles ago
#pragma unroll
      for (int k = 0; k + 1 < kLook2; ++k) tokq[k] = tokq[k + 1];
      tokq[kLook2 - 1] = fetch_tok(issued + kLook2 - 1);
    }
    float sv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) {
      const float4 p0 = xb[2 * (w * 32 + lane)];
      const float4 p1 = xb[2 * (w * 32 + lane) + 1];
      sv[0] += p0.x;
      sv[1] += p0.y;
      sv[2] += p0.z;
      sv[3] += p0.w;
      sv[4] += p1.x;
      sv[5] += p1.y;
      sv[6] += p1.z;
      sv[7] += p1.w;
    }
    float tmax = -INFINITY;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
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
    uint32_t pb[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) pb[k] = pack_bf16x2(exp2f(sv[2 * k] - m_use), exp2f(sv[2 * k + 1] - m_use));
    // the weights the product uses are the rounded ones: so is their sum
    l_run = l_run * alpha + (((bf16_lo(pb[0]) + bf16_hi(pb[0])) + (bf16_lo(pb[1]) + bf16_hi(pb[1]))) +
                             ((bf16_lo(pb[2]) + bf16_hi(pb[2])) + (bf16_lo(pb[3]) + bf16_hi(pb[3]))));
    if (__any_sync(0xffffffffu, alpha != 1.f)) {  // some head's maximum moved
      // O^T's columns are heads 2q, 2q+1, whose factors lanes 8q and 8q+4 hold
      const float al0 = __shfl_sync(0xffffffffu, alpha, 8 * q);
      const float al1 = __shfl_sync(0xffffffffu, alpha, 8 * q + 4);
#pragma unroll
      for (int t = 0; t < Geo::kMT; ++t) {
        acc[t][0] *= al0;
        acc[t][2] *= al0;
        acc[t][1] *= al1;
        acc[t][3] *= al1;
      }
    }

    // ---- O^T += V^T P^T for this warp's m-tiles T = warp * kMT + t: rows g,
    // g+8 of m-tile T are dims 8(g + 8c) + 2e, +1 with c = T / 4, e = T % 4
    // (in a partial tile a token outside the list contributes zeros: its stage
    // row may hold anything)
    auto pv = [&](const int ks, const uint32_t z0, const uint32_t z1, const uint32_t z2,
                  const uint32_t z3) {  // k-step ks: tile tokens 16 ks .. 16 ks + 15
      const int c = (warp * Geo::kMT) / 4;
      const int off = 16 * (g + 8 * c);
      const uint8_t *vk = vt + (16 * ks) * Geo::kStride;
      const uint4 v0 = *reinterpret_cast<const uint4 *>(vk + (2 * q) * Geo::kStride + off);
      const uint4 v1 = *reinterpret_cast<const uint4 *>(vk + (2 * q + 1) * Geo::kStride + off);
      const uint4 v2 = *reinterpret_cast<const uint4 *>(vk + (2 * q + 8) * Geo::kStride + off);
      const uint4 v3 = *reinterpret_cast<const uint4 *>(vk + (2 * q + 9) * Geo::kStride + off);
      // words e = (warp * kMT) % 4 + t of the chunk: dims 8(g + 8c) + 2e, +1
      uint32_t w0[Geo::kMT], w1[Geo::kMT], w2[Geo::kMT], w3[Geo::kMT];
      if constexpr (Geo::kMT == 4) {
        w0[0] = v0.x; w0[1] = v0.y; w0[2] = v0.z; w0[3] = v0.w;
        w1[0] = v1.x; w1[1] = v1.y; w1[2] = v1.z; w1[3] = v1.w;
        w2[0] = v2.x; w2[1] = v2.y; w2[2] = v2.z; w2[3] = v2.w;
        w3[0] = v3.x; w3[1] = v3.y; w3[2] = v3.z; w3[3] = v3.w;
      } else {  // two m-tiles: the low or the high half of the chunk
        const bool hi = (warp & 1) != 0;
        w0[0] = hi ? v0.z : v0.x; w0[1] = hi ? v0.w : v0.y;
        w1[0] = hi ? v1.z : v1.x; w1[1] = hi ? v1.w : v1.y;
        w2[0] = hi ? v2.z : v2.x; w2[1] = hi ? v2.w : v2.y;
        w3[0] = hi ? v3.z : v3.x; w3[1] = hi ? v3.w : v3.y;
      }
#pragma unroll
      for (int t = 0; t < Geo::kMT; ++t) {
        const uint32_t x0 = w0[t] & z0, x1 = w1[t] & z1, x2 = w2[t] & z2, x3 = w3[t] & z3;
        mma_bf16(acc[t], prmt(x0, x1, 0x5410u), prmt(x0, x1, 0x7632u), prmt(x2, x3, 0x5410u),
                 prmt(x2, x3, 0x7632u), pb[2 * ks], pb[2 * ks + 1]);
      }
    };
    if (vb == 0xFFFFFFFFu) {  // a whole tile (uniform over the CTA): constant masks fold away
      pv(0, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu);
      pv(1, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu);
    } else {
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        const uint32_t vk = vb >> (16 * ks);
        pv(ks, (vk >> (2 * q)) & 1u ? 0xFFFFFFFFu : 0u, (vk >> (2 * q + 1)) & 1u ? 0xFFFFFFFFu : 0u,
           (vk >> (2 * q + 8)) & 1u ? 0xFFFFFFFFu : 0u, (vk >> (2 * q + 9)) & 1u ? 0xFFFFFFFFu : 0u);
      }
    }
  }

  // ---- output: head h = 2q, 2q+1 of this warp's dims, normalised by the
  // head's weight sum (every warp holds the same one)
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
  const float l0 = __shfl_sync(0xffffffffu, l_run, 8 * q);
  const float l1 = __shfl_sync(0xffffffffu, l_run, 8 * q + 4);
  const float inv0 = l0 == 0.f ? 0.f : 1.f / l0;  // no selected token: zeros
  const float inv1 = l1 == 0.f ? 0.f : 1.f / l1;
  uint16_t *orow = a.out + (int64_t)row * a.out_stride + (int64_t)(kvh * a.group + hc * 8) * HD;
  {
    const int c = (warp * Geo::kMT) / 4;
    const int d0 = 8 * (g + 8 * c) + 2 * ((warp * Geo::kMT) % 4);  // this warp's first dim here
    uint32_t h0[Geo::kMT], h1[Geo::kMT];
#pragma unroll
    for (int t = 0; t < Geo::kMT; ++t) {
      h0[t] = pack_bf16x2(acc[t][0] * inv0, acc[t][2] * inv0);
      h1[t] = pack_bf16x2(acc[t][1] * inv1, acc[t][3] * inv1);
    }
    if constexpr (Geo::kMT == 4) {
      if (2 * q < heads_here)
        *reinterpret_cast<uint4 *>(orow + (int64_t)(2 * q) * HD + d0) = make_uint4(h0[0], h0[1], h0[2], h0[3]);
      if (2 * q + 1 < heads_here)
        *reinterpret_cast<uint4 *>(orow + (int64_t)(2 * q + 1) * HD + d0) = make_uint4(h1[0], h1[1], h1[2], h1[3]);
    } else {
      if (2 * q < heads_here)
        *reinterpret_cast<uint2 *>(orow + (int64_t)(2 * q) * HD + d0) = make_uint2(h0[0], h0[1]);
      if (2 * q + 1 < heads_here)
        *reinterpret_cast<uint2 *>(orow + (int64_t)(2 * q + 1) * HD + d0) = make_uint2(h1[0], h1[1]);
    }
  }
  if (*abort_flag && threadIdx.x == 0) report_error(a.status, kErrTimeout, row);
  // the copies issued land before the CTA's shared memory is released (in a
  // run that completed, every tile was waited for already)
  if (lane == 0) {
    for (int k = max(0, issued - Geo::kStages); k < issued; ++k)
      attn_wait(smem_u32(&C.full[k % Geo::kStages]), (uint32_t)(k / Geo::kStages) & 1u, nullptr);
  }
}

template <int HD>
cudaError_t launch_attn_hd(const AttnArgs &a, int32_t n_rows, cudaStream_t stream) {
  static PerDevice smem_attr;
  const cudaError_t e = set_smem_once(smem_attr, sparse_attn_kernel<HD>, AttnGeom<HD>::kSmem);
  if (e != cudaSuccess) return e;
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
  // Division by the page size as a multiply-high and a shift (Granlund and
  // Montgomery, "Division by invariant integers using multiplication", 1994):
  // with l = ceil(log2 d), p = 31 + l and m = ceil(2^p / d) < 2^32, every
  // 0 <= t < 2^31 has t / d == (t * m) >> p, since t * (m d - 2^p) < 2^31 d
  // <= 2^p keeps the error below 1/d.
  if (page_size == 1) {
    a.pg_mul = 1u;
    a.pg_shift = -1;
  } else {
    int l = 0;
    while ((1ll << l) < page_size) ++l;
    const int p = 31 + l;
    a.pg_mul = (uint32_t)((((uint64_t)1 << p) + (uint64_t)page_size - 1) / (uint64_t)page_size);
    a.pg_shift = p - 32;
  }
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
