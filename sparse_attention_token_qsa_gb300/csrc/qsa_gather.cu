// Selected token lists and the gather of their K/V rows.
//
// metrale layers/qsa.rs, decode_select after its top-k: the selected tokens
// are every kept block's four tokens, blocks ascending, then the row's tail --
// exactly the tokens whose mask byte is set, in ascending order -- and their
// K and V rows are gathered from the paged attention cache into a contiguous
// scratch (QsaSelection: NHD k/v scratch that the paged decode attention reads
// through an identity block table).
//
// mask_tokens_kernel: one CTA per row; 64 mask bytes per thread per chunk of
// 65536 tokens, the set bytes of each 4-byte word found with a carry-free byte
// test, a block scan of the per-thread counts gives each thread its output
// offset, and the list is written in ascending order.  Traffic: 1 B read per
// token, 4 B written per selected token.
//
// gather_kv_kernel: one warp per selected token; the token's page comes from
// the row's page table, and its K and V rows (width bf16 each) are copied with
// 16-byte loads, all of a lane's loads in flight before its stores.  Traffic:
// 4 * width B per selected token (read K and V, write both), HBM-bound.
#include "qsa_device.cuh"
#include "qsa_launch.h"

namespace qsa {

namespace {

constexpr int kTokThreads = 1024;
constexpr int kTokPerThread = 64;  // four 16-byte words of mask
constexpr int64_t kTokChunk = (int64_t)kTokThreads * kTokPerThread;
constexpr int kGatherWarps = 8;  // tokens per CTA

// Bit e of the result is set iff byte e of w is non-zero (e < 4): a byte's top
// bit after adding 0x7F to its low seven bits, or'ed with the byte itself, is
// set iff the byte is non-zero (no carry crosses bytes).
__device__ __forceinline__ uint32_t nonzero_nibble(uint32_t w) {
  const uint32_t x = ((((w & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) | w) & 0x80808080u) >> 7;
  return (x | (x >> 7) | (x >> 14) | (x >> 21)) & 0xFu;
}

// One CTA per row.  The row is read from its first 16-byte boundary on in
// chunks of 65536 tokens, 64 per thread, all of a thread's loads in flight at
// once; the bytes before that boundary (fewer than 16) are thread 0's, ahead of
// its own 64, and a ragged end is read byte by byte.  One block scan per chunk
// gives every thread the place of its first token in the list.
__global__ void __launch_bounds__(kTokThreads)
mask_tokens_kernel(const uint8_t *__restrict__ mask, int32_t tokens, int32_t *__restrict__ sel,
                   int64_t sel_cols, int32_t *__restrict__ n_sel) {
  __shared__ uint32_t warp_tot[kTokThreads / 32];
  grid_dependency_sync();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t row = blockIdx.x;
  const uint8_t *mrow = mask + (int64_t)row * tokens;
  int32_t *srow = sel + (int64_t)row * sel_cols;
  const int head = (int)min((int64_t)tokens, (int64_t)((16u - (reinterpret_cast<uintptr_t>(mrow) & 15u)) & 15u));
  uint32_t hbits = 0;  // thread 0: tokens [0, head)
  if (tid == 0)
    for (int e = 0; e < head; ++e) hbits |= (mrow[e] != 0 ? 1u : 0u) << e;
  uint32_t base = 0;  // tokens listed by earlier chunks
  for (int64_t c0 = head; c0 == head || c0 < tokens; c0 += kTokChunk) {
    const int64_t t0 = c0 + (int64_t)kTokPerThread * tid;  // this thread's 64 tokens
    const int64_t here = min((int64_t)kTokPerThread, max((int64_t)0, (int64_t)tokens - t0));
    uint64_t bits = 0;  // bit e: token t0 + e is selected
    if (here == kTokPerThread) {
      uint4 v[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) v[k] = *reinterpret_cast<const uint4 *>(mrow + t0 + 16 * k);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        bits |= (uint64_t)nonzero_nibble(v[k].x) << (16 * k);
        bits |= (uint64_t)nonzero_nibble(v[k].y) << (16 * k + 4);
        bits |= (uint64_t)nonzero_nibble(v[k].z) << (16 * k + 8);
        bits |= (uint64_t)nonzero_nibble(v[k].w) << (16 * k + 12);
      }
    } else {
      for (int e = 0; e < here; ++e) bits |= (uint64_t)(mrow[t0 + e] != 0 ? 1u : 0u) << e;
    }
    const bool lead = tid == 0 && c0 == head;  // thread 0 lists the head first
    const uint32_t cnt = (uint32_t)__popcll(bits) + (lead ? (uint32_t)__popc(hbits) : 0u);
    uint32_t incl = cnt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    uint32_t before = 0, total = 0;
#pragma unroll
    for (int j = 0; j < kTokThreads / 32; ++j) {
      const uint32_t t = warp_tot[j];
      before += j < warp ? t : 0u;
      total += t;
    }
    uint32_t at = base + before + incl - cnt;
    if (lead) {
      for (uint32_t h = hbits; h; h &= h - 1) {
        if ((int64_t)at < sel_cols) srow[at] = __ffs(h) - 1;
        ++at;
      }
    }
    for (; bits; bits &= bits - 1) {
      if ((int64_t)at < sel_cols) srow[at] = (int32_t)(t0 + __ffsll((long long)bits) - 1);
      ++at;
    }
    base += total;
    __syncthreads();  // warp_tot is rewritten by the next chunk
  }
  if (tid == 0) n_sel[row] = (int32_t)base;
}

// Row `row`'s j-th selected token, copied by the calling warp.
__device__ __forceinline__ void gather_one(const uint16_t *__restrict__ k_pool,
                                           const uint16_t *__restrict__ v_pool, int32_t width,
                                           int32_t pool_pages, const int32_t *__restrict__ table,
                                           int32_t table_len, int64_t table_cols, int32_t page_size,
                                           const int32_t *__restrict__ sel, int64_t sel_cols,
                                           const int32_t *__restrict__ n_sel, int32_t max_sel,
                                           uint16_t *__restrict__ k_out,
                                           uint16_t *__restrict__ v_out, int64_t out_rows,
                                           int32_t *status, int32_t row, int32_t j, int lane) {
  const int32_t n = min(n_sel[row], max_sel);
  if (j >= n) return;
  const int32_t t = sel[(int64_t)row * sel_cols + j];
  const int32_t pg = t >= 0 ? t / page_size : -1;
  if (t < 0 || pg >= table_len) {
    if (lane == 0) report_error(status, kErrTokenRange, row);
    return;
  }
  const int32_t phys = table[(int64_t)row * table_cols + pg];
  if (phys < 0 || phys >= pool_pages) {  // a page the pool does not have: nothing is read
    if (lane == 0) report_error(status, kErrTokenRange, row);
    return;
  }
  const int64_t slot = (int64_t)phys * page_size + t % page_size;
  const uint4 *ks = reinterpret_cast<const uint4 *>(k_pool + slot * width);
  const uint4 *vs = reinterpret_cast<const uint4 *>(v_pool + slot * width);
  uint4 *kd = reinterpret_cast<uint4 *>(k_out + ((int64_t)row * out_rows + j) * width);
  uint4 *vd = reinterpret_cast<uint4 *>(v_out + ((int64_t)row * out_rows + j) * width);
  const int nv = width / 8;  // 16-byte vectors per row
  for (int v0 = 0; v0 < nv; v0 += 64) {  // 2 K + 2 V vectors per lane in flight
    uint4 a[2], b[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int v = v0 + u * 32 + lane;
      if (v < nv) {
        a[u] = ldg_nc_v4(ks + v);
        b[u] = ldg_nc_v4(vs + v);
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int v = v0 + u * 32 + lane;
      if (v < nv) {
        kd[v] = a[u];
        vd[v] = b[u];
      }
    }
  }
}

__global__ void __launch_bounds__(32 * kGatherWarps)
gather_kv_kernel(const uint16_t *__restrict__ k_pool, const uint16_t *__restrict__ v_pool,
                 int32_t width, int32_t pool_pages, const int32_t *__restrict__ table,
                 int32_t table_len, int64_t table_cols, int32_t page_size,
                 const int32_t *__restrict__ sel,
                 int64_t sel_cols, const int32_t *__restrict__ n_sel, int32_t max_sel,
                 uint16_t *__restrict__ k_out, uint16_t *__restrict__ v_out, int64_t out_rows,
                 int32_t *status, int32_t n_rows) {
  grid_dependency_sync();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int32_t j = blockIdx.x * kGatherWarps + warp;
  for (int32_t row = blockIdx.y; row < n_rows; row += gridDim.y)
    gather_one(k_pool, v_pool, width, pool_pages, table, table_len, table_cols, page_size, sel,
               sel_cols, n_sel, max_sel, k_out, v_out, out_rows, status, row, j, lane);
}

}  // namespace

cudaError_t launch_mask_tokens(const uint8_t *mask, int32_t n_rows, int32_t tokens, int32_t *sel,
                               int64_t sel_cols, int32_t *n_sel, cudaStream_t stream) {
  return launch_dependent(mask_tokens_kernel, dim3((unsigned)n_rows), dim3(kTokThreads), 0, stream,
                          1u, mask, tokens, sel, sel_cols, n_sel);
}

cudaError_t launch_gather_kv(const uint16_t *k_pool, const uint16_t *v_pool, int32_t width,
                             int32_t pool_pages, const int32_t *table, int32_t table_len,
                             int64_t table_cols,
                             int32_t page_size, const int32_t *sel, int64_t sel_cols,
                             const int32_t *n_sel, int32_t n_rows, int32_t max_sel,
                             uint16_t *k_out, uint16_t *v_out, int64_t out_rows, int32_t *status,
                             cudaStream_t stream) {
  const dim3 grid((unsigned)((max_sel + kGatherWarps - 1) / kGatherWarps),
                  (unsigned)min(n_rows, 65535));
  return launch_dependent(gather_kv_kernel, grid, dim3(32 * kGatherWarps), 0, stream, 1u, k_pool,
                          v_pool, width, pool_pages, table, table_len, table_cols, page_size, sel,
                          sel_cols, n_sel, max_sel, k_out, v_out, out_rows, status, n_rows);
}

}  // namespace qsa
