// Selection helpers shared by the selection kernel and the fused decode
// kernel: the monotonic order key of a score, mask-row writers, and the bin
// searches of a radix round.
//
// PR #1178 "select QSA indexer blocks", "Exact semantics": scores compare as
// floats with -0.0 equal to +0.0; a row at position p keeps the top blocks
// and its tail; mask byte t is 1 for a kept block's tokens and for t in the
// tail (4 * blocks <= t <= p).
#pragma once

#include "qsa_device.cuh"

namespace qsa {

constexpr uint32_t kZeroKey = 0x80000000u;  // order key of +0.0 (and folded -0.0)

// Monotonic u32 key of a score.  -0.0 folds into +0.0 on the bit pattern: a
// float select (s == 0 ? 0 : s) may be rewritten by the compiler in ways that
// do not keep a NaN's bits, and NaNs must land in the outer bins.
__device__ __forceinline__ uint32_t order_key(float s) {
  uint32_t u = __float_as_uint(s);
  u = (u << 1) ? u : 0u;
  // negative: all bits flipped; non-negative: the sign bit set
  return u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
}

// The float whose order key is k (for finite keys): key >= k exactly when the
// score >= key_to_float(k), since the key is monotone in the score and -0.0
// compares equal to +0.0 on both sides.
__device__ __forceinline__ float key_to_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Write bytes [a, b) of a mask row: byte t = (t <= p).
__device__ inline void fill_visible(uint8_t *mrow, int64_t a, int64_t b, int64_t p) {
  if (a >= b) return;
  const uintptr_t base = reinterpret_cast<uintptr_t>(mrow);
  int64_t va = (int64_t)(((base + (uintptr_t)a + 15) & ~(uintptr_t)15) - base);
  if (va > b) va = b;
  for (int64_t t = a + threadIdx.x; t < va; t += blockDim.x) mrow[t] = (t <= p) ? 1 : 0;
  const int64_t nvec = (b - va) >> 4;
  for (int64_t v = threadIdx.x; v < nvec; v += blockDim.x) {
    const int64_t t0 = va + 16 * v;
    uint4 w;
    if (t0 + 15 <= p) {
      w = make_uint4(0x01010101u, 0x01010101u, 0x01010101u, 0x01010101u);
    } else if (t0 > p) {
      w = make_uint4(0u, 0u, 0u, 0u);
    } else {
      uint32_t q[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint32_t x = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) x |= (t0 + 4 * k + e <= p ? 1u : 0u) << (8 * e);
        q[k] = x;
      }
      w = make_uint4(q[0], q[1], q[2], q[3]);
    }
    *reinterpret_cast<uint4 *>(mrow + t0) = w;
  }
  for (int64_t t = va + 16 * nvec + threadIdx.x; t < b; t += blockDim.x) mrow[t] = (t <= p) ? 1 : 0;
}

// Store the 4 mask bytes of blocks [blk, blk+cnt) (cnt <= 4) from bit flags.
__device__ __forceinline__ void store_blocks(uint8_t *mrow, int64_t blk, int cnt, uint32_t kept,
                                             bool aligned16, bool aligned4) {
  uint8_t *dst = mrow + 4 * blk;
  if (cnt == 4 && aligned16) {
    *reinterpret_cast<uint4 *>(dst) =
        make_uint4((kept & 1) ? 0x01010101u : 0u, (kept & 2) ? 0x01010101u : 0u,
                   (kept & 4) ? 0x01010101u : 0u, (kept & 8) ? 0x01010101u : 0u);
  } else if (aligned4) {
    for (int e = 0; e < cnt; ++e)
      reinterpret_cast<uint32_t *>(dst)[e] = ((kept >> e) & 1) ? 0x01010101u : 0u;
  } else {
    for (int e = 0; e < 4 * cnt; ++e) dst[e] = ((kept >> (e >> 2)) & 1) ? 1 : 0;
  }
}

// Exclusive block-wide scan of v (all threads call); returns the exclusive
// prefix and writes the block total to *total.
template <int NT>
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t *warp_tot, uint32_t &total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  uint32_t before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) {
    const uint32_t t = warp_tot[w];
    before += (w < warp) ? t : 0u;
    tot += t;
  }
  __syncthreads();
  total = tot;
  return before + incl - v;
}

// Find the bin of histogram M[nb] (shared memory) that holds the need-th
// largest key, scanning bins from the top: *sel_bin gets the bin, *sel_above
// the number of keys in higher bins, *sel_total (if given) the histogram's
// total (all in shared memory, read after the call; *sel_bin is left as it was
// when the total is below need).  Every thread of the CTA calls it; warp_tot
// holds NT / 32 words.
template <int NT>
__device__ __forceinline__ void find_bin(const uint32_t *M, int nb, uint32_t need,
                                         uint32_t *warp_tot, int32_t *sel_bin,
                                         uint32_t *sel_above, uint32_t *sel_total = nullptr) {
  const int tid = threadIdx.x;
  const int per = (nb + NT - 1) / NT;
  const int hi = nb - 1 - tid * per;  // this thread's bins: hi, hi-1, ..., hi-per+1
  uint32_t sum = 0;
  for (int j = 0; j < per; ++j)
    if (hi - j >= 0) sum += M[hi - j];
  uint32_t total;
  const uint32_t before = block_excl_scan<NT>(sum, warp_tot, total);
  if (sel_total != nullptr && tid == 0) *sel_total = total;
  if (before < need && need <= before + sum) {
    uint32_t acc = before;
    for (int j = 0; j < per; ++j) {
      const uint32_t c = M[hi - j];
      if (acc + c >= need) {
        *sel_bin = hi - j;
        *sel_above = acc;
        break;
      }
      acc += c;
    }
  }
  __syncthreads();
}

// find_bin for two ranks at once (one scan): the bins holding the need_a-th
// and the need_b-th largest keys (1 <= need_a, need_b <= the histogram's
// total), written to bins[0] and bins[1] (shared memory, read after the call).
template <int NT>
__device__ __forceinline__ void find_two_bins(const uint32_t *M, int nb, uint32_t need_a,
                                              uint32_t need_b, uint32_t *warp_tot, int32_t *bins) {
  const int tid = threadIdx.x;
  const int per = (nb + NT - 1) / NT;
  const int hi = nb - 1 - tid * per;  // this thread's bins: hi, hi-1, ..., hi-per+1
  uint32_t sum = 0;
  for (int j = 0; j < per; ++j)
    if (hi - j >= 0) sum += M[hi - j];
  uint32_t total;
  const uint32_t before = block_excl_scan<NT>(sum, warp_tot, total);
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const uint32_t need = k == 0 ? need_a : need_b;
    if (before < need && need <= before + sum) {
      uint32_t acc = before;
      for (int j = 0; j < per; ++j) {
        acc += M[hi - j];
        if (acc >= need) {
          bins[k] = hi - j;
          break;
        }
      }
    }
  }
  __syncthreads();
}

// One warp's version of find_bin for the small rounds (nb <= 256): the bin
// of H holding the need-th largest key and the count above it, returned to
// every lane.  Warp-synchronous: no block barrier.
__device__ __forceinline__ void warp_find_bin(const uint32_t *H, int nb, uint32_t need, int lane,
                                              uint32_t &bin, uint32_t &above) {
  const int per = (nb + 31) / 32;
  const int hi = nb - 1 - lane * per;  // this lane's bins, from the top
  uint32_t sum = 0;
  for (int j = 0; j < per; ++j)
    if (hi - j >= 0) sum += H[hi - j];
  uint32_t incl = sum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  const uint32_t before = incl - sum;
  const bool mine = before < need && need <= incl;
  uint32_t mb = 0, ma = 0;
  if (mine) {
    uint32_t acc = before;
    for (int j = 0; j < per; ++j) {
      const uint32_t c = H[hi - j];
      if (acc + c >= need) {
        mb = (uint32_t)(hi - j);
        ma = acc;
        break;
      }
      acc += c;
    }
  }
  const int src = __ffs(__ballot_sync(0xffffffffu, mine)) - 1;
  bin = __shfl_sync(0xffffffffu, mb, src);
  above = __shfl_sync(0xffffffffu, ma, src);
}

}  // namespace qsa
