// Exact top-(budget/4) block selection into a u8 visibility mask.
//
// PR #1178 "select QSA indexer blocks", "Exact semantics": for a row at
// position p, blocks = (p+1)/4, tail = (p+1)%4, keep = min(budget/4, blocks);
// the keep highest scores under (score descending, block index ascending) are
// kept; the mask is 1 on their 4 tokens and on the tail, 0 elsewhere.  A row
// with blocks <= budget/4 writes its visible prefix in one pass and reads no
// score.  Otherwise each finite score maps to a monotonic u32 key (-0.0 folded
// to +0.0), 8-bit radix passes find the keep-th key, keys above it are kept
// and threshold-equal keys fill the remaining slots in ascending block order.
// A non-finite score in a truncating row's prefix is an error (recorded in the
// status word, the row left untouched; no trap).
//
// GB300 design:
//  * a row is split over a cluster of C CTAs (C = 1..16): each CTA owns a
//    contiguous, 4-aligned slice of the row's blocks and keeps its keys in
//    shared memory, so HBM sees each score once;
//  * per pass every CTA builds a 256-bin histogram of its candidates
//    (warp-aggregated with match.any), the cluster merges the C histograms
//    through distributed shared memory, and every CTA derives the same digit;
//  * ties at the final key are ranked in index order by the count of equal
//    keys in lower-ranked CTAs (read from their last histogram) plus an
//    in-CTA block scan;
//  * the mask row is written with 16-byte stores where the row is aligned.
#include "qsa_device.cuh"
#include "qsa_launch.h"

namespace qsa {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelMaxCluster = 16;
constexpr int kSelCapMax = 16384;  // keys cached per CTA (64 KiB)

struct SelectSmem {
  uint32_t hist[2][257];  // [buffer][bin], slot 256 = non-finite count
  uint32_t merged[256];
  uint32_t warp_tot[kSelWarps];
  uint32_t scan_tot[kSelWarps];
  int32_t sel_bin;
  uint32_t sel_above;
  uint32_t eq_base;
  uint32_t nonfinite;
  // keys[] follows (dynamic)
};

__device__ __forceinline__ uint32_t order_key(float s) {
  const uint32_t u = __float_as_uint(s == 0.0f ? 0.0f : s);  // fold -0.0 into +0.0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

__device__ __forceinline__ uint32_t ld_dsmem(const uint32_t *local, uint32_t rank) {
  uint32_t laddr = (uint32_t)__cvta_generic_to_shared(local);
  uint32_t raddr, v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(raddr) : "r"(laddr), "r"(rank));
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(raddr) : "memory");
  return v;
}

// Warp-aggregated histogram increment; every lane of the warp must call it.
__device__ __forceinline__ void hist_add(uint32_t *h, uint32_t bin, bool valid) {
  const unsigned act = __ballot_sync(0xffffffffu, valid);
  if (valid) {
    const unsigned peers = __match_any_sync(act, bin);
    if ((int)(threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&h[bin], (uint32_t)__popc(peers));
  }
}

// Write bytes [a, b) of a mask row: byte t = (t <= p).
__device__ void fill_visible(uint8_t *mrow, int64_t a, int64_t b, int64_t p) {
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
  for (int w = 0; w < kSelWarps; ++w) {
    const uint32_t t = warp_tot[w];
    before += (w < warp) ? t : 0u;
    tot += t;
  }
  __syncthreads();
  total = tot;
  return before + incl - v;
}

__global__ void __launch_bounds__(kSelThreads)
select_kernel(const float *__restrict__ scores, int64_t score_cols, const int32_t *__restrict__ pos,
              int32_t tokens, int32_t keep_max, uint8_t *__restrict__ mask, int32_t *status,
              int32_t C, int32_t cap) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SelectSmem &S = *reinterpret_cast<SelectSmem *>(smem_raw);
  uint32_t *keys_s = reinterpret_cast<uint32_t *>(smem_raw + ((sizeof(SelectSmem) + 15) & ~size_t(15)));

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t row = blockIdx.x / C;
  const uint32_t rank = (C > 1) ? cluster_rank() : 0u;
  const int32_t p = pos[row];
  if (p < 0 || p >= tokens) {  // uniform over the cluster: no barrier is reached
    if (rank == 0 && tid == 0) report_error(status, kErrRowRange, row);
    return;
  }
  const int32_t n = (p + 1) >> 2;
  uint8_t *mrow = mask + (int64_t)row * tokens;

  if (n <= keep_max) {  // every block kept: the visible prefix, one pass
    const int64_t span = ((int64_t)tokens + C - 1) / C;
    const int64_t a = (int64_t)rank * span;
    const int64_t b = a + span < tokens ? a + span : tokens;
    fill_visible(mrow, a, b, p);
    return;
  }

  // this CTA's slice [b0, b1) of the row's blocks, 4-aligned
  const int32_t per = (((n + C - 1) / C) + 3) & ~3;
  const int32_t b0 = min(n, (int32_t)rank * per);
  const int32_t b1 = min(n, b0 + per);
  const int32_t cnt = b1 - b0;
  const float *srow = scores + (int64_t)row * score_cols + b0;
  const int32_t cached = min(cnt, cap);

  for (int i = tid; i < 2 * 257; i += kSelThreads) (&S.hist[0][0])[i] = 0u;
  if (tid == 0) S.eq_base = 0u;
  __syncthreads();

  // ---- pass 0: load, check, key, histogram of the top byte
  {
    const int32_t nq = (cnt + 3) >> 2;
    uint32_t nonfinite = 0;
    for (int32_t qb = warp * 32; qb < nq; qb += kSelThreads) {
      const int32_t qd = qb + lane;
      const bool qv = qd < nq;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (qv) v = __ldg(reinterpret_cast<const float4 *>(srow) + qd);
      const float sv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int32_t i = 4 * qd + e;
        const bool valid = qv && i < cnt;
        uint32_t key = 0;
        if (valid) {
          if (!isfinite(sv[e])) nonfinite = 1;
          key = order_key(sv[e]);
          if (i < cached) keys_s[i] = key;
        }
        hist_add(S.hist[0], key >> 24, valid);
      }
    }
    if (nonfinite) atomicAdd(&S.hist[0][256], 1u);
  }

  uint32_t prefix = 0;   // digits found so far
  int bits = 0;          // how many of the key's top bits `prefix` holds
  uint32_t need = (uint32_t)min(keep_max, n);  // keys still to keep at/below the prefix
  bool done = false;     // every key matching the prefix is kept
  bool bad = false;      // a non-finite score somewhere in the row

  for (int pass = 0; pass < 4; ++pass) {
    const int buf = pass & 1;
    const int shift = 24 - 8 * pass;
    if (pass > 0) {  // histogram the next digit of the candidates
      for (int32_t ib = warp * 32; ib < cnt; ib += kSelThreads) {
        const int32_t i = ib + lane;
        const bool in = i < cnt;
        uint32_t key = 0;
        if (in) key = (i < cached) ? keys_s[i] : order_key(__ldg(srow + i));
        const bool cand = in && ((key >> (shift + 8)) == prefix);
        hist_add(S.hist[buf], (key >> shift) & 0xffu, cand);
      }
    }
    // publish this CTA's histogram to the cluster, then merge all of them
    if (C > 1) cluster_sync_all(); else __syncthreads();
    if (tid < 256) {
      uint32_t t = 0;
      for (int r = 0; r < C; ++r)
        t += (C > 1) ? ld_dsmem(&S.hist[buf][tid], (uint32_t)r) : S.hist[buf][tid];
      S.merged[tid] = t;
    } else if (pass == 0 && tid == 256) {
      uint32_t nf = 0;
      for (int r = 0; r < C; ++r)
        nf += (C > 1) ? ld_dsmem(&S.hist[0][256], (uint32_t)r) : S.hist[0][256];
      S.nonfinite = nf;
    }
    // the next pass fills the other buffer; every peer finished reading it
    // (previous pass's merge) before arriving at the barrier above
    if (tid < 257) S.hist[buf ^ 1][tid] = 0u;
    __syncthreads();
    if (pass == 0 && S.nonfinite != 0) {
      bad = true;
      break;
    }
    // find the digit holding the need-th largest key: inclusive scan of the
    // merged histogram from the top bin down (threads 0..255 = bins 255..0)
    uint32_t c = 0, incl = 0;
    if (tid < 256) {
      c = S.merged[255 - tid];
      incl = c;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      if (lane == 31) S.scan_tot[warp] = incl;
    }
    __syncthreads();
    if (tid < 256) {
      uint32_t before = 0;
      for (int w = 0; w < warp; ++w) before += S.scan_tot[w];
      const uint32_t hi_incl = before + incl, hi_excl = hi_incl - c;
      if (hi_excl < need && need <= hi_incl) {
        S.sel_bin = 255 - tid;
        S.sel_above = hi_excl;
      }
    }
    __syncthreads();
    const uint32_t B = (uint32_t)S.sel_bin;
    need -= S.sel_above;
    prefix = (prefix << 8) | B;
    bits += 8;
    if (S.merged[B] == need) {
      done = true;  // the whole bin is kept: no tie to rank
    } else if (pass == 3 && tid == 0) {
      // keys equal to the threshold in lower-ranked CTAs precede ours in block order
      uint32_t e = 0;
      for (uint32_t r = 0; r < rank; ++r) e += ld_dsmem(&S.hist[buf][B], r);
      S.eq_base = e;
    }
    __syncthreads();
    if (done) break;
  }

  if (!bad) {
    const uintptr_t rb = reinterpret_cast<uintptr_t>(mrow);
    const bool al16 = (rb & 15u) == 0, al4 = (rb & 3u) == 0;
    const uint32_t thresh = prefix;
    const int tshift = 32 - bits;
    uint32_t running = done ? 0u : S.eq_base;
    for (int32_t tb = 0; tb < cnt; tb += 4 * kSelThreads) {
      const int32_t i = tb + 4 * tid;
      const int m = max(0, min(4, cnt - i));
      uint32_t k[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int32_t ie = i + e;
        k[e] = (e < m) ? ((ie < cached) ? keys_s[ie] : order_key(__ldg(srow + ie))) : 0u;
      }
      uint32_t kept = 0;
      if (done) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (e < m && (k[e] >> tshift) >= thresh) kept |= 1u << e;
      } else {
        uint32_t eqc = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) eqc += (e < m && k[e] == thresh) ? 1u : 0u;
        uint32_t total;
        uint32_t r = running + block_excl_scan(eqc, S.warp_tot, total);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (e >= m) continue;
          if (k[e] > thresh) {
            kept |= 1u << e;
          } else if (k[e] == thresh) {
            if (r < need) kept |= 1u << e;
            ++r;
          }
        }
        running += total;
      }
      if (m > 0) store_blocks(mrow, (int64_t)b0 + i, m, kept, al16, al4);
    }
    // tokens past the complete blocks: the tail is visible, the rest zero
    const int64_t lo = 4 * (int64_t)n;
    const int64_t span = ((int64_t)tokens - lo + C - 1) / C;
    const int64_t a = lo + (int64_t)rank * span;
    const int64_t b = a + span < tokens ? a + span : tokens;
    fill_visible(mrow, a, b, p);
  } else if (rank == 0 && tid == 0) {
    report_error(status, kErrNonFinite, row);
  }
  // no CTA may leave while a peer can still read its histograms
  if (C > 1) cluster_sync_all();
}

static int g_max_cluster = -1;

static size_t select_smem_bytes(int32_t cap) {
  return ((sizeof(SelectSmem) + 15) & ~size_t(15)) + 4 * (size_t)(cap > 0 ? cap : 1);
}

// Largest cluster the select kernel can be co-scheduled with (16 needs the
// non-portable opt-in; fall back to 8, 4, 2 if the GPU refuses).
static int max_cluster_size() {
  if (g_max_cluster >= 0) return g_max_cluster;
  int best = 1;
  cudaFuncSetAttribute(select_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)select_smem_bytes(kSelCapMax));
  for (int c = kSelMaxCluster; c >= 2; c >>= 1) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = c;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(c);
    cfg.blockDim = dim3(kSelThreads);
    cfg.dynamicSmemBytes = select_smem_bytes(kSelCapMax);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, select_kernel, &cfg) == cudaSuccess && n > 0) {
      best = c;
      break;
    }
  }
  cudaGetLastError();  // a refused query leaves no sticky error
  g_max_cluster = best;
  return best;
}

// Cluster size for a launch: split rows whose slice would overflow the key
// cache, then keep splitting while the grid cannot fill the GPU.
int select_cluster_size(int64_t n_rows, int64_t tokens) {
  const int64_t n_max = tokens / kRatio;
  const int cmax = max_cluster_size();
  int C = 1;
  while (C < cmax && (n_max + C - 1) / C > kSelCapMax) C <<= 1;
  while (C < cmax && n_rows * C < 2 * 152 && n_max / (2 * C) >= 1024) C <<= 1;
  return C;
}

cudaError_t launch_select(const float *scores, int64_t score_cols, const int32_t *pos,
                          int32_t n_rows, int32_t tokens, int32_t budget, uint8_t *mask,
                          int32_t *status, cudaStream_t stream) {
  const int32_t keep_max = budget / kRatio;
  const int64_t n_max = (int64_t)tokens / kRatio;
  const int C = select_cluster_size(n_rows, tokens);
  const int64_t per = (((n_max + C - 1) / C) + 3) & ~int64_t(3);
  const int32_t cap = (int32_t)(per < kSelCapMax ? per : kSelCapMax);

  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3((unsigned)((int64_t)n_rows * C));
  cfg.blockDim = dim3(kSelThreads);
  cfg.dynamicSmemBytes = select_smem_bytes(cap);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = C > 1 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, select_kernel, scores, score_cols, pos, tokens, keep_max, mask,
                            status, (int32_t)C, cap);
}

}  // namespace qsa
