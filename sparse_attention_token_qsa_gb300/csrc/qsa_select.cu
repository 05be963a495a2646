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
//  * a row is split over a cluster of C CTAs (C = 1..16) only when its blocks
//    overflow one CTA's key cache: each CTA owns a contiguous, 4-aligned slice
//    of the row's blocks and keeps its keys in shared memory, so HBM sees
//    each score once;
//  * the first round histograms the top 12 bits of every key as it is loaded
//    (exact zeros, the heavy bin of relu scores, go to one spare bin per lane
//    and are folded in afterwards); a non-finite score shows up as a count in
//    one of the 16 outer bins, so no per-key check is needed.  In a cluster
//    every CTA finds the selected bin itself from its peers' shared memory,
//    without merging the 4096 bins: a window below its own highest bin in one
//    read, else the ranks' sums over runs of 64 bins, then the chosen run's;
//  * one pass over the keys then writes the final mask bytes of every key
//    outside the selected bin and marks the quads that hold the bin's keys; a
//    second, short walk over the marked quads lists those keys (with their
//    block indices) as candidates; rounds of 8, 8 and 4 bits run on the
//    candidates only (stopping once the keys left are all one key), and exact
//    ties at the final key are cut on the block index (lowest indices kept).
//    On one CTA the rounds run on its list, ties cut by a bitmap or radix
//    rounds on the indices.  In a cluster of the key-caching shape each list
//    stays in its CTA: a round's digit counts, and each rank's key range and
//    count under the prefix, are read from the peers, every CTA reaches the
//    same bins, and ties are cut by the ranks' counts (ranks own ascending
//    slices) and a bitmap in the one CTA where the cut falls.  (Clusters of
//    the other shape, for rows past 65536 blocks in many-row launches, gather
//    the lists in rank 0, which runs the rounds and hands out the result);
//  * every CTA then patches the mask bytes of its own candidates.  A bin too
//    large for the candidate list falls back to rounds over every key, with
//    ties ranked by a block scan in the mask pass.
#include "qsa_device.cuh"
#include "qsa_launch.h"
#include "qsa_select_util.cuh"

namespace qsa {

// Two block shapes: 512 threads with the row's keys cached in shared memory
// (two CTAs per SM) for launches with few rows, where latency matters; 256
// threads that re-read keys from L2 instead (four smaller CTAs per SM hide
// each other's barrier phases) for launches with many rows.
constexpr int kSelMaxWarps = 16;
constexpr int kSelMaxCluster = 16;
constexpr int kSelCapMax = 16384;  // keys cached per CTA (64 KiB)

// Radix rounds over the 32-bit order key: round 0 takes the top 12 bits
// (4096 bins: sign, exponent and 3 mantissa bits, so one round already splits
// a binade eight ways), rounds 1..3 take 8, 8 and 4 bits.
constexpr int kRounds = 4;
__host__ __device__ constexpr int round_bins(int r) { return r == 0 ? 4096 : (r == 3 ? 16 : 256); }
// key >> round_shift(r) = the prefix known after round r
__host__ __device__ constexpr int round_shift(int r) { return r == 0 ? 20 : (r == 1 ? 12 : (r == 2 ? 4 : 0)); }
constexpr int kCandCap = 4096;  // keys of round 0's bin kept for rounds 1..3
// The shape without a key cache holds half as many when no row of the launch
// can take the sampled band (rows up to 32768 blocks), which lets six CTAs
// share an SM instead of five (the 64k prefill chunk: 197 -> 192 us a step).
constexpr int kCandCapShort = 2048;

constexpr int kZeroLanes = 32;  // round 0 counts exact zeros in one spare bin per lane

struct SelectSmem {
  // per-round histograms; in a cluster round 0's is merged in place.  Round
  // 0's has kZeroLanes spare bins past its 4096, folded into the zero bin.
  uint32_t hist0[4096 + kZeroLanes];
  uint32_t hist1[256];
  uint32_t hist2[256];
  uint32_t hist3[16];
  uint32_t warp_tot[kSelMaxWarps];
  uint32_t msmall[256];  // rounds 1..3 merged over a cluster (fallback path)
  uint32_t roff[kSelMaxCluster + 1];  // rank 0: where each rank's candidates start
  uint32_t rule_prefix;  // the kept set: (key >> rule_shift) > rule_prefix, or equal
  uint32_t rule_shift;   //   to it at a block index <= rule_cut
  int32_t rule_cut;
  uint32_t ncand;
  int32_t sel_bin;
  uint32_t sel_above;
  uint32_t eq_base;
  uint32_t band_hi;  // sampled band: keys at or above its upper edge
  int32_t band_bin[2];  // sampled band: its top and bottom bins
  int32_t rsel[kRounds];     // each candidate round's bin ...
  uint32_t rabove[kRounds];  // ... and the keys above it
  uint32_t kmin, kmax;       // the candidates under the prefix: their key range
  uint32_t coarse[64];       // in a cluster: this CTA's round-0 counts over runs of 64 bins
  uint32_t lmax;             // in a cluster: this CTA's highest non-empty round-0 bin
  uint32_t rowmax;           // ... and the row's
  uint32_t sel_cnt;          // in a cluster: the selected round-0 bin's count over the cluster
  // in a cluster, per candidate round r (1..3, and 4 for a final check):
  uint32_t rcnt[kRounds];          //   the round's bin count over the cluster
  uint32_t kmin_r[kRounds + 1];    //   this CTA's candidates under the prefix: lowest key,
  uint32_t kmax_r[kRounds + 1];    //   highest key
  uint32_t kcnt_r[kRounds + 1];    //   and count
  uint32_t one_key;                // every rank's candidates under the prefix hold one key ...
  uint32_t one_key_val;            // ... this one
  uint32_t tbefore;                // ... and the lower ranks hold this many of them
  // cand keys [CAND] u32, cand local indices [CAND] u16, keys[] follow (dynamic)
};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Cluster barrier whose release covers shared memory only: the CTAs of a
// cluster exchange nothing but their shared memory (no CTA reads another's
// global writes), so an arrive need not wait for the mask stores in flight.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "fence.release.sync_restrict::shared::cta.cluster;\n\t"
      "barrier.cluster.arrive.relaxed.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}

__device__ __forceinline__ uint32_t ld_dsmem(const uint32_t *local, uint32_t rank) {
  uint32_t laddr = (uint32_t)__cvta_generic_to_shared(local);
  uint32_t raddr, v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(raddr) : "r"(laddr), "r"(rank));
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(raddr) : "memory");
  return v;
}

__device__ __forceinline__ uint16_t ld_dsmem_u16(const uint16_t *local, uint32_t rank) {
  uint32_t laddr = (uint32_t)__cvta_generic_to_shared(local);
  uint32_t raddr;
  uint16_t v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(raddr) : "r"(laddr), "r"(rank));
  asm volatile("ld.shared::cluster.u16 %0, [%1];" : "=h"(v) : "r"(raddr) : "memory");
  return v;
}

// Bin b of H summed over the cluster's C ranks (one thread per bin: the
// loads of a warp read 32 consecutive bins of one rank at a time).
__device__ __forceinline__ uint32_t cluster_bin(const uint32_t *H, int b, int C) {
  uint32_t v[kSelMaxCluster];
#pragma unroll
  for (int q = 0; q < kSelMaxCluster; ++q) v[q] = q < C ? ld_dsmem(&H[b], (uint32_t)q) : 0u;
  uint32_t t = 0;
#pragma unroll
  for (int q = 0; q < kSelMaxCluster; ++q) t += v[q];
  return t;
}

// Round 0's bin over a cluster and the non-finite verdict (the 16 outer
// bins).  First, in one read of the peers: the kWin0 bins ending 32 above
// this CTA's own highest one, summed over the ranks, with the ranks' highest
// bins.  If that window reaches the row's highest bin and holds at least
// need keys, the need-th key's bin is in it (no key lies above it).
// Otherwise, in two levels: the ranks' 64 run sums, then the chosen run's 64
// bins of every rank.  Every CTA reaches the same bin, whichever way.  Every
// thread of the CTA calls it; the results land in S.sel_bin / sel_above /
// sel_cnt and the verdict is returned.
constexpr int kWin0 = 128;

template <int NT>
__device__ __forceinline__ bool cluster_find_round0(SelectSmem &S, int C, uint32_t need) {
  static_assert(NT >= kWin0 + 64, "the window, the outer bins and the ranks' maxima need their own threads");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t *M = S.msmall;  // merged window bins; else run sums, then the run's bins
  const int w0 = min(max((int)S.lmax + 32 - (kWin0 - 1), 0), 4096 - kWin0);
  bool nf = false;
  if (tid < kWin0) {
    M[tid] = cluster_bin(S.hist0, w0 + tid, C);
  } else if (tid < kWin0 + 16) {
    const int o = tid - kWin0;
    nf = cluster_bin(S.hist0, o < 8 ? o : 4088 + (o - 8), C) != 0u;
  } else if (warp == kWin0 / 32 + 1) {
    uint32_t m = lane < C ? ld_dsmem(&S.lmax, (uint32_t)lane) : 0u;
    m = __reduce_max_sync(0xffffffffu, m);
    if (lane == 0) S.rowmax = m;
  }
  if (__syncthreads_or(nf)) return true;
  if (S.rowmax <= (uint32_t)(w0 + kWin0 - 1)) {
    if (warp == 0) {
      uint32_t sum = 0;
#pragma unroll
      for (int j = 0; j < kWin0 / 32; ++j) sum += M[lane * (kWin0 / 32) + j];
      const uint32_t total = __reduce_add_sync(0xffffffffu, sum);
      int32_t sb = -1;
      uint32_t ab = 0, cb = 0;
      if (total >= need) {
        uint32_t B, above;
        warp_find_bin(M, kWin0, need, lane, B, above);
        sb = w0 + (int32_t)B;
        ab = above;
        cb = M[B];
      }
      if (lane == 0) {
        S.sel_bin = sb;
        S.sel_above = ab;
        S.sel_cnt = cb;
      }
    }
    __syncthreads();
    if (S.sel_bin >= 0) return false;
    __syncthreads();  // (M and sel_bin are rewritten below)
  }
  if (tid < 64) M[tid] = cluster_bin(S.coarse, tid, C);
  __syncthreads();
  if (warp == 0) {
    uint32_t B, above;
    warp_find_bin(M, 64, need, lane, B, above);
    if (lane == 0) {
      S.sel_bin = (int32_t)B;
      S.sel_above = above;
    }
  }
  __syncthreads();
  const uint32_t run = (uint32_t)S.sel_bin, above_run = S.sel_above;
  __syncthreads();  // (M and sel_bin are rewritten below)
  if (tid < 64) M[tid] = cluster_bin(S.hist0, (int)(64 * run) + tid, C);
  __syncthreads();
  if (warp == 0) {
    uint32_t B, above;
    warp_find_bin(M, 64, need - above_run, lane, B, above);
    if (lane == 0) {
      S.sel_bin = (int32_t)(64 * run + B);
      S.sel_above = above_run + above;
      S.sel_cnt = M[B];
    }
  }
  __syncthreads();
  return false;
}

// Candidate round r's bin over a cluster (H's nb bins summed over the ranks;
// nb = 0 for the final check) into S.rsel / rabove / rcnt[r]; and, from every
// rank's key range and count of the candidates under the prefix, whether
// they all hold one key (S.one_key, S.one_key_val) and how many of them the
// ranks below this one hold (S.tbefore).  Every thread of the CTA calls it.
template <int NT>
__device__ __forceinline__ void cluster_find_round(SelectSmem &S, const uint32_t *H, int nb, int r, int C,
                                                   uint32_t need, uint32_t rank) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t *M = S.msmall;
  if (tid < nb) M[tid] = cluster_bin(H, tid, C);
  if (warp == NT / 32 - 1) {  // the last warp: the ranks' key ranges and counts
    uint32_t lo = 0xFFFFFFFFu, hi = 0u, c = 0u;
    if (lane < C) {
      lo = ld_dsmem(&S.kmin_r[r], (uint32_t)lane);
      hi = ld_dsmem(&S.kmax_r[r], (uint32_t)lane);
      c = ld_dsmem(&S.kcnt_r[r], (uint32_t)lane);
    }
    lo = __reduce_min_sync(0xffffffffu, lo);
    hi = __reduce_max_sync(0xffffffffu, hi);
    const uint32_t below = __reduce_add_sync(0xffffffffu, lane < (int)rank ? c : 0u);
    if (lane == 0) {
      S.one_key = lo == hi ? 1u : 0u;
      S.one_key_val = lo;
      S.tbefore = below;
    }
  }
  __syncthreads();
  if (nb > 0 && !S.one_key && warp == 0) {
    uint32_t B, above;
    warp_find_bin(M, nb, need, lane, B, above);
    if (lane == 0) {
      S.rsel[r] = (int32_t)B;
      S.rabove[r] = above;
      S.rcnt[r] = M[B];
    }
  }
  __syncthreads();
}

// Histogram increment for one key per lane (exact zeros, the one heavy bin of
// relu scores, are counted separately by the caller with a ballot, so the
// remaining lanes of a warp rarely hit the same bin).
__device__ __forceinline__ void hist_add(uint32_t *h, uint32_t bin, bool valid) {
  if (valid) atomicAdd(&h[bin], 1u);
}

template <int NT, bool CACHE, int CAND = kCandCap>
__global__ void __launch_bounds__(NT, NT == 256 ? (CAND <= kCandCapShort ? 6 : 5) : 2)
select_kernel(const float *__restrict__ scores, int64_t score_cols, const int32_t *__restrict__ pos,
              int32_t tokens, int32_t keep_max, uint8_t *__restrict__ mask, int32_t *status,
              int32_t C, int32_t cap) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SelectSmem &S = *reinterpret_cast<SelectSmem *>(smem_raw);
  uint32_t *cand_s =
      reinterpret_cast<uint32_t *>(smem_raw + ((sizeof(SelectSmem) + 15) & ~size_t(15)));
  uint16_t *cand_li = reinterpret_cast<uint16_t *>(cand_s + CAND);
  uint32_t *keys_s = reinterpret_cast<uint32_t *>(cand_li + CAND);

  grid_dependency_sync();
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
  const int32_t cached = CACHE ? min(cnt, cap) : 0;
  {
    // tokens past the complete blocks (the tail visible, the rest zero) depend
    // on no score: their stores drain while the scores load
    const int64_t lo = 4 * (int64_t)n;
    const int64_t span = ((int64_t)tokens - lo + C - 1) / C;
    const int64_t a = lo + (int64_t)rank * span;
    const int64_t b = a + span < tokens ? a + span : tokens;
    fill_visible(mrow, a, b, p);
  }
  if (!CACHE && cnt <= 16384) {
    // a slice of up to 64 KiB heads for L2 at once (two requests a thread):
    // the loads below then wait on L2, not on HBM.  (A longer slice would
    // crowd L2 out across the resident CTAs; the sampled band prefetches its
    // own first batches.)
    for (int32_t l = 32 * tid; l < cnt; l += 32 * NT)  // 32 scores: one 128-byte line
      asm volatile("prefetch.global.L2 [%0];" ::"l"(srow + l));
  }

  for (int i = tid; i < 4096 + kZeroLanes + 256 + 256 + 16; i += NT) (&S.hist0[0])[i] = 0u;
  if (tid == 0) {
    S.ncand = 0u;
    S.eq_base = 0u;
    S.band_hi = 0u;
    S.lmax = 0u;
#pragma unroll
    for (int r = 0; r <= kRounds; ++r) {
      S.kmin_r[r] = 0xFFFFFFFFu;
      S.kmax_r[r] = 0u;
      S.kcnt_r[r] = 0u;
    }
  }
  __syncthreads();

  uint32_t need = (uint32_t)min(keep_max, n);  // keys still to keep at/below the prefix
  bool bad = false;        // a non-finite score somewhere in the row
  bool scan_ties = false;  // fallback: ties ranked by a block scan in the mask pass
  bool cand_path = false;  // mask written during compaction; candidates patched after
  uint32_t own_n = 0;      // this CTA's own candidates (at the start of its list)
  uint32_t prefix = 0;     // fallback state: the threshold's top bits so far ...
  int shift = 32;          // ... prefix = threshold >> shift
  bool rule_ready = false;  // the kept set is known: no candidate rounds

  // ---- sampled band (a row on one CTA, long enough for a sample).  kRun * NT
  // scores in runs of kRun, spread evenly over the row, are histogrammed on the
  // top 12 key bits.  With r = need * samples / n, the bins holding the
  // sample's (r - d)-th and (r + d)-th largest keys (d = 3 sqrt(r) + 2) bound
  // a band [t_lo, t_hi) that holds the row's keep-th key unless the sample is
  // far off.  One pass over the row then writes every key's mask bytes (kept
  // at or above t_hi, dropped below t_lo, dropped for now inside the band),
  // counts the kept keys and lists the band's keys as candidates.  If the
  // counts put the keep-th key in the band and the list fits, the candidate
  // rounds finish the selection; otherwise (or on a non-finite score) the row
  // is selected again by the full-histogram path, which rewrites every byte.
  bool sampled = false;
  {
    constexpr int kRun = 8;  // (runs of 16 or 32 measured slower on 256k rows)
    constexpr int kSamp = kRun * NT;
    // (rows whose keys a second pass would still find in L2 are faster on the
    // full-histogram path, and the cached shape never reads a key twice)
    const bool try_sample = !CACHE && C == 1 && cnt > 32768 && cnt <= 65536 &&
                            need * (uint32_t)kSamp >= 16u * (uint32_t)cnt;
    if (try_sample) {
      const float r = (float)need * (float)kSamp / (float)cnt;
      const float d = ceilf(3.f * sqrtf(r)) + 2.f;
      const uint32_t r_hi = (uint32_t)fmaxf(1.f, floorf(r - d));
      const uint32_t r_lo = (uint32_t)ceilf(r + d);
      bool ok;
      {
        // the pass's first two batches head for L2 while the sample is read
        for (int u = 0; u < 8; ++u) {
          const int32_t qd = warp * 32 + (u >> 2) * 4 * NT + (u & 3) * NT + lane;
          if (4 * qd < cnt)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(srow + 4 * (int64_t)qd));
        }
        // run `tid` starts at a multiple of 4 at most cnt - kRun (rows are 16-byte aligned)
        const int32_t at = (int32_t)((((int64_t)tid * (cnt - kRun)) / (NT - 1)) & ~int64_t(3));
        float v[kRun];
#pragma unroll
        for (int u = 0; u < kRun / 4; ++u) {
          const float4 f = __ldg(reinterpret_cast<const float4 *>(srow + at + 4 * u));
          v[4 * u] = f.x;
          v[4 * u + 1] = f.y;
          v[4 * u + 2] = f.z;
          v[4 * u + 3] = f.w;
        }
        bool nf = false;
#pragma unroll
        for (int e = 0; e < kRun; ++e) {
          nf |= (__float_as_uint(v[e]) & 0x7F800000u) == 0x7F800000u;
          atomicAdd(&S.hist0[order_key(v[e]) >> 20], 1u);
        }
        ok = __syncthreads_or(nf) == 0;
      }
      int32_t bhi = 0, blo = 0;
      if (ok) {
        find_two_bins<NT>(S.hist0, 4096, r_hi, r_lo, S.warp_tot, S.band_bin);
        bhi = S.band_bin[0];
        blo = S.band_bin[1];
        // finite edges, and a band the 256-bin histogram below can hold
        ok = blo >= 8 && bhi <= 0xFF6 && bhi - blo < 256;
      }
      if (ok) {
        const float t_lo = key_to_float((uint32_t)blo << 20);
        const float t_hi = key_to_float((uint32_t)(bhi + 1) << 20);
        const uintptr_t rbm = reinterpret_cast<uintptr_t>(mrow);
        const bool m16 = (rbm & 15u) == 0, m4 = (rbm & 3u) == 0;
        uint32_t kept_n = 0;
        float chk = 0.f;  // stays +0 unless a score is non-finite (or a quad's sum overflows)
        // one quad of scores (mq of them in the row): its mask bytes, kept
        // count and candidates
        auto band_quad = [&](int32_t i, const float4 &f, int mq) {
          const float x[4] = {f.x, f.y, f.z, f.w};
          uint32_t w[4], bits = 0;
          float s = 0.f;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const bool in = e < mq;
            const bool kp = in && x[e] >= t_hi;
            w[e] = kp ? 0x01010101u : 0u;
            kept_n += kp ? 1u : 0u;
            bits |= (in && !kp && x[e] >= t_lo) ? (1u << e) : 0u;
            s += in ? x[e] : 0.f;
          }
          chk = fmaf(s, 0.f, chk);  // inf * 0 and NaN * 0 are NaN
          if (mq == 4 && m16) {
            *reinterpret_cast<uint4 *>(mrow + 4 * (int64_t)i) = make_uint4(w[0], w[1], w[2], w[3]);
          } else {
            store_blocks(mrow, (int64_t)i, mq,
                         (w[0] & 1u) | ((w[1] & 1u) << 1) | ((w[2] & 1u) << 2) | ((w[3] & 1u) << 3),
                         m16, m4);
          }
          if (bits) {
            uint32_t at = atomicAdd(&S.ncand, (uint32_t)__popc(bits));
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              if (bits & (1u << e)) {
                if (at < (uint32_t)CAND) {
                  cand_s[at] = order_key(x[e]);
                  cand_li[at] = (uint16_t)(i + e);
                }
                ++at;
              }
            }
          }
        };
        constexpr int kLoadsInFlight = 4;  // float4 loads issued per thread before use
        const float4 *srow4 = reinterpret_cast<const float4 *>(srow);
        const int32_t nq = (cnt + 3) >> 2, nq_full = cnt >> 2;
        int32_t qb = warp * 32;
        for (; qb + (kLoadsInFlight - 1) * NT + 32 <= nq_full; qb += NT * kLoadsInFlight) {
          float4 v[kLoadsInFlight];
#pragma unroll
          for (int u = 0; u < kLoadsInFlight; ++u) v[u] = __ldg(srow4 + qb + u * NT + lane);
#pragma unroll
          for (int u = 0; u < kLoadsInFlight; ++u) band_quad(4 * (qb + u * NT + lane), v[u], 4);
        }
        for (; qb < nq; qb += NT * kLoadsInFlight) {
          float4 v[kLoadsInFlight];
#pragma unroll
          for (int u = 0; u < kLoadsInFlight; ++u) {
            const int32_t qd = qb + u * NT + lane;
            v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (qd < nq) v[u] = __ldg(srow4 + qd);
          }
#pragma unroll
          for (int u = 0; u < kLoadsInFlight; ++u) {
            const int32_t qd = qb + u * NT + lane;
            if (qd < nq) band_quad(4 * qd, v[u], min(4, cnt - 4 * qd));
          }
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) kept_n += __shfl_xor_sync(0xffffffffu, kept_n, off);
        if (lane == 0 && kept_n) atomicAdd(&S.band_hi, kept_n);
        const bool nf = !(chk == 0.f);
        ok = __syncthreads_or(nf) == 0;  // (also the barrier before the totals are read)
        const uint32_t hi_n = S.band_hi, nc = S.ncand;
        ok = ok && hi_n <= need && hi_n + nc >= need && nc <= (uint32_t)CAND;
        if (ok) {
          sampled = true;
          cand_path = true;
          need -= hi_n;
          if (need == 0) {  // exactly the keys at or above t_hi: no candidate is kept
            rule_ready = true;
            if (tid == 0) {
              S.rule_prefix = (uint32_t)bhi;
              S.rule_shift = 20;
              S.rule_cut = -1;
            }
          } else {
            // the candidates' bins within the band: the one holding the need-th
            for (uint32_t j = tid; j < nc; j += NT)
              atomicAdd(&S.hist1[(cand_s[j] >> 20) - (uint32_t)blo], 1u);
            __syncthreads();
            if (warp == 0) {
              uint32_t B, above;
              warp_find_bin(S.hist1, bhi - blo + 1, need, lane, B, above);
              if (lane == 0) {
                S.sel_bin = (int32_t)B;
                S.sel_above = above;
              }
            }
            __syncthreads();
            need -= S.sel_above;
            prefix = (uint32_t)blo + (uint32_t)S.sel_bin;
            shift = 20;
            if (tid < 256) S.hist1[tid] = 0u;  // round 1 histograms here again
          }
        }
      }
      if (!sampled) {  // start over on the full histogram
        __syncthreads();
        for (int i = tid; i < 4096; i += NT) S.hist0[i] = 0u;
        if (tid == 0) S.ncand = 0u;
        __syncthreads();
      }
    }
  }

  if (!sampled) {
    // ---- round 0 while loading: key cache and top-12-bit histogram.  Exact
    // zeros (relu outputs, the one heavy bin) go to the lane's own spare bin,
    // so the lanes of a warp rarely add to the same bin; the spare bins are
    // folded into the zero bin afterwards.
    {
      constexpr int kLoadsInFlight = 4;  // float4 loads issued per thread before use
      const int32_t nq = (cnt + 3) >> 2;
      const uint32_t zbin = 4096u + (uint32_t)lane;
      // one quad's keys into the histogram (and the key cache); ne = its keys in
      // the slice, a constant 4 on the fast path below
      auto take = [&](const float4 &f, int32_t qd, int ne) {
        if constexpr (CACHE) {
          const uint32_t kq[4] = {order_key(f.x), order_key(f.y), order_key(f.z), order_key(f.w)};
          if (4 * qd + 3 < cached) {  // one 16-byte store per quad
            *reinterpret_cast<uint4 *>(keys_s + 4 * qd) = make_uint4(kq[0], kq[1], kq[2], kq[3]);
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (4 * qd + e < cached) keys_s[4 * qd + e] = kq[e];
          }
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (e < ne) atomicAdd(&S.hist0[kq[e] == kZeroKey ? zbin : kq[e] >> 20], 1u);
        } else {
          // no copy to keep: zeros of either sign are found on the raw bits,
          // and no other key needs the -0.0 fold
          const uint32_t uq[4] = {__float_as_uint(f.x), __float_as_uint(f.y), __float_as_uint(f.z),
                                  __float_as_uint(f.w)};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if (e < ne) {
              const uint32_t key = uq[e] ^ ((uint32_t)((int32_t)uq[e] >> 31) | 0x80000000u);
              atomicAdd(&S.hist0[(uq[e] << 1) == 0u ? zbin : key >> 20], 1u);
            }
          }
        }
      };
      const float4 *srow4 = reinterpret_cast<const float4 *>(srow);
      const int32_t nq_full = cnt >> 2;  // quads whose four keys all lie in the slice
      int32_t qb = warp * 32;
      // whole batches first: every lane's quads are full, no per-quad tests
      for (; qb + (kLoadsInFlight - 1) * NT + 32 <= nq_full; qb += NT * kLoadsInFlight) {
        float4 v[kLoadsInFlight];
#pragma unroll
        for (int u = 0; u < kLoadsInFlight; ++u) v[u] = __ldg(srow4 + qb + u * NT + lane);
#pragma unroll
        for (int u = 0; u < kLoadsInFlight; ++u) take(v[u], qb + u * NT + lane, 4);
      }
      // the rest of the slice, quad by quad
      for (; qb < nq; qb += NT * kLoadsInFlight) {
        float4 v[kLoadsInFlight];
#pragma unroll
        for (int u = 0; u < kLoadsInFlight; ++u) {
          const int32_t qd = qb + u * NT + lane;
          v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (qd < nq) v[u] = __ldg(srow4 + qd);
        }
#pragma unroll
        for (int u = 0; u < kLoadsInFlight; ++u) {
          const int32_t qd = qb + u * NT + lane;
          if (qd < nq) take(v[u], qd, min(4, cnt - 4 * qd));
        }
      }
      // the spare bins into the zero bin
      __syncthreads();
      if (tid < kZeroLanes) {
        const uint32_t z = S.hist0[4096 + tid];
        if (z) atomicAdd(&S.hist0[kZeroKey >> 20], z);
      }
    }

    // ---- round 0 over a cluster, in two levels: each CTA sums its bins in
    // runs of 64; after one cluster barrier every CTA reads the ranks' 64 run
    // sums (and the 16 outer bins), finds the run holding the need-th key,
    // then reads that run's 64 bins from every rank and finds the bin.  Every
    // CTA reaches the same bin without merging the 4096 bins.
    //
    // A score is non-finite exactly when its key lands in one of the 16 outer
    // bins: keys of -inf and negative NaNs are below 0x00800000 (bins 0..7),
    // keys of +inf and positive NaNs at or above 0xFF800000 (bins 0xFF8..0xFFF),
    // and every finite score's key lies between.
    if (C > 1) {
      __syncthreads();  // the spare bins are folded in
      {
        constexpr int kPer = 4096 / NT;    // bins per thread: 8 or 16
        constexpr int kGroup = 64 / kPer;  // threads per run of 64 bins
        const uint4 *h4 = reinterpret_cast<const uint4 *>(S.hist0 + tid * kPer);
        uint32_t t = 0, hb = 0;  // (hb: the thread's highest non-empty bin)
#pragma unroll
        for (int k = 0; k < kPer / 4; ++k) {
          const uint4 v = h4[k];
          t += v.x + v.y + v.z + v.w;
          const uint32_t b = (uint32_t)(tid * kPer + 4 * k);
          hb = v.x ? b : hb;
          hb = v.y ? b + 1u : hb;
          hb = v.z ? b + 2u : hb;
          hb = v.w ? b + 3u : hb;
        }
#pragma unroll
        for (int off = 1; off < kGroup; off <<= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
        if ((tid & (kGroup - 1)) == 0) S.coarse[tid / kGroup] = t;
        hb = __reduce_max_sync(0xffffffffu, hb);
        if (lane == 0 && hb) atomicMax(&S.lmax, hb);
      }
      cluster_sync_all();  // every rank's bins and run sums are final until the next one
      bad = cluster_find_round0<NT>(S, C, need);  // the same verdict in every CTA of the cluster
    } else {
      __syncthreads();
      const bool nf = tid < 16 && S.hist0[tid < 8 ? tid : 0xFF0 + tid] != 0u;
      bad = __syncthreads_or(nf) != 0;
    }

    if (!bad) {
      if (C == 1) find_bin<NT>(S.hist0, 4096, need, S.warp_tot, &S.sel_bin, &S.sel_above);
      const uint32_t B0 = (uint32_t)S.sel_bin;
      const uint32_t cnt0 = C > 1 ? S.sel_cnt : S.hist0[B0];
      need -= S.sel_above;
      prefix = B0;
      shift = 20;
      if (cnt0 == need) {  // the whole bin is kept
        if (tid == 0) {
          S.rule_prefix = B0;
          S.rule_shift = 20;
          S.rule_cut = INT32_MAX;
        }
        __syncthreads();
      } else if (cnt0 <= (uint32_t)CAND && per <= 65536) {
        // ---- candidate path.  One pass over this CTA's keys: the mask bytes of
        // keys above the bin (kept) and below it (dropped) are final; the bin's
        // own keys are written as dropped, appended with their local block
        // index to the candidate list (slots from a shared counter, so the list
        // is unordered) and patched once the threshold inside the bin is known.
        // About one key in 25 lies in the bin, so nearly every warp step would
        // take a listing branch: the pass only marks the thread's quads that
        // hold one, and reads those few again afterwards to list them.
        {
          const uintptr_t rbm = reinterpret_cast<uintptr_t>(mrow);
          const bool m16 = (rbm & 15u) == 0, m4 = (rbm & 3u) == 0;
          // B0 < 0xFF8 (a finite key's bin), so the upper edge does not wrap
          const uint32_t bin_lo = B0 << 20, bin_hi = (B0 + 1u) << 20;
          const float t_lo = key_to_float(bin_lo), t_hi = key_to_float(bin_hi);
          // one quad's keys against the bin's edges (keys, or raw scores against
          // the edges' floats): w = mask words (>= hi kept), bits = [lo, hi)
          auto classify = [&](const uint32_t (&k)[4], int mq, uint32_t (&w)[4]) {
            uint32_t bits = 0;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const bool in = e < mq;
              bool kp, lo;
              if constexpr (CACHE) {
                kp = k[e] >= bin_hi;
                lo = k[e] >= bin_lo;
              } else {
                kp = __uint_as_float(k[e]) >= t_hi;
                lo = __uint_as_float(k[e]) >= t_lo;
              }
              w[e] = (in && kp) ? 0x01010101u : 0u;
              bits |= (in && !kp && lo) ? (1u << e) : 0u;
            }
            return bits;
          };
          // quad i's keys (order keys from the cache, else raw score bits)
          auto fetch = [&](int32_t i, uint32_t (&k)[4]) {
            if (i + 3 < cnt && (!CACHE || i + 3 < cached)) {  // a whole quad, one 16-byte load
              if constexpr (CACHE) {
                const uint4 kv = *reinterpret_cast<const uint4 *>(keys_s + i);
                k[0] = kv.x;
                k[1] = kv.y;
                k[2] = kv.z;
                k[3] = kv.w;
              } else {
                const float4 f = __ldg(reinterpret_cast<const float4 *>(srow + i));
                k[0] = __float_as_uint(f.x);
                k[1] = __float_as_uint(f.y);
                k[2] = __float_as_uint(f.z);
                k[3] = __float_as_uint(f.w);
              }
            } else {  // the slice's last quad, or past the key cache
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                if constexpr (CACHE)
                  k[e] = (i + e < cnt) ? (i + e < cached ? keys_s[i + e] : order_key(__ldg(srow + i + e)))
                                       : 0u;
                else
                  k[e] = (i + e < cnt) ? __float_as_uint(__ldg(srow + i + e)) : 0u;
              }
            }
          };
          uint64_t marked = 0;  // bit t: the thread's t-th quad holds candidates (per <= 65536)
          // quad i (the thread's t-th): its final mask words, and its mark
          auto place = [&](int32_t i, int t, const uint32_t (&k)[4]) {
            uint32_t w[4];
            const int mq = min(4, cnt - i);
            const uint32_t bits = classify(k, mq, w);
            if (mq == 4 && m16) {
              *reinterpret_cast<uint4 *>(mrow + 4 * ((int64_t)b0 + i)) = make_uint4(w[0], w[1], w[2], w[3]);
            } else {
              store_blocks(mrow, (int64_t)b0 + i, mq,
                           (w[0] & 1u) | ((w[1] & 1u) << 1) | ((w[2] & 1u) << 2) | ((w[3] & 1u) << 3),
                           m16, m4);
            }
            marked |= bits ? (1ull << t) : 0ull;
          };
          // a whole quad, at a 16-byte aligned mask word: no per-key bounds
          // tests, and only whether it holds a candidate (the listing below
          // classifies marked quads again)
          auto place4 = [&](int32_t i, int t, const uint32_t (&k)[4]) {
            uint32_t w[4];
            bool any = false;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              bool kp, lo;
              if constexpr (CACHE) {
                kp = k[e] >= bin_hi;
                lo = k[e] >= bin_lo;
              } else {
                kp = __uint_as_float(k[e]) >= t_hi;
                lo = __uint_as_float(k[e]) >= t_lo;
              }
              w[e] = kp ? 0x01010101u : 0u;
              any |= lo && !kp;
            }
            *reinterpret_cast<uint4 *>(mrow + 4 * ((int64_t)b0 + i)) = make_uint4(w[0], w[1], w[2], w[3]);
            marked |= any ? (1ull << t) : 0ull;
          };
          int32_t i = 4 * tid, t = 0;
          if (m16) {  // two whole quads per step, both loads in flight
            for (; i + 4 * NT + 3 < cnt; i += 8 * NT, t += 2) {
              uint32_t k0[4], k1[4];
              fetch(i, k0);
              fetch(i + 4 * NT, k1);
              place4(i, t, k0);
              place4(i + 4 * NT, t + 1, k1);
            }
          }
          for (; i < cnt; i += 4 * NT, ++t) {
            uint32_t k[4];
            fetch(i, k);
            place(i, t, k);
          }
          // the marked quads again: their bin keys into the candidate list
          while (marked) {
            const int t = __ffsll((long long)marked) - 1;
            marked &= marked - 1ull;
            const int32_t i = 4 * tid + t * 4 * NT;
            uint32_t k[4], w[4];
            fetch(i, k);
            const uint32_t bits = classify(k, min(4, cnt - i), w);
            uint32_t at = atomicAdd(&S.ncand, (uint32_t)__popc(bits));
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              if (bits & (1u << e)) {
                const uint32_t key = CACHE ? k[e] : order_key(__uint_as_float(k[e]));
                cand_s[at] = key;
                cand_li[at] = (uint16_t)(i + e);
                ++at;
                // a cluster's first candidate round histograms the lists as they form
                if (CACHE && C > 1) atomicAdd(&S.hist1[(key >> 12) & 255u], 1u);
              }
            }
          }

        }
        cand_path = true;
      } else {
        scan_ties = true;  // ---- fallback: rounds over every key (part B)
      }
    }
  }

  if (CACHE && cand_path && C > 1) {
    // ---- a cluster's candidate rounds, each over the CTAs' own lists: one
    // warp merges the round's digit counts from every rank's histogram, with
    // every rank's key range and count of the candidates under the prefix;
    // every CTA reaches the same bins, and no list leaves its CTA.  Once the
    // candidates under the prefix all hold one key (exact ties, as quantised
    // scores give), no key round can split them: the ranks' counts place the
    // cut, in block order, at once.
    __syncthreads();  // this CTA's list is complete
    own_n = S.ncand;
    {
      // round 1's key range (its digits were counted as the list formed)
      uint32_t lo = 0xFFFFFFFFu, hi = 0u;
      for (uint32_t j = tid; j < own_n; j += NT) {
        lo = min(lo, cand_s[j]);
        hi = max(hi, cand_s[j]);
      }
      lo = __reduce_min_sync(0xffffffffu, lo);
      hi = __reduce_max_sync(0xffffffffu, hi);
      if (lane == 0 && lo <= hi) {
        atomicMin(&S.kmin_r[1], lo);
        atomicMax(&S.kmax_r[1], hi);
      }
      if (tid == 0) S.kcnt_r[1] = own_n;
    }
    bool done = false;
    int r_one = 0;  // the round whose check found one key
    for (int r = 1; r <= kRounds && !done; ++r) {
      uint32_t *H = r == 1 ? S.hist1 : (r == 2 ? S.hist2 : S.hist3);
      const int nb = r < kRounds ? round_bins(r) : 0, sh = r < kRounds ? round_shift(r) : 0;
      if (r > 1) {  // this CTA's candidates under the prefix: digits, key range, count
        uint32_t lo = 0xFFFFFFFFu, hi = 0u, c = 0u;
        for (uint32_t j = tid; j < own_n; j += NT) {
          const uint32_t key = cand_s[j];
          if ((key >> shift) == prefix) {
            if (nb > 0) atomicAdd(&H[(key >> sh) & (uint32_t)(nb - 1)], 1u);
            lo = min(lo, key);
            hi = max(hi, key);
            ++c;
          }
        }
        lo = __reduce_min_sync(0xffffffffu, lo);
        hi = __reduce_max_sync(0xffffffffu, hi);
        c = __reduce_add_sync(0xffffffffu, c);
        if (lane == 0 && c) {
          atomicMin(&S.kmin_r[r], lo);
          atomicMax(&S.kmax_r[r], hi);
          atomicAdd(&S.kcnt_r[r], c);
        }
      }
      cluster_sync_all();
      cluster_find_round<NT>(S, H, nb, r, C, need, rank);
      if (S.one_key || r == kRounds) {  // (after round 3 the prefix is a whole key)
        if (r < kRounds) {
          prefix = S.one_key_val;
          shift = 0;
        }
        r_one = r;
        break;
      }
      need -= S.rabove[r];
      prefix = (prefix << (shift - sh)) | (uint32_t)S.rsel[r];
      shift = sh;
      done = S.rcnt[r] == need;
    }
    int32_t cut = INT32_MAX;  // keys equal to the prefix: kept up to this block index
    if (!done) {
      // the need lowest block indices among the keys equal to `prefix` are
      // kept; ranks own ascending slices, so the lower ranks' come first
      const uint32_t before = S.tbefore, mine = S.kcnt_r[r_one];
      if (need <= before) {
        cut = -1;
      } else if (need < before + mine) {
        // this CTA keeps its m lowest: a bitmap of their local indices and a
        // scan of its words' bit counts
        const uint32_t m = need - before;
        const int words = (cnt + 31) >> 5;  // cnt <= 65536 on this path
        const int per_t = (words + NT - 1) / NT;
        uint32_t *bm = S.hist0;  // no rank reads round 0's bins any more
        for (int i = tid; i < words; i += NT) bm[i] = 0u;
        __syncthreads();
        for (uint32_t j = tid; j < own_n; j += NT) {
          if (cand_s[j] == prefix) {
            const uint32_t li = cand_li[j];
            atomicOr(&bm[li >> 5], 1u << (li & 31u));
          }
        }
        __syncthreads();
        uint32_t c = 0;
        for (int k = 0; k < per_t; ++k) {
          const int w = tid * per_t + k;
          if (w < words) c += (uint32_t)__popc(bm[w]);
        }
        uint32_t total;
        const uint32_t below = block_excl_scan<NT>(c, S.warp_tot, total);
        if (below < m && m <= below + c) {
          uint32_t acc = below;
          for (int k = 0; k < per_t; ++k) {
            const int w = tid * per_t + k;
            uint32_t word = bm[w];
            const uint32_t cw = (uint32_t)__popc(word);
            if (acc + cw >= m) {
              for (uint32_t q = m - acc; q > 1u; --q) word &= word - 1u;  // drop the lower set bits
              S.sel_bin = (int32_t)(32 * w + __ffs((int)word) - 1);
              break;
            }
            acc += cw;
          }
        }
        __syncthreads();
        cut = b0 + S.sel_bin;
      }
    }
    if (tid == 0) {
      S.rule_prefix = prefix;
      S.rule_shift = (uint32_t)shift;
      S.rule_cut = cut;
    }
    __syncthreads();
  } else if (cand_path) {
    if (C > 1) cluster_sync_all(); else __syncthreads();
    own_n = S.ncand;
    if (rank == 0 && !rule_ready) {
      // rank 0 gathers every CTA's candidates after its own, rank by rank,
      // so an entry's rank (and with it its global block index) follows
      // from where it sits in the list
      if (warp == 0) {  // every rank's count at once, then a warp prefix sum
        uint32_t c = 0;
        if (lane < C) c = lane == 0 ? S.ncand : ld_dsmem(&S.ncand, (uint32_t)lane);
        uint32_t incl = c;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const uint32_t o = __shfl_up_sync(0xffffffffu, incl, off);
          if (lane >= off) incl += o;
        }
        if (lane < C) S.roff[lane] = incl - c;
        if (lane == C - 1) S.roff[C] = incl;
      }
      __syncthreads();
      // one thread per remote entry across all ranks, loads independent
      const uint32_t own = S.roff[1], all = S.roff[C];
      for (uint32_t j = own + tid; j < all; j += NT) {
        int q = 1;
        while (q + 1 < C && S.roff[q + 1] <= j) ++q;
        const uint32_t jj = j - S.roff[q];
        cand_s[j] = ld_dsmem(&cand_s[jj], (uint32_t)q);
        cand_li[j] = ld_dsmem_u16(&cand_li[jj], (uint32_t)q);
      }
      __syncthreads();
      // Every candidate of the gathered list, strided over the CTA by whole
      // warps (lanes past the end hold valid = false): fn(valid, key, global
      // block index).
      const int32_t nl = (int32_t)S.roff[C];
      auto each = [&](auto &&fn) {
        for (int32_t j0 = warp * 32; j0 < nl; j0 += NT) {
          const int32_t j = j0 + lane;
          const bool v = j < nl;
          int q = 0;
          while (q + 1 < C && v && (int32_t)S.roff[q + 1] <= j) ++q;
          fn(v, v ? cand_s[j] : 0u, v ? (uint32_t)(q * per) + (uint32_t)cand_li[j] : 0u);
        }
      };
      // rounds 1..3 on the candidates: every thread histograms, one warp
      // finds the bin (two barriers a round)
      bool done = false;
      for (int r = 1; r < kRounds && !done; ++r) {
        uint32_t *H = r == 1 ? S.hist1 : (r == 2 ? S.hist2 : S.hist3);
        const int nb = round_bins(r), sh = round_shift(r);
        each([&](bool v, uint32_t key, uint32_t) {
          if (v && (key >> shift) == prefix) atomicAdd(&H[(key >> sh) & (uint32_t)(nb - 1)], 1u);
        });
        __syncthreads();
        if (warp == 0) {
          uint32_t B, above;
          warp_find_bin(H, nb, need, lane, B, above);
          if (lane == 0) {
            S.rsel[r] = (int32_t)B;
            S.rabove[r] = above;
          }
        }
        __syncthreads();
        const uint32_t B = (uint32_t)S.rsel[r];
        const uint32_t cB = H[B];
        need -= S.rabove[r];
        prefix = (prefix << (shift - sh)) | B;
        shift = sh;
        done = cB == need;
        if (!done && r < kRounds - 1 && cB > 64u) {
          // many keys left under the prefix: if they all hold one key (exact
          // ties, as quantised scores give) the remaining key rounds are moot
          // and the index rounds below cut the ties
          if (tid == 0) {
            S.kmin = 0xFFFFFFFFu;
            S.kmax = 0u;
          }
          __syncthreads();
          uint32_t lo = 0xFFFFFFFFu, hi = 0u;
          each([&](bool v, uint32_t key, uint32_t) {
            if (v && (key >> shift) == prefix) {
              lo = min(lo, key);
              hi = max(hi, key);
            }
          });
          lo = __reduce_min_sync(0xffffffffu, lo);
          hi = __reduce_max_sync(0xffffffffu, hi);
          if (lane == 0) {
            atomicMin(&S.kmin, lo);
            atomicMax(&S.kmax, hi);
          }
          __syncthreads();
          if (S.kmin == S.kmax) {
            prefix = S.kmin;
            shift = 0;
            break;
          }
        }
      }
      if (done) {
        if (tid == 0) {
          S.rule_prefix = prefix;
          S.rule_shift = (uint32_t)shift;
          S.rule_cut = INT32_MAX;
        }
      } else if (C == 1 && n <= 65536) {
        // ties at the full key, on one CTA: of the keys equal to `prefix`,
        // the `need` with the lowest block indices are kept.  Their indices
        // are marked in a bitmap (round 0's histogram is no longer read) and
        // a scan of its words' bit counts finds the need-th lowest.
        constexpr int kWords = 65536 / 32, kPer = kWords / NT;
        uint32_t *bm = S.hist0;
        for (int i = tid; i < kWords; i += NT) bm[i] = 0u;
        __syncthreads();
        each([&](bool v, uint32_t key, uint32_t gi) {
          if (v && key == prefix) atomicOr(&bm[gi >> 5], 1u << (gi & 31u));
        });
        __syncthreads();
        uint32_t c = 0;
#pragma unroll
        for (int k = 0; k < kPer; ++k) c += (uint32_t)__popc(bm[tid * kPer + k]);
        uint32_t total;
        const uint32_t before = block_excl_scan<NT>(c, S.warp_tot, total);
        if (before < need && need <= before + c) {
          uint32_t acc = before;
          for (int k = 0; k < kPer; ++k) {
            uint32_t w = bm[tid * kPer + k];
            const uint32_t cw = (uint32_t)__popc(w);
            if (acc + cw >= need) {
              for (uint32_t r = need - acc; r > 1u; --r) w &= w - 1u;  // drop the lower set bits
              S.rule_cut = (int32_t)(32 * (tid * kPer + k) + __ffs((int)w) - 1);
              break;
            }
            acc += cw;
          }
        }
        if (tid == 0) {
          S.rule_prefix = prefix;
          S.rule_shift = 0;
        }
      } else {
        // ties at the full key: of the keys equal to `prefix`, the `need`
        // with the lowest block indices are kept.  Radix rounds over the
        // equal candidates' block indices, 8 bits at a time from the highest
        // bit an index < n can have, find the cut index.
        const uint32_t top = (uint32_t)n - 1u;
        int ish = top ? ((32 - __clz((int)top) + 7) & ~7) : 8;  // index bits, rounded up
        uint32_t iprefix = 0;  // the cut index's bits above ish
        uint32_t *H = S.hist0;  // round 0's histogram is no longer read
        for (int ir = 0; ir < 4; ++ir) {
          const int sh = ish - 8;
          if (tid < 256) H[tid] = 0u;
          __syncthreads();
          each([&](bool v, uint32_t key, uint32_t gi) {
            if (v && key == prefix && (ish >= 32 || (gi >> ish) == iprefix))  // ascending: digit d in bin 255-d
              atomicAdd(&H[255u - ((gi >> sh) & 255u)], 1u);
          });
          __syncthreads();
          if (warp == 0) {
            uint32_t B, above;
            warp_find_bin(H, 256, need, lane, B, above);
            if (lane == 0) {
              S.sel_bin = (int32_t)B;
              S.sel_above = above;
            }
          }
          __syncthreads();
          const uint32_t cB = H[S.sel_bin];
          need -= S.sel_above;
          iprefix = (iprefix << 8) | (255u - (uint32_t)S.sel_bin);
          ish = sh;
          __syncthreads();  // sel_bin and H are rewritten next round
          if (cB == need || ish == 0) break;  // at ish == 0 a bin holds one index
        }
        if (tid == 0) {
          S.rule_prefix = prefix;
          S.rule_shift = 0;
          S.rule_cut = (int32_t)((((uint64_t)iprefix + 1u) << ish) - 1u);
        }
      }
      __syncthreads();
    }
    // every CTA takes rank 0's rule
    if (C > 1) cluster_sync_all();
    if (rank != 0 && tid == 0) {
      S.rule_prefix = ld_dsmem(&S.rule_prefix, 0u);
      S.rule_shift = ld_dsmem(&S.rule_shift, 0u);
      S.rule_cut = (int32_t)ld_dsmem(reinterpret_cast<const uint32_t *>(&S.rule_cut), 0u);
    }
    __syncthreads();
  }

  if (scan_ties) {
    // ---- fallback (round 0's bin holds more than CAND keys): rounds 1..3
    // over every key, each histogram merged over the cluster
    bool done = false;
    for (int r = 1; r < kRounds && !done; ++r) {
      uint32_t *H = r == 1 ? S.hist1 : (r == 2 ? S.hist2 : S.hist3);
      const int nb = round_bins(r), sh = round_shift(r);
      for (int32_t ib = warp * 32; ib < cnt; ib += NT) {
        const int32_t i = ib + lane;
        const bool in = i < cnt;
        uint32_t key = 0;
        if (in) key = i < cached ? keys_s[i] : order_key(__ldg(srow + i));
        hist_add(H, (key >> sh) & (uint32_t)(nb - 1), in && (key >> shift) == prefix);
      }
      if (C > 1) cluster_sync_all(); else __syncthreads();
      const uint32_t *M = H;
      if (C > 1) {
        for (int b = tid; b < nb; b += NT) {
          uint32_t v[kSelMaxCluster];
#pragma unroll
          for (int q = 0; q < kSelMaxCluster; ++q) v[q] = q < C ? ld_dsmem(&H[b], (uint32_t)q) : 0u;
          uint32_t t = 0;
#pragma unroll
          for (int q = 0; q < kSelMaxCluster; ++q) t += v[q];
          S.msmall[b] = t;
        }
        __syncthreads();
        M = S.msmall;
      }
      find_bin<NT>(M, nb, need, S.warp_tot, &S.sel_bin, &S.sel_above);
      const uint32_t B = (uint32_t)S.sel_bin;
      const uint32_t cB = M[B];
      need -= S.sel_above;
      prefix = (prefix << (shift - sh)) | B;
      shift = sh;
      done = cB == need;
      if (!done && r == kRounds - 1 && tid == 0) {
        // keys equal to the threshold in lower-ranked CTAs precede ours in block order
        uint32_t e = 0;
        for (uint32_t q = 0; q < rank; ++q) e += ld_dsmem(&S.hist3[B], q);
        S.eq_base = e;
      }
      __syncthreads();
    }
    if (done) {
      scan_ties = false;
      if (tid == 0) {
        S.rule_prefix = prefix;
        S.rule_shift = (uint32_t)shift;
        S.rule_cut = INT32_MAX;
      }
      __syncthreads();
    }
  }

  if (!bad) {
    const uintptr_t rb = reinterpret_cast<uintptr_t>(mrow);
    const bool al16 = (rb & 15u) == 0, al4 = (rb & 3u) == 0;
    const uint32_t rp = S.rule_prefix, rs = S.rule_shift;
    const int32_t rc = S.rule_cut;
    uint32_t running = S.eq_base;
    if (cand_path) {  // the mask is written but for this CTA's candidates
      for (uint32_t j = tid; j < own_n; j += NT) {
        const uint32_t kk = cand_s[j] >> rs;
        const int32_t li = (int32_t)cand_li[j];
        if (kk > rp || (kk == rp && b0 + li <= rc)) store_blocks(mrow, (int64_t)b0 + li, 1, 1u, false, al4);
      }
    }
    for (int32_t tb = 0; tb < (cand_path ? 0 : cnt); tb += 4 * NT) {
      const int32_t i = tb + 4 * tid;
      const int m = max(0, min(4, cnt - i));
      uint32_t k[4];
      if (m == 4 && i + 3 < cached) {  // one 16-byte load per thread
        const uint4 kv = *reinterpret_cast<const uint4 *>(keys_s + i);
        k[0] = kv.x;
        k[1] = kv.y;
        k[2] = kv.z;
        k[3] = kv.w;
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int32_t ie = i + e;
          k[e] = (e < m) ? ((ie < cached) ? keys_s[ie] : order_key(__ldg(srow + ie))) : 0u;
        }
      }
      uint32_t kept = 0;
      if (!scan_ties) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t kk = k[e] >> rs;
          if (e < m && (kk > rp || (kk == rp && b0 + i + e <= rc))) kept |= 1u << e;
        }
      } else {  // the threshold key itself: ties filled in block order by a scan
        uint32_t eqc = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) eqc += (e < m && k[e] == prefix) ? 1u : 0u;
        uint32_t total;
        uint32_t rk = running + block_excl_scan<NT>(eqc, S.warp_tot, total);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (e >= m) continue;
          if (k[e] > prefix) {
            kept |= 1u << e;
          } else if (k[e] == prefix) {
            if (rk < need) kept |= 1u << e;
            ++rk;
          }
        }
        running += total;
      }
      if (m > 0) store_blocks(mrow, (int64_t)b0 + i, m, kept, al16, al4);
    }
  } else if (rank == 0 && tid == 0) {
    report_error(status, kErrNonFinite, row);
  }
  // no CTA may leave while a peer can still read its shared memory
  if (C > 1) cluster_sync_all();
}

static size_t select_smem_bytes(int32_t cap, int cand = kCandCap) {
  return ((sizeof(SelectSmem) + 15) & ~size_t(15)) + 6 * (size_t)cand +
         4 * (size_t)(cap > 0 ? cap : 1);
}

// Largest cluster the select kernel can be co-scheduled with (16 needs the
// non-portable opt-in; fall back to 8, 4, 2 if the GPU refuses).  Both block
// shapes get their attributes here, once per device.
static int probe_max_cluster();

static int max_cluster_size() {
  static PerDevice cache;
  return cache.get(probe_max_cluster);
}

static int probe_max_cluster() {
  int best = 1;
  for (auto fn : {select_kernel<512, true>, select_kernel<256, false>}) {
    cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)select_smem_bytes(kSelCapMax));
  }
  for (int c = kSelMaxCluster; c >= 2; c >>= 1) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = c;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(c);
    cfg.blockDim = dim3(512);
    cfg.dynamicSmemBytes = select_smem_bytes(kSelCapMax);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, select_kernel<512, true>, &cfg) == cudaSuccess && n > 0) {
      best = c;
      break;
    }
  }
  cudaGetLastError();  // a refused query leaves no sticky error
  return best;
}

static int sm_count() { return device_sm_count(); }

// Cluster size for a launch: split a row over a cluster when its blocks
// overflow one CTA's key cache, and, for launches of a few rows, further, up
// to 8 CTAs a row, while the whole launch stays within half the GPU and every
// CTA keeps at least 4096 keys (one 16384-block row: 8.6 us on 1 CTA, 8.1 on
// 2, 7.5 on 4; one 65536-block row: 12.3 us on 4, 9.5 on 8, 10.1 on 16; 32 rows
// of 32768-65536 blocks: 11.2 us on 4 CTAs each, 12.8 on 8 -- past one wave
// the cluster barriers and remote reads cost more than the split gains).
int select_cluster_size(int64_t n_rows, int64_t tokens) {
  const int64_t n_max = tokens / kRatio;
  const int cmax = max_cluster_size();
  int C = 1;
  if (n_rows > 2 * (int64_t)sm_count()) {
    // many rows take the shape without a key cache: a row needs a cluster only
    // past 65536 blocks (16-bit local indices); 1024 rows x 65536 blocks run
    // in 206 us on one CTA each, 224 us on clusters of 4
    while (C < cmax && (n_max + C - 1) / C > 65536) C <<= 1;
    return C;
  }
  while (C < cmax && (n_max + C - 1) / C > kSelCapMax) C <<= 1;
  while (2 * C <= (cmax < 8 ? cmax : 8) && n_rows * 2 * C <= sm_count() / 2 && n_max / (2 * C) >= 4096)
    C <<= 1;
  return C;
}

cudaError_t launch_select(const float *scores, int64_t score_cols, const int32_t *pos,
                          int32_t n_rows, int32_t tokens, int32_t budget, uint8_t *mask,
                          int32_t *status, cudaStream_t stream) {
  const int32_t keep_max = budget / kRatio;
  const int64_t n_max = (int64_t)tokens / kRatio;
  const int C = select_cluster_size(n_rows, tokens);
  const int64_t per = (((n_max + C - 1) / C) + 3) & ~int64_t(3);
  const int64_t ctas = (int64_t)n_rows * C;
  // more CTAs than two waves of the wide shape: small CTAs, keys re-read from L2
  const bool narrow = ctas > 2 * (int64_t)sm_count();
  const int32_t cap = narrow ? 0 : (int32_t)(per < kSelCapMax ? per : kSelCapMax);

  if (narrow && C == 1 && n_max <= 32768)  // no row can take the sampled band
    return launch_dependent(select_kernel<256, false, kCandCapShort>, dim3((unsigned)ctas), dim3(256),
                            select_smem_bytes(0, kCandCapShort), stream, 1u, scores, score_cols, pos,
                            tokens, keep_max, mask, status, (int32_t)1, 0);
  const size_t smem = select_smem_bytes(cap);
  if (narrow)
    return launch_dependent(select_kernel<256, false>, dim3((unsigned)ctas), dim3(256), smem, stream,
                            (unsigned)C, scores, score_cols, pos, tokens, keep_max, mask, status,
                            (int32_t)C, cap);
  return launch_dependent(select_kernel<512, true>, dim3((unsigned)ctas), dim3(512), smem, stream,
                          (unsigned)C, scores, score_cols, pos, tokens, keep_max, mask, status,
                          (int32_t)C, cap);
}

}  // namespace qsa
