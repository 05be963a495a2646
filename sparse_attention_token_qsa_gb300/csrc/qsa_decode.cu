// Fused decode step: score a few query rows against every visible block key
// and select each row's top blocks into its mask, in one launch.
//
// The operation is the scorer's and the selector's, unchanged (PR #1160
// "score QSA token-indexer blocks in native CUDA": S[p, b] = sum_h relu(q_h .
// k_b) / sqrt(128) over the row's visible blocks; PR #1178 "select QSA indexer
// blocks", "Exact semantics": the keep = min(budget / 4, blocks) highest
// scores under (score descending, block index ascending), their tokens and the
// row's tail visible).  metrale layers/qsa.rs decode_select runs the two back
// to back for each decode step; at one row per step the second launch and
// the selector's single-CTA passes over the row are most of the step's time,
// so here the row's scoring CTAs also do the selection:
//
//  1. each CTA scores its contiguous range of the row's blocks (the streaming
//     core shared with the decode scorer), keeps its scores in shared memory
//     and adds their top-12-bit order-key histogram into the row's workspace
//     (exact zeros counted per warp);
//  2. the row's CTAs meet at a grid barrier (the launch is cooperative, so
//     they are co-resident; the wait is bounded);
//  3. every CTA reads the row's histogram, finds the bin holding the keep-th
//     key (a non-finite score shows up in the 16 outer bins), writes the final
//     mask bytes of its own blocks outside that bin, and appends the bin's
//     keys with their block indices to the row's candidate list;
//  4. the last CTA of the row to finish (an atomic ticket) zeroes the row's
//     workspace for the next call (its stores drain while it works on), runs
//     the remaining radix rounds (8, 8, 4 bits) over the candidates, cuts
//     exact ties at the final key by radix rounds on the block index (lowest
//     kept), and writes the kept candidates' mask bytes.
//
// Workspace per row: the 4096-bin histogram, three counters, and room for
// tokens / 4 candidates (key, block index).  It must be zero before the first
// call; every call that completes leaves it zero.  A call that reports an
// error may leave it dirty: zero it again before the next call.
#include "qsa_score_simt.cuh"
#include "qsa_select_util.cuh"

namespace qsa {

namespace {

constexpr int kDecThreads = kSimtThreads;
constexpr int kDecMaxBpc = 512;      // blocks per CTA (their scores stay in shared memory)
constexpr int kDecCandCache = 8192;  // candidates the last CTA copies into shared memory
constexpr long long kDecSpinLimit = 4000000000LL;  // ~2 s of SM clock

struct RowHdr {  // per row, at the start of the row's workspace
  uint32_t hist0[4096];
  uint32_t arrive;  // CTAs whose histogram is in
  uint32_t pad0;
  // candidates listed (low 32 bits) and CTAs done writing their blocks (high
  // 32 bits): the last CTA's ticket returns the list's length with it
  unsigned long long tc;
  uint32_t maxbin[8];  // the highest bin any key landed in (CTA y adds to slot y % 8)
  uint32_t lowbad;     // a key landed below bin 8 (a negative non-finite score)
  uint32_t pad[51];
};
static_assert(sizeof(RowHdr) == 16640, "the workspace layout is part of the ABI");

// Keys of the keep-th largest score and everything above it sit in the top few
// dozen bins of a row's histogram, so each CTA first reads only this many bins
// below the row's highest one (and the whole histogram if they fall short).
constexpr int kDecWindow = 256;

struct DecSmem {  // selection scratch, laid over the key ring once scoring is done
  uint32_t hist0[4096];
  uint32_t hist1[256];
  uint32_t hist2[256];
  uint32_t hist3[16];
  uint32_t warp_tot[kDecThreads / 32];
  int32_t sel_bin;
  uint32_t sel_above;
  int32_t flag;
  uint32_t rule_prefix;
  uint32_t rule_shift;
  int32_t rule_cut;
  uint32_t nl;         // candidates listed over the row (the last CTA)
  int32_t rsel[4];     // each candidate round's bin ...
  uint32_t rabove[4];  // ... and the keys above it
};
constexpr size_t kDecCandOff = (sizeof(DecSmem) + 127) & ~size_t(127);
static_assert(kDecCandOff + (size_t)kDecCandCache * 8 <= kSimtRingBytes, "scratch overflows the ring");
constexpr size_t kDecSmemBytes = kSimtStageOff + kSimtRingBytes + kDecMaxBpc * sizeof(float);

__device__ __forceinline__ void red_add_release_gpu(uint32_t *p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

struct PoolArgs {         // newly complete blocks to pool in the same launch
  const uint16_t *keys;  // token 4 * first's raw key
  int64_t key_stride;
  int32_t first, n;      // blocks [first, first + n); n = 0: none
  const uint16_t *k_norm_w;
  uint16_t *block_keys;  // the scorer's block-key cache, written here
};

constexpr int kDecPoolOverlap = 12;  // blocks a scoring CTA pools in its copy window (warps 2..7)

__global__ void __launch_bounds__(kDecThreads)
decode_fused_kernel(const ScoreArgs a, int32_t keep_max, uint8_t *__restrict__ mask,
                    uint8_t *__restrict__ ws, int64_t row_ws_bytes, int32_t bpc,
                    const PoolArgs pa) {
  extern __shared__ __align__(128) uint8_t dec_smem[];
  __shared__ uint32_t s_maxbin, s_low;  // this CTA's highest bin, any bin below 8
  SimtSmem &S = *reinterpret_cast<SimtSmem *>(dec_smem);
  uint8_t *ring = dec_smem + kSimtStageOff;
  float *sc_s = reinterpret_cast<float *>(ring + kSimtRingBytes);
  DecSmem &D = *reinterpret_cast<DecSmem *>(ring);
  uint32_t *ck_s = reinterpret_cast<uint32_t *>(ring + kDecCandOff);  // cached candidate keys
  uint32_t *ci_s = ck_s + kDecCandCache;                              // ... and block indices
  grid_dependency_sync();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = blockIdx.x, y = blockIdx.y, ny = gridDim.y;
  // the query row's load is issued beside the position's (both may live in
  // host memory: two round trips side by side instead of one after the other)
  const uint4 qchunk = load_query_chunk(a, row);
  if (tid == 0) {
    s_maxbin = 0u;
    s_low = 0u;
  }
  const int32_t p = a.pos[row];
  const bool valid = p >= 0 && p < a.tokens;
  const int32_t n = valid ? (p + 1) >> 2 : 0;

  // ---- 0. the newly complete blocks in this CTA's range are pooled here
  // (every row's CTAs pool them, writing identical keys, so the range is
  // covered whatever each row sees).  A CTA that scores them does it in its
  // copy window and patches its landed stage; any other CTA, or one with more
  // than kDecPoolOverlap of them, pools before it scores.
  const int pr0 = max(pa.first, y * bpc);
  const int pr1 = min(pa.first + pa.n, min(y * bpc + bpc, a.tokens >> 2));
  const int npool = max(0, pr1 - pr0);
  const int c0_ = y * bpc;
  const int cnt_ = max(0, min(n, c0_ + bpc) - c0_);
  const bool overlap = npool > 0 && cnt_ > 0 && npool <= kDecPoolOverlap;
  auto pool_one = [&](int b) {  // both half-warps of the calling warp call it
    return pool_block_16(pa.keys + (int64_t)(b - pa.first) * kRatio * pa.key_stride,
                         pa.key_stride, b, pa.k_norm_w, a.cos_t, a.sin_t, a.eps, lane & 15);
  };
  if (npool > 0 && !overlap) {
    for (int j0 = 0; j0 < npool; j0 += kDecThreads / 16) {
      const int j = j0 + (tid >> 4);
      const uint4 key = pool_one(pr0 + min(j, npool - 1));
      if (j < npool)
        *reinterpret_cast<uint4 *>(pa.block_keys + (int64_t)(pr0 + j) * kHeadDim + 8 * (lane & 15)) = key;
    }
    __syncthreads();
    // the bulk copies below read these keys through the async proxy
    if (tid == 0) asm volatile("fence.proxy.async.global;" ::: "memory");
  }
  if (!valid) {  // uniform over the row's CTAs: nobody waits for them
    if (y == 0 && tid == 0) report_error(a.status, kErrRowRange, row);
    return;
  }
  uint8_t *mrow = mask + (int64_t)row * a.tokens;
  uint8_t *wrow = ws + (int64_t)row * row_ws_bytes;
  RowHdr &W = *reinterpret_cast<RowHdr *>(wrow);
  uint32_t *cand_key = reinterpret_cast<uint32_t *>(wrow + sizeof(RowHdr));
  uint32_t *cand_idx = cand_key + (a.tokens >> 2);
  const int c0 = y * bpc;
  const int c1 = min(n, c0 + bpc);
  const int cnt = max(0, c1 - c0);

  // ---- 1. scores of this CTA's blocks
  const int pj = (warp - 2) * 2 + (lane >> 4);  // warps 2..7: pooled block pr0 + pj
  uint4 pooled = make_uint4(0u, 0u, 0u, 0u);
  auto prologue = [&]() {
    if (overlap && warp >= 2) {
      pooled = pool_one(pr0 + min(pj, npool - 1));
      if (pj < npool)
        *reinterpret_cast<uint4 *>(pa.block_keys + (int64_t)(pr0 + pj) * kHeadDim + 8 * (lane & 15)) =
            pooled;
    }
  };
  auto patch = [&](int base, uint8_t *st) {  // the stage read the keys before pooling
    if (overlap && pr0 < base + kSimtBlocksPerIter && pr1 > base) {
      const int b = pr0 + pj;
      if (warp >= 2 && pj < npool && b >= base && b < base + kSimtBlocksPerIter)
        *reinterpret_cast<uint4 *>(st + (size_t)(b - base) * (kHeadDim * 2) + 16 * (lane & 15)) =
            pooled;
      __syncthreads();
    }
  };
  if (cnt > 0 && !simt_score_blocks(a, row, p, c0, c1, S, ring,
                                    [&](int b, float sc) { sc_s[b - c0] = sc; }, prologue, patch,
                                    &qchunk)) {
    if (tid == 0) report_error(a.status, kErrTimeout, row);
    return;  // the row's other CTAs time out at the barrier below
  }
  if (n <= keep_max) {  // every block kept: this CTA's share of the visible prefix
    const int64_t span = ((int64_t)a.tokens + ny - 1) / ny;
    const int64_t lo = (int64_t)y * span;
    fill_visible(mrow, lo, min((int64_t)a.tokens, lo + span), p);
    return;
  }
  __syncthreads();  // sc_s complete; the ring is free
  // one add per distinct bin per warp: a row's keys crowd into a few hundred
  // bins, and every CTA of the row adds into the same workspace counters
  uint32_t my_max = 0u, my_low = 0u;
  for (int i0 = warp * 32; i0 < cnt; i0 += kDecThreads) {
    const int i = i0 + lane;
    const uint32_t bin = i < cnt ? order_key(sc_s[i]) >> 20 : 0xFFFFFFFFu;
    const uint32_t peers = __match_any_sync(0xffffffffu, bin);
    if (bin != 0xFFFFFFFFu) {
      if (lane == __ffs(peers) - 1) atomicAdd(&W.hist0[bin], (uint32_t)__popc(peers));
      my_max = max(my_max, bin);
      my_low |= bin < 8u ? 1u : 0u;
    }
  }
  my_max = __reduce_max_sync(0xffffffffu, my_max);
  my_low = __reduce_or_sync(0xffffffffu, my_low);
  if (lane == 0) {
    atomicMax(&s_maxbin, my_max);
    if (my_low) s_low = 1u;
  }

  // ---- 2. grid barrier over the row's CTAs
  __syncthreads();
  if (tid == 0) {
    asm volatile("red.relaxed.gpu.global.max.u32 [%0], %1;" ::"l"(&W.maxbin[y & 7]), "r"(s_maxbin)
                 : "memory");
    if (s_low) asm volatile("red.relaxed.gpu.global.or.b32 [%0], 1;" ::"l"(&W.lowbad) : "memory");
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
  // A non-finite score lands above bin 0xFF7 (positive) or below bin 8
  // (negative); every finite one between.  The row's histogram comes into
  // shared memory by bulk copies (the copy engine reads global memory through
  // the async proxy, so that proxy is fenced after the acquire that made the
  // other CTAs' adds visible): first the kDecWindow bins ending at the row's
  // highest one, then, only if they hold fewer than keep keys, all 4096.
  if (tid == 0) {
    uint32_t mx = 0u;
#pragma unroll
    for (int k = 0; k < 8; ++k) mx = max(mx, __ldcg(&W.maxbin[k]));
    const bool nf = __ldcg(&W.lowbad) != 0u || mx >= 0xFF8u;
    D.rule_prefix = nf ? 1u : 0u;  // (scratch: the non-finite verdict)
    // window start: 16-byte aligned, rounded up so the highest bin stays inside
    // (mx <= 0xFF7 for a finite row, so the window ends inside the histogram)
    D.rule_shift = ((uint32_t)max(0, (int)mx + 1 - kDecWindow) + 3u) & ~3u;
  }
  __syncthreads();
  const bool bad = D.rule_prefix != 0u;
  const uint32_t wlo = D.rule_shift;
  auto fetch_hist = [&](uint32_t first, uint32_t nbins, uint32_t parity) {
    if (tid == 0) {
      const uint32_t mb = simt_smem_u32(&S.full[0]);  // the ring's barriers are free again
      if (parity == 0u) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(mb) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      }
      asm volatile("fence.proxy.async.global;" ::: "memory");
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mb), "r"(4u * nbins)
                   : "memory");
      asm volatile(
          "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
              "r"(simt_smem_u32(D.hist0)),
          "l"(W.hist0 + first), "r"(4u * nbins), "r"(mb)
          : "memory");
      D.flag = simt_wait(mb, parity) ? 1 : 0;
      D.sel_bin = -1;
    }
    __syncthreads();
    return D.flag != 0;
  };
  uint32_t need = (uint32_t)min(keep_max, n);
  uint32_t hbase = wlo;  // D.hist0[i] holds bin hbase + i
  if (!bad) {
    if (!fetch_hist(wlo, kDecWindow, 0u)) {
      if (tid == 0) report_error(a.status, kErrTimeout, row);
      return;
    }
    find_bin<kDecThreads>(D.hist0, kDecWindow, need, D.warp_tot, &D.sel_bin, &D.sel_above);
    if (D.sel_bin < 0) {  // the keep-th key lies below the window
      __syncthreads();    // every thread has read sel_bin
      hbase = 0u;
      if (!fetch_hist(0u, 4096u, 1u)) {
        if (tid == 0) report_error(a.status, kErrTimeout, row);
        return;
      }
      find_bin<kDecThreads>(D.hist0, 4096, need, D.warp_tot, &D.sel_bin, &D.sel_above);
    }
  }
  uint32_t B0 = 0;
  bool whole = false;  // the bin's keys are all kept
  if (bad) {
    if (y == 0 && tid == 0) report_error(a.status, kErrNonFinite, row);
  } else {
    B0 = hbase + (uint32_t)D.sel_bin;
    need -= D.sel_above;
    whole = D.hist0[B0 - hbase] == need;
    const uintptr_t rb = reinterpret_cast<uintptr_t>(mrow);
    const bool al16 = (rb & 15u) == 0, al4 = (rb & 3u) == 0;
    for (int i = 4 * tid; i < cnt; i += 4 * kDecThreads) {
      const int mq = min(4, cnt - i);
      uint32_t kept = 0, bits = 0, k[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        k[e] = e < mq ? order_key(sc_s[i + e]) : 0u;
        const uint32_t d = k[e] >> 20;
        if (e < mq) {
          kept |= (d > B0 || (whole && d == B0) ? 1u : 0u) << e;
          bits |= (!whole && d == B0 ? 1u : 0u) << e;
        }
      }
      store_blocks(mrow, (int64_t)c0 + i, mq, kept, al16, al4);
      if (bits) {
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
    // tokens past the complete blocks: the tail is visible, the rest zero
    if (y == ny - 1) fill_visible(mrow, 4 * (int64_t)n, a.tokens, p);
  }

  // ---- 4. the last CTA of the row resolves the candidates
  __syncthreads();
  if (tid == 0) {
    // release this CTA's mask bytes and candidates; the last CTA acquires all
    unsigned long long t;
    asm volatile("atom.acq_rel.gpu.global.add.u64 %0, [%1], %2;"
                 : "=l"(t)
                 : "l"(&W.tc), "l"(1ull << 32)
                 : "memory");
    D.flag = (uint32_t)(t >> 32) == (uint32_t)(ny - 1);
    D.nl = (uint32_t)t;  // every CTA's candidates are listed by now
  }
  __syncthreads();
  if (!D.flag) return;
  // every CTA has read the histogram and taken its ticket: clear it for the
  // next call now, so that the stores drain while the candidates are resolved
  for (int i = tid; i < 4096 / 4; i += kDecThreads)
    reinterpret_cast<uint4 *>(W.hist0)[i] = make_uint4(0u, 0u, 0u, 0u);
  auto clear_counters = [&]() {
    if (tid == 0) {
      W.arrive = 0u;
      W.tc = 0ull;
#pragma unroll
      for (int k = 0; k < 8; ++k) W.maxbin[k] = 0u;
      W.lowbad = 0u;
    }
  };
  if (bad || whole) clear_counters();
  if (!bad && !whole) {
    const int32_t nl = (int32_t)D.nl;
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
    for (int i = tid; i < 256 + 256 + 16; i += kDecThreads) (&D.hist1[0])[i] = 0u;
    __syncthreads();
    clear_counters();
    auto ckey = [&](int32_t j) { return j < kDecCandCache ? ck_s[j] : __ldcg(&cand_key[j]); };
    auto cidx = [&](int32_t j) { return j < kDecCandCache ? ci_s[j] : __ldcg(&cand_idx[j]); };
    uint32_t prefix = B0;
    int shift = 20;
    bool done = false;
    // rounds of 8, 8 and 4 bits on the candidates (each round's result in its
    // own slot: two barriers a round)
    for (int r = 1; r < 4 && !done; ++r) {
      uint32_t *H = r == 1 ? D.hist1 : (r == 2 ? D.hist2 : D.hist3);
      const int nb = r == 3 ? 16 : 256, sh = r == 1 ? 12 : (r == 2 ? 4 : 0);
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
    // the kept candidates' mask bytes (every candidate was written as dropped)
    const uint32_t rp = D.rule_prefix, rs = D.rule_shift;
    const int32_t rc = D.rule_cut;
    const bool al4 = (reinterpret_cast<uintptr_t>(mrow) & 3u) == 0;
    for (int32_t j = tid; j < nl; j += kDecThreads) {
      const uint32_t kk = ckey(j) >> rs;
      const int32_t gi = (int32_t)cidx(j);
      if (kk > rp || (kk == rp && gi <= rc)) store_blocks(mrow, gi, 1, 1u, false, al4);
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
  if (n_max == 0 || cap <= 0) return cudaSuccess;
  // the fewest blocks per CTA (128 .. 512) that keep every CTA co-resident
  int32_t bpc = 0;
  for (int32_t k = kSimtBlocksPerIter; k <= kDecMaxBpc; k += kSimtBlocksPerIter) {
    if ((int64_t)a.n_rows * ((n_max + k - 1) / k) <= cap && (n_max + k - 1) / k <= 65535) {
      bpc = k;
      break;
    }
  }
  if (bpc == 0) return cudaSuccess;  // too many rows: the caller takes the two-kernel path
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
      cudaLaunchKernelEx(&cfg, decode_fused_kernel, a, budget / kRatio, mask,
                         static_cast<uint8_t *>(ws), decode_row_ws_bytes(a.tokens), bpc, pa);
  if (e == cudaSuccess) *launched = true;
  return e;
}

}  // namespace qsa
