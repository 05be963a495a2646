// Streaming block scorer core, shared by the decode scorer kernel and the
// fused decode kernel.
//
// PR #1160 "score QSA token-indexer blocks in native CUDA", description: each
// query row's four heads are normed with (1 + q_norm_w) and rotated at the
// row's own position, then score(p, b) = sum_h relu(q_h . k_b) / sqrt(128), with
// relu applied per head before the head sum and written as a comparison so a
// NaN key keeps its NaN.
//
// A CTA of kSimtThreads owns a contiguous range [c0, c1) of one row's blocks,
// whose keys are contiguous in memory.  One thread streams them into shared
// memory with the bulk-copy engine (cp.async.bulk, 1-D TMA), 128 keys
// (32 KiB) per stage in a ring of three, each stage completing an mbarrier;
// the first copies are in flight while the CTA prepares the row's four heads.
// 8-lane groups reduce keys from shared memory: lane g of a group owns dims
// {8(8j+g)+e : j<2, e<8}, so a quarter-warp's 16-byte loads cover one 128-byte
// run of a key (no bank conflicts).  The 4 head partial dots are
// reduce-scattered over the 8 lanes (4 shuffles) and gathered to lane 0
// (3 shuffles), which applies relu, sums heads in order 0..3 and scales.
// Every wait is bounded.
#pragma once

#include "qsa_device.cuh"
#include "qsa_launch.h"

namespace qsa {

constexpr int kSimtThreads = 256;
constexpr int kSimtGroups = kSimtThreads / 8;  // 32 groups of 8 lanes
constexpr int kSimtUnroll = 4;
constexpr int kSimtBlocksPerIter = kSimtGroups * kSimtUnroll;  // 128 keys: one stage
constexpr int kSimtStages = 3;
constexpr uint32_t kSimtStageBytes = kSimtBlocksPerIter * kHeadDim * 2;  // 32 KiB
constexpr long long kSimtSpinLimit = 4000000000LL;                      // ~2 s of SM clock

// The limit of a wait the caller may shorten (ScoreArgs::wait_limit).
__device__ __forceinline__ long long caller_wait_limit(const ScoreArgs &a) {
  return a.wait_limit > 0 ? a.wait_limit : kSimtSpinLimit;
}

struct SimtSmem {
  float q_s[kHeads][kHeadDim];
  uint64_t full[kSimtStages];
};
constexpr size_t kSimtStageOff = (sizeof(SimtSmem) + 127) & ~size_t(127);
constexpr size_t kSimtRingBytes = kSimtStages * (size_t)kSimtStageBytes;

__device__ __forceinline__ uint32_t simt_smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// Bounded wait on an mbarrier phase: a non-blocking test, then the limit,
// then a test that may sleep in hardware until the phase completes.  Returns
// false once `limit` cycles have passed (a phase still open at the first test
// with a limit of a few cycles gives up at once).
__device__ __forceinline__ bool simt_wait(uint32_t mbar, uint32_t parity,
                                          long long limit = kSimtSpinLimit) {
  const long long t0 = clock64();
  while (true) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(mbar), "r"(parity)
        : "memory");
    if (ok) return true;
    if (clock64() - t0 > limit) return false;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(mbar), "r"(parity), "r"(20000u)
        : "memory");
    if (ok) return true;
  }
}

// This thread's 16 bytes of the row's query heads (warps 0 and 1: 4 half-warps
// = 4 heads); they do not depend on the row's position, so a caller may load
// them before it reads the position.
__device__ __forceinline__ uint4 load_query_chunk(const ScoreArgs &a, int row) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp >= 2) return make_uint4(0u, 0u, 0u, 0u);
  const int h = warp * 2 + (lane >> 4);
  return ldg_nc_v4(a.q + (int64_t)row * a.q_stride + h * kHeadDim + 8 * (lane & 15));
}

__device__ __forceinline__ void prep_query_heads(const ScoreArgs &a, int row, int p,
                                                 float (*q_s)[kHeadDim], const uint4 *preloaded) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp < 2) {  // 4 half-warps = 4 heads
    const int h = warp * 2 + (lane >> 4);
    const int g = lane & 15;
    const uint4 v = preloaded ? *preloaded
                              : ldg_nc_v4(a.q + (int64_t)row * a.q_stride + h * kHeadDim + 8 * g);
    const uint4 w8 = ldg_nc_v4(a.q_norm_w + 8 * g);
    uint4 c8 = make_uint4(0, 0, 0, 0), s8 = make_uint4(0, 0, 0, 0);
    if (g < 8) {
      c8 = ldg_nc_v4(a.cos_t + (int64_t)p * kRot + 8 * g);
      s8 = ldg_nc_v4(a.sin_t + (int64_t)p * kRot + 8 * g);
    }
    float x[8];
    unpack8(v, x);
    const uint4 o = norm_rope_16(x, w8, c8, s8, a.eps, g);
    float y[8];
    unpack8(o, y);
#pragma unroll
    for (int e = 0; e < 8; ++e) q_s[h][8 * g + e] = y[e];
  }
}

// Hooks that do nothing (the plain scorer's).
struct SimtNoHook {
  __device__ void operator()() const {}
  __device__ void operator()(int, uint8_t *) const {}
};

// Score blocks [c0, c1) of `row` (c0 < c1), writing scores[row, b] and calling
// emit(b, score) from the one lane that holds each score.  All kSimtThreads
// threads call it.  Two hooks let a caller work in the copy window: prologue()
// runs on every thread once the first copies are in flight (warps 0 and 1 are
// busy with the query heads meanwhile), and patch(base, stage) runs on every
// thread when the stage of keys [base, base + 128) has landed, before it is
// read (a patch that writes the stage ends with a CTA barrier).  Returns false
// if a wait timed out (the CTA's own copies have then landed, and the caller
// reports the error).
template <typename Emit, typename Prologue = SimtNoHook, typename Patch = SimtNoHook>
__device__ __forceinline__ bool simt_score_blocks(const ScoreArgs &a, int row, int p, int c0, int c1,
                                                  SimtSmem &S, uint8_t *stages, Emit emit,
                                                  Prologue prologue = SimtNoHook(),
                                                  Patch patch = SimtNoHook(),
                                                  const uint4 *preloaded_q = nullptr) {
  const int n_it = (c1 - c0 + kSimtBlocksPerIter - 1) / kSimtBlocksPerIter;
  const uint16_t *kb = a.block_keys + (a.key_base ? a.key_base[row] : 0) * kHeadDim;
  const int tid = threadIdx.x;

  // stage `it` of the range: keys [c0 + 128 it, ...) into ring slot it % 3
  auto issue = [&](int it) {
    const int base = c0 + it * kSimtBlocksPerIter;
    const uint32_t bytes = (uint32_t)min(kSimtBlocksPerIter, c1 - base) * (kHeadDim * 2);
    const uint32_t mb = simt_smem_u32(&S.full[it % kSimtStages]);
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mb), "r"(bytes)
                 : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(simt_smem_u32(stages + (size_t)(it % kSimtStages) * kSimtStageBytes)),
        "l"(kb + (int64_t)base * kHeadDim), "r"(bytes), "r"(mb)
        : "memory");
  };
  if (tid == 0) {
    for (int s = 0; s < kSimtStages; ++s)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(simt_smem_u32(&S.full[s]))
                   : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    for (int it = 0; it < min(kSimtStages, n_it); ++it) issue(it);
  }
  // the first stages are in flight while the query heads are prepared
  prep_query_heads(a, row, p, S.q_s, preloaded_q);
  prologue();
  __syncthreads();

  const int gi = tid >> 3;
  const int g = tid & 7;
  // the lane's 16 query dims per head as (even, odd) pairs for packed FMAs
  float2 qr[kHeads][2][4];
#pragma unroll
  for (int h = 0; h < kHeads; ++h)
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int i = 0; i < 4; ++i)
        qr[h][j][i] = make_float2(S.q_s[h][8 * (8 * j + g) + 2 * i], S.q_s[h][8 * (8 * j + g) + 2 * i + 1]);

  float *srow = a.scores + (int64_t)row * a.score_cols;
  const float inv_sqrt_hd = 0.08838834764831845f;  // 1/sqrt(128)

  int it = 0;
  bool failed = false;
  for (; it < n_it; ++it) {
    const int s = it % kSimtStages;
    const bool ok = simt_wait(simt_smem_u32(&S.full[s]), (uint32_t)(it / kSimtStages) & 1u,
                              caller_wait_limit(a));
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
    const int base = c0 + it * kSimtBlocksPerIter;
    uint8_t *st = stages + (size_t)s * kSimtStageBytes;
    patch(base, st);
    uint4 kv[kSimtUnroll][2];
#pragma unroll
    for (int u = 0; u < kSimtUnroll; ++u) {
      const int lb = u * kSimtGroups + gi;  // key within the stage
      const uint8_t *kp = st + (size_t)(base + lb < c1 ? lb : 0) * (kHeadDim * 2) + 16 * g;
      kv[u][0] = *reinterpret_cast<const uint4 *>(kp);
      kv[u][1] = *reinterpret_cast<const uint4 *>(kp + 128);
    }
#pragma unroll
    for (int u = 0; u < kSimtUnroll; ++u) {
      // per head, the even and the odd dims summed apart by one packed FMA
      // per dim pair (the two bf16 of a key word unpacked side by side), then
      // added
      float2 acc2[kHeads];
#pragma unroll
      for (int h = 0; h < kHeads; ++h) acc2[h] = make_float2(0.f, 0.f);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint32_t w[4] = {kv[u][j].x, kv[u][j].y, kv[u][j].z, kv[u][j].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 kk = make_float2(lo_bf16(w[i]), hi_bf16(w[i]));
#pragma unroll
          for (int h = 0; h < kHeads; ++h) acc2[h] = __ffma2_rn(qr[h][j][i], kk, acc2[h]);
        }
      }
      float acc[kHeads];
#pragma unroll
      for (int h = 0; h < kHeads; ++h) acc[h] = acc2[h].x + acc2[h].y;
      // reduce-scatter the 4 head sums over the 8 lanes of the group
      const bool up4 = g & 4;
      float keep0 = up4 ? acc[2] : acc[0];
      float keep1 = up4 ? acc[3] : acc[1];
      const float send0 = up4 ? acc[0] : acc[2];
      const float send1 = up4 ? acc[1] : acc[3];
      keep0 += __shfl_xor_sync(0xffffffffu, send0, 4);
      keep1 += __shfl_xor_sync(0xffffffffu, send1, 4);
      const bool up2 = g & 2;
      float d = up2 ? keep1 : keep0;
      d += __shfl_xor_sync(0xffffffffu, up2 ? keep0 : keep1, 2);
      d += __shfl_xor_sync(0xffffffffu, d, 1);
      // lanes 0,2,4,6 of the group now hold heads 0,1,2,3
      const float r = (d < 0.f) ? 0.f : d;  // relu as a comparison: NaN stays NaN
      const float r1 = __shfl_down_sync(0xffffffffu, r, 2);
      const float r2 = __shfl_down_sync(0xffffffffu, r, 4);
      const float r3 = __shfl_down_sync(0xffffffffu, r, 6);
      const int b = base + u * kSimtGroups + gi;
      if (g == 0 && b < c1) {
        const float sc = __fmul_rn(__fadd_rn(__fadd_rn(__fadd_rn(r, r1), r2), r3), inv_sqrt_hd);
        srow[b] = sc;
        emit(b, sc);
      }
    }
    __syncthreads();  // every warp is done with slot s
    if (tid == 0 && it + kSimtStages < n_it) issue(it + kSimtStages);
  }
  if (failed && tid == 0) {
    // let this CTA's own copies land before its shared memory is reused (at
    // the fixed limit: a copy in flight lands within microseconds)
    for (int k = it; k < min(n_it, it + kSimtStages); ++k)
      simt_wait(simt_smem_u32(&S.full[k % kSimtStages]), (uint32_t)(k / kSimtStages) & 1u);
  }
  return !failed;
}

}  // namespace qsa
