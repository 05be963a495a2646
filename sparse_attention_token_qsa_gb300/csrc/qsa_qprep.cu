// Query preparation into a workspace: every (row, head) vector normed with
// (1 + q_norm_w) and rotated at the row's own position, once per launch.
//
// PR #1160 "score QSA token-indexer blocks in native CUDA", description: each
// query row's four heads are normed and rotated like a pooled key before the
// relu-head-sum score; metrale layers/qsa.rs (qsa_qprep) and atlas
// layers/qsa_select.rs (qsa_qprep_rows) likewise prepare the query rows of a
// slab before scoring them.  The prepared heads go to workspace rows
// 4 * row + head (bf16, 128 values, 256 bytes each): exactly the [rows * 4,
// 128] K-major operand the tensor-core scorer fetches with TMA.  Rows with an
// invalid position or visible length get zero vectors (the scorer writes
// nothing for them and reports the error itself).
//
// The same launch may also pool the blocks completed since the last call
// (metrale layers/qsa.rs pool_new_blocks, run just before scoring): CTAs past
// the query vectors' do it, half a warp per block as in the pool kernel, so a
// prefill chunk's pooling costs no launch of its own; the scorer waits for
// this whole launch before it reads a key.
#include "qsa_device.cuh"
#include "qsa_launch.h"

namespace qsa {

constexpr int kPrepThreads = 256;                 // 16 vectors per CTA
constexpr int kPrepVecsPerCta = kPrepThreads / 16;

__global__ void __launch_bounds__(kPrepThreads)
qprep_kernel(const ScoreArgs a, uint16_t *__restrict__ qws, const PoolArgs pa, int32_t prep_ctas) {
  grid_dependency_sync();
  const int lane = threadIdx.x & 31;
  const int g = lane & 15;
  if ((int)blockIdx.x >= prep_ctas) {
    // pooling CTAs: an idle half-warp works on a clamped block and drops its
    // store (both half-warps reach the shuffles in norm_rope_16)
    const int64_t i = (int64_t)(blockIdx.x - prep_ctas) * kPrepVecsPerCta + (threadIdx.x >> 4);
    const bool active = i < pa.n;
    const int64_t ii = active ? i : (int64_t)pa.n - 1;
    const int64_t b = (int64_t)pa.first + ii;
    const uint4 out = pool_block_16(pa.keys + (int64_t)kRatio * ii * pa.key_stride, pa.key_stride,
                                    b, pa.k_norm_w, a.cos_t, a.sin_t, a.eps, g);
    if (active) *reinterpret_cast<uint4 *>(pa.block_keys + b * kHeadDim + 8 * g) = out;
    return;
  }
  const int64_t nvec = (int64_t)a.n_rows * kHeads;
  const int64_t v = (int64_t)blockIdx.x * kPrepVecsPerCta + (threadIdx.x >> 4);
  // both half-warps reach the shuffles inside norm_rope_16; an idle one works
  // on a clamped vector and drops its store
  const int64_t vc = v < nvec ? v : nvec - 1;
  const int64_t row = vc >> 2;
  const int h = (int)(vc & 3);
  const int32_t p = a.pos[row];
  const int32_t vis = a.visible_len ? a.visible_len[row] : p + 1;
  const bool ok = !(p < 0 || p >= a.tokens || vis < 0 || vis > p + 1);
  const int32_t pc = ok ? p : 0;
  uint4 x4 = make_uint4(0, 0, 0, 0);
  if (ok) x4 = ldg_nc_v4(a.q + row * a.q_stride + h * kHeadDim + 8 * g);
  const uint4 w8 = ldg_nc_v4(a.q_norm_w + 8 * g);
  uint4 c8 = make_uint4(0, 0, 0, 0), s8 = make_uint4(0, 0, 0, 0);
  if (g < 8) {
    c8 = ldg_nc_v4(a.cos_t + (int64_t)pc * kRot + 8 * g);
    s8 = ldg_nc_v4(a.sin_t + (int64_t)pc * kRot + 8 * g);
  }
  float x[8];
  unpack8(x4, x);
  uint4 o = norm_rope_16(x, w8, c8, s8, a.eps, g);
  if (!ok) o = make_uint4(0, 0, 0, 0);
  if (v < nvec) *reinterpret_cast<uint4 *>(qws + v * kHeadDim + 8 * g) = o;
}

cudaError_t launch_qprep(const ScoreArgs &a, uint16_t *qws, cudaStream_t stream,
                         const PoolArgs *pool) {
  const int64_t nvec = (int64_t)a.n_rows * kHeads;
  const int64_t prep = (nvec + kPrepVecsPerCta - 1) / kPrepVecsPerCta;
  const PoolArgs pa = pool ? *pool : PoolArgs{nullptr, 0, 0, 0, nullptr, nullptr};
  const int64_t grid = prep + ((int64_t)pa.n + kPrepVecsPerCta - 1) / kPrepVecsPerCta;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  return launch_dependent(qprep_kernel, dim3((unsigned)grid), dim3(kPrepThreads), 0, stream, 1u, a,
                          qws, pa, (int32_t)prep);
}

}  // namespace qsa
