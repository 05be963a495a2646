// Bandwidth-bound block scorer (decode shape, and any row set).
//
// PR #1160 "score QSA token-indexer blocks in native CUDA", description: each
// query row's four heads are normed with (1 + q_norm_w) and rotated at the
// row's own position, then score(p, b) = sum_h relu(q_h . k_b) / sqrt(128), with
// relu applied per head before the head sum and written as a comparison so a
// NaN key keeps its NaN.  Only b < visible_len / 4 is written.
// metrale layers/qsa.rs decode_select (qsa_qprep then qsa_score over the
// complete blocks) is the decode use: one row streams every block key once.
//
// The kernel splits each row's visible blocks into contiguous ranges, one per
// CTA, and streams them through the shared core (bulk copies into a shared
// memory ring, 8-lane dot products, relu and head sum).  HBM traffic: 256 B of
// key read + 4 B of score written per (row, block).  On a timed-out wait the
// CTA records QSA_ERR_TIMEOUT once its own copies have landed.
#include "qsa_score_simt.cuh"

namespace qsa {

constexpr size_t kSimtSmemBytes = kSimtStageOff + kSimtRingBytes;

__global__ void __launch_bounds__(kSimtThreads)
score_simt_kernel(const ScoreArgs a, int32_t blocks_per_cta) {
  extern __shared__ __align__(128) uint8_t simt_smem_raw[];
  SimtSmem &S = *reinterpret_cast<SimtSmem *>(simt_smem_raw);
  uint8_t *stages = simt_smem_raw + kSimtStageOff;
  grid_dependency_sync();
  const int row = blockIdx.x;
  const int p = a.pos[row];
  const int vis = a.visible_len ? a.visible_len[row] : p + 1;
  if (p < 0 || p >= a.tokens || vis < 0 || vis > p + 1) {
    if (blockIdx.y == 0 && threadIdx.x == 0) report_error(a.status, kErrRowRange, row);
    return;
  }
  const int n = vis >> 2;
  const int c0 = blockIdx.y * blocks_per_cta;
  if (c0 >= n) return;
  const int c1 = min(n, c0 + blocks_per_cta);
  if (!simt_score_blocks(a, row, p, c0, c1, S, stages, [](int, float) {}) && threadIdx.x == 0)
    report_error(a.status, kErrTimeout, row);
}

cudaError_t launch_score_simt(const ScoreArgs &a, cudaStream_t stream) {
  const int64_t n_max = (int64_t)a.tokens / kRatio;
  if (n_max == 0) return cudaSuccess;
  static PerDevice smem_attr;
  const cudaError_t e = set_smem_once(smem_attr, score_simt_kernel, kSimtSmemBytes);
  if (e != cudaSuccess) return e;
  const int64_t iters = (n_max + kSimtBlocksPerIter - 1) / kSimtBlocksPerIter;
  // enough CTAs to cover ~8 per SM, each streaming at least 128 blocks
  int64_t k = ((int64_t)a.n_rows * iters) / (8 * (int64_t)device_sm_count());
  k = k < 1 ? 1 : (k > 16 ? 16 : k);
  while ((iters + k - 1) / k > 65535) ++k;
  const int32_t bpc = (int32_t)(k * kSimtBlocksPerIter);
  dim3 grid((unsigned)a.n_rows, (unsigned)((n_max + bpc - 1) / bpc));
  return launch_dependent(score_simt_kernel, grid, dim3(kSimtThreads), kSimtSmemBytes, stream, 1u,
                          a, bpc);
}

}  // namespace qsa
