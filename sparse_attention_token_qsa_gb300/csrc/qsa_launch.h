// Internal launchers of the QSA kernels (host side, one per kernel family).
// Arguments are validated by the C ABI layer before these are called.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "qsa_per_device.h"

namespace qsa {

// Launch `kernel` so that it may begin while the previous kernel in `stream`
// finishes (programmatic stream serialization).  The kernel must call
// grid_dependency_sync() before it touches global memory; an optional cluster
// shape is passed through.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, unsigned cluster_x, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  if (cluster_x > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = cluster_x;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

cudaError_t launch_pool_blocks(const uint16_t *keys, int64_t key_stride, int32_t first_block,
                               int32_t n_blocks, const uint16_t *k_norm_w, const uint16_t *cos_t,
                               const uint16_t *sin_t, float eps, uint16_t *block_keys,
                               cudaStream_t stream);

// Newly complete blocks that a scoring launch pools itself, before any of
// their keys are read (the cos/sin tables and eps are the scorer's).
struct PoolArgs {
  const uint16_t *keys;  // token 4 * first's raw key
  int64_t key_stride;
  int32_t first, n;      // blocks [first, first + n); n = 0: none
  const uint16_t *k_norm_w;
  uint16_t *block_keys;  // the scorer's block-key cache, written here
};

struct ScoreArgs {
  const uint16_t *q;
  int64_t q_stride;
  const int32_t *pos;
  const int32_t *visible_len;
  int32_t n_rows;
  int32_t tokens;
  const uint16_t *q_norm_w;
  const uint16_t *cos_t;
  const uint16_t *sin_t;
  float eps;
  const uint16_t *block_keys;
  const int64_t *key_base;
  float *scores;
  int64_t score_cols;
  int32_t *status;
  // limit of the waits a caller may shorten (the streaming scorers' waits
  // for their key copies, query operand and accumulators, the fused decode
  // step's waits and grid barrier), in SM clock cycles; <= 0 means the default
  long long wait_limit;
};

// The limit qsa_set_wait_limit_cycles set (process-wide), read at each launch.
long long wait_limit_cycles();

cudaError_t launch_score_simt(const ScoreArgs &a, cudaStream_t stream);
// Streaming tensor-core scorer: the SIMT scorer's rows and ranges, each
// 128-block tile scored by tcgen05 MMAs from TMA-fetched keys.
cudaError_t launch_score_stream(const ScoreArgs &a, cudaStream_t stream);
// Prepared query heads, [n_rows * 4, 128] bf16, into a workspace; the same
// launch pools `pool`'s blocks when it is given (its own CTAs).
cudaError_t launch_qprep(const ScoreArgs &a, uint16_t *qws, cudaStream_t stream,
                         const PoolArgs *pool = nullptr);
// Tensor-core scorer; qws is a workspace of n_rows * 1024 bytes (16-byte
// aligned).  `pool`'s blocks are pooled by the query-prep launch in front of it.
cudaError_t launch_score_tc(const ScoreArgs &a, uint16_t *qws, cudaStream_t stream,
                            const PoolArgs *pool = nullptr);
extern const bool kTcScorerReady;

// Fused decode step (pool the given new blocks, score, select: one
// cooperative launch; pool_n = 0 pools nothing, and the blocks must lie below
// tokens / 4).  Sets *launched; returns cudaSuccess with *launched false when
// the rows' CTAs cannot all be co-resident (the caller then launches the pool,
// score and select kernels itself).
int64_t decode_row_ws_bytes(int32_t tokens);
cudaError_t launch_decode_fused(const ScoreArgs &a, int32_t budget, uint8_t *mask, void *ws,
                                const uint16_t *pool_keys, int64_t pool_key_stride,
                                int32_t pool_first, int32_t pool_n, const uint16_t *k_norm_w,
                                uint16_t *block_keys, cudaStream_t stream, bool *launched);

// Selected token lists of mask rows, and the gather of their K/V rows.
cudaError_t launch_mask_tokens(const uint8_t *mask, int32_t n_rows, int32_t tokens, int32_t *sel,
                               int64_t sel_cols, int32_t *n_sel, cudaStream_t stream);
cudaError_t launch_gather_kv(const uint16_t *k_pool, const uint16_t *v_pool, int32_t width,
                             int32_t pool_pages, const int32_t *table, int32_t table_len,
                             int64_t table_cols,
                             int32_t page_size, const int32_t *sel, int64_t sel_cols,
                             const int32_t *n_sel, int32_t n_rows, int32_t max_sel,
                             uint16_t *k_out, uint16_t *v_out, int64_t out_rows, int32_t *status,
                             cudaStream_t stream);

cudaError_t launch_select(const float *scores, int64_t score_cols, const int32_t *pos,
                          int32_t n_rows, int32_t tokens, int32_t budget, uint8_t *mask,
                          int32_t *status, cudaStream_t stream);

// Sparse attention of each row over its selected tokens (qsa_attn.cu);
// head_dim is 128 or 256, nq a multiple of nkv.
cudaError_t launch_sparse_attn(const uint16_t *q, int64_t q_stride, int32_t nq, int32_t nkv,
                               int32_t head_dim, const uint16_t *k_pool, const uint16_t *v_pool,
                               int32_t pool_pages, int32_t page_size, const int32_t *table,
                               int32_t table_len, int64_t table_cols, const int32_t *sel,
                               int64_t sel_cols, const int32_t *n_sel, int32_t n_rows,
                               int32_t max_sel, float scale, uint16_t *out, int64_t out_stride,
                               int32_t *status, cudaStream_t stream);

// The indexer's qk projection y = x W^T on tcgen05 (qsa_proj.cu).
cudaError_t launch_proj(const uint16_t *x, int64_t x_stride, const uint16_t *w, int32_t n_rows,
                        int32_t hidden, int32_t out_cols, uint16_t *y, int64_t y_stride,
                        int32_t *status, cudaStream_t stream);

}  // namespace qsa
