// C ABI of libqsa.so: host-side validation, launch configuration and the
// RoPE table builder.  Every refusal happens here, before any launch; the
// kernels only see arguments that passed these checks.
//
// Interface conventions follow PR #1178 "select QSA indexer blocks" (explicit
// score_cols with spare capacity; budget a positive multiple of 4 keeping at
// most 512 blocks; empty launch is a no-op at the wrapper; refusal before any
// pointer is formed) and PR #1160 "score QSA token-indexer blocks in native
// CUDA" (rows and visible_len as separate device arrays; the RoPE tables are
// inputs; only rms_eps is a run-time scalar).
#include <atomic>
#include <cmath>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <cuda_runtime.h>

#include "../../include/qsa.h"
#include "qsa_launch.h"

namespace {

constexpr int32_t kVersion = 100;  // 0.1.0
constexpr int kHeadDim = 128;
constexpr int kRatio = 4;
constexpr int kRot = 64;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr long long kDefaultWaitLimit = 4000000000LL;  // ~2 s of SM clock at 2 GHz
std::atomic<long long> g_wait_limit{kDefaultWaitLimit};

qsa_status from_cuda(cudaError_t e) { return e == cudaSuccess ? QSA_OK : QSA_ERR_LAUNCH; }

bool eps_ok(float eps) { return !(eps < 0.0f) && !isnan(eps) && !isinf(eps); }

// Checks shared by every scoring entry.
qsa_status check_score_args(const uint16_t *q, int64_t q_stride, const int32_t *pos,
                            int32_t n_rows, int32_t tokens, const uint16_t *q_norm_w,
                            const uint16_t *cos_t, const uint16_t *sin_t, int32_t table_rows,
                            float eps, const uint16_t *block_keys, float *scores,
                            int64_t score_cols) {
  if (n_rows < 0 || tokens < 0 || table_rows < 0 || score_cols < 0) return QSA_ERR_INVALID_VALUE;
  if (!eps_ok(eps)) return QSA_ERR_INVALID_VALUE;
  if (n_rows == 0 || tokens == 0) return QSA_OK;
  if (!q || !pos || !q_norm_w || !cos_t || !sin_t || !block_keys || !scores)
    return QSA_ERR_INVALID_VALUE;
  if (q_stride < 4 * kHeadDim || (q_stride & 7) != 0) return QSA_ERR_INVALID_VALUE;
  if (!aligned16(q) || !aligned16(q_norm_w) || !aligned16(cos_t) || !aligned16(sin_t) ||
      !aligned16(block_keys) || !aligned16(scores))
    return QSA_ERR_INVALID_VALUE;
  if (score_cols < tokens / kRatio || (score_cols & 3) != 0) return QSA_ERR_INVALID_VALUE;
  if (table_rows < tokens) return QSA_ERR_INVALID_VALUE;
  // overflow: row offsets must fit in int64 element counts
  if ((int64_t)n_rows > INT64_MAX / (score_cols > 0 ? score_cols : 1)) return QSA_ERR_INVALID_VALUE;
  if ((int64_t)n_rows > INT64_MAX / q_stride) return QSA_ERR_INVALID_VALUE;
  return QSA_OK;
}

qsa_status check_select_args(const float *scores, int64_t score_cols, const int32_t *pos,
                             int32_t n_rows, int32_t tokens, int32_t budget, uint8_t *mask) {
  if (n_rows < 0 || tokens < 0 || score_cols < 0) return QSA_ERR_INVALID_VALUE;
  if (budget <= 0 || budget % kRatio != 0 || budget / kRatio > 512) return QSA_ERR_INVALID_VALUE;
  if (n_rows == 0 || tokens == 0) return QSA_OK;
  if (!scores || !pos || !mask) return QSA_ERR_INVALID_VALUE;
  if (!aligned16(scores) || (score_cols & 3) != 0 || score_cols < tokens / kRatio)
    return QSA_ERR_INVALID_VALUE;
  if ((int64_t)n_rows > INT64_MAX / (score_cols > 0 ? score_cols : 1)) return QSA_ERR_INVALID_VALUE;
  if ((int64_t)n_rows > INT64_MAX / tokens) return QSA_ERR_INVALID_VALUE;
  if ((int64_t)n_rows * 16 > (int64_t)INT32_MAX) return QSA_ERR_INVALID_VALUE;  // grid.x = rows * cluster
  return QSA_OK;
}

qsa_status check_pool_args(const uint16_t *keys, int64_t key_stride, int32_t first_block,
                           int32_t n_blocks, const uint16_t *k_norm_w, const uint16_t *cos_t,
                           const uint16_t *sin_t, int32_t table_rows, float eps,
                           uint16_t *block_keys) {
  if (n_blocks < 0 || first_block < 0 || table_rows < 0) return QSA_ERR_INVALID_VALUE;
  if (!eps_ok(eps)) return QSA_ERR_INVALID_VALUE;
  if (n_blocks == 0) return QSA_OK;
  if (!keys || !k_norm_w || !cos_t || !sin_t || !block_keys) return QSA_ERR_INVALID_VALUE;
  if (key_stride < kHeadDim || (key_stride & 7) != 0) return QSA_ERR_INVALID_VALUE;
  if (!aligned16(keys) || !aligned16(k_norm_w) || !aligned16(cos_t) || !aligned16(sin_t) ||
      !aligned16(block_keys))
    return QSA_ERR_INVALID_VALUE;
  const int64_t last = (int64_t)first_block + n_blocks - 1;
  if (last > INT32_MAX / kRatio) return QSA_ERR_INVALID_VALUE;
  if ((int64_t)table_rows <= kRatio * last) return QSA_ERR_INVALID_VALUE;  // position 4*last is read
  if ((int64_t)kRatio * n_blocks > INT64_MAX / key_stride) return QSA_ERR_INVALID_VALUE;
  return QSA_OK;
}

}  // namespace

long long qsa::wait_limit_cycles() { return g_wait_limit.load(std::memory_order_relaxed); }

extern "C" {

int32_t qsa_version(void) { return kVersion; }

qsa_status qsa_set_wait_limit_cycles(int64_t cycles) {
  if (cycles <= 0) return QSA_ERR_INVALID_VALUE;
  g_wait_limit.store(cycles, std::memory_order_relaxed);
  return QSA_OK;
}

int64_t qsa_wait_limit_cycles(void) { return g_wait_limit.load(std::memory_order_relaxed); }

const char *qsa_status_string(int32_t status) {
  switch (status) {
    case QSA_OK: return "ok";
    case QSA_ERR_INVALID_VALUE: return "invalid value (refused on the host, nothing launched)";
    case QSA_ERR_LAUNCH: return "kernel launch failed";
    case QSA_ERR_ROW_RANGE: return "row position or visible length out of range";
    case QSA_ERR_NONFINITE: return "non-finite score in a truncating row";
    case QSA_ERR_TIMEOUT: return "a bounded device wait gave up";
    case QSA_ERR_TOKEN_RANGE: return "a selected token or its page lies outside the page table or the pool";
    default: return "unknown status";
  }
}

qsa_status qsa_rope_tables(int32_t max_pos, double theta, uint16_t *cos_out, uint16_t *sin_out) {
  if (max_pos < 0 || !(theta > 0.0) || isinf(theta)) return QSA_ERR_INVALID_VALUE;
  if (max_pos == 0) return QSA_OK;
  if (!cos_out || !sin_out) return QSA_ERR_INVALID_VALUE;
  float inv_freq[kRot / 2];
  for (int j = 0; j < kRot / 2; ++j)
    inv_freq[j] = (float)(1.0 / pow(theta, (double)(2 * j) / (double)kRot));
  auto narrow = [](float f) -> uint16_t {  // f32 -> bf16, nearest-even, NaN kept
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40u);
    return (uint16_t)((u + 0x7fffu + ((u >> 16) & 1u)) >> 16);
  };
  for (int64_t p = 0; p < max_pos; ++p) {
    uint16_t *cr = cos_out + p * kRot;
    uint16_t *sr = sin_out + p * kRot;
    for (int j = 0; j < kRot / 2; ++j) {
      const float ang = (float)p * inv_freq[j];
      cr[j] = cr[j + kRot / 2] = narrow((float)cos((double)ang));
      sr[j] = sr[j + kRot / 2] = narrow((float)sin((double)ang));
    }
  }
  return QSA_OK;
}

qsa_status qsa_pool_blocks(const uint16_t *keys, int64_t key_stride, int32_t first_block,
                           int32_t n_blocks, const uint16_t *k_norm_w, const uint16_t *cos_t,
                           const uint16_t *sin_t, int32_t table_rows, float eps,
                           uint16_t *block_keys, void *stream) {
  qsa_status st = check_pool_args(keys, key_stride, first_block, n_blocks, k_norm_w, cos_t, sin_t,
                                  table_rows, eps, block_keys);
  if (st != QSA_OK || n_blocks == 0) return st;
  return from_cuda(qsa::launch_pool_blocks(keys, key_stride, first_block, n_blocks, k_norm_w,
                                           cos_t, sin_t, eps, block_keys,
                                           (cudaStream_t)stream));
}

int64_t qsa_score_workspace_bytes(int32_t n_rows) {
  return n_rows < 0 ? -1 : (int64_t)n_rows * 4 * kHeadDim * 2;
}

namespace {

// A caller workspace the tensor-core scorer can use for n_rows query rows.
bool score_ws_ok(const void *workspace, int64_t workspace_bytes, int32_t n_rows) {
  return workspace != nullptr && aligned16(workspace) &&
         workspace_bytes >= qsa_score_workspace_bytes(n_rows) && (int64_t)n_rows * 4 <= INT32_MAX;
}

// QSA_SCORE_AUTO's choice: the tensor-core tile scorer once there are enough
// rows to fill its 64-row tiles and blocks to fill a key tile, else the
// streaming tensor-core scorer.
bool auto_picks_tc(const int64_t *key_base, bool ws_ok, int32_t n_rows, int32_t tokens) {
  return qsa::kTcScorerReady && key_base == nullptr && ws_ok && n_rows >= 64 && tokens >= 2048;
}

}  // namespace

qsa_status qsa_score_rows_with(const uint16_t *q, int64_t q_stride, const int32_t *pos,
                               const int32_t *visible_len, int32_t n_rows, int32_t tokens,
                               const uint16_t *q_norm_w, const uint16_t *cos_t,
                               const uint16_t *sin_t, int32_t table_rows, float eps,
                               const uint16_t *block_keys, const int64_t *key_base,
                               float *scores, int64_t score_cols, int32_t *dev_status,
                               int32_t path, void *workspace, int64_t workspace_bytes,
                               void *stream) {
  if (path != QSA_SCORE_AUTO && path != QSA_SCORE_SIMT && path != QSA_SCORE_TCGEN05 &&
      path != QSA_SCORE_STREAM)
    return QSA_ERR_INVALID_VALUE;
  if (workspace_bytes < 0) return QSA_ERR_INVALID_VALUE;
  qsa_status st = check_score_args(q, q_stride, pos, n_rows, tokens, q_norm_w, cos_t, sin_t,
                                   table_rows, eps, block_keys, scores, score_cols);
  if (st != QSA_OK || n_rows == 0 || tokens == 0) return st;
  const bool ws_ok = score_ws_ok(workspace, workspace_bytes, n_rows);
  if (path == QSA_SCORE_TCGEN05 && (key_base != nullptr || !ws_ok)) return QSA_ERR_INVALID_VALUE;
  qsa::ScoreArgs a{q,          q_stride, pos,   visible_len, n_rows,     tokens,
                   q_norm_w,   cos_t,    sin_t, eps,         block_keys, key_base,
                   scores,     score_cols, dev_status, qsa::wait_limit_cycles()};
  if (path == QSA_SCORE_AUTO)
    path = auto_picks_tc(key_base, ws_ok, n_rows, tokens) ? QSA_SCORE_TCGEN05 : QSA_SCORE_STREAM;
  if (path == QSA_SCORE_TCGEN05)
    return from_cuda(qsa::launch_score_tc(a, static_cast<uint16_t *>(workspace), (cudaStream_t)stream));
  if (path == QSA_SCORE_STREAM) return from_cuda(qsa::launch_score_stream(a, (cudaStream_t)stream));
  return from_cuda(qsa::launch_score_simt(a, (cudaStream_t)stream));
}

qsa_status qsa_score_rows(const uint16_t *q, int64_t q_stride, const int32_t *pos,
                          const int32_t *visible_len, int32_t n_rows, int32_t tokens,
                          const uint16_t *q_norm_w, const uint16_t *cos_t, const uint16_t *sin_t,
                          int32_t table_rows, float eps, const uint16_t *block_keys,
                          const int64_t *key_base, float *scores, int64_t score_cols,
                          int32_t *dev_status, void *workspace, int64_t workspace_bytes,
                          void *stream) {
  return qsa_score_rows_with(q, q_stride, pos, visible_len, n_rows, tokens, q_norm_w, cos_t, sin_t,
                             table_rows, eps, block_keys, key_base, scores, score_cols, dev_status,
                             QSA_SCORE_AUTO, workspace, workspace_bytes, stream);
}

qsa_status qsa_select_mask(const float *scores, int64_t score_cols, const int32_t *pos,
                           int32_t n_rows, int32_t tokens, int32_t budget, uint8_t *mask,
                           int32_t *dev_status, void *stream) {
  qsa_status st = check_select_args(scores, score_cols, pos, n_rows, tokens, budget, mask);
  if (st != QSA_OK || n_rows == 0 || tokens == 0) return st;
  return from_cuda(qsa::launch_select(scores, score_cols, pos, n_rows, tokens, budget, mask,
                                      dev_status, (cudaStream_t)stream));
}

qsa_status qsa_index_select(const uint16_t *keys, int64_t key_stride, int32_t pool_first_block,
                            int32_t pool_n_blocks, const uint16_t *k_norm_w, const uint16_t *q,
                            int64_t q_stride, const int32_t *pos, int32_t n_rows, int32_t tokens,
                            const uint16_t *q_norm_w, const uint16_t *cos_t,
                            const uint16_t *sin_t, int32_t table_rows, float eps, int32_t budget,
                            uint16_t *block_keys, float *scores, int64_t score_cols,
                            uint8_t *mask, int32_t *dev_status, void *workspace,
                            int64_t workspace_bytes, void *stream) {
  // validate all three stages before launching any of them
  qsa_status st = check_pool_args(keys, key_stride, pool_first_block, pool_n_blocks, k_norm_w,
                                  cos_t, sin_t, table_rows, eps, block_keys);
  if (st != QSA_OK) return st;
  st = check_score_args(q, q_stride, pos, n_rows, tokens, q_norm_w, cos_t, sin_t, table_rows, eps,
                        block_keys, scores, score_cols);
  if (st != QSA_OK) return st;
  st = check_select_args(scores, score_cols, pos, n_rows, tokens, budget, mask);
  if (st != QSA_OK) return st;
  if (workspace_bytes < 0) return QSA_ERR_INVALID_VALUE;
  cudaStream_t s = (cudaStream_t)stream;
  // on the tensor-core path the new blocks are pooled by the query-prep launch
  const bool tc = n_rows > 0 && tokens > 0 &&
                  auto_picks_tc(nullptr, score_ws_ok(workspace, workspace_bytes, n_rows), n_rows,
                                tokens);
  if (pool_n_blocks > 0 && !tc) {
    st = from_cuda(qsa::launch_pool_blocks(keys, key_stride, pool_first_block, pool_n_blocks,
                                           k_norm_w, cos_t, sin_t, eps, block_keys, s));
    if (st != QSA_OK) return st;
  }
  if (n_rows == 0 || tokens == 0) return QSA_OK;
  if (tc) {
    const qsa::ScoreArgs a{q,          q_stride, pos,   nullptr, n_rows,     tokens,
                           q_norm_w,   cos_t,    sin_t, eps,     block_keys, nullptr,
                           scores,     score_cols, dev_status, qsa::wait_limit_cycles()};
    const qsa::PoolArgs pa{keys, key_stride, pool_first_block, pool_n_blocks, k_norm_w, block_keys};
    st = from_cuda(qsa::launch_score_tc(a, static_cast<uint16_t *>(workspace), s, &pa));
  } else {
    st = qsa_score_rows_with(q, q_stride, pos, nullptr, n_rows, tokens, q_norm_w, cos_t, sin_t,
                             table_rows, eps, block_keys, nullptr, scores, score_cols, dev_status,
                             QSA_SCORE_AUTO, workspace, workspace_bytes, stream);
  }
  if (st != QSA_OK) return st;
  return from_cuda(qsa::launch_select(scores, score_cols, pos, n_rows, tokens, budget, mask,
                                      dev_status, s));
}

int64_t qsa_decode_workspace_bytes(int32_t n_rows, int32_t tokens) {
  if (n_rows < 0 || tokens < 0) return -1;
  return (int64_t)n_rows * qsa::decode_row_ws_bytes(tokens);
}

qsa_status qsa_decode_index_select(const uint16_t *keys, int64_t key_stride,
                                   int32_t pool_first_block, int32_t pool_n_blocks,
                                   const uint16_t *k_norm_w, const uint16_t *q, int64_t q_stride,
                                   const int32_t *pos, int32_t n_rows, int32_t tokens,
                                   const uint16_t *q_norm_w, const uint16_t *cos_t,
                                   const uint16_t *sin_t, int32_t table_rows, float eps,
                                   int32_t budget, uint16_t *block_keys, float *scores,
                                   int64_t score_cols, uint8_t *mask, int32_t *dev_status,
                                   void *decode_ws, int64_t decode_ws_bytes, void *stream) {
  qsa_status st = check_pool_args(keys, key_stride, pool_first_block, pool_n_blocks, k_norm_w,
                                  cos_t, sin_t, table_rows, eps, block_keys);
  if (st != QSA_OK) return st;
  st = check_score_args(q, q_stride, pos, n_rows, tokens, q_norm_w, cos_t, sin_t, table_rows, eps,
                        block_keys, scores, score_cols);
  if (st != QSA_OK) return st;
  st = check_select_args(scores, score_cols, pos, n_rows, tokens, budget, mask);
  if (st != QSA_OK) return st;
  const int64_t need = qsa_decode_workspace_bytes(n_rows, tokens);
  if (n_rows > 0 && tokens > 0 &&
      (decode_ws == nullptr || decode_ws_bytes < need ||
       (reinterpret_cast<uintptr_t>(decode_ws) & 15u) != 0))
    return QSA_ERR_INVALID_VALUE;
  cudaStream_t s = (cudaStream_t)stream;
  auto pool_launch = [&]() -> qsa_status {
    if (pool_n_blocks == 0) return QSA_OK;
    return from_cuda(qsa::launch_pool_blocks(keys, key_stride, pool_first_block, pool_n_blocks,
                                             k_norm_w, cos_t, sin_t, eps, block_keys, s));
  };
  if (n_rows == 0 || tokens == 0) return pool_launch();
  // new blocks inside the token range are pooled by the fused launch itself
  const bool pool_inside =
      (int64_t)pool_first_block + pool_n_blocks <= (int64_t)(tokens / 4);
  if (!pool_inside && (st = pool_launch()) != QSA_OK) return st;
  qsa::ScoreArgs a = {q,        q_stride, pos,        nullptr,    n_rows, tokens, q_norm_w,
                      cos_t,    sin_t,    eps,        block_keys, nullptr, scores, score_cols,
                      dev_status, qsa::wait_limit_cycles()};
  bool launched = false;
  st = from_cuda(qsa::launch_decode_fused(a, budget, mask, decode_ws, keys, key_stride,
                                          pool_first_block, pool_inside ? pool_n_blocks : 0,
                                          k_norm_w, block_keys, s, &launched));
  if (st != QSA_OK || launched) return st;
  // more rows than can be co-resident: pool, score and select in turn
  if (pool_inside && (st = pool_launch()) != QSA_OK) return st;
  st = from_cuda(qsa::launch_score_stream(a, s));
  if (st != QSA_OK) return st;
  return from_cuda(qsa::launch_select(scores, score_cols, pos, n_rows, tokens, budget, mask,
                                      dev_status, s));
}

qsa_status qsa_mask_tokens(const uint8_t *mask, int32_t n_rows, int32_t tokens, int32_t *sel,
                           int64_t sel_cols, int32_t *n_sel, void *stream) {
  if (n_rows < 0 || tokens < 0 || sel_cols < 0) return QSA_ERR_INVALID_VALUE;
  if (n_rows == 0) return QSA_OK;
  if (!n_sel || (tokens > 0 && !mask) || (sel_cols > 0 && !sel)) return QSA_ERR_INVALID_VALUE;
  if ((int64_t)n_rows * tokens > ((int64_t)1 << 46) || (int64_t)n_rows * sel_cols > ((int64_t)1 << 46))
    return QSA_ERR_INVALID_VALUE;
  return from_cuda(qsa::launch_mask_tokens(mask, n_rows, tokens, sel, sel_cols, n_sel,
                                           (cudaStream_t)stream));
}

qsa_status qsa_gather_kv(const uint16_t *k_pool, const uint16_t *v_pool, int32_t width,
                         int32_t pool_pages, const int32_t *table, int32_t table_len,
                         int64_t table_cols, int32_t page_size, const int32_t *sel,
                         int64_t sel_cols, const int32_t *n_sel, int32_t n_rows, int32_t max_sel,
                         uint16_t *k_out, uint16_t *v_out, int64_t out_rows, int32_t *dev_status,
                         void *stream) {
  if (n_rows < 0 || max_sel < 0 || width < 0 || pool_pages < 0 || table_len < 0 ||
      table_cols < 0 || sel_cols < 0 || out_rows < 0)
    return QSA_ERR_INVALID_VALUE;
  if (n_rows == 0 || max_sel == 0 || width == 0) return QSA_OK;
  if (width % 8 != 0 || page_size <= 0 || max_sel > sel_cols || max_sel > out_rows)
    return QSA_ERR_INVALID_VALUE;
  if (table_cols != 0 && table_cols < table_len) return QSA_ERR_INVALID_VALUE;
  if (!k_pool || !v_pool || !table || !sel || !n_sel || !k_out || !v_out || !dev_status)
    return QSA_ERR_INVALID_VALUE;
  if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(k_out) || !aligned16(v_out))
    return QSA_ERR_INVALID_VALUE;
  if ((int64_t)pool_pages * page_size * width > ((int64_t)1 << 46) ||
      (int64_t)n_rows * out_rows * width > ((int64_t)1 << 46) ||
      (int64_t)n_rows * sel_cols > ((int64_t)1 << 46) ||
      (int64_t)table_len * page_size > INT32_MAX)
    return QSA_ERR_INVALID_VALUE;
  return from_cuda(qsa::launch_gather_kv(k_pool, v_pool, width, pool_pages, table, table_len,
                                         table_cols, page_size, sel, sel_cols, n_sel, n_rows,
                                         max_sel, k_out, v_out, out_rows, dev_status,
                                         (cudaStream_t)stream));
}

qsa_status qsa_sparse_attn(const uint16_t *q, int64_t q_stride, int32_t nq, int32_t nkv,
                           int32_t head_dim, const uint16_t *k_pool, const uint16_t *v_pool,
                           int32_t pool_pages, int32_t page_size, const int32_t *table,
                           int32_t table_len, int64_t table_cols, const int32_t *sel,
                           int64_t sel_cols, const int32_t *n_sel, int32_t n_rows, int32_t max_sel,
                           float scale, uint16_t *out, int64_t out_stride, int32_t *dev_status,
                           void *stream) {
  if (n_rows < 0 || max_sel < 0 || pool_pages < 0 || table_len < 0 || table_cols < 0 ||
      sel_cols < 0 || q_stride < 0 || out_stride < 0)
    return QSA_ERR_INVALID_VALUE;
  if (n_rows == 0) return QSA_OK;
  if (nq <= 0 || nkv <= 0 || nq % nkv != 0 || (head_dim != 128 && head_dim != 256) ||
      page_size <= 0 || max_sel > sel_cols || !std::isfinite(scale))
    return QSA_ERR_INVALID_VALUE;
  if (table_cols != 0 && table_cols < table_len) return QSA_ERR_INVALID_VALUE;
  const int64_t row_len = (int64_t)nq * head_dim;
  if (q_stride < row_len || out_stride < row_len || (q_stride & 7) != 0 || (out_stride & 7) != 0)
    return QSA_ERR_INVALID_VALUE;
  if (!q || !k_pool || !v_pool || !out || !n_sel || !dev_status ||
      (max_sel > 0 && (!sel || !table)))
    return QSA_ERR_INVALID_VALUE;
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out))
    return QSA_ERR_INVALID_VALUE;
  const int64_t chunks = (nq / nkv + 7) / 8;
  if ((int64_t)n_rows * nkv * chunks > INT32_MAX || (int64_t)table_len * page_size > INT32_MAX ||
      (int64_t)pool_pages * page_size * nkv * head_dim > ((int64_t)1 << 46) ||
      (int64_t)n_rows * (q_stride > out_stride ? q_stride : out_stride) > ((int64_t)1 << 46) ||
      (int64_t)n_rows * sel_cols > ((int64_t)1 << 46))
    return QSA_ERR_INVALID_VALUE;
  return from_cuda(qsa::launch_sparse_attn(q, q_stride, nq, nkv, head_dim, k_pool, v_pool,
                                           pool_pages, page_size, table, table_len, table_cols,
                                           sel, sel_cols, n_sel, n_rows, max_sel, scale, out,
                                           out_stride, dev_status, (cudaStream_t)stream));
}

qsa_status qsa_qk_proj(const uint16_t *x, int64_t x_stride, const uint16_t *w, int32_t n_rows,
                       int32_t hidden, int32_t out_cols, uint16_t *y, int64_t y_stride,
                       int32_t *dev_status, void *stream) {
  if (n_rows < 0 || hidden < 0 || out_cols < 0 || x_stride < 0 || y_stride < 0)
    return QSA_ERR_INVALID_VALUE;
  if (n_rows == 0) return QSA_OK;
  if (hidden == 0 || hidden % 8 != 0 || out_cols == 0 || out_cols % 16 != 0)
    return QSA_ERR_INVALID_VALUE;
  if (x_stride < hidden || x_stride % 8 != 0 || y_stride < out_cols || y_stride % 8 != 0)
    return QSA_ERR_INVALID_VALUE;
  if (!x || !w || !y || !dev_status) return QSA_ERR_INVALID_VALUE;
  if (!aligned16(x) || !aligned16(w) || !aligned16(y)) return QSA_ERR_INVALID_VALUE;
  if ((int64_t)n_rows > (int64_t)65535 * 128 ||
      (int64_t)n_rows * (x_stride > y_stride ? x_stride : y_stride) > ((int64_t)1 << 46) ||
      (int64_t)hidden * out_cols > ((int64_t)1 << 46))
    return QSA_ERR_INVALID_VALUE;
  return from_cuda(qsa::launch_proj(x, x_stride, w, n_rows, hidden, out_cols, y, y_stride,
                                    dev_status, (cudaStream_t)stream));
}

qsa_status qsa_reset_status(int32_t *dev_status, void *stream) {
  if (!dev_status) return QSA_ERR_INVALID_VALUE;
  return from_cuda(cudaMemsetAsync(dev_status, 0, 2 * sizeof(int32_t), (cudaStream_t)stream));
}

qsa_status qsa_read_status(const int32_t *dev_status, void *stream, int32_t *host_code,
                           int32_t *host_row) {
  if (!dev_status || !host_code || !host_row) return QSA_ERR_INVALID_VALUE;
  int32_t h[2] = {0, 0};
  cudaError_t e = cudaMemcpyAsync(h, dev_status, sizeof(h), cudaMemcpyDeviceToHost,
                                  (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return QSA_ERR_LAUNCH;
  *host_code = h[0];
  *host_row = h[1];
  return QSA_OK;
}

}  // extern "C"
