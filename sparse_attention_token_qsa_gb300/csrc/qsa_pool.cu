// Block pooling kernel: one pooled bf16 key per complete 4-token block.
//
// PR #1160 "score QSA token-indexer blocks in native CUDA", description: every
// complete micro-block of compress_ratio = 4 raw keys is averaged in float32,
// cast back to bf16, (1 + w) RMSNorm'd and rotated (partial RoPE, 64 of 128
// dims) at the block's FIRST token; one pass over the keys serves every row.
// metrale layers/qsa.rs (pool_new_blocks) pools only newly complete blocks,
// which is why the launch takes [first_block, first_block + n_blocks).
//
// Layout: a half-warp (16 lanes) owns one block; lane g loads the 16-byte
// slice (dims 8g..8g+7) of each of the four token rows, so each token row is
// one coalesced 256-byte read and the output row one 256-byte write.  HBM
// traffic per block: 1024 B keys + 256 B out + 256 B cos/sin rows.
#include "qsa_device.cuh"
#include "qsa_launch.h"

namespace qsa {

// 8 blocks per CTA: with 56 registers a thread, 128-thread CTAs leave a
// smaller partial last wave than 256-thread ones (3-4 % faster at 16k and at
// 1.5M blocks)
constexpr int kPoolThreads = 128;
constexpr int kPoolBlocksPerCta = kPoolThreads / 16;

__global__ void __launch_bounds__(kPoolThreads)
pool_blocks_kernel(const uint16_t *__restrict__ keys, int64_t key_stride, int32_t first_block,
                   int32_t n_blocks, const uint16_t *__restrict__ k_norm_w,
                   const uint16_t *__restrict__ cos_t, const uint16_t *__restrict__ sin_t,
                   float eps, uint16_t *__restrict__ block_keys) {
  grid_dependency_sync();
  const int lane = threadIdx.x & 31;
  const int g = lane & 15;
  const int64_t i = (int64_t)blockIdx.x * kPoolBlocksPerCta + (threadIdx.x >> 4);
  // Both half-warps must reach the shuffles in norm_rope_16: clamp the block
  // index of an idle half-warp and drop its store instead of returning early.
  const bool active = i < n_blocks;
  const int64_t ii = active ? i : (int64_t)n_blocks - 1;
  const int64_t b = (int64_t)first_block + ii;

  const uint4 out = pool_block_16(keys + (int64_t)kRatio * ii * key_stride, key_stride, b, k_norm_w,
                                  cos_t, sin_t, eps, g);
  if (active) *reinterpret_cast<uint4 *>(block_keys + b * kHeadDim + 8 * g) = out;
}

cudaError_t launch_pool_blocks(const uint16_t *keys, int64_t key_stride, int32_t first_block,
                               int32_t n_blocks, const uint16_t *k_norm_w, const uint16_t *cos_t,
                               const uint16_t *sin_t, float eps, uint16_t *block_keys,
                               cudaStream_t stream) {
  const int64_t grid = ((int64_t)n_blocks + kPoolBlocksPerCta - 1) / kPoolBlocksPerCta;
  return launch_dependent(pool_blocks_kernel, dim3((unsigned)grid), dim3(kPoolThreads), 0, stream,
                          1u, keys, key_stride, first_block, n_blocks, k_norm_w, cos_t, sin_t,
                          eps, block_keys);
}

}  // namespace qsa
