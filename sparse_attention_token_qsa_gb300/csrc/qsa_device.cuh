// Device helpers for the QSA indexer kernels (sm_103a).
//
// Arithmetic conventions (PR #1160 "score QSA token-indexer blocks in native
// CUDA": block keys are averaged in float32 and cast back to bf16, then (1 + w)
// RMSNorm and partial RoPE, every bf16 rounding point of the reference kept;
// its "Tolerance" section: the reference rounds float32 reductions):
//  * the 4-token sum and the 128-term sum of squares are computed error-free
//    (TwoSum cascades), so each equals the exact sum rounded once to f32;
//  * every other step is one IEEE f32 operation (explicit _rn intrinsics, so
//    no FMA contraction changes a rounding), then bf16 where the reference
//    rounds to bf16.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace qsa {

constexpr int kHeads = 4;
constexpr int kHeadDim = 128;
constexpr int kRatio = 4;
constexpr int kRot = 64;
constexpr int kHalf = 32;
constexpr int kMaxKeep = 512;  // budget / 4 <= 512

enum : int32_t {
  kOk = 0,
  kErrRowRange = 3,
  kErrNonFinite = 4,
  kErrTimeout = 5,
  kErrTokenRange = 6,
};

__device__ __forceinline__ float bf16_to_f32(uint32_t h16) { return __uint_as_float(h16 << 16); }

__device__ __forceinline__ uint32_t f32_to_bf16(float f) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f));
}

__device__ __forceinline__ float round_bf16(float f) { return bf16_to_f32(f32_to_bf16(f)); }

// Low / high bf16 of a packed pair.
__device__ __forceinline__ float lo_bf16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_bf16(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16(uint32_t lo, uint32_t hi) { return lo | (hi << 16); }

// Error-free transformation: a + b = s + e exactly (Knuth's TwoSum).
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
  s = __fadd_rn(a, b);
  float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// Programmatic dependent launch.  Every kernel of the library is launched so
// that it may start while the previous kernel in its stream is finishing;
// this call, made by every thread before its first global memory access and
// before any early return, waits until that kernel has completed and its
// writes are visible, then lets the next kernel in the stream begin to
// launch.  A launch without the programmatic attribute passes both at once.
__device__ __forceinline__ void grid_dependency_sync() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Record the first device-side error: {code, row}.  Never traps.
__device__ __forceinline__ void report_error(int32_t *status, int32_t code, int32_t row) {
  if (status == nullptr) return;
  if (atomicCAS(status, 0, code) == 0) atomicExch(status + 1, row);
}

// (1 + w) RMSNorm then partial RoPE of one 128-vector held by a 16-lane group:
// lane g (0..15 within the group) holds dims 8g..8g+7 in x[] (bf16 values as
// f32).  Lanes 0-3 hold dims 0..31, lanes 4-7 dims 32..63 (the rotated half,
// paired (i, i+32)), lanes 8-15 the unrotated dims.  `w8` holds the weight's
// 8 bf16 for those dims, `c8`/`s8` the cos/sin row's entries 8g..8g+7 (lanes
// 0..7 only).  Returns the 8 output bf16 packed in a uint4.  All 32 lanes of
// the warp must call this (two groups per warp).
__device__ __forceinline__ uint4 norm_rope_16(const float (&x)[8], const uint4 &w8, const uint4 &c8,
                                              const uint4 &s8, float eps, int g) {
  // sum of squares, error-free: squares of bf16 values are exact in f32
  float hi = 0.f, lo = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    float sq = __fmul_rn(x[e], x[e]);
    float s, err;
    two_sum(hi, sq, s, err);
    hi = s;
    lo = __fadd_rn(lo, err);
  }
#pragma unroll
  for (int off = 8; off >= 1; off >>= 1) {
    float ohi = __shfl_xor_sync(0xffffffffu, hi, off);
    float olo = __shfl_xor_sync(0xffffffffu, lo, off);
    float s, err;
    two_sum(hi, ohi, s, err);
    hi = s;
    lo = __fadd_rn(__fadd_rn(lo, olo), err);
  }
  const float ms = __fmul_rn(__fadd_rn(hi, lo), 1.0f / 128.0f);
  const float r = __frcp_rn(__fsqrt_rn(__fadd_rn(ms, eps)));

  const uint32_t wv[4] = {w8.x, w8.y, w8.z, w8.w};
  float n[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float w = (e & 1) ? hi_bf16(wv[e >> 1]) : lo_bf16(wv[e >> 1]);
    n[e] = round_bf16(__fmul_rn(__fmul_rn(x[e], r), __fadd_rn(1.0f, w)));
  }
  // partner half of the rotary pair lives 4 lanes away
  float part[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) part[e] = __shfl_xor_sync(0xffffffffu, n[e], 4);

  const uint32_t cv[4] = {c8.x, c8.y, c8.z, c8.w};
  const uint32_t sv[4] = {s8.x, s8.y, s8.z, s8.w};
  // out_i = x_i c - x_{i+32} s (lanes 0-3), out_{i+32} = x_{i+32} c + x_i s
  // (lanes 4-7), unrotated dims pass (lanes 8-15); branch-free, with a - b
  // taken as a + (-b), which IEEE defines to be the same operation
  const bool rot = g < 8, neg = g < 4;
  uint32_t o[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float c = (e & 1) ? hi_bf16(cv[e >> 1]) : lo_bf16(cv[e >> 1]);
    const float s = (e & 1) ? hi_bf16(sv[e >> 1]) : lo_bf16(sv[e >> 1]);
    const float t1 = round_bf16(__fmul_rn(n[e], c));
    const float t2 = round_bf16(__fmul_rn(part[e], s));
    const float r = __fadd_rn(t1, neg ? -t2 : t2);
    o[e] = f32_to_bf16(rot ? r : n[e]);
  }
  return make_uint4(pack_bf16(o[0], o[1]), pack_bf16(o[2], o[3]), pack_bf16(o[4], o[5]),
                    pack_bf16(o[6], o[7]));
}

__device__ __forceinline__ void unpack8(const uint4 &v, float (&x)[8]) {
  x[0] = lo_bf16(v.x); x[1] = hi_bf16(v.x);
  x[2] = lo_bf16(v.y); x[3] = hi_bf16(v.y);
  x[4] = lo_bf16(v.z); x[5] = hi_bf16(v.z);
  x[6] = lo_bf16(v.w); x[7] = hi_bf16(v.w);
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// The pooled key of block b, computed by a 16-lane group (every lane calls
// it; lane g returns dims 8g..8g+7): tok0 points at the block's first raw key,
// the next three follow key_stride apart.  PR #1160 "score QSA token-indexer
// blocks in native CUDA", description: the four keys averaged in float32 (the
// exact sum rounded once, then x 1/4), cast back to bf16, (1 + w) RMSNorm, and
// partial RoPE at the block's first token, 4b.
__device__ __forceinline__ uint4 pool_block_16(const uint16_t *tok0, int64_t key_stride, int64_t b,
                                               const uint16_t *k_norm_w, const uint16_t *cos_t,
                                               const uint16_t *sin_t, float eps, int g) {
  const uint16_t *k0 = tok0 + 8 * g;
  uint4 t0 = ldg_nc_v4(k0);
  uint4 t1 = ldg_nc_v4(k0 + key_stride);
  uint4 t2 = ldg_nc_v4(k0 + 2 * key_stride);
  uint4 t3 = ldg_nc_v4(k0 + 3 * key_stride);
  const uint4 w8 = ldg_nc_v4(k_norm_w + 8 * g);
  uint4 c8 = make_uint4(0, 0, 0, 0), s8 = make_uint4(0, 0, 0, 0);
  if (g < 8) {
    const int64_t P = (int64_t)kRatio * b;  // the block's first token
    c8 = ldg_nc_v4(cos_t + P * kRot + 8 * g);
    s8 = ldg_nc_v4(sin_t + P * kRot + 8 * g);
  }
  float a[8], bb[8], c[8], d[8], m[8];
  unpack8(t0, a);
  unpack8(t1, bb);
  unpack8(t2, c);
  unpack8(t3, d);
  // The mean needs the exact sum of the 4 bf16 values rounded once to f32.
  // When the smallest magnitude of a dim's four is at least 2^-14 of the
  // largest (their exponents at most 14 apart) and the largest is below 2^125,
  // every partial sum is a multiple of the smallest value's bf16 quantum below
  // 2^24 quanta, so plain f32 additions are exact; a warp whose lanes all meet
  // that takes them, any other the TwoSum cascade (same result).  A zero sum
  // is +0 on both (the plain one adds +0 last: four -0 keys sum to +0, as the
  // exact definition, which starts from +0, gives).
  bool plain = true;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float hi = fmaxf(fmaxf(fabsf(a[e]), fabsf(bb[e])), fmaxf(fabsf(c[e]), fabsf(d[e])));
    const float lo = fminf(fminf(fabsf(a[e]), fabsf(bb[e])), fminf(fabsf(c[e]), fabsf(d[e])));
    plain = plain && hi < 0x1p125f && __fmul_rn(lo, 16384.0f) >= hi;
  }
  if (__all_sync(0xffffffffu, plain)) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float sum =
          __fadd_rn(__fadd_rn(__fadd_rn(__fadd_rn(a[e], bb[e]), c[e]), d[e]), 0.0f);
      m[e] = round_bf16(__fmul_rn(sum, 0.25f));  // f32 mean, cast back to bf16
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      // exact sum of the 4 bf16 values, rounded once to f32 (TwoSum cascade)
      float s1, e1, s2, e2, s3, e3;
      two_sum(a[e], bb[e], s1, e1);
      two_sum(s1, c[e], s2, e2);
      two_sum(s2, d[e], s3, e3);
      const float sum = __fadd_rn(s3, __fadd_rn(__fadd_rn(e1, e2), e3));
      m[e] = round_bf16(__fmul_rn(sum, 0.25f));  // f32 mean, cast back to bf16
    }
  }
  return norm_rope_16(m, w8, c8, s8, eps, g);
}

__device__ __forceinline__ uint4 ldg_v4(const void *p) {
  return *reinterpret_cast<const uint4 *>(p);
}

}  // namespace qsa
