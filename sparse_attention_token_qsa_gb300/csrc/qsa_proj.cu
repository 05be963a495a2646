// The index_qk_proj projection: fused_qk = x W^T, a dense bf16 GEMM.
//
// atlas layers/qsa_select.rs prefill_select projects each 2048-row slab of
// the normed hidden states with the indexer's qk projection (hidden -> 640:
// four query heads and the raw key) before q-prep and scoring; W is a linear
// layer's weight, [out, in].  Both operands are K-major, which is the
// tcgen05 layout: D[row, col] = sum_k x[row, k] W[col, k].
//
// One CTA per output tile of 128 rows x BN columns, BN = 160 when such tiles
// alone fill most of the GPU (4096 x 640: 128 CTAs) and 80 otherwise (a 2048 x
// 640 slab: 16 x 8 = 128 CTAs): a tcgen05.mma takes about as long at N = 80 as
// at N = 160, so the wider tile does twice the work per instruction.  Warp 0's
// lane 0 streams 128-wide K slices of both operands with TMA (two 64-wide
// boxes each, 128-byte swizzle, zero fill past the matrix edges) into a ring
// of four (BN = 80) or three (BN = 160) stages; warp 1's lane 0 issues
// tcgen05.mma M128 N=BN K16 eight times per slice into a TMEM accumulator
// (f32) -- one barrier wait per eight instructions: 64-wide slices, one wait
// per four, took a quarter longer -- then all four warps drain their 32 TMEM
// lanes (one output row per thread), round to bf16 and store.  Every wait is
// bounded; on a timeout the CTA records QSA_ERR_TIMEOUT.
#include <cuda.h>  // CUtensorMap and its enums (the encoder comes from the runtime)

#include "qsa_device.cuh"
#include "qsa_launch.h"

namespace qsa {

namespace {

constexpr int kPM = 128;        // output rows per tile (TMEM lanes)
constexpr int kPK = 64;         // K per TMA box: one 128-byte swizzled row of bf16
constexpr int kPKS = 128;       // K per stage: two boxes
constexpr int kPStages = 4;     // ring slots (the most any tile width uses)
constexpr int kPThreads = 128;
constexpr uint32_t kPAStage = kPM * kPKS * 2;  // 32 KiB
constexpr uint32_t kPAChunk = kPM * kPK * 2;   // 16 KiB
constexpr long long kPSpinLimit = 4000000000LL;

// Tile geometry for BN output columns per tile (80 or 160).  A tcgen05.mma
// costs about the same time at N = 80 as at N = 160, so wide tiles pay when
// there are enough of them to fill the GPU.
template <int BN>
struct ProjGeom {
  static constexpr int kStages = BN <= 96 ? 4 : 3;
  static constexpr uint32_t kBStage = BN * kPKS * 2;
  static constexpr uint32_t kBChunk = BN * kPK * 2;
  static constexpr uint32_t kAOff = 0;
  static constexpr uint32_t kBOff = kStages * kPAStage;
  static constexpr uint32_t kCtrlOff = kBOff + kStages * kBStage;
  static constexpr uint32_t kTmemCols = BN <= 128 ? 128 : 256;  // a power of two >= BN
  // instruction descriptor, kind::f16: D f32, A and B bf16, both K-major, M = 128, N = BN
  static constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                                     ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(kPM >> 4) << 24);
};

struct ProjCtrl {
  uint64_t full[kPStages];
  uint64_t empty[kPStages];
  uint64_t done;
  uint32_t tmem_base;
  int32_t abort;
};
template <int BN>
constexpr size_t proj_smem() { return ProjGeom<BN>::kCtrlOff + sizeof(ProjCtrl) + 1024; }

__device__ __forceinline__ uint32_t p_smem(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ bool p_try(uint32_t a, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(a), "r"(parity), "r"(20000u)
      : "memory");
  return ok != 0;
}

// Bounded wait; raises the CTA's abort flag at the limit, gives up when
// another role has raised it.
__device__ bool p_wait(uint32_t a, uint32_t parity, volatile int32_t *abort_flag) {
  const long long t0 = clock64();
  while (true) {
    if (p_try(a, parity)) return true;
    if (abort_flag != nullptr && *abort_flag) return false;
    if (clock64() - t0 > kPSpinLimit) {
      if (abort_flag != nullptr) *abort_flag = 1;
      return false;
    }
  }
}

__device__ __forceinline__ void p_expect_tx(uint32_t a, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(a), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void p_tma_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                         uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(mbar)
      : "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart, descriptor version 1.
__device__ __forceinline__ uint64_t p_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)1u << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)2u << 61;
  return d;
}

__device__ __forceinline__ void p_mma(uint32_t dtmem, uint64_t adesc, uint64_t bdesc,
                                      uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(dtmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void p_commit(uint32_t mbar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar)
      : "memory");
}

__device__ __forceinline__ void p_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
        "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ uint32_t p_pack(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

template <int BN>
__global__ void __launch_bounds__(kPThreads, 1)
proj_kernel(const __grid_constant__ CUtensorMap amap, const __grid_constant__ CUtensorMap bmap,
            uint16_t *__restrict__ y, int64_t y_stride, int32_t n_rows, int32_t out_cols,
            int32_t nk, int32_t *status) {
  using G = ProjGeom<BN>;
  extern __shared__ uint8_t p_smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(p_smem_raw) + 1023) & ~uintptr_t(1023));
  ProjCtrl &C = *reinterpret_cast<ProjCtrl *>(smem + G::kCtrlOff);
  const uint32_t sA = p_smem(smem + G::kAOff), sB = p_smem(smem + G::kBOff);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n0 = blockIdx.x * BN, m0 = blockIdx.y * kPM;
  grid_dependency_sync();  // before TMEM too: an earlier launch may hold it

  if (tid == 0) {
    for (int s = 0; s < G::kStages; ++s) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(p_smem(&C.full[s])) : "memory");
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(p_smem(&C.empty[s])) : "memory");
    }
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(p_smem(&C.done)) : "memory");
    C.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 2) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     p_smem(&C.tmem_base)),
                 "r"(G::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = C.tmem_base;
  volatile int32_t *abort_flag = &C.abort;

  if (warp == 0) {
    // ---- TMA producer
    if (lane == 0) {
      int issued = 0;
      for (int kb = 0; kb < nk; ++kb) {
        const int s = kb % G::kStages;
        const uint32_t it = (uint32_t)(kb / G::kStages);
        if (!p_wait(p_smem(&C.empty[s]), (it & 1u) ^ 1u, abort_flag)) break;
        const uint32_t fb = p_smem(&C.full[s]);
        p_expect_tx(fb, kPAStage + G::kBStage);
        p_tma_2d(sA + s * kPAStage, &amap, kb * kPKS, m0, fb);
        p_tma_2d(sA + s * kPAStage + kPAChunk, &amap, kb * kPKS + kPK, m0, fb);
        p_tma_2d(sB + s * G::kBStage, &bmap, kb * kPKS, n0, fb);
        p_tma_2d(sB + s * G::kBStage + G::kBChunk, &bmap, kb * kPKS + kPK, n0, fb);
        issued = kb + 1;
      }
      if (*abort_flag) {  // let our own copies land before the CTA leaves
        for (int kb = issued - G::kStages < 0 ? 0 : issued - G::kStages; kb < issued; ++kb)
          p_wait(p_smem(&C.full[kb % G::kStages]), (uint32_t)(kb / G::kStages) & 1u, nullptr);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---- MMA issuer
    if (lane == 0) {
      bool ok = true;
      for (int kb = 0; kb < nk && ok; ++kb) {
        const int s = kb % G::kStages;
        const uint32_t it = (uint32_t)(kb / G::kStages);
        {
          // non-suspending polls: the stage has usually landed already (a
          // suspending wait here cost about 2 % at 2048 and 4096 rows)
          const uint32_t fa = p_smem(&C.full[s]);
          const long long t0 = clock64();
          while (true) {
            uint32_t done;
            asm volatile(
                "{\n\t.reg .pred p;\n\t"
                "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                "selp.u32 %0, 1, 0, p;\n\t}"
                : "=r"(done)
                : "r"(fa), "r"(it & 1u)
                : "memory");
            if (done) break;
            if (*abort_flag) {
              ok = false;
              break;
            }
            if (clock64() - t0 > kPSpinLimit) {
              *abort_flag = 1;
              ok = false;
              break;
            }
          }
        }
        if (!ok) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll
        for (int kk = 0; kk < kPKS / 16; ++kk) {  // K = 16 per MMA: 32 bytes along the swizzled row
          const uint32_t ka = (uint32_t)(kk >> 2) * kPAChunk + (uint32_t)(kk & 3) * 32u;
          const uint32_t kbb = (uint32_t)(kk >> 2) * G::kBChunk + (uint32_t)(kk & 3) * 32u;
          p_mma(tmem, p_desc(sA + s * kPAStage + ka), p_desc(sB + s * G::kBStage + kbb),
                G::kIdesc, (kb > 0 || kk > 0) ? 1u : 0u);
        }
        p_commit(p_smem(&C.empty[s]));
      }
      // the accumulator is complete (or the CTA aborted) once every MMA issued has drained
      p_commit(p_smem(&C.done));
    }
    __syncwarp();
  }

  // ---- epilogue: warp w drains TMEM lanes 32w .. 32w + 31 (output rows m0 + 32w + lane)
  uint32_t ok = 0;
  if (lane == 0) ok = (p_wait(p_smem(&C.done), 0u, abort_flag) && !*abort_flag) ? 1u : 0u;
  ok = __shfl_sync(0xffffffffu, ok, 0);  // one verdict per warp
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (ok) {
    const int r = m0 + 32 * warp + lane;
    const uint32_t taddr = tmem + ((uint32_t)(32 * warp) << 16);
    uint16_t *dst = y + (int64_t)r * y_stride + n0;
#pragma unroll
    for (int c = 0; c < BN / 16; ++c) {
      uint32_t v[16];
      p_ld16(taddr + (uint32_t)(16 * c), v);  // every lane of the warp takes part
      if (r < n_rows && n0 + 16 * c < out_cols) {
        uint4 lo, hi;
        lo.x = p_pack(__uint_as_float(v[0]), __uint_as_float(v[1]));
        lo.y = p_pack(__uint_as_float(v[2]), __uint_as_float(v[3]));
        lo.z = p_pack(__uint_as_float(v[4]), __uint_as_float(v[5]));
        lo.w = p_pack(__uint_as_float(v[6]), __uint_as_float(v[7]));
        hi.x = p_pack(__uint_as_float(v[8]), __uint_as_float(v[9]));
        hi.y = p_pack(__uint_as_float(v[10]), __uint_as_float(v[11]));
        hi.z = p_pack(__uint_as_float(v[12]), __uint_as_float(v[13]));
        hi.w = p_pack(__uint_as_float(v[14]), __uint_as_float(v[15]));
        *reinterpret_cast<uint4 *>(dst + 16 * c) = lo;
        *reinterpret_cast<uint4 *>(dst + 16 * c + 8) = hi;
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (*abort_flag && tid == 0) report_error(status, kErrTimeout, (int32_t)blockIdx.y);
  if (warp == 2) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(G::kTmemCols)
                 : "memory");
  }
}

using PEncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                               const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                               const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                               CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder (process-wide; looked up once, thread-safe).
PEncodeFn p_encoder() {
  static const PEncodeFn fn = []() -> PEncodeFn {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PEncodeFn>(p);
    cudaGetLastError();
    return nullptr;
  }();
  return fn;
}

}  // namespace

cudaError_t launch_proj(const uint16_t *x, int64_t x_stride, const uint16_t *w, int32_t n_rows,
                        int32_t hidden, int32_t out_cols, uint16_t *y, int64_t y_stride,
                        int32_t *status, cudaStream_t stream) {
  if (n_rows == 0) return cudaSuccess;
  PEncodeFn enc = p_encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  const cuuint32_t estr[2] = {1, 1};
  CUtensorMap amap;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)hidden, (cuuint64_t)n_rows};
    const cuuint64_t strides[1] = {(cuuint64_t)x_stride * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kPK, (cuuint32_t)kPM};
    if (enc(&amap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(x), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const int32_t nk = (hidden + kPKS - 1) / kPKS;
  const int64_t m_tiles = (n_rows + kPM - 1) / kPM;
  // wide tiles once they alone fill most of the GPU
  const bool wide = m_tiles * ((out_cols + 159) / 160) >= (int64_t)device_sm_count() * 3 / 4;
  auto run = [&](auto kernel, int bn, size_t smem, PerDevice &smem_attr) -> cudaError_t {
    CUtensorMap bmap;
    const cuuint64_t dims[2] = {(cuuint64_t)hidden, (cuuint64_t)out_cols};
    const cuuint64_t strides[1] = {(cuuint64_t)hidden * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kPK, (cuuint32_t)bn};
    if (enc(&bmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(w), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    const cudaError_t e = set_smem_once(smem_attr, kernel, smem);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)((out_cols + bn - 1) / bn), (unsigned)m_tiles);
    return launch_dependent(kernel, grid, dim3(kPThreads), smem, stream, 1u, amap, bmap, y, y_stride,
                            n_rows, out_cols, nk, status);
  };
  static PerDevice set80, set160;
  if (wide) return run(proj_kernel<160>, 160, proj_smem<160>(), set160);
  return run(proj_kernel<80>, 80, proj_smem<80>(), set80);
}

}  // namespace qsa
