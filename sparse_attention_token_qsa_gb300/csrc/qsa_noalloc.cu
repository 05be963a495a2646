// qsa_score_rows_noalloc: the tensor-core scorer with a built-in workspace.
//
// The pages have no counterpart to this entry point.  It exists for callers
// that cannot allocate device memory at the point where they score rows:
// serving engines that hand every free byte of HBM to their KV cache at start
// and forbid allocation afterwards, code running where the CUDA allocator may
// not be called (a host callback, for one), and real-time loops that cannot
// take the allocator's latency, or its failure, in the middle of a step.
// Everything qsa_score_rows asks of a caller-provided workspace is served by a
// file-scope device array instead; the caller still passes every input and
// output buffer.
//
// The array is QSA_NOALLOC_MAX_ROWS * 1024 bytes (8 MiB) and every GPU that
// loads this library holds it until the process exits.  Calls are limited to
// QSA_NOALLOC_MAX_ROWS rows; larger calls are refused before any launch.
// Every call shares the one array: its contents persist from the last call,
// but the query-prep kernel overwrites every vector a call reads, so nothing
// has to start at zero.  Calls whose kernels overlap on the GPU (different
// streams, or different host threads on one device, without ordering between
// them) race on the array.
//
// The array's device address belongs to the CUDA context that loaded this
// module.  A device reset (cudaDeviceReset, or the primary context released
// and created again) loads the module anew, possibly elsewhere, so the address
// is looked up once per device and context: each call compares the current
// context's ID with the one the address was looked up under and looks it up
// again when they differ (or when the ID cannot be read).
#include <mutex>

#include <cuda.h>  // CUcontext (the two driver calls come through the runtime)
#include <cuda_runtime.h>

#include "../../include/qsa.h"

namespace {

constexpr int64_t kNoAllocBytes = (int64_t)QSA_NOALLOC_MAX_ROWS * 4 * 128 * 2;

// The workspace itself.  In host code this name is only a host-side stand-in
// for the device object, never a device address: kernels get the address that
// cudaGetSymbolAddress returns for the current device.
static __device__ __align__(256) unsigned char g_noalloc_ws[kNoAllocBytes];

constexpr int kMaxDevices = 64;

struct WsAddr {
  void *addr;                  // the array's device address ...
  unsigned long long ctx_id;   // ... in the context with this ID (0: unknown)
};
std::mutex g_mu;
WsAddr g_ws[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

// The ID of the calling thread's current context (unique per context the
// driver creates, never reused), or 0 if it cannot be read.
unsigned long long current_context_id() {
  struct Calls {
    CtxGetCurrentFn get_current;
    CtxGetIdFn get_id;
  };
  static const Calls calls = []() -> Calls {
    void *a = nullptr, *b = nullptr;
    cudaDriverEntryPointQueryResult qa, qb;
    const bool ok =
        cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) ==
            cudaSuccess &&
        qa == cudaDriverEntryPointSuccess &&
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) ==
            cudaSuccess &&
        qb == cudaDriverEntryPointSuccess;
    if (!ok) {
      cudaGetLastError();
      return Calls{nullptr, nullptr};
    }
    return Calls{reinterpret_cast<CtxGetCurrentFn>(a), reinterpret_cast<CtxGetIdFn>(b)};
  }();
  if (calls.get_current == nullptr) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (calls.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
      calls.get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Set-up, once per device and context, with that device current: look up the
// array's device address (cudaGetSymbolAddress also makes the device's
// primary context current on this thread).  Returns nullptr if the lookup
// fails.
void *workspace_for_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  const unsigned long long id = current_context_id();
  if (g_ws[dev].addr == nullptr || id == 0 || id != g_ws[dev].ctx_id) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_ws) != cudaSuccess) {
      cudaGetLastError();  // leave no sticky error behind
      g_ws[dev] = WsAddr{nullptr, 0};
      return nullptr;
    }
    g_ws[dev] = WsAddr{p, current_context_id()};
  }
  return g_ws[dev].addr;
}

}  // namespace

extern "C" qsa_status qsa_score_rows_noalloc(const uint16_t *q, int64_t q_stride,
                                             const int32_t *pos, const int32_t *visible_len,
                                             int32_t n_rows, int32_t tokens,
                                             const uint16_t *q_norm_w, const uint16_t *cos_t,
                                             const uint16_t *sin_t, int32_t table_rows, float eps,
                                             const uint16_t *block_keys, float *scores,
                                             int64_t score_cols, int32_t *dev_status,
                                             void *stream) {
  if (n_rows < 0 || n_rows > QSA_NOALLOC_MAX_ROWS) return QSA_ERR_INVALID_VALUE;
  if (n_rows == 0 || tokens == 0)  // an empty launch needs no workspace either
    return qsa_score_rows_with(q, q_stride, pos, visible_len, n_rows, tokens, q_norm_w, cos_t,
                               sin_t, table_rows, eps, block_keys, nullptr, scores, score_cols,
                               dev_status, QSA_SCORE_TCGEN05, nullptr, 0, stream);
  void *ws = workspace_for_current_device();
  if (ws == nullptr) return QSA_ERR_LAUNCH;
  return qsa_score_rows_with(q, q_stride, pos, visible_len, n_rows, tokens, q_norm_w, cos_t, sin_t,
                             table_rows, eps, block_keys, nullptr, scores, score_cols, dev_status,
                             QSA_SCORE_TCGEN05, ws, kNoAllocBytes, stream);
}
