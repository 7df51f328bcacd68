// AnnCA prompt selection for callers that cannot allocate device memory.
//
// fastar_annca_select needs a scratch array for the per-token scores whenever the
// caller does not want them back, and asks the caller to allocate it.  Some callers
// cannot do that at the point where they run the step: a serving process that
// reserves all of its device memory up front and forbids later allocations, code
// that runs under a fixed memory budget shared with other tenants, or a host thread
// on a latency-critical path where cudaMalloc may block or synchronise the device.
// This variant keeps its scratch in a fixed array that lives in the library's own
// device image instead, so a call needs no allocation at all.
//
// Limits and rules:
//   * the scratch holds FASTAR_NOALLOC_MAX_SCORES floats (1 MiB); calls with
//     H * F * P above that are rejected with FASTAR_ECAPACITY;
//   * every GPU that loads the library holds the array until the process exits;
//   * the array's device address is looked up once per device, on the first call
//     made with that device current; make that first call before any stream
//     capture begins;
//   * all calls share the one array and it keeps the last call's contents.  Every
//     score the ranking reads is written earlier in the same call, so nothing needs
//     clearing, but two calls whose work overlaps on the GPU (different streams,
//     no ordering between them) race on the array: order them.
#include <mutex>

#include "fastar.h"
#include "kernels.h"

namespace fastar {
namespace {

static __device__ __align__(256) float g_annca_scratch[FASTAR_NOALLOC_MAX_SCORES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
float* g_scratch_addr[kMaxDevices] = {};

// The device address of g_annca_scratch on the current device (looked up once).
int scratch_for_current_device(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FASTAR_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return FASTAR_EUNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_annca_scratch) != cudaSuccess || !p) return FASTAR_ECUDA;
    g_scratch_addr[dev] = static_cast<float*>(p);
  }
  *out = g_scratch_addr[dev];
  return FASTAR_OK;
}

}  // namespace
}  // namespace fastar

extern "C" int fastar_annca_select_noalloc(const void* q, int dtype, int H, int F, int64_t tpf, int d,
                                           int64_t q_head_stride, int64_t q_token_stride, const int32_t* qb,
                                           int r, const void* kp, const int32_t* pb, int64_t P, float tau_ca,
                                           int topk, int gate, uint8_t* keep, int32_t* kidx, int32_t* kcnt,
                                           cudaStream_t stream) {
  if (H < 0 || F < 0 || P < 0) return FASTAR_EINVAL;
  if ((int64_t)H * F * P > FASTAR_NOALLOC_MAX_SCORES) return FASTAR_ECAPACITY;
  if (H == 0 || F == 0) return FASTAR_OK;
  float* scratch = nullptr;
  const int rc = fastar::scratch_for_current_device(&scratch);
  if (rc != FASTAR_OK) return rc;
  // the scores land in the fixed scratch array, which is passed as the (otherwise
  // caller-owned) score output of the regular entry point
  return fastar_annca_select(q, dtype, H, F, tpf, d, q_head_stride, q_token_stride, qb, r, kp, pb, P, tau_ca,
                             topk, gate, 0, nullptr, nullptr, nullptr, keep, kidx, kcnt, scratch, nullptr, nullptr, nullptr,
                             nullptr, 0, stream);
}
