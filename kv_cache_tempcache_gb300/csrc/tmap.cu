// Host-side TMA tensor-map encoding (driver entry point looked up through the runtime,
// so the library does not link libcuda directly).
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "tmap.h"

namespace fastar {

namespace {
using EncodeFn = decltype(&cuTensorMapEncodeTiled);

EncodeFn encode_fn() {
  static EncodeFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeFn>(nullptr);
    return reinterpret_cast<EncodeFn>(p);
  }();
  return fn;
}
}  // namespace

bool make_tmap_bf16_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                       uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0, uint32_t box1,
                       uint32_t box2) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {d0, d1, d2 > 0 ? d2 : 1};
  cuuint64_t strides[2] = {stride1_bytes, stride2_bytes > 0 ? stride2_bytes : stride1_bytes * d1};
  cuuint32_t box[3] = {box0, box1, box2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {
constexpr int kMaxDevices = 64;
constexpr int kMaxOptIns = 512;
std::mutex g_dev_mutex;
std::atomic<int> g_sms[kMaxDevices];
struct OptIn {
  const void* func;
  int dev, bytes;
};
OptIn g_opt_in[kMaxOptIns];   // a fixed table: set-up allocates nothing, not even on the host
int g_n_opt_in = 0;
}  // namespace

int sm_count() {
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  const int cached = g_sms[dev].load(std::memory_order_relaxed);
  if (cached > 0) return cached;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) return 148;
  g_sms[dev].store(v, std::memory_order_relaxed);
  return v;
}

cudaError_t opt_in_smem(const void* func, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  for (int i = 0; i < g_n_opt_in; ++i)
    if (g_opt_in[i].func == func && g_opt_in[i].dev == dev && g_opt_in[i].bytes >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  if (g_n_opt_in < kMaxOptIns) g_opt_in[g_n_opt_in++] = OptIn{func, dev, bytes};   // else: set again next time
  return cudaSuccess;
}

}  // namespace fastar
