// ANN bucket assignment (argmax / top-r over per-head unit centroids) and the
// stable counting sort that groups tokens by bucket.
//
// FAST-AR technical summary §2.C (AnnSA: tokens assigned to ANN buckets; each
// query restricted to the keys of its own bucket(s)) and §2.B (AnnCA shares the
// buckets).  The centroid-argmax ANN is the method spec's fixed choice.
#include <climits>

#include "common.cuh"
#include "kernels.h"

namespace fastar {

constexpr int kAssignWarps = 8;

// One warp per token row.  Centroids of the head are staged transposed in shared
// memory ([d][Bp], Bp = B rounded up to 32) so lane c reads centroid c without bank
// conflicts; the token row is broadcast from a per-warp staging row.  Scores are
// exact fp32 FMA chains over c = 0..d-1.
template <typename T, int D>
__global__ void __launch_bounds__(kAssignWarps * 32)
bucket_assign_kernel(const T* __restrict__ x, int64_t hs, int64_t ts, int64_t n,
                     const T* __restrict__ cent, int B, int r, int32_t* __restrict__ ids,
                     float* __restrict__ scores, float* __restrict__ norms) {
  extern __shared__ float smem[];
  const int Bp = (B + 31) & ~31;
  float* ct = smem;                 // [D][Bp]
  float* xs = smem + D * Bp;        // [warps][D]
  const int h = blockIdx.y;
  for (int idx = threadIdx.x; idx < Bp * D; idx += blockDim.x) {
    const int c = idx / D, k = idx - c * D;
    ct[k * Bp + c] = c < B ? to_f(cent[((int64_t)h * B + c) * D + k]) : 0.f;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nc = Bp >> 5;
  float* xrow = xs + warp * D;
  for (int64_t t = (int64_t)blockIdx.x * kAssignWarps + warp; t < n;
       t += (int64_t)gridDim.x * kAssignWarps) {
    const T* row = x + h * hs + t * ts;
    float ss = 0.f;
    for (int k = lane; k < D; k += 32) {
      const float v = to_f(row[k]);
      xrow[k] = v;
      ss = fmaf(v, v, ss);
    }
    ss = warp_sum(ss);
    __syncwarp();
    float acc[FASTAR_MAX_B / 32];
#pragma unroll
    for (int c = 0; c < FASTAR_MAX_B / 32; ++c) acc[c] = 0.f;
#pragma unroll 4
    for (int k = 0; k < D; ++k) {
      const float xv = xrow[k];
      const float* crow = ct + k * Bp + lane;
#pragma unroll
      for (int c = 0; c < FASTAR_MAX_B / 32; ++c)
        if (c < nc) acc[c] = fmaf(xv, crow[c * 32], acc[c]);
    }
    unsigned taken = 0;
    for (int s = 0; s < r; ++s) {
      float bv = neg_inf();
      int bi = INT_MAX;
#pragma unroll
      for (int c = 0; c < FASTAR_MAX_B / 32; ++c) {
        const int idx = c * 32 + lane;
        if (c < nc && idx < B && !((taken >> c) & 1u) && beats(acc[c], idx, bv, bi)) {
          bv = acc[c];
          bi = idx;
        }
      }
      warp_argmax(bv, bi);
      if (lane == 0) {
        ids[(h * n + t) * r + s] = bi;
        if (scores) scores[(h * n + t) * r + s] = bv;
      }
      if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    }
    if (norms && lane == 0) norms[h * n + t] = sqrtf(ss);
    __syncwarp();
  }
}

template <typename T, int D>
static cudaError_t assign_impl(TokView x, int H, int64_t n, const void* cent, int B, int r,
                               int32_t* ids, float* scores, float* norms, cudaStream_t s) {
  const int Bp = (B + 31) & ~31;
  const size_t smem = sizeof(float) * ((size_t)D * Bp + (size_t)kAssignWarps * D);
  auto kern = bucket_assign_kernel<T, D>;
  // opt in once to the largest footprint (B = FASTAR_MAX_B); no per-launch attribute calls
  static const cudaError_t attr = cudaFuncSetAttribute(
      kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
      (int)(sizeof(float) * ((size_t)D * FASTAR_MAX_B + (size_t)kAssignWarps * D)));
  if (attr != cudaSuccess) return attr;
  int64_t gx = (n + kAssignWarps - 1) / kAssignWarps;
  const int64_t cap = (4 * 152 + H - 1) / H;
  if (gx > cap) gx = cap;
  if (gx < 1) gx = 1;
  kern<<<dim3((unsigned)gx, H), kAssignWarps * 32, smem, s>>>(
      static_cast<const T*>(x.p), x.hs, x.ts, n, static_cast<const T*>(cent), B, r, ids, scores, norms);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_bucket_assign(int dtype, int d, TokView x, int H, int64_t n, const void* cent,
                                 int B, int r, int32_t* ids, float* scores, float* norms,
                                 cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  if (dtype == FASTAR_BF16) {
    // tensor cores (the SIMT kernel below only if the set-up is refused)
    if (launch_assign_tc(d, x, H, n, cent, B, r, ids, scores, norms, s)) return cudaGetLastError();
    if (d == 128) return assign_impl<__nv_bfloat16, 128>(x, H, n, cent, B, r, ids, scores, norms, s);
    return assign_impl<__nv_bfloat16, 64>(x, H, n, cent, B, r, ids, scores, norms, s);
  }
  if (d == 128) return assign_impl<float, 128>(x, H, n, cent, B, r, ids, scores, norms, s);
  return assign_impl<float, 64>(x, H, n, cent, B, r, ids, scores, norms, s);
}

// ---------------------------------------------------------------------------------------
// Stable counting sort, one CTA per head.
// Each warp owns a contiguous segment of the element range.  Pass 1 builds a
// per-warp histogram (warp-level match gives each bucket one leader per batch of
// 32 elements); an exclusive scan over (bucket, warp) then gives every warp its
// first position in every bucket; pass 2 replays the segment and scatters each
// element to start + its rank among same-bucket lanes of the batch.  Element order
// inside a bucket is therefore ascending element id.  No block waits on another.
// ---------------------------------------------------------------------------------------
constexpr int kSortWarps = 32;

__global__ void __launch_bounds__(kSortWarps * 32)
bucket_sort_kernel(const int32_t* __restrict__ ids, int64_t n, int r, int B,
                   const int32_t* __restrict__ n_valid, int32_t* __restrict__ perm,
                   int32_t* __restrict__ offsets, int32_t* status, int stage) {
  extern __shared__ int sm_sort[];
  int* cnt = sm_sort;               // [kSortWarps][B]
  int* tot = sm_sort + kSortWarps * B;  // [B + 1]
  const int h = blockIdx.x;
  int64_t nv = n;
  if (n_valid) {
    nv = n_valid[h];
    if (nv < 0 || nv > n) {
      if (threadIdx.x == 0) flag_status(status, FASTAR_DEV_BAD_LEN);
      nv = nv < 0 ? 0 : n;
    }
  }
  const int64_t E = nv * r;
  const int32_t* id = ids + (int64_t)h * n * r;
  int32_t* out = perm + (int64_t)h * n * r;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < kSortWarps * B; i += blockDim.x) cnt[i] = 0;
  if (stage) {
    // both passes read the ids: stage them once, coalesced, in shared memory
    int* ids_s = tot + ((B + 1 + 3) & ~3);
    for (int64_t e = threadIdx.x; e < E; e += blockDim.x) ids_s[e] = id[e];
    id = ids_s;
  }
  __syncthreads();
  const int64_t seg = (E + kSortWarps - 1) / kSortWarps;
  const int64_t beg = warp * seg;
  const int64_t end = beg + seg < E ? beg + seg : E;
  for (int64_t base = beg; base < end; base += 32) {
    const int64_t e = base + lane;
    int b = e < end ? id[e] : -1;
    if (e < end && (b < 0 || b >= B)) {
      flag_status(status, FASTAR_DEV_BAD_BUCKET);
      b = -1;
    }
    const unsigned peers = __match_any_sync(0xffffffffu, b);
    if (b >= 0 && lane == __ffs(peers) - 1) cnt[warp * B + b] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    int s = 0;
    for (int w = 0; w < kSortWarps; ++w) s += cnt[w * B + b];
    tot[b] = s;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int b = 0; b < B; ++b) {
      const int t = tot[b];
      tot[b] = acc;
      acc += t;
    }
    tot[B] = acc;
  }
  __syncthreads();
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    int acc = tot[b];
    for (int w = 0; w < kSortWarps; ++w) {
      const int t = cnt[w * B + b];
      cnt[w * B + b] = acc;
      acc += t;
    }
  }
  for (int b = threadIdx.x; b <= B; b += blockDim.x) offsets[(int64_t)h * (B + 1) + b] = tot[b];
  __syncthreads();
  for (int64_t base = beg; base < end; base += 32) {
    const int64_t e = base + lane;
    int b = e < end ? id[e] : -1;
    if (b >= B) b = -1;
    if (b < -1) b = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, b);
    int start = 0;
    if (b >= 0) start = cnt[warp * B + b];
    __syncwarp();
    if (b >= 0) {
      out[start + __popc(peers & ((1u << lane) - 1u))] = (int32_t)e;
      if (lane == __ffs(peers) - 1) cnt[warp * B + b] = start + __popc(peers);
    }
    __syncwarp();
  }
}

cudaError_t launch_bucket_sort(const int32_t* ids, int H, int64_t n, int r, int B,
                               const int32_t* n_valid, int32_t* perm, int32_t* offsets,
                               int32_t* status, cudaStream_t s) {
  // histograms (<= 33.8 KB) plus, when they fit, the head's ids staged in shared memory
  const size_t base = sizeof(int) * ((size_t)kSortWarps * B + ((B + 1 + 3) & ~3));
  const size_t staged = base + sizeof(int) * (size_t)(n * r);
  constexpr size_t kMaxSmem = 200 * 1024;
  static const cudaError_t attr =
      cudaFuncSetAttribute(bucket_sort_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxSmem);
  const int stage = (attr == cudaSuccess && staged <= kMaxSmem) ? 1 : 0;
  bucket_sort_kernel<<<H, kSortWarps * 32, stage ? staged : base, s>>>(ids, n, r, B, n_valid, perm, offsets,
                                                                         status, stage);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace fastar
