// ANN bucket assignment (argmax / top-r over per-head unit centroids) and the
// stable counting sort that groups tokens by bucket.
//
// FAST-AR technical summary §2.C (AnnSA: tokens assigned to ANN buckets; each
// query restricted to the keys of its own bucket(s)) and §2.B (AnnCA shares the
// buckets).  The centroid-argmax ANN is the method spec's fixed choice.
#include <climits>

#include "cluster_sort.cuh"
#include "common.cuh"
#include "kernels.h"
#include "tmap.h"

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
  // opt in to the largest footprint (B = FASTAR_MAX_B), once per device
  const cudaError_t attr = opt_in_smem(
      (const void*)kern, (int)(sizeof(float) * ((size_t)D * FASTAR_MAX_B + (size_t)kAssignWarps * D)));
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

cudaError_t launch_bucket_assign_qk(int dtype, int d, TokView q, TokView k, int H, int64_t n, const void* cent,
                                    int B, int r, int32_t* qb, int32_t* kb, float* knorm, float* qnorm,
                                    cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  if (dtype == FASTAR_BF16 && launch_assign_qk_tc(d, q, k, H, n, cent, B, r, qb, kb, knorm, qnorm, s))
    return cudaGetLastError();
  // otherwise the two assignments one after the other
  cudaError_t e = launch_bucket_assign(dtype, d, q, H, n, cent, B, r, qb, nullptr, qnorm, s);
  if (e != cudaSuccess) return e;
  return launch_bucket_assign(dtype, d, k, H, n, cent, B, 1, kb, nullptr, knorm, s);
}

// ---------------------------------------------------------------------------------------
// Stable counting sort: one thread-block cluster of kSortCtas CTAs per head (the body is
// cluster_counting_sort in cluster_sort.cuh, shared with the compaction's plan kernel).
// ---------------------------------------------------------------------------------------
__global__ void __cluster_dims__(kSortCtas, 1, 1) __launch_bounds__(kSortWarpsC * 32)
bucket_sort_kernel(const int32_t* __restrict__ ids, int64_t n, int r, int B, const int32_t* __restrict__ n_valid,
                   int32_t* __restrict__ perm, int32_t* __restrict__ offsets, int32_t* __restrict__ inv,
                   int32_t* status) {
  __shared__ SortSmem sm;
  const int h = blockIdx.x / kSortCtas;
  int64_t nv = n;
  if (n_valid) {
    nv = n_valid[h];
    if (nv < 0 || nv > n) {
      if (threadIdx.x == 0 && blockIdx.x % kSortCtas == 0) flag_status(status, FASTAR_DEV_BAD_LEN);
      nv = nv < 0 ? 0 : n;
    }
  }
  cluster_counting_sort(sm, ids + (int64_t)h * n * r, nv * r, B, perm + (int64_t)h * n * r,
                        offsets + (int64_t)h * (B + 1), inv ? inv + (int64_t)h * n * r : nullptr, status);
}

cudaError_t launch_bucket_sort(const int32_t* ids, int H, int64_t n, int r, int B,
                               const int32_t* n_valid, int32_t* perm, int32_t* offsets,
                               int32_t* status, cudaStream_t s, int32_t* inv) {
  bucket_sort_kernel<<<H * kSortCtas, kSortWarpsC * 32, 0, s>>>(ids, n, r, B, n_valid, perm, offsets, inv, status);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace fastar
