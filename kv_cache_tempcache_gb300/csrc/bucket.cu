// ANN bucket assignment (argmax / top-r over per-head unit centroids) and the
// stable counting sort that groups tokens by bucket.
//
// FAST-AR technical summary §2.C (AnnSA: tokens assigned to ANN buckets; each
// query restricted to the keys of its own bucket(s)) and §2.B (AnnCA shares the
// buckets).  The centroid-argmax ANN is the method spec's fixed choice.
#include <climits>

#include <cooperative_groups.h>

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
                                    int B, int r, int32_t* qb, int32_t* kb, float* knorm, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  if (dtype == FASTAR_BF16 && launch_assign_qk_tc(d, q, k, H, n, cent, B, r, qb, kb, knorm, s))
    return cudaGetLastError();
  // otherwise the two assignments one after the other
  cudaError_t e = launch_bucket_assign(dtype, d, q, H, n, cent, B, r, qb, nullptr, nullptr, s);
  if (e != cudaSuccess) return e;
  return launch_bucket_assign(dtype, d, k, H, n, cent, B, 1, kb, nullptr, knorm, s);
}

// ---------------------------------------------------------------------------------------
// Stable counting sort: one thread-block cluster of kSortCtas CTAs per head.
// CTA c of the cluster owns the c-th contiguous chunk of the head's element range and,
// inside it, each warp a contiguous segment.  Pass 1 builds per-warp histograms (a
// warp-level match gives each bucket one leader per batch of 32 elements).  The CTA's
// histogram sits in its shared memory; after a cluster barrier every CTA reads all of
// the cluster's histograms through distributed shared memory, which gives per bucket
// the total (the bucket offsets) and the count in the chunks before its own.  Pass 2
// replays the chunk and scatters each element to bucket offset + earlier chunks +
// earlier warps + its rank among same-bucket lanes of the batch, so the order inside
// a bucket is ascending element id.  Optionally each element's sorted position is written
// too (the inverse permutation).  The CTAs of a cluster are co-scheduled by the
// hardware and every thread executes both cluster barriers unconditionally.
// ---------------------------------------------------------------------------------------
constexpr int kSortCtas = 8;
constexpr int kSortWarpsC = 8;
constexpr int kSortStage = 8192;   // ids of a chunk staged in shared memory when they fit

__global__ void __cluster_dims__(kSortCtas, 1, 1) __launch_bounds__(kSortWarpsC * 32)
bucket_sort_kernel(const int32_t* __restrict__ ids, int64_t n, int r, int B, const int32_t* __restrict__ n_valid,
                   int32_t* __restrict__ perm, int32_t* __restrict__ offsets, int32_t* __restrict__ inv,
                   int32_t* status) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  __shared__ int cnt[kSortWarpsC][FASTAR_MAX_B];
  __shared__ int hist[FASTAR_MAX_B];
  __shared__ int base[FASTAR_MAX_B];
  __shared__ int wsum[kSortWarpsC];
  __shared__ int ids_s[kSortStage];
  const int c = (int)cluster.block_rank();
  const int h = blockIdx.x / kSortCtas;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, t = threadIdx.x;
  int64_t nv = n;
  if (n_valid) {
    nv = n_valid[h];
    if (nv < 0 || nv > n) {
      if (t == 0 && c == 0) flag_status(status, FASTAR_DEV_BAD_LEN);
      nv = nv < 0 ? 0 : n;
    }
  }
  const int64_t E = nv * r;
  const int64_t per = (E + kSortCtas - 1) / kSortCtas;
  const int64_t cb = (int64_t)c * per < E ? (int64_t)c * per : E;
  const int64_t ce = cb + per < E ? cb + per : E;
  const int32_t* id = ids + (int64_t)h * n * r;
  int32_t* out = perm + (int64_t)h * n * r;
  int32_t* where = inv ? inv + (int64_t)h * n * r : nullptr;   // element -> its sorted position
  for (int i = t; i < kSortWarpsC * FASTAR_MAX_B; i += blockDim.x) (&cnt[0][0])[i] = 0;
  const bool staged = ce - cb <= kSortStage;
  if (staged)
    for (int64_t e = cb + t; e < ce; e += blockDim.x) ids_s[e - cb] = id[e];
  __syncthreads();
  auto bucket_of = [&](int64_t e) -> int { return staged ? ids_s[e - cb] : id[e]; };
  const int64_t wseg = (ce - cb + kSortWarpsC - 1) / kSortWarpsC;
  const int64_t wb = cb + warp * wseg < ce ? cb + warp * wseg : ce;
  const int64_t we = wb + wseg < ce ? wb + wseg : ce;
  for (int64_t bse = wb; bse < we; bse += 32) {
    const int64_t e = bse + lane;
    int b = e < we ? bucket_of(e) : -1;
    if (e < we && (b < 0 || b >= B)) {
      flag_status(status, FASTAR_DEV_BAD_BUCKET);
      b = -1;
    }
    const unsigned peers = __match_any_sync(0xffffffffu, b);
    if (b >= 0 && lane == __ffs(peers) - 1) cnt[warp][b] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  if (t < B) {
    int sum = 0;
#pragma unroll
    for (int w = 0; w < kSortWarpsC; ++w) sum += cnt[w][t];
    hist[t] = sum;
  }
  cluster.sync();   // every CTA's histogram is complete
  int total = 0, before = 0;
  if (t < B) {
    for (int k = 0; k < kSortCtas; ++k) {
      const int v = cluster.map_shared_rank(hist, k)[t];
      total += v;
      if (k < c) before += v;
    }
  }
  cluster.sync();   // no CTA leaves (its histogram) while another may still read it
  // exclusive scan of the bucket totals (B <= blockDim.x)
  int incl = total;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  int wpre = 0;
  for (int w = 0; w < warp; ++w) wpre += wsum[w];
  const int off = wpre + incl - total;
  if (t < B) {
    base[t] = off + before;
    if (c == 0) offsets[(int64_t)h * (B + 1) + t] = off;
  }
  if (c == 0 && t == B - 1) offsets[(int64_t)h * (B + 1) + B] = off + total;
  __syncthreads();
  if (t < B) {
    int acc = base[t];
#pragma unroll
    for (int w = 0; w < kSortWarpsC; ++w) {
      const int x = cnt[w][t];
      cnt[w][t] = acc;
      acc += x;
    }
  }
  __syncthreads();
  for (int64_t bse = wb; bse < we; bse += 32) {
    const int64_t e = bse + lane;
    int b = e < we ? bucket_of(e) : -1;
    if (b >= B || b < -1) b = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, b);
    int start = 0;
    if (b >= 0) start = cnt[warp][b];
    __syncwarp();
    if (b >= 0) {
      const int dst = start + __popc(peers & ((1u << lane) - 1u));
      out[dst] = (int32_t)e;
      if (where) where[e] = dst;
      if (lane == __ffs(peers) - 1) cnt[warp][b] = start + __popc(peers);
    }
    __syncwarp();
  }
}

cudaError_t launch_bucket_sort(const int32_t* ids, int H, int64_t n, int r, int B,
                               const int32_t* n_valid, int32_t* perm, int32_t* offsets,
                               int32_t* status, cudaStream_t s, int32_t* inv) {
  bucket_sort_kernel<<<H * kSortCtas, kSortWarpsC * 32, 0, s>>>(ids, n, r, B, n_valid, perm, offsets, inv, status);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace fastar
