// Stable counting sort by bucket of one head's elements, run by the CTAs of one
// thread-block cluster (FAST-AR technical summary §2.C: the bucket-grouped, block-sparse
// layout of the restricted attention).
//
// CTA c of the cluster owns the c-th contiguous chunk of the element range and, inside
// it, each warp a contiguous segment.  Pass 1 builds per-warp histograms (shared-memory
// atomic adds).  The CTA's histogram
// sits in its shared memory; after a cluster barrier every CTA reads all of the
// cluster's histograms through distributed shared memory, which gives per bucket the
// total (the bucket offsets) and the count in the chunks before its own.  Pass 2 replays
// the chunk and scatters each element to bucket offset + earlier chunks + earlier warps +
// its rank among same-bucket lanes of the batch, so the order inside a bucket is
// ascending element id.  Every thread of every CTA of the cluster must call it (it holds
// two cluster barriers).
#pragma once

#include <cooperative_groups.h>

#include "common.cuh"

namespace fastar {

constexpr int kSortCtas = 8;
constexpr int kSortWarpsC = 8;
constexpr int kSortStage = 8192;   // ids of a chunk staged in shared memory when they fit

struct SortSmem {
  int cnt[kSortWarpsC][FASTAR_MAX_B];
  int hist[FASTAR_MAX_B];
  int base[FASTAR_MAX_B];
  int wsum[kSortWarpsC];
  int ids_s[kSortStage];
};

// id[0..E): the elements' buckets.  Writes out[0..E) (element ids in bucket order),
// offsets[0..B] (first position of each bucket, offsets[B] = E; by the cluster's CTA 0)
// and, when where is not null, where[e] = the sorted position of element e.  Ids outside
// [0, B) are skipped and flag FASTAR_DEV_BAD_BUCKET.
__device__ __forceinline__ void cluster_counting_sort(SortSmem& sm, const int32_t* __restrict__ id, int64_t E,
                                                      int B, int32_t* __restrict__ out,
                                                      int32_t* __restrict__ offsets, int32_t* __restrict__ where,
                                                      int32_t* status) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  const int c = (int)cluster.block_rank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, t = threadIdx.x;
  const int64_t per = (E + kSortCtas - 1) / kSortCtas;
  const int64_t cb = (int64_t)c * per < E ? (int64_t)c * per : E;
  const int64_t ce = cb + per < E ? cb + per : E;
  for (int i = t; i < kSortWarpsC * FASTAR_MAX_B; i += blockDim.x) (&sm.cnt[0][0])[i] = 0;
  const bool staged = ce - cb <= kSortStage;
  if (staged)
    for (int64_t e = cb + t; e < ce; e += blockDim.x) sm.ids_s[e - cb] = id[e];
  __syncthreads();
  auto bucket_of = [&](int64_t e) -> int { return staged ? sm.ids_s[e - cb] : id[e]; };
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
    if (b >= 0) atomicAdd(&sm.cnt[warp][b], 1);   // counts only: the order of the adds is immaterial
  }
  __syncthreads();
  if (t < B) {
    int sum = 0;
#pragma unroll
    for (int w = 0; w < kSortWarpsC; ++w) sum += sm.cnt[w][t];
    sm.hist[t] = sum;
  }
  cluster.sync();   // every CTA's histogram is complete
  int total = 0, before = 0;
  if (t < B) {
    for (int k = 0; k < kSortCtas; ++k) {
      const int v = cluster.map_shared_rank(sm.hist, k)[t];
      total += v;
      if (k < c) before += v;
    }
  }
  cluster.sync();   // no CTA overwrites (or leaves) its histogram while another may still read it
  // exclusive scan of the bucket totals (B <= blockDim.x)
  int incl = total;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sm.wsum[warp] = incl;
  __syncthreads();
  int wpre = 0;
  for (int w = 0; w < warp; ++w) wpre += sm.wsum[w];
  const int off = wpre + incl - total;
  if (t < B) {
    sm.base[t] = off + before;
    if (c == 0) offsets[t] = off;
  }
  if (c == 0 && t == B - 1) offsets[B] = off + total;
  __syncthreads();
  if (t < B) {
    int acc = sm.base[t];
#pragma unroll
    for (int w = 0; w < kSortWarpsC; ++w) {
      const int x = sm.cnt[w][t];
      sm.cnt[w][t] = acc;
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
    if (b >= 0) start = sm.cnt[warp][b];
    __syncwarp();
    if (b >= 0) {
      const int dst = start + __popc(peers & ((1u << lane) - 1u));
      out[dst] = (int32_t)e;
      if (where) where[e] = dst;
      if (lane == __ffs(peers) - 1) sm.cnt[warp][b] = start + __popc(peers);
    }
    __syncwarp();
  }
  __syncthreads();   // the staged ids and counts may be reused by the caller's next phase
}

}  // namespace fastar
