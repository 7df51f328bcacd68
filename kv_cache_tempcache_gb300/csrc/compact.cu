// TempCache compaction: drop evicted entries, append the current chunk as the most
// recent representatives, keep at most M entries (oldest dropped first).
//
// FAST-AR technical summary §2.A ("bounds the growth of the KV cache") and blog §1
// ("only the most recent representative stays in the cache"); the FIFO hard cap is
// the method spec's.
//
// Two kernels: a one-CTA-per-head scan that writes the slot -> source map and the
// new length, then a bandwidth kernel that moves rows with 16-byte accesses.  The sorted
// form plans with one thread-block cluster per head instead: the survivor scan across
// the cluster's CTAs (chunk totals exchanged through distributed shared memory), the new
// slots' bucket ids, their stable counting sort, and optionally the step's (query, slot)
// pairs' counting sort as well, so that the copy can also write each row to its place in
// a bucket-ordered copy (the layout the bucket-restricted attention reads as contiguous
// tiles) and the step needs no separate sort launch.
//
// The merge variant (technical summary §2.A, Theoretical Basis: Lemma 5.1 — identical
// keys merge exactly when their values are averaged and the logit is shifted by the
// group size) keeps a group count g per entry: an evicted entry j is folded into its
// owner, the lowest current entry i that evicted it, whose value becomes
// (v_i + g_j v_j) / (1 + g_j) and whose count becomes 1 + g_j; i's key stays.  The slot
// order is the replace variant's.
#include "cluster_sort.cuh"
#include "common.cuh"
#include "kernels.h"
#include "tmap.h"

namespace fastar {

constexpr int kScanThreads = 1024;

// Slot s of the new cache takes: survivor number (s + drop) if s + drop < S, else
// current token (s + drop - S); drop = max(0, S + nq - M).
__global__ void __launch_bounds__(kScanThreads)
compact_scan_kernel(int64_t nq, int64_t M, const int32_t* __restrict__ len_in,
                    const uint8_t* __restrict__ evict, int32_t* __restrict__ len_out,
                    int32_t* __restrict__ index_map, int32_t* status) {
  __shared__ int warp_tot[kScanThreads / 32];
  __shared__ int s_total;
  const int h = blockIdx.x;
  int64_t n = len_in[h];
  if (n < 0 || n > M) {
    if (threadIdx.x == 0) flag_status(status, FASTAR_DEV_BAD_LEN);
    n = n < 0 ? 0 : M;
  }
  const uint8_t* e = evict + (int64_t)h * M;
  int32_t* imap = index_map + (int64_t)h * M;
  const int64_t per = (n + kScanThreads - 1) / kScanThreads;
  const int64_t beg = threadIdx.x * per;
  const int64_t end = beg + per < n ? beg + per : n;
  int local = 0;
  for (int64_t j = beg; j < end; ++j) local += e[j] ? 0 : 1;
  // block exclusive scan of the per-thread survivor counts
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int t = warp_tot[lane];
    int ti = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, ti, o);
      if (lane >= o) ti += v;
    }
    warp_tot[lane] = ti - t;
    if (lane == 31) s_total = ti;
  }
  __syncthreads();
  const int64_t S = s_total;
  const int64_t total = S + nq;
  const int64_t drop = total > M ? total - M : 0;
  const int64_t L = total - drop;
  int64_t rank = warp_tot[warp] + incl - local;
  for (int64_t j = beg; j < end; ++j) {
    if (!e[j]) {
      const int64_t slot = rank - drop;
      if (slot >= 0) imap[slot] = (int32_t)j;
      ++rank;
    }
  }
  for (int64_t i = threadIdx.x; i < nq; i += blockDim.x) {
    const int64_t slot = S + i - drop;
    if (slot >= 0) imap[slot] = (int32_t)(n + i);
  }
  for (int64_t s = L + threadIdx.x; s < M; s += blockDim.x) imap[s] = -1;
  if (threadIdx.x == 0) len_out[h] = (int32_t)L;
}

// The sorted compaction's plan, clusters of kSortCtas CTAs (every thread of a cluster's
// CTAs runs every phase of its role, so the cluster barriers always fill).  Per head, one
// cluster runs
//   the survivor scan: slot s takes survivor number (s + drop) if s + drop < S, else current
//   token (s + drop - S), drop = max(0, S + nq - M); writes index_map, len_out and the new
//   slots' bucket ids kbout (the source entry's);
//   then the stable counting sort of kbout over the len_out slots -> kperm, koff, kpos;
// and, when qb is given, a second cluster the stable counting sort of the (query, slot)
// pairs' buckets qb -> qperm, qoff at the same time (clusters 2h and 2h + 1).
__global__ void __cluster_dims__(kSortCtas, 1, 1) __launch_bounds__(kSortWarpsC * 32)
compact_plan_kernel(int64_t nq, int64_t M, const int32_t* __restrict__ len_in, const uint8_t* __restrict__ evict,
                    int32_t* __restrict__ len_out, int32_t* __restrict__ index_map, const int32_t* __restrict__ kcb,
                    const int32_t* __restrict__ kbin, int32_t* __restrict__ kbout, int B, int32_t* __restrict__ kperm,
                    int32_t* __restrict__ koff, int32_t* __restrict__ kpos, const int32_t* __restrict__ qb, int r,
                    int32_t* __restrict__ qperm, int32_t* __restrict__ qoff, int32_t* status) {
  pdl_wait();   // the eviction flags of the match before it in the stream
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  __shared__ SortSmem sm;
  __shared__ int warp_tot[kSortWarpsC];
  __shared__ int cta_tot;
  const int c = (int)cluster.block_rank();
  const int cid = blockIdx.x / kSortCtas;
  const int h = qb ? cid >> 1 : cid;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  constexpr int kT = kSortWarpsC * 32;
  if (qb && (cid & 1)) {   // the pairs' sort, beside the other cluster's scan and key sort
    cluster_counting_sort(sm, qb + (int64_t)h * nq * r, nq * r, B, qperm + (int64_t)h * nq * r,
                          qoff + (int64_t)h * (B + 1), nullptr, status);
    return;
  }
  // ---- survivor scan: CTA c owns a contiguous chunk, each thread a contiguous piece ----
  int64_t n = len_in[h];
  if (n < 0 || n > M) {
    if (t == 0 && c == 0) flag_status(status, FASTAR_DEV_BAD_LEN);
    n = n < 0 ? 0 : M;
  }
  const uint8_t* e = evict + (int64_t)h * M;
  const int64_t cper = (n + kSortCtas - 1) / kSortCtas;
  const int64_t cb = (int64_t)c * cper < n ? (int64_t)c * cper : n;
  const int64_t ce = cb + cper < n ? cb + cper : n;
  const int64_t tper = (ce - cb + kT - 1) / kT;
  const int64_t beg = cb + t * tper < ce ? cb + t * tper : ce;
  const int64_t end = beg + tper < ce ? beg + tper : ce;
  const int32_t* kbi = kbin + (int64_t)h * M;
  // a piece of up to kPre entries has its flags and bucket ids loaded here, all at once,
  // for both passes (longer pieces read them entry by entry)
  constexpr int kPre = 16;
  const bool pre = end - beg <= kPre;
  uint8_t ev[kPre];
  int32_t kbv[kPre];
  int local = 0;
  if (pre) {
#pragma unroll
    for (int k = 0; k < kPre; ++k) {
      ev[k] = 1;
      kbv[k] = 0;
      if (beg + k < end) {
        ev[k] = e[beg + k];
        kbv[k] = kbi[beg + k];
      }
    }
#pragma unroll
    for (int k = 0; k < kPre; ++k) local += ev[k] ? 0 : 1;
  } else {
    for (int64_t j = beg; j < end; ++j) local += e[j] ? 0 : 1;
  }
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  int wpre = 0;
  for (int w = 0; w < warp; ++w) wpre += warp_tot[w];
  if (t == kT - 1) cta_tot = wpre + incl;
  cluster.sync();   // every CTA's survivor count is published
  int64_t S = 0, before = 0;
  for (int k = 0; k < kSortCtas; ++k) {
    const int v = *cluster.map_shared_rank(&cta_tot, k);
    S += v;
    if (k < c) before += v;
  }
  const int64_t total = S + nq;
  const int64_t drop = total > M ? total - M : 0;
  const int64_t L = total - drop;
  int32_t* imap = index_map + (int64_t)h * M;
  int32_t* kbo = kbout + (int64_t)h * M;
  int64_t rank = before + wpre + incl - local;
  if (pre) {
#pragma unroll
    for (int k = 0; k < kPre; ++k) {
      if (!ev[k]) {
        const int64_t slot = rank - drop;
        if (slot >= 0) {
          imap[slot] = (int32_t)(beg + k);
          kbo[slot] = kbv[k];
        }
        ++rank;
      }
    }
  } else {
    for (int64_t j = beg; j < end; ++j) {
      if (!e[j]) {
        const int64_t slot = rank - drop;
        if (slot >= 0) {
          imap[slot] = (int32_t)j;
          kbo[slot] = kbi[j];
        }
        ++rank;
      }
    }
  }
  // the new entries, four per thread and round: their bucket ids loaded before any store
  for (int64_t i0 = (int64_t)c * kT + t; i0 < nq; i0 += 4 * (int64_t)kSortCtas * kT) {
    int32_t b4[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int64_t i = i0 + (int64_t)k * kSortCtas * kT;
      b4[k] = i < nq ? kcb[(int64_t)h * nq + i] : 0;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int64_t i = i0 + (int64_t)k * kSortCtas * kT;
      const int64_t slot = S + i - drop;
      if (i < nq && slot >= 0) {
        imap[slot] = (int32_t)(n + i);
        kbo[slot] = b4[k];
      }
    }
  }
  for (int64_t s2 = L + (int64_t)c * kT + t; s2 < M; s2 += (int64_t)kSortCtas * kT) imap[s2] = -1;
  if (t == 0 && c == 0) len_out[h] = (int32_t)L;
  // the slots' bucket ids are written (global memory, ordered by the barrier's release and
  // acquire) and no CTA reads cta_tot any more
  cluster.sync();
  cluster_counting_sort(sm, kbo, L, B, kperm + (int64_t)h * M, koff + (int64_t)h * (B + 1), kpos + (int64_t)h * M,
                        status);
}

// The group-merge inputs and outputs of the merge variant (all null otherwise).
struct MergeIO {
  const int32_t* top1;    // [H, nq] the match's top-1 cache index per current entry
  const int32_t* owner;   // [H, M] lowest evicting current entry per cached entry, -1 none
  const int32_t* g_in;    // [H, M] incoming group counts
  int32_t* g_out;         // [H, M] outgoing group counts
};

// The bucket-ordered copy written beside the cache (all null otherwise): slot s of head h
// also goes to row kpos[h, s] of ksorted / vsorted.
struct SortedIO {
  const int32_t* kpos;
  void* ksorted;
  void* vsorted;
};

// wa * a + wb * b element-wise over one 16-byte chunk (fp32 arithmetic, rounded once).
template <typename T>
__device__ __forceinline__ uint4 blend16(uint4 a, uint4 b, float wa, float wb) {
  constexpr int N = 16 / (int)sizeof(T);
  const T* x = reinterpret_cast<const T*>(&a);
  const T* y = reinterpret_cast<const T*>(&b);
  uint4 r;
  T* z = reinterpret_cast<T*>(&r);
#pragma unroll
  for (int e = 0; e < N; ++e) z[e] = from_f<T>(fmaf(wa, to_f(x[e]), wb * to_f(y[e])));
  return r;
}

// One 16-byte chunk per thread; VPR chunks per row.  Metadata moves with the row.
template <typename T, int D, bool kMerge>
__global__ void __launch_bounds__(256)
compact_copy_kernel(int H, int64_t nq, int64_t M, const T* __restrict__ kc, const T* __restrict__ vc,
                    int64_t hs, int64_t ts, const float* __restrict__ kcn, const int32_t* __restrict__ kcb,
                    const T* __restrict__ kin, const T* __restrict__ vin, const float* __restrict__ knin,
                    const int32_t* __restrict__ kbin, const int32_t* __restrict__ len_in,
                    const int32_t* __restrict__ len_out, const int32_t* __restrict__ index_map,
                    T* __restrict__ kout, T* __restrict__ vout, float* __restrict__ knout,
                    int32_t* __restrict__ kbout, int32_t* status, const MergeIO mg, const SortedIO so) {
  pdl_wait();   // the index map of the planning kernel before it in the stream
  // grid: (CTAs per head, heads); a head's occupied slots [0, len_out) in 16-byte chunks
  constexpr int VPR = D * (int)sizeof(T) / 16;
  const int h = (int)blockIdx.y;
  int64_t n = len_in[h];
  n = n < 0 ? 0 : (n > M ? M : n);
  int64_t lo = len_out[h];
  lo = lo < 0 ? 0 : (lo > M ? M : lo);
  const int64_t total = lo * VPR;
  for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total;
       g += (int64_t)gridDim.x * blockDim.x) {
    const int64_t slot = g / VPR;
    const int c = (int)(g - slot * VPR);
    const int64_t row = (int64_t)h * M + slot;
    const int64_t src = index_map[row];
    const uint4* ks;
    const uint4* vs;
    float kn;
    int32_t kb;
    int32_t gc = 1;
    int64_t absorb = -1;   // merge variant: the cached entry this current entry owns
    if (src >= 0 && src < n) {
      ks = reinterpret_cast<const uint4*>(kin + ((int64_t)h * M + src) * D) + c;
      vs = reinterpret_cast<const uint4*>(vin + ((int64_t)h * M + src) * D) + c;
      kn = knin[(int64_t)h * M + src];
      kb = kbin[(int64_t)h * M + src];
      if (kMerge) gc = mg.g_in[(int64_t)h * M + src];
    } else if (src >= n && src < n + nq) {
      const int64_t i = src - n;
      ks = reinterpret_cast<const uint4*>(kc + h * hs + i * ts) + c;
      vs = reinterpret_cast<const uint4*>(vc + h * hs + i * ts) + c;
      kn = kcn[(int64_t)h * nq + i];
      kb = kcb[(int64_t)h * nq + i];
      if (kMerge) {
        const int32_t j = mg.top1[(int64_t)h * nq + i];
        if (j >= 0 && j < n && mg.owner[(int64_t)h * M + j] == (int32_t)i) absorb = j;
      }
    } else {
      if (c == 0) flag_status(status, FASTAR_DEV_BAD_INDEX);
      continue;
    }
    // the bucket-ordered row this slot also goes to (null: none)
    uint4* ksd = nullptr;
    uint4* vsd = nullptr;
    if (so.kpos) {
      const int32_t p = so.kpos[row];
      if (p >= 0 && p < M) {
        ksd = reinterpret_cast<uint4*>(static_cast<T*>(so.ksorted) + ((int64_t)h * M + p) * D) + c;
        vsd = reinterpret_cast<uint4*>(static_cast<T*>(so.vsorted) + ((int64_t)h * M + p) * D) + c;
      } else if (c == 0) {
        flag_status(status, FASTAR_DEV_BAD_INDEX);
      }
    }
    const uint4 kr = __ldg(ks);
    reinterpret_cast<uint4*>(kout + row * D)[c] = kr;
    if (ksd) *ksd = kr;
    if (kMerge && absorb >= 0) {
      int32_t gj = mg.g_in[(int64_t)h * M + absorb];
      if (gj < 0) {
        if (c == 0) flag_status(status, FASTAR_DEV_BAD_INDEX);
        gj = 0;
      }
      const float inv = 1.0f / (1.0f + (float)gj);
      const uint4 vj = __ldg(reinterpret_cast<const uint4*>(vin + ((int64_t)h * M + absorb) * D) + c);
      const uint4 vr = blend16<T>(__ldg(vs), vj, inv, (float)gj * inv);
      reinterpret_cast<uint4*>(vout + row * D)[c] = vr;
      if (vsd) *vsd = vr;
      gc = 1 + gj;
    } else {
      const uint4 vr = __ldg(vs);
      reinterpret_cast<uint4*>(vout + row * D)[c] = vr;
      if (vsd) *vsd = vr;
    }
    if (c == 0) {
      knout[row] = kn;
      kbout[row] = kb;
      if (kMerge) mg.g_out[row] = gc;
    }
  }
}

template <typename T, int D>
static cudaError_t copy_impl(int H, int64_t nq, int64_t M, TokView kc, TokView vc, const float* kcn,
                             const int32_t* kcb, const void* kin, const void* vin, const float* knin,
                             const int32_t* kbin, const int32_t* len_in, const int32_t* len_out,
                             const int32_t* imap, void* kout, void* vout, float* knout, int32_t* kbout,
                             int32_t* status, const MergeIO& mg, cudaStream_t s, const SortedIO& so = SortedIO{}) {
  constexpr int VPR = D * (int)sizeof(T) / 16;
  // about 16 CTAs of 256 threads per SM over all heads, each head's CTAs striding its slots
  int64_t blocks = ((int64_t)M * VPR + 255) / 256;
  const int64_t cap = ((int64_t)sm_count() * 16 + H - 1) / H;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  auto kern = mg.g_out ? compact_copy_kernel<T, D, true> : compact_copy_kernel<T, D, false>;
  const cudaError_t e = launch_dependent(
      kern, dim3((unsigned)blocks, (unsigned)H), dim3(256), 0, s, H, nq, M, static_cast<const T*>(kc.p),
      static_cast<const T*>(vc.p), kc.hs, kc.ts, kcn, kcb, static_cast<const T*>(kin), static_cast<const T*>(vin),
      knin, kbin, len_in, len_out, imap, static_cast<T*>(kout), static_cast<T*>(vout), knout, kbout, status, mg,
      so);
  count_launches(1);
  return e;
}

cudaError_t launch_cache_compact(int dtype, int d, int H, int64_t nq, int64_t M, TokView kc,
                                 TokView vc, const float* kcn, const int32_t* kcb, const void* kin,
                                 const void* vin, const float* knin, const int32_t* kbin,
                                 const int32_t* len_in, const uint8_t* evict, void* kout, void* vout,
                                 float* knout, int32_t* kbout, int32_t* len_out, int32_t* imap,
                                 int32_t* status, const int32_t* top1, const int32_t* owner,
                                 const int32_t* g_in, int32_t* g_out, cudaStream_t s) {
  compact_scan_kernel<<<H, kScanThreads, 0, s>>>(nq, M, len_in, evict, len_out, imap, status);
  count_launches(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const MergeIO mg{top1, owner, g_in, g_out};
  if (dtype == FASTAR_BF16) {
    if (d == 128)
      return copy_impl<__nv_bfloat16, 128>(H, nq, M, kc, vc, kcn, kcb, kin, vin, knin, kbin, len_in, len_out, imap,
                                           kout, vout, knout, kbout, status, mg, s);
    return copy_impl<__nv_bfloat16, 64>(H, nq, M, kc, vc, kcn, kcb, kin, vin, knin, kbin, len_in, len_out, imap,
                                        kout, vout, knout, kbout, status, mg, s);
  }
  if (d == 128)
    return copy_impl<float, 128>(H, nq, M, kc, vc, kcn, kcb, kin, vin, knin, kbin, len_in, len_out, imap, kout,
                                 vout, knout, kbout, status, mg, s);
  return copy_impl<float, 64>(H, nq, M, kc, vc, kcn, kcb, kin, vin, knin, kbin, len_in, len_out, imap, kout, vout,
                              knout, kbout, status, mg, s);
}

cudaError_t launch_cache_compact_sorted(int dtype, int d, int H, int64_t nq, int64_t M, TokView kc, TokView vc,
                                        const float* kcn, const int32_t* kcb, const void* kin, const void* vin,
                                        const float* knin, const int32_t* kbin, const int32_t* len_in,
                                        const uint8_t* evict, void* kout, void* vout, float* knout,
                                        int32_t* kbout, int32_t* len_out, int32_t* imap, int B, int32_t* kperm,
                                        int32_t* koff, int32_t* kpos, void* ksorted, void* vsorted,
                                        const int32_t* qb, int r, int32_t* qperm, int32_t* qoff, int32_t* status,
                                        cudaStream_t s) {
  // one cluster per head plans the step: the query pairs' sort, the survivor scan with
  // the new slots' bucket ids, and the key sort
  cudaError_t e = launch_dependent(compact_plan_kernel, dim3(H * kSortCtas * (qb ? 2 : 1)), dim3(kSortWarpsC * 32),
                                   0, s, nq, M, len_in, evict, len_out, imap, kcb, kbin, kbout, B, kperm, koff,
                                   kpos, qb, r, qperm, qoff, status);
  count_launches(1);
  if (e != cudaSuccess) return e;
  const MergeIO mg{nullptr, nullptr, nullptr, nullptr};
  const SortedIO so{kpos, ksorted, vsorted};
  if (dtype == FASTAR_BF16) {
    if (d == 128)
      return copy_impl<__nv_bfloat16, 128>(H, nq, M, kc, vc, kcn, kcb, kin, vin, knin, kbin, len_in, len_out, imap,
                                           kout, vout, knout, kbout, status, mg, s, so);
    return copy_impl<__nv_bfloat16, 64>(H, nq, M, kc, vc, kcn, kcb, kin, vin, knin, kbin, len_in, len_out, imap,
                                        kout, vout, knout, kbout, status, mg, s, so);
  }
  if (d == 128)
    return copy_impl<float, 128>(H, nq, M, kc, vc, kcn, kcb, kin, vin, knin, kbin, len_in, len_out, imap, kout,
                                 vout, knout, kbout, status, mg, s, so);
  return copy_impl<float, 64>(H, nq, M, kc, vc, kcn, kcb, kin, vin, knin, kbin, len_in, len_out, imap, kout, vout,
                              knout, kbout, status, mg, s, so);
}

// ---------------------------------------------------------------------------------------
// Dense baseline: append the current chunk to an append-only cache.
// ---------------------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(256)
dense_append_kernel(int H, int64_t nq, const T* __restrict__ kc, const T* __restrict__ vc, int64_t hs,
                    int64_t ts, T* __restrict__ kd, T* __restrict__ vd, int64_t cap, int64_t at) {
  constexpr int VPR = D * (int)sizeof(T) / 16;
  const int64_t total = (int64_t)H * nq * VPR;
  for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total;
       g += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = g / VPR;
    const int c = (int)(g - row * VPR);
    const int h = (int)(row / nq);
    const int64_t i = row - (int64_t)h * nq;
    const int64_t dst = ((int64_t)h * cap + at + i) * D;
    reinterpret_cast<uint4*>(kd + dst)[c] = __ldg(reinterpret_cast<const uint4*>(kc + h * hs + i * ts) + c);
    reinterpret_cast<uint4*>(vd + dst)[c] = __ldg(reinterpret_cast<const uint4*>(vc + h * hs + i * ts) + c);
  }
}

template <typename T, int D>
static cudaError_t append_impl(int H, int64_t nq, TokView kc, TokView vc, void* kd, void* vd, int64_t cap,
                               int64_t at, cudaStream_t s) {
  constexpr int VPR = D * (int)sizeof(T) / 16;
  int64_t blocks = ((int64_t)H * nq * VPR + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks < 1) blocks = 1;
  dense_append_kernel<T, D><<<(unsigned)blocks, 256, 0, s>>>(
      H, nq, static_cast<const T*>(kc.p), static_cast<const T*>(vc.p), kc.hs, kc.ts,
      static_cast<T*>(kd), static_cast<T*>(vd), cap, at);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_dense_append(int dtype, int d, int H, int64_t nq, TokView kc, TokView vc, void* kd,
                                void* vd, int64_t cap, int64_t at, cudaStream_t s) {
  if (nq == 0) return cudaSuccess;
  if (dtype == FASTAR_BF16) {
    if (d == 128) return append_impl<__nv_bfloat16, 128>(H, nq, kc, vc, kd, vd, cap, at, s);
    return append_impl<__nv_bfloat16, 64>(H, nq, kc, vc, kd, vd, cap, at, s);
  }
  if (d == 128) return append_impl<float, 128>(H, nq, kc, vc, kd, vd, cap, at, s);
  return append_impl<float, 64>(H, nq, kc, vc, kd, vd, cap, at, s);
}

}  // namespace fastar
