// TempCache top-1 temporal-correspondence match and eviction flags (SIMT path).
//
// FAST-AR technical summary §2.A / blog §1: for each current-frame query find the
// top-1 nearest cached key from previous frames; a cached key whose content the
// current chunk re-expresses (similarity >= tau) is merged away, so only the most
// recent representative stays.
//
// Matching is by cosine.  Since |q_i| is constant along a row, the row arg-max of
// cos(q_i, k_j) is the arg-max of (q_i . k_j) * (1/|k_j|); the kernel tracks the
// top two of that value per row and the finaliser divides by |q_i| once.
#include <climits>

#include "common.cuh"
#include "kernels.h"
#include "tmap.h"

namespace fastar {

constexpr int kMT = 64;  // queries per tile
constexpr int kNT = 64;  // keys per tile

struct Top2 {
  float m1;
  int i1;
  float m2;
};

// Folds value v of column j into a running top-2; columns arrive in increasing j,
// so a strict > keeps the lowest index on ties.
__device__ __forceinline__ void top2_push(Top2& t, float v, int j) {
  if (v > t.m1) {
    t.m2 = t.m1;
    t.m1 = v;
    t.i1 = j;
  } else if (v > t.m2) {
    t.m2 = v;
  }
}

// Merges two top-2 summaries of disjoint column sets.
__device__ __forceinline__ Top2 top2_merge(Top2 a, Top2 b) {
  Top2 o;
  if (beats(b.m1, b.i1, a.m1, a.i1)) {
    o.m1 = b.m1;
    o.i1 = b.i1;
    o.m2 = fmaxf(a.m1, b.m2);
  } else {
    o.m1 = a.m1;
    o.i1 = a.i1;
    o.m2 = fmaxf(a.m2, b.m1);
  }
  return o;
}

int match_splits(int H, int64_t nq, int64_t M) {
  const int64_t tiles = (nq + kMT - 1) / kMT * H;
  int64_t s = (2 * 152 + tiles - 1) / (tiles > 0 ? tiles : 1);
  const int64_t max_s = (M + kNT - 1) / kNT;
  if (s > max_s) s = max_s;
  if (s > 64) s = 64;
  if (s < 1) s = 1;
  return (int)s;
}

size_t match_workspace(int H, int64_t nq, int64_t M) {
  const size_t simt = sizeof(float4) * (size_t)match_splits(H, nq, M) * H * (size_t)nq;
  const size_t tcw = match_tc_workspace(H, nq, M);
  return simt > tcw ? simt : tcw;
}

// grid (ceil(nq/64), H, splits); 256 threads; thread (ty, tx) owns rows ty*4..+3 and
// columns tx*4..+3 of each 64x64 tile.  Q and K tiles are staged transposed in fp32.
template <typename T, int D>
__global__ void __launch_bounds__(256)
match_simt_kernel(const T* __restrict__ q, int64_t hs, int64_t ts, int64_t nq,
                  const T* __restrict__ ck, const float* __restrict__ cknorm,
                  const int32_t* __restrict__ clen, int64_t M, int64_t chunk,
                  float4* __restrict__ part, uint8_t* __restrict__ evict, int32_t* __restrict__ owner,
                  int32_t* status) {
  extern __shared__ float sm_match[];
  float* Qs = sm_match;            // [D][kMT]
  float* Ks = Qs + D * kMT;        // [D][kNT]
  float* invk = Ks + D * kNT;      // [kNT]
  const int h = blockIdx.y;
  const int tid = threadIdx.x;
  // clear the eviction flags and owners of this head (the finaliser sets them afterwards)
  {
    const int64_t nblk = (int64_t)gridDim.x * gridDim.z;
    const int64_t b = (int64_t)blockIdx.z * gridDim.x + blockIdx.x;
    for (int64_t j = b * blockDim.x + tid; j < M; j += nblk * blockDim.x) {
      evict[h * M + j] = 0;
      if (owner) owner[h * M + j] = -1;
    }
  }
  int64_t n = clen[h];
  if (n < 0 || n > M) {
    if (tid == 0 && blockIdx.x == 0 && blockIdx.z == 0) flag_status(status, FASTAR_DEV_BAD_LEN);
    n = n < 0 ? 0 : M;
  }
  const int64_t i0 = (int64_t)blockIdx.x * kMT;
  const int64_t jbeg = (int64_t)blockIdx.z * chunk;
  const int64_t jend = jbeg + chunk < n ? jbeg + chunk : n;
  // stage Q transposed
  for (int idx = tid; idx < kMT * (D / 8); idx += blockDim.x) {
    const int row = idx % kMT, c8 = idx / kMT;
    float v[8];
    if (i0 + row < nq) {
      load8(q + h * hs + (i0 + row) * ts + c8 * 8, v);
    } else {
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = 0.f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) Qs[(c8 * 8 + u) * kMT + row] = v[u];
  }
  const int ty = tid >> 4, tx = tid & 15;
  Top2 best[4];
#pragma unroll
  for (int a = 0; a < 4; ++a) best[a] = Top2{neg_inf(), INT_MAX, neg_inf()};
  const T* ckh = ck + (int64_t)h * M * D;
  for (int64_t j0 = jbeg; j0 < jend; j0 += kNT) {
    __syncthreads();
    for (int idx = tid; idx < kNT * (D / 8); idx += blockDim.x) {
      const int col = idx % kNT, c8 = idx / kNT;
      float v[8];
      if (j0 + col < jend) {
        load8(ckh + (j0 + col) * D + c8 * 8, v);
      } else {
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = 0.f;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) Ks[(c8 * 8 + u) * kNT + col] = v[u];
    }
    if (tid < kNT) {
      const float kn = j0 + tid < jend ? cknorm[(int64_t)h * M + j0 + tid] : 0.f;
      invk[tid] = kn > 0.f ? 1.0f / kn : 0.f;
    }
    __syncthreads();
    float acc[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
#pragma unroll 8
    for (int k = 0; k < D; ++k) {
      const float4 qa = *reinterpret_cast<const float4*>(Qs + k * kMT + ty * 4);
      const float4 kb = *reinterpret_cast<const float4*>(Ks + k * kNT + tx * 4);
      const float qv[4] = {qa.x, qa.y, qa.z, qa.w};
      const float kv[4] = {kb.x, kb.y, kb.z, kb.w};
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(qv[a], kv[b], acc[a][b]);
    }
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int64_t j = j0 + tx * 4 + b;
      if (j < jend) {
        const float s = invk[tx * 4 + b];
#pragma unroll
        for (int a = 0; a < 4; ++a) top2_push(best[a], acc[a][b] * s, (int)j);
      }
    }
  }
  // combine the 16 column groups of each row (lanes tx of one half-warp)
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    Top2 t = best[a];
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) {
      Top2 u;
      u.m1 = __shfl_xor_sync(0xffffffffu, t.m1, o);
      u.i1 = __shfl_xor_sync(0xffffffffu, t.i1, o);
      u.m2 = __shfl_xor_sync(0xffffffffu, t.m2, o);
      t = top2_merge(t, u);
    }
    const int64_t i = i0 + ty * 4 + a;
    if (tx == 0 && i < nq)
      part[((int64_t)blockIdx.z * gridDim.y + h) * nq + i] =
          make_float4(t.m1, __int_as_float(t.i1), t.m2, 0.f);
  }
}

// Eight lanes per (head, query): merge the split partials, turn the best values into
// cosines, and test the matched entry for eviction: cos(kcur_i, k_top1) >= tau.  The
// owner of an evicted entry is the lowest evicting query (an atomic minimum over the
// unsigned view, where the cleared value -1 is the largest).
constexpr int kFinLanes = 4;   // finaliser lanes per query

template <typename T, int D>
__global__ void __launch_bounds__(256)
match_finalize_kernel(const T* __restrict__ q, const T* __restrict__ kc, int64_t hs, int64_t ts,
                      int64_t nq, int H, const T* __restrict__ ck, const float* __restrict__ cknorm,
                      const int32_t* __restrict__ clen, int64_t M, float tau, int splits,
                      const float4* __restrict__ part, int32_t* __restrict__ top1,
                      float* __restrict__ s1, float* __restrict__ s2, uint8_t* __restrict__ evict,
                      int32_t* __restrict__ owner, int qn_part) {
  pdl_wait();   // the partials (and cleared flags) of the match kernel before it in the stream
  // kFinLanes lanes per query: each lane owns D / kFinLanes consecutive elements (vector
  // loads); four lanes keep every warp of the layer resident at once
  // grid: (queries / (256 / kFinLanes), heads)
  const int sub = threadIdx.x & (kFinLanes - 1);
  const int h = (int)blockIdx.y;
  const int64_t iq = (int64_t)blockIdx.x * (256 / kFinLanes) + threadIdx.x / kFinLanes;
  const bool in = iq < nq;
  const int64_t i = in ? iq : 0;   // (out-of-range lanes still take part in the shuffles)
  int64_t n = clen[h];
  n = n < 0 ? 0 : (n > M ? M : n);
  // this lane's first partial and the two rows are loaded before any of them is used
  float4 p0 = make_float4(neg_inf(), __int_as_float(INT_MAX), neg_inf(), 0.f);
  if (sub < splits) p0 = part[((int64_t)sub * H + h) * nq + i];
  // |q_i| (from the partials when the match kernel summed it: qn_part) and |kcur_i|
  constexpr int E = D / kFinLanes;
  const T* qr = q + h * hs + i * ts + sub * E;
  const T* kr = kc + h * hs + i * ts + sub * E;
  float kv[E];
  float qq = 0.f, kk = 0.f;
#pragma unroll
  for (int c = 0; c < E; c += 8) {
    load8(kr + c, kv + c);
    if (!qn_part) {
      float a[8];
      load8(qr + c, a);
#pragma unroll
      for (int u = 0; u < 8; ++u) qq = fmaf(a[u], a[u], qq);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) kk = fmaf(kv[c + u], kv[c + u], kk);
  }
  if (qn_part) qq = sub == 0 ? p0.w : 0.f;   // segment 0's |q|^2, summed below like the shares
#pragma unroll
  for (int o = kFinLanes / 2; o > 0; o >>= 1) {
    qq += __shfl_xor_sync(0xffffffffu, qq, o);
    kk += __shfl_xor_sync(0xffffffffu, kk, o);
  }
  Top2 t{p0.x, __float_as_int(p0.y), p0.z};
  for (int s = sub + kFinLanes; s < splits; s += kFinLanes) {
    const float4 p = part[((int64_t)s * H + h) * nq + i];
    t = top2_merge(t, Top2{p.x, __float_as_int(p.y), p.z});
  }
#pragma unroll
  for (int o = kFinLanes / 2; o > 0; o >>= 1) {
    Top2 u;
    u.m1 = __shfl_xor_sync(0xffffffffu, t.m1, o);
    u.i1 = __shfl_xor_sync(0xffffffffu, t.i1, o);
    u.m2 = __shfl_xor_sync(0xffffffffu, t.m2, o);
    t = top2_merge(t, u);
  }
  qq = sqrtf(qq);
  kk = sqrtf(kk);
  const bool any = n > 0 && t.i1 != INT_MAX;
  const int j = any ? t.i1 : -1;
  float dot = 0.f;
  if (any) {
    const T* jr = ck + ((int64_t)h * M + j) * D + sub * E;
#pragma unroll
    for (int c = 0; c < E; c += 8) {
      float b[8];
      load8(jr + c, b);
#pragma unroll
      for (int u = 0; u < 8; ++u) dot = fmaf(kv[c + u], b[u], dot);
    }
  }
#pragma unroll
  for (int o = kFinLanes / 2; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
  if (in && sub == 0) {
    top1[(int64_t)h * nq + i] = j;
    const float inv_q = qq > 0.f ? 1.0f / qq : 0.f;
    if (s1) s1[(int64_t)h * nq + i] = any ? t.m1 * inv_q : neg_inf();
    if (s2) s2[(int64_t)h * nq + i] = (n > 1 && t.m2 != neg_inf()) ? t.m2 * inv_q : neg_inf();
    if (any) {
      const float den = kk * cknorm[(int64_t)h * M + j];
      const float c = den > 0.f ? dot / den : 0.f;
      if (c >= tau) {
        evict[(int64_t)h * M + j] = 1;
        if (owner) atomicMin(reinterpret_cast<unsigned int*>(owner) + (int64_t)h * M + j, (unsigned int)i);
      }
    }
  }
}

template <typename T, int D>
static cudaError_t match_impl(TokView q, TokView kc, int H, int64_t nq, const void* ck,
                              const float* cknorm, const int32_t* clen, int64_t M, float tau,
                              int32_t* top1, float* s1, float* s2, uint8_t* evict, int32_t* owner,
                              int32_t* status, void* ws, cudaStream_t s, const void* ck_ev = nullptr,
                              const float* kn_ev = nullptr) {
  // the keys ranked (ck, cknorm) and the keys the eviction test uses (ck_ev, kn_ev) are
  // the same except in the quantised match, which ranks decoded keys
  if (!ck_ev) {
    ck_ev = ck;
    kn_ev = cknorm;
  }
  float4* part = static_cast<float4*>(ws);
  if (sizeof(T) == 2 && nq > 0) {
    // bf16: the tensor-core kernel (the SIMT kernel below only if its set-up is refused)
    const int tsplits =
        launch_match_tc(D, q, H, nq, ck, cknorm, clen, M, s2 != nullptr, part, evict, owner, status, s);
    if (tsplits > 0) {
      cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return e;
      e = launch_dependent(match_finalize_kernel<T, D>,
                           dim3((unsigned)((nq * kFinLanes + 255) / 256), (unsigned)H), dim3(256), 0, s, static_cast<const T*>(q.p), static_cast<const T*>(kc.p), q.hs,
                           q.ts, nq, H, static_cast<const T*>(ck_ev), kn_ev, clen, M, tau, tsplits,
                           (const float4*)part, top1, s1, s2, evict, owner, 1);
      count_launches(1);
      return e;
    }
  }
  const int splits = match_splits(H, nq, M);
  int64_t chunk = (M + splits - 1) / splits;
  chunk = (chunk + kNT - 1) / kNT * kNT;
  const size_t smem = sizeof(float) * ((size_t)D * kMT + (size_t)D * kNT + kNT);
  auto k1 = match_simt_kernel<T, D>;
  const cudaError_t attr = opt_in_smem((const void*)k1, (int)smem);
  if (attr != cudaSuccess) return attr;
  cudaError_t e;
  const unsigned gx = (unsigned)((nq + kMT - 1) / kMT);
  if (nq > 0) {
    k1<<<dim3(gx, H, splits), 256, smem, s>>>(static_cast<const T*>(q.p), q.hs, q.ts, nq,
                                              static_cast<const T*>(ck), cknorm, clen, M, chunk,
                                              part, evict, owner, status);
    count_launches(1);
  } else {
    e = cudaMemsetAsync(evict, 0, (size_t)H * M, s);
    if (e != cudaSuccess) return e;
    if (owner) {
      e = cudaMemsetAsync(owner, 0xff, sizeof(int32_t) * (size_t)H * M, s);
      if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  match_finalize_kernel<T, D><<<dim3((unsigned)((nq * kFinLanes + 255) / 256), (unsigned)H), 256, 0, s>>>(
      static_cast<const T*>(q.p), static_cast<const T*>(kc.p), q.hs, q.ts, nq, H,
      static_cast<const T*>(ck_ev), kn_ev, clen, M, tau, splits, part, top1, s1, s2, evict, owner, 0);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_tempcache_match(int dtype, int d, TokView q, TokView kc, int H, int64_t nq,
                                   const void* ck, const float* cknorm, const int32_t* clen,
                                   int64_t M, float tau, int32_t* top1, float* s1, float* s2,
                                   uint8_t* evict, int32_t* owner, int32_t* status, void* ws, cudaStream_t s) {
  if (dtype == FASTAR_BF16) {
    if (d == 128)
      return match_impl<__nv_bfloat16, 128>(q, kc, H, nq, ck, cknorm, clen, M, tau, top1, s1, s2, evict, owner,
                                            status, ws, s);
    return match_impl<__nv_bfloat16, 64>(q, kc, H, nq, ck, cknorm, clen, M, tau, top1, s1, s2, evict, owner,
                                         status, ws, s);
  }
  if (d == 128)
    return match_impl<float, 128>(q, kc, H, nq, ck, cknorm, clen, M, tau, top1, s1, s2, evict, owner, status, ws, s);
  return match_impl<float, 64>(q, kc, H, nq, ck, cknorm, clen, M, tau, top1, s1, s2, evict, owner, status, ws, s);
}

// The quantised match: the cached keys' codes decoded into the workspace (bf16 rows and
// their norms), ranked by the tensor-core match, the eviction tested on the true keys.
size_t match_pq_workspace(int H, int64_t nq, int64_t M, int d) {
  const size_t part = (match_workspace(H, nq, M) + 1023) & ~(size_t)1023;
  return part + sizeof(uint16_t) * (size_t)H * M * d + sizeof(float) * (size_t)H * M + 1024;
}

cudaError_t launch_tempcache_match_pq(int d, TokView q, TokView kc, int H, int64_t nq, const void* ck,
                                      const float* cknorm, const uint8_t* codes, const int32_t* clen, int64_t M,
                                      const void* cb, int m, int Kc, float tau, int32_t* top1, float* s1,
                                      uint8_t* evict, int32_t* owner, int32_t* status, void* ws, cudaStream_t s) {
  const uintptr_t base = (reinterpret_cast<uintptr_t>(ws) + 1023) & ~static_cast<uintptr_t>(1023);
  uint8_t* khat = reinterpret_cast<uint8_t*>(base) + ((match_workspace(H, nq, M) + 1023) & ~(size_t)1023);
  float* khat_norm = reinterpret_cast<float*>(khat + sizeof(uint16_t) * (size_t)H * M * d);
  cudaError_t e = launch_pq_decode(d, H, M, m, Kc, codes, clen, cb, khat, khat_norm, status, s);
  if (e != cudaSuccess) return e;
  void* part = reinterpret_cast<void*>(base);
  if (d == 128)
    return match_impl<__nv_bfloat16, 128>(q, kc, H, nq, khat, khat_norm, clen, M, tau, top1, s1, nullptr, evict,
                                          owner, status, part, s, ck, cknorm);
  return match_impl<__nv_bfloat16, 64>(q, kc, H, nq, khat, khat_norm, clen, M, tau, top1, s1, nullptr, evict, owner,
                                       status, part, s, ck, cknorm);
}

}  // namespace fastar
