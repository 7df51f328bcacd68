// Softmax attention over gathered key sets, SIMT fp32 path (the f32 dtype, and
// the reference path every other kernel is checked against on the GPU).
//
// Three work decoders share one tile engine:
//   dense  — FAST-AR's dense baseline (technical summary, Key Results: dense
//            FlashAttention-3): every query against keys [0, nk).
//   cross  — AnnCA (technical summary §2.B): the queries of frame f against the
//            kept prompt tokens kidx[h, f, 0..kcnt).
//   sparse — AnnSA (technical summary §2.C): the (query, slot) pairs of bucket b
//            against the cache keys of bucket b; one partial (o, lse) per pair,
//            merged over the r slots afterwards (the slots' key sets are disjoint
//            because every key has exactly one bucket, so the merge is exact).
// Online softmax over 64-key tiles with running max and sum in fp32.  With group counts
// (the merge variant, technical summary §2.A, Lemma 5.1) every key's logit is shifted
// by ln g.
#include <climits>

#include "common.cuh"
#include "kernels.h"
#include "tmap.h"

namespace fastar {

constexpr int kAQ = 64;
constexpr int kAK = 64;

template <int D>
__host__ __device__ constexpr size_t attn_simt_smem() {
  return sizeof(float) * ((size_t)D * kAQ + (size_t)D * kAK + (size_t)kAK * D + (size_t)kAQ * kAK + kAK) +
         sizeof(int64_t) * (kAQ + kAK) + sizeof(int) * (kAQ + FASTAR_MAX_B + 8);
}

template <typename T, int D>
__global__ void __launch_bounds__(256) attn_simt_kernel(const AttnArgs a) {
  extern __shared__ __align__(16) float sm_attn[];
  float* Qs = sm_attn;              // [D][kAQ]
  float* Ks = Qs + D * kAQ;         // [D][kAK]
  float* Vs = Ks + D * kAK;         // [kAK][D]
  float* Ps = Vs + kAK * D;         // [kAQ][kAK]
  int64_t* qoffs = reinterpret_cast<int64_t*>(Ps + kAQ * kAK);  // [kAQ] query row offset or -1
  int64_t* koffs = qoffs + kAQ;                                  // [kAK] key row offset or -1
  int* qdst = reinterpret_cast<int*>(koffs + kAK);               // [kAQ] output row id or -1
  int* pre = qdst + kAQ;                                         // [B + 1] tile prefix (sparse)
  int* info = pre + FASTAR_MAX_B + 1;                            // misc
  float* kbias = reinterpret_cast<float*>(info + 7);             // [kAK] ln g per key (merge variant)

  const int tid = threadIdx.x;
  const int h = blockIdx.y;
  const T* Q = static_cast<const T*>(a.q.p);
  const T* K = static_cast<const T*>(a.k);
  const T* V = static_cast<const T*>(a.v);

  // ---- decode the work item -------------------------------------------------------
  int64_t nkeys = 0;
  int64_t kbase = 0;   // sparse: first position in kperm of the bucket
  int bucket = -1;
  if (a.mode == kSparse) {
    const int32_t* qo = a.qoff + (int64_t)h * (a.B + 1);
    if (tid == 0) {
      int acc = 0;
      for (int b = 0; b < a.B; ++b) {
        pre[b] = acc;
        const int c = qo[b + 1] - qo[b];
        acc += c > 0 ? (c + kAQ - 1) / kAQ : 0;
      }
      pre[a.B] = acc;
      int found = -1;
      if ((int)blockIdx.x < acc) {
        int lo = 0, hi = a.B - 1;   // last b with pre[b] <= blockIdx.x
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (pre[mid] <= (int)blockIdx.x) lo = mid; else hi = mid - 1;
        }
        found = lo;
      }
      info[0] = found;
    }
    __syncthreads();
    bucket = info[0];
    if (bucket < 0) return;
    const int64_t qb0 = qo[bucket] + (int64_t)(blockIdx.x - pre[bucket]) * kAQ;
    const int64_t qb1 = qo[bucket + 1];
    const int64_t np = a.nq * a.r;
    for (int row = tid; row < kAQ; row += blockDim.x) {
      const int64_t pos = qb0 + row;
      int64_t off = -1;
      int dst = -1;
      if (pos < qb1) {
        const int e = a.qperm[(int64_t)h * np + pos];
        if (e >= 0 && e < np) {
          const int64_t i = e / a.r;
          off = h * a.q.hs + i * a.q.ts;
          dst = e;
        } else {
          flag_status(a.status, FASTAR_DEV_BAD_INDEX);
        }
      }
      qoffs[row] = off;
      qdst[row] = dst;
    }
    const int32_t* ko = a.koff + (int64_t)h * (a.B + 1);
    kbase = ko[bucket];
    nkeys = ko[bucket + 1] - kbase;
  } else if (a.mode == kCross) {
    const int f = blockIdx.z;
    const int64_t t0 = (int64_t)blockIdx.x * kAQ;
    for (int row = tid; row < kAQ; row += blockDim.x) {
      const int64_t t = t0 + row;
      const int64_t i = (int64_t)f * a.tpf + t;
      qoffs[row] = t < a.tpf ? h * a.q.hs + i * a.q.ts : -1;
      qdst[row] = t < a.tpf ? (int)i : -1;
    }
    nkeys = a.kcnt[(int64_t)h * a.F + f];
    if (nkeys < 0 || nkeys > a.P) {
      if (tid == 0) flag_status(a.status, FASTAR_DEV_BAD_INDEX);
      nkeys = nkeys < 0 ? 0 : a.P;
    }
  } else {
    const int64_t i0 = (int64_t)blockIdx.x * kAQ;
    for (int row = tid; row < kAQ; row += blockDim.x) {
      const int64_t i = i0 + row;
      qoffs[row] = i < a.nq ? h * a.q.hs + i * a.q.ts : -1;
      qdst[row] = i < a.nq ? (int)i : -1;
    }
    nkeys = a.nk;
  }
  __syncthreads();

  // ---- stage Q (transposed) -------------------------------------------------------
  for (int idx = tid; idx < kAQ * (D / 8); idx += blockDim.x) {
    const int row = idx % kAQ, c8 = idx / kAQ;
    float v[8];
    if (qoffs[row] >= 0) {
      load8(Q + qoffs[row] + c8 * 8, v);
    } else {
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = 0.f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) Qs[(c8 * 8 + u) * kAQ + row] = v[u];
  }

  const int ty = tid >> 4, tx = tid & 15;
  constexpr int OC = D / 16;     // output columns per thread
  float o[4][OC];
  float m[4], l[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    m[r] = neg_inf();
    l[r] = 0.f;
#pragma unroll
    for (int c = 0; c < OC; ++c) o[r][c] = 0.f;
  }

  for (int64_t u0 = 0; u0 < nkeys; u0 += kAK) {
    __syncthreads();
    for (int col = tid; col < kAK; col += blockDim.x) {
      const int64_t u = u0 + col;
      int64_t off = -1;
      int32_t gk = 1;
      if (u < nkeys) {
        if (a.mode == kSparse) {
          const int s = a.kperm[(int64_t)h * a.M + kbase + u];
          if (s >= 0 && s < a.M) {
            off = ((int64_t)h * a.M + s) * D;
            if (a.gcount) gk = a.gcount[(int64_t)h * a.M + s];
          } else {
            flag_status(a.status, FASTAR_DEV_BAD_INDEX);
          }
        } else if (a.mode == kCross) {
          const int p = a.kidx[((int64_t)h * a.F + blockIdx.z) * a.P + u];
          if (p >= 0 && p < a.P) off = ((int64_t)h * a.P + p) * D;
          else flag_status(a.status, FASTAR_DEV_BAD_INDEX);
        } else {
          off = h * a.kv_hs + u * a.kv_ts;
          if (a.gcount) gk = a.gcount[(int64_t)h * a.gc_hs + u];
        }
      }
      koffs[col] = off;
      if (gk < 0) flag_status(a.status, FASTAR_DEV_BAD_INDEX);
      kbias[col] = gk > 0 ? logf((float)gk) : neg_inf();
    }
    __syncthreads();
    for (int idx = tid; idx < kAK * (D / 8); idx += blockDim.x) {
      const int col = idx % kAK, c8 = idx / kAK;
      float kv[8], vv[8];
      if (koffs[col] >= 0) {
        load8(K + koffs[col] + c8 * 8, kv);
        load8(V + koffs[col] + c8 * 8, vv);
      } else {
#pragma unroll
        for (int u = 0; u < 8; ++u) kv[u] = vv[u] = 0.f;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        Ks[(c8 * 8 + u) * kAK + col] = kv[u];
        Vs[col * D + c8 * 8 + u] = vv[u];
      }
    }
    __syncthreads();
    float s[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) s[r][c] = 0.f;
#pragma unroll 8
    for (int k = 0; k < D; ++k) {
      const float4 qa = *reinterpret_cast<const float4*>(Qs + k * kAQ + ty * 4);
      const float4 kb = *reinterpret_cast<const float4*>(Ks + k * kAK + tx * 4);
      const float qv[4] = {qa.x, qa.y, qa.z, qa.w};
      const float kv[4] = {kb.x, kb.y, kb.z, kb.w};
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) s[r][c] = fmaf(qv[r], kv[c], s[r][c]);
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      float mx = neg_inf();
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        s[r][c] = koffs[tx * 4 + c] >= 0 ? fmaf(s[r][c], a.scale, kbias[tx * 4 + c]) : neg_inf();
        mx = fmaxf(mx, s[r][c]);
      }
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float mnew = fmaxf(m[r], mx);
      const float corr = mnew == neg_inf() ? 1.f : __expf(m[r] - mnew);
      float sum = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float p = mnew == neg_inf() ? 0.f : __expf(s[r][c] - mnew);
        Ps[(ty * 4 + r) * kAK + tx * 4 + c] = p;
        sum += p;
      }
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      l[r] = l[r] * corr + sum;
      m[r] = mnew;
#pragma unroll
      for (int c = 0; c < OC; ++c) o[r][c] *= corr;
    }
    __syncthreads();
#pragma unroll 4
    for (int u = 0; u < kAK; ++u) {
      float vv[OC];
#pragma unroll
      for (int c = 0; c < OC; ++c) vv[c] = Vs[u * D + tx * OC + c];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float p = Ps[(ty * 4 + r) * kAK + u];
#pragma unroll
        for (int c = 0; c < OC; ++c) o[r][c] = fmaf(p, vv[c], o[r][c]);
      }
    }
  }

  // ---- epilogue --------------------------------------------------------------------------
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int row = ty * 4 + r;
    const int dst = qdst[row];
    if (dst < 0) continue;
    const bool live = l[r] > 0.f;
    const float inv = live ? 1.0f / l[r] : 0.f;
    const float lse = live ? m[r] + __logf(l[r]) : neg_inf();
    if (a.mode == kSparse) {
      float* po = a.part_o + ((int64_t)h * a.nq * a.r + dst) * D + tx * OC;
#pragma unroll
      for (int c = 0; c < OC; ++c) po[c] = o[r][c] * inv;
      if (tx == 0) a.part_lse[(int64_t)h * a.nq * a.r + dst] = lse;
    } else {
      T* out = static_cast<T*>(a.out) + h * a.o_hs + (int64_t)dst * a.o_ts + tx * OC;
#pragma unroll
      for (int c = 0; c < OC; ++c) out[c] = from_f<T>(o[r][c] * inv);
      const int64_t nrow = a.mode == kCross ? (int64_t)a.F * a.tpf : a.nq;
      if (tx == 0 && a.lse) a.lse[(int64_t)h * nrow + dst] = lse;
    }
  }
}

// One warp per (head, query): exact LSE merge of the r bucket-slot partials.
template <typename T, int D>
__global__ void __launch_bounds__(256) attn_merge_kernel(const AttnArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (wid >= (int64_t)a.H * a.nq) return;
  const int h = (int)(wid / a.nq);
  const int64_t i = wid - (int64_t)h * a.nq;
  const int64_t base = (int64_t)h * a.nq * a.r + i * a.r;
  float mx = neg_inf();
  for (int s = 0; s < a.r; ++s) mx = fmaxf(mx, a.part_lse[base + s]);
  float w[FASTAR_MAX_R];
  float W = 0.f;
  for (int s = 0; s < a.r; ++s) {
    const float ls = a.part_lse[base + s];
    w[s] = (mx == neg_inf() || ls == neg_inf()) ? 0.f : __expf(ls - mx);
    W += w[s];
  }
  const float invW = W > 0.f ? 1.0f / W : 0.f;
  T* out = static_cast<T*>(a.out) + h * a.o_hs + i * a.o_ts;
  for (int c = lane; c < D; c += 32) {
    float acc = 0.f;
    for (int s = 0; s < a.r; ++s)
      if (w[s] > 0.f) acc = fmaf(w[s], a.part_o[(base + s) * D + c], acc);
    out[c] = from_f<T>(acc * invW);
  }
  if (lane == 0 && a.lse) a.lse[(int64_t)h * a.nq + i] = W > 0.f ? mx + __logf(W) : neg_inf();
}

size_t sparse_attn_workspace(int H, int64_t nq, int d, int r, int B, int64_t M) {
  // fp32 partials (o, lse) per (query, slot); then (16-byte aligned) the tensor-core
  // path's work list and its length; then (1024-byte aligned) its bucket-ordered copy
  // of the cache K and V (bf16) and of the keys' log2 group counts (float)
  const size_t head = sizeof(float) * (size_t)H * nq * r * (d + 1);
  const size_t plan = ((head + 15) & ~(size_t)15) + sparse_plan_bytes(H, nq, r, B);
  return ((plan + 1023) & ~(size_t)1023) + 2 * sizeof(uint16_t) * (size_t)H * M * d + sizeof(float) * (size_t)H * M +
         1024;
}

template <typename T, int D>
static cudaError_t attn_impl(const AttnArgs& a, cudaStream_t s) {
  constexpr size_t smem = attn_simt_smem<D>();
  auto kern = attn_simt_kernel<T, D>;
  const cudaError_t attr = opt_in_smem((const void*)kern, (int)smem);
  if (attr != cudaSuccess) return attr;
  cudaError_t e;
  dim3 grid;
  if (a.mode == kDense) {
    if (a.nq == 0) return cudaSuccess;
    grid = dim3((unsigned)((a.nq + kAQ - 1) / kAQ), a.H, 1);
  } else if (a.mode == kCross) {
    if (a.tpf == 0 || a.F == 0) return cudaSuccess;
    grid = dim3((unsigned)((a.tpf + kAQ - 1) / kAQ), a.H, a.F);
  } else {
    if (a.nq == 0) return cudaSuccess;
    const int64_t tiles = (a.nq * a.r + kAQ - 1) / kAQ + a.B;
    grid = dim3((unsigned)tiles, a.H, 1);
  }
  if (sizeof(T) == 2) {
    // bf16: the tensor-core kernels (for AnnSA: planning, attention, slot merge)
    if (launch_attn_tc(D, a, s)) return cudaGetLastError();
  }
  // cross-attention over the caller's kept-row planes has no index list for this path
  if (a.mode == kCross && a.presorted) return cudaErrorNotSupported;
  {
    AttnArgs b = a;
    kern<<<grid, 256, smem, s>>>(b);
  }
  count_launches(1);
  e = cudaGetLastError();
  if (e != cudaSuccess || a.mode != kSparse) return e;
  const int64_t warps = (int64_t)a.H * a.nq;
  attn_merge_kernel<T, D><<<(unsigned)((warps * 32 + 255) / 256), 256, 0, s>>>(a);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_attention(int dtype, int d, const AttnArgs& a, cudaStream_t s) {
  if (dtype == FASTAR_BF16) {
    if (d == 128) return attn_impl<__nv_bfloat16, 128>(a, s);
    return attn_impl<__nv_bfloat16, 64>(a, s);
  }
  if (d == 128) return attn_impl<float, 128>(a, s);
  return attn_impl<float, 64>(a, s);
}

}  // namespace fastar
