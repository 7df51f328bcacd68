// AnnCA: frame-relevant prompt tokens (SIMT path).
//
// FAST-AR technical summary §2.B / blog §2: a prompt token is kept for a frame
// when it shares an ANN bucket with at least one of the frame's queries; the
// score (max bucket-sharing query cosine), the threshold tau_ca and the
// always-keep top-k are the method spec's.
//
// Kernel 1 scores every (head, frame, prompt token); kernel 2 ranks the scores of
// one (head, frame) in a single CTA and writes the keep mask and the compacted,
// ascending index list.
#include <climits>

#include "common.cuh"
#include "kernels.h"
#include "tmap.h"

namespace fastar {

constexpr int kCQ = 64;  // queries per tile
constexpr int kCP = 64;  // prompt tokens per tile

template <typename T, int D>
__global__ void __launch_bounds__(256)
annca_score_kernel(const T* __restrict__ q, int64_t hs, int64_t ts, int F, int64_t tpf,
                   const int32_t* __restrict__ qb, int r, const T* __restrict__ kp,
                   const int32_t* __restrict__ pb, int64_t P, int gate, float* __restrict__ score) {
  extern __shared__ __align__(16) float sm_ca[];
  float* Qs = sm_ca;                // [D][kCQ]
  float* Ks = Qs + D * kCQ;         // [D][kCP]
  float* qinv = Ks + D * kCP;       // [kCQ]
  float* pinv = qinv + kCQ;         // [kCP]
  float* red = pinv + kCP;          // [16][kCP]
  int* qbs = reinterpret_cast<int*>(red + 16 * kCP);   // [kCQ][FASTAR_MAX_R]
  int* pbs = qbs + kCQ * FASTAR_MAX_R;                  // [kCP]
  const int tid = threadIdx.x;
  const int h = blockIdx.y, f = blockIdx.z;
  const int64_t p0 = (int64_t)blockIdx.x * kCP;
  const int64_t nq = (int64_t)F * tpf;
  // stage the prompt tile (transposed) and its norms / buckets
  for (int idx = tid; idx < kCP * (D / 8); idx += blockDim.x) {
    const int col = idx % kCP, c8 = idx / kCP;
    float v[8];
    if (p0 + col < P) {
      load8(kp + ((int64_t)h * P + p0 + col) * D + c8 * 8, v);
    } else {
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = 0.f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) Ks[(c8 * 8 + u) * kCP + col] = v[u];
  }
  __syncthreads();
  if (tid < kCP) {
    float ss = 0.f;
    for (int k = 0; k < D; ++k) ss = fmaf(Ks[k * kCP + tid], Ks[k * kCP + tid], ss);
    const float nrm = sqrtf(ss);
    pinv[tid] = nrm > 0.f ? 1.0f / nrm : 0.f;
    pbs[tid] = p0 + tid < P ? pb[(int64_t)h * P + p0 + tid] : -1;
  }
  const int ty = tid >> 4, tx = tid & 15;
  float best[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) best[c] = neg_inf();
  for (int64_t t0 = 0; t0 < tpf; t0 += kCQ) {
    __syncthreads();
    for (int idx = tid; idx < kCQ * (D / 8); idx += blockDim.x) {
      const int row = idx % kCQ, c8 = idx / kCQ;
      float v[8];
      if (t0 + row < tpf) {
        load8(q + h * hs + ((int64_t)f * tpf + t0 + row) * ts + c8 * 8, v);
      } else {
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = 0.f;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) Qs[(c8 * 8 + u) * kCQ + row] = v[u];
    }
    for (int idx = tid; idx < kCQ * r; idx += blockDim.x) {
      const int row = idx / r, s = idx - row * r;
      qbs[row * FASTAR_MAX_R + s] =
          t0 + row < tpf ? qb[((int64_t)h * nq + (int64_t)f * tpf + t0 + row) * r + s] : -2;
    }
    __syncthreads();
    if (tid < kCQ) {
      float ss = 0.f;
      for (int k = 0; k < D; ++k) ss = fmaf(Qs[k * kCQ + tid], Qs[k * kCQ + tid], ss);
      const float nrm = sqrtf(ss);
      qinv[tid] = (t0 + tid < tpf && nrm > 0.f) ? 1.0f / nrm : 0.f;
    }
    __syncthreads();
    float acc[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
#pragma unroll 8
    for (int k = 0; k < D; ++k) {
      const float4 qa = *reinterpret_cast<const float4*>(Qs + k * kCQ + ty * 4);
      const float4 kb = *reinterpret_cast<const float4*>(Ks + k * kCP + tx * 4);
      const float qv[4] = {qa.x, qa.y, qa.z, qa.w};
      const float kv[4] = {kb.x, kb.y, kb.z, kb.w};
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(qv[a], kv[b], acc[a][b]);
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int row = ty * 4 + a;
      if (t0 + row >= tpf) continue;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int col = tx * 4 + b;
        bool ok = pbs[col] >= 0;
        if (ok && gate) {
          bool shared = false;
          for (int s = 0; s < r; ++s) shared |= qbs[row * FASTAR_MAX_R + s] == pbs[col];
          ok = shared;
        }
        if (ok) best[b] = fmaxf(best[b], acc[a][b] * qinv[row] * pinv[col]);
      }
    }
  }
  __syncthreads();
#pragma unroll
  for (int b = 0; b < 4; ++b) red[ty * kCP + tx * 4 + b] = best[b];
  __syncthreads();
  if (tid < kCP && p0 + tid < P) {
    float mx = neg_inf();
    for (int y = 0; y < 16; ++y) mx = fmaxf(mx, red[y * kCP + tid]);
    score[((int64_t)h * F + f) * P + p0 + tid] = mx;
  }
}

// The kept rows' copy written beside the selection (all null otherwise): kp_kept /
// vp_kept [H, F, P, d] receive, for each (head, frame), kp / vp rows kidx[0..kcnt) in
// order, then zero rows up to the next multiple of 64 (at most P); cpr 16-byte chunks
// per row.
struct KeptPlanes {
  const uint4* kp;
  const uint4* vp;
  uint4* kk;
  uint4* vk;
  int cpr;
};

// gridDim.y CTAs per (head, frame): rank = #{p' : (s', p') precedes (s, p)} in the order
// (score desc, index asc), -inf last; keep = s >= tau_ca or rank < min(topk, P).
// A (head, frame) holding a NaN score is not ranked: kcnt = -1, no token kept.  Every CTA
// of a (head, frame) ranks (P scores: cheap); the first writes keep / kidx / kcnt and all
// share the copy of the kept rows when planes are asked for.
__global__ void __launch_bounds__(1024)
annca_rank_kernel(int F, int64_t P, float tau_ca, int topk, const float* __restrict__ score,
                  uint8_t* __restrict__ keep, int32_t* __restrict__ kidx, int32_t* __restrict__ kcnt,
                  const KeptPlanes kpl) {
  __shared__ float s[FASTAR_MAX_P];
  __shared__ int kl[FASTAR_MAX_P];   // the kept list, ascending
  __shared__ int wsum[32];
  const int hf = blockIdx.x;
  const bool lead = blockIdx.y == 0;
  const int p = threadIdx.x;
  const float* sc = score + (int64_t)hf * P;
  __shared__ int bad;
  if (p == 0) bad = 0;
  __syncthreads();
  if (p < P) {
    s[p] = sc[p];
    if (s[p] != s[p]) bad = 1;   // a NaN score: the scorer timed out, or an input held a NaN
  }
  __syncthreads();
  if (bad) {
    // the (head, frame) cannot be ranked: no kept token, kcnt = -1 marks it
    if (lead && p < P) {
      keep[(int64_t)hf * P + p] = 0;
      kidx[(int64_t)hf * P + p] = -1;
    }
    if (lead && p == 0) kcnt[hf] = -1;
    return;
  }
  int k = 0;
  if (p < P) {
    const float mine = s[p];
    const int lim = topk < P ? topk : (int)P;
    if (mine >= tau_ca) {
      k = 1;
    } else {
      // only "rank < lim" matters: stop counting once lim tokens are known to precede p
      int rank = 0;
      for (int u = 0; u < P && rank < lim; ++u) {
        const float o = s[u];
        rank += (o > mine || (o == mine && u < p)) ? 1 : 0;
      }
      k = rank < lim ? 1 : 0;
    }
    if (lead) keep[(int64_t)hf * P + p] = (uint8_t)k;
  }
  // exclusive scan of the keep flags in index order
  const int lane = p & 31, warp = p >> 5;
  int incl = k;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int t = wsum[lane];
    int ti = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, ti, o);
      if (lane >= o) ti += v;
    }
    wsum[lane] = ti - t;
  }
  __syncthreads();
  const int pos = wsum[warp] + incl - k;
  __shared__ int total;
  if (p == blockDim.x - 1) total = pos + k;
  __syncthreads();
  if (p < P && k) kl[pos] = p;
  if (lead) {
    if (p < P) {
      int32_t* out = kidx + (int64_t)hf * P;
      if (k) out[pos] = p;
      if (p >= total) out[p] = -1;
    }
    if (p == 0) kcnt[hf] = total;
  }
  if (!kpl.kk) return;
  __syncthreads();
  // the kept rows of this (head, frame), then zero rows to the next 64-row boundary; the
  // gridDim.y CTAs take interleaved 16-byte chunks, four in flight per thread
  const int64_t lim = (int64_t)(total + 63) / 64 * 64 < P ? (int64_t)(total + 63) / 64 * 64 : P;
  const int64_t chunks = lim * kpl.cpr;
  const int64_t h = hf / F;
  const uint4* ksrc = kpl.kp + h * P * kpl.cpr;
  const uint4* vsrc = kpl.vp + h * P * kpl.cpr;
  uint4* kdst = kpl.kk + (int64_t)hf * P * kpl.cpr;
  uint4* vdst = kpl.vk + (int64_t)hf * P * kpl.cpr;
  const int64_t step = (int64_t)gridDim.y * blockDim.x;
  for (int64_t g0 = (int64_t)blockIdx.y * blockDim.x + p; g0 < chunks; g0 += 4 * step) {
    uint4 kv[4], vv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t g = g0 + u * step;
      kv[u] = vv[u] = make_uint4(0, 0, 0, 0);
      if (g < chunks) {
        const int64_t row = g / kpl.cpr;
        if (row < total) {
          const int64_t src = (int64_t)kl[row] * kpl.cpr + (g - row * kpl.cpr);
          kv[u] = __ldg(ksrc + src);
          vv[u] = __ldg(vsrc + src);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t g = g0 + u * step;
      if (g < chunks) {
        kdst[g] = kv[u];
        vdst[g] = vv[u];
      }
    }
  }
}

size_t annca_workspace(int H, int F, int64_t P) { return sizeof(float) * (size_t)H * F * P + 256; }

// ---------------------------------------------------------------------------------------
// Bucket-gated scoring by bucket.  With the gate, prompt token p can only be scored by
// queries whose bucket set holds pb[p], so one CTA per (head, bucket b) visits exactly
// the pairs (query with b in R(i), prompt token with pb = b): the ANN buckets turn the
// frame x prompt score matrix into a union of small dense blocks.  The CTA collects its
// query list (any order: only maxima are taken), then for chunks of 32 of its prompt
// tokens and 64 of its queries forms the dot products in fp32 and keeps, per prompt
// token and latent frame, the largest q.kp/|q|; the score is that times 1/|kp|.
// ---------------------------------------------------------------------------------------
// Optional bucket order of the (query, slot) pairs (B buckets; qperm/qoff as the
// counting sort writes them).  qperm == nullptr: scan the query buckets instead.
struct BucketOrder {
  int B;
  const int32_t* qperm;
  const int32_t* qoff;
};

constexpr int kBP = 32;          // prompt tokens per chunk
constexpr int kBQ = 64;          // queries per chunk
constexpr int kBMaxF = 16;       // frames per chunk supported by this path
constexpr int kBMaxQ = 16384;    // queries per head supported by this path

// Shared memory of the bucket kernel for a query list of up to `maxq` entries.
template <int D>
constexpr size_t annca_bucket_smem(int64_t maxq) {
  return sizeof(float) * ((size_t)kBP * (D + 4) + (size_t)kBQ * (D + 4) + kBQ + kBP) +
         sizeof(unsigned) * (size_t)kBP * kBMaxF + sizeof(int) * ((size_t)maxq + FASTAR_MAX_P + kBQ + 4);
}

template <typename T, int D>
__global__ void __launch_bounds__(256)
annca_bucket_kernel(const T* __restrict__ q, int64_t hs, int64_t ts, int F, int64_t tpf,
                    const int32_t* __restrict__ qb, int r, const T* __restrict__ kp,
                    const int32_t* __restrict__ pb, int64_t P, const BucketOrder bo, float* __restrict__ score) {
  extern __shared__ __align__(16) float sm_b[];
  constexpr int LD = D + 4;                       // padded row stride (floats)
  float* Ks = sm_b;                               // [kBP][LD]
  float* Qs = Ks + kBP * LD;                      // [kBQ][LD]
  float* qinv = Qs + kBQ * LD;                    // [kBQ]
  float* pinv = qinv + kBQ;                       // [kBP]
  unsigned* best = reinterpret_cast<unsigned*>(pinv + kBP);   // [kBP][kBMaxF] ordered floats
  int* plist = reinterpret_cast<int*>(best + kBP * kBMaxF);   // [FASTAR_MAX_P]
  int* qlist = plist + FASTAR_MAX_P;                           // [F * tpf], placed last
  int* qfr = qlist + F * tpf;                                  // [kBQ] frame of each chunk query
  int* cnt = qfr + kBQ;                                        // [0]: queries, [1]: prompt tokens
  const int tid = threadIdx.x;
  const int b = blockIdx.x, h = blockIdx.y;
  const int64_t nq = (int64_t)F * tpf;
  if (tid < 2) cnt[tid] = 0;
  __syncthreads();
  for (int64_t p = tid; p < P; p += blockDim.x)
    if (pb[(int64_t)h * P + p] == b) plist[atomicAdd(&cnt[1], 1)] = (int)p;
  __syncthreads();
  const int npb = cnt[1];
  if (npb == 0) return;   // no prompt token in this bucket (uniform across the CTA)
  if (bo.qperm) {
    // the bucket's (query, slot) pairs are one contiguous range of the sorted order
    const int32_t* qo = bo.qoff + (int64_t)h * (bo.B + 1);
    const int64_t beg = qo[b], end = qo[b + 1];
    const int64_t np = nq * r;
    for (int64_t pos = beg + tid; pos < end; pos += blockDim.x) {
      const int e = bo.qperm[(int64_t)h * np + pos];
      if (e >= 0 && e < np) qlist[atomicAdd(&cnt[0], 1)] = e / r;
    }
  } else {
    for (int64_t i = tid; i < nq; i += blockDim.x) {
      bool in = false;
      for (int s = 0; s < r; ++s) in |= qb[((int64_t)h * nq + i) * r + s] == b;
      if (in) qlist[atomicAdd(&cnt[0], 1)] = (int)i;
    }
  }
  __syncthreads();
  const int nqb = cnt[0];
  const unsigned kNegKey = float_to_ordered(neg_inf());
  for (int pc = 0; pc < npb; pc += kBP) {
    const int np = npb - pc < kBP ? npb - pc : kBP;
    __syncthreads();
    for (int idx = tid; idx < kBP * (D / 8); idx += blockDim.x) {
      const int row = idx / (D / 8), c8 = idx % (D / 8);
      float v[8];
      if (row < np) {
        load8(kp + ((int64_t)h * P + plist[pc + row]) * D + c8 * 8, v);
      } else {
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = 0.f;
      }
      *reinterpret_cast<float4*>(Ks + row * LD + c8 * 8) = make_float4(v[0], v[1], v[2], v[3]);
      *reinterpret_cast<float4*>(Ks + row * LD + c8 * 8 + 4) = make_float4(v[4], v[5], v[6], v[7]);
    }
    for (int idx = tid; idx < kBP * kBMaxF; idx += blockDim.x) best[idx] = kNegKey;
    __syncthreads();
    if (tid < kBP) {
      float ss = 0.f;
      for (int k = 0; k < D; ++k) ss = fmaf(Ks[tid * LD + k], Ks[tid * LD + k], ss);
      const float nrm = sqrtf(ss);
      pinv[tid] = nrm > 0.f ? 1.0f / nrm : 0.f;
    }
    for (int qc = 0; qc < nqb; qc += kBQ) {
      const int nqc = nqb - qc < kBQ ? nqb - qc : kBQ;
      __syncthreads();
      for (int idx = tid; idx < kBQ * (D / 8); idx += blockDim.x) {
        const int row = idx / (D / 8), c8 = idx % (D / 8);
        float v[8];
        if (row < nqc) {
          load8(q + h * hs + (int64_t)qlist[qc + row] * ts + c8 * 8, v);
        } else {
#pragma unroll
          for (int u = 0; u < 8; ++u) v[u] = 0.f;
        }
        *reinterpret_cast<float4*>(Qs + row * LD + c8 * 8) = make_float4(v[0], v[1], v[2], v[3]);
        *reinterpret_cast<float4*>(Qs + row * LD + c8 * 8 + 4) = make_float4(v[4], v[5], v[6], v[7]);
      }
      if (tid < kBQ) qfr[tid] = tid < nqc ? (int)(qlist[qc + tid] / tpf) : -1;
      __syncthreads();
      if (tid < kBQ) {
        float ss = 0.f;
        for (int k = 0; k < D; ++k) ss = fmaf(Qs[tid * LD + k], Qs[tid * LD + k], ss);
        const float nrm = sqrtf(ss);
        qinv[tid] = nrm > 0.f ? 1.0f / nrm : 0.f;
      }
      __syncthreads();
      // thread: prompt row pr, queries qg*8 .. qg*8+7
      const int pr = tid & (kBP - 1), qg = tid >> 5;
      float acc[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) acc[u] = 0.f;
#pragma unroll 4
      for (int k = 0; k < D; k += 4) {
        const float4 a = *reinterpret_cast<const float4*>(Ks + pr * LD + k);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float4 bq = *reinterpret_cast<const float4*>(Qs + (qg * 8 + u) * LD + k);
          acc[u] = fmaf(a.x, bq.x, acc[u]);
          acc[u] = fmaf(a.y, bq.y, acc[u]);
          acc[u] = fmaf(a.z, bq.z, acc[u]);
          acc[u] = fmaf(a.w, bq.w, acc[u]);
        }
      }
      if (pr < np) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int qi = qg * 8 + u;
          const int f = qfr[qi];
          if (qi < nqc && f >= 0 && f < kBMaxF)
            atomicMax(&best[pr * kBMaxF + f], float_to_ordered(acc[u] * qinv[qi]));
        }
      }
    }
    __syncthreads();
    for (int idx = tid; idx < np * F; idx += blockDim.x) {
      const int row = idx / F, f = idx % F;
      const unsigned key = best[row * kBMaxF + f];
      float sc = neg_inf();
      if (key != kNegKey) sc = ordered_to_float(key) * pinv[row];
      score[((int64_t)h * F + f) * P + plist[pc + row]] = sc;
    }
  }
}

template <typename T, int D>
static cudaError_t annca_impl(TokView q, int H, int F, int64_t tpf, const int32_t* qb, int r,
                              const void* kp, const int32_t* pb, int64_t P, int gate, const BucketOrder bo,
                              const float* qnorm, float* score, cudaStream_t s) {
  // bf16: the tensor-core scorer (dense Kp.Q^T with the bucket condition as a mask)
  if (sizeof(T) == 2 && gate &&
      launch_annca_tc(D, q, H, F, tpf, qb, r, kp, pb, P, bo.B > 0 ? bo.B : FASTAR_MAX_B, qnorm, score, nullptr, s))
    return cudaGetLastError();
  if (gate && F <= kBMaxF && (int64_t)F * tpf <= kBMaxQ && P <= FASTAR_MAX_P) {
    // prompt tokens whose bucket no CTA visits would keep stale scores: the bucket
    // kernel covers every p (each has exactly one bucket, and every bucket has a CTA)
    const size_t bsmem = annca_bucket_smem<D>((int64_t)F * tpf);
    const cudaError_t battr =
        opt_in_smem((const void*)annca_bucket_kernel<T, D>, (int)annca_bucket_smem<D>(kBMaxQ));
    if (battr != cudaSuccess) return battr;
    const unsigned nb = bo.B > 0 ? (unsigned)bo.B : (unsigned)FASTAR_MAX_B;
    annca_bucket_kernel<T, D><<<dim3(nb, H), 256, bsmem, s>>>(
        static_cast<const T*>(q.p), q.hs, q.ts, F, tpf, qb, r, static_cast<const T*>(kp), pb, P, bo, score);
    count_launches(1);
    return cudaGetLastError();
  }
  const size_t smem = sizeof(float) * ((size_t)D * kCQ + (size_t)D * kCP + kCQ + kCP + 16 * kCP) +
                      sizeof(int) * ((size_t)kCQ * FASTAR_MAX_R + kCP);
  auto kern = annca_score_kernel<T, D>;
  const cudaError_t attr = opt_in_smem((const void*)kern, (int)smem);
  if (attr != cudaSuccess) return attr;
  kern<<<dim3((unsigned)((P + kCP - 1) / kCP), H, F), 256, smem, s>>>(
      static_cast<const T*>(q.p), q.hs, q.ts, F, tpf, qb, r, static_cast<const T*>(kp), pb, P, gate, score);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_annca_select(int dtype, int d, TokView q, int H, int F, int64_t tpf, const int32_t* qb,
                                int r, const void* kp, const int32_t* pb, int64_t P, float tau_ca, int topk,
                                int gate, int B, const int32_t* qperm, const int32_t* qoff, const float* qnorm,
                                uint8_t* keep,
                                int32_t* kidx, int32_t* kcnt, float* score, const void* vp, void* kp_kept,
                                void* vp_kept, void* ws, cudaStream_t s) {
  if (H == 0 || F == 0) return cudaSuccess;
  float* sc = score ? score : static_cast<float*>(ws);
  cudaError_t e = cudaSuccess;
  const BucketOrder bo{B, qperm, qoff};
  if (P > 0) {
    if (dtype == FASTAR_BF16) {
      e = d == 128 ? annca_impl<__nv_bfloat16, 128>(q, H, F, tpf, qb, r, kp, pb, P, gate, bo, qnorm, sc, s)
                   : annca_impl<__nv_bfloat16, 64>(q, H, F, tpf, qb, r, kp, pb, P, gate, bo, qnorm, sc, s);
    } else {
      e = d == 128 ? annca_impl<float, 128>(q, H, F, tpf, qb, r, kp, pb, P, gate, bo, qnorm, sc, s)
                   : annca_impl<float, 64>(q, H, F, tpf, qb, r, kp, pb, P, gate, bo, qnorm, sc, s);
    }
    if (e != cudaSuccess) return e;
  }
  int threads = (int)((P + 31) / 32 * 32);
  if (threads < 32) threads = 32;
  KeptPlanes kpl{nullptr, nullptr, nullptr, nullptr, 0};
  unsigned copiers = 1;
  if (kp_kept && P > 0) {
    const int esize = dtype == FASTAR_BF16 ? 2 : 4;
    kpl = KeptPlanes{static_cast<const uint4*>(kp), static_cast<const uint4*>(vp), static_cast<uint4*>(kp_kept),
                     static_cast<uint4*>(vp_kept), d * esize / 16};
    copiers = 4;   // CTAs per (head, frame) sharing the copy of its kept rows
  }
  annca_rank_kernel<<<dim3((unsigned)(H * F), copiers), threads, 0, s>>>(F, P, tau_ca, topk, sc, keep, kidx, kcnt,
                                                                         kpl);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace fastar
