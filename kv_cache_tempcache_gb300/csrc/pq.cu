// Product quantization for the quantization variant of the TempCache match (FAST-AR
// technical summary §2.A: the top-1 correspondence is searched with a lightweight ANN,
// "LSH or Quantization").
//
// A key of dimension d is m consecutive sub-vectors of DS = d/m elements; each is
// replaced by the nearest (smallest squared Euclidean distance, lowest index on ties) of
// the Kc codewords of its sub-space.  Codebooks are per head, [H, m, Kc, DS].
//
//   pq_encode_kernel   a block per 64 keys, its 8 warps splitting the m sub-spaces (two keys
//                      per lane, packed f32x2 arithmetic); the head's codebook staged in
//                      shared memory as fp32 (every lane of a warp reads the same codeword:
//                      a broadcast); the one-byte codes staged and written as 32-bit words;
//   pq_decode_kernel   the head's codebook in shared memory; a warp decodes four cached
//                      keys per round (their code loads issued together): lane s writes
//                      sub-vector s (bf16, exactly the codeword), the warp reduces |k^|;
//   pq_gather_codes    the codes follow the cache through a compaction (its index map).
// The match itself is the tensor-core match over the decoded keys (match.cu).
#include <climits>
#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "tmap.h"

namespace fastar {

namespace {

constexpr int kEncKeys = 64;    // keys per encode block (each of its 8 warps: all 64 keys, m/8 sub-spaces)

// (a.x, a.y) - (b, b) and acc + d * d, two lanes of fp32 per instruction (PTX f32x2).
__device__ __forceinline__ unsigned long long pack2(float x, float y) {
  return (unsigned long long)__float_as_uint(x) | ((unsigned long long)__float_as_uint(y) << 32);
}
__device__ __forceinline__ unsigned long long sub2(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b, unsigned long long c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

template <typename T, int DS>
__global__ void __launch_bounds__(256)
    pq_encode_kernel(TokView x, int64_t n, int m, int Kc, const T* __restrict__ cb, uint8_t* __restrict__ codes) {
  // shared memory: the head's codebook [m][Kc][DS] (fp32), the block's key rows
  // [kEncKeys][d + 4] (fp32; the 4-float pad spreads a warp's row reads over all banks),
  // then the block's codes [kEncKeys][m]
  extern __shared__ __align__(16) float cbs[];
  const int d = m * DS, xstride = d + 4;
  float* xs = cbs + m * Kc * DS;
  uint8_t* cs = reinterpret_cast<uint8_t*>(xs + kEncKeys * xstride);
  const int h = blockIdx.y;
  const int64_t t0 = (int64_t)blockIdx.x * kEncKeys;
  const T* cbh = cb + (int64_t)h * m * Kc * DS;
  for (int i = threadIdx.x; i < m * Kc * DS; i += 256) cbs[i] = to_f(cbh[i]);
  // the key rows with coalesced 8-element loads (rows past n read as zero)
  for (int i = threadIdx.x; i < kEncKeys * d / 8; i += 256) {
    const int row = i / (d / 8), c8 = i % (d / 8);
    float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (t0 + row < n) load8(static_cast<const T*>(x.p) + h * x.hs + (t0 + row) * x.ts + c8 * 8, v);
    float4* dst = reinterpret_cast<float4*>(xs + row * xstride + c8 * 8);
    dst[0] = make_float4(v[0], v[1], v[2], v[3]);
    dst[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // every lane takes two keys (rows lane and lane + 32), packed into the two halves of
  // f32x2 operations; the block's 8 warps split the sub-spaces, so all lanes of a warp
  // read the same codeword (a shared-memory broadcast)
  const float* xa = xs + lane * xstride;
  const float* xb = xs + (lane + 32) * xstride;
  for (int s = warp; s < m; s += 8) {
    float va[DS], vb[DS];
#pragma unroll
    for (int e = 0; e < DS; e += 4) {
      const float4 a = *reinterpret_cast<const float4*>(xa + s * DS + e);
      const float4 b = *reinterpret_cast<const float4*>(xb + s * DS + e);
      va[e] = a.x; va[e + 1] = a.y; va[e + 2] = a.z; va[e + 3] = a.w;
      vb[e] = b.x; vb[e + 1] = b.y; vb[e + 2] = b.z; vb[e + 3] = b.w;
    }
    unsigned long long v2[DS];
#pragma unroll
    for (int e = 0; e < DS; ++e) v2[e] = pack2(va[e], vb[e]);
    const float4* c4 = reinterpret_cast<const float4*>(cbs + s * Kc * DS);
    float best_a = __int_as_float(0x7f800000u), best_b = best_a;
    int arg_a = 0, arg_b = 0;
#pragma unroll 4
    for (int k = 0; k < Kc; ++k) {
      unsigned long long acc = 0ull;
#pragma unroll
      for (int e4 = 0; e4 < DS / 4; ++e4) {
        const float4 c = c4[k * (DS / 4) + e4];
        const float ce[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const unsigned long long df = sub2(v2[e4 * 4 + e], pack2(ce[e], ce[e]));
          acc = fma2(df, df, acc);
        }
      }
      const float da = __uint_as_float((unsigned)(acc & 0xffffffffull));
      const float db = __uint_as_float((unsigned)(acc >> 32));
      // strict: the lowest index keeps a tie
      arg_a = da < best_a ? k : arg_a;
      best_a = da < best_a ? da : best_a;
      arg_b = db < best_b ? k : arg_b;
      best_b = db < best_b ? db : best_b;
    }
    cs[lane * m + s] = (uint8_t)arg_a;
    cs[(lane + 32) * m + s] = (uint8_t)arg_b;
  }
  __syncthreads();
  // the block's codes leave as 32-bit words (rows of m bytes, m a multiple of 4)
  const int64_t keys = n - t0 < kEncKeys ? n - t0 : kEncKeys;
  const int words = (int)keys * m / 4;
  uint32_t* out = reinterpret_cast<uint32_t*>(codes + ((int64_t)h * n + t0) * m);
  const uint32_t* in = reinterpret_cast<const uint32_t*>(cs);
  for (int i = threadIdx.x; i < words; i += 256) out[i] = in[i];
}

constexpr int kDecKeys = 4;     // keys per warp and round of the decode (their loads issued together)

template <int DS>
__global__ void __launch_bounds__(256)
    pq_decode_kernel(int H, int64_t M, int m, int Kc, const uint8_t* __restrict__ codes,
                     const int32_t* __restrict__ clen, const __nv_bfloat16* __restrict__ cb,
                     __nv_bfloat16* __restrict__ khat, float* __restrict__ khat_norm, int32_t* status) {
  // grid (blocks, H): the head's codebook in shared memory (bf16, as stored); each warp
  // decodes kDecKeys keys per round, lane s writing sub-vector s of each (m <= 32)
  using Vec = typename std::conditional<DS == 4, uint2, uint4>::type;
  extern __shared__ __align__(16) uint8_t cbsm[];
  const Vec* cbv = reinterpret_cast<const Vec*>(cbsm);   // [m][Kc] sub-vectors
  const int h = blockIdx.y;
  {
    const uint4* src = reinterpret_cast<const uint4*>(cb + (int64_t)h * m * Kc * DS);
    uint4* dst = reinterpret_cast<uint4*>(cbsm);
    for (int i = threadIdx.x; i < m * Kc * DS * 2 / 16; i += 256) dst[i] = src[i];
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  int64_t n = clen[h];
  n = n < 0 ? 0 : (n > M ? M : n);
  const int d = m * DS;
  const int64_t step = (int64_t)gridDim.x * 8 * kDecKeys;
  for (int64_t j0 = ((int64_t)blockIdx.x * 8 + (threadIdx.x >> 5)) * kDecKeys; j0 < M; j0 += step) {
    int c[kDecKeys];
#pragma unroll
    for (int u = 0; u < kDecKeys; ++u) {
      const int64_t j = j0 + u;
      c[u] = (lane < m && j < n) ? codes[((int64_t)h * M + j) * m + lane] : -1;
    }
#pragma unroll
    for (int u = 0; u < kDecKeys; ++u) {
      const int64_t j = j0 + u;
      if (j >= M) break;
      Vec v = Vec();
      if (c[u] >= Kc) {
        flag_status(status, FASTAR_DEV_BAD_INDEX);
        c[u] = 0;
      }
      if (c[u] >= 0) v = cbv[lane * Kc + c[u]];
      float ss = 0.f;
      const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
      for (int e = 0; e < DS / 2; ++e) {
        const float2 f = __bfloat1622float2(p2[e]);
        ss = fmaf(f.x, f.x, ss);
        ss = fmaf(f.y, f.y, ss);
      }
      const int64_t w = (int64_t)h * M + j;
      if (lane < m) *reinterpret_cast<Vec*>(khat + w * d + lane * DS) = v;
      ss = warp_sum(ss);
      if (lane == 0) khat_norm[w] = sqrtf(ss);
    }
  }
}

__global__ void __launch_bounds__(256)
    pq_gather_codes_kernel(int H, int64_t nq, int64_t M, int words, const uint32_t* __restrict__ codes_in,
                           const int32_t* __restrict__ len_in, const uint32_t* __restrict__ codes_cur,
                           const int32_t* __restrict__ imap, const int32_t* __restrict__ len_out,
                           uint32_t* __restrict__ codes_out, int32_t* status) {
  const int64_t total = (int64_t)H * M * words;
  for (int64_t g = (int64_t)blockIdx.x * 256 + threadIdx.x; g < total; g += (int64_t)gridDim.x * 256) {
    const int64_t row = g / words;
    const int c = (int)(g % words);
    const int h = (int)(row / M);
    const int64_t slot = row - (int64_t)h * M;
    if (slot >= len_out[h]) continue;
    int64_t n = len_in[h];
    n = n < 0 ? 0 : (n > M ? M : n);
    const int64_t src = imap[row];
    if (src >= 0 && src < n) {
      codes_out[g] = codes_in[((int64_t)h * M + src) * words + c];
    } else if (src >= n && src < n + nq) {
      codes_out[g] = codes_cur[((int64_t)h * nq + (src - n)) * words + c];
    } else if (c == 0) {
      flag_status(status, FASTAR_DEV_BAD_INDEX);
    }
  }
}

template <typename T, int DS>
cudaError_t encode_impl(TokView x, int H, int64_t n, int m, int Kc, const void* cb, uint8_t* codes, cudaStream_t s) {
  const size_t smem =
      sizeof(float) * ((size_t)m * Kc * DS + (size_t)kEncKeys * (m * DS + 4)) + (size_t)kEncKeys * m;
  auto kern = pq_encode_kernel<T, DS>;
  if (smem > 48 * 1024) {
    const cudaError_t e = opt_in_smem((const void*)kern, (int)smem);
    if (e != cudaSuccess) return e;
  }
  const dim3 grid((unsigned)((n + kEncKeys - 1) / kEncKeys), (unsigned)H);
  kern<<<grid, 256, smem, s>>>(x, n, m, Kc, static_cast<const T*>(cb), codes);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_pq_encode(int dtype, int d, TokView x, int H, int64_t n, int m, int Kc, const void* cb,
                             uint8_t* codes, cudaStream_t s) {
  const int ds = d / m;
  if (dtype == FASTAR_BF16)
    return ds == 4 ? encode_impl<__nv_bfloat16, 4>(x, H, n, m, Kc, cb, codes, s)
                   : encode_impl<__nv_bfloat16, 8>(x, H, n, m, Kc, cb, codes, s);
  return ds == 4 ? encode_impl<float, 4>(x, H, n, m, Kc, cb, codes, s)
                 : encode_impl<float, 8>(x, H, n, m, Kc, cb, codes, s);
}

cudaError_t launch_pq_decode(int d, int H, int64_t M, int m, int Kc, const uint8_t* codes, const int32_t* clen,
                             const void* cb, void* khat, float* khat_norm, int32_t* status, cudaStream_t s) {
  // m <= 32 sub-spaces (one lane each); about 152 x 4 blocks in all, over the heads
  const size_t smem = (size_t)m * Kc * (d / m) * 2;
  int64_t per_head = (152 * 4 + H - 1) / H;
  const int64_t need = (M + 8 * kDecKeys - 1) / (8 * kDecKeys);
  if (per_head > need) per_head = need;
  if (per_head < 1) per_head = 1;
  const dim3 blocks((unsigned)per_head, (unsigned)H);
  const __nv_bfloat16* c = static_cast<const __nv_bfloat16*>(cb);
  __nv_bfloat16* k = static_cast<__nv_bfloat16*>(khat);
  cudaError_t e;
  if (d / m == 4) {
    if (smem > 48 * 1024 &&
        (e = opt_in_smem((const void*)pq_decode_kernel<4>, (int)smem)) != cudaSuccess)
      return e;
    pq_decode_kernel<4><<<blocks, 256, smem, s>>>(H, M, m, Kc, codes, clen, c, k, khat_norm, status);
  } else {
    if (smem > 48 * 1024 &&
        (e = opt_in_smem((const void*)pq_decode_kernel<8>, (int)smem)) != cudaSuccess)
      return e;
    pq_decode_kernel<8><<<blocks, 256, smem, s>>>(H, M, m, Kc, codes, clen, c, k, khat_norm, status);
  }
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_pq_gather_codes(int H, int64_t nq, int64_t M, int m, const uint8_t* codes_in,
                                   const int32_t* len_in, const uint8_t* codes_cur, const int32_t* imap,
                                   const int32_t* len_out, uint8_t* codes_out, int32_t* status, cudaStream_t s) {
  const int words = m / 4;
  int64_t blocks = ((int64_t)H * M * words + 255) / 256;
  if (blocks > 152 * 8) blocks = 152 * 8;
  if (blocks < 1) blocks = 1;
  pq_gather_codes_kernel<<<(unsigned)blocks, 256, 0, s>>>(
      H, nq, M, words, reinterpret_cast<const uint32_t*>(codes_in), len_in,
      reinterpret_cast<const uint32_t*>(codes_cur), imap, len_out, reinterpret_cast<uint32_t*>(codes_out), status);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace fastar
