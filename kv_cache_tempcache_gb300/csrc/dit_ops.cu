// Row-wise operations of the transformer around the attention step (the Wan-1.3B-shaped
// DiT): layer norm with adaptive modulation, RMS norm with rotary positions, and the
// sinusoidal timestep embedding.  One warp per token row; rows of C <= 4096 channels are
// held in registers (C / 256 16-byte vectors per lane), statistics in fp32.
#include <climits>

#include "common.cuh"
#include "kernels.h"

namespace fastar {

namespace {

constexpr int kMaxV = 16;   // 16-byte vectors per lane: C <= 32 * 8 * 16 = 4096

__device__ __forceinline__ void unpack8(const uint4& u, float* f) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 t = __bfloat1622float2(h[e]);
    f[2 * e] = t.x;
    f[2 * e + 1] = t.y;
  }
}

__device__ __forceinline__ uint4 pack8(const float* f) {
  uint4 u;
  uint32_t* w = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * e], f[2 * e + 1]);
    w[e] = *reinterpret_cast<uint32_t*>(&h);
  }
  return u;
}

__device__ __forceinline__ float vsum(const float* a, const float* b, int i) {
  return (a ? a[i] : 0.f) + (b ? b[i] : 0.f);
}

// y = LN(x) [* w + b] then y * (1 + scale) + shift, scale = scale_a + scale_b, shift =
// shift_a + shift_b (any may be null).  Lane l owns vectors l, l + 32, ... (8 channels).
template <int NV>
__global__ void __launch_bounds__(256)
    layernorm_mod_kernel(const __nv_bfloat16* __restrict__ x, int64_t ldx, int64_t n, int C, float eps,
                         const float* __restrict__ w, const float* __restrict__ b, const float* shift_a,
                         const float* shift_b, const float* scale_a, const float* scale_b,
                         __nv_bfloat16* __restrict__ out, int64_t ldo) {
  const int64_t row = ((int64_t)blockIdx.x * 256 + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= n) return;
  const int nv = C / 8;
  float v[NV][8];
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int c8 = lane + 32 * k;
    if (c8 < nv) {
      unpack8(reinterpret_cast<const uint4*>(x + row * ldx)[c8], v[k]);
#pragma unroll
      for (int e = 0; e < 8; ++e) s += v[k][e];
    }
  }
  const float mean = warp_sum(s) / (float)C;
  float q = 0.f;
#pragma unroll
  for (int k = 0; k < NV; ++k)
    if (lane + 32 * k < nv)
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float dlt = v[k][e] - mean;
        q = fmaf(dlt, dlt, q);
      }
  const float rstd = rsqrtf(warp_sum(q) / (float)C + eps);
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int c8 = lane + 32 * k;
    if (c8 >= nv) continue;
    float y[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int c = c8 * 8 + e;
      float t = (v[k][e] - mean) * rstd;
      if (w) t = fmaf(t, w[c], b ? b[c] : 0.f);
      const float sc = vsum(scale_a, scale_b, c), sh = vsum(shift_a, shift_b, c);
      y[e] = fmaf(t, 1.0f + sc, sh);
    }
    reinterpret_cast<uint4*>(out + row * ldo)[c8] = pack8(y);
  }
}

// In place on a token-major row of C = H * d channels: optional RMS norm over the whole
// row (x / sqrt(mean x^2 + eps) * w), then optional rotary positions per head: the head
// dimension splits into frame / row / column parts of dt = d - 4 (d / 6), dh = dw = 2 (d / 6)
// channels; within a part of width da, the pair (2j, 2j + 1) turns by pos * theta^(-2j/da).
// Token i of the chunk sits at frame t0 + i / (gh gw), row (i / gw) % gh, column i % gw.
template <int NV>
__global__ void __launch_bounds__(256)
    rmsnorm_rope_kernel(__nv_bfloat16* __restrict__ x, int64_t ldx, int64_t n, int C, int d, float eps,
                        const float* __restrict__ w, int rope, int t0, const int32_t* t0_dev, int gh, int gw,
                        float theta) {
  const int64_t row = ((int64_t)blockIdx.x * 256 + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= n) return;
  const int nv = C / 8;
  float v[NV][8];
  float q = 0.f;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int c8 = lane + 32 * k;
    if (c8 < nv) {
      unpack8(reinterpret_cast<const uint4*>(x + row * ldx)[c8], v[k]);
#pragma unroll
      for (int e = 0; e < 8; ++e) q = fmaf(v[k][e], v[k][e], q);
    }
  }
  const float r = w ? rsqrtf(warp_sum(q) / (float)C + eps) : 1.f;
  const int f0 = t0 + (t0_dev ? t0_dev[0] : 0);   // a device offset keeps replayed graphs current
  const int pos[3] = {f0 + (int)(row / ((int64_t)gh * gw)), (int)((row / gw) % gh), (int)(row % gw)};
  const int part = 2 * (d / 6);
  const int dt = d - 2 * part;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int c8 = lane + 32 * k;
    if (c8 >= nv) continue;
    float y[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) y[e] = w ? v[k][e] * r * w[c8 * 8 + e] : v[k][e];
    if (rope) {
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        const int cin = (c8 * 8 + e) % d;   // even channel of the pair inside its head
        int axis, j, da;
        if (cin < dt) {
          axis = 0, j = cin / 2, da = dt;
        } else if (cin < dt + part) {
          axis = 1, j = (cin - dt) / 2, da = part;
        } else {
          axis = 2, j = (cin - dt - part) / 2, da = part;
        }
        const float ang = (float)pos[axis] * powf(theta, -2.0f * (float)j / (float)da);
        float sn, cs;
        sincosf(ang, &sn, &cs);
        const float a0 = y[e], a1 = y[e + 1];
        y[e] = a0 * cs - a1 * sn;
        y[e + 1] = a0 * sn + a1 * cs;
      }
    }
    reinterpret_cast<uint4*>(x + row * ldx)[c8] = pack8(y);
  }
}

// out[b, i] = cos(t_b f_i) and out[b, half + i] = sin(t_b f_i), f_i = 10000^(-i / half).
__global__ void sinusoidal_kernel(const float* __restrict__ t, int nb, int dim, __nv_bfloat16* __restrict__ out,
                                  int64_t ldo) {
  const int half = dim / 2;
  const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= (int64_t)nb * half) return;
  const int bi = (int)(g / half), i = (int)(g % half);
  const float a = t[bi] * powf(10000.0f, -(float)i / (float)half);
  float sn, cs;
  sincosf(a, &sn, &cs);
  out[bi * ldo + i] = __float2bfloat16_rn(cs);
  out[bi * ldo + half + i] = __float2bfloat16_rn(sn);
}

template <int NV>
cudaError_t ln_impl(const void* x, int64_t ldx, int64_t n, int C, float eps, const float* w, const float* b,
                    const float* sha, const float* shb, const float* sca, const float* scb, void* out, int64_t ldo,
                    cudaStream_t s) {
  const int64_t blocks = (n * 32 + 255) / 256;
  layernorm_mod_kernel<NV><<<(unsigned)blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(x), ldx, n, C, eps, w,
                                                            b, sha, shb, sca, scb,
                                                            static_cast<__nv_bfloat16*>(out), ldo);
  count_launches(1);
  return cudaGetLastError();
}

template <int NV>
cudaError_t rope_impl(void* x, int64_t ldx, int64_t n, int C, int d, float eps, const float* w, int rope, int t0,
                      const int32_t* t0_dev, int gh, int gw, float theta, cudaStream_t s) {
  const int64_t blocks = (n * 32 + 255) / 256;
  rmsnorm_rope_kernel<NV><<<(unsigned)blocks, 256, 0, s>>>(static_cast<__nv_bfloat16*>(x), ldx, n, C, d, eps, w,
                                                           rope, t0, t0_dev, gh, gw, theta);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_layernorm_mod(const void* x, int64_t ldx, int64_t n, int C, float eps, const float* w,
                                 const float* b, const float* sha, const float* shb, const float* sca,
                                 const float* scb, void* out, int64_t ldo, cudaStream_t s) {
  const int nv = (C / 8 + 31) / 32;
  if (nv <= 2) return ln_impl<2>(x, ldx, n, C, eps, w, b, sha, shb, sca, scb, out, ldo, s);
  if (nv <= 6) return ln_impl<6>(x, ldx, n, C, eps, w, b, sha, shb, sca, scb, out, ldo, s);
  return ln_impl<kMaxV>(x, ldx, n, C, eps, w, b, sha, shb, sca, scb, out, ldo, s);
}

cudaError_t launch_rmsnorm_rope(void* x, int64_t ldx, int64_t n, int C, int d, float eps, const float* w, int rope,
                                int t0, const int32_t* t0_dev, int gh, int gw, float theta, cudaStream_t s) {
  const int nv = (C / 8 + 31) / 32;
  if (nv <= 2) return rope_impl<2>(x, ldx, n, C, d, eps, w, rope, t0, t0_dev, gh, gw, theta, s);
  if (nv <= 6) return rope_impl<6>(x, ldx, n, C, d, eps, w, rope, t0, t0_dev, gh, gw, theta, s);
  return rope_impl<kMaxV>(x, ldx, n, C, d, eps, w, rope, t0, t0_dev, gh, gw, theta, s);
}

cudaError_t launch_sinusoidal(const float* t, int nb, int dim, void* out, int64_t ldo, cudaStream_t s) {
  const int64_t total = (int64_t)nb * (dim / 2);
  sinusoidal_kernel<<<(unsigned)((total + 255) / 256), 256, 0, s>>>(t, nb, dim, static_cast<__nv_bfloat16*>(out),
                                                                      ldo);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace fastar
