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

// The 8 fp32 values of a vector starting at channel c (16-byte aligned), or zeros.
__device__ __forceinline__ void load8f(const float* p, int c, float* f) {
  if (!p) {
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] = 0.f;
    return;
  }
  const float4 x = reinterpret_cast<const float4*>(p + c)[0], y = reinterpret_cast<const float4*>(p + c)[1];
  f[0] = x.x, f[1] = x.y, f[2] = x.z, f[3] = x.w, f[4] = y.x, f[5] = y.y, f[6] = y.z, f[7] = y.w;
}

// y = LN(x) [* w + b] then y * (1 + scale) + shift, scale = scale_a + scale_b, shift =
// shift_a + shift_b (any may be null).  Lane l owns vectors l, l + 32, ... (8 channels);
// the per-channel vectors are read 16 bytes at a time (they are 16-byte aligned).
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
    float y[8], p0[8], p1[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) y[e] = (v[k][e] - mean) * rstd;
    if (w) {
      load8f(w, c8 * 8, p0);
      load8f(b, c8 * 8, p1);
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] = fmaf(y[e], p0[e], p1[e]);
    }
    if (scale_a || scale_b || shift_a || shift_b) {
      float q0[8], q1[8];
      load8f(scale_a, c8 * 8, p0);
      load8f(scale_b, c8 * 8, p1);
      load8f(shift_a, c8 * 8, q0);
      load8f(shift_b, c8 * 8, q1);
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] = fmaf(y[e], 1.0f + (p0[e] + p1[e]), q0[e] + q1[e]);
    }
    reinterpret_cast<uint4*>(out + row * ldo)[c8] = pack8(y);
  }
}

// The rotation of the channel pair (cin, cin + 1) inside a head of width d: the head
// splits into frame / row / column parts of dt = d - 4 (d / 6), dh = dw = 2 (d / 6) channels;
// within a part of width da, the pair (2j, 2j + 1) turns by pos * theta^(-2j/da).
__device__ __forceinline__ void rope_angle(int cin, int d, int pf, int ph, int pw, float theta, float& sn,
                                           float& cs) {
  const int part = 2 * (d / 6);
  const int dt = d - 2 * part;
  int p, j, da;
  if (cin < dt) {
    p = pf, j = cin / 2, da = dt;
  } else if (cin < dt + part) {
    p = ph, j = (cin - dt) / 2, da = part;
  } else {
    p = pw, j = (cin - dt - part) / 2, da = part;
  }
  const float ang = (float)p * powf(theta, -2.0f * (float)j / (float)da);
  sincosf(ang, &sn, &cs);
}

// In place on a token-major row of C = H * d channels: optional RMS norm over the whole
// row (x / sqrt(mean x^2 + eps) * w), then optional rotary positions per head (rope_angle).
// Token i of the chunk sits at frame t0 + i / (gh gw), row (i / gw) % gh, column i % gw.
// Lane l owns vectors l + 32 k; when d divides 256 their channels sit at the same offsets
// inside their heads for every k, so the lane's four rotations are computed once per row.
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
  const int pf = f0 + (int)(row / ((int64_t)gh * gw)), ph = (int)((row / gw) % gh), pw = (int)(row % gw);
  const bool shared_rot = (256 % d) == 0;
  float sn[4], cs[4];
  if (rope && shared_rot) {
#pragma unroll
    for (int e = 0; e < 4; ++e) rope_angle((8 * lane) % d + 2 * e, d, pf, ph, pw, theta, sn[e], cs[e]);
  }
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int c8 = lane + 32 * k;
    if (c8 >= nv) continue;
    float y[8];
    if (w) {
      float wv[8];
      load8f(w, c8 * 8, wv);
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] = v[k][e] * r * wv[e];
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] = v[k][e];
    }
    if (rope) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (!shared_rot) rope_angle((c8 * 8 + 2 * e) % d, d, pf, ph, pw, theta, sn[e], cs[e]);
        const float a0 = y[2 * e], a1 = y[2 * e + 1];
        y[2 * e] = a0 * cs[e] - a1 * sn[e];
        y[2 * e + 1] = a0 * sn[e] + a1 * cs[e];
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
