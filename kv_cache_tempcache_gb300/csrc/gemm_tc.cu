// Dense bf16 GEMM on the 5th-generation tensor cores for the transformer around the
// attention step (the Wan-1.3B-shaped DiT: projections, FFN, embeddings):
//
//   C[m, n] = epilogue( sum_k A[m, k] W[n, k] ),  A [M, K], W [N, K] row-major bf16, C [M, N]
//   row-major bf16 (or fp32)
//   epilogue: v = acc + bias[n];  v = act(v)  (none, GELU with the tanh form, SiLU);
//             with a residual: v = R[m, n] + (gate_a[n] + gate_b[n]) * v  (gates optional,
//             a missing gate counts as 1 / 0 as documented in the header).
//
// One persistent CTA per SM, warp-specialised:
//   warp 0      TMA producer: 128 x 64 tiles of A and 256 x 64 tiles of W through a
//               4-stage shared-memory ring (128-byte swizzle);
//   warp 1      owns TMEM (2 accumulator stages x 256 fp32 columns) and issues
//               tcgen05.mma (M = 128, N = 256, K = 16) from one thread;
//   warps 2..9  epilogue: each reads 32 rows x 128 columns of the accumulator (its TMEM
//               lane quadrant, its column half), hands the stage back, applies the
//               epilogue in fp32 and stores bf16 rows with 16-byte writes.
// Output tiles are taken round-robin (M fastest, so CTAs in flight share W tiles in L2).
// Every wait is bounded; a timeout sets FASTAR_DEV_TIMEOUT and unwinds.
#include <climits>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"
#include "tmap.h"

namespace fastar {

namespace {

constexpr int kBM = 128, kBN = 256, kBK = 64, kGS = 4;
constexpr int kEpiW = 8;
constexpr int kThreadsG = (2 + kEpiW) * 32;
constexpr int kABytes = kBM * kBK * 2;   // 16 KB
constexpr int kBBytes = kBN * kBK * 2;   // 32 KB

struct alignas(1024) GemmSmem {
  uint8_t a[kGS][kABytes];
  uint8_t b[kGS][kBBytes];
  uint64_t full[kGS], empty[kGS];
  uint64_t acc_full[2], acc_empty[2];
  uint32_t tmem_base;
  int abort;
};

struct GemmArgs {
  int64_t M, N, K;
  const float* bias;
  const __nv_bfloat16* res;
  int64_t ldr;
  const float* gate_a;
  const float* gate_b;
  void* C;
  int64_t ldc;
  int c_f32;   // C is fp32 instead of bf16
  int act;
  int32_t* status;
};

__device__ __forceinline__ float act_fn(float v, int act) {
  if (act == FASTAR_ACT_GELU_TANH) {
    // 0.5 v (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3)))
    const float u = 0.7978845608028654f * fmaf(0.044715f * v, v * v, v);
    return 0.5f * v * (1.0f + tanhf(u));
  }
  if (act == FASTAR_ACT_SILU) return v / (1.0f + __expf(-v));
  return v;
}

__global__ void __launch_bounds__(kThreadsG, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_w,
                   const GemmArgs g) {
  extern __shared__ uint8_t smem_raw[];
  GemmSmem& sm = *reinterpret_cast<GemmSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int MT = (int)((g.M + kBM - 1) / kBM), NT = (int)(g.N / kBN), KT = (int)(g.K / kBK);
  const int tiles = MT * NT;
  constexpr uint32_t kIdesc = tc::idesc_bf16_f32(kBM, kBN);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGS; ++s) {
      tc::mbar_init(&sm.full[s], 1);
      tc::mbar_init(&sm.empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&sm.acc_full[s], 1);
      tc::mbar_init(&sm.acc_empty[s], kEpiW);
    }
    sm.abort = 0;
    tc::mbar_fence_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(&sm.tmem_base, 512);
    tc::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tc::tma_prefetch_desc(&tm_a);
    tc::tma_prefetch_desc(&tm_w);
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort = &sm.abort;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int stage = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        const int tm = t % MT, tn = t / MT;
        for (int kb = 0; kb < KT; ++kb) {
          if (!tc::mbar_wait(&sm.empty[stage], ph ^ 1, abort)) {
            ok = false;
            break;
          }
          tc::mbar_arrive_tx(&sm.full[stage], (uint32_t)(kABytes + kBBytes));
          tc::tma_load_3d(sm.a[stage], &tm_a, kb * kBK, tm * kBM, 0, &sm.full[stage]);
          tc::tma_load_3d(sm.b[stage], &tm_w, kb * kBK, tn * kBN, 0, &sm.full[stage]);
          if (++stage == kGS) {
            stage = 0;
            ph ^= 1;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      int stage = 0, acc = 0;
      uint32_t ph = 0, aph = 0;
      bool ok = true;
      const uint64_t a0 = tc::sw128_desc(tc::smem_u32(sm.a[0]));
      const uint64_t b0 = tc::sw128_desc(tc::smem_u32(sm.b[0]));
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        if (!tc::mbar_wait(&sm.acc_empty[acc], aph ^ 1, abort)) break;
        tc::tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(acc * kBN);
        for (int kb = 0; kb < KT; ++kb) {
          if (!tc::mbar_wait(&sm.full[stage], ph, abort)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            const uint64_t ad = a0 + (uint64_t)((stage * kABytes + k * 32) >> 4);
            const uint64_t bd = b0 + (uint64_t)((stage * kBBytes + k * 32) >> 4);
            tc::mma_bf16(d, ad, bd, kIdesc, (kb > 0 || k > 0) ? 1u : 0u);
          }
          tc::mma_commit(&sm.empty[stage]);
          if (++stage == kGS) {
            stage = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
        tc::mma_commit(&sm.acc_full[acc]);
        if (++acc == 2) {
          acc = 0;
          aph ^= 1;
        }
      }
    }
  } else {
    // ---------------- epilogue ----------------
    const int quad = warp & 3;              // the TMEM lane quadrant this warp may read
    const int half = (warp - 2) >> 2;       // which 128 columns of the 256-column tile
    const int row = quad * 32 + lane;
    int acc = 0;
    uint32_t aph = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
      const int tm = t % MT, tn = t / MT;
      if (!tc::mbar_wait(&sm.acc_full[acc], aph, abort)) break;
      tc::tc_fence_after();
      const int64_t m = (int64_t)tm * kBM + row;
      const int64_t n0 = (int64_t)tn * kBN + half * 128;
      const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(acc * kBN + half * 128);
      // two passes of 64 columns (64 registers of scores at a time); the accumulator
      // stage is handed back once the second pass's scores are in registers
#pragma unroll 1
      for (int pass = 0; pass < 2; ++pass) {
        float v[2][32];
        __syncwarp();   // the TMEM loads are warp-collective: every lane, converged
        tc::tmem_ld32(taddr + (uint32_t)(pass * 64), v[0]);
        tc::tmem_ld32(taddr + (uint32_t)(pass * 64 + 32), v[1]);
        tc::tmem_wait_ld();
        tc::tmem_pin32(v[0]);
        tc::tmem_pin32(v[1]);
        if (pass == 1) {
          tc::tc_fence_before();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&sm.acc_empty[acc]);
        }
#pragma unroll
        for (int c = 0; c < 2 && m < g.M; ++c) {   // rows past M: nothing to store
          const int64_t nc = n0 + pass * 64 + c * 32;
          float r[32];
          if (g.res) {
            const uint4* rp = reinterpret_cast<const uint4*>(g.res + m * g.ldr + nc);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint4 u = rp[q];
              const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 f = __bfloat1622float2(h2[e]);
                r[q * 8 + 2 * e] = f.x;
                r[q * 8 + 2 * e + 1] = f.y;
              }
            }
          }
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            float x0 = v[c][i], x1 = v[c][i + 1];
            if (g.bias) {
              x0 += g.bias[nc + i];
              x1 += g.bias[nc + i + 1];
            }
            x0 = act_fn(x0, g.act);
            x1 = act_fn(x1, g.act);
            if (g.res) {
              float g0 = 1.f, g1 = 1.f;
              if (g.gate_a) {
                g0 = g.gate_a[nc + i] + (g.gate_b ? g.gate_b[nc + i] : 0.f);
                g1 = g.gate_a[nc + i + 1] + (g.gate_b ? g.gate_b[nc + i + 1] : 0.f);
              }
              x0 = fmaf(g0, x0, r[i]);
              x1 = fmaf(g1, x1, r[i + 1]);
            }
            if (g.c_f32) {
              *reinterpret_cast<float2*>(static_cast<float*>(g.C) + m * g.ldc + nc + i) = make_float2(x0, x1);
            } else {
              __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
              pk[i >> 1] = *reinterpret_cast<uint32_t*>(&h);
            }
          }
          if (!g.c_f32) {
            uint4* cp = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(g.C) + m * g.ldc + nc);
#pragma unroll
            for (int q = 0; q < 4; ++q) cp[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
          }
        }
      }
      if (++acc == 2) {
        acc = 0;
        aph ^= 1;
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && sm.abort) flag_status(g.status, FASTAR_DEV_TIMEOUT);
}

}  // namespace

cudaError_t launch_gemm_tc(const void* A, int64_t lda, const void* W, int64_t ldw, const float* bias,
                           const void* res, int64_t ldr, const float* gate_a, const float* gate_b, void* C, int64_t ldc,
                           int c_f32, int64_t M, int64_t N, int64_t K, int act, int32_t* status, cudaStream_t s) {
  constexpr size_t smem = sizeof(GemmSmem) + 1024;
  static const cudaError_t attr =
      cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (attr != cudaSuccess) return attr;
  CUtensorMap ta, tw;
  if (!make_tmap_bf16_3d(&ta, A, (uint64_t)K, (uint64_t)M, 1, (uint64_t)lda * 2, 0, kBK, kBM) ||
      !make_tmap_bf16_3d(&tw, W, (uint64_t)K, (uint64_t)N, 1, (uint64_t)ldw * 2, 0, kBK, kBN))
    return cudaErrorInvalidValue;
  GemmArgs g;
  g.M = M;
  g.N = N;
  g.K = K;
  g.bias = bias;
  g.res = static_cast<const __nv_bfloat16*>(res);
  g.ldr = ldr;
  g.gate_a = gate_a;
  g.gate_b = gate_b;
  g.C = C;
  g.ldc = ldc;
  g.c_f32 = c_f32;
  g.act = act;
  g.status = status;
  const int64_t tiles = ((M + kBM - 1) / kBM) * (N / kBN);
  const int grid = (int)(tiles < sm_count() ? tiles : sm_count());
  gemm_tc_kernel<<<grid, kThreadsG, smem, s>>>(ta, tw, g);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace fastar
