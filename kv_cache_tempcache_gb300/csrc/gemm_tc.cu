// Dense bf16 GEMM on the 5th-generation tensor cores for the transformer around the
// attention step (the Wan-1.3B-shaped DiT: projections, FFN, embeddings):
//
//   C[m, n] = epilogue( sum_k A[m, k] W[n, k] ),  A [M, K], W [N, K] row-major bf16, C [M, N]
//   row-major bf16 (or fp32)
//   epilogue: v = acc + bias[n];  v = act(v)  (none, GELU with the tanh form, SiLU; one
//             kernel instance per activation);
//             with a residual: v = R[m, n] + (gate_a[n] + gate_b[n]) * v  (gates optional,
//             a missing gate counts as 1 / 0 as documented in the header).
//
// One persistent CTA per SM, warp-specialised, output tiles of 128 x BN (BN = 256, or 128
// when 256-column tiles would leave the last wave of CTAs mostly idle):
//   warp 0      TMA producer: 128 x 64 tiles of A and BN x 64 tiles of W through a
//               shared-memory ring of 4 (BN 256) or 6 (BN 128) stages (128-byte swizzle);
//   warp 1      owns TMEM (2 accumulator stages x BN fp32 columns) and issues
//               tcgen05.mma (M = 128, N = BN, K = 16) from one thread;
//   warps 2..9  epilogue: each reads 32 rows x BN/2 columns of the accumulator (its TMEM
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

constexpr int kBM = 128, kBK = 64;
constexpr int kEpiW = 8;
constexpr int kThreadsG = (2 + kEpiW) * 32;
constexpr int kABytes = kBM * kBK * 2;   // 16 KB

// Output tiles of 128 x BN; the ring holds as many 64-column stages as fit 192 KB.
template <int BN>
struct GemmShape {
  static constexpr int kBBytes = BN * kBK * 2;
  static constexpr int kStages = (192 * 1024) / (kABytes + kBBytes);   // 4 (BN 256) or 6 (BN 128)
};

template <int BN>
struct alignas(1024) GemmSmem {
  uint8_t a[GemmShape<BN>::kStages][kABytes];
  uint8_t b[GemmShape<BN>::kStages][GemmShape<BN>::kBBytes];
  uint64_t full[GemmShape<BN>::kStages], empty[GemmShape<BN>::kStages];
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
  int32_t* status;
};

// Hyperbolic tangent from the SFU (PTX tanh.approx.f32; its error, about 2^-11, is below
// the bf16 rounding of the output).
__device__ __forceinline__ float tanh_sfu(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int kAct>
__device__ __forceinline__ float act_fn(float v) {
  if (kAct == FASTAR_ACT_GELU_TANH) {
    // 0.5 v (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3)))
    const float u = 0.7978845608028654f * fmaf(0.044715f * v, v * v, v);
    return 0.5f * v * (1.0f + tanh_sfu(u));
  }
  if (kAct == FASTAR_ACT_SILU) return v / (1.0f + __expf(-v));
  return v;
}

// kAct (the activation) and kRes (a residual is added) are fixed per instance, so that
// the epilogue carries one body without per-element branches.
template <int kBN, int kAct, bool kRes>
__global__ void __launch_bounds__(kThreadsG, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_w,
                   const GemmArgs g) {
  constexpr int kGS = GemmShape<kBN>::kStages;
  constexpr int kBBytes = GemmShape<kBN>::kBBytes;
  extern __shared__ uint8_t smem_raw[];
  GemmSmem<kBN>& sm =
      *reinterpret_cast<GemmSmem<kBN>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
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
    tc::tmem_alloc(&sm.tmem_base, 2 * kBN);
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
    const int half = (warp - 2) >> 2;       // which half of the tile's columns
    const int row = quad * 32 + lane;
    int acc = 0;
    uint32_t aph = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
      const int tm = t % MT, tn = t / MT;
      if (!tc::mbar_wait(&sm.acc_full[acc], aph, abort)) break;
      tc::tc_fence_after();
      const int64_t m = (int64_t)tm * kBM + row;
      const int64_t n0 = (int64_t)tn * kBN + half * (kBN / 2);
      const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(acc * kBN + half * (kBN / 2));
      // passes of 64 columns (64 registers of scores at a time); the accumulator stage is
      // handed back once the last pass's scores are in registers
      constexpr int kPasses = kBN / 128;
#pragma unroll 1
      for (int pass = 0; pass < kPasses; ++pass) {
        float v[2][32];
        __syncwarp();   // the TMEM loads are warp-collective: every lane, converged
        tc::tmem_ld32(taddr + (uint32_t)(pass * 64), v[0]);
        tc::tmem_ld32(taddr + (uint32_t)(pass * 64 + 32), v[1]);
        tc::tmem_wait_ld();
        tc::tmem_pin32(v[0]);
        tc::tmem_pin32(v[1]);
        if (pass == kPasses - 1) {
          tc::tc_fence_before();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&sm.acc_empty[acc]);
        }
#pragma unroll
        for (int c = 0; c < 2 && m < g.M; ++c) {   // rows past M: nothing to store
          const int64_t nc = n0 + pass * 64 + c * 32;
          float r[32];
          if (kRes) {
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
          // four columns at a time: their bias and gate values as 16-byte loads (the
          // same for every lane)
          uint32_t pk[16];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 b4 = g.bias ? reinterpret_cast<const float4*>(g.bias + nc)[q] : make_float4(0.f, 0.f, 0.f, 0.f);
            float4 g4 = make_float4(1.f, 1.f, 1.f, 1.f);
            if (kRes && g.gate_a) {
              g4 = reinterpret_cast<const float4*>(g.gate_a + nc)[q];
              if (g.gate_b) {
                const float4 h4 = reinterpret_cast<const float4*>(g.gate_b + nc)[q];
                g4.x += h4.x, g4.y += h4.y, g4.z += h4.z, g4.w += h4.w;
              }
            }
            const float bq[4] = {b4.x, b4.y, b4.z, b4.w}, gq[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
            for (int u = 0; u < 4; u += 2) {
              const int i = 4 * q + u;
              float x0 = act_fn<kAct>(v[c][i] + bq[u]), x1 = act_fn<kAct>(v[c][i + 1] + bq[u + 1]);
              if (kRes) {
                x0 = fmaf(gq[u], x0, r[i]);
                x1 = fmaf(gq[u + 1], x1, r[i + 1]);
              }
              if (g.c_f32) {
                *reinterpret_cast<float2*>(static_cast<float*>(g.C) + m * g.ldc + nc + i) = make_float2(x0, x1);
              } else {
                __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
                pk[i >> 1] = *reinterpret_cast<uint32_t*>(&h);
              }
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
    tc::tmem_dealloc(tmem, 2 * kBN);
  }
  if (threadIdx.x == 0 && sm.abort) flag_status(g.status, FASTAR_DEV_TIMEOUT);
}

}  // namespace

template <int kBN, int kAct, bool kRes>
static cudaError_t gemm_launch(const void* A, int64_t lda, const void* W, int64_t ldw, const GemmArgs& g,
                               cudaStream_t s) {
  constexpr size_t smem = sizeof(GemmSmem<kBN>) + 1024;
  const cudaError_t attr = opt_in_smem((const void*)gemm_tc_kernel<kBN, kAct, kRes>, (int)smem);
  if (attr != cudaSuccess) return attr;
  CUtensorMap ta, tw;
  if (!make_tmap_bf16_3d(&ta, A, (uint64_t)g.K, (uint64_t)g.M, 1, (uint64_t)lda * 2, 0, kBK, kBM) ||
      !make_tmap_bf16_3d(&tw, W, (uint64_t)g.K, (uint64_t)g.N, 1, (uint64_t)ldw * 2, 0, kBK, kBN))
    return cudaErrorInvalidValue;
  const int64_t tiles = ((g.M + kBM - 1) / kBM) * (g.N / kBN);
  const int grid = (int)(tiles < sm_count() ? tiles : sm_count());
  gemm_tc_kernel<kBN, kAct, kRes><<<grid, kThreadsG, smem, s>>>(ta, tw, g);
  count_launches(1);
  return cudaGetLastError();
}

template <int kAct>
static cudaError_t gemm_pick(bool res, bool narrow, const void* A, int64_t lda, const void* W, int64_t ldw,
                             const GemmArgs& g, cudaStream_t s) {
  if (res)
    return narrow ? gemm_launch<128, kAct, true>(A, lda, W, ldw, g, s)
                  : gemm_launch<256, kAct, true>(A, lda, W, ldw, g, s);
  return narrow ? gemm_launch<128, kAct, false>(A, lda, W, ldw, g, s)
                : gemm_launch<256, kAct, false>(A, lda, W, ldw, g, s);
}

cudaError_t launch_gemm_tc(const void* A, int64_t lda, const void* W, int64_t ldw, const float* bias,
                           const void* res, int64_t ldr, const float* gate_a, const float* gate_b, void* C, int64_t ldc,
                           int c_f32, int64_t M, int64_t N, int64_t K, int act, int32_t* status, cudaStream_t s) {
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
  g.status = status;
  // 128 x 256 tiles, unless 128 x 128 tiles fill the machine enough better: waves of the
  // narrow tiles are half as long but cost about 0.6 of a wide one when K is short (the
  // epilogue and the pipeline fill dominate a tile); with a long K the narrow tiles' main
  // loop is markedly slower (measured), so they are kept to K <= 2048
  const int64_t sms = sm_count();
  const int64_t t256 = ((M + kBM - 1) / kBM) * (N / 256);
  const int64_t w256 = (t256 + sms - 1) / sms, w128 = (2 * t256 + sms - 1) / sms;
  const bool narrow = K <= 2048 && 3 * w128 < 5 * w256;
  switch (act) {
    case FASTAR_ACT_GELU_TANH:
      return gemm_pick<FASTAR_ACT_GELU_TANH>(res != nullptr, narrow, A, lda, W, ldw, g, s);
    case FASTAR_ACT_SILU:
      return gemm_pick<FASTAR_ACT_SILU>(res != nullptr, narrow, A, lda, W, ldw, g, s);
    default:
      return gemm_pick<FASTAR_ACT_NONE>(res != nullptr, narrow, A, lda, W, ldw, g, s);
  }
}

}  // namespace fastar
