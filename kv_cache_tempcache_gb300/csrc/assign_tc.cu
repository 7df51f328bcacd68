// ANN bucket assignment on the tensor cores (bf16): scores of 128 tokens against all
// B centroids of their head in one tcgen05.mma (N = B rounded up to 32), then a
// per-row top-r in the epilogue.
//
// FAST-AR technical summary §2.C / §2.B: tokens go to ANN buckets; the key bucket is
// the arg-max centroid, a query's set the r best (ties to the lower index).
//
// One CTA per (head, 128-token tile), 4 warps (a step's query and key assignments can
// also run as one launch, one grid plane each).  Thread 0 loads the token tile and the
// head's centroids with TMA and issues the MMA; every thread then owns one token row:
// it reads its scores from TMEM in 32-column chunks, keeps a sorted top-r, and
// computes |x| from the token tile still in shared memory.  Several CTAs share an SM
// (small shared-memory and TMEM footprints), which hides the load latency.
#include <climits>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"
#include "tmap.h"

namespace fastar {
namespace {

constexpr int kRows = 128;
constexpr int kBlk = 128 * 128;   // 128 rows x 64 bf16 (swizzled)

// Shared memory (1024-byte aligned): the token tile (D/64 blocks of 128 rows x 128 B),
// the centroid tile (D/64 blocks of NP rows x 128 B), then two mbarriers and the TMEM
// address.
struct AssignCtl {
  uint64_t tma_bar, mma_bar;
  uint32_t tmem_base;
  int abort;
};

// The assignment of one (head h, 128-token tile) (every thread of the CTA calls it).
template <int D, int RT>
__device__ __forceinline__ void assign_tile(const CUtensorMap* tm_x, const CUtensorMap* tm_c, int h, int64_t t0,
                                            int64_t n, int token_major, int B, int NP, int r, uint32_t tcols,
                                            int32_t* __restrict__ ids, float* __restrict__ scores,
                                            float* __restrict__ norms, int32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  constexpr int KH = D / 64;
  uint8_t* sa = base;                                  // [KH][kBlk]
  uint8_t* sb = base + KH * kBlk;                      // [KH][NP * 128]
  AssignCtl& sm = *reinterpret_cast<AssignCtl*>(sb + KH * NP * 128);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    tc::mbar_init(&sm.tma_bar, 1);
    tc::mbar_init(&sm.mma_bar, 1);
    sm.abort = 0;
    tc::mbar_fence_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(&sm.tmem_base, tcols);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort = &sm.abort;
  if (threadIdx.x == 0) {
    tc::mbar_arrive_tx(&sm.tma_bar, (uint32_t)(KH * kBlk + KH * NP * 128));
    for (int kh = 0; kh < KH; ++kh) {
      if (token_major)
        tc::tma_load_3d(sa + kh * kBlk, tm_x, kh * 64, h, (int)t0, &sm.tma_bar);
      else
        tc::tma_load_3d(sa + kh * kBlk, tm_x, kh * 64, (int)t0, h, &sm.tma_bar);
      tc::tma_load_3d(sb + kh * NP * 128, tm_c, kh * 64, 0, h, &sm.tma_bar);
    }
    if (tc::mbar_wait(&sm.tma_bar, 0, abort)) {
      tc::tc_fence_after();
      const uint32_t idesc = tc::idesc_bf16_f32(128, NP);
#pragma unroll
      for (int k = 0; k < D / 16; ++k) {
        const uint32_t ko = (uint32_t)((k & 3) * 32);
        tc::mma_bf16(tmem, tc::sw128_desc(tc::smem_u32(sa + (k >> 2) * kBlk) + ko),
                     tc::sw128_desc(tc::smem_u32(sb + (k >> 2) * NP * 128) + ko), idesc, k > 0 ? 1u : 0u);
      }
      tc::mma_commit(&sm.mma_bar);
    }
  }
  __syncwarp();
  const bool ok = __all_sync(0xffffffffu, tc::mbar_wait(&sm.mma_bar, 0, abort));
  tc::tc_fence_after();
  const int row = warp * 32 + lane;
  const int64_t t = t0 + row;
  // sorted top-r (score desc, index asc); ties keep the earlier (lower) index.  RT > 0
  // fixes r at compile time so the list lives in registers.
  constexpr int NR = RT > 0 ? RT : FASTAR_MAX_R;
  float bv[NR];
  int bi[NR];
#pragma unroll
  for (int s = 0; s < NR; ++s) {
    bv[s] = neg_inf();
    bi[s] = INT_MAX;
  }
  if (ok) {
    for (int c = 0; c < NP; c += 32) {
      float v[32];
      tc::tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c, v);
      tc::tmem_wait_ld();
#pragma unroll
      for (int x = 0; x < 32; ++x) {
        const int j = c + x;
        const float s = v[x];
        if (j >= B) continue;
        if (RT == 1) {
          if (s > bv[0]) {
            bv[0] = s;
            bi[0] = j;
          }
        } else if (RT == 2) {
          if (s > bv[NR - 1]) {
            if (s > bv[0]) {
              bv[NR - 1] = bv[0];
              bi[NR - 1] = bi[0];
              bv[0] = s;
              bi[0] = j;
            } else {
              bv[NR - 1] = s;
              bi[NR - 1] = j;
            }
          }
        } else if (s > bv[r - 1]) {
          // insert j keeping the order; equal scores stay ahead of it
          int pos = r - 1;
          while (pos > 0 && s > bv[pos - 1]) {
            bv[pos] = bv[pos - 1];
            bi[pos] = bi[pos - 1];
            --pos;
          }
          bv[pos] = s;
          bi[pos] = j;
        }
      }
    }
  }
  tc::tc_fence_before();
  if (t < n && ok) {
#pragma unroll
    for (int s = 0; s < NR; ++s) {
      if (s < r) {
        ids[((int64_t)h * n + t) * r + s] = bi[s];
        if (scores) scores[((int64_t)h * n + t) * r + s] = bv[s];
      }
    }
    if (norms) {
      float ss = 0.f;
#pragma unroll
      for (int kh = 0; kh < KH; ++kh) {
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
          float e[8];
          load8(reinterpret_cast<const __nv_bfloat16*>(sa + kh * kBlk + tc::sw128_off(row, c8)), e);
#pragma unroll
          for (int u = 0; u < 8; ++u) ss = fmaf(e[u], e[u], ss);
        }
      }
      norms[(int64_t)h * n + t] = sqrtf(ss);
    }
  }
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, tcols);
  }
  if (threadIdx.x == 0 && sm.abort) flag_status(status, FASTAR_DEV_TIMEOUT);
}

template <int D, int RT>
__global__ void __launch_bounds__(128)
assign_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_c, int H,
                 int64_t n, int token_major, int B, int NP, int r, uint32_t tcols, int32_t* __restrict__ ids,
                 float* __restrict__ scores, float* __restrict__ norms, int32_t* status) {
  assign_tile<D, RT>(&tm_x, &tm_c, blockIdx.y, (int64_t)blockIdx.x * kRows, n, token_major, B, NP, r, tcols, ids,
                     scores, norms, status);
}

// Both assignments of a step in one launch: blockIdx.z = 0 takes a query tile (top-r
// sets), blockIdx.z = 1 a current-key tile (arg-max bucket and |k|).
template <int D, int RTQ>
__global__ void __launch_bounds__(128)
assign_qk_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_c, int64_t n, int token_major, int B, int NP, int r,
                    uint32_t tcols, int32_t* __restrict__ qb, int32_t* __restrict__ kb, float* __restrict__ knorm,
                    float* __restrict__ qnorm) {
  if (blockIdx.z == 0)
    assign_tile<D, RTQ>(&tm_q, &tm_c, blockIdx.y, (int64_t)blockIdx.x * kRows, n, token_major, B, NP, r, tcols, qb,
                        nullptr, qnorm, nullptr);
  else
    assign_tile<D, 1>(&tm_k, &tm_c, blockIdx.y, (int64_t)blockIdx.x * kRows, n, token_major, B, NP, 1, tcols, kb,
                      nullptr, knorm, nullptr);
}

template <int D>
size_t assign_tc_smem(int NP) {
  return (size_t)(D / 64) * (kBlk + (size_t)NP * 128) + sizeof(AssignCtl) + 1024;
}

template <int D>
bool assign_tc_impl(TokView x, int H, int64_t n, const void* cent, int B, int r, int32_t* ids, float* scores,
                    float* norms, cudaStream_t s) {
  const int NP = (B + 31) / 32 * 32;
  if (NP > 256 || n > INT32_MAX) return false;
  CUtensorMap tx, tcen;
  const bool token_major = H > 1 && x.hs < x.ts;
  if (token_major) {
    if (!make_tmap_bf16_3d(&tx, x.p, D, (uint64_t)H, (uint64_t)n, (uint64_t)x.hs * 2, (uint64_t)x.ts * 2, 64, 1, 128))
      return false;
  } else if (!make_tmap_bf16_3d(&tx, x.p, D, (uint64_t)n, (uint64_t)H, (uint64_t)x.ts * 2, (uint64_t)x.hs * 2, 64,
                                128)) {
    return false;
  }
  if (!make_tmap_bf16_3d(&tcen, cent, D, (uint64_t)B, (uint64_t)H, (uint64_t)D * 2, (uint64_t)B * D * 2, 64,
                         (uint32_t)NP))
    return false;
  uint32_t tcols = 32;
  while ((int)tcols < NP) tcols <<= 1;
  const size_t smem = assign_tc_smem<D>(NP);
  const int smax = (int)assign_tc_smem<D>(256);
  const cudaError_t a1 = opt_in_smem((const void*)assign_tc_kernel<D, 1>, smax);
  const cudaError_t a2 = opt_in_smem((const void*)assign_tc_kernel<D, 2>, smax);
  const cudaError_t a0 = opt_in_smem((const void*)assign_tc_kernel<D, 0>, smax);
  if (a1 != cudaSuccess || a2 != cudaSuccess || a0 != cudaSuccess) return false;
  const dim3 grid((unsigned)((n + kRows - 1) / kRows), H);
  const int tm = token_major ? 1 : 0;
  if (r == 1)
    assign_tc_kernel<D, 1><<<grid, 128, smem, s>>>(tx, tcen, H, n, tm, B, NP, r, tcols, ids, scores, norms, nullptr);
  else if (r == 2)
    assign_tc_kernel<D, 2><<<grid, 128, smem, s>>>(tx, tcen, H, n, tm, B, NP, r, tcols, ids, scores, norms, nullptr);
  else
    assign_tc_kernel<D, 0><<<grid, 128, smem, s>>>(tx, tcen, H, n, tm, B, NP, r, tcols, ids, scores, norms, nullptr);
  count_launches(1);
  return true;
}

template <int D>
bool assign_qk_tc_impl(TokView q, TokView k, int H, int64_t n, const void* cent, int B, int r, int32_t* qb,
                       int32_t* kb, float* knorm, float* qnorm, cudaStream_t s) {
  const int NP = (B + 31) / 32 * 32;
  if (NP > 256 || n > INT32_MAX) return false;
  CUtensorMap tq, tk, tcen;
  const bool token_major = H > 1 && q.hs < q.ts;
  for (int i = 0; i < 2; ++i) {
    const TokView& x = i == 0 ? q : k;
    CUtensorMap* m = i == 0 ? &tq : &tk;
    if (token_major) {
      if (!make_tmap_bf16_3d(m, x.p, D, (uint64_t)H, (uint64_t)n, (uint64_t)x.hs * 2, (uint64_t)x.ts * 2, 64, 1,
                             128))
        return false;
    } else if (!make_tmap_bf16_3d(m, x.p, D, (uint64_t)n, (uint64_t)H, (uint64_t)x.ts * 2, (uint64_t)x.hs * 2, 64,
                                  128)) {
      return false;
    }
  }
  if (!make_tmap_bf16_3d(&tcen, cent, D, (uint64_t)B, (uint64_t)H, (uint64_t)D * 2, (uint64_t)B * D * 2, 64,
                         (uint32_t)NP))
    return false;
  uint32_t tcols = 32;
  while ((int)tcols < NP) tcols <<= 1;
  const size_t smem = assign_tc_smem<D>(NP);
  const int smax = (int)assign_tc_smem<D>(256);
  const cudaError_t a2 = opt_in_smem((const void*)assign_qk_tc_kernel<D, 2>, smax);
  const cudaError_t a0 = opt_in_smem((const void*)assign_qk_tc_kernel<D, 0>, smax);
  if (a2 != cudaSuccess || a0 != cudaSuccess) return false;
  const dim3 grid((unsigned)((n + kRows - 1) / kRows), H, 2);
  const int tm = token_major ? 1 : 0;
  if (r == 2)
    assign_qk_tc_kernel<D, 2><<<grid, 128, smem, s>>>(tq, tk, tcen, n, tm, B, NP, r, tcols, qb, kb, knorm, qnorm);
  else
    assign_qk_tc_kernel<D, 0><<<grid, 128, smem, s>>>(tq, tk, tcen, n, tm, B, NP, r, tcols, qb, kb, knorm, qnorm);
  count_launches(1);
  return true;
}

}  // namespace

bool launch_assign_tc(int d, TokView x, int H, int64_t n, const void* cent, int B, int r, int32_t* ids,
                      float* scores, float* norms, cudaStream_t s) {
  return d == 128 ? assign_tc_impl<128>(x, H, n, cent, B, r, ids, scores, norms, s)
                  : assign_tc_impl<64>(x, H, n, cent, B, r, ids, scores, norms, s);
}

bool launch_assign_qk_tc(int d, TokView q, TokView k, int H, int64_t n, const void* cent, int B, int r,
                         int32_t* qb, int32_t* kb, float* knorm, float* qnorm, cudaStream_t s) {
  return d == 128 ? assign_qk_tc_impl<128>(q, k, H, n, cent, B, r, qb, kb, knorm, qnorm, s)
                  : assign_qk_tc_impl<64>(q, k, H, n, cent, B, r, qb, kb, knorm, qnorm, s);
}

}  // namespace fastar
