// AnnCA frame-relevance scores on the 5th-generation tensor cores (bf16, gated).
//
// FAST-AR technical summary §2.B / blog §2: for latent frame f and prompt token p,
//   score(h, f, p) = max over the frame's queries i whose bucket set R(i) holds the
//                    prompt token's bucket pb[p] of cos(q_i, kp_p)
// (−inf when no such query).  The dense form S = Kp · Q_f^T is cheap on the tensor
// cores (2·P·T_f·d flops per head and frame), so the bucket condition becomes a mask
// in the epilogue instead of a gather.
//
// One persistent CTA per SM; a work unit is (head, frame, 128-prompt tile):
//   warp 0     TMA: the unit's prompt tile (M = 128 rows) once, then the frame's query
//              tiles (N = 128 rows each) through a 4-deep shared-memory ring;
//   warp 1     owns TMEM (2 accumulator stages of 128 columns) and issues tcgen05.mma;
//   warps 2-5  column facts, one query column per thread, a tile ahead of the fold:
//              1/|q_j| (from the caller's query norms when given, loaded a tile ahead with
//              the bucket ids; else the fp32 sum of squares of the shared-memory Q row, and
//              only then do these warps wait for the Q tile) and, per bucket b,
//              the 128-bit mask of the tile's columns whose bucket set holds b (built with
//              shared-memory atomics from qb; a column with an id outside [0, B) gets no
//              bit); two buffers;
//   warps 6-13 fold, two warps per TMEM lane quadrant (each takes half of the tile's
//              columns): prompt row p reads the two mask words of its own bucket pb[p] and
//              keeps the running maximum of s_pj / |q_j| over the columns whose bit is
//              set; at the end score = max / |kp_p|.
// Every wait is bounded; a timeout sets FASTAR_DEV_TIMEOUT, every role still walks every
// unit (a wait after the timeout returns at once), so the named barriers of the facts and
// fold groups always fill, and the rows of every unit that was not scored completely are
// written as NaN.
#include <climits>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"
#include "tmap.h"

namespace fastar {
namespace {

constexpr int kCaStages = 4;          // Q ring depth
constexpr int kCaTS = 2;              // TMEM accumulator stages (and column-fact buffers)
constexpr int kCaFactW = 4;           // column-fact warps (one query column per thread)
constexpr int kCaFoldW = 8;           // fold warps: 4 lane quadrants x 2 column halves
constexpr int kCaFact0 = 2;           // first column-fact warp
constexpr int kCaFold0 = kCaFact0 + kCaFactW;
constexpr int kCaThreads = (kCaFold0 + kCaFoldW) * 32;
constexpr int kCaTile = 128 * 128;    // one 128-row x 64-element bf16 block (128-B swizzle)

template <int D>
struct alignas(1024) CaSmem {
  uint8_t a[D / 64][kCaTile];               // prompt tile
  uint8_t b[kCaStages][D / 64][kCaTile];    // query tiles
  float inv[kCaTS][128];                    // 1/|q_j| per query column
  uint32_t mask[kCaTS][FASTAR_MAX_B][4];    // per bucket: the columns whose bucket set holds it
  float bx[128];                            // second column half's row maxima
  uint64_t a_full, a_empty;
  uint64_t b_full[kCaStages], b_empty[kCaStages];
  uint64_t t_full[kCaTS], t_empty[kCaTS];
  uint64_t f_full[kCaTS], f_empty[kCaTS];
  uint32_t tmem_base;
  int abort;
};

struct CaGeom {
  int H, F, PT, r, B;
  int q_token_major;
  int64_t tpf, P;
};

__device__ __forceinline__ bool ca_wait_all(uint64_t* bar, uint32_t parity, volatile int* abort) {
  const bool ok = tc::mbar_wait(bar, parity, abort);
  return __all_sync(0xffffffffu, ok);
}

// fp32 sum of squares of row `row` of a 128-row bf16 tile stored as D/64 swizzled blocks.
template <int D>
__device__ __forceinline__ float row_sumsq(const uint8_t* tile, int row) {
  float s0 = 0.f, s1 = 0.f;
#pragma unroll
  for (int kh = 0; kh < D / 64; ++kh) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint4 v = *reinterpret_cast<const uint4*>(tile + kh * kCaTile + tc::sw128_off(row, c));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float lo = __uint_as_float(w[i] << 16), hi = __uint_as_float(w[i] & 0xffff0000u);
        s0 = fmaf(lo, lo, s0);
        s1 = fmaf(hi, hi, s1);
      }
    }
  }
  return s0 + s1;
}

template <int D>
__global__ void __launch_bounds__(kCaThreads, 1)
    annca_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_p,
                    const int32_t* __restrict__ qb, const int32_t* __restrict__ pb,
                    const float* __restrict__ qn, CaGeom g, float* __restrict__ score, int32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  CaSmem<D>& sm = *reinterpret_cast<CaSmem<D>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  constexpr int KH = D / 64;
  constexpr uint32_t kIdesc = tc::idesc_bf16_f32(128, 128);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int units = g.H * g.F * g.PT;
  const int nch = (int)((g.tpf + 127) / 128);   // query tiles per frame
  if (threadIdx.x == 0) {
    tc::mbar_init(&sm.a_full, 1);
    tc::mbar_init(&sm.a_empty, 1 + kCaFoldW / 2);   // the MMA's commit + the half-0 fold warps
    for (int s = 0; s < kCaStages; ++s) {
      tc::mbar_init(&sm.b_full[s], 1);
      // the MMA's commit + the column-fact warps when they read the Q tile themselves
      tc::mbar_init(&sm.b_empty[s], qn ? 1 : 1 + kCaFactW);
    }
    for (int s = 0; s < kCaTS; ++s) {
      tc::mbar_init(&sm.t_full[s], 1);
      tc::mbar_init(&sm.t_empty[s], kCaFoldW);
      tc::mbar_init(&sm.f_full[s], kCaFactW);
      tc::mbar_init(&sm.f_empty[s], kCaFoldW);
    }
    sm.abort = 0;
    tc::mbar_fence_init();
  }
  if ((int)blockIdx.x >= units) return;   // uniform, before any allocation
  if (warp == 1) {
    tc::tmem_alloc(&sm.tmem_base, 256);
    tc::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tc::tma_prefetch_desc(&tm_q);
    tc::tma_prefetch_desc(&tm_p);
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
      uint32_t ph = 0, aph = 0;
      for (int u = blockIdx.x; u < units && !*abort; u += gridDim.x) {
        const int pt = u % g.PT, f = (u / g.PT) % g.F, h = u / (g.PT * g.F);
        if (!tc::mbar_wait(&sm.a_empty, aph ^ 1, abort)) break;
        aph ^= 1;
        tc::mbar_arrive_tx(&sm.a_full, (uint32_t)(KH * kCaTile));
        for (int kh = 0; kh < KH; ++kh) tc::tma_load_3d(sm.a[kh], &tm_p, kh * 64, pt * 128, h, &sm.a_full);
        for (int c = 0; c < nch; ++c) {
          if (!tc::mbar_wait(&sm.b_empty[stage], ph ^ 1, abort)) break;
          tc::mbar_arrive_tx(&sm.b_full[stage], (uint32_t)(KH * kCaTile));
          const int t0 = (int)(f * g.tpf + c * 128);
          for (int kh = 0; kh < KH; ++kh) {
            if (g.q_token_major)
              tc::tma_load_3d(sm.b[stage][kh], &tm_q, kh * 64, h, t0, &sm.b_full[stage]);
            else
              tc::tma_load_3d(sm.b[stage][kh], &tm_q, kh * 64, t0, h, &sm.b_full[stage]);
          }
          if (++stage == kCaStages) {
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
      uint32_t ph = 0, aph = 0, tph = 0;
      const uint64_t a_desc = tc::sw128_desc(tc::smem_u32(&sm.a[0][0]));
      const uint64_t b_desc0 = tc::sw128_desc(tc::smem_u32(&sm.b[0][0][0]));
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        if (!tc::mbar_wait(&sm.a_full, aph, abort)) break;
        aph ^= 1;
        tc::tc_fence_after();
        for (int c = 0; c < nch; ++c) {
          if (!tc::mbar_wait(&sm.b_full[stage], ph, abort) || !tc::mbar_wait(&sm.t_empty[acc], tph ^ 1, abort)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t off = (uint32_t)((k >> 2) * kCaTile + (k & 3) * 32);
            tc::mma_bf16(tmem + (uint32_t)(acc * 128), a_desc + (off >> 4),
                         b_desc0 + ((uint32_t)(stage * KH * kCaTile + off) >> 4), kIdesc, k > 0 ? 1u : 0u);
          }
          tc::mma_commit(&sm.b_empty[stage]);
          tc::mma_commit(&sm.t_full[acc]);
          if (++stage == kCaStages) {
            stage = 0;
            ph ^= 1;
          }
          if (++acc == kCaTS) {
            acc = 0;
            tph ^= 1;
          }
        }
        if (!ok) break;
        tc::mma_commit(&sm.a_empty);
      }
    }
  } else if (warp < kCaFold0) {
    // ---------------- column facts: thread ft owns query column ft of every tile ----------------
    const int ft = (warp - kCaFact0) * 32 + lane;
    const int nmask = g.B * 4;
    int stage = 0, fb = 0;
    uint32_t ph = 0, fph = 0;
    // the column's bucket ids (and norm, when given) of tile c of (h, f), loaded a tile
    // ahead of their use
    auto load_ids = [&](int h, int f, int c, int (&ids)[FASTAR_MAX_R], float& nrm) -> bool {
      const int64_t tl = (int64_t)c * 128 + ft;
      if (c >= nch || tl >= g.tpf) return false;
      const int64_t qi = (int64_t)h * g.F * g.tpf + (int64_t)f * g.tpf + tl;
      const int32_t* src = qb + qi * g.r;
#pragma unroll
      for (int sl = 0; sl < FASTAR_MAX_R; ++sl) ids[sl] = sl < g.r ? src[sl] : 0;
      if (qn) nrm = qn[qi];
      return true;
    };
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      const int f = (u / g.PT) % g.F, h = u / (g.PT * g.F);
      int nids[FASTAR_MAX_R];
      float nnrm = 0.f;
      bool nok = load_ids(h, f, 0, nids, nnrm);
      for (int c = 0; c < nch; ++c) {
        int ids[FASTAR_MAX_R];
#pragma unroll
        for (int sl = 0; sl < FASTAR_MAX_R; ++sl) ids[sl] = nids[sl];
        const float nrm = nnrm;
        bool okc = nok;
        nok = load_ids(h, f, c + 1, nids, nnrm);   // in flight during this tile's waits and math
        bool live = ca_wait_all(&sm.f_empty[fb], fph ^ 1, abort);
        if (live)
          for (int i = ft; i < nmask; i += kCaFactW * 32) (&sm.mask[fb][0][0])[i] = 0u;
        live = tc::named_bar_and(2, kCaFactW * 32, live);   // cleared before any bit is set
        if (!qn) live = live && ca_wait_all(&sm.b_full[stage], ph, abort);
        if (live) {
          float qi = 0.f;
          if (okc) {
            if (qn) {
              qi = nrm > 0.f ? 1.0f / nrm : 0.f;
            } else {
              const float ss = row_sumsq<D>(&sm.b[stage][0][0], ft);
              qi = ss > 0.f ? 1.0f / sqrtf(ss) : 0.f;
            }
#pragma unroll
            for (int sl = 0; sl < FASTAR_MAX_R; ++sl)
              if (sl < g.r && (ids[sl] < 0 || ids[sl] >= g.B)) okc = false;
          }
          sm.inv[fb][ft] = qi;
          if (okc) {
#pragma unroll
            for (int sl = 0; sl < FASTAR_MAX_R; ++sl)
              if (sl < g.r) atomicOr(&sm.mask[fb][ids[sl]][ft >> 5], 1u << (ft & 31));
          }
        }
        __syncwarp();
        if (lane == 0) {
          if (!qn) tc::mbar_arrive(&sm.b_empty[stage]);
          tc::mbar_arrive(&sm.f_full[fb]);
        }
        if (++stage == kCaStages) {
          stage = 0;
          ph ^= 1;
        }
        if (++fb == kCaTS) {
          fb = 0;
          fph ^= 1;
        }
      }
    }
  } else {
    // ---------------- fold: warp (quad, half) takes prompt rows quad*32.. and the tile's
    // columns half*64 .. half*64+63 ----------------
    const int fw = warp - kCaFold0;
    const int quad = warp & 3, half = fw >> 2;
    const int row = quad * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
    int acc = 0;
    uint32_t aph = 0, tph = 0;
    bool alive = true;   // false from the first timed-out wait on
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      const int pt = u % g.PT, f = (u / g.PT) % g.F, h = u / (g.PT * g.F);
      const int64_t p = (int64_t)pt * 128 + row;
      int mypb = -1;
      if (p < g.P) {
        mypb = pb[(int64_t)h * g.P + p];
        if (mypb < 0 || mypb >= g.B) {
          flag_status(status, FASTAR_DEV_BAD_BUCKET);
          mypb = -1;
        }
      }
      // 1/|kp_p| from the prompt tile, then hand the tile's shared memory back
      bool got = ca_wait_all(&sm.a_full, aph, abort);
      aph ^= 1;
      alive = alive && got;
      float pinv = 0.f;
      if (half == 0) {
        if (got) {
          const float ss = row_sumsq<D>(&sm.a[0][0], row);
          pinv = ss > 0.f ? 1.0f / sqrtf(ss) : 0.f;
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&sm.a_empty);
      }
      float best = neg_inf();
      for (int c = 0; c < nch; ++c) {
        got = ca_wait_all(&sm.t_full[acc], tph, abort);
        float v[64];
        if (got) {
          tc::tc_fence_after();
          tc::tmem_ld32(tmem + lane_addr + (uint32_t)(acc * 128 + half * 64), v);
          tc::tmem_ld32(tmem + lane_addr + (uint32_t)(acc * 128 + half * 64 + 32), v + 32);
          tc::tmem_wait_ld();
          tc::tmem_pin32(v);
          tc::tmem_pin32(v + 32);
          tc::tc_fence_before();
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&sm.t_empty[acc]);
        got = got && ca_wait_all(&sm.f_full[acc], tph, abort);
        alive = alive && got;
        if (got && mypb >= 0) {
          const uint32_t m0 = sm.mask[acc][mypb][half * 2], m1 = sm.mask[acc][mypb][half * 2 + 1];
          const float* iv = sm.inv[acc] + half * 64;
#pragma unroll
          for (int j4 = 0; j4 < 16; ++j4) {
            const float4 s4 = *reinterpret_cast<const float4*>(iv + j4 * 4);
            const float sc[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int j = j4 * 4 + e;
              const uint32_t m = j < 32 ? m0 : m1;
              if ((m >> (j & 31)) & 1u) best = fmaxf(best, v[j] * sc[e]);
            }
          }
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&sm.f_empty[acc]);
        if (++acc == kCaTS) {
          acc = 0;
          tph ^= 1;
        }
      }
      // combine the two column halves of each row; a unit not scored completely (a wait
      // timed out) writes NaN, so that the ranking sees the failure
      if (half == 1) sm.bx[row] = best;
      const bool unit_ok = tc::named_bar_and(1, kCaFoldW * 32, alive);
      if (half == 0 && p < g.P) {
        best = fmaxf(best, sm.bx[row]);
        const float sc = best == neg_inf() ? neg_inf() : best * pinv;
        score[((int64_t)h * g.F + f) * g.P + p] = unit_ok ? sc : __uint_as_float(0x7fc00000u);
      }
      tc::named_bar(1, kCaFoldW * 32);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 256);
  }
  if (threadIdx.x == 0 && sm.abort) flag_status(status, FASTAR_DEV_TIMEOUT);
}

template <int D>
bool launch_annca_tc_impl(TokView q, int H, int F, int64_t tpf, const int32_t* qb, int r, const void* kp,
                          const int32_t* pb, int64_t P, int B, const float* qnorm, float* score, int32_t* status,
                          cudaStream_t s) {
  const int64_t nq = (int64_t)F * tpf;
  if (P <= 0 || tpf <= 0 || nq > INT_MAX || P > INT_MAX) return false;
  CUtensorMap tq, tp;
  const bool token_major = H > 1 && q.hs < q.ts;
  if (token_major) {
    if (!make_tmap_bf16_3d(&tq, q.p, D, (uint64_t)H, (uint64_t)nq, (uint64_t)q.hs * 2, (uint64_t)q.ts * 2, 64, 1,
                           128))
      return false;
  } else if (!make_tmap_bf16_3d(&tq, q.p, D, (uint64_t)nq, (uint64_t)H, (uint64_t)q.ts * 2, (uint64_t)q.hs * 2, 64,
                                128)) {
    return false;
  }
  if (!make_tmap_bf16_3d(&tp, kp, D, (uint64_t)P, (uint64_t)H, (uint64_t)D * 2, (uint64_t)P * D * 2, 64, 128))
    return false;
  CaGeom g;
  g.H = H;
  g.F = F;
  g.PT = (int)((P + 127) / 128);
  g.r = r;
  g.B = B;
  g.q_token_major = token_major ? 1 : 0;
  g.tpf = tpf;
  g.P = P;
  const int units = H * F * g.PT;
  const int grid = units < sm_count() ? units : sm_count();
  constexpr size_t smem = sizeof(CaSmem<D>) + 1024;
  const cudaError_t a = opt_in_smem((const void*)annca_tc_kernel<D>, (int)smem);
  if (a != cudaSuccess) return false;
  annca_tc_kernel<D><<<grid, kCaThreads, smem, s>>>(tq, tp, qb, pb, qnorm, g, score, status);
  count_launches(1);
  return true;
}

}  // namespace

bool launch_annca_tc(int d, TokView q, int H, int F, int64_t tpf, const int32_t* qb, int r, const void* kp,
                     const int32_t* pb, int64_t P, int B, const float* qnorm, float* score, int32_t* status,
                     cudaStream_t s) {
  if (B < 1 || B > FASTAR_MAX_B || r < 1 || r > FASTAR_MAX_R) return false;
  if (d == 128) return launch_annca_tc_impl<128>(q, H, F, tpf, qb, r, kp, pb, P, B, qnorm, score, status, s);
  return launch_annca_tc_impl<64>(q, H, F, tpf, qb, r, kp, pb, P, B, qnorm, score, status, s);
}

}  // namespace fastar
