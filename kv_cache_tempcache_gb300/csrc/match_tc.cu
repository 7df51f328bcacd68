// TempCache top-1 match on the 5th-generation tensor cores (bf16 inputs).
//
// FAST-AR technical summary §2.A / blog §1: for each current-frame query, the top-1
// nearest cached key (cosine).  Per head this is a GEMM S = Q K^T (M = Nq, N = n,
// K = d) whose N dimension is reduced on the fly by an arg-max epilogue: scores
// never leave the SM.
//
// One persistent CTA per SM, warp-specialised:
//   warp 0      TMA producer: the unit's 256 query rows once (two M=128 tiles), then
//               128-key tiles of the cache through a 4-deep shared-memory ring;
//   warp 1      owns TMEM (512 columns = 2 accumulator stages x 2 M-tiles x 128
//               columns) and issues tcgen05.mma (one thread, operand descriptors
//               as precomputed offsets), committing to the ring's "empty" barriers
//               and the accumulator's "full" barrier;
//   warps 2..17 epilogue, four warps per TMEM lane quadrant (4 column parts of 32
//               keys): each thread owns the same row of both M-tiles, reads the 32
//               scores of each in two 16-column halves, scales them by 1/|k_j| (norms
//               prefetched a tile ahead, packed f32x2 multiplies) and keeps the
//               running top-1 (and top-2 when asked) of both rows with three-input
//               max trees over groups of four columns.  The
//               1/|k_j| values reach the lanes as shared-memory broadcasts, which
//               share the data pipe with the tensor core's operand reads: one
//               broadcast serving both M-tiles halves that traffic.  16 warps keep
//               enough of the latency-bound reduction in flight per SM.
// The MMA of tile t+1 overlaps the epilogue of tile t.  A work unit is (head,
// 256-query block, key segment); segments split the cache so the unit count
// fills the machine; the column parts of a row are merged in shared memory at the
// end of each unit, and a small finaliser merges the segments' partial top-2s.
// Every wait is bounded; a timeout sets FASTAR_DEV_TIMEOUT and unwinds.
#include <climits>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"
#include "tmap.h"

namespace fastar {

namespace {

constexpr int kQ = 256;         // queries per unit
constexpr int kN = 128;         // keys per tile
constexpr int kStages = 4;      // B ring depth
constexpr int kTS = 2;          // TMEM accumulator stages (kTS x 2 M-tiles x kN = 512 columns)
constexpr int kEpW = 16;        // epilogue warps: 4 lane quadrants x kParts column parts
constexpr int kParts = kEpW / 4;
constexpr int kCW = kN / kParts;   // key columns per epilogue thread and tile
constexpr int kCPL = kCW / 32;     // key columns per epilogue lane for the norm loads
constexpr int kThreads = (2 + kEpW) * 32;
constexpr int kTile = 128 * 128; // bytes of one 128-row x 64-element bf16 swizzled block

template <int D>
struct alignas(1024) MatchSmem {
  uint8_t a[2][D / 64][kTile];
  uint8_t b[kStages][D / 64][kN * 128];
  float invk[kEpW][kCW];
  float4 best[kParts][kQ];
  float qsq[kParts][kQ];     // per-unit shares of |q|^2 of every row, one per column part   // per-unit (m1, i1, m2) of every column part, merged in place
  uint64_t a_full, a_empty;
  uint64_t b_full[kStages], b_empty[kStages];
  uint64_t t_full[kTS], t_empty[kTS];
  uint32_t tmem_base;
  int abort;
};

struct MatchGeom {
  int H, QB, S;
  int q_token_major;   // Q's tensor map is (d, H, nq) instead of (d, nq, H)
  int64_t nq, M;
};

struct Unit {
  int h, qb, seg, nm, rows;
  int t_beg, t_end;   // key tiles [t_beg, t_end)
  int64_t n;
};

__device__ __forceinline__ Unit decode(const MatchGeom& g, int u, const int32_t* clen) {
  Unit w;
  w.seg = u % g.S;
  const int t = u / g.S;
  w.qb = t % g.QB;
  w.h = t / g.QB;
  const int64_t r = g.nq - (int64_t)w.qb * kQ;
  w.rows = (int)(r < kQ ? r : kQ);
  w.nm = (w.rows + 127) / 128;
  int64_t n = clen[w.h];
  n = n < 0 ? 0 : (n > g.M ? g.M : n);
  w.n = n;
  const int tiles = (int)((n + kN - 1) / kN);
  const int per = (tiles + g.S - 1) / g.S;
  w.t_beg = w.seg * per;
  w.t_end = w.t_beg + per < tiles ? w.t_beg + per : tiles;
  if (w.t_end < w.t_beg) w.t_end = w.t_beg;
  return w;
}

struct Best {
  float m1;
  int i1;
  float m2;
};

// (a, b) *= (x, y) with one packed f32x2 multiply (each lane rounded to nearest).
__device__ __forceinline__ void mul2(float& a, float& b, float x, float y) {
  unsigned long long p =
      (unsigned long long)__float_as_uint(a) | ((unsigned long long)__float_as_uint(b) << 32);
  const unsigned long long q =
      (unsigned long long)__float_as_uint(x) | ((unsigned long long)__float_as_uint(y) << 32);
  asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(p) : "l"(q));
  a = __uint_as_float((unsigned)(p & 0xffffffffull));
  b = __uint_as_float((unsigned)(p >> 32));
}

// Three-input maximum (sm_100-family PTX max.f32 with three sources).
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

template <bool kTop2>
__device__ __forceinline__ void fold16(Best& b, const float* w, int j0) {
  if (kTop2) {
    float a0 = max3f(w[0], w[1], w[2]), a1 = max3f(w[3], w[4], w[5]);
    float a2 = max3f(w[6], w[7], w[8]), a3 = max3f(w[9], w[10], w[11]);
    a0 = max3f(a0, w[12], w[13]);
    a1 = max3f(a1, w[14], w[15]);
    const float gm = max3f(a0, a1, fmaxf(a2, a3));
    if (gm > b.m2) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float v = w[i];
        if (v > b.m1) {
          b.m2 = b.m1;
          b.m1 = v;
          b.i1 = j0 + i;
        } else if (v > b.m2) {
          b.m2 = v;
        }
      }
    }
  } else {
    // maxima of four groups of consecutive columns, so that a new best is located by
    // its group first (the lowest group holding it, then the lowest column in it)
    const float g0 = fmaxf(max3f(w[0], w[1], w[2]), w[3]);
    const float g1 = fmaxf(max3f(w[4], w[5], w[6]), w[7]);
    const float g2 = fmaxf(max3f(w[8], w[9], w[10]), w[11]);
    const float g3 = fmaxf(max3f(w[12], w[13], w[14]), w[15]);
    const float gm = max3f(g0, g1, fmaxf(g2, g3));
    if (gm > b.m1) {
      const bool in0 = g0 == gm, in1 = g1 == gm, in2 = g2 == gm;
      const int base = in0 ? 0 : in1 ? 4 : in2 ? 8 : 12;
      const float x0 = in0 ? w[0] : in1 ? w[4] : in2 ? w[8] : w[12];
      const float x1 = in0 ? w[1] : in1 ? w[5] : in2 ? w[9] : w[13];
      const float x2 = in0 ? w[2] : in1 ? w[6] : in2 ? w[10] : w[14];
      const int k = x0 == gm ? 0 : x1 == gm ? 1 : x2 == gm ? 2 : 3;
      b.m1 = gm;
      b.i1 = j0 + base + k;
    }
  }
}

template <int D, bool kTop2>
__global__ void __launch_bounds__(kThreads, 1)
match_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const float* __restrict__ cknorm, const int32_t* __restrict__ clen, MatchGeom g,
                float4* __restrict__ part_out, uint8_t* __restrict__ evict, int32_t* __restrict__ owner,
                int32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  MatchSmem<D>& sm = *reinterpret_cast<MatchSmem<D>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int KH = D / 64;
  constexpr uint32_t kIdesc = tc::idesc_bf16_f32(128, kN);

  // clear the eviction flags and owners (the finaliser sets them after this kernel)
  {
    const int64_t total = (int64_t)g.H * g.M;
    for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < total; j += (int64_t)gridDim.x * blockDim.x) {
      evict[j] = 0;
      if (owner) owner[j] = -1;
    }
  }
  if (threadIdx.x == 0) {
    tc::mbar_init(&sm.a_full, 1);
    tc::mbar_init(&sm.a_empty, 1 + kEpW);   // the MMA's commit + the epilogue warps (|q|^2 read)
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&sm.b_full[s], 1);
      tc::mbar_init(&sm.b_empty[s], 1);
    }
    for (int s = 0; s < kTS; ++s) {
      tc::mbar_init(&sm.t_full[s], 1);
      tc::mbar_init(&sm.t_empty[s], kEpW);
    }
    sm.abort = 0;
    tc::mbar_fence_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(&sm.tmem_base, 512);
    tc::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tc::tma_prefetch_desc(&tm_q);
    tc::tma_prefetch_desc(&tm_k);
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort = &sm.abort;
  const int units = g.H * g.QB * g.S;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int stage = 0;
      uint32_t ph = 0, aph = 0;
      for (int u = blockIdx.x; u < units && !*abort; u += gridDim.x) {
        const Unit w = decode(g, u, clen);
        if (w.t_end <= w.t_beg) continue;
        if (!tc::mbar_wait(&sm.a_empty, aph ^ 1, abort)) break;
        aph ^= 1;
        tc::mbar_arrive_tx(&sm.a_full, (uint32_t)(w.nm * KH * kTile));
        for (int m = 0; m < w.nm; ++m)
          for (int kh = 0; kh < KH; ++kh)
            if (g.q_token_major)
              tc::tma_load_3d(sm.a[m][kh], &tm_q, kh * 64, w.h, w.qb * kQ + m * 128, &sm.a_full);
            else
              tc::tma_load_3d(sm.a[m][kh], &tm_q, kh * 64, w.qb * kQ + m * 128, w.h, &sm.a_full);
        for (int t = w.t_beg; t < w.t_end; ++t) {
          if (!tc::mbar_wait(&sm.b_empty[stage], ph ^ 1, abort)) break;
          tc::mbar_arrive_tx(&sm.b_full[stage], (uint32_t)(KH * kN * 128));
          for (int kh = 0; kh < KH; ++kh)
            tc::tma_load_3d(sm.b[stage][kh], &tm_k, kh * 64, t * kN, w.h, &sm.b_full[stage]);
          if (++stage == kStages) {
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
      // descriptors of the first block of A and of the B ring; every other operand
      // address is a compile-time offset from them (16-byte units in the low field)
      const uint64_t a_desc0 = tc::sw128_desc(tc::smem_u32(&sm.a[0][0][0]));
      const uint64_t b_desc0 = tc::sw128_desc(tc::smem_u32(&sm.b[0][0][0]));
      for (int u = blockIdx.x; u < units && !*abort; u += gridDim.x) {
        const Unit w = decode(g, u, clen);
        if (w.t_end <= w.t_beg) continue;
        if (!tc::mbar_wait(&sm.a_full, aph, abort)) break;
        aph ^= 1;
        tc::tc_fence_after();
        for (int t = w.t_beg; t < w.t_end; ++t) {
          if (!tc::mbar_wait(&sm.b_full[stage], ph, abort)) break;
          if (!tc::mbar_wait(&sm.t_empty[acc], tph ^ 1, abort)) break;
          tc::tc_fence_after();
          const uint64_t bd0 = b_desc0 + (uint64_t)((stage * KH * kN * 128) >> 4);
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            if (m < w.nm) {
              const uint32_t d = tmem + (uint32_t)(acc * 2 * kN + m * kN);
#pragma unroll
              for (int k = 0; k < D / 16; ++k) {
                const uint64_t ad = a_desc0 + (uint64_t)((m * KH * kTile + (k >> 2) * kTile + (k & 3) * 32) >> 4);
                const uint64_t bd = bd0 + (uint64_t)(((k >> 2) * kN * 128 + (k & 3) * 32) >> 4);
                tc::mma_bf16(d, ad, bd, kIdesc, k > 0 ? 1u : 0u);
              }
            }
          }
          tc::mma_commit(&sm.b_empty[stage]);
          tc::mma_commit(&sm.t_full[acc]);
          if (++stage == kStages) {
            stage = 0;
            ph ^= 1;
          }
          if (++acc == kTS) {
            acc = 0;
            tph ^= 1;
          }
        }
        tc::mma_commit(&sm.a_empty);
      }
    }
  } else {
    // ---------------- epilogue ----------------
    // kEpW warps: (lane quadrant, column part).  Each thread owns one query row in each
    // M-tile and kCW of the tile's key columns: it loads both rows' scores from TMEM,
    // hands the stage back to the MMA, then scales by 1/|k_j| and folds them into the
    // two running bests.
    static_assert(kCW == 32 && kCPL == 1, "one 32-column chunk per M-tile and tile");
    const int ew = warp - 2;          // 0..kEpW-1
    const int quad = warp & 3;        // TMEM lane quadrant this warp may access
    const int part = ew >> 2;         // which kCW-column part of the tile
    float* inv = sm.invk[ew];
    int acc = 0;
    uint32_t tph = 0;
    // Every epilogue warp walks every unit (no early exit on abort: after one, each
    // wait returns at once), so the two named barriers per unit always fill.
    uint32_t aph = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      const Unit w = decode(g, u, clen);
      const bool two = w.nm > 1;      // warp-uniform: the second M-tile holds queries
      Best b0{neg_inf(), INT_MAX, neg_inf()}, b1{neg_inf(), INT_MAX, neg_inf()};
      // this part's share of |q|^2 of both rows, from the unit's query tile (for the
      // finaliser's cosine; the parts' shares are summed in the merge below)
      // (a unit without key tiles loads no query tile and reports no match: nothing to read)
      if (w.t_end > w.t_beg) {
        float qs0 = 0.f, qs1 = 0.f;
        const int r0 = quad * 32 + lane;
        if (tc::mbar_wait(&sm.a_full, aph, abort)) {
#pragma unroll
          for (int i = 0; i < D / 32; ++i) {
            const int gc = part * (D / 32) + i;   // 16-byte chunk of the row
#pragma unroll
            for (int mm = 0; mm < 2; ++mm) {
              const uint4 v = *reinterpret_cast<const uint4*>(&sm.a[mm][gc >> 3][0] + tc::sw128_off(r0, gc & 7));
              const uint32_t x[4] = {v.x, v.y, v.z, v.w};
              float acc = 0.f;
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float lo = __uint_as_float(x[e] << 16), hi = __uint_as_float(x[e] & 0xffff0000u);
                acc = fmaf(lo, lo, acc);
                acc = fmaf(hi, hi, acc);
              }
              if (mm == 0) qs0 += acc; else qs1 += acc;
            }
          }
        }
        aph ^= 1;
        sm.qsq[part][r0] = qs0;
        sm.qsq[part][r0 + 128] = qs1;
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&sm.a_empty);
      }
      const float* kn = cknorm + (int64_t)w.h * g.M;
      // |k_j| of this lane's column of the first tile (prefetched one tile ahead)
      float kx = 0.f;
      if (w.t_beg < w.t_end) {
        const int64_t j = (int64_t)w.t_beg * kN + part * kCW + lane;
        kx = j < w.n ? kn[j] : 0.f;
      }
      for (int t = w.t_beg; t < w.t_end; ++t) {
        const int64_t j0 = (int64_t)t * kN + part * kCW;
        if (!tc::mbar_wait(&sm.t_full[acc], tph, abort)) break;
        tc::tc_fence_after();
        const uint32_t taddr =
            tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(acc * 2 * kN + part * kCW);
        // 1/|k_j| of this tile into the warp's buffer while the first TMEM loads are in flight
        float v0[16], v1[16];
        tc::tmem_ld16(taddr, v0);
        if (two) tc::tmem_ld16(taddr + (uint32_t)kN, v1);
        inv[lane] = kx > 0.f ? __frcp_rn(kx) : 0.f;
        // prefetch the next tile's norms
        if (t + 1 < w.t_end) {
          const int64_t j = j0 + kN + lane;
          kx = j < w.n ? kn[j] : 0.f;
        }
        __syncwarp();
        // two 16-column halves; each broadcast of four scales serves both M-tiles
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          if (c > 0) {
            tc::tmem_ld16(taddr + 16u, v0);
            if (two) tc::tmem_ld16(taddr + (uint32_t)kN + 16u, v1);
          }
          tc::tmem_wait_ld();
          tc::tmem_pin16(v0);
          if (two) tc::tmem_pin16(v1);
          if (c == 1) {
            // both rows' scores are in registers: hand the stage back to the MMA now
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&sm.t_empty[acc]);
          }
          // scale by 1/|k_j| two lanes at a time (packed f32x2 multiply, round to nearest)
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const float4 s = *reinterpret_cast<const float4*>(inv + c * 16 + q4 * 4);
            mul2(v0[q4 * 4 + 0], v0[q4 * 4 + 1], s.x, s.y);
            mul2(v0[q4 * 4 + 2], v0[q4 * 4 + 3], s.z, s.w);
            if (two) {
              mul2(v1[q4 * 4 + 0], v1[q4 * 4 + 1], s.x, s.y);
              mul2(v1[q4 * 4 + 2], v1[q4 * 4 + 3], s.z, s.w);
            }
          }
          const int64_t jc = j0 + c * 16;
          if (jc + 16 > w.n) {
#pragma unroll
            for (int x = 0; x < 16; ++x)
              if (jc + x >= w.n) v0[x] = v1[x] = neg_inf();
          }
          fold16<kTop2>(b0, v0, (int)jc);
          if (two) fold16<kTop2>(b1, v1, (int)jc);
        }
        if (++acc == kTS) {
          acc = 0;
          tph ^= 1;
        }
        __syncwarp();   // every lane is done with inv before the next tile rewrites it
      }
      // the four column parts of each row meet in shared memory; the part-0 warps merge
      // them (ties to the lower key index) and write one partial top-2 per segment
      const int r0 = quad * 32 + lane;
      sm.best[part][r0] = make_float4(b0.m1, __int_as_float(b0.i1), b0.m2, 0.f);
      sm.best[part][r0 + 128] = make_float4(b1.m1, __int_as_float(b1.i1), b1.m2, 0.f);
      tc::named_bar(1, kEpW * 32);
      if (part == 0) {
        const int64_t base = ((int64_t)w.seg * g.H + w.h) * g.nq + (int64_t)w.qb * kQ;
#pragma unroll
        for (int mm = 0; mm < 2; ++mm) {
          const int r = r0 + mm * 128;
          float4 a = sm.best[0][r];
          a.w = sm.qsq[0][r];
#pragma unroll
          for (int p2 = 1; p2 < kParts; ++p2) {
            const float4 c = sm.best[p2][r];
            a.w += sm.qsq[p2][r];   // |q|^2, summed over the parts in order
            if (beats(c.x, __float_as_int(c.y), a.x, __float_as_int(a.y))) {
              a.z = fmaxf(a.x, c.z);
              a.x = c.x;
              a.y = c.y;
            } else {
              a.z = fmaxf(a.z, c.x);
            }
          }
          if (r < w.rows && !*abort) part_out[base + r] = a;
        }
      }
      tc::named_bar(1, kEpW * 32);   // the merge has read sm.best before the next unit refills it
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && sm.abort) flag_status(status, FASTAR_DEV_TIMEOUT);
}

template <int D>
constexpr size_t match_tc_smem() {
  return sizeof(MatchSmem<D>) + 1024;
}

}  // namespace

int match_tc_splits(int H, int64_t nq, int64_t M) {
  const int nsm = sm_count();
  const int64_t qb = (nq + kQ - 1) / kQ;
  const int64_t tiles = (M + kN - 1) / kN;
  int best_s = 1;
  double best = 1e30;
  for (int s = 1; s <= 8; ++s) {
    const int64_t units = H * qb * s;
    const int64_t waves = (units + nsm - 1) / nsm;
    const double cost = (double)waves * ((double)((tiles + s - 1) / s) + 2.0);
    if (cost < best - 1e-9) {
      best = cost;
      best_s = s;
    }
  }
  return best_s;
}

size_t match_tc_workspace(int H, int64_t nq, int64_t M) {
  return sizeof(float4) * (size_t)8 * H * (size_t)nq;   // up to 8 segments
}

// Launches the tensor-core match (writes `part` as [S, H, nq] and clears evict).
// Returns the number of segments S the finaliser must merge, or -1 on a failure to
// set the kernel up (tensor maps, attributes).
template <int D>
static int launch_match_tc_impl(TokView q, int H, int64_t nq, const void* ck, const float* cknorm,
                                const int32_t* clen, int64_t M, bool top2, float4* part, uint8_t* evict,
                                int32_t* owner, int32_t* status, cudaStream_t s) {
  CUtensorMap tq, tk;
  const bool token_major = H > 1 && q.hs < q.ts;   // e.g. [N, H, d] storage
  if (token_major) {
    if (!make_tmap_bf16_3d(&tq, q.p, D, (uint64_t)H, (uint64_t)nq, (uint64_t)q.hs * 2, (uint64_t)q.ts * 2, 64, 1,
                           128))
      return -1;
  } else if (!make_tmap_bf16_3d(&tq, q.p, D, (uint64_t)nq, (uint64_t)H, (uint64_t)q.ts * 2, (uint64_t)q.hs * 2, 64,
                                128)) {
    return -1;
  }
  if (!make_tmap_bf16_3d(&tk, ck, D, (uint64_t)M, (uint64_t)H, (uint64_t)D * 2, (uint64_t)M * D * 2, 64, kN))
    return -1;
  MatchGeom g;
  g.H = H;
  g.nq = nq;
  g.M = M;
  g.QB = (int)((nq + kQ - 1) / kQ);
  g.q_token_major = token_major ? 1 : 0;
  g.S = match_tc_splits(H, nq, M);
  const int units = g.H * g.QB * g.S;
  const int grid = units < sm_count() ? units : sm_count();
  constexpr size_t smem = match_tc_smem<D>();
  if (top2) {
    const cudaError_t a = opt_in_smem((const void*)match_tc_kernel<D, true>, (int)smem);
    if (a != cudaSuccess) return -1;
    match_tc_kernel<D, true><<<grid, kThreads, smem, s>>>(tq, tk, cknorm, clen, g, part, evict, owner, status);
  } else {
    const cudaError_t a = opt_in_smem((const void*)match_tc_kernel<D, false>, (int)smem);
    if (a != cudaSuccess) return -1;
    match_tc_kernel<D, false><<<grid, kThreads, smem, s>>>(tq, tk, cknorm, clen, g, part, evict, owner, status);
  }
  count_launches(1);
  return g.S;   // partial top-2s, one per segment
}

int launch_match_tc(int d, TokView q, int H, int64_t nq, const void* ck, const float* cknorm, const int32_t* clen,
                    int64_t M, bool top2, float4* part, uint8_t* evict, int32_t* owner, int32_t* status,
                    cudaStream_t s) {
  if (d == 128) return launch_match_tc_impl<128>(q, H, nq, ck, cknorm, clen, M, top2, part, evict, owner, status, s);
  return launch_match_tc_impl<64>(q, H, nq, ck, cknorm, clen, M, top2, part, evict, owner, status, s);
}

}  // namespace fastar
