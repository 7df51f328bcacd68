// Softmax attention over gathered key sets on the 5th-generation tensor cores (bf16).
//
// Serves the three attention rows of the step with one engine:
//   sparse — AnnSA (FAST-AR technical summary §2.C, blog §3): the (query, slot) pairs
//            of one bucket against that bucket's cache keys, one fp32 partial (o, lse)
//            per pair (merged over the r slots afterwards);
//   cross  — AnnCA (technical summary §2.B, blog §2): one latent frame's queries
//            against its kept prompt tokens;
//   dense  — the dense baseline (technical summary, Key Results): every key.
//
// One CTA per 128-query tile, warp-specialised:
//   warps 0-3  gather rows with 16-byte cp.async into 128-byte-swizzled tiles (the
//              Q tile once, then K and V tiles through a 2-deep ring, warps 0-1 the
//              even tiles and 2-3 the odd ones), fence them to the async proxy and
//              arrive on mbarriers;
//   warp 4     owns TMEM (S0, S1: 2 x 128 columns, O: d columns) and issues
//              tcgen05.mma from one thread: S_j = Q K_j^T into S[j%2] as soon as
//              K_j is in, then O += P_j V_j once the softmax has written P_j —
//              so QK_{j+1} overlaps the softmax of tile j;
//   warps 5-8  softmax, one query row per thread: S row from TMEM, running max in
//              log2 units with lazy rescaling (O in TMEM is rescaled only when the
//              max grows by more than 2^8), P as bf16 into shared memory, and the
//              final O / l written out.
// Every wait is bounded; a timeout sets FASTAR_DEV_TIMEOUT and unwinds.
#include <climits>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace fastar {
namespace {

constexpr int kAT = 128;         // query rows per CTA and keys per tile
constexpr int kKV = 2;           // K/V ring depth
constexpr int kThreadsA = 288;   // 9 warps
constexpr int kBlkA = 128 * 128; // one 128-row x 64-element bf16 block (128-B swizzle)
constexpr int kMmaWarpA = 4;

template <int D>
struct alignas(1024) AttnSmem {
  uint8_t q[D / 64][kBlkA];
  uint8_t k[kKV][D / 64][kBlkA];
  uint8_t v[kKV][D / 64][kBlkA];
  uint8_t p[2][kBlkA];
  int64_t qsrc[kAT];
  int64_t ksrc[kKV][kAT];
  int qdst[kAT];
  int pre[FASTAR_MAX_B + 1];
  uint64_t q_full;
  uint64_t kv_full[kKV], kv_empty[kKV];
  uint64_t s_full[2], s_free[2];
  uint64_t p_full, p_empty;
  uint32_t tmem_base;
  int abort;
  int item[4];       // valid, h, bucket (sparse) / frame (cross)
  int64_t range[3];  // query range begin/end (sparse: positions in qperm; else token index), key base
  int64_t nkeys;
};

__device__ __forceinline__ bool wait_all(uint64_t* bar, uint32_t parity, volatile int* abort) {
  const bool ok = tc::mbar_wait(bar, parity, abort);
  return __all_sync(0xffffffffu, ok);
}

// 2^x with the SFU's approximate base-2 exponential (PTX ex2.approx; 2^-inf = 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <int D>
__global__ void __launch_bounds__(kThreadsA, 1) attn_tc_kernel(const AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  AttnSmem<D>& sm = *reinterpret_cast<AttnSmem<D>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  constexpr int KH = D / 64;
  constexpr int CPR = D / 8;   // 16-byte chunks per row
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const __nv_bfloat16* Q = static_cast<const __nv_bfloat16*>(a.q.p);
  const __nv_bfloat16* K = static_cast<const __nv_bfloat16*>(a.k);
  const __nv_bfloat16* V = static_cast<const __nv_bfloat16*>(a.v);
  const int h = blockIdx.y;
  const int64_t np = a.nq * a.r;

  if (threadIdx.x == 0) {
    tc::mbar_init(&sm.q_full, 128);
    for (int s = 0; s < kKV; ++s) {
      tc::mbar_init(&sm.kv_full[s], 64);   // one loader group of 64 threads per stage
      tc::mbar_init(&sm.kv_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&sm.s_full[s], 1);
      tc::mbar_init(&sm.s_free[s], 4);
    }
    tc::mbar_init(&sm.p_full, 4);
    tc::mbar_init(&sm.p_empty, 1);
    sm.abort = 0;
    // decode the work item
    int valid = 1;
    if (a.mode == kSparse) {
      const int32_t* qo = a.qoff + (int64_t)h * (a.B + 1);
      int acc = 0;
      for (int b = 0; b < a.B; ++b) {
        sm.pre[b] = acc;
        const int c = qo[b + 1] - qo[b];
        acc += c > 0 ? (c + kAT - 1) / kAT : 0;
      }
      int b = -1;
      if ((int)blockIdx.x < acc) {
        int lo = 0, hi = a.B - 1;
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (sm.pre[mid] <= (int)blockIdx.x) lo = mid; else hi = mid - 1;
        }
        b = lo;
      }
      valid = b >= 0;
      if (valid) {
        const int64_t q0 = qo[b] + (int64_t)(blockIdx.x - sm.pre[b]) * kAT;
        const int64_t q1 = qo[b + 1];
        sm.range[0] = q0;
        sm.range[1] = q0 + kAT < q1 ? q0 + kAT : q1;
        const int32_t* ko = a.koff + (int64_t)h * (a.B + 1);
        sm.range[2] = ko[b];
        sm.nkeys = ko[b + 1] - ko[b];
        if (sm.nkeys < 0 || sm.range[2] < 0 || sm.range[2] + sm.nkeys > a.M) {
          flag_status(a.status, FASTAR_DEV_BAD_INDEX);
          sm.nkeys = 0;
        }
      }
      sm.item[2] = b;
    } else if (a.mode == kCross) {
      const int f = blockIdx.z;
      const int64_t t0 = (int64_t)blockIdx.x * kAT;
      sm.range[0] = (int64_t)f * a.tpf + t0;
      sm.range[1] = (int64_t)f * a.tpf + (t0 + kAT < a.tpf ? t0 + kAT : a.tpf);
      int64_t nk = a.kcnt[(int64_t)h * a.F + f];
      if (nk < 0 || nk > a.P) {
        flag_status(a.status, FASTAR_DEV_BAD_INDEX);
        nk = nk < 0 ? 0 : a.P;
      }
      sm.nkeys = nk;
      sm.item[2] = f;
    } else {
      const int64_t i0 = (int64_t)blockIdx.x * kAT;
      sm.range[0] = i0;
      sm.range[1] = i0 + kAT < a.nq ? i0 + kAT : a.nq;
      sm.nkeys = a.nk;
    }
    sm.item[0] = valid;
    tc::mbar_fence_init();
  }
  __syncthreads();
  // query rows of the tile: source offset and output row (read by the loaders and,
  // at the end, by the softmax warps)
  if (threadIdx.x < kAT) {
    const int lt = threadIdx.x;
    const int64_t pos = sm.range[0] + lt;
    int64_t src = -1;
    int dst = -1;
    if (sm.item[0] && pos < sm.range[1]) {
      if (a.mode == kSparse) {
        const int e = a.qperm[(int64_t)h * np + pos];
        if (e >= 0 && e < np) {
          src = h * a.q.hs + (int64_t)(e / a.r) * a.q.ts;
          dst = e;
        } else {
          flag_status(a.status, FASTAR_DEV_BAD_INDEX);
        }
      } else {
        src = h * a.q.hs + pos * a.q.ts;
        dst = (int)pos;
      }
    }
    sm.qsrc[lt] = src;
    sm.qdst[lt] = dst;
  }
  if (warp == kMmaWarpA) {
    tc::tmem_alloc(&sm.tmem_base, 512);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort = &sm.abort;
  const bool valid = sm.item[0] != 0;
  const int64_t nkeys = valid ? sm.nkeys : 0;
  const int T = (int)((nkeys + kAT - 1) / kAT);

  if (valid && warp < 4) {
    // ---------------- row gathers (128 threads) ----------------
    const int lt = threadIdx.x;
#pragma unroll 4
    for (int g = lt; g < kAT * CPR; g += 128) {
      const int row = g / CPR, c = g % CPR;
      const int64_t s = sm.qsrc[row];
      tc::cp_async16(tc::smem_u32(sm.q[c >> 3]) + tc::sw128_off(row, c & 7), s >= 0 ? Q + s + c * 8 : Q,
                     s >= 0 ? 16u : 0u);
    }
    tc::cp_async_commit();
    tc::cp_async_wait<0>();
    tc::fence_proxy_async();
    tc::mbar_arrive(&sm.q_full);
    // K/V tiles: warps 0-1 load the even tiles into stage 0, warps 2-3 the odd ones
    // into stage 1, so two tiles are in flight and each group signals its own tile
    // as soon as it has landed (no group waits on the other's progress).
    const int grp = warp >> 1;
    const int gt = threadIdx.x & 63;
    for (int j = grp; j < T && !*abort; j += kKV) {
      const int st = grp;
      if (!tc::mbar_wait(&sm.kv_empty[st], ((j / kKV) & 1) ^ 1, abort)) break;
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int row = gt + rr * 64;
        const int64_t u = (int64_t)j * kAT + row;
        int64_t off = -1;
        if (u < nkeys) {
          if (a.mode == kSparse) {
            const int s = a.kperm[(int64_t)h * a.M + sm.range[2] + u];
            if (s >= 0 && s < a.M) off = ((int64_t)h * a.M + s) * D;
            else flag_status(a.status, FASTAR_DEV_BAD_INDEX);
          } else if (a.mode == kCross) {
            const int p = a.kidx[((int64_t)h * a.F + sm.item[2]) * a.P + u];
            if (p >= 0 && p < a.P) off = ((int64_t)h * a.P + p) * D;
            else flag_status(a.status, FASTAR_DEV_BAD_INDEX);
          } else {
            off = h * a.kv_hs + u * a.kv_ts;
          }
        }
        sm.ksrc[st][row] = off;
      }
      tc::named_bar(1 + grp, 64);
#pragma unroll 4
      for (int g = gt; g < kAT * CPR; g += 64) {
        const int row = g / CPR, c = g % CPR;
        const int64_t s = sm.ksrc[st][row];
        const uint32_t o = tc::sw128_off(row, c & 7);
        tc::cp_async16(tc::smem_u32(sm.k[st][c >> 3]) + o, s >= 0 ? K + s + c * 8 : K, s >= 0 ? 16u : 0u);
        tc::cp_async16(tc::smem_u32(sm.v[st][c >> 3]) + o, s >= 0 ? V + s + c * 8 : V, s >= 0 ? 16u : 0u);
      }
      tc::cp_async_commit();
      tc::cp_async_wait<0>();
      tc::fence_proxy_async();
      tc::mbar_arrive(&sm.kv_full[st]);
    }
  } else if (valid && warp == kMmaWarpA) {
    // ---------------- MMA issuer ----------------
    if (lane == 0 && T > 0) {
      constexpr uint32_t idesc_qk = tc::idesc_bf16_f32(128, kAT);
      constexpr uint32_t idesc_pv = tc::idesc_bf16_f32_bmn(128, D);
      auto issue_qk = [&](int j) -> bool {
        const int st = j % kKV, b = j & 1;
        if (!tc::mbar_wait(&sm.kv_full[st], (j / kKV) & 1, abort)) return false;
        if (!tc::mbar_wait(&sm.s_free[b], ((j >> 1) & 1) ^ 1, abort)) return false;
        tc::tc_fence_after();
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t ko = (uint32_t)((k & 3) * 32);
          tc::mma_bf16(tmem + (uint32_t)(b * 128), tc::sw128_desc(tc::smem_u32(sm.q[k >> 2]) + ko),
                       tc::sw128_desc(tc::smem_u32(sm.k[st][k >> 2]) + ko), idesc_qk, k > 0 ? 1u : 0u);
        }
        tc::mma_commit(&sm.s_full[b]);
        return true;
      };
      bool ok = tc::mbar_wait(&sm.q_full, 0, abort);
      if (ok) tc::tc_fence_after();
      ok = ok && issue_qk(0);
      for (int j = 0; j < T && ok; ++j) {
        if (j + 1 < T && !issue_qk(j + 1)) break;
        if (!tc::mbar_wait(&sm.p_full, j & 1, abort)) break;
        tc::tc_fence_after();
        const int st = j % kKV;
#pragma unroll
        for (int ks = 0; ks < kAT / 16; ++ks) {
          const uint64_t ad = tc::sw128_desc(tc::smem_u32(sm.p[ks >> 2]) + (uint32_t)((ks & 3) * 32));
          const uint64_t bd = tc::sw128_mn_desc(tc::smem_u32(sm.v[st][0]) + (uint32_t)(ks * 2048), kBlkA);
          tc::mma_bf16(tmem + 256u, ad, bd, idesc_pv, (j > 0 || ks > 0) ? 1u : 0u);
        }
        tc::mma_commit(&sm.kv_empty[st]);
        tc::mma_commit(&sm.p_empty);
      }
    }
  } else if (valid && warp >= 5) {
    // ---------------- softmax and output ----------------
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
    const float sl2 = a.scale * 1.4426950408889634f;   // scores in log2 units
    float m_used = neg_inf(), l = 0.f;
    bool ok = true;
    for (int j = 0; j < T; ++j) {
      const int b = j & 1;
      if (!wait_all(&sm.s_full[b], (j >> 1) & 1, abort)) {
        ok = false;
        break;
      }
      tc::tc_fence_after();
      float x[kAT];
#pragma unroll
      for (int c = 0; c < kAT / 32; ++c) tc::tmem_ld32(tmem + lane_addr + (uint32_t)(b * 128 + c * 32), x + c * 32);
      tc::tmem_wait_ld();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sm.s_free[b]);
      const int64_t left = nkeys - (int64_t)j * kAT;
      const int vcols = left < kAT ? (int)left : kAT;
      float mt = neg_inf();
#pragma unroll
      for (int i = 0; i < kAT; ++i) {
        x[i] = i < vcols ? x[i] * sl2 : neg_inf();
        mt = fmaxf(mt, x[i]);
      }
      float alpha = 1.f;
      bool resc = false;
      if (mt > m_used + 8.f) {
        resc = m_used != neg_inf();
        alpha = resc ? ex2(m_used - mt) : 0.f;
        m_used = mt;
      }
      float sum = 0.f;
      uint32_t pk[kAT / 2];
#pragma unroll
      for (int i = 0; i < kAT; i += 2) {
        const float p0 = m_used == neg_inf() ? 0.f : ex2(x[i] - m_used);
        const float p1 = m_used == neg_inf() ? 0.f : ex2(x[i + 1] - m_used);
        sum += p0 + p1;
        pk[i >> 1] = pack_bf16(p0, p1);
      }
      l = l * alpha + sum;
      if (j > 0 && !wait_all(&sm.p_empty, (j - 1) & 1, abort)) {
        ok = false;
        break;
      }
      tc::tc_fence_after();
      if (__any_sync(0xffffffffu, resc)) {
        const float f = resc ? alpha : 1.f;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          tc::tmem_ld32(tmem + lane_addr + 256u + (uint32_t)(c * 32), o);
          tc::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= f;
          tc::tmem_st32(tmem + lane_addr + 256u + (uint32_t)(c * 32), o);
        }
        tc::tmem_wait_st();
      }
#pragma unroll
      for (int c16 = 0; c16 < kAT / 8; ++c16) {
        const uint32_t addr = tc::smem_u32(sm.p[c16 >> 3]) + tc::sw128_off(row, c16 & 7);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[c16 * 4]),
                     "r"(pk[c16 * 4 + 1]), "r"(pk[c16 * 4 + 2]), "r"(pk[c16 * 4 + 3])
                     : "memory");
      }
      tc::fence_proxy_async();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sm.p_full);
    }
    if (ok && T > 0 && !wait_all(&sm.p_empty, (T - 1) & 1, abort)) ok = false;
    tc::tc_fence_after();
    const int dst = sm.qdst[row];
    const bool live = ok && T > 0 && l > 0.f;
    const float inv = live ? 1.0f / l : 0.f;
    const float lse = live ? (m_used + __log2f(l)) * 0.6931471805599453f : neg_inf();
#pragma unroll 1
    for (int c = 0; c < D / 32; ++c) {
      float o[32];
      if (ok && T > 0) {
        tc::tmem_ld32(tmem + lane_addr + 256u + (uint32_t)(c * 32), o);
        tc::tmem_wait_ld();
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = 0.f;
      }
      if (dst >= 0 && ok) {
        if (a.mode == kSparse) {
          float4* po = reinterpret_cast<float4*>(a.part_o + ((int64_t)h * np + dst) * D + c * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            po[i] = make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv, o[4 * i + 3] * inv);
        } else {
          uint4* po = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + h * a.o_hs +
                                               (int64_t)dst * a.o_ts + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            po[i] = make_uint4(pack_bf16(o[8 * i] * inv, o[8 * i + 1] * inv), pack_bf16(o[8 * i + 2] * inv, o[8 * i + 3] * inv),
                               pack_bf16(o[8 * i + 4] * inv, o[8 * i + 5] * inv), pack_bf16(o[8 * i + 6] * inv, o[8 * i + 7] * inv));
        }
      }
    }
    if (dst >= 0 && ok) {
      if (a.mode == kSparse) {
        a.part_lse[(int64_t)h * np + dst] = lse;
      } else if (a.lse) {
        const int64_t nrow = a.mode == kCross ? (int64_t)a.F * a.tpf : a.nq;
        a.lse[(int64_t)h * nrow + dst] = lse;
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarpA) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && sm.abort) flag_status(a.status, FASTAR_DEV_TIMEOUT);
}

template <int D>
constexpr size_t attn_tc_smem() {
  return sizeof(AttnSmem<D>) + 1024;
}

template <int D>
bool attn_tc_impl(const AttnArgs& a, cudaStream_t s) {
  dim3 grid;
  if (a.mode == kDense) {
    grid = dim3((unsigned)((a.nq + kAT - 1) / kAT), a.H, 1);
  } else if (a.mode == kCross) {
    grid = dim3((unsigned)((a.tpf + kAT - 1) / kAT), a.H, a.F);
  } else {
    grid = dim3((unsigned)((a.nq * a.r + kAT - 1) / kAT + a.B), a.H, 1);
  }
  constexpr size_t smem = attn_tc_smem<D>();
  static const cudaError_t attr =
      cudaFuncSetAttribute(attn_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (attr != cudaSuccess) return false;
  attn_tc_kernel<D><<<grid, kThreadsA, smem, s>>>(a);
  count_launches(1);
  return true;
}

}  // namespace

bool launch_attn_tc(int d, const AttnArgs& a, cudaStream_t s) {
  return d == 128 ? attn_tc_impl<128>(a, s) : attn_tc_impl<64>(a, s);
}

}  // namespace fastar
