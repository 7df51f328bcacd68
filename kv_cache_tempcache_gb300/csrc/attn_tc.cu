// Softmax attention over gathered key sets on the 5th-generation tensor cores (bf16).
//
// Serves the three attention rows of the step with one engine:
//   sparse — AnnSA (FAST-AR technical summary §2.C, blog §3): the (query, slot) pairs
//            of one bucket against that bucket's cache keys; the r slots of a query
//            use disjoint key sets (every key has one bucket), so their partial
//            (o, lse) merge exactly — the last slot to finish merges them in place;
//   cross  — AnnCA (technical summary §2.B, blog §2): one latent frame's queries
//            against its kept prompt tokens;
//   dense  — the dense baseline (technical summary, Key Results): every key.
//
// One CTA per 128-query tile, warp-specialised:
//   warps 0-3  gather rows with 16-byte cp.async into 128-byte-swizzled tiles, fence
//              them to the async proxy and arrive on mbarriers;
//   warp 4     owns TMEM and issues tcgen05.mma from one thread: S_j = Q K_j^T, then
//              O += P_j V_j once the softmax has written P_j;
//   warps 5-8  softmax, one query row per thread: S row from TMEM, running max in
//              log2 units with lazy rescaling (O in TMEM is rescaled only when the
//              max grows by more than 2^8), P as bf16 into shared memory, and the
//              final O / l written out.
// Two variants (template KV):
//   KV = 2  streaming: a 2-deep K/V ring (warps 0-1 load even tiles, 2-3 odd ones),
//           S double-buffered in TMEM so QK_{j+1} overlaps the softmax of tile j.
//           For long key lists (the dense baseline).  ~195 KB shared, 1 CTA/SM.
//   KV = 1  compact: one K/V stage, one S buffer, P written over the consumed K tile
//           (d = 128).  ~100 KB shared and 256 TMEM columns, so two CTAs share an SM
//           and hide each other's gather latency.  For the short per-bucket and
//           per-frame lists of AnnSA and AnnCA.
// Every wait is bounded; a timeout sets FASTAR_DEV_TIMEOUT and unwinds.
#include <climits>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace fastar {
namespace {

constexpr int kAT = 128;         // query rows per CTA and keys per tile
constexpr int kThreadsA = 288;   // 9 warps
constexpr int kBlkA = 128 * 128; // one 128-row x 64-element bf16 block (128-B swizzle)
constexpr int kMmaWarpA = 4;

struct AttnCtl {
  int64_t qsrc[kAT];
  int64_t ksrc[2][kAT];
  int qdst[kAT];
  int pre[FASTAR_MAX_B + 1];
  int wsum[kThreadsA / 32];
  uint64_t q_full;
  uint64_t kv_full[2], kv_empty[2];
  uint64_t s_full[2], s_free[2];
  uint64_t p_full, p_empty;
  uint32_t tmem_base;
  int abort;
  int item[4];       // valid, -, bucket (sparse) / frame (cross)
  int64_t range[3];  // query range begin/end (sparse: positions in qperm; else token index), key base
  int64_t nkeys;
};

// Shared-memory layout (bytes from the 1024-aligned base).
template <int D, int KV>
struct AttnLayout {
  static constexpr int KH = D / 64;
  static constexpr bool kPAliasK = (KV == 1 && D == 128);   // P (32 KB) over the consumed K tile
  static constexpr size_t q = 0;
  static constexpr size_t k = q + (size_t)KH * kBlkA;
  static constexpr size_t v = k + (size_t)KV * KH * kBlkA;
  static constexpr size_t p = kPAliasK ? k : v + (size_t)KV * KH * kBlkA;
  static constexpr size_t ctl = (kPAliasK ? v + (size_t)KV * KH * kBlkA : p + 2 * (size_t)kBlkA);
  static constexpr size_t bytes = ctl + sizeof(AttnCtl) + 1024;
  static constexpr uint32_t tmem_cols = KV == 2 ? 512 : 256;   // S buffers (KV x 128) + O (128)
  static constexpr uint32_t o_col = KV * 128;
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

// Element offset of key u of the CTA's key list (-1 if out of range).
__device__ __forceinline__ int64_t key_offset(const AttnArgs& a, const AttnCtl& c, int h, int64_t u, int D) {
  if (u >= c.nkeys) return -1;
  if (a.mode == kSparse) {
    const int s = a.kperm[(int64_t)h * a.M + c.range[2] + u];
    if (s >= 0 && s < a.M) return ((int64_t)h * a.M + s) * D;
    flag_status(a.status, FASTAR_DEV_BAD_INDEX);
    return -1;
  }
  if (a.mode == kCross) {
    const int p = a.kidx[((int64_t)h * a.F + c.item[2]) * a.P + u];
    if (p >= 0 && p < a.P) return ((int64_t)h * a.P + p) * D;
    flag_status(a.status, FASTAR_DEV_BAD_INDEX);
    return -1;
  }
  return h * a.kv_hs + u * a.kv_ts;
}

template <int D, int KV>
__global__ void __launch_bounds__(kThreadsA, KV == 1 ? 2 : 1) attn_tc_kernel(const AttnArgs a) {
  using Lay = AttnLayout<D, KV>;
  constexpr int KH = D / 64;
  constexpr int CPR = D / 8;   // 16-byte chunks per row
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sq = base + Lay::q;
  uint8_t* sk = base + Lay::k;   // [KV][KH][kBlkA]
  uint8_t* sv = base + Lay::v;   // [KV][KH][kBlkA]
  uint8_t* sp = base + Lay::p;   // [2][kBlkA]
  AttnCtl& sm = *reinterpret_cast<AttnCtl*>(base + Lay::ctl);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const __nv_bfloat16* Q = static_cast<const __nv_bfloat16*>(a.q.p);
  const __nv_bfloat16* K = static_cast<const __nv_bfloat16*>(a.k);
  const __nv_bfloat16* V = static_cast<const __nv_bfloat16*>(a.v);
  const int h = blockIdx.y;
  const int64_t np = a.nq * a.r;

  if (a.mode == kSparse) {
    // exclusive prefix over buckets of their 128-pair tile counts, all threads at once
    const int t = threadIdx.x;
    const int32_t* qo = a.qoff + (int64_t)h * (a.B + 1);
    int v = 0;
    if (t < a.B) {
      const int c = qo[t + 1] - qo[t];
      v = c > 0 ? (c + kAT - 1) / kAT : 0;
    }
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) sm.wsum[warp] = incl;
    __syncthreads();
    if (t == 0) {
      int run = 0;
      for (int w2 = 0; w2 < kThreadsA / 32; ++w2) {
        const int x = sm.wsum[w2];
        sm.wsum[w2] = run;
        run += x;
      }
    }
    __syncthreads();
    if (t < a.B) sm.pre[t] = sm.wsum[warp] + incl - v;
    if (t == a.B - 1) sm.pre[a.B] = sm.wsum[warp] + incl;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    tc::mbar_init(&sm.q_full, 128);
    for (int s = 0; s < KV; ++s) {
      tc::mbar_init(&sm.kv_full[s], KV == 2 ? 64 : 128);   // the loader group of the stage
      tc::mbar_init(&sm.kv_empty[s], 1);
    }
    for (int s = 0; s < KV; ++s) {
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
      const int acc = sm.pre[a.B];
      int b = -1;
      if ((int)blockIdx.x < acc) {
        int lo = 0, hi = a.B - 1;   // last b with pre[b] <= blockIdx.x
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
  if (!sm.item[0]) return;   // no work for this CTA (uniform; nothing allocated yet)
  // query rows of the tile: source offset and output row
  if (threadIdx.x < kAT) {
    const int lt = threadIdx.x;
    const int64_t pos = sm.range[0] + lt;
    int64_t src = -1;
    int dst = -1;
    if (pos < sm.range[1]) {
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
    tc::tmem_alloc(&sm.tmem_base, Lay::tmem_cols);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort = &sm.abort;
  const int64_t nkeys = sm.nkeys;
  const int T = (int)((nkeys + kAT - 1) / kAT);

  if (warp < 4) {
    // ---------------- row gathers (128 threads) ----------------
    const int lt = threadIdx.x;
#pragma unroll 4
    for (int g = lt; g < kAT * CPR; g += 128) {
      const int row = g / CPR, c = g % CPR;
      const int64_t s = sm.qsrc[row];
      tc::cp_async16(tc::smem_u32(sq + (c >> 3) * kBlkA) + tc::sw128_off(row, c & 7), s >= 0 ? Q + s + c * 8 : Q,
                     s >= 0 ? 16u : 0u);
    }
    tc::cp_async_commit();
    tc::cp_async_wait<0>();
    tc::fence_proxy_async();
    tc::mbar_arrive(&sm.q_full);
    // K/V tiles.  KV = 2: warps 0-1 load the even tiles into stage 0, warps 2-3 the odd
    // ones into stage 1 (two tiles in flight, each group signals its own tile).
    // KV = 1: all four warps load every tile into the single stage.
    constexpr int GT = KV == 2 ? 64 : 128;
    const int grp = KV == 2 ? (warp >> 1) : 0;
    const int gt = threadIdx.x & (GT - 1);
    for (int j = grp; j < T && !*abort; j += KV) {
      const int st = grp;
      if (!tc::mbar_wait(&sm.kv_empty[st], ((j / KV) & 1) ^ 1, abort)) break;
      for (int row = gt; row < kAT; row += GT) sm.ksrc[st][row] = key_offset(a, sm, h, (int64_t)j * kAT + row, D);
      tc::named_bar(1 + grp, GT);
      uint8_t* kst = sk + (size_t)st * KH * kBlkA;
      uint8_t* vst = sv + (size_t)st * KH * kBlkA;
#pragma unroll 4
      for (int g = gt; g < kAT * CPR; g += GT) {
        const int row = g / CPR, c = g % CPR;
        const int64_t s = sm.ksrc[st][row];
        const uint32_t o = (uint32_t)((c >> 3) * kBlkA) + tc::sw128_off(row, c & 7);
        tc::cp_async16(tc::smem_u32(kst) + o, s >= 0 ? K + s + c * 8 : K, s >= 0 ? 16u : 0u);
        tc::cp_async16(tc::smem_u32(vst) + o, s >= 0 ? V + s + c * 8 : V, s >= 0 ? 16u : 0u);
      }
      tc::cp_async_commit();
      tc::cp_async_wait<0>();
      tc::fence_proxy_async();
      tc::mbar_arrive(&sm.kv_full[st]);
    }
  } else if (warp == kMmaWarpA) {
    // ---------------- MMA issuer ----------------
    if (lane == 0 && T > 0) {
      constexpr uint32_t idesc_qk = tc::idesc_bf16_f32(128, kAT);
      constexpr uint32_t idesc_pv = tc::idesc_bf16_f32_bmn(128, D);
      const uint64_t q_desc = tc::sw128_desc(tc::smem_u32(sq));
      const uint64_t k_desc = tc::sw128_desc(tc::smem_u32(sk));
      const uint64_t p_desc = tc::sw128_desc(tc::smem_u32(sp));
      const uint64_t v_desc = tc::sw128_mn_desc(tc::smem_u32(sv), kBlkA);
      auto issue_qk = [&](int j) -> bool {
        const int st = j % KV, b = j % KV;
        if (!tc::mbar_wait(&sm.kv_full[st], (j / KV) & 1, abort)) return false;
        if (!tc::mbar_wait(&sm.s_free[b], ((j / KV) & 1) ^ 1, abort)) return false;
        tc::tc_fence_after();
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (uint32_t)((k >> 2) * kBlkA + (k & 3) * 32);
          tc::mma_bf16(tmem + (uint32_t)(b * 128), q_desc + (off >> 4),
                       k_desc + ((uint32_t)(st * KH * kBlkA + off) >> 4), idesc_qk, k > 0 ? 1u : 0u);
        }
        tc::mma_commit(&sm.s_full[b]);
        return true;
      };
      auto issue_pv = [&](int j) -> bool {
        if (!tc::mbar_wait(&sm.p_full, j & 1, abort)) return false;
        tc::tc_fence_after();
        const int st = j % KV;
#pragma unroll
        for (int ks = 0; ks < kAT / 16; ++ks) {
          const uint32_t aoff = (uint32_t)((ks >> 2) * kBlkA + (ks & 3) * 32);
          const uint32_t boff = (uint32_t)(st * KH * kBlkA + ks * 2048);
          tc::mma_bf16(tmem + Lay::o_col, p_desc + (aoff >> 4), v_desc + (boff >> 4), idesc_pv,
                       (j > 0 || ks > 0) ? 1u : 0u);
        }
        tc::mma_commit(&sm.kv_empty[st]);
        tc::mma_commit(&sm.p_empty);
        return true;
      };
      bool ok = tc::mbar_wait(&sm.q_full, 0, abort);
      if (ok) tc::tc_fence_after();
      ok = ok && issue_qk(0);
      for (int j = 0; j < T && ok; ++j) {
        if (KV == 2) {
          // the next score tile goes into the other S buffer while the softmax runs
          if (j + 1 < T && !issue_qk(j + 1)) break;
          if (!issue_pv(j)) break;
        } else {
          // one stage: the next K tile can only land once PV_j has consumed this one
          if (!issue_pv(j)) break;
          if (j + 1 < T && !issue_qk(j + 1)) break;
        }
      }
    }
  } else {
    // ---------------- softmax and output ----------------
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
    const float sl2 = a.scale * 1.4426950408889634f;   // scores in log2 units
    float m_used = neg_inf(), l = 0.f;
    bool ok = true;
    for (int j = 0; j < T; ++j) {
      const int b = j % KV;
      if (!wait_all(&sm.s_full[b], (j / KV) & 1, abort)) {
        ok = false;
        break;
      }
      tc::tc_fence_after();
      const int64_t left = nkeys - (int64_t)j * kAT;
      const int vcols = left < kAT ? (int)left : kAT;
      if (KV == 1) {
        // compact variant (two CTAs per SM, ~100 registers): two passes over the S row in
        // TMEM, 32 columns at a time — the row maximum, then exp / pack / store of P
        float mt = neg_inf();
#pragma unroll 1
        for (int c = 0; c < kAT / 32; ++c) {
          float x[32];
          tc::tmem_ld32(tmem + lane_addr + (uint32_t)(c * 32), x);
          tc::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) mt = fmaxf(mt, c * 32 + i < vcols ? x[i] * sl2 : neg_inf());
        }
        float alpha = 1.f;
        bool resc = false;
        if (mt > m_used + 8.f) {
          resc = m_used != neg_inf();
          alpha = resc ? ex2(m_used - mt) : 0.f;
          m_used = mt;
        }
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
            tc::tmem_ld32(tmem + lane_addr + Lay::o_col + (uint32_t)(c * 32), o);
            tc::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= f;
            tc::tmem_st32(tmem + lane_addr + Lay::o_col + (uint32_t)(c * 32), o);
          }
          tc::tmem_wait_st();
        }
        float sum = 0.f;
#pragma unroll 1
        for (int c = 0; c < kAT / 32; ++c) {
          float x[32];
          tc::tmem_ld32(tmem + lane_addr + (uint32_t)(c * 32), x);
          tc::tmem_wait_ld();
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float s0 = c * 32 + i < vcols ? x[i] * sl2 : neg_inf();
            const float s1 = c * 32 + i + 1 < vcols ? x[i + 1] * sl2 : neg_inf();
            const float p0 = m_used == neg_inf() ? 0.f : ex2(s0 - m_used);
            const float p1 = m_used == neg_inf() ? 0.f : ex2(s1 - m_used);
            sum += p0 + p1;
            pk[i >> 1] = pack_bf16(p0, p1);
          }
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int c16 = c * 4 + q4;
            const uint32_t addr = tc::smem_u32(sp + (c16 >> 3) * kBlkA) + tc::sw128_off(row, c16 & 7);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[q4 * 4]),
                         "r"(pk[q4 * 4 + 1]), "r"(pk[q4 * 4 + 2]), "r"(pk[q4 * 4 + 3])
                         : "memory");
          }
        }
        l = l * alpha + sum;
        tc::fence_proxy_async();
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          tc::mbar_arrive(&sm.s_free[b]);
          tc::mbar_arrive(&sm.p_full);
        }
        continue;
      }
      float x[kAT];
#pragma unroll
      for (int c = 0; c < kAT / 32; ++c) tc::tmem_ld32(tmem + lane_addr + (uint32_t)(b * 128 + c * 32), x + c * 32);
      tc::tmem_wait_ld();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sm.s_free[b]);
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
          tc::tmem_ld32(tmem + lane_addr + Lay::o_col + (uint32_t)(c * 32), o);
          tc::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= f;
          tc::tmem_st32(tmem + lane_addr + Lay::o_col + (uint32_t)(c * 32), o);
        }
        tc::tmem_wait_st();
      }
#pragma unroll
      for (int c16 = 0; c16 < kAT / 8; ++c16) {
        const uint32_t addr = tc::smem_u32(sp + (c16 >> 3) * kBlkA) + tc::sw128_off(row, c16 & 7);
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
        tc::tmem_ld32(tmem + lane_addr + Lay::o_col + (uint32_t)(c * 32), o);
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
            po[i] = make_uint4(pack_bf16(o[8 * i] * inv, o[8 * i + 1] * inv),
                               pack_bf16(o[8 * i + 2] * inv, o[8 * i + 3] * inv),
                               pack_bf16(o[8 * i + 4] * inv, o[8 * i + 5] * inv),
                               pack_bf16(o[8 * i + 6] * inv, o[8 * i + 7] * inv));
        }
      }
    }
    if (dst >= 0 && ok) {
      if (a.mode == kSparse) {
        a.part_lse[(int64_t)h * np + dst] = lse;
        if (a.cnt) {
          // the last of the query's r slots to finish merges them (no waiting: the
          // earlier slots only publish their partials)
          const int64_t qi = dst / a.r;
          __threadfence();
          const int old = atomicAdd(&a.cnt[(int64_t)h * a.nq + qi], 1);
          if (old == a.r - 1) {
            __threadfence();
            const int64_t pb = (int64_t)h * np + qi * a.r;
            float mx = neg_inf();
            for (int s = 0; s < a.r; ++s) mx = fmaxf(mx, __ldcg(a.part_lse + pb + s));
            float w[FASTAR_MAX_R];
            float W = 0.f;
            for (int s = 0; s < a.r; ++s) {
              const float ls = __ldcg(a.part_lse + pb + s);
              w[s] = (mx == neg_inf() || ls == neg_inf()) ? 0.f : __expf(ls - mx);
              W += w[s];
            }
            const float invW = W > 0.f ? 1.0f / W : 0.f;
            __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.out) + h * a.o_hs + qi * a.o_ts;
#pragma unroll 1
            for (int c = 0; c < D / 8; ++c) {
              float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
              for (int s = 0; s < a.r; ++s) {
                if (w[s] == 0.f) continue;
                const float4* src = reinterpret_cast<const float4*>(a.part_o + (pb + s) * D + c * 8);
                const float4 u0 = __ldcg(src), u1 = __ldcg(src + 1);
                acc[0] = fmaf(w[s], u0.x, acc[0]);
                acc[1] = fmaf(w[s], u0.y, acc[1]);
                acc[2] = fmaf(w[s], u0.z, acc[2]);
                acc[3] = fmaf(w[s], u0.w, acc[3]);
                acc[4] = fmaf(w[s], u1.x, acc[4]);
                acc[5] = fmaf(w[s], u1.y, acc[5]);
                acc[6] = fmaf(w[s], u1.z, acc[6]);
                acc[7] = fmaf(w[s], u1.w, acc[7]);
              }
              reinterpret_cast<uint4*>(orow)[c] =
                  make_uint4(pack_bf16(acc[0] * invW, acc[1] * invW), pack_bf16(acc[2] * invW, acc[3] * invW),
                             pack_bf16(acc[4] * invW, acc[5] * invW), pack_bf16(acc[6] * invW, acc[7] * invW));
            }
            if (a.lse) a.lse[(int64_t)h * a.nq + qi] = W > 0.f ? mx + __logf(W) : neg_inf();
            a.cnt[(int64_t)h * a.nq + qi] = 0;   // ready for the next call
          }
        }
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
    tc::tmem_dealloc(tmem, Lay::tmem_cols);
  }
  if (threadIdx.x == 0 && sm.abort) flag_status(a.status, FASTAR_DEV_TIMEOUT);
}

template <int D, int KV>
bool attn_tc_impl(const AttnArgs& a, cudaStream_t s) {
  dim3 grid;
  if (a.mode == kDense) {
    grid = dim3((unsigned)((a.nq + kAT - 1) / kAT), a.H, 1);
  } else if (a.mode == kCross) {
    grid = dim3((unsigned)((a.tpf + kAT - 1) / kAT), a.H, a.F);
  } else {
    grid = dim3((unsigned)((a.nq * a.r + kAT - 1) / kAT + a.B), a.H, 1);
  }
  constexpr size_t smem = AttnLayout<D, KV>::bytes;
  static const cudaError_t attr =
      cudaFuncSetAttribute(attn_tc_kernel<D, KV>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (attr != cudaSuccess) return false;
  attn_tc_kernel<D, KV><<<grid, kThreadsA, smem, s>>>(a);
  count_launches(1);
  return true;
}

}  // namespace

bool launch_attn_tc(int d, const AttnArgs& a, cudaStream_t s) {
  // long key lists stream through a 2-deep ring; the short per-bucket / per-frame lists
  // use the compact variant so that two CTAs share an SM
  const bool streaming = a.mode == kDense;
  if (d == 128) return streaming ? attn_tc_impl<128, 2>(a, s) : attn_tc_impl<128, 1>(a, s);
  return streaming ? attn_tc_impl<64, 2>(a, s) : attn_tc_impl<64, 1>(a, s);
}

}  // namespace fastar
