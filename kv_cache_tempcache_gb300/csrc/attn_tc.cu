// Softmax attention over gathered key sets on the 5th-generation tensor cores (bf16).
//
// Serves the three attention rows of the step with one engine:
//   sparse — AnnSA (FAST-AR technical summary §2.C, blog §3): the (query, slot) pairs
//            of one bucket against that bucket's cache keys; the r slots of a query
//            use disjoint key sets (every key has one bucket), so their partial
//            (o, lse) merge exactly;
//   cross  — AnnCA (technical summary §2.B, blog §2): one latent frame's queries
//            against its kept prompt tokens;
//   dense  — the dense baseline (technical summary, Key Results): every key.
//
// A work item is one tile of up to 128 query rows with its key list.  The kernel is
// persistent (one CTA per SM, items taken round-robin) and warp-specialised so that
// the gathers of the next item overlap the arithmetic of this one:
//   warps 0-3   gather rows with 16-byte cp.async into 128-byte-swizzled tiles: the
//               item's Q tile (two Q stages) and its 128-key K/V tiles (two K/V
//               stages), keeping up to three copy groups in flight per thread;
//   warp 4      owns TMEM (S double buffer + one O accumulator per Q stage) and
//               issues tcgen05.mma from one thread: S_j = Q K_j^T, and O += P_j V_j
//               once the softmax has written P_j (QK_{j+1} is issued before PV_j);
//   warps 5-8   softmax, one query row per thread: S row from TMEM, running max in
//               log2 units with lazy rescaling (O in TMEM is rescaled only when the
//               max grows by more than 2^8), P as bf16 into shared memory (over the
//               consumed K tile when d = 128);
//   warps 9-12  epilogue: O / l from TMEM to the output (or, for AnnSA, the slot
//               partial and the merge) while the next item is being computed.
// AnnSA's items (head, bucket, 128-pair tile) are planned by every CTA in its prologue
// (an exclusive prefix of the tile counts in shared memory, searched per item) when
// H·B < 2048, else listed by a one-CTA planning kernel;
// each item writes its slot partials (o in bf16, lse in fp32) at the (query, slot) pair
// rows — staged through shared memory so every store is a full row segment — and a merge
// kernel combines the r adjacent slot rows of every query afterwards.
// Every wait is bounded; a timeout sets FASTAR_DEV_TIMEOUT and unwinds.
#include <climits>
#include <cstring>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"
#include "tmap.h"

namespace fastar {
namespace {

constexpr int kAT = 128;          // query rows per item
constexpr int kKT = 64;           // keys per K/V tile
constexpr int kKS = 4;            // K/V stages (and S buffers)
constexpr int kThreadsA = 416;    // 13 warps
constexpr int kBlkA = 128 * 128;  // one 128-row x 64-element bf16 block (128-B swizzle)
constexpr int kBlkK = kKT * 128;  // one kKT-row x 64-element bf16 block
constexpr int kMmaWarpA = 4;
constexpr int kSoftWarp0 = 5;
constexpr int kEpiWarp0 = 9;
constexpr int kPlanThreads = 1024;
constexpr int kPrefixMax = 2048;  // (head, bucket) entries + 1 planned inside the kernel
constexpr int kMatchAux = 80 * 4; // bytes of 1/|k| (or of indices) staged per key tile in match mode

// One AnnSA work item, as listed by the planning kernel.
struct SparseItem {
  int h, q0, q1, kbase, nkeys, pad0, pad1, pad2;
};

struct ItemInfo {
  int h, T, f, nrows;
  int64_t nkeys, kbase, q0;
};

struct AttnCtl {
  int64_t qsrc[2][kAT];   // loader-private: source offset of each query row, per Q stage
  union {
    int64_t ksrc[kKS][kKT]; // row gathers, loader-private: source offset of each key row, per stage
    float kbias[kKS][kKT];  // tensor-engine K/V with group counts: log2 g of each key, per stage
  };
  int qdst[2][kAT];       // output row of each query row (-1: none), per Q stage
  float mrow[2][kAT], lrow[2][kAT];   // softmax max (log2 units) and sum, per Q stage
  int edst[kAT];          // epilogue-private: output row of each row of the item being stored
  ItemInfo info[2];
  uint64_t q_full[2], q_empty[2], dst_free[2];
  uint64_t kv_full[kKS], kv_empty[kKS];
  uint64_t s_full[kKS], s_free[kKS], p_full[kKS];
  uint64_t pv_done, fin;
  uint64_t ml_full[2], o_full[2], o_empty[2];
  uint32_t tmem_base;
  int abort;
  int n_items;
};

// Shared-memory layout (bytes from the 1024-aligned base).
template <int D>
struct AttnLayout {
  static constexpr int KH = D / 64;
  static constexpr size_t qstage = (size_t)KH * kBlkA;   // one 128-row Q tile
  static constexpr size_t kstage = (size_t)KH * kBlkK;   // one kKT-row K (or V) tile
  static constexpr size_t pbytes = (size_t)kAT * kKT * 2; // P: 128 x kKT bf16, one swizzled block
  static constexpr bool kPAliasK = kstage >= pbytes;     // P over the consumed K tile
  static constexpr size_t q = 0;
  static constexpr size_t k = q + 2 * qstage;
  static constexpr size_t v = k + kKS * kstage;
  static constexpr size_t p = kPAliasK ? k : v + kKS * kstage;
  static constexpr size_t pstride = kPAliasK ? kstage : pbytes;
  // 128 rows x 32 fp32: the epilogue's transpose buffer for coalesced partial stores
  static constexpr size_t ostage = kPAliasK ? v + kKS * kstage : p + kKS * pstride;
  static constexpr size_t ctl = ostage + 128 * 32 * sizeof(float);
  static constexpr size_t prefix = ctl + ((sizeof(AttnCtl) + 15) & ~(size_t)15);   // kPrefixMax ints
  static constexpr size_t bytes = prefix + kPrefixMax * sizeof(int) + 1024;
  static constexpr uint32_t s_col = 0;      // S buffers: kKS x kKT columns from 0
  static constexpr uint32_t o_col = 256;    // O accumulators: [256 + 128 * stage, ...)
  static_assert(kKS * kKT <= 256, "S buffers overlap the O accumulators");
  static_assert(pbytes == kBlkA * (kKT / 64), "P is one 128-row block per 64 keys");
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

// The logit shift of a key that stands for a group of g keys, in log2 units (the merge
// variant, Lemma 5.1): log2 g; an empty group (g = 0) gets -inf, a negative count is a
// bad input (flagged) and counts as empty.
__device__ __forceinline__ float group_log2(int32_t g, int32_t* status) {
  if (g < 0) flag_status(status, FASTAR_DEV_BAD_INDEX);
  return g > 0 ? log2f((float)g) : neg_inf();
}

// 16 consecutive 32-bit TMEM columns of this thread's lane (P as packed bf16 pairs).
__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t* v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
               : "memory");
}

// D[tmem] (+)= A B^T with A read from TMEM (M = 128 rows on the lanes, each 32-bit column a
// bf16 pair of consecutive K elements: a K = 16 step reads 8 columns) and B from shared
// memory.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(acc)
      : "memory");
}

// Three-input maximum (PTX max.f32 with three sources).
__device__ __forceinline__ float max3(float a, float b, float c) {
  float y;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
  return y;
}

// Maximum of 32 scores; with kFull = false the columns from `valid` on count as -inf.
template <bool kFull>
__device__ __forceinline__ float max32(const float* v, int valid) {
  float t[11];
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    const float a = kFull || 3 * i < valid ? v[3 * i] : neg_inf();
    const float b = kFull || 3 * i + 1 < valid ? v[3 * i + 1] : neg_inf();
    const float c = kFull || 3 * i + 2 < valid ? v[3 * i + 2] : neg_inf();
    t[i] = max3(a, b, c);
  }
  t[10] = fmaxf(kFull || 30 < valid ? v[30] : neg_inf(), kFull || 31 < valid ? v[31] : neg_inf());
  return max3(max3(t[0], t[1], t[2]), max3(t[3], t[4], t[5]), max3(max3(t[6], t[7], t[8]), t[9], t[10]));
}

// Softmax pass 1 over one kKT-column S row in TMEM, 64 columns per TMEM round trip: the
// raw row maximum (scores not yet scaled); with kBias, the maximum of the shifted logits
// s * sl2 + bias[c] (log2 units).
template <bool kFull, bool kBias = false>
__device__ __forceinline__ float row_max(uint32_t s_addr, int vcols, float sl2 = 0.f, const float* bias = nullptr) {
  float m = neg_inf();
#pragma unroll 1
  for (int hh = 0; hh < kKT / 64; ++hh) {
    float x[64];
    tc::tmem_ld32(s_addr + (uint32_t)(hh * 64), x);
    tc::tmem_ld32(s_addr + (uint32_t)(hh * 64 + 32), x + 32);
    tc::tmem_wait_ld();
    tc::tmem_pin32(x);
    tc::tmem_pin32(x + 32);
    if (kBias) {
#pragma unroll
      for (int c = 0; c < 64; c += 4) {
        const float4 b = *reinterpret_cast<const float4*>(bias + hh * 64 + c);
        x[c] = fmaf(x[c], sl2, b.x);
        x[c + 1] = fmaf(x[c + 1], sl2, b.y);
        x[c + 2] = fmaf(x[c + 2], sl2, b.z);
        x[c + 3] = fmaf(x[c + 3], sl2, b.w);
      }
    }
    m = max3(m, max32<kFull>(x, vcols - hh * 64), max32<kFull>(x + 32, vcols - hh * 64 - 32));
  }
  return m;
}

// Softmax pass 2: P = 2^(s * sl2 + bias - m) as bf16 pairs into this thread's TMEM lane,
// over the S columns already read (P's kKT / 2 columns start at s_addr: chunk c of 32
// scores becomes columns 16c .. 16c + 15, after S columns 0 .. 32c + 31 have been loaded);
// returns the row sum of P.  The P.V product then reads P from TMEM as its A operand.
template <bool kFull, bool kBias = false>
__device__ __forceinline__ float row_exp(uint32_t s_addr, int vcols, float sl2, float m, const float* bias = nullptr) {
  const float nm = m == neg_inf() ? 0.f : -m;
  float xa[32], xb[32];
  float s0 = 0.f, s1 = 0.f;
  tc::tmem_ld32(s_addr, xa);
  tc::tmem_wait_ld();
  tc::tmem_pin32(xa);
#pragma unroll
  for (int c = 0; c < kKT / 32; ++c) {
    float* cur = (c & 1) ? xb : xa;
    float* nxt = (c & 1) ? xa : xb;
    if (c + 1 < kKT / 32) tc::tmem_ld32(s_addr + (uint32_t)((c + 1) * 32), nxt);
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      float b0 = nm, b1 = nm;
      if (kBias) {
        const float2 b = *reinterpret_cast<const float2*>(bias + c * 32 + i);
        b0 = b.x + nm;
        b1 = b.y + nm;
      }
      float a0 = fmaf(cur[i], sl2, b0), a1 = fmaf(cur[i + 1], sl2, b1);
      if (!kFull) {
        a0 = c * 32 + i < vcols ? a0 : neg_inf();
        a1 = c * 32 + i + 1 < vcols ? a1 : neg_inf();
      }
      const float p0 = ex2(a0), p1 = ex2(a1);
      s0 += p0;
      s1 += p1;
      pk[i >> 1] = pack_bf16(p0, p1);
    }
    tmem_st16u(s_addr + (uint32_t)(c * 16), pk);
    if (c + 1 < kKT / 32) {
      tc::tmem_wait_ld();
      tc::tmem_pin32(nxt);
    }
  }
  return s0 + s1;
}

__device__ __forceinline__ int64_t items_of(const AttnArgs& a) {
  if (a.mode == kCross) return (int64_t)a.H * a.F * ((a.tpf + kAT - 1) / kAT);
  if (a.mode == kDense) return (int64_t)a.H * ((a.nq + kAT - 1) / kAT);
  return 0;   // sparse: from the planning kernel
}

// Items over (query, slot) pairs in bucket order: AnnSA and the ANN-restricted match.
__device__ __forceinline__ bool pair_items(const AttnArgs& a) { return a.mode == kSparse || a.mode == kMatchAnn; }

// AnnSA entry k = (head, bucket): its query-pair range [q0, q1) in the head's sorted
// order, its key range (kbase, nk) and the number of 128-pair tiles; malformed offsets
// give no tiles (or no keys) and a status bit.
__device__ __forceinline__ int sparse_entry(const AttnArgs& a, int k, int& q0, int& q1, int& kb, int& nk) {
  const int64_t np = a.nq * a.r;
  const int h = k / a.B, b = k % a.B;
  const int32_t* qo = a.qoff + (int64_t)h * (a.B + 1);
  const int32_t* ko = a.koff + (int64_t)h * (a.B + 1);
  q0 = qo[b];
  q1 = qo[b + 1];
  kb = ko[b];
  nk = ko[b + 1] - kb;
  if (q0 < 0 || q1 < q0 || q1 > np) {
    flag_status(a.status, FASTAR_DEV_BAD_INDEX);
    return 0;
  }
  if (kb < 0 || nk < 0 || (int64_t)kb + nk > a.M) {
    flag_status(a.status, FASTAR_DEV_BAD_INDEX);
    nk = 0;
  }
  return (q1 - q0 + kAT - 1) / kAT;
}

// Work item u: its head, key count and key base, and its query range [q0, q1) (sparse:
// positions in the head's qperm row; otherwise token rows).
__device__ __forceinline__ void decode_item(const AttnArgs& a, int64_t u, ItemInfo& it, int64_t& q0,
                                            int64_t& q1, const int* pre) {
  it.f = 0;
  it.kbase = 0;
  if (pair_items(a) && !a.items) {
    // planned in the kernel: pre[k] = tiles of the entries before k; find the entry
    int lo = 0, hi = a.H * a.B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] <= u) lo = mid; else hi = mid - 1;
    }
    int e0, e1, kb, nk;
    sparse_entry(a, lo, e0, e1, kb, nk);
    it.h = lo / a.B;
    q0 = e0 + (u - pre[lo]) * kAT;
    q1 = q0 + kAT < e1 ? q0 + kAT : e1;
    it.kbase = kb;
    it.nkeys = nk;
    it.q0 = q0;
    it.nrows = (int)(q1 - q0);
    it.T = (int)((it.nkeys + kKT - 1) / kKT);
    return;
  }
  if (pair_items(a)) {
    const int4* p = reinterpret_cast<const int4*>(static_cast<const SparseItem*>(a.items) + u);
    const int4 x = p[0], y = p[1];
    it.h = x.x;
    q0 = x.y;
    q1 = x.z;
    it.kbase = x.w;
    it.nkeys = y.x;
    it.q0 = q0;
    it.nrows = (int)(q1 - q0);
    it.T = (int)((it.nkeys + kKT - 1) / kKT);
    return;
  } else if (a.mode == kCross) {
    const int64_t nqt = (a.tpf + kAT - 1) / kAT;
    const int64_t per = (int64_t)a.F * nqt;
    it.h = (int)(u / per);
    const int64_t rem = u % per;
    it.f = (int)(rem / nqt);
    const int64_t t0 = (rem % nqt) * kAT;
    q0 = (int64_t)it.f * a.tpf + t0;
    q1 = (int64_t)it.f * a.tpf + (t0 + kAT < a.tpf ? t0 + kAT : a.tpf);
    int64_t nk = a.kcnt[(int64_t)it.h * a.F + it.f];
    if (nk < 0 || nk > a.P) {
      flag_status(a.status, FASTAR_DEV_BAD_INDEX);
      nk = nk < 0 ? 0 : a.P;
    }
    it.nkeys = nk;
  } else {
    const int64_t nqt = (a.nq + kAT - 1) / kAT;
    it.h = (int)(u / nqt);
    q0 = (u % nqt) * kAT;
    q1 = q0 + kAT < a.nq ? q0 + kAT : a.nq;
    it.nkeys = a.nk;
  }
  it.q0 = q0;
  it.nrows = (int)(q1 - q0);
  it.T = (int)((it.nkeys + kKT - 1) / kKT);
}

// Element offset of key u of the item's key list (-1 if out of range).
__device__ __forceinline__ int64_t key_offset(const AttnArgs& a, const ItemInfo& it, int64_t u, int D) {
  if (u >= it.nkeys) return -1;
  if (pair_items(a)) {
    const int s = a.kperm[(int64_t)it.h * a.M + it.kbase + u];
    if (s >= 0 && s < a.M) return ((int64_t)it.h * a.M + s) * D;
    flag_status(a.status, FASTAR_DEV_BAD_INDEX);
    return -1;
  }
  if (a.mode == kCross) {
    const int p = a.kidx[((int64_t)it.h * a.F + it.f) * a.P + u];
    if (p >= 0 && p < a.P) return ((int64_t)it.h * a.P + p) * D;
    flag_status(a.status, FASTAR_DEV_BAD_INDEX);
    return -1;
  }
  return it.h * a.kv_hs + u * a.kv_ts;
}

// The logit shift (log2 units) of key u of the item's key list when keys stand for
// groups (the merge variant): AnnSA reads the bucket-ordered copy the sort kernel wrote,
// the dense path the caller's counts; 0 past the list (those columns are masked).
__device__ __forceinline__ float key_bias(const AttnArgs& a, const ItemInfo& it, int64_t u) {
  if (u >= it.nkeys) return 0.f;
  if (a.mode == kSparse) return a.lg_sorted[(int64_t)it.h * a.M + it.kbase + u];
  return group_log2(a.gcount[(int64_t)it.h * a.gc_hs + u], a.status);
}

// The third tensor-map coordinate of the item's K/V tiles: the head, or for AnnCA the
// (head, frame) plane of the gathered kept-prompt rows.
__device__ __forceinline__ int kv_plane(const AttnArgs& a, const ItemInfo& it) {
  return a.mode == kCross ? it.h * a.F + it.f : it.h;
}

// Query row `pos` of item `it` (valid below q1): its source offset and output row
// (sparse: the (query, slot) pair index; otherwise the token row), or -1 for none.
__device__ __forceinline__ void query_row(const AttnArgs& a, const ItemInfo& it, int64_t pos, int64_t q1,
                                          int64_t np, int64_t& src, int& dst) {
  src = -1;
  dst = -1;
  if (pos >= q1) return;
  if (pair_items(a)) {
    const int e = a.qperm[(int64_t)it.h * np + pos];
    if (e >= 0 && e < np) {
      src = it.h * a.q.hs + (int64_t)(e / a.r) * a.q.ts;
      dst = e;
    } else {
      flag_status(a.status, FASTAR_DEV_BAD_INDEX);
    }
  } else {
    src = it.h * a.q.hs + pos * a.q.ts;
    dst = (int)pos;
  }
}

// Copy groups a loader thread has committed but not yet signalled (at most four are
// kept in flight; before any blocking wait all of them are signalled, so a consumer
// is never left waiting on a copy whose producer is itself waiting).
struct Pending {
  uint64_t* b0 = nullptr;
  uint64_t* b1 = nullptr;
  uint64_t* b2 = nullptr;
  uint64_t* b3 = nullptr;
  int n = 0;
  __device__ __forceinline__ void flush() {
    if (n == 0) return;
    tc::cp_async_wait<0>();
    tc::fence_proxy_async();
    tc::mbar_arrive(b0);
    if (n > 1) tc::mbar_arrive(b1);
    if (n > 2) tc::mbar_arrive(b2);
    if (n > 3) tc::mbar_arrive(b3);
    n = 0;
  }
  __device__ __forceinline__ void push(uint64_t* b) {
    if (n == 4) {
      tc::cp_async_wait<4>();   // the oldest of the five groups has landed
      tc::fence_proxy_async();
      tc::mbar_arrive(b0);
      b0 = b1;
      b1 = b2;
      b2 = b3;
      b3 = b;
      return;
    }
    if (n == 0) b0 = b;
    else if (n == 1) b1 = b;
    else if (n == 2) b2 = b;
    else b3 = b;
    ++n;
  }
  __device__ __forceinline__ bool acquire(uint64_t* bar, uint32_t parity, volatile int* abort) {
    if (tc::mbar_test(bar, parity)) return true;
    flush();
    return tc::mbar_wait(bar, parity, abort);
  }
};

// kMode is the AttnMode of the launch, fixed per instance: every mode test below folds at
// compile time, so an instance carries only its own mode's code (one instance serving all
// modes spent a large share of its cycles waiting on instruction fetches).
template <int D, bool kGrouped, int kMode>
__global__ void __launch_bounds__(kThreadsA, 1)
    attn_tc_kernel(const AttnArgs args, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_q) {
  AttnArgs a = args;
  a.mode = kMode;
  using Lay = AttnLayout<D>;
  constexpr int CPR = D / 8;   // 16-byte chunks per row
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sq = base + Lay::q;   // [2][KH][kBlkA]
  uint8_t* sk = base + Lay::k;   // [kKS][KH][kBlkK]
  uint8_t* sv = base + Lay::v;   // [kKS][KH][kBlkK]
  uint8_t* sp = base + Lay::p;   // [2] x pstride
  float* so = reinterpret_cast<float*>(base + Lay::ostage);   // [128][32], 16-byte chunks swizzled
  AttnCtl& sm = *reinterpret_cast<AttnCtl*>(base + Lay::ctl);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const __nv_bfloat16* Q = static_cast<const __nv_bfloat16*>(a.q.p);
  const __nv_bfloat16* K = static_cast<const __nv_bfloat16*>(a.k);
  const __nv_bfloat16* V = static_cast<const __nv_bfloat16*>(a.v);
  const int64_t np = a.nq * a.r;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&sm.q_full[s], a.q_tma ? 1 : 128);
      tc::mbar_init(&sm.q_empty[s], 1);
      tc::mbar_init(&sm.dst_free[s], 4);
      tc::mbar_init(&sm.ml_full[s], 4);
      tc::mbar_init(&sm.o_full[s], 1);
      tc::mbar_init(&sm.o_empty[s], 4);
    }
    for (int s = 0; s < kKS; ++s) {
      tc::mbar_init(&sm.kv_full[s], a.kv_tma ? 1 : 128);
      // match mode: the softmax warps release a stage (they read its 1/|k| and indices)
      tc::mbar_init(&sm.kv_empty[s], a.mode == kMatchAnn ? 4 : 1);
      tc::mbar_init(&sm.s_full[s], 1);
      tc::mbar_init(&sm.s_free[s], 4);
      tc::mbar_init(&sm.p_full[s], 4);
    }
    tc::mbar_init(&sm.pv_done, 1);
    tc::mbar_init(&sm.fin, 1);
    sm.abort = 0;
    tc::mbar_fence_init();
  }
  // the slot merge after it (AnnSA) may start launching: its CTAs are small and wait for
  // this grid to finish
  pdl_trigger();
  // the inputs written by the kernel before it in the stream (the sorted compaction's
  // bucket-ordered rows and offsets, the AnnCA selection's kept rows): everything above
  // touched shared memory only
  pdl_wait();
  int* pre = reinterpret_cast<int*>(base + Lay::prefix);
  if (pair_items(a) && !a.items) {
    // plan the AnnSA items here: exclusive prefix over the (head, bucket) entries of
    // their tile counts (every thread takes a contiguous run of entries)
    const int ne = a.H * a.B;
    const int per = (ne + kThreadsA - 1) / kThreadsA;
    const int k0 = threadIdx.x * per, k1 = k0 + per < ne ? k0 + per : ne;
    int mine = 0;
    for (int k = k0; k < k1; ++k) {
      int e0, e1, kb, nk;
      mine += sparse_entry(a, k, e0, e1, kb, nk);
    }
    int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    __shared__ int wtot[kThreadsA / 32];
    if (lane == 31) wtot[warp] = incl;
    __syncthreads();
    int run = 0;
    for (int w = 0; w < warp; ++w) run += wtot[w];
    int at = run + incl - mine;
    for (int k = k0; k < k1; ++k) {
      pre[k] = at;
      int e0, e1, kb, nk;
      at += sparse_entry(a, k, e0, e1, kb, nk);
    }
    if (threadIdx.x == kThreadsA - 1) sm.n_items = run + incl;
  } else if (threadIdx.x == 0) {
    const int64_t n = pair_items(a) ? (int64_t)*a.n_items : items_of(a);
    sm.n_items = (int)(n < INT_MAX ? n : INT_MAX);
  }
  __syncthreads();
  const int n_items = sm.n_items;
  if ((int)blockIdx.x >= n_items) return;   // no work for this CTA (uniform; nothing allocated)
  if (warp == kMmaWarpA) {
    tc::tmem_alloc(&sm.tmem_base, 512);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort = &sm.abort;
  const bool amatch = a.mode == kMatchAnn;   // arg-max of cosines instead of softmax.V
  constexpr bool grouped = kGrouped;  // keys stand for groups: logit shift log2 g per key

  if (warp < 4 && a.q_tma) {
    // ---------------- tensor-engine loads (thread 0 issues every copy) ----------------
    // Q, K and V tiles are all contiguous rows: thread 0 issues them; the other loader
    // threads only record their row's output destination.  Nobody holds an unsignalled
    // copy, so the only barrier (per item) cannot wait on a stuck copy.
    const int t = threadIdx.x;
    int g = 0, n = 0;
    bool tiles_ok = true;
    for (int u = blockIdx.x; u < n_items; u += gridDim.x, ++n) {
      const int qs = n & 1;
      const uint32_t qph = (n >> 1) & 1;
      bool got = true;
      if (n >= 2) got = tc::mbar_wait(&sm.q_empty[qs], qph ^ 1, abort) && tc::mbar_wait(&sm.dst_free[qs], qph ^ 1, abort);
      ItemInfo it;
      int64_t q0, q1, src;
      int dst;
      decode_item(a, u, it, q0, q1, pre);
      query_row(a, it, q0 + t, q1, np, src, dst);
      if (got) {
        sm.qdst[qs][t] = dst;
        if (t == 0) sm.info[qs] = it;
      }
      if (!tc::named_bar_and(1, 128, got && tiles_ok)) break;
      if (t < 32) {
        if (t == 0) {
          tc::mbar_arrive_tx(&sm.q_full[qs], (uint32_t)Lay::qstage);
          for (int kh = 0; kh < D / 64; ++kh) {
            uint8_t* dq = sq + (size_t)qs * Lay::qstage + kh * kBlkA;
            if (!a.q_token_major)
              tc::tma_load_3d(dq, &tm_q, kh * 64, (int)q0, it.h, &sm.q_full[qs]);
            else
              tc::tma_load_3d(dq, &tm_q, kh * 64, it.h, (int)q0, &sm.q_full[qs]);
          }
        }
        // warp 0: lane 0 issues the K/V copies; with group counts every lane also stages
        // two keys' logit shifts, written before lane 0's arrival publishes the stage
        for (int j = 0; j < it.T; ++j) {
          const int st = (g + j) % kKS;
          const uint32_t ph = ((g + j) / kKS) & 1;
          float b0 = 0.f, b1 = 0.f;
          if (grouped) {
            b0 = key_bias(a, it, (int64_t)j * kKT + t);
            b1 = key_bias(a, it, (int64_t)j * kKT + t + 32);
          }
          bool fr = true;
          if (t == 0 || grouped) fr = tc::mbar_wait(&sm.kv_empty[st], ph ^ 1, abort);
          if (!__all_sync(0xffffffffu, fr)) {
            tiles_ok = false;
            break;
          }
          if (grouped) {
            sm.kbias[st][t] = b0;
            sm.kbias[st][t + 32] = b1;
            __syncwarp();
          }
          if (t == 0) {
            const int y = (int)(it.kbase + (int64_t)j * kKT);
            tc::mbar_arrive_tx(&sm.kv_full[st], (uint32_t)(2 * Lay::kstage));
            for (int kh = 0; kh < D / 64; ++kh) {
              tc::tma_load_3d(sk + (size_t)st * Lay::kstage + kh * kBlkK, &tm_k, kh * 64, y, kv_plane(a, it),
                              &sm.kv_full[st]);
              tc::tma_load_3d(sv + (size_t)st * Lay::kstage + kh * kBlkK, &tm_v, kh * 64, y, kv_plane(a, it),
                              &sm.kv_full[st]);
            }
          }
        }
      }
      g += it.T;
    }
  } else if (warp < 4) {
    // ---------------- row gathers (128 threads) ----------------
    const int t = threadIdx.x;
    // Every exit decision is taken by all 128 threads together (named_bar_and): a
    // thread that left alone would strand the others in the next named barrier.
    // Index loads run one step ahead of the copies that use them: the next item's query
    // row and first key tile while this item's tiles are copied, the next key tile's
    // rows while this one waits for its stage.
    Pending pend;
    int g = 0, n = 0;
    bool ok = true;
    ItemInfo it;
    int64_t qsrc = -1, ksrc = -1;
    int qdst = -1;
    auto load_item = [&](int64_t v, ItemInfo& x, int64_t& src, int& dst, int64_t& k0) {
      int64_t p0, p1;
      decode_item(a, v, x, p0, p1, pre);
      query_row(a, x, p0 + t, p1, np, src, dst);
      k0 = !a.kv_tma && t < kKT && x.T > 0 ? key_offset(a, x, t, D) : -1;
    };
    if ((int)blockIdx.x < n_items) load_item(blockIdx.x, it, qsrc, qdst, ksrc);
    for (int u = blockIdx.x; u < n_items && ok; u += gridDim.x, ++n) {
      const int qs = n & 1;
      const uint32_t qph = (n >> 1) & 1;
      ItemInfo nit{};
      int64_t nqsrc = -1, nksrc = -1;
      int nqdst = -1;
      if (u + (int)gridDim.x < n_items) load_item(u + gridDim.x, nit, nqsrc, nqdst, nksrc);
      bool got = true;
      if (n >= 2)
        got = pend.acquire(&sm.q_empty[qs], qph ^ 1, abort) && pend.acquire(&sm.dst_free[qs], qph ^ 1, abort);
      if (got) {
        sm.qsrc[qs][t] = qsrc;
        sm.qdst[qs][t] = qdst;
        if (t == 0) sm.info[qs] = it;
      }
      if (!tc::named_bar_and(1, 128, got)) {
        ok = false;
        break;
      }
      {
        uint8_t* qst = sq + (size_t)qs * Lay::qstage;
#pragma unroll 4
        for (int gi = t; gi < kAT * CPR; gi += 128) {
          const int row = gi / CPR, c = gi % CPR;
          const int64_t s = sm.qsrc[qs][row];
          tc::cp_async16(tc::smem_u32(qst + (c >> 3) * kBlkA) + tc::sw128_off(row, c & 7),
                         s >= 0 ? Q + s + c * 8 : Q, s >= 0 ? 16u : 0u);
        }
        tc::cp_async_commit();
        pend.push(&sm.q_full[qs]);
        // K/V by TMA: nothing else of this thread's is in flight, so signal Q now (no
        // thread may hold an unsignalled copy while it waits in a named barrier below)
        if (a.kv_tma) pend.flush();
      }
      for (int j = 0; j < it.T; ++j, ++g) {
        const int st = g % kKS;
        const uint32_t ph = (g / kKS) & 1;
        if (a.kv_tma) {
          // one thread brings the K and V tiles (contiguous rows) with the tensor engine
          bool free = true;
          if (grouped) {
            // warp 0 stages the tile's logit shifts (loaded before the wait), then lane 0
            // issues the copies; nothing of this thread's is in flight (Q was signalled)
            if (t < 32) {
              const float b0 = key_bias(a, it, (int64_t)j * kKT + t);
              const float b1 = key_bias(a, it, (int64_t)j * kKT + t + 32);
              free = __all_sync(0xffffffffu, tc::mbar_wait(&sm.kv_empty[st], ph ^ 1, abort));
              if (free) {
                sm.kbias[st][t] = b0;
                sm.kbias[st][t + 32] = b1;
                __syncwarp();
                if (t == 0) {
                  const int y = (int)(it.kbase + (int64_t)j * kKT);
                  tc::mbar_arrive_tx(&sm.kv_full[st], (uint32_t)(2 * Lay::kstage));
                  for (int kh = 0; kh < D / 64; ++kh) {
                    tc::tma_load_3d(sk + (size_t)st * Lay::kstage + kh * kBlkK, &tm_k, kh * 64, y, kv_plane(a, it),
                                    &sm.kv_full[st]);
                    tc::tma_load_3d(sv + (size_t)st * Lay::kstage + kh * kBlkK, &tm_v, kh * 64, y, kv_plane(a, it),
                                    &sm.kv_full[st]);
                  }
                }
              }
            }
          } else if (t == 0) {
            free = pend.acquire(&sm.kv_empty[st], ph ^ 1, abort);
            if (free) {
              const int y = (int)(it.kbase + (int64_t)j * kKT);
              if (amatch) {
                // K, and per key 1/|k| and the cache index, into the (unused) V stage: 80
                // entries from y rounded down to 16 bytes
                const int64_t y0 = (int64_t)it.h * a.mstride + (y & ~3);
                uint8_t* vst = sv + (size_t)st * Lay::kstage;
                tc::mbar_arrive_tx(&sm.kv_full[st], (uint32_t)(Lay::kstage + 2 * kMatchAux));
                for (int kh = 0; kh < D / 64; ++kh)
                  tc::tma_load_3d(sk + (size_t)st * Lay::kstage + kh * kBlkK, &tm_k, kh * 64, y, it.h, &sm.kv_full[st]);
                tc::bulk_load(vst, a.inv_sorted + y0, kMatchAux, &sm.kv_full[st]);
                tc::bulk_load(vst + kMatchAux, a.j_sorted + y0, kMatchAux, &sm.kv_full[st]);
              } else {
                tc::mbar_arrive_tx(&sm.kv_full[st], (uint32_t)(2 * Lay::kstage));
                for (int kh = 0; kh < D / 64; ++kh) {
                  tc::tma_load_3d(sk + (size_t)st * Lay::kstage + kh * kBlkK, &tm_k, kh * 64, y, kv_plane(a, it),
                                  &sm.kv_full[st]);
                  tc::tma_load_3d(sv + (size_t)st * Lay::kstage + kh * kBlkK, &tm_v, kh * 64, y, kv_plane(a, it),
                                  &sm.kv_full[st]);
                }
              }
            }
          }
          if (!tc::named_bar_and(1, 128, free)) {
            ok = false;
            break;
          }
          continue;
        }
        const int64_t cur = ksrc;
        ksrc = t < kKT && j + 1 < it.T ? key_offset(a, it, (int64_t)(j + 1) * kKT + t, D) : -1;
        const bool free = pend.acquire(&sm.kv_empty[st], ph ^ 1, abort);
        if (free && t < kKT) sm.ksrc[st][t] = cur;
        if (!tc::named_bar_and(1, 128, free)) {
          ok = false;
          break;
        }
        uint8_t* kst = sk + (size_t)st * Lay::kstage;
        uint8_t* vst = sv + (size_t)st * Lay::kstage;
#pragma unroll 4
        for (int gi = t; gi < kKT * CPR; gi += 128) {
          const int row = gi / CPR, c = gi % CPR;
          const int64_t s = sm.ksrc[st][row];
          const uint32_t o = (uint32_t)((c >> 3) * kBlkK) + tc::sw128_off(row, c & 7);
          tc::cp_async16(tc::smem_u32(kst) + o, s >= 0 ? K + s + c * 8 : K, s >= 0 ? 16u : 0u);
          tc::cp_async16(tc::smem_u32(vst) + o, s >= 0 ? V + s + c * 8 : V, s >= 0 ? 16u : 0u);
        }
        tc::cp_async_commit();
        pend.push(&sm.kv_full[st]);
      }
      it = nit;
      qsrc = nqsrc;
      qdst = nqdst;
      ksrc = nksrc;
    }
    pend.flush();
  } else if (warp == kMmaWarpA) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc_qk = tc::idesc_bf16_f32(128, kKT);
      constexpr uint32_t idesc_pv = tc::idesc_bf16_f32_bmn(128, D);
      const uint64_t q_desc = tc::sw128_desc(tc::smem_u32(sq));
      const uint64_t k_desc = tc::sw128_desc(tc::smem_u32(sk));
      const uint64_t p_desc = tc::sw128_desc(tc::smem_u32(sp));
      const uint64_t v_desc = tc::sw128_mn_desc(tc::smem_u32(sv), kBlkK);
      // O_qs += P_gt V_gt for global tile gt; `first` starts the accumulator
      auto issue_pv = [&](int gt, int qs, bool first) -> bool {
        const int st = gt % kKS;
        if (!tc::mbar_wait(&sm.p_full[st], (gt / kKS) & 1, abort)) return false;
        tc::tc_fence_after();
        // A = P from TMEM (the stage's S columns, 8 per 16 keys), B = V from shared memory
#pragma unroll
        for (int ks = 0; ks < kKT / 16; ++ks) {
          const uint32_t boff = (uint32_t)(st * Lay::kstage + ks * 2048);
          mma_bf16_ts(tmem + Lay::o_col + (uint32_t)(qs * 128), tmem + Lay::s_col + (uint32_t)(st * kKT + ks * 8),
                      v_desc + (boff >> 4), idesc_pv, (!first || ks > 0) ? 1u : 0u);
        }
        tc::mma_commit(&sm.kv_empty[st]);
        tc::mma_commit(&sm.pv_done);
        return true;
      };
      int g = 0, n = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < n_items && ok; u += gridDim.x, ++n) {
        const int qs = n & 1;
        const uint32_t qph = (n >> 1) & 1;
        if (!tc::mbar_wait(&sm.q_full[qs], qph, abort)) break;
        const int T = sm.info[qs].T;
        if (!tc::mbar_wait(&sm.o_empty[qs], qph ^ 1, abort)) break;
        tc::tc_fence_after();
        for (int j = 0; j < T; ++j, ++g) {
          const int st = g % kKS;
          const uint32_t ph = (g / kKS) & 1;
          if (!tc::mbar_wait(&sm.kv_full[st], ph, abort) || !tc::mbar_wait(&sm.s_free[st], ph ^ 1, abort)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t qoff = (uint32_t)(qs * Lay::qstage + (k >> 2) * kBlkA + (k & 3) * 32);
            const uint32_t koff = (uint32_t)(st * Lay::kstage + (k >> 2) * kBlkK + (k & 3) * 32);
            tc::mma_bf16(tmem + Lay::s_col + (uint32_t)(st * kKT), q_desc + (qoff >> 4), k_desc + (koff >> 4),
                         idesc_qk, k > 0 ? 1u : 0u);
          }
          tc::mma_commit(&sm.s_full[st]);
          // the previous tile's P.V goes after this tile's Q.K^T (overlaps the softmax)
          if (j > 0 && !amatch && !issue_pv(g - 1, qs, j == 1)) {
            ok = false;
            break;
          }
        }
        if (!ok) break;
        if (T > 0 && !amatch && !issue_pv(g - 1, qs, T == 1)) break;
        tc::mma_commit(&sm.q_empty[qs]);
        tc::mma_commit(&sm.o_full[qs]);
      }
      // let every issued MMA finish before TMEM is released
      tc::mma_commit(&sm.fin);
      volatile int never = 0;
      tc::mbar_wait(&sm.fin, 0, &never, 400000000LL);
    }
  } else if (warp >= kSoftWarp0 && warp < kEpiWarp0) {
    // ---------------- softmax ----------------
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
    const float sl2 = a.scale * 1.4426950408889634f;   // scores in log2 units
    int g = 0, n = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < n_items && ok; u += gridDim.x, ++n) {
      const int qs = n & 1;
      const uint32_t qph = (n >> 1) & 1;
      if (!wait_all(&sm.q_full[qs], qph, abort)) break;
      const int T = sm.info[qs].T;
      const int64_t nkeys = sm.info[qs].nkeys;
      const uint32_t o_addr = tmem + lane_addr + Lay::o_col + (uint32_t)(qs * 128);
      float m_used = neg_inf(), l = 0.f;
      float best = neg_inf();   // match mode: best q.k/|k| of the row and its cache index
      int bidx = -1;
      const int64_t kbase = sm.info[qs].kbase;
      for (int j = 0; j < T; ++j, ++g) {
        const int st = g % kKS;
        if (!wait_all(&sm.s_full[st], (g / kKS) & 1, abort)) {
          ok = false;
          break;
        }
        tc::tc_fence_after();
        if (amatch) {
          // the staged 1/|k| and indices landed with the K tile (kv_full, already complete)
          if (!wait_all(&sm.kv_full[st], (g / kKS) & 1, abort)) {
            ok = false;
            break;
          }
          const int64_t left = nkeys - (int64_t)j * kKT;
          const int vcols = left < kKT ? (int)left : kKT;
          const int off = (int)((kbase + (int64_t)j * kKT) & 3);
          const uint8_t* vst = sv + (size_t)st * Lay::kstage;
          const float* iv = reinterpret_cast<const float*>(vst) + off;
          const int32_t* jv = reinterpret_cast<const int32_t*>(vst + kMatchAux) + off;
          const uint32_t s_addr = tmem + lane_addr + Lay::s_col + (uint32_t)(st * kKT);
          float x[64];
          tc::tmem_ld32(s_addr, x);
          tc::tmem_ld32(s_addr + 32, x + 32);
          tc::tmem_wait_ld();
          tc::tmem_pin32(x);
          tc::tmem_pin32(x + 32);
          // ascending keys: a strict improvement keeps the lowest cache index on ties
          // (branch-free: masked columns score -inf, the choice is a select)
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const float v = c < vcols ? x[c] * iv[c] : neg_inf();
            const int jc = jv[c];
            const bool gt = v > best;
            best = gt ? v : best;
            bidx = gt ? jc : bidx;
          }
          tc::tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            tc::mbar_arrive(&sm.s_free[st]);
            tc::mbar_arrive(&sm.kv_empty[st]);
          }
          continue;
        }
        const int64_t left = nkeys - (int64_t)j * kKT;
        const int vcols = left < kKT ? (int)left : kKT;
        const uint32_t s_addr = tmem + lane_addr + Lay::s_col + (uint32_t)(st * kKT);
        const bool full = vcols == kKT;
        const float* bias = sm.kbias[st];
        // group counts: the staged shifts were published with the K/V tile (kv_full)
        if (grouped && !wait_all(&sm.kv_full[st], (g / kKS) & 1, abort)) {
          ok = false;
          break;
        }
        // pass 1: the row maximum (the scale is positive, so the maximum of the scaled
        // scores is the scaled maximum, exactly; with shifts, of the shifted logits)
        float mt;
        if (grouped) {
          mt = full ? row_max<true, true>(s_addr, vcols, sl2, bias) : row_max<false, true>(s_addr, vcols, sl2, bias);
        } else {
          const float mr = full ? row_max<true>(s_addr, vcols) : row_max<false>(s_addr, vcols);
          mt = mr * sl2;
        }
        float alpha = 1.f;
        bool resc = false;
        if (mt > m_used + 8.f) {
          resc = m_used != neg_inf();
          alpha = resc ? ex2(m_used - mt) : 0.f;
          m_used = mt;
        }
        if (__any_sync(0xffffffffu, resc)) {
          // O holds the previous tiles' P.V: rescale it once that product has landed
          if (!wait_all(&sm.pv_done, (g - 1) & 1, abort)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const float f = resc ? alpha : 1.f;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            float o[32];
            tc::tmem_ld32(o_addr + (uint32_t)(c * 32), o);
            tc::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= f;
            tc::tmem_st32(o_addr + (uint32_t)(c * 32), o);
          }
          tc::tmem_wait_st();
        }
        // pass 2: P = 2^(s - m) as bf16 into TMEM over the consumed S columns, and its row sum
        float sum;
        if (grouped)
          sum = full ? row_exp<true, true>(s_addr, vcols, sl2, m_used, bias)
                     : row_exp<false, true>(s_addr, vcols, sl2, m_used, bias);
        else
          sum = full ? row_exp<true>(s_addr, vcols, sl2, m_used) : row_exp<false>(s_addr, vcols, sl2, m_used);
        l = l * alpha + sum;
        tc::tmem_wait_st();   // P has landed in TMEM before the P.V product may read it
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          tc::mbar_arrive(&sm.s_free[st]);
          tc::mbar_arrive(&sm.p_full[st]);
        }
      }
      if (!ok) break;
      sm.mrow[qs][row] = amatch ? best : m_used;
      sm.lrow[qs][row] = amatch ? __int_as_float(bidx) : l;
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sm.ml_full[qs]);
    }
  } else {
    // ---------------- epilogue ----------------
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
    int n = 0;
    for (int u = blockIdx.x; u < n_items; u += gridDim.x, ++n) {
      const int qs = n & 1;
      const uint32_t qph = (n >> 1) & 1;
      const bool got = wait_all(&sm.q_full[qs], qph, abort) && wait_all(&sm.ml_full[qs], qph, abort) &&
                       wait_all(&sm.o_full[qs], qph, abort);
      // the four epilogue warps leave together (they share named barriers below)
      if (!tc::named_bar_and(3, 128, got)) break;
      tc::tc_fence_after();
      // everything this item needs from the stage's shared slots is read before dst_free
      // lets the loader reuse them
      const int h = sm.info[qs].h;
      const int T = sm.info[qs].T;
      const int nrows = sm.info[qs].nrows;
      const int dst = sm.qdst[qs][row];
      const float m_used = sm.mrow[qs][row], l = sm.lrow[qs][row];
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sm.dst_free[qs]);
      if (amatch) {
        // the row's best scaled score and cache index for its (query, slot) pair
        if (dst >= 0) {
          a.mbest[(int64_t)h * np + dst] = m_used;
          a.midx[(int64_t)h * np + dst] = __float_as_int(l);
        }
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&sm.o_empty[qs]);
        continue;
      }
      const uint32_t o_addr = tmem + lane_addr + Lay::o_col + (uint32_t)(qs * 128);
      const bool live = T > 0 && l > 0.f;
      const float inv = live ? 1.0f / l : 0.f;
      const float lse = live ? (m_used + __log2f(l)) * 0.6931471805599453f : neg_inf();
      if (a.mode == kSparse) {
        // slot partials (bf16) at their (query, slot) pair rows: each 32-column slice goes
        // through the transpose buffer and leaves as 64-byte row segments (edst: the row of
        // each)
        const int64_t prow0 = (int64_t)h * np;
        __nv_bfloat16* part16 = reinterpret_cast<__nv_bfloat16*>(a.part_o);
        sm.edst[row] = dst;
        const int ew = warp - kEpiWarp0;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          if (T > 0) {
            tc::tmem_ld32(o_addr + (uint32_t)(c * 32), o);
            tc::tmem_wait_ld();
            tc::tmem_pin32(o);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = 0.f;
          }
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float4 v4 = make_float4(o[4 * k] * inv, o[4 * k + 1] * inv, o[4 * k + 2] * inv, o[4 * k + 3] * inv);
            *reinterpret_cast<float4*>(so + row * 32 + ((k ^ (row & 7)) << 2)) = v4;
          }
          tc::named_bar(2, 128);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int rr = ew * 32 + k * 4 + (lane >> 3), ch = lane & 7;
            const int er = sm.edst[rr];
            if (rr < nrows && er >= 0) {
              const float4 v4 = *reinterpret_cast<const float4*>(so + rr * 32 + ((ch ^ (rr & 7)) << 2));
              *reinterpret_cast<uint2*>(part16 + (prow0 + er) * D + c * 32 + ch * 4) =
                  make_uint2(pack_bf16(v4.x, v4.y), pack_bf16(v4.z, v4.w));
            }
          }
          tc::named_bar(2, 128);
        }
        if (dst >= 0) a.part_lse[prow0 + dst] = lse;
      } else {
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          if (T > 0) {
            tc::tmem_ld32(o_addr + (uint32_t)(c * 32), o);
            tc::tmem_wait_ld();
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = 0.f;
          }
          if (dst >= 0) {
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
        if (dst >= 0 && a.lse) {
          const int64_t nrow = a.mode == kCross ? (int64_t)a.F * a.tpf : a.nq;
          a.lse[(int64_t)h * nrow + dst] = lse;
        }
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sm.o_empty[qs]);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarpA) {
    __syncwarp();
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && sm.abort) flag_status(a.status, FASTAR_DEV_TIMEOUT);
}

// Lists AnnSA's work items — (head, bucket, 128-pair tile) in head-major, bucket order,
// so that the tiles of one bucket run side by side and share its keys in L2.  One CTA.
__global__ void __launch_bounds__(kPlanThreads) sparse_plan_kernel(const AttnArgs a) {
  __shared__ int wsum[kPlanThreads / 32];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int n = a.H * a.B;
  const int per = (n + kPlanThreads - 1) / kPlanThreads;
  const int k0 = t * per, k1 = k0 + per < n ? k0 + per : n;
  auto tiles = [&](int k, int& q0, int& q1, int& kb, int& nk) -> int { return sparse_entry(a, k, q0, q1, kb, nk); };
  int mine = 0;
  for (int k = k0; k < k1; ++k) {
    int q0, q1, kb, nk;
    mine += tiles(k, q0, q1, kb, nk);
  }
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int x = wsum[lane];
    int s = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    wsum[lane] = s - x;   // exclusive prefix of the warp totals
    if (lane == 31) *a.n_items = s;
  }
  __syncthreads();
  int at = wsum[warp] + incl - mine;
  SparseItem* items = static_cast<SparseItem*>(a.items);
  for (int k = k0; k < k1; ++k) {
    int q0, q1, kb, nk;
    const int nt = tiles(k, q0, q1, kb, nk);
    for (int i = 0; i < nt; ++i, ++at) {
      const int s = q0 + i * kAT;
      items[at] = SparseItem{k / a.B, s, s + kAT < q1 ? s + kAT : q1, kb, nk, 0, 0, 0};
    }
  }
}

// Copies each head's cache K/V rows into bucket order — rows [koff[b], koff[b+1]) of
// head h are bucket b's keys — so that the attention kernel reads a bucket's keys as
// contiguous TMA tiles.  Rows past the head's sorted length are zeroed (a tile may
// reach into them; their scores are masked and their values must stay finite).
template <int D>
__global__ void __launch_bounds__(256) sparse_sort_rows_kernel(const AttnArgs a) {
  constexpr int CPR = D / 8;   // 16-byte chunks per row
  const int64_t total = (int64_t)a.H * a.M * CPR;
  const uint4* K = static_cast<const uint4*>(a.k);
  const uint4* V = static_cast<const uint4*>(a.v);
  uint4* KS = static_cast<uint4*>(a.ksorted);
  uint4* VS = static_cast<uint4*>(a.vsorted);
  for (int64_t g = (int64_t)blockIdx.x * 256 + threadIdx.x; g < total; g += (int64_t)gridDim.x * 256) {
    const int64_t row = g / CPR;
    const int c = (int)(g % CPR);
    const int h = (int)(row / a.M);
    const int64_t pos = row % a.M;
    const int32_t n = a.koff[(int64_t)h * (a.B + 1) + a.B];
    uint4 kv = make_uint4(0, 0, 0, 0), vv = kv;
    float lg = 0.f;
    if (pos < n && n <= a.M) {
      const int s = a.kperm[(int64_t)h * a.M + pos];
      if (s >= 0 && s < a.M) {
        const int64_t src = ((int64_t)h * a.M + s) * CPR + c;
        kv = K[src];
        vv = V[src];
        if (a.gcount && c == 0) lg = group_log2(a.gcount[(int64_t)h * a.M + s], a.status);
      } else if (c == 0) {
        flag_status(a.status, FASTAR_DEV_BAD_INDEX);
      }
    }
    KS[g] = kv;
    VS[g] = vv;
    if (a.gcount && c == 0) a.lg_sorted[row] = lg;   // group counts: log2 g in bucket order
  }
}

// AnnCA's kept prompt rows gathered into contiguous (head, frame) planes [H*F, P, d]
// (kept order), so that the attention reads them as tiled TMA boxes; the rows from the
// kept count up to the next 64-row tile are zeroed (they are masked, and P = 0 times a
// finite value stays 0 in the P.V product).
template <int D>
__global__ void __launch_bounds__(256) cross_gather_rows_kernel(const AttnArgs a) {
  constexpr int CPR = D / 8;
  const int64_t total = (int64_t)a.H * a.F * a.P * CPR;
  const uint4* K = static_cast<const uint4*>(a.k);
  const uint4* V = static_cast<const uint4*>(a.v);
  uint4* KS = static_cast<uint4*>(a.ksorted);
  uint4* VS = static_cast<uint4*>(a.vsorted);
  for (int64_t g = (int64_t)blockIdx.x * 256 + threadIdx.x; g < total; g += (int64_t)gridDim.x * 256) {
    const int64_t row = g / CPR;
    const int c = (int)(g % CPR);
    const int64_t hf = row / a.P, t = row % a.P;
    int64_t n = a.kcnt[hf];
    n = n < 0 ? 0 : (n > a.P ? a.P : n);
    int64_t lim = (n + kKT - 1) / kKT * kKT;
    lim = lim < a.P ? lim : a.P;
    if (t >= lim) continue;
    uint4 kv = make_uint4(0, 0, 0, 0), vv = kv;
    if (t < n) {
      const int p = a.kidx[hf * a.P + t];
      if (p >= 0 && p < a.P) {
        const int64_t src = ((hf / a.F) * a.P + p) * CPR + c;
        kv = K[src];
        vv = V[src];
      } else if (c == 0) {
        flag_status(a.status, FASTAR_DEV_BAD_INDEX);
      }
    }
    KS[g] = kv;
    VS[g] = vv;
  }
}

// Merges the r slot partials of every AnnSA query by the exact log-sum-exp rule:
// o = sum_s w_s o_s / sum_s w_s with w_s = exp(lse_s - max_s lse_s), and
// lse = max + log(sum_s w_s).  One warp per (head, query); lane l owns columns
// [l*D/32, (l+1)*D/32), so every slot row (bf16, as the attention stored it) is read as
// one coalesced 2*D-byte line.  Grid: (queries / 8, heads), eight warps per CTA.
template <int D>
__global__ void __launch_bounds__(256) sparse_merge_kernel(const AttnArgs a) {
  pdl_wait();   // the slot partials of the attention before it in the stream
  constexpr int E = D / 32;
  const int h = (int)blockIdx.y;
  const int64_t qi = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (qi >= a.nq) return;
  const int64_t np = a.nq * a.r;
  const int64_t pb = (int64_t)h * np + qi * a.r;   // the query's r slots are adjacent rows
  // the first two slot rows are loaded together with the lse values, before the weights
  // are known (every pair has a row in the partial buffer; a row is used only when its
  // weight is nonzero)
  float4 p0 = make_float4(0.f, 0.f, 0.f, 0.f), p1 = p0;
  const __nv_bfloat16* part16 = reinterpret_cast<const __nv_bfloat16*>(a.part_o);
  auto load_row = [&](int sl) -> float4 {
    const __nv_bfloat16* src = part16 + (pb + sl) * D + lane * E;
    if (E == 4) {
      const uint2 u = __ldcs(reinterpret_cast<const uint2*>(src));
      const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
      const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
      return make_float4(x.x, x.y, y.x, y.y);
    }
    const unsigned u = __ldcs(reinterpret_cast<const unsigned*>(src));
    const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u));
    return make_float4(x.x, x.y, 0.f, 0.f);
  };
  p0 = load_row(0);
  if (a.r > 1) p1 = load_row(1);
  const float ls = lane < a.r ? a.part_lse[pb + lane] : neg_inf();
  float mx = ls;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  const float w = (mx == neg_inf() || ls == neg_inf()) ? 0.f : __expf(ls - mx);
  float W = w;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) W += __shfl_xor_sync(0xffffffffu, W, o);
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  auto add_row = [&](float ws, const float4& v) {
    acc[0] = fmaf(ws, v.x, acc[0]);
    acc[1] = fmaf(ws, v.y, acc[1]);
    acc[2] = fmaf(ws, v.z, acc[2]);
    acc[3] = fmaf(ws, v.w, acc[3]);
  };
  const float w0 = __shfl_sync(0xffffffffu, w, 0), w1 = __shfl_sync(0xffffffffu, w, 1);
  if (w0 != 0.f) add_row(w0, p0);
  if (a.r > 1 && w1 != 0.f) add_row(w1, p1);
  for (int sl = 2; sl < a.r; ++sl) {
    const float ws = __shfl_sync(0xffffffffu, w, sl);
    if (ws != 0.f) add_row(ws, load_row(sl));
  }
  const float invW = W > 0.f ? 1.0f / W : 0.f;
  __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.out) + h * a.o_hs + qi * a.o_ts + lane * E;
  if (E == 4) {
    *reinterpret_cast<uint2*>(orow) =
        make_uint2(pack_bf16(acc[0] * invW, acc[1] * invW), pack_bf16(acc[2] * invW, acc[3] * invW));
  } else {
    *reinterpret_cast<uint32_t*>(orow) = pack_bf16(acc[0] * invW, acc[1] * invW);
  }
  if (lane == 0 && a.lse) a.lse[(int64_t)h * a.nq + qi] = W > 0.f ? mx + __logf(W) : neg_inf();
}

// Launches the instance of one (group counts, mode) pair, setting its shared-memory size
// once; false if the attribute is refused.
template <int D, bool kGrouped, int kMode>
bool attn_launch(int grid, cudaStream_t s, const AttnArgs& b, const CUtensorMap& tk, const CUtensorMap& tv,
                 const CUtensorMap& tq) {
  constexpr size_t smem = AttnLayout<D>::bytes;
  const cudaError_t attr = opt_in_smem((const void*)attn_tc_kernel<D, kGrouped, kMode>, (int)smem);
  if (attr != cudaSuccess) return false;
  const cudaError_t e =
      launch_dependent(attn_tc_kernel<D, kGrouped, kMode>, dim3(grid), dim3(kThreadsA), smem, s, b, tk, tv, tq);
  count_launches(1);
  return e == cudaSuccess;
}

template <int D>
bool attn_tc_impl(const AttnArgs& a, cudaStream_t s) {
  int64_t upper;
  AttnArgs b = a;
  CUtensorMap tk, tv, tq;
  memset(&tk, 0, sizeof(tk));
  memset(&tv, 0, sizeof(tv));
  memset(&tq, 0, sizeof(tq));
  b.kv_tma = 0;
  b.q_tma = 0;
  b.q_token_major = 0;
  if (a.mode == kSparse && a.presorted) {
    // the caller's bucket-ordered copies (written by the compaction as it moved the rows)
    if (make_tmap_bf16_3d(&tk, a.ksorted, D, (uint64_t)a.M, (uint64_t)a.H, (uint64_t)D * 2, (uint64_t)a.M * D * 2,
                          64, kKT) &&
        make_tmap_bf16_3d(&tv, a.vsorted, D, (uint64_t)a.M, (uint64_t)a.H, (uint64_t)D * 2, (uint64_t)a.M * D * 2,
                          64, kKT))
      b.kv_tma = 1;
  } else if (a.mode == kSparse) {
    // bucket-ordered copies of the cache rows, read as contiguous tiles
    // (the queries stay gathered: copying the pairs' rows costs more than it saves)
    if (a.ksorted && a.vsorted &&
        make_tmap_bf16_3d(&tk, a.ksorted, D, (uint64_t)a.M, (uint64_t)a.H, (uint64_t)D * 2,
                          (uint64_t)a.M * D * 2, 64, kKT) &&
        make_tmap_bf16_3d(&tv, a.vsorted, D, (uint64_t)a.M, (uint64_t)a.H, (uint64_t)D * 2,
                          (uint64_t)a.M * D * 2, 64, kKT)) {
      const int64_t chunks = (int64_t)a.H * a.M * (D / 8);
      const int64_t blocks = (chunks + 255) / 256;   // one 16-byte chunk per thread
      if (blocks <= INT_MAX) {
        sparse_sort_rows_kernel<D><<<(unsigned)blocks, 256, 0, s>>>(a);
        count_launches(1);
        b.kv_tma = 1;
      }
    }
  } else if (a.mode == kCross) {
    // with a workspace: the kept rows gathered into contiguous planes, read (like the
    // queries of each frame, which are contiguous rows) by tiled TMA
    if (a.ksorted && a.vsorted && a.P <= INT_MAX &&
        make_tmap_bf16_3d(&tk, a.ksorted, D, (uint64_t)a.P, (uint64_t)a.H * a.F, (uint64_t)D * 2,
                          (uint64_t)a.P * D * 2, 64, kKT) &&
        make_tmap_bf16_3d(&tv, a.vsorted, D, (uint64_t)a.P, (uint64_t)a.H * a.F, (uint64_t)D * 2,
                          (uint64_t)a.P * D * 2, 64, kKT)) {
      const int64_t chunks = (int64_t)a.H * a.F * a.P * (D / 8);
      const int64_t blocks = (chunks + 255) / 256;
      if (blocks > 0 && blocks <= INT_MAX) {
        if (!a.presorted) {   // (the caller's planes hold the kept rows already)
          cross_gather_rows_kernel<D><<<(unsigned)blocks, 256, 0, s>>>(a);
          count_launches(1);
        }
        b.kv_tma = 1;
        const int64_t nrow = (int64_t)a.F * a.tpf;
        const bool tmaj = a.H > 1 && a.q.hs < a.q.ts;
        const bool qok = nrow <= INT_MAX &&
                         (tmaj ? make_tmap_bf16_3d(&tq, a.q.p, D, (uint64_t)a.H, (uint64_t)nrow, (uint64_t)a.q.hs * 2,
                                                   (uint64_t)a.q.ts * 2, 64, 1, kAT)
                               : make_tmap_bf16_3d(&tq, a.q.p, D, (uint64_t)nrow, (uint64_t)a.H, (uint64_t)a.q.ts * 2,
                                                   (uint64_t)a.q.hs * 2, 64, kAT));
        if (qok) {
          b.q_tma = 1;
          b.q_token_major = tmaj ? 1 : 0;
        }
      }
    }
  } else if (a.mode == kDense && a.kv_ts == D && a.nk <= INT_MAX &&
             make_tmap_bf16_3d(&tk, a.k, D, (uint64_t)a.nk, (uint64_t)a.H, (uint64_t)a.kv_ts * 2,
                               (uint64_t)a.kv_hs * 2, 64, kKT) &&
             make_tmap_bf16_3d(&tv, a.v, D, (uint64_t)a.nk, (uint64_t)a.H, (uint64_t)a.kv_ts * 2,
                               (uint64_t)a.kv_hs * 2, 64, kKT)) {
    b.kv_tma = 1;   // the dense keys are contiguous rows already
    // and so are the queries (a token-major view is read as (d, H, tokens) boxes)
    const bool tmaj = a.H > 1 && a.q.hs < a.q.ts;
    const bool qok = tmaj ? make_tmap_bf16_3d(&tq, a.q.p, D, (uint64_t)a.H, (uint64_t)a.nq, (uint64_t)a.q.hs * 2,
                                              (uint64_t)a.q.ts * 2, 64, 1, kAT)
                          : make_tmap_bf16_3d(&tq, a.q.p, D, (uint64_t)a.nq, (uint64_t)a.H, (uint64_t)a.q.ts * 2,
                                              (uint64_t)a.q.hs * 2, 64, kAT);
    if (qok && a.nq <= INT_MAX) {
      b.q_tma = 1;
      b.q_token_major = tmaj ? 1 : 0;
    }
  }
  // group counts need the tensor-engine K/V path (the shifts are staged with its tiles)
  if (a.gcount && !b.kv_tma) return false;
  // so do the caller's kept-row planes (there is no index list to gather by)
  if (a.mode == kCross && a.presorted && !b.kv_tma) return false;
  if (a.mode == kSparse) {
    if (!a.items || !a.n_items) return false;
    if ((int64_t)a.H * a.B + 1 <= kPrefixMax) {
      b.items = nullptr;   // planned inside the attention kernel
    } else {
      sparse_plan_kernel<<<1, kPlanThreads, 0, s>>>(a);
      count_launches(1);
    }
    upper = (int64_t)a.H * ((a.nq * a.r + kAT - 1) / kAT + a.B);
  } else if (a.mode == kCross) {
    upper = (int64_t)a.H * a.F * ((a.tpf + kAT - 1) / kAT);
  } else {
    upper = (int64_t)a.H * ((a.nq + kAT - 1) / kAT);
  }
  if (upper <= 0) return true;
  const int sms = sm_count();
  const int grid = (int)(upper < sms ? upper : sms);
  // group counts (the merge variant) select the instances that stage the logit shifts
  bool ok;
  if (a.mode == kSparse)
    ok = a.gcount ? attn_launch<D, true, kSparse>(grid, s, b, tk, tv, tq)
                  : attn_launch<D, false, kSparse>(grid, s, b, tk, tv, tq);
  else if (a.mode == kCross)
    ok = !a.gcount && attn_launch<D, false, kCross>(grid, s, b, tk, tv, tq);
  else
    ok = a.gcount ? attn_launch<D, true, kDense>(grid, s, b, tk, tv, tq)
                  : attn_launch<D, false, kDense>(grid, s, b, tk, tv, tq);
  if (!ok) return false;
  if (a.mode == kSparse) {
    if (launch_dependent(sparse_merge_kernel<D>, dim3((unsigned)((a.nq + 7) / 8), (unsigned)a.H), dim3(256), 0, s,
                         a) != cudaSuccess)
      return false;
    count_launches(1);
  }
  return true;
}

}  // namespace

// ---------------------------------------------------------------------------------------
// ANN-restricted TempCache match (FAST-AR technical summary §2.A: a lightweight ANN search
// for the temporal correspondence instead of full attention matrices): each query is
// compared only with the incoming cache's keys in its own buckets.  The attention engine
// runs in match mode over (head, bucket, 128-pair) items; a finaliser merges the r slots.
// ---------------------------------------------------------------------------------------

// The incoming cache in bucket order: K rows (bf16, [H, M, d]), 1/|k| and the cache index
// of every sorted key ([H, mstride]; past the sorted length: zero row, 0, -1).  Also
// clears the eviction flags and owners.
template <int D>
__global__ void __launch_bounds__(256)
    ann_sort_rows_kernel(const AttnArgs a, const float* __restrict__ knorm, float* inv_sorted, int32_t* j_sorted,
                         uint4* ks, uint8_t* evict, int32_t* owner) {
  constexpr int CPR = D / 8;
  const uint4* K = static_cast<const uint4*>(a.k);
  const int64_t total = (int64_t)a.H * a.mstride * CPR;
  for (int64_t g = (int64_t)blockIdx.x * 256 + threadIdx.x; g < total; g += (int64_t)gridDim.x * 256) {
    const int64_t row = g / CPR;
    const int c = (int)(g % CPR);
    const int h = (int)(row / a.mstride);
    const int64_t pos = row % a.mstride;
    int32_t n = a.koff[(int64_t)h * (a.B + 1) + a.B];
    n = n < 0 ? 0 : (n > a.M ? (int32_t)a.M : n);
    int s = -1;
    if (pos < n) {
      s = a.kperm[(int64_t)h * a.M + pos];
      if (s < 0 || s >= a.M) {
        if (c == 0) flag_status(a.status, FASTAR_DEV_BAD_INDEX);
        s = -1;
      }
    }
    if (pos < a.M) ks[((int64_t)h * a.M + pos) * CPR + c] = s >= 0 ? K[((int64_t)h * a.M + s) * CPR + c] : make_uint4(0, 0, 0, 0);
    if (c == 0) {
      const float kn = s >= 0 ? knorm[(int64_t)h * a.M + s] : 0.f;
      inv_sorted[row] = kn > 0.f ? 1.0f / kn : 0.f;
      j_sorted[row] = s;
    }
  }
  for (int64_t g = (int64_t)blockIdx.x * 256 + threadIdx.x; g < (int64_t)a.H * a.M; g += (int64_t)gridDim.x * 256) {
    evict[g] = 0;
    if (owner) owner[g] = -1;
  }
}

// Per query (one warp): the best of its r slots — largest q.k/|k|, then lowest cache
// index — is top1; s1 = that / |q|; the entry is evicted when cos(kcur_i, k_top1) >= tau,
// and its owner is the lowest evicting query (atomic minimum over the unsigned view).
template <int D>
__global__ void __launch_bounds__(256)
    ann_match_finalize_kernel(const AttnArgs a, TokView kcur, const float* __restrict__ knorm, float tau,
                              int32_t* top1, float* s1, uint8_t* evict, int32_t* owner) {
  constexpr int E = D / 32;
  const int64_t wq = ((int64_t)blockIdx.x * 256 + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wq >= (int64_t)a.H * a.nq) return;
  const int h = (int)(wq / a.nq);
  const int64_t i = wq % a.nq;
  const int64_t pb = ((int64_t)h * a.nq + i) * a.r;
  float b = neg_inf();
  int j = -1;
  if (lane < a.r) {
    j = a.midx[pb + lane];
    b = j >= 0 ? a.mbest[pb + lane] : neg_inf();
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ob = __shfl_xor_sync(0xffffffffu, b, o);
    const int oj = __shfl_xor_sync(0xffffffffu, j, o);
    if (oj >= 0 && (j < 0 || ob > b || (ob == b && oj < j))) {
      b = ob;
      j = oj;
    }
  }
  const __nv_bfloat16* Q = static_cast<const __nv_bfloat16*>(a.q.p) + h * a.q.hs + i * a.q.ts + lane * E;
  const __nv_bfloat16* Kc = static_cast<const __nv_bfloat16*>(kcur.p) + h * kcur.hs + i * kcur.ts + lane * E;
  float qq = 0.f, kk = 0.f, dk = 0.f;
  const bool have = j >= 0 && j < a.M;
  const __nv_bfloat16* Kj = static_cast<const __nv_bfloat16*>(a.k) + ((int64_t)h * a.M + (have ? j : 0)) * D + lane * E;
  __nv_bfloat16 qe[E], ce[E], ke[E];
  if (E == 4) {
    *reinterpret_cast<uint2*>(qe) = *reinterpret_cast<const uint2*>(Q);
    if (have) {
      *reinterpret_cast<uint2*>(ce) = *reinterpret_cast<const uint2*>(Kc);
      *reinterpret_cast<uint2*>(ke) = *reinterpret_cast<const uint2*>(Kj);
    }
  } else {
    *reinterpret_cast<uint32_t*>(qe) = *reinterpret_cast<const uint32_t*>(Q);
    if (have) {
      *reinterpret_cast<uint32_t*>(ce) = *reinterpret_cast<const uint32_t*>(Kc);
      *reinterpret_cast<uint32_t*>(ke) = *reinterpret_cast<const uint32_t*>(Kj);
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const float qv = __bfloat162float(qe[e]);
    qq = fmaf(qv, qv, qq);
    if (have) {
      const float cv = __bfloat162float(ce[e]), kv = __bfloat162float(ke[e]);
      kk = fmaf(cv, cv, kk);
      dk = fmaf(cv, kv, dk);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    qq += __shfl_xor_sync(0xffffffffu, qq, o);
    kk += __shfl_xor_sync(0xffffffffu, kk, o);
    dk += __shfl_xor_sync(0xffffffffu, dk, o);
  }
  if (lane != 0) return;
  const float nq_ = sqrtf(qq);
  top1[(int64_t)h * a.nq + i] = have ? j : -1;
  s1[(int64_t)h * a.nq + i] = have ? (nq_ > 0.f ? b / nq_ : 0.f) : neg_inf();
  if (have) {
    const float den = sqrtf(kk) * knorm[(int64_t)h * a.M + j];
    const float c = den > 0.f ? dk / den : 0.f;
    if (c >= tau) {
      evict[(int64_t)h * a.M + j] = 1;
      if (owner) atomicMin(reinterpret_cast<unsigned int*>(owner) + (int64_t)h * a.M + j, (unsigned int)i);
    }
  }
}

template <int D>
cudaError_t launch_match_ann_impl(TokView q, TokView kcur, int H, int64_t nq, int r, int B, const int32_t* qperm,
                                  const int32_t* qoff, const void* cache_k, const float* cache_knorm, int64_t M,
                                  const int32_t* kperm, const int32_t* koff, float tau, int32_t* top1, float* s1,
                                  uint8_t* evict, int32_t* owner, int32_t* status, void* ws, cudaStream_t s) {
  AttnArgs a{};
  a.mode = kMatchAnn;
  a.H = H;
  a.q = q;
  a.nq = nq;
  a.k = cache_k;
  a.r = r;
  a.B = B;
  a.qperm = qperm;
  a.qoff = qoff;
  a.kperm = kperm;
  a.koff = koff;
  a.M = M;
  a.status = status;
  a.mstride = (M + 80 + 3) & ~(int64_t)3;
  const int64_t np = nq * r;
  uint8_t* w = static_cast<uint8_t*>(ws);
  a.mbest = reinterpret_cast<float*>(w);
  a.midx = reinterpret_cast<int32_t*>(w + sizeof(float) * (size_t)H * np);
  size_t at = (2 * sizeof(float) * (size_t)H * np + 15) & ~(size_t)15;
  a.items = w + at;
  a.n_items = reinterpret_cast<int32_t*>(w + at + sparse_plan_bytes(H, nq, r, B) - 16);
  at = (at + sparse_plan_bytes(H, nq, r, B) + 1023) & ~(size_t)1023;
  uint4* ks = reinterpret_cast<uint4*>(w + at);
  at += sizeof(uint16_t) * (size_t)H * M * D;
  float* inv_sorted = reinterpret_cast<float*>(w + at);
  at += sizeof(float) * (size_t)H * a.mstride;
  int32_t* j_sorted = reinterpret_cast<int32_t*>(w + at);
  a.inv_sorted = inv_sorted;
  a.j_sorted = j_sorted;
  const int64_t chunks = (int64_t)H * a.mstride * (D / 8);
  const int64_t blocks = (chunks + 255) / 256;
  ann_sort_rows_kernel<D><<<(unsigned)blocks, 256, 0, s>>>(a, cache_knorm, inv_sorted, j_sorted, ks, evict, owner);
  count_launches(1);
  CUtensorMap tk, tz;
  memset(&tz, 0, sizeof(tz));
  if (!make_tmap_bf16_3d(&tk, ks, D, (uint64_t)M, (uint64_t)H, (uint64_t)D * 2, (uint64_t)M * D * 2, 64, kKT))
    return cudaErrorInvalidValue;
  AttnArgs b = a;
  b.kv_tma = 1;
  if ((int64_t)H * B + 1 <= kPrefixMax) {
    b.items = nullptr;
  } else {
    sparse_plan_kernel<<<1, kPlanThreads, 0, s>>>(a);
    count_launches(1);
  }
  const int64_t upper = (int64_t)H * ((np + kAT - 1) / kAT + B);
  const int grid = (int)(upper < sm_count() ? upper : sm_count());
  if (!attn_launch<D, false, kMatchAnn>(grid, s, b, tk, tz, tz)) return cudaErrorInvalidValue;
  const int64_t threads = (int64_t)H * nq * 32;
  ann_match_finalize_kernel<D><<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(a, kcur, cache_knorm, tau, top1,
                                                                                   s1, evict, owner);
  count_launches(1);
  return cudaGetLastError();
}

size_t match_ann_workspace(int H, int64_t nq, int d, int r, int B, int64_t M) {
  const int64_t mstride = (M + 80 + 3) & ~(int64_t)3;
  size_t at = (2 * sizeof(float) * (size_t)H * nq * r + 15) & ~(size_t)15;
  at = (at + sparse_plan_bytes(H, nq, r, B) + 1023) & ~(size_t)1023;
  return at + sizeof(uint16_t) * (size_t)H * M * d + 2 * sizeof(float) * (size_t)H * mstride + 1024;
}

cudaError_t launch_match_ann(int d, TokView q, TokView kcur, int H, int64_t nq, int r, int B, const int32_t* qperm,
                             const int32_t* qoff, const void* cache_k, const float* cache_knorm,
                             const int32_t* cache_len, int64_t M, const int32_t* kperm, const int32_t* koff,
                             float tau, int32_t* top1, float* s1, uint8_t* evict, int32_t* owner, int32_t* status,
                             void* ws, cudaStream_t s) {
  (void)cache_len;   // the incoming cache's bucket order (koff) carries its length
  if (d == 128)
    return launch_match_ann_impl<128>(q, kcur, H, nq, r, B, qperm, qoff, cache_k, cache_knorm, M, kperm, koff, tau,
                                      top1, s1, evict, owner, status, ws, s);
  return launch_match_ann_impl<64>(q, kcur, H, nq, r, B, qperm, qoff, cache_k, cache_knorm, M, kperm, koff, tau,
                                   top1, s1, evict, owner, status, ws, s);
}

size_t sparse_plan_bytes(int H, int64_t nq, int r, int B) {
  const int64_t upper = (int64_t)H * ((nq * r + kAT - 1) / kAT + B);
  return sizeof(SparseItem) * (size_t)upper + 16;
}

bool launch_attn_tc(int d, const AttnArgs& a, cudaStream_t s) {
  if (d == 128) return attn_tc_impl<128>(a, s);
  return attn_tc_impl<64>(a, s);
}

}  // namespace fastar
