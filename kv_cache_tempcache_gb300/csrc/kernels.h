// Internal launch interface between the C ABI (abi.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "fastar.h"

namespace fastar {

// A token tensor: element (h, t, c) lives at p + h*hs + t*ts + c (elements).
struct TokView {
  const void* p;
  int64_t hs, ts;
};

// Counts kernels enqueued by the library (a diagnostic the ABI exports).
void count_launches(int n);

// ---- buckets ------------------------------------------------------------------------
cudaError_t launch_bucket_assign(int dtype, int d, TokView x, int H, int64_t n, const void* centroids,
                                 int B, int r, int32_t* ids, float* scores, float* norms,
                                 cudaStream_t s);
// Tensor-core bucket assignment (bf16); false if it could not be set up.
bool launch_assign_tc(int d, TokView x, int H, int64_t n, const void* cent, int B, int r, int32_t* ids,
                      float* scores, float* norms, cudaStream_t s);
// Both assignments of a step in one launch (bf16): queries' top-r sets into qb
// [H, n, r], current keys' buckets into kb [H, n] and their norms into knorm [H, n];
// the queries' norms into qnorm [H, n] when it is not null.
bool launch_assign_qk_tc(int d, TokView q, TokView k, int H, int64_t n, const void* cent, int B, int r,
                         int32_t* qb, int32_t* kb, float* knorm, float* qnorm, cudaStream_t s);
cudaError_t launch_bucket_assign_qk(int dtype, int d, TokView q, TokView k, int H, int64_t n, const void* cent,
                                    int B, int r, int32_t* qb, int32_t* kb, float* knorm, float* qnorm,
                                    cudaStream_t s);
// inv (optional, [H, n*r]): each element's position in its head's sorted order.
cudaError_t launch_bucket_sort(const int32_t* ids, int H, int64_t n, int r, int B,
                               const int32_t* n_valid, int32_t* perm, int32_t* offsets,
                               int32_t* status, cudaStream_t s, int32_t* inv = nullptr);

// ---- TempCache ----------------------------------------------------------------------
int match_splits(int H, int64_t nq, int64_t M);
size_t match_workspace(int H, int64_t nq, int64_t M);
int match_tc_splits(int H, int64_t nq, int64_t M);
size_t match_tc_workspace(int H, int64_t nq, int64_t M);
// Tensor-core match (bf16): writes [S, H, nq] partial top-2s and clears evict;
// returns S, or -1 if the launch could not be set up (the caller falls back).
int launch_match_tc(int d, TokView q, int H, int64_t nq, const void* ck, const float* cknorm,
                    const int32_t* clen, int64_t M, bool top2, float4* part, uint8_t* evict,
                    int32_t* owner, int32_t* status, cudaStream_t s);
cudaError_t launch_tempcache_match(int dtype, int d, TokView q, TokView kcur, int H, int64_t nq,
                                   const void* cache_k, const float* cache_knorm,
                                   const int32_t* cache_len, int64_t M, float tau, int32_t* top1,
                                   float* s1, float* s2, uint8_t* evict, int32_t* owner,
                                   int32_t* status, void* ws, cudaStream_t s);
// ---- product quantization (the quantised match) ---------------------------------------
cudaError_t launch_pq_encode(int dtype, int d, TokView x, int H, int64_t n, int m, int Kc, const void* cb,
                             uint8_t* codes, cudaStream_t s);
cudaError_t launch_pq_decode(int d, int H, int64_t M, int m, int Kc, const uint8_t* codes, const int32_t* clen,
                             const void* cb, void* khat, float* khat_norm, int32_t* status, cudaStream_t s);
cudaError_t launch_pq_gather_codes(int H, int64_t nq, int64_t M, int m, const uint8_t* codes_in,
                                   const int32_t* len_in, const uint8_t* codes_cur, const int32_t* imap,
                                   const int32_t* len_out, uint8_t* codes_out, int32_t* status, cudaStream_t s);
size_t match_pq_workspace(int H, int64_t nq, int64_t M, int d);
cudaError_t launch_tempcache_match_pq(int d, TokView q, TokView kc, int H, int64_t nq, const void* ck,
                                      const float* cknorm, const uint8_t* codes, const int32_t* clen, int64_t M,
                                      const void* cb, int m, int Kc, float tau, int32_t* top1, float* s1,
                                      uint8_t* evict, int32_t* owner, int32_t* status, void* ws, cudaStream_t s);
cudaError_t launch_cache_compact(int dtype, int d, int H, int64_t nq, int64_t M, TokView kcur,
                                 TokView vcur, const float* kcur_norm, const int32_t* kcur_bucket,
                                 const void* k_in, const void* v_in, const float* knorm_in,
                                 const int32_t* kb_in, const int32_t* len_in, const uint8_t* evict,
                                 void* k_out, void* v_out, float* knorm_out, int32_t* kb_out,
                                 int32_t* len_out, int32_t* index_map, int32_t* status,
                                 const int32_t* top1, const int32_t* owner, const int32_t* g_in,
                                 int32_t* g_out, cudaStream_t s);

// The compaction that also leaves AnnSA's input ready: the new cache's bucket ids, their
// stable counting sort (kperm, koff, and kpos = each slot's position in bucket order), a
// bucket-ordered copy of the new K/V rows (ksorted, vsorted), written as the rows move,
// and (qb non-null) the (query, slot) pairs' counting sort (qperm, qoff): two launches.
cudaError_t launch_cache_compact_sorted(int dtype, int d, int H, int64_t nq, int64_t M, TokView kc, TokView vc,
                                        const float* kcn, const int32_t* kcb, const void* kin, const void* vin,
                                        const float* knin, const int32_t* kbin, const int32_t* len_in,
                                        const uint8_t* evict, void* kout, void* vout, float* knout,
                                        int32_t* kbout, int32_t* len_out, int32_t* imap, int B, int32_t* kperm,
                                        int32_t* koff, int32_t* kpos, void* ksorted, void* vsorted,
                                        const int32_t* qb, int r, int32_t* qperm, int32_t* qoff, int32_t* status,
                                        cudaStream_t s);

// ---- attention ------------------------------------------------------------------------
enum AttnMode { kDense = 0, kCross = 1, kSparse = 2, kMatchAnn = 3 };

struct AttnArgs {
  int mode;
  int H;
  TokView q;
  int64_t nq;
  // keys/values: dense -> (k, v, kv_hs, kv_ts, nk); cross -> prompt [H,P,d]; sparse -> cache [H,M,d]
  const void* k;
  const void* v;
  int64_t kv_hs, kv_ts, nk;
  // cross
  int F;
  int64_t tpf;
  const int32_t* kidx;
  const int32_t* kcnt;
  int64_t P;
  // sparse
  int r, B;
  const int32_t* qperm;
  const int32_t* qoff;
  const int32_t* kperm;
  const int32_t* koff;
  int64_t M;
  float scale;
  // outputs
  void* out;
  int64_t o_hs, o_ts;
  float* lse;
  float* part_o;    // sparse partials [H, nq*r, d], row = (query, slot) pair (bf16 on the tensor-core path)
  float* part_lse;  // [H, nq*r]
  void* items;      // sparse: work list written by the planning kernel (tensor-core path)
  void* ksorted;    // sparse: the cache K/V rows in bucket order [H, M, d] (tensor-core path)
  void* vsorted;
  int presorted;    // sparse: ksorted / vsorted already hold that copy (the caller's buffers)
                    // cross: ksorted / vsorted are the caller's kept-row planes [H, F, P, d]
  int kv_tma;       // keys/values arrive as contiguous TMA tiles (set by the launcher)
  int q_tma;        // so do the query tiles: one thread drives every copy (set by the launcher)
  int q_token_major;  // the query tensor map is (d, H, tokens) rather than (d, tokens, H)
  // ANN-restricted match: per bucket-ordered key, 1/|k| and its cache index ([H, mstride]);
  // per (query, slot) pair, the best scaled score and its index
  const float* inv_sorted;
  const int32_t* j_sorted;
  int64_t mstride;
  float* mbest;
  int32_t* midx;
  int32_t* n_items; // sparse: its length
  // merge variant (Lemma 5.1): keys stand for groups of gcount keys and get the logit
  // shift ln g.  sparse: [H, M] per cache slot (gc_hs = M); dense: h * gc_hs + key.
  // lg_sorted: the tensor-core AnnSA path's log2 g in bucket order ([H, M], workspace).
  const int32_t* gcount;
  int64_t gc_hs;
  float* lg_sorted;
  int32_t* status;
};

size_t sparse_attn_workspace(int H, int64_t nq, int d, int r, int B, int64_t M);
// ANN-restricted TempCache match (bf16, tensor cores): workspace and launch.  The pair
// order (qperm/qoff) and the incoming cache's bucket order (kperm/koff) are inputs.
size_t match_ann_workspace(int H, int64_t nq, int d, int r, int B, int64_t M);
cudaError_t launch_match_ann(int d, TokView q, TokView kcur, int H, int64_t nq, int r, int B, const int32_t* qperm,
                             const int32_t* qoff, const void* cache_k, const float* cache_knorm,
                             const int32_t* cache_len, int64_t M, const int32_t* kperm, const int32_t* koff,
                             float tau, int32_t* top1, float* s1, uint8_t* evict, int32_t* owner, int32_t* status,
                             void* ws, cudaStream_t s);
// Bytes of the tensor-core AnnSA work list (inside the sparse workspace).
size_t sparse_plan_bytes(int H, int64_t nq, int r, int B);
// Tensor-core attention (bf16); false if it could not be set up (caller falls back).
bool launch_attn_tc(int d, const AttnArgs& a, cudaStream_t s);
cudaError_t launch_attention(int dtype, int d, const AttnArgs& a, cudaStream_t s);

// ---- AnnCA --------------------------------------------------------------------------
size_t annca_workspace(int H, int F, int64_t P);
// Tensor-core AnnCA scores (bf16, bucket-gated); false if it could not be set up.
// qnorm (optional, [H, F * tpf]): the queries' norms, used instead of forming them.
bool launch_annca_tc(int d, TokView q, int H, int F, int64_t tpf, const int32_t* qb, int r, const void* kp,
                     const int32_t* pb, int64_t P, int B, const float* qnorm, float* score, int32_t* status,
                     cudaStream_t s);
cudaError_t launch_annca_select(int dtype, int d, TokView q, int H, int F, int64_t tpf,
                                const int32_t* qb, int r, const void* kp, const int32_t* pb,
                                int64_t P, float tau_ca, int topk, int gate, int B,
                                const int32_t* qperm, const int32_t* qoff, const float* qnorm, uint8_t* keep,
                                int32_t* kidx, int32_t* kcnt, float* score, const void* vp,
                                void* kp_kept, void* vp_kept, void* ws, cudaStream_t s);

// ---- the transformer around the attention step ----------------------------------------
cudaError_t launch_gemm_tc(const void* A, int64_t lda, const void* W, int64_t ldw, const float* bias,
                           const void* res, int64_t ldr, const float* gate_a, const float* gate_b, void* C, int64_t ldc,
                           int c_f32, int64_t M, int64_t N, int64_t K, int act, int32_t* status, cudaStream_t s);

cudaError_t launch_layernorm_mod(const void* x, int64_t ldx, int64_t n, int C, float eps, const float* w,
                                 const float* b, const float* sha, const float* shb, const float* sca,
                                 const float* scb, void* out, int64_t ldo, cudaStream_t s);
cudaError_t launch_rmsnorm_rope(void* x, int64_t ldx, int64_t n, int C, int d, float eps, const float* w, int rope,
                                int t0, const int32_t* t0_dev, int gh, int gw, float theta, cudaStream_t s);
cudaError_t launch_sinusoidal(const float* t, int nb, int dim, void* out, int64_t ldo, cudaStream_t s);

// ---- dense cache append --------------------------------------------------------------
cudaError_t launch_dense_append(int dtype, int d, int H, int64_t nq, TokView kcur, TokView vcur,
                                void* k_cache, void* v_cache, int64_t cap, int64_t at,
                                cudaStream_t s);

}  // namespace fastar
