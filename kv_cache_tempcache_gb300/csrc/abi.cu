// The C ABI of libfastar: argument validation, workspace sizing and dispatch.
// Every check runs on the host before anything is enqueued.
#include <atomic>
#include <cstdint>

#include "fastar.h"
#include "kernels.h"

using fastar::TokView;

namespace fastar {
static std::atomic<long long> g_launches{0};
void count_launches(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
}  // namespace fastar

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t esize(int dtype) { return dtype == FASTAR_BF16 ? 2 : 4; }

int check_dtype_d(int dtype, int d) {
  if (dtype != FASTAR_F32 && dtype != FASTAR_BF16) return FASTAR_EUNSUPPORTED;
  if (d != 64 && d != 128) return FASTAR_EUNSUPPORTED;
  return FASTAR_OK;
}

// A token tensor: non-null (when rows exist), 16-byte aligned base and strides, and
// rows that do not overlap.
int check_tok(const void* p, int dtype, int d, int64_t hs, int64_t ts, int64_t nrows, int H) {
  if (nrows == 0 || H == 0) return FASTAR_OK;
  if (!p || !aligned16(p)) return FASTAR_EINVAL;
  const int64_t es = (int64_t)esize(dtype);
  if (ts < d || hs < 0 || ((ts * es) & 15) || ((hs * es) & 15)) return FASTAR_EINVAL;
  if (H > 1 && hs < d) return FASTAR_EINVAL;
  return FASTAR_OK;
}

thread_local cudaError_t g_last_cuda = cudaSuccess;

int cuda_rc(cudaError_t e) {
  if (e == cudaSuccess) return FASTAR_OK;
  g_last_cuda = e;
  return FASTAR_ECUDA;
}

}  // namespace

extern "C" {

int fastar_version(void) { return 110; }

const char* fastar_last_cuda_error(void) { return cudaGetErrorString(g_last_cuda); }

long long fastar_kernel_launches(void) { return fastar::g_launches.load(std::memory_order_relaxed); }

const char* fastar_status_string(int status) {
  switch (status) {
    case FASTAR_OK: return "ok";
    case FASTAR_EINVAL: return "invalid argument (null or misaligned pointer, bad size or stride)";
    case FASTAR_EUNSUPPORTED: return "unsupported dtype or head dimension";
    case FASTAR_ECAPACITY: return "shape beyond a documented capacity limit";
    case FASTAR_EWORKSPACE: return "workspace smaller than fastar_workspace_bytes()";
    case FASTAR_ECUDA: return "CUDA launch failed";
    default: return "unknown status";
  }
}

size_t fastar_workspace_bytes(int op, int H, int64_t n, int64_t M, int d, int B, int r, int64_t P,
                              int F) {
  if (H <= 0 || n < 0) return 0;
  switch (op) {
    case FASTAR_OP_MATCH: return fastar::match_workspace(H, n, M);
    case FASTAR_OP_SORT: return 0;
    case FASTAR_OP_SPARSE_ATTN: return fastar::sparse_attn_workspace(H, n, d, r, B, M);
    case FASTAR_OP_ANNCA: return fastar::annca_workspace(H, F, P);
    case FASTAR_OP_MATCH_ANN:
      if ((d != 64 && d != 128) || B < 1 || r < 1 || M < 1) return 0;
      return fastar::match_ann_workspace(H, n, d, r, B, M);
    case FASTAR_OP_MATCH_PQ:
      if ((d != 64 && d != 128) || M < 1) return 0;
      return fastar::match_pq_workspace(H, n, M, d);
    case FASTAR_OP_CROSS_ATTN:
      if ((d != 64 && d != 128) || P < 1 || F < 1) return 0;
      return 2 * sizeof(uint16_t) * (size_t)H * F * P * d + 1024;
    default: return 0;
  }
}

int fastar_bucket_assign(const void* x, int dtype, int H, int64_t n, int d, int64_t head_stride,
                         int64_t token_stride, const void* centroids, int B, int r, int32_t* ids,
                         float* scores, float* norms, cudaStream_t stream) {
  int rc = check_dtype_d(dtype, d);
  if (rc) return rc;
  if (H < 0 || n < 0 || B < 1 || r < 1) return FASTAR_EINVAL;
  if (B > FASTAR_MAX_B || r > FASTAR_MAX_R || r > B) return FASTAR_ECAPACITY;
  if (H == 0 || n == 0) return FASTAR_OK;
  if ((rc = check_tok(x, dtype, d, head_stride, token_stride, n, H))) return rc;
  if (!centroids || !aligned16(centroids) || !ids) return FASTAR_EINVAL;
  return cuda_rc(fastar::launch_bucket_assign(dtype, d, TokView{x, head_stride, token_stride}, H, n,
                                              centroids, B, r, ids, scores, norms, stream));
}

int fastar_bucket_assign_qk(const void* q, const void* k_cur, int dtype, int H, int64_t n, int d,
                            int64_t head_stride, int64_t token_stride, const void* centroids, int B, int r,
                            int32_t* q_ids, int32_t* k_ids, float* k_norms, float* q_norms, cudaStream_t stream) {
  int rc = check_dtype_d(dtype, d);
  if (rc) return rc;
  if (H < 0 || n < 0 || B < 1 || r < 1) return FASTAR_EINVAL;
  if (B > FASTAR_MAX_B || r > FASTAR_MAX_R || r > B) return FASTAR_ECAPACITY;
  if (H == 0 || n == 0) return FASTAR_OK;
  if ((rc = check_tok(q, dtype, d, head_stride, token_stride, n, H))) return rc;
  if ((rc = check_tok(k_cur, dtype, d, head_stride, token_stride, n, H))) return rc;
  if (!centroids || !aligned16(centroids) || !q_ids || !k_ids) return FASTAR_EINVAL;
  return cuda_rc(fastar::launch_bucket_assign_qk(dtype, d, TokView{q, head_stride, token_stride},
                                                 TokView{k_cur, head_stride, token_stride}, H, n, centroids, B, r,
                                                 q_ids, k_ids, k_norms, q_norms, stream));
}

int fastar_tempcache_match(const void* q, const void* k_cur, int dtype, int H, int64_t nq, int d,
                           int64_t head_stride, int64_t token_stride, const void* cache_k,
                           const float* cache_knorm, const int32_t* cache_len, int64_t M, float tau,
                           int32_t* top1, float* s1, float* s2, uint8_t* evict, int32_t* owner,
                           int32_t* dev_status, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  int rc = check_dtype_d(dtype, d);
  if (rc) return rc;
  if (H < 0 || nq < 0 || M < 1 || M > INT32_MAX || nq > INT32_MAX) return FASTAR_EINVAL;
  if (H == 0) return FASTAR_OK;
  if ((rc = check_tok(q, dtype, d, head_stride, token_stride, nq, H))) return rc;
  if ((rc = check_tok(k_cur, dtype, d, head_stride, token_stride, nq, H))) return rc;
  if (!cache_k || !aligned16(cache_k) || !cache_knorm || !cache_len || !evict) return FASTAR_EINVAL;
  if (nq > 0 && !top1) return FASTAR_EINVAL;
  if (nq > 0) {
    const size_t need = fastar::match_workspace(H, nq, M);
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return FASTAR_EWORKSPACE;
  }
  return cuda_rc(fastar::launch_tempcache_match(
      dtype, d, TokView{q, head_stride, token_stride}, TokView{k_cur, head_stride, token_stride}, H, nq,
      cache_k, cache_knorm, cache_len, M, tau, top1, s1, s2, evict, owner, dev_status, workspace, stream));
}

int fastar_tempcache_match_ann(const void* q, const void* k_cur, int dtype, int H, int64_t nq, int d,
                               int64_t head_stride, int64_t token_stride, int r, int B,
                               const int32_t* qperm, const int32_t* qoff, const void* cache_k,
                               const float* cache_knorm, const int32_t* cache_len, int64_t M,
                               const int32_t* kperm, const int32_t* koff, float tau, int32_t* top1,
                               float* s1, uint8_t* evict, int32_t* owner, int32_t* dev_status, void* workspace,
                               size_t workspace_bytes, cudaStream_t stream) {
  int rc = check_dtype_d(dtype, d);
  if (rc) return rc;
  if (dtype != FASTAR_BF16) return FASTAR_EUNSUPPORTED;
  if (H < 0 || nq < 0 || M < 1 || M > INT32_MAX || r < 1 || B < 1) return FASTAR_EINVAL;
  if (B > FASTAR_MAX_B || r > FASTAR_MAX_R || nq * r > INT32_MAX) return FASTAR_ECAPACITY;
  if (H == 0) return FASTAR_OK;
  if ((rc = check_tok(q, dtype, d, head_stride, token_stride, nq, H))) return rc;
  if ((rc = check_tok(k_cur, dtype, d, head_stride, token_stride, nq, H))) return rc;
  if (!cache_k || !aligned16(cache_k) || !cache_knorm || !cache_len || !evict || !qperm || !qoff || !kperm ||
      !koff)
    return FASTAR_EINVAL;
  if (nq > 0 && (!top1 || !s1)) return FASTAR_EINVAL;
  const size_t need = fastar::match_ann_workspace(H, nq, d, r, B, M);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return FASTAR_EWORKSPACE;
  if (nq == 0) {
    // no current entries: nothing is matched or evicted
    cudaError_t e = cudaMemsetAsync(evict, 0, (size_t)H * M, stream);
    if (e == cudaSuccess && owner) e = cudaMemsetAsync(owner, 0xff, sizeof(int32_t) * (size_t)H * M, stream);
    return cuda_rc(e);
  }
  return cuda_rc(fastar::launch_match_ann(d, TokView{q, head_stride, token_stride},
                                          TokView{k_cur, head_stride, token_stride}, H, nq, r, B, qperm, qoff,
                                          cache_k, cache_knorm, cache_len, M, kperm, koff, tau, top1, s1, evict,
                                          owner, dev_status, workspace, stream));
}

int fastar_cache_compact(int dtype, int H, int64_t nq, int d, int64_t M, const void* k_cur,
                         const void* v_cur, int64_t head_stride, int64_t token_stride,
                         const float* kcur_norm, const int32_t* kcur_bucket, const void* k_in,
                         const void* v_in, const float* knorm_in, const int32_t* kb_in,
                         const int32_t* len_in, const uint8_t* evict, void* k_out, void* v_out,
                         float* knorm_out, int32_t* kb_out, int32_t* len_out, int32_t* index_map,
                         int32_t* dev_status, cudaStream_t stream) {
  int rc = check_dtype_d(dtype, d);
  if (rc) return rc;
  if (H < 0 || nq < 0 || M < 1 || M > INT32_MAX) return FASTAR_EINVAL;
  if (M < nq) return FASTAR_ECAPACITY;
  if (H == 0) return FASTAR_OK;
  if ((rc = check_tok(k_cur, dtype, d, head_stride, token_stride, nq, H))) return rc;
  if ((rc = check_tok(v_cur, dtype, d, head_stride, token_stride, nq, H))) return rc;
  if (nq > 0 && (!kcur_norm || !kcur_bucket)) return FASTAR_EINVAL;
  const void* ptrs[] = {k_in, v_in, k_out, v_out};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return FASTAR_EINVAL;
  if (!knorm_in || !kb_in || !len_in || !evict || !knorm_out || !kb_out || !len_out || !index_map)
    return FASTAR_EINVAL;
  if (k_in == k_out || v_in == v_out || knorm_in == knorm_out || kb_in == kb_out) return FASTAR_EINVAL;
  return cuda_rc(fastar::launch_cache_compact(
      dtype, d, H, nq, M, TokView{k_cur, head_stride, token_stride}, TokView{v_cur, head_stride, token_stride},
      kcur_norm, kcur_bucket, k_in, v_in, knorm_in, kb_in, len_in, evict, k_out, v_out, knorm_out, kb_out,
      len_out, index_map, dev_status, nullptr, nullptr, nullptr, nullptr, stream));
}

int fastar_cache_compact_sorted(int dtype, int H, int64_t nq, int d, int64_t M, const void* k_cur,
                                const void* v_cur, int64_t head_stride, int64_t token_stride,
                                const float* kcur_norm, const int32_t* kcur_bucket, const void* k_in,
                                const void* v_in, const float* knorm_in, const int32_t* kb_in,
                                const int32_t* len_in, const uint8_t* evict, void* k_out, void* v_out,
                                float* knorm_out, int32_t* kb_out, int32_t* len_out, int32_t* index_map, int B,
                                int32_t* kperm, int32_t* koff, int32_t* kpos, void* k_sorted, void* v_sorted,
                                const int32_t* qb, int r, int32_t* qperm, int32_t* qoff, int32_t* dev_status,
                                cudaStream_t stream) {
  int rc = check_dtype_d(dtype, d);
  if (rc) return rc;
  if (H < 0 || nq < 0 || M < 1 || M > INT32_MAX || B < 1) return FASTAR_EINVAL;
  if (B > FASTAR_MAX_B) return FASTAR_ECAPACITY;
  if (M < nq) return FASTAR_ECAPACITY;
  if (H == 0) return FASTAR_OK;
  if ((rc = check_tok(k_cur, dtype, d, head_stride, token_stride, nq, H))) return rc;
  if ((rc = check_tok(v_cur, dtype, d, head_stride, token_stride, nq, H))) return rc;
  if (nq > 0 && (!kcur_norm || !kcur_bucket)) return FASTAR_EINVAL;
  const void* ptrs[] = {k_in, v_in, k_out, v_out, k_sorted, v_sorted};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return FASTAR_EINVAL;
  if (!knorm_in || !kb_in || !len_in || !evict || !knorm_out || !kb_out || !len_out || !index_map || !kperm ||
      !koff || !kpos)
    return FASTAR_EINVAL;
  if (k_in == k_out || v_in == v_out || knorm_in == knorm_out || kb_in == kb_out) return FASTAR_EINVAL;
  if (k_sorted == k_in || k_sorted == k_out || v_sorted == v_in || v_sorted == v_out) return FASTAR_EINVAL;
  if (qb) {
    if (r < 1) return FASTAR_EINVAL;
    if (r > FASTAR_MAX_R || nq * r > INT32_MAX) return FASTAR_ECAPACITY;
    if (!qperm || !qoff) return FASTAR_EINVAL;
  }
  return cuda_rc(fastar::launch_cache_compact_sorted(
      dtype, d, H, nq, M, TokView{k_cur, head_stride, token_stride}, TokView{v_cur, head_stride, token_stride},
      kcur_norm, kcur_bucket, k_in, v_in, knorm_in, kb_in, len_in, evict, k_out, v_out, knorm_out, kb_out,
      len_out, index_map, B, kperm, koff, kpos, k_sorted, v_sorted, qb, qb ? r : 0, qb ? qperm : nullptr,
      qb ? qoff : nullptr, dev_status, stream));
}

int fastar_cache_compact_merge(int dtype, int H, int64_t nq, int d, int64_t M, const void* k_cur,
                               const void* v_cur, int64_t head_stride, int64_t token_stride,
                               const float* kcur_norm, const int32_t* kcur_bucket, const void* k_in,
                               const void* v_in, const float* knorm_in, const int32_t* kb_in,
                               const int32_t* g_in, const int32_t* len_in, const uint8_t* evict,
                               const int32_t* top1, const int32_t* owner, void* k_out, void* v_out,
                               float* knorm_out, int32_t* kb_out, int32_t* g_out, int32_t* len_out,
                               int32_t* index_map, int32_t* dev_status, cudaStream_t stream) {
  int rc = check_dtype_d(dtype, d);
  if (rc) return rc;
  if (H < 0 || nq < 0 || M < 1 || M > INT32_MAX) return FASTAR_EINVAL;
  if (M < nq) return FASTAR_ECAPACITY;
  if (H == 0) return FASTAR_OK;
  if ((rc = check_tok(k_cur, dtype, d, head_stride, token_stride, nq, H))) return rc;
  if ((rc = check_tok(v_cur, dtype, d, head_stride, token_stride, nq, H))) return rc;
  if (nq > 0 && (!kcur_norm || !kcur_bucket || !top1)) return FASTAR_EINVAL;
  const void* ptrs[] = {k_in, v_in, k_out, v_out};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return FASTAR_EINVAL;
  if (!knorm_in || !kb_in || !g_in || !len_in || !evict || !owner || !knorm_out || !kb_out || !g_out || !len_out ||
      !index_map)
    return FASTAR_EINVAL;
  if (k_in == k_out || v_in == v_out || knorm_in == knorm_out || kb_in == kb_out || g_in == g_out)
    return FASTAR_EINVAL;
  return cuda_rc(fastar::launch_cache_compact(
      dtype, d, H, nq, M, TokView{k_cur, head_stride, token_stride}, TokView{v_cur, head_stride, token_stride},
      kcur_norm, kcur_bucket, k_in, v_in, knorm_in, kb_in, len_in, evict, k_out, v_out, knorm_out, kb_out,
      len_out, index_map, dev_status, top1, owner, g_in, g_out, stream));
}

int fastar_pq_encode(const void* x, int dtype, int H, int64_t n, int d, int64_t head_stride, int64_t token_stride,
                     const void* codebooks, int m, int Kc, uint8_t* codes, cudaStream_t stream) {
  int rc = check_dtype_d(dtype, d);
  if (rc) return rc;
  if (H < 0 || n < 0 || m < 1 || Kc < 1) return FASTAR_EINVAL;
  if (d % m || (d / m != 4 && d / m != 8) || Kc > FASTAR_MAX_PQ_KC) return FASTAR_EUNSUPPORTED;
  if (H == 0 || n == 0) return FASTAR_OK;
  if ((rc = check_tok(x, dtype, d, head_stride, token_stride, n, H))) return rc;
  if (!codebooks || !aligned16(codebooks) || !codes || (reinterpret_cast<uintptr_t>(codes) & 3)) return FASTAR_EINVAL;
  return cuda_rc(fastar::launch_pq_encode(dtype, d, TokView{x, head_stride, token_stride}, H, n, m, Kc, codebooks,
                                          codes, stream));
}

int fastar_tempcache_match_pq(const void* q, const void* k_cur, int dtype, int H, int64_t nq, int d,
                              int64_t head_stride, int64_t token_stride, const void* cache_k,
                              const float* cache_knorm, const uint8_t* cache_codes, const int32_t* cache_len,
                              int64_t M, const void* codebooks, int m, int Kc, float tau, int32_t* top1, float* s1,
                              uint8_t* evict, int32_t* owner, int32_t* dev_status, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream) {
  int rc = check_dtype_d(dtype, d);
  if (rc) return rc;
  if (dtype != FASTAR_BF16) return FASTAR_EUNSUPPORTED;
  if (H < 0 || nq < 0 || M < 1 || M > INT32_MAX || nq > INT32_MAX || m < 1 || Kc < 1) return FASTAR_EINVAL;
  if (d % m || (d / m != 4 && d / m != 8) || Kc > FASTAR_MAX_PQ_KC) return FASTAR_EUNSUPPORTED;
  if (H == 0) return FASTAR_OK;
  if ((rc = check_tok(q, dtype, d, head_stride, token_stride, nq, H))) return rc;
  if ((rc = check_tok(k_cur, dtype, d, head_stride, token_stride, nq, H))) return rc;
  if (!cache_k || !aligned16(cache_k) || !cache_knorm || !cache_codes || !cache_len || !evict || !codebooks ||
      !aligned16(codebooks))
    return FASTAR_EINVAL;
  if (nq > 0 && (!top1 || !s1)) return FASTAR_EINVAL;
  const size_t need = fastar::match_pq_workspace(H, nq, M, d);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return FASTAR_EWORKSPACE;
  if (nq == 0) {
    cudaError_t e = cudaMemsetAsync(evict, 0, (size_t)H * M, stream);
    if (e == cudaSuccess && owner) e = cudaMemsetAsync(owner, 0xff, sizeof(int32_t) * (size_t)H * M, stream);
    return cuda_rc(e);
  }
  return cuda_rc(fastar::launch_tempcache_match_pq(
      d, TokView{q, head_stride, token_stride}, TokView{k_cur, head_stride, token_stride}, H, nq, cache_k,
      cache_knorm, cache_codes, cache_len, M, codebooks, m, Kc, tau, top1, s1, evict, owner, dev_status, workspace,
      stream));
}

int fastar_pq_gather_codes(int H, int64_t nq, int64_t M, int m, const uint8_t* codes_in, const int32_t* len_in,
                           const uint8_t* codes_cur, const int32_t* index_map, const int32_t* len_out,
                           uint8_t* codes_out, int32_t* dev_status, cudaStream_t stream) {
  if (H < 0 || nq < 0 || M < 1 || m < 4 || (m & 3) || M > INT32_MAX) return FASTAR_EINVAL;
  if (H == 0) return FASTAR_OK;
  const void* ptrs[] = {codes_in, codes_out};
  for (const void* p : ptrs)
    if (!p || (reinterpret_cast<uintptr_t>(p) & 3)) return FASTAR_EINVAL;
  if (nq > 0 && (!codes_cur || (reinterpret_cast<uintptr_t>(codes_cur) & 3))) return FASTAR_EINVAL;
  if (!len_in || !index_map || !len_out || codes_in == codes_out) return FASTAR_EINVAL;
  return cuda_rc(fastar::launch_pq_gather_codes(H, nq, M, m, codes_in, len_in, codes_cur, index_map, len_out,
                                                codes_out, dev_status, stream));
}

int fastar_bucket_sort(const int32_t* ids, int H, int64_t n, int r, int B, const int32_t* n_valid,
                       int32_t* perm, int32_t* offsets, int32_t* dev_status, cudaStream_t stream) {
  if (H < 0 || n < 0 || r < 1 || B < 1) return FASTAR_EINVAL;
  if (B > FASTAR_MAX_B || r > FASTAR_MAX_R || n * r > INT32_MAX) return FASTAR_ECAPACITY;
  if (H == 0) return FASTAR_OK;
  if ((n > 0 && (!ids || !perm)) || !offsets) return FASTAR_EINVAL;
  return cuda_rc(fastar::launch_bucket_sort(ids, H, n, r, B, n_valid, perm, offsets, dev_status, stream));
}

}  // extern "C"

namespace {

int sparse_attn_impl(const void* q, int dtype, int H, int64_t nq, int d, int64_t q_head_stride,
                     int64_t q_token_stride, int r, int B, const int32_t* qperm, const int32_t* qoff,
                     const void* k, const void* v, int64_t M, const int32_t* kperm, const int32_t* koff,
                     const int32_t* group_count, float scale, void* out, int64_t o_head_stride,
                     int64_t o_token_stride, float* lse, int32_t* dev_status, void* workspace,
                     size_t workspace_bytes, cudaStream_t stream, const void* k_sorted = nullptr,
                     const void* v_sorted = nullptr) {
  int rc = check_dtype_d(dtype, d);
  if (rc) return rc;
  if (H < 0 || nq < 0 || M < 1 || r < 1 || B < 1 || M > INT32_MAX) return FASTAR_EINVAL;
  if (B > FASTAR_MAX_B || r > FASTAR_MAX_R || nq * r > INT32_MAX) return FASTAR_ECAPACITY;
  if (H == 0 || nq == 0) return FASTAR_OK;
  if ((rc = check_tok(q, dtype, d, q_head_stride, q_token_stride, nq, H))) return rc;
  if ((rc = check_tok(out, dtype, d, o_head_stride, o_token_stride, nq, H))) return rc;
  if (!qperm || !qoff || !kperm || !koff || !k || !v || !aligned16(k) || !aligned16(v)) return FASTAR_EINVAL;
  const size_t need = fastar::sparse_attn_workspace(H, nq, d, r, B, M);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return FASTAR_EWORKSPACE;
  if (!(scale > 0.f) || !(scale < 3.0e38f)) return FASTAR_EINVAL;
  fastar::AttnArgs a{};
  a.mode = fastar::kSparse;
  a.H = H;
  a.q = TokView{q, q_head_stride, q_token_stride};
  a.nq = nq;
  a.k = k;
  a.v = v;
  a.r = r;
  a.B = B;
  a.qperm = qperm;
  a.qoff = qoff;
  a.kperm = kperm;
  a.koff = koff;
  a.M = M;
  a.scale = scale;
  a.out = out;
  a.o_hs = o_head_stride;
  a.o_ts = o_token_stride;
  a.lse = lse;
  a.part_o = static_cast<float*>(workspace);
  a.part_lse = a.part_o + (size_t)H * nq * r * d;
  {
    const uintptr_t at = reinterpret_cast<uintptr_t>(a.part_lse + (size_t)H * nq * r);
    uint8_t* plan = reinterpret_cast<uint8_t*>((at + 15) & ~static_cast<uintptr_t>(15));
    a.items = plan;
    a.n_items = reinterpret_cast<int32_t*>(plan + fastar::sparse_plan_bytes(H, nq, r, B) - 16);
    const uintptr_t kat = reinterpret_cast<uintptr_t>(plan + fastar::sparse_plan_bytes(H, nq, r, B));
    uint8_t* ks = reinterpret_cast<uint8_t*>((kat + 1023) & ~static_cast<uintptr_t>(1023));
    a.ksorted = ks;
    a.vsorted = ks + sizeof(uint16_t) * (size_t)H * M * d;
    a.lg_sorted = reinterpret_cast<float*>(ks + 2 * sizeof(uint16_t) * (size_t)H * M * d);
  }
  if (k_sorted) {   // the caller's bucket-ordered copy replaces the workspace one
    a.ksorted = const_cast<void*>(k_sorted);
    a.vsorted = const_cast<void*>(v_sorted);
    a.presorted = 1;
  }
  a.gcount = group_count;
  a.gc_hs = M;
  a.status = dev_status;
  return cuda_rc(fastar::launch_attention(dtype, d, a, stream));
}

int dense_attn_impl(const void* q, int dtype, int H, int64_t nq, int d, int64_t q_head_stride, int64_t q_token_stride,
                    const void* k, const void* v, int64_t nk, int64_t kv_head_stride, int64_t kv_token_stride,
                    const int32_t* group_count, int64_t g_head_stride, float scale, void* out, int64_t o_head_stride,
                    int64_t o_token_stride, float* lse, cudaStream_t stream);

}  // namespace

extern "C" {

int fastar_sparse_attn(const void* q, int dtype, int H, int64_t nq, int d, int64_t q_head_stride,
                       int64_t q_token_stride, int r, int B, const int32_t* qperm, const int32_t* qoff,
                       const void* k, const void* v, int64_t M, const int32_t* kperm, const int32_t* koff,
                       float scale, void* out, int64_t o_head_stride, int64_t o_token_stride, float* lse,
                       int32_t* dev_status, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return sparse_attn_impl(q, dtype, H, nq, d, q_head_stride, q_token_stride, r, B, qperm, qoff, k, v, M, kperm, koff,
                          nullptr, scale, out, o_head_stride, o_token_stride, lse, dev_status, workspace,
                          workspace_bytes, stream);
}

int fastar_sparse_attn_grouped(const void* q, int dtype, int H, int64_t nq, int d, int64_t q_head_stride,
                               int64_t q_token_stride, int r, int B, const int32_t* qperm, const int32_t* qoff,
                               const void* k, const void* v, int64_t M, const int32_t* kperm, const int32_t* koff,
                               const int32_t* group_count, float scale, void* out, int64_t o_head_stride,
                               int64_t o_token_stride, float* lse, int32_t* dev_status, void* workspace,
                               size_t workspace_bytes, cudaStream_t stream) {
  if (!group_count) return FASTAR_EINVAL;
  return sparse_attn_impl(q, dtype, H, nq, d, q_head_stride, q_token_stride, r, B, qperm, qoff, k, v, M, kperm, koff,
                          group_count, scale, out, o_head_stride, o_token_stride, lse, dev_status, workspace,
                          workspace_bytes, stream);
}

int fastar_sparse_attn_presorted(const void* q, int dtype, int H, int64_t nq, int d, int64_t q_head_stride,
                                 int64_t q_token_stride, int r, int B, const int32_t* qperm, const int32_t* qoff,
                                 const void* k, const void* v, int64_t M, const int32_t* kperm,
                                 const int32_t* koff, const void* k_sorted, const void* v_sorted, float scale,
                                 void* out, int64_t o_head_stride, int64_t o_token_stride, float* lse,
                                 int32_t* dev_status, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!k_sorted || !v_sorted || !aligned16(k_sorted) || !aligned16(v_sorted)) return FASTAR_EINVAL;
  return sparse_attn_impl(q, dtype, H, nq, d, q_head_stride, q_token_stride, r, B, qperm, qoff, k, v, M, kperm, koff,
                          nullptr, scale, out, o_head_stride, o_token_stride, lse, dev_status, workspace,
                          workspace_bytes, stream, k_sorted, v_sorted);
}

int fastar_annca_select(const void* q, int dtype, int H, int F, int64_t tpf, int d, int64_t q_head_stride,
                        int64_t q_token_stride, const int32_t* qb, int r, const void* kp, const int32_t* pb,
                        int64_t P, float tau_ca, int topk, int gate, int B, const int32_t* qperm,
                        const int32_t* qoff, const float* q_norms, uint8_t* keep, int32_t* kidx, int32_t* kcnt,
                        float* score,
                        const void* vp, void* kp_kept, void* vp_kept, void* workspace, size_t workspace_bytes,
                        cudaStream_t stream) {
  int rc = check_dtype_d(dtype, d);
  if (rc) return rc;
  if (B < 0 || B > FASTAR_MAX_B) return FASTAR_EINVAL;
  if ((qperm != nullptr) != (qoff != nullptr) || (qperm && B < 1)) return FASTAR_EINVAL;
  if (H < 0 || F < 0 || tpf < 0 || r < 1 || P < 0 || topk < 0) return FASTAR_EINVAL;
  if (P > FASTAR_MAX_P || r > FASTAR_MAX_R) return FASTAR_ECAPACITY;
  if (H == 0 || F == 0) return FASTAR_OK;
  if (!kcnt) return FASTAR_EINVAL;
  if (P > 0) {
    if ((rc = check_tok(q, dtype, d, q_head_stride, q_token_stride, (int64_t)F * tpf, H))) return rc;
    if (tpf > 0 && !qb) return FASTAR_EINVAL;
    if (!kp || !aligned16(kp) || !pb || !keep || !kidx) return FASTAR_EINVAL;
    if ((kp_kept != nullptr) != (vp_kept != nullptr)) return FASTAR_EINVAL;
    if (kp_kept) {
      if (dtype != FASTAR_BF16) return FASTAR_EUNSUPPORTED;
      if (!vp || !aligned16(vp) || !aligned16(kp_kept) || !aligned16(vp_kept)) return FASTAR_EINVAL;
      if (kp_kept == vp_kept || kp_kept == kp || kp_kept == vp || vp_kept == kp || vp_kept == vp)
        return FASTAR_EINVAL;
    }
    if (!score) {
      const size_t need = fastar::annca_workspace(H, F, P);
      if (!workspace || workspace_bytes < need || !aligned16(workspace)) return FASTAR_EWORKSPACE;
    }
  }
  return cuda_rc(fastar::launch_annca_select(dtype, d, TokView{q, q_head_stride, q_token_stride}, H, F, tpf,
                                             qb, r, kp, pb, P, tau_ca, topk, gate, B, qperm, qoff, q_norms, keep, kidx,
                                             kcnt, score, P > 0 ? vp : nullptr, P > 0 ? kp_kept : nullptr,
                                             P > 0 ? vp_kept : nullptr, workspace, stream));
}

int fastar_cross_attn_subset(const void* q, int dtype, int H, int F, int64_t tpf, int d, int64_t q_head_stride,
                             int64_t q_token_stride, const void* kp, const void* vp, int64_t P,
                             const int32_t* kidx, const int32_t* kcnt, float scale, void* out,
                             int64_t o_head_stride, int64_t o_token_stride, float* lse, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream) {
  int rc = check_dtype_d(dtype, d);
  if (rc) return rc;
  if (H < 0 || F < 0 || tpf < 0 || P < 0) return FASTAR_EINVAL;
  if (P > FASTAR_MAX_P) return FASTAR_ECAPACITY;
  if (H == 0 || F == 0 || tpf == 0) return FASTAR_OK;
  if ((rc = check_tok(q, dtype, d, q_head_stride, q_token_stride, (int64_t)F * tpf, H))) return rc;
  if ((rc = check_tok(out, dtype, d, o_head_stride, o_token_stride, (int64_t)F * tpf, H))) return rc;
  if (!kcnt || (P > 0 && (!kp || !vp || !kidx || !aligned16(kp) || !aligned16(vp)))) return FASTAR_EINVAL;
  if (!(scale > 0.f) || !(scale < 3.0e38f)) return FASTAR_EINVAL;
  fastar::AttnArgs a{};
  a.mode = fastar::kCross;
  a.H = H;
  a.q = TokView{q, q_head_stride, q_token_stride};
  a.nq = (int64_t)F * tpf;
  a.k = kp;
  a.v = vp;
  a.F = F;
  a.tpf = tpf;
  a.kidx = kidx;
  a.kcnt = kcnt;
  a.P = P;
  a.scale = scale;
  a.out = out;
  a.o_hs = o_head_stride;
  a.o_ts = o_token_stride;
  a.lse = lse;
  if (workspace && dtype == FASTAR_BF16 && P > 0) {
    const size_t plane = sizeof(uint16_t) * (size_t)H * F * P * d;
    if (workspace_bytes < 2 * plane + 1024) return FASTAR_EWORKSPACE;
    const uintptr_t at = (reinterpret_cast<uintptr_t>(workspace) + 1023) & ~static_cast<uintptr_t>(1023);
    a.ksorted = reinterpret_cast<void*>(at);
    a.vsorted = reinterpret_cast<uint8_t*>(at) + plane;
  }
  return cuda_rc(fastar::launch_attention(dtype, d, a, stream));
}

int fastar_cross_attn_kept(const void* q, int dtype, int H, int F, int64_t tpf, int d, int64_t q_head_stride,
                           int64_t q_token_stride, const void* kp_kept, const void* vp_kept, int64_t P,
                           const int32_t* kcnt, float scale, void* out, int64_t o_head_stride,
                           int64_t o_token_stride, float* lse, cudaStream_t stream) {
  int rc = check_dtype_d(dtype, d);
  if (rc) return rc;
  if (dtype != FASTAR_BF16) return FASTAR_EUNSUPPORTED;
  if (H < 0 || F < 0 || tpf < 0 || P < 0) return FASTAR_EINVAL;
  if (P > FASTAR_MAX_P) return FASTAR_ECAPACITY;
  if (H == 0 || F == 0 || tpf == 0) return FASTAR_OK;
  if ((rc = check_tok(q, dtype, d, q_head_stride, q_token_stride, (int64_t)F * tpf, H))) return rc;
  if ((rc = check_tok(out, dtype, d, o_head_stride, o_token_stride, (int64_t)F * tpf, H))) return rc;
  if (!kcnt) return FASTAR_EINVAL;
  if (P > 0 && (!kp_kept || !vp_kept || !aligned16(kp_kept) || !aligned16(vp_kept))) return FASTAR_EINVAL;
  if (!(scale > 0.f) || !(scale < 3.0e38f)) return FASTAR_EINVAL;
  fastar::AttnArgs a{};
  a.mode = fastar::kCross;
  a.H = H;
  a.q = TokView{q, q_head_stride, q_token_stride};
  a.nq = (int64_t)F * tpf;
  a.F = F;
  a.tpf = tpf;
  a.kcnt = kcnt;
  a.P = P;
  a.scale = scale;
  a.out = out;
  a.o_hs = o_head_stride;
  a.o_ts = o_token_stride;
  a.lse = lse;
  a.ksorted = const_cast<void*>(kp_kept);
  a.vsorted = const_cast<void*>(vp_kept);
  a.presorted = 1;
  return cuda_rc(fastar::launch_attention(dtype, d, a, stream));
}

int fastar_dense_attn(const void* q, int dtype, int H, int64_t nq, int d, int64_t q_head_stride,
                      int64_t q_token_stride, const void* k, const void* v, int64_t nk, int64_t kv_head_stride,
                      int64_t kv_token_stride, float scale, void* out, int64_t o_head_stride,
                      int64_t o_token_stride, float* lse, cudaStream_t stream) {
  return dense_attn_impl(q, dtype, H, nq, d, q_head_stride, q_token_stride, k, v, nk, kv_head_stride,
                         kv_token_stride, nullptr, 0, scale, out, o_head_stride, o_token_stride, lse, stream);
}

int fastar_dense_attn_grouped(const void* q, int dtype, int H, int64_t nq, int d, int64_t q_head_stride,
                              int64_t q_token_stride, const void* k, const void* v, int64_t nk,
                              int64_t kv_head_stride, int64_t kv_token_stride, const int32_t* group_count,
                              int64_t g_head_stride, float scale, void* out, int64_t o_head_stride,
                              int64_t o_token_stride, float* lse, cudaStream_t stream) {
  if (!group_count || g_head_stride < 0 || (H > 1 && g_head_stride < nk)) return FASTAR_EINVAL;
  return dense_attn_impl(q, dtype, H, nq, d, q_head_stride, q_token_stride, k, v, nk, kv_head_stride,
                         kv_token_stride, group_count, g_head_stride, scale, out, o_head_stride, o_token_stride, lse,
                         stream);
}

}  // extern "C"

namespace {

int dense_attn_impl(const void* q, int dtype, int H, int64_t nq, int d, int64_t q_head_stride, int64_t q_token_stride,
                    const void* k, const void* v, int64_t nk, int64_t kv_head_stride, int64_t kv_token_stride,
                    const int32_t* group_count, int64_t g_head_stride, float scale, void* out, int64_t o_head_stride,
                    int64_t o_token_stride, float* lse, cudaStream_t stream) {
  int rc = check_dtype_d(dtype, d);
  if (rc) return rc;
  if (H < 0 || nq < 0 || nk < 0 || nq > INT32_MAX) return FASTAR_EINVAL;
  if (H == 0 || nq == 0) return FASTAR_OK;
  if ((rc = check_tok(q, dtype, d, q_head_stride, q_token_stride, nq, H))) return rc;
  if ((rc = check_tok(out, dtype, d, o_head_stride, o_token_stride, nq, H))) return rc;
  if ((rc = check_tok(k, dtype, d, kv_head_stride, kv_token_stride, nk, H))) return rc;
  if ((rc = check_tok(v, dtype, d, kv_head_stride, kv_token_stride, nk, H))) return rc;
  if (!(scale > 0.f) || !(scale < 3.0e38f)) return FASTAR_EINVAL;
  fastar::AttnArgs a{};
  a.mode = fastar::kDense;
  a.H = H;
  a.q = TokView{q, q_head_stride, q_token_stride};
  a.nq = nq;
  a.k = k;
  a.v = v;
  a.kv_hs = kv_head_stride;
  a.kv_ts = kv_token_stride;
  a.nk = nk;
  a.scale = scale;
  a.out = out;
  a.o_hs = o_head_stride;
  a.o_ts = o_token_stride;
  a.lse = lse;
  a.gcount = group_count;
  a.gc_hs = g_head_stride;
  return cuda_rc(fastar::launch_attention(dtype, d, a, stream));
}

}  // namespace

extern "C" {

int fastar_gemm(const void* A, int64_t lda, const void* W, int64_t ldw, const float* bias, const void* R,
                int64_t ldr, const float* gate_a, const float* gate_b, void* C, int64_t ldc, int c_dtype, int64_t M,
                int64_t N, int64_t K, int act, int32_t* dev_status, cudaStream_t stream) {
  if (M < 0 || N < 0 || K < 0 || act < FASTAR_ACT_NONE || act > FASTAR_ACT_SILU) return FASTAR_EINVAL;
  if (c_dtype != FASTAR_BF16 && c_dtype != FASTAR_F32) return FASTAR_EUNSUPPORTED;
  if (M == 0 || N == 0) return FASTAR_OK;
  if (K == 0 || N % 256 || K % 64) return FASTAR_EUNSUPPORTED;
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return FASTAR_ECAPACITY;
  if (!A || !W || !C || !aligned16(A) || !aligned16(W) || !aligned16(C)) return FASTAR_EINVAL;
  if (lda < K || ldw < K || ldc < N || (lda & 7) || (ldw & 7) || (ldc & 7)) return FASTAR_EINVAL;
  if (R && (!aligned16(R) || ldr < N || (ldr & 7))) return FASTAR_EINVAL;
  if (C == A || C == W) return FASTAR_EINVAL;
  if ((bias && !aligned16(bias)) || (gate_a && !aligned16(gate_a)) || (gate_b && !aligned16(gate_b)))
    return FASTAR_EINVAL;
  return cuda_rc(fastar::launch_gemm_tc(A, lda, W, ldw, bias, R, ldr, gate_a, gate_b, C, ldc,
                                        c_dtype == FASTAR_F32 ? 1 : 0, M, N, K, act, dev_status, stream));
}

int fastar_layernorm_mod(const void* x, int64_t ldx, int64_t n, int C, float eps, const float* weight,
                         const float* bias, const float* shift_a, const float* shift_b, const float* scale_a,
                         const float* scale_b, void* out, int64_t ldo, cudaStream_t stream) {
  if (n < 0 || C < 8 || C % 8 || C > 4096 || !(eps > 0.f)) return FASTAR_EINVAL;
  if (n == 0) return FASTAR_OK;
  if (!x || !out || !aligned16(x) || !aligned16(out) || ldx < C || ldo < C || (ldx & 7) || (ldo & 7))
    return FASTAR_EINVAL;
  if (bias && !weight) return FASTAR_EINVAL;
  for (const float* v : {weight, bias, shift_a, shift_b, scale_a, scale_b})
    if (v && !aligned16(v)) return FASTAR_EINVAL;   // read as 16-byte vectors
  return cuda_rc(fastar::launch_layernorm_mod(x, ldx, n, C, eps, weight, bias, shift_a, shift_b, scale_a, scale_b,
                                              out, ldo, stream));
}

int fastar_rmsnorm_rope(void* x, int64_t ldx, int64_t n, int C, int d, float eps, const float* weight, int rope,
                        int t0, const int32_t* t0_dev, int grid_h, int grid_w, float theta, cudaStream_t stream) {
  if (n < 0 || C < 8 || C % 8 || C > 4096 || d < 12 || d % 2 || C % d || !(eps > 0.f)) return FASTAR_EINVAL;
  if (rope && (grid_h < 1 || grid_w < 1 || !(theta > 1.f) || t0 < 0)) return FASTAR_EINVAL;
  if (n == 0) return FASTAR_OK;
  if (!x || !aligned16(x) || ldx < C || (ldx & 7)) return FASTAR_EINVAL;
  if (weight && !aligned16(weight)) return FASTAR_EINVAL;   // read as 16-byte vectors
  return cuda_rc(
      fastar::launch_rmsnorm_rope(x, ldx, n, C, d, eps, weight, rope, t0, t0_dev, grid_h, grid_w, theta, stream));
}

int fastar_sinusoidal_embedding(const float* t, int nb, int dim, void* out, int64_t ldo, cudaStream_t stream) {
  if (nb < 0 || dim < 2 || dim % 2 || ldo < dim) return FASTAR_EINVAL;
  if (nb == 0) return FASTAR_OK;
  if (!t || !out) return FASTAR_EINVAL;
  return cuda_rc(fastar::launch_sinusoidal(t, nb, dim, out, ldo, stream));
}

int fastar_dense_append(int dtype, int H, int64_t nq, int d, const void* k_cur, const void* v_cur,
                        int64_t head_stride, int64_t token_stride, void* k_cache, void* v_cache, int64_t cap,
                        int64_t at, cudaStream_t stream) {
  int rc = check_dtype_d(dtype, d);
  if (rc) return rc;
  if (H < 0 || nq < 0 || at < 0 || cap < 0) return FASTAR_EINVAL;
  if (at + nq > cap) return FASTAR_ECAPACITY;
  if (H == 0 || nq == 0) return FASTAR_OK;
  if ((rc = check_tok(k_cur, dtype, d, head_stride, token_stride, nq, H))) return rc;
  if ((rc = check_tok(v_cur, dtype, d, head_stride, token_stride, nq, H))) return rc;
  if (!k_cache || !v_cache || !aligned16(k_cache) || !aligned16(v_cache)) return FASTAR_EINVAL;
  return cuda_rc(fastar::launch_dense_append(dtype, d, H, nq, TokView{k_cur, head_stride, token_stride},
                                             TokView{v_cur, head_stride, token_stride}, k_cache, v_cache, cap,
                                             at, stream));
}

}  // extern "C"
