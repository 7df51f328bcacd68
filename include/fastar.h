/*
 * fastar.h — C ABI of libfastar.so: the per-chunk attention step of FAST-AR
 * ("Fast Autoregressive Video Diffusion and World Models with Temporal Cache
 * Compression and Sparse Attention") on one NVIDIA GB300 (sm_103a).
 *
 * One layer step for one chunk of Nq = F * Tf current tokens is
 *   1. fastar_bucket_assign   (queries: top-r buckets; current keys: 1 bucket + norm)
 *   2. fastar_tempcache_match (top-1 cosine match against the cache + eviction flags)
 *   3. fastar_cache_compact   (drop evicted entries, append the chunk, FIFO cap M)
 *   4. fastar_bucket_sort     (cache keys and (query, slot) pairs grouped by bucket)
 *   5. fastar_sparse_attn     (bucket-restricted self-attention)
 *   6. fastar_annca_select    (frame-relevant prompt tokens)
 *   7. fastar_cross_attn_subset (cross-attention over the kept prompt tokens)
 * and fastar_dense_attn is the dense baseline the speed-up is measured against.
 * The merge variant (technical summary §2.A, Theoretical Basis: Lemma 5.1 — merging
 * identical keys is exact when their values are averaged and their logit is shifted
 * by the group size) replaces step 3 with fastar_cache_compact_merge and step 5 with
 * fastar_sparse_attn_grouped, using the owner output of step 2.
 * Steps 3-5 can also run as fastar_cache_compact_sorted (the compaction, both sorts of
 * step 4 and a bucket-ordered copy of the new K/V rows, written as the rows move) followed
 * by fastar_sparse_attn_presorted, which reads that copy instead of making its own.
 *
 * Conventions shared by every entry point
 *   - Pointers are DEVICE pointers unless stated otherwise.  The caller allocates
 *     and owns every buffer, including the workspace sized by
 *     fastar_workspace_bytes(); the library never allocates or frees memory and
 *     keeps no pointer after a call returns.
 *   - dtype is FASTAR_F32 or FASTAR_BF16 and applies to every floating-point
 *     tensor input and attention output of the call; scores, norms and lse are
 *     always float32.  The arithmetic is fp32 (bf16 inputs, fp32 accumulation).
 *   - Head dimension d is 64 or 128 and is contiguous.  Token tensors are
 *     addressed as base + h*head_stride + t*token_stride + c (strides in
 *     ELEMENTS), so both [H,N,d] and [N,H,d] layouts work without copies; strides
 *     and base pointers must be 16-byte aligned.  Cache tensors are contiguous
 *     [H, M, d]; per-entry metadata is [H, M]; prompt tensors are [H, P, d].
 *   - All work is enqueued on `stream`; no call synchronises the host.  Lengths
 *     that change from step to step (cache length, bucket counts, kept counts)
 *     live in device memory, so a whole step can be captured in a CUDA graph.
 *   - Every call returns FASTAR_OK or a negative FASTAR_E* code.  Arguments are
 *     validated on the host before anything is enqueued; an error return
 *     enqueues nothing.  Data-dependent faults found on the device (a cache
 *     length above M, a bucket id out of range) are OR-ed as FASTAR_DEV_* bits
 *     into the caller's int32 dev_status word (optional where noted) and the
 *     offending element is skipped.  No kernel traps or asserts, and none
 *     waits on a block outside its own thread-block cluster (whose blocks the
 *     hardware schedules together).
 *   - Devices: a call works on the device current on the calling thread.  Per-device
 *     set-up (kernel shared-memory opt-ins, the no-allocation entry's scratch address)
 *     is done on the first call on each device and kept for the life of the process;
 *     do not call the library on a device after cudaDeviceReset.
 *   - Ties of every arg-max / top-k decision go to the lowest index.
 *   - The softmax scale of every attention call must be positive and finite
 *     (FASTAR_EINVAL otherwise).
 */
#ifndef FASTAR_H_
#define FASTAR_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- element types ---------------------------------------------------------- */
#define FASTAR_F32 0
#define FASTAR_BF16 1

/* ---- host return codes -------------------------------------------------------- */
#define FASTAR_OK 0
#define FASTAR_EINVAL (-1)       /* null/misaligned pointer, bad size or stride   */
#define FASTAR_EUNSUPPORTED (-2) /* dtype or head dimension not built             */
#define FASTAR_ECAPACITY (-3)    /* shape beyond a documented limit (M < Nq, ...) */
#define FASTAR_EWORKSPACE (-4)   /* workspace smaller than fastar_workspace_bytes */
#define FASTAR_ECUDA (-5)        /* a launch failed (cudaGetLastError captured)   */

/* ---- device status bits (OR-ed into *dev_status) ------------------------------ */
#define FASTAR_DEV_BAD_LEN 1      /* a cache length was outside [0, M]            */
#define FASTAR_DEV_BAD_BUCKET 2   /* a bucket id was outside [0, B)               */
#define FASTAR_DEV_BAD_INDEX 4    /* an index list pointed outside its range      */
#define FASTAR_DEV_TIMEOUT 8      /* a bounded on-chip wait gave up; outputs invalid */

/* ---- limits ------------------------------------------------------------------------ */
#define FASTAR_MAX_B 256          /* buckets per head                              */
#define FASTAR_MAX_R 8            /* buckets per query                             */
#define FASTAR_MAX_P 1024         /* prompt tokens per head                        */
#define FASTAR_MAX_PQ_KC 256      /* codewords per product-quantization sub-space  */

/* ---- workspace queries --------------------------------------------------------- */
#define FASTAR_OP_MATCH 1
#define FASTAR_OP_SORT 2
#define FASTAR_OP_SPARSE_ATTN 3
#define FASTAR_OP_ANNCA 4
#define FASTAR_OP_MATCH_ANN 5
#define FASTAR_OP_CROSS_ATTN 6
#define FASTAR_OP_MATCH_PQ 7

/* Bytes of workspace `op` needs for the given sizes (0 if it needs none).
 * MATCH: n = Nq, M = cache capacity.  SORT: n = elements per head before the
 * r fan-out.  SPARSE_ATTN: n = Nq, M = cache capacity (the bf16 path keeps a
 * bucket-ordered copy of the cache K/V in it).  ANNCA: F frames, P prompt tokens.
 * MATCH_ANN: n = Nq, M, d, B, r.  CROSS_ATTN: d, P, F (the bf16 path's gathered copy of
 * the kept prompt rows).  MATCH_PQ: n = Nq, M, d (the decoded cached keys).
 * Unused arguments are ignored.  Returns 0 for an unknown op. */
size_t fastar_workspace_bytes(int op, int H, int64_t n, int64_t M, int d, int B, int r,
                              int64_t P, int F);

/* Human-readable text for a FASTAR_* return code (static storage). */
const char* fastar_status_string(int status);

/* Library ABI version (major*100 + minor). */
int fastar_version(void);

/* Text of the CUDA error behind the calling thread's most recent FASTAR_ECUDA
 * return ("no error" if there was none); static storage. */
const char* fastar_last_cuda_error(void);

/* Number of kernels the library has enqueued in this process so far (a
 * diagnostic: the difference across a captured step is that step's launch count). */
long long fastar_kernel_launches(void);

/* ---- 1. ANN bucket assignment ---------------------------------------------------
 * FAST-AR technical summary §2.C (AnnSA assigns tokens to ANN buckets, "semantic
 * neighbourhoods") and §2.B (AnnCA shares the buckets); the random unit-centroid
 * ANN itself is fixed by the method spec (the pages name only "LSH or
 * quantization").
 * For every row x = X[h, t, :] (t < n) and centroids C[h] ([H, B, d], same dtype,
 * contiguous):
 *   score_c = <C[h, c], x>;  ids[h, t, 0..r) = the r largest scores, ordered by
 *   (score desc, c asc).  r = 1 gives the key bucket argmax_c score_c.
 * Outputs: ids int32 [H, n, r] (required); scores float [H, n, r] (optional, the
 * chosen scores); norms float [H, n] (optional, |x|_2).  n = 0 is a no-op.
 * Limits: 1 <= r <= min(B, FASTAR_MAX_R), B <= FASTAR_MAX_B. */
int fastar_bucket_assign(const void* x, int dtype, int H, int64_t n, int d,
                         int64_t head_stride, int64_t token_stride,
                         const void* centroids, int B, int r,
                         int32_t* ids, float* scores, float* norms, cudaStream_t stream);

/* ---- 1b. both assignments of a step in one call ---------------------------------------
 * The two uses of 1 in a layer step, one launch: q_ids [H, n, r] = the queries' top-r
 * sets, k_ids [H, n] = the current keys' arg-max buckets, k_norms [H, n] (optional) =
 * |k_cur|, q_norms [H, n] (optional) = |q| (for fastar_annca_select's q_norms).
 * Identical results to fastar_bucket_assign(q, ..., r, q_ids, NULL, q_norms) and
 * fastar_bucket_assign(k_cur, ..., 1, k_ids, NULL, k_norms).  q and k_cur share
 * (head_stride, token_stride).  Limits and errors as 1. */
int fastar_bucket_assign_qk(const void* q, const void* k_cur, int dtype, int H, int64_t n, int d,
                            int64_t head_stride, int64_t token_stride, const void* centroids, int B, int r,
                            int32_t* q_ids, int32_t* k_ids, float* k_norms, float* q_norms, cudaStream_t stream);

/* ---- 2. TempCache match + eviction flags ------------------------------------------
 * FAST-AR technical summary §2.A and blog §1: for each current-frame query, the
 * top-1 nearest key among the cached (previous-frame) keys; a cached entry whose
 * content the current chunk re-expresses closely enough (similarity threshold)
 * is merged away, leaving the most recent representative.
 * For each head h and query i < nq, over the n = cache_len[h] cached entries
 * (age order, oldest first):
 *   top1[h,i] = argmax_j cos(q_i, k_j)   (lowest j on ties; -1 when n == 0)
 *   s1[h,i], s2[h,i] = best and second-best cosine (-inf when absent)
 *   evict[h, top1] = 1 if cos(kcur_i, k_top1) >= tau (kcur_i = current key i).
 *   owner[h, j] (optional, int32 [H, M]; NULL to skip) = the lowest i that evicts j,
 *               -1 where no query evicts j (the merge variant folds j into owner[j]).
 * cos(a,b) = a.b/(|a||b|), 0 on a zero norm.  cache_knorm[h,j] must hold |k_j|
 * (fastar_bucket_assign's norms / fastar_cache_compact maintain it).
 * q and k_cur share (head_stride, token_stride).  evict is [H, M] uint8 and is
 * cleared to 0 (owner to -1) inside the call before the flags are set.  s1/s2 may be
 * NULL.
 * Workspace: fastar_workspace_bytes(FASTAR_OP_MATCH, H, nq, M, d, ...).
 * cache_len values outside [0, M] are clamped and flag FASTAR_DEV_BAD_LEN. */
int fastar_tempcache_match(const void* q, const void* k_cur, int dtype, int H, int64_t nq, int d,
                           int64_t head_stride, int64_t token_stride,
                           const void* cache_k, const float* cache_knorm,
                           const int32_t* cache_len, int64_t M, float tau,
                           int32_t* top1, float* s1, float* s2, uint8_t* evict, int32_t* owner,
                           int32_t* dev_status, void* workspace, size_t workspace_bytes,
                           cudaStream_t stream);

/* ---- 2b. ANN-restricted TempCache match (a variant of 2) -----------------------------
 * FAST-AR technical summary §2.A: the temporal correspondence is searched with a
 * lightweight approximate nearest-neighbour method instead of full attention
 * matrices.  Here the ANN is the bucketing that AnnSA and AnnCA share: query i is
 * compared only with the cached keys whose bucket is one of its r buckets R(i):
 *   top1[h,i] = argmax_{j < n, kb(k_j) in R(i)} cos(q_i, k_j)  (lowest j on ties;
 *               -1 when no cached key shares a bucket with q_i)
 *   s1[h,i]   = that cosine (-inf when top1 = -1)
 *   evict[h, top1] = 1 if cos(kcur_i, k_top1) >= tau, and owner (optional) as in 2
 *   (both cleared first).
 * Inputs beyond 2's: the (query, slot) pairs in bucket order (qperm/qoff from
 * fastar_bucket_sort of the query buckets, r per query) and the INCOMING cache's keys
 * in bucket order (kperm/koff from fastar_bucket_sort of its key buckets with
 * n_valid = cache_len).  bf16 only (FASTAR_EUNSUPPORTED otherwise).
 * Workspace: fastar_workspace_bytes(FASTAR_OP_MATCH_ANN, H, nq, M, d, B, r, ...). */
int fastar_tempcache_match_ann(const void* q, const void* k_cur, int dtype, int H, int64_t nq, int d,
                               int64_t head_stride, int64_t token_stride, int r, int B,
                               const int32_t* qperm, const int32_t* qoff, const void* cache_k,
                               const float* cache_knorm, const int32_t* cache_len, int64_t M,
                               const int32_t* kperm, const int32_t* koff, float tau, int32_t* top1,
                               float* s1, uint8_t* evict, int32_t* owner, int32_t* dev_status,
                               void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ---- 2c. quantised TempCache match (a variant of 2) -----------------------------------
 * FAST-AR technical summary §2.A: the top-1 nearest key is searched with a lightweight
 * ANN, "LSH or Quantization"; this is the quantization family (product quantization).
 * A key of dimension d is m consecutive sub-vectors of d/m elements (d/m = 4 or 8, so m
 * is a multiple of 4); each is coded by the nearest (smallest squared distance, lowest
 * index on ties) of the Kc <= FASTAR_MAX_PQ_KC codewords of its sub-space.  Codebooks
 * are per head, [H, m, Kc, d/m], same dtype, contiguous, 16-byte aligned.
 *
 * fastar_pq_encode: codes [H, n, m] uint8 (4-byte aligned) of the rows of x.
 * fastar_tempcache_match_pq: as 2 with every cached key k_j replaced by its
 *   reconstruction k^_j (its codewords concatenated; cache_codes [H, M, m] from
 *   fastar_pq_encode, moved through compactions by fastar_pq_gather_codes):
 *     top1[h,i] = argmax_{j < n} cos(q_i, k^_j) (lowest j on ties; -1 when n == 0),
 *     s1 = that cosine; evict / owner as in 2, tested on the TRUE keys:
 *     cos(kcur_i, k_top1) >= tau, with cache_knorm = |k_j|.  bf16 only.
 *   Workspace: fastar_workspace_bytes(FASTAR_OP_MATCH_PQ, H, nq, M, d, ...).
 * fastar_pq_gather_codes: the codes of a compacted cache: codes_out[h, s] =
 *   codes_in[h, j] for index_map[h, s] = j < len_in[h], codes_cur[h, i] for
 *   index_map[h, s] = len_in[h] + i, for s < len_out[h] (index_map / len_out from
 *   fastar_cache_compact).  codes_in and codes_out must differ. */
int fastar_pq_encode(const void* x, int dtype, int H, int64_t n, int d, int64_t head_stride,
                     int64_t token_stride, const void* codebooks, int m, int Kc, uint8_t* codes,
                     cudaStream_t stream);
int fastar_tempcache_match_pq(const void* q, const void* k_cur, int dtype, int H, int64_t nq, int d,
                              int64_t head_stride, int64_t token_stride, const void* cache_k,
                              const float* cache_knorm, const uint8_t* cache_codes,
                              const int32_t* cache_len, int64_t M, const void* codebooks, int m, int Kc,
                              float tau, int32_t* top1, float* s1, uint8_t* evict, int32_t* owner,
                              int32_t* dev_status, void* workspace, size_t workspace_bytes,
                              cudaStream_t stream);
int fastar_pq_gather_codes(int H, int64_t nq, int64_t M, int m, const uint8_t* codes_in,
                           const int32_t* len_in, const uint8_t* codes_cur, const int32_t* index_map,
                           const int32_t* len_out, uint8_t* codes_out, int32_t* dev_status,
                           cudaStream_t stream);

/* ---- 3. cache compaction -------------------------------------------------------
 * FAST-AR technical summary §2.A ("merging ... bounds the growth of the KV
 * cache") and blog §1 ("only the most recent representative stays in the
 * cache"); FIFO hard cap M from the method spec.
 * Per head: the new cache is [old entries j < len_in with evict[j] == 0, in age
 * order] ++ [current tokens i = 0..nq-1]; while longer than M the oldest entries
 * are dropped.  Written: k_out, v_out [H,M,d]; knorm_out [H,M] (|k|);
 * kb_out [H,M] (key bucket); len_out [H]; index_map [H,M] int32 with the source
 * of each slot: j (< n) for an old entry, n + i for current token i, -1 past
 * len_out.  Slots past len_out keep stale rows.
 * Current rows come from k_cur/v_cur (head_stride, token_stride) with their norm
 * kcur_norm [H,nq] and bucket kcur_bucket [H,nq] (from fastar_bucket_assign).
 * Out-of-place: the *_in and *_out buffers must not overlap.
 * Requires M >= nq (else FASTAR_ECAPACITY).  dev_status optional. */
int fastar_cache_compact(int dtype, int H, int64_t nq, int d, int64_t M,
                         const void* k_cur, const void* v_cur, int64_t head_stride,
                         int64_t token_stride, const float* kcur_norm, const int32_t* kcur_bucket,
                         const void* k_in, const void* v_in, const float* knorm_in,
                         const int32_t* kb_in, const int32_t* len_in, const uint8_t* evict,
                         void* k_out, void* v_out, float* knorm_out, int32_t* kb_out,
                         int32_t* len_out, int32_t* index_map, int32_t* dev_status,
                         cudaStream_t stream);

/* ---- 3b. cache compaction, merge variant ----------------------------------------
 * FAST-AR technical summary §2.A, Theoretical Basis (Lemma 5.1): identical keys merge
 * with no error when their values are averaged and the logit is shifted by the group
 * size.  Every entry carries a group count g (int32 [H, M], >= 0; a fresh entry is 1).
 * The slot order, lengths, index_map, keys, norms and buckets are those of
 * fastar_cache_compact with the same evict flags.  In addition, current entry i that
 * owns an evicted entry j (owner[h, j] == i from fastar_tempcache_match, j = top1[h, i])
 * takes the group: its value becomes (v_i + g_j v_j) / (1 + g_j) (fp32 arithmetic,
 * rounded once to dtype) and its count 1 + g_j; its key stays k_i.  Other current
 * entries get g = 1 and their own value; survivors keep theirs.  g_out [H, M] is
 * written for slots below len_out.  A negative g_j flags FASTAR_DEV_BAD_INDEX and
 * counts as 0.  Out-of-place like 3 (g_in and g_out must differ). */
int fastar_cache_compact_merge(int dtype, int H, int64_t nq, int d, int64_t M,
                               const void* k_cur, const void* v_cur, int64_t head_stride,
                               int64_t token_stride, const float* kcur_norm, const int32_t* kcur_bucket,
                               const void* k_in, const void* v_in, const float* knorm_in,
                               const int32_t* kb_in, const int32_t* g_in, const int32_t* len_in,
                               const uint8_t* evict, const int32_t* top1, const int32_t* owner,
                               void* k_out, void* v_out, float* knorm_out, int32_t* kb_out,
                               int32_t* g_out, int32_t* len_out, int32_t* index_map,
                               int32_t* dev_status, cudaStream_t stream);

/* ---- 3+4. compaction that also leaves AnnSA's input ready ---------------------------
 * Exactly fastar_cache_compact (same outputs, same slot order), then the stable counting
 * sort of the new cache's bucket ids kb_out over its first len_out[h] slots (fastar_
 * bucket_sort with r = 1, n_valid = len_out: kperm int32 [H, M], koff int32 [H, B+1]),
 * and a copy of the new K/V rows in that bucket order: k_sorted[h, p] = k_out[h,
 * kperm[h, p]] for p < len_out[h] (same for V; [H, M, d], dtype; rows past len_out
 * untouched).  kpos int32 [H, M] receives each slot's position in the bucket order (the
 * inverse of kperm; caller-owned scratch).  The sorted copy is written as the rows move,
 * instead of being re-read from the new cache by fastar_sparse_attn.  1 <= B <=
 * FASTAR_MAX_B; k_sorted / v_sorted 16-byte aligned and distinct from the in and out
 * caches; a bucket id outside [0, B) flags FASTAR_DEV_BAD_BUCKET.
 * qb int32 [H, nq, r] (may be NULL): the step's query buckets.  When given, the same
 * launch also writes AnnSA's query-side order, exactly fastar_bucket_sort(qb, H, nq, r, B,
 * NULL, qperm, qoff): qperm int32 [H, nq*r], qoff int32 [H, B+1] (both required then;
 * 1 <= r <= FASTAR_MAX_R, else FASTAR_EINVAL / FASTAR_ECAPACITY before any work), so
 * that the step needs no separate sort launch.  Without qb, r, qperm and qoff are
 * ignored.  Two kernel launches either way: one thread-block cluster per head plans
 * (the pairs' sort, the survivor scan, the key sort), then the rows move. */
int fastar_cache_compact_sorted(int dtype, int H, int64_t nq, int d, int64_t M,
                                const void* k_cur, const void* v_cur, int64_t head_stride,
                                int64_t token_stride, const float* kcur_norm, const int32_t* kcur_bucket,
                                const void* k_in, const void* v_in, const float* knorm_in,
                                const int32_t* kb_in, const int32_t* len_in, const uint8_t* evict,
                                void* k_out, void* v_out, float* knorm_out, int32_t* kb_out,
                                int32_t* len_out, int32_t* index_map, int B, int32_t* kperm,
                                int32_t* koff, int32_t* kpos, void* k_sorted, void* v_sorted,
                                const int32_t* qb, int r, int32_t* qperm, int32_t* qoff,
                                int32_t* dev_status, cudaStream_t stream);

/* ---- 4. counting sort by bucket --------------------------------------------------
 * Groups tokens by ANN bucket so that bucket-restricted attention runs on dense
 * blocks (FAST-AR technical summary §2.C: "block-sparse operation"; the
 * semantic-aware token permutation of Sparse VideoGen2, which the paper builds
 * on, is the same idea).
 * ids int32 [H, n, r]; per head the elements are e = t*r + s for t < n_valid[h]
 * (n_valid may be NULL: all n).  A stable counting sort by ids[e] writes
 * perm[h, 0..E) (E = n_valid*r; element ids e in bucket order, ascending e within
 * a bucket) and offsets[h, 0..B] (offsets[b] = first position of bucket b,
 * offsets[B] = E).  Ids outside [0,B) are skipped and flag FASTAR_DEV_BAD_BUCKET. */
int fastar_bucket_sort(const int32_t* ids, int H, int64_t n, int r, int B,
                       const int32_t* n_valid, int32_t* perm, int32_t* offsets,
                       int32_t* dev_status, cudaStream_t stream);

/* ---- 5. bucket-restricted (AnnSA) self-attention -------------------------------------
 * FAST-AR technical summary §2.C and blog §3: each query attends only to the keys
 * in its own bucket(s).
 *   O[h,i] = sum_{s < len, kb[s] in R(i)} softmax_s(q_i . k_s * scale) v_s
 * over the compacted cache k, v [H,M,d].  The caller passes the two bucket
 * orders from fastar_bucket_sort: qperm/qoff over the (query, slot) pairs of
 * the [H,nq,r] query buckets, kperm/koff over the cache's key buckets.  A query
 * whose buckets hold no key gets O = 0 and lse = -inf.
 * out: dtype, addressed with (o_head_stride, o_token_stride); lse float [H,nq]
 * (optional).  Workspace: fastar_workspace_bytes(FASTAR_OP_SPARSE_ATTN, H, nq, M, d, B, r, ...). */
int fastar_sparse_attn(const void* q, int dtype, int H, int64_t nq, int d,
                       int64_t q_head_stride, int64_t q_token_stride, int r, int B,
                       const int32_t* qperm, const int32_t* qoff,
                       const void* k, const void* v, int64_t M,
                       const int32_t* kperm, const int32_t* koff, float scale,
                       void* out, int64_t o_head_stride, int64_t o_token_stride, float* lse,
                       int32_t* dev_status, void* workspace, size_t workspace_bytes,
                       cudaStream_t stream);

/* ---- 5b. bucket-restricted self-attention over grouped keys (merge variant) ---------
 * As 5, with group counts group_count int32 [H, M] (per cache slot, from
 * fastar_cache_compact_merge): every key's logit is shifted by ln g,
 *   O[h,i] = sum_s g_s exp(q_i.k_s*scale) v_s / sum_s g_s exp(q_i.k_s*scale)
 * over the same key sets; lse includes the shifts.  A key with g = 0 is an empty group
 * (weight 0); a negative g flags FASTAR_DEV_BAD_INDEX and counts as 0.  Same workspace. */
int fastar_sparse_attn_grouped(const void* q, int dtype, int H, int64_t nq, int d,
                               int64_t q_head_stride, int64_t q_token_stride, int r, int B,
                               const int32_t* qperm, const int32_t* qoff,
                               const void* k, const void* v, int64_t M,
                               const int32_t* kperm, const int32_t* koff, const int32_t* group_count,
                               float scale, void* out, int64_t o_head_stride, int64_t o_token_stride,
                               float* lse, int32_t* dev_status, void* workspace, size_t workspace_bytes,
                               cudaStream_t stream);

/* ---- 5c. bucket-restricted self-attention reading a caller-made bucket-ordered copy ---
 * As 5, with k_sorted / v_sorted ([H, M, d], dtype, 16-byte aligned) the rows of k / v in
 * kperm order, as fastar_cache_compact_sorted writes them: the tensor-core path reads
 * them directly instead of copying the rows itself; k, v and kperm are still required
 * (any other path gathers through them).  Same outputs, workspace and errors as 5. */
int fastar_sparse_attn_presorted(const void* q, int dtype, int H, int64_t nq, int d,
                                 int64_t q_head_stride, int64_t q_token_stride, int r, int B,
                                 const int32_t* qperm, const int32_t* qoff,
                                 const void* k, const void* v, int64_t M,
                                 const int32_t* kperm, const int32_t* koff,
                                 const void* k_sorted, const void* v_sorted, float scale,
                                 void* out, int64_t o_head_stride, int64_t o_token_stride, float* lse,
                                 int32_t* dev_status, void* workspace, size_t workspace_bytes,
                                 cudaStream_t stream);

/* ---- 6. AnnCA prompt selection ---------------------------------------------------
 * FAST-AR technical summary §2.B and blog §2: keep the prompt tokens that share
 * an ANN bucket with at least one of the frame's queries; the always-keep top-k
 * by max query cosine and the threshold tau_ca are fixed by the method spec.
 * Queries i of frame f are i in [f*tpf, (f+1)*tpf).  For prompt token p (< P):
 *   score[h,f,p] = max over the frame's i with pb[h,p] in qb[h,i,0..r) of
 *                  cos(q_i, kp_p)   (gate = 0 drops the bucket condition);
 *                  -inf when there is no such i.
 *   keep[h,f,p] = score >= tau_ca, or p is among the first min(topk, P) in the
 *                 order (score desc, p asc) with -inf after every finite score.
 * Outputs: keep uint8 [H,F,P]; kidx int32 [H,F,P] (kept p ascending, then -1);
 * kcnt int32 [H,F]; score float [H,F,P] (optional).  kp is [H,P,d] contiguous.
 * B: the bucket count (0 if unknown).  qperm/qoff (optional, need B > 0): the
 * (query, slot) pairs of qb grouped by bucket, as fastar_bucket_sort writes them;
 * with them the gated scoring reads each bucket's queries directly instead of
 * scanning qb (same results either way).  q_norms (optional, float [H, F*tpf]): |q_i|
 * as fastar_bucket_assign / _qk write it (fp32 sum of squares); the bf16 tensor-core
 * scorer then divides by these instead of forming |q_i| itself (the cosines agree to
 * fp32 rounding); the other scorers ignore it.  NULL: the call forms the norms.
 * Failure: a (head, frame) whose scores could not all be formed (a bounded wait of the
 * tensor-core scorer timed out, which a working device never does) or hold a NaN (NaN
 * inputs) is not ranked: kcnt = -1, keep 0 and kidx -1 throughout, score NaN.
 * fastar_cross_attn_subset and fastar_cross_attn_kept (no status word) attend to no
 * prompt token for such a frame, exactly as for kcnt = 0: the count is the signal.
 * kp_kept, vp_kept (optional, together; bf16 only, else FASTAR_EUNSUPPORTED): [H,F,P,d]
 * planes that the ranking launch fills with the kept rows: kp_kept[h,f,t] =
 * kp[h, kidx[h,f,t]] for t < kcnt[h,f] (vp_kept from vp, [H,P,d] contiguous, required
 * then), zero rows from kcnt up to the next multiple of 64 (at most P), other rows
 * untouched; after a failure (kcnt = -1) nothing is written.  16-byte aligned and distinct
 * from kp and vp.  They are fastar_cross_attn_kept's input, so that the cross-attention
 * needs no gather launch of its own.
 * Workspace: fastar_workspace_bytes(FASTAR_OP_ANNCA, H, ..., P, F).  P <= FASTAR_MAX_P. */
int fastar_annca_select(const void* q, int dtype, int H, int F, int64_t tpf, int d,
                        int64_t q_head_stride, int64_t q_token_stride,
                        const int32_t* qb, int r, const void* kp, const int32_t* pb, int64_t P,
                        float tau_ca, int topk, int gate, int B,
                        const int32_t* qperm, const int32_t* qoff, const float* q_norms,
                        uint8_t* keep, int32_t* kidx, int32_t* kcnt, float* score,
                        const void* vp, void* kp_kept, void* vp_kept,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ---- 6b. AnnCA prompt selection without any caller allocation ------------------------
 * The paper has no counterpart: this is a convenience for callers that cannot
 * allocate device memory when they run the step (a server that reserves all
 * device memory at start-up, a process under a fixed shared memory budget, a
 * latency-critical host thread where cudaMalloc may block or synchronise).
 * Same arguments and results as fastar_annca_select without the query norms, the
 * score output and the workspace: the per-token scores go to a fixed scratch array inside the
 * library's device image (FASTAR_NOALLOC_MAX_SCORES floats, 1 MiB, held on every
 * GPU that loads the library until the process exits).  H * F * P above that
 * limit returns FASTAR_ECAPACITY.  The first call on a device (with that device
 * current) looks up the array's address; make it before any stream capture.  The
 * address, like every other per-device set-up of the library, lasts for the process:
 * after a cudaDeviceReset the library is not to be called on that device again.
 * All calls share the array: calls that may overlap on the GPU race and must be
 * ordered by the caller.  A call never reads scores that it did not write itself,
 * so a smaller call after a larger one needs no clearing.  The failure rule of 6
 * applies (kcnt = -1).  Calls no allocation routine of any kind. */
#define FASTAR_NOALLOC_MAX_SCORES 262144
int fastar_annca_select_noalloc(const void* q, int dtype, int H, int F, int64_t tpf, int d,
                                int64_t q_head_stride, int64_t q_token_stride,
                                const int32_t* qb, int r, const void* kp, const int32_t* pb, int64_t P,
                                float tau_ca, int topk, int gate,
                                uint8_t* keep, int32_t* kidx, int32_t* kcnt, cudaStream_t stream);

/* ---- 7. cross-attention over the kept prompt subset --------------------------------
 * FAST-AR technical summary §2.B ("cross-attention computed over ... the
 * frame-relevant prompt subset").  For query i of frame f:
 *   O[h,i] = sum_{t < kcnt[h,f]} softmax_t(q_i . kp_{kidx[h,f,t]} * scale) vp_{kidx[h,f,t]}
 * kp, vp [H,P,d] contiguous; kidx/kcnt from fastar_annca_select.  kcnt = 0 gives
 * O = 0, lse = -inf.  lse float [H, F*tpf] optional.
 * workspace (optional, bf16 only): fastar_workspace_bytes(FASTAR_OP_CROSS_ATTN, H, 0, 0,
 * d, 0, 0, P, F) bytes; with it the kept rows are first gathered into contiguous
 * per-frame planes and read as tensor-engine tiles (faster); NULL reads them in place.
 * Same results either way.  A non-NULL workspace that is too small: FASTAR_EWORKSPACE. */
int fastar_cross_attn_subset(const void* q, int dtype, int H, int F, int64_t tpf, int d,
                             int64_t q_head_stride, int64_t q_token_stride,
                             const void* kp, const void* vp, int64_t P,
                             const int32_t* kidx, const int32_t* kcnt, float scale,
                             void* out, int64_t o_head_stride, int64_t o_token_stride,
                             float* lse, void* workspace, size_t workspace_bytes,
                             cudaStream_t stream);

/* ---- 7b. cross-attention over kept-row planes ------------------------------------------
 * 7 with the kept rows already gathered by fastar_annca_select into kp_kept / vp_kept
 * [H,F,P,d] (rows 0..kcnt[h,f) of plane (h,f) are the kept prompt tokens in kidx order):
 *   O[h,i] = sum_{t < kcnt[h,f]} softmax_t(q_i . kp_kept[h,f,t] * scale) vp_kept[h,f,t]
 * for query i of frame f.  The same results as fastar_cross_attn_subset with a workspace
 * on the same selection, in one kernel launch (the tensor-core engine reads the planes as
 * tiles).  bf16 only (FASTAR_EUNSUPPORTED otherwise); planes 16-byte aligned; a frame with
 * kcnt <= 0 (kcnt = -1: a failed selection) attends to nothing (O = 0, lse = -inf), as in 7. */
int fastar_cross_attn_kept(const void* q, int dtype, int H, int F, int64_t tpf, int d,
                           int64_t q_head_stride, int64_t q_token_stride,
                           const void* kp_kept, const void* vp_kept, int64_t P, const int32_t* kcnt,
                           float scale, void* out, int64_t o_head_stride, int64_t o_token_stride,
                           float* lse, cudaStream_t stream);

/* ---- 8. dense attention (the baseline) ------------------------------------------
 * The dense softmax attention FAST-AR is compared against (technical summary,
 * Key Results: speed-ups versus dense FlashAttention-3).
 *   O[h,i] = sum_{j < nk} softmax_j(q_i . k_j * scale) v_j
 * k, v addressed with (kv_head_stride, kv_token_stride).  lse optional. */
int fastar_dense_attn(const void* q, int dtype, int H, int64_t nq, int d,
                      int64_t q_head_stride, int64_t q_token_stride,
                      const void* k, const void* v, int64_t nk,
                      int64_t kv_head_stride, int64_t kv_token_stride, float scale,
                      void* out, int64_t o_head_stride, int64_t o_token_stride, float* lse,
                      cudaStream_t stream);

/* ---- 8b. dense attention over grouped keys (merge variant) ----------------------------
 * As 8, with the count of key j of head h at group_count[h * g_head_stride + j]
 * (g_head_stride >= nk when H > 1): logits shifted by ln g, as in 5b.  Dense attention
 * over a merged cache; with g = 1 everywhere it equals 8. */
int fastar_dense_attn_grouped(const void* q, int dtype, int H, int64_t nq, int d,
                              int64_t q_head_stride, int64_t q_token_stride,
                              const void* k, const void* v, int64_t nk,
                              int64_t kv_head_stride, int64_t kv_token_stride,
                              const int32_t* group_count, int64_t g_head_stride, float scale,
                              void* out, int64_t o_head_stride, int64_t o_token_stride, float* lse,
                              cudaStream_t stream);

/* ---- 9. the transformer around the attention step (a Wan-1.3B-shaped DiT) ---------
 * Not on the pages: the dense operations of the diffusion transformer the attention
 * layer sits in (projections, FFN, embeddings, norms, rotary positions), so that a
 * whole chunk denoise runs on the library.  bf16 tensors, fp32 arithmetic. */

#define FASTAR_ACT_NONE 0
#define FASTAR_ACT_GELU_TANH 1    /* 0.5 v (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3))) */
#define FASTAR_ACT_SILU 2         /* v / (1 + exp(-v))                              */

/* C[m, n] = R[m, n] + gate[n] * act(sum_k A[m, k] W[n, k] + bias[n])  on the tensor cores.
 * A [M, K], W [N, K] (a torch Linear weight), C [M, N], R [M, N]: row-major bf16 with
 * leading dimensions lda, ldw, ldc, ldr in elements (multiples of 8; 16-byte aligned
 * bases).  bias [N] fp32 (NULL: 0).  R NULL: no residual term (C = act(...)).  With R,
 * gate[n] = gate_a[n] + gate_b[n] (fp32; gate_b may be NULL; gate_a NULL: gate 1).
 * c_dtype: FASTAR_BF16 or FASTAR_F32 for C (R is always bf16).  bias and the gates must be
 * 16-byte aligned.
 * M >= 1, N a multiple of 256, K a multiple of 64 (FASTAR_EUNSUPPORTED otherwise).
 * C must not overlap A or W; it may be R (in-place residual update). */
int fastar_gemm(const void* A, int64_t lda, const void* W, int64_t ldw, const float* bias,
                const void* R, int64_t ldr, const float* gate_a, const float* gate_b, void* C,
                int64_t ldc, int c_dtype, int64_t M, int64_t N, int64_t K, int act, int32_t* dev_status,
                cudaStream_t stream);

/* Layer norm of the n rows of x [n, C] (row stride ldx; bf16, C a multiple of 8, <= 4096)
 * with adaptive modulation, into out (row stride ldo; may be x):
 *   y = (x - mean) / sqrt(var + eps)  [* weight[c] + bias[c]]  (weight NULL: no affine)
 *   out = y * (1 + scale[c]) + shift[c],  scale = scale_a + scale_b, shift = shift_a + shift_b
 * (fp32 vectors [C]; any of the four may be NULL, counting 0).  var is the biased
 * variance.  eps > 0.  x, out and every non-NULL vector 16-byte aligned (the vectors
 * are read 16 bytes at a time); FASTAR_EINVAL otherwise. */
int fastar_layernorm_mod(const void* x, int64_t ldx, int64_t n, int C, float eps, const float* weight,
                         const float* bias, const float* shift_a, const float* shift_b,
                         const float* scale_a, const float* scale_b, void* out, int64_t ldo,
                         cudaStream_t stream);

/* In place on the n rows of x [n, C] (bf16, row stride ldx), C = H * d:
 *   weight non-NULL: RMS norm over the row, x / sqrt(mean(x^2) + eps) * weight[c];
 *   rope != 0: rotary positions per head of d channels, split into frame / row / column
 *   parts of dt = d - 4 floor(d / 6), dh = dw = 2 floor(d / 6) channels; in a part of da
 *   channels the pair (2j, 2j + 1) turns by the angle pos * theta^(-2j / da), where token i
 *   sits at frame f0 + i / (grid_h grid_w), row (i / grid_w) % grid_h, column i % grid_w,
 *   f0 = t0 + *t0_dev (t0_dev optional, device int32: lets a captured graph follow the
 *   rollout).
 * d even and >= 12, C a multiple of d and of 8, C <= 4096; x and weight (fp32 [C], read
 * 16 bytes at a time) 16-byte aligned, else FASTAR_EINVAL. */
int fastar_rmsnorm_rope(void* x, int64_t ldx, int64_t n, int C, int d, float eps, const float* weight,
                        int rope, int t0, const int32_t* t0_dev, int grid_h, int grid_w, float theta,
                        cudaStream_t stream);

/* The sinusoidal timestep embedding of the nb timesteps t (device fp32): out[b, i] =
 * cos(t_b f_i), out[b, dim/2 + i] = sin(t_b f_i), f_i = 10000^(-i / (dim/2)); bf16 rows of
 * stride ldo. */
int fastar_sinusoidal_embedding(const float* t, int nb, int dim, void* out, int64_t ldo, cudaStream_t stream);

/* Appends nq rows of k_cur/v_cur to an append-only dense cache [H, cap, d] at row
 * `at` (the dense baseline's growing cache).  Requires at + nq <= cap. */
int fastar_dense_append(int dtype, int H, int64_t nq, int d, const void* k_cur, const void* v_cur,
                        int64_t head_stride, int64_t token_stride, void* k_cache, void* v_cache,
                        int64_t cap, int64_t at, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FASTAR_H_ */
