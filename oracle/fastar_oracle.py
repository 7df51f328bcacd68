"""Plain CPU oracle of the FAST-AR per-chunk attention step.  TEST INFRASTRUCTURE.

Only the tests, the package's smoke check and the benchmark's CPU-baseline arm may
import or run this module.  It shares no code with the CUDA path and imports nothing
from it; the product path never calls it.

Everything is computed in float64 NumPy (FLOAT), one head at a time, straight from
the definitions.  The benchmark's CPU-baseline leg may set FLOAT to float32, the
precision the method spec names for a CPU baseline, to time the same code in fp32;
the parity tests always run it in float64.  Source: "Fast Autoregressive Video Diffusion and World Models with
Temporal Cache Compression and Sparse Attention" (FAST-AR), as described on the
pages about it:
  * TempCache (technical summary §2.A; blog §1): for each current-frame query, the
    top-1 nearest cached key from previous frames; keys that track the same content
    are grouped, only the most recent representative stays; in practice keys merge
    when their similarity passes a threshold.
  * AnnCA (technical summary §2.B; blog §2): keep the prompt tokens that share an
    ANN bucket with at least one of the frame's queries; cross-attention over that
    subset only.
  * AnnSA (technical summary §2.C; blog §3): reuse the same buckets; each query
    attends only to keys in its own bucket(s).
  * Problem statement: the cache grows with the rollout and is to be bounded.
  * The quantization variant of the match (technical summary §2.A: the ANN is LSH or
    quantization): product quantization of the cached keys, the top-1 searched among
    the decoded keys.
  * The merge variant (technical summary §2.A, "Theoretical Basis", Lemma 5.1):
    identical keys merge with no error when their values are averaged and their
    logit is shifted by the size of the group.
The pages leave the ANN method open; the spec that accompanies them fixes it:
per-head unit centroids, key -> argmax-dot centroid, query -> top-r centroids, ties
to the lowest index, softmax scale 1/sqrt(d), inclusive thresholds, FIFO cap M.

Conventions: a "cosine" of two vectors is a.b / (|a| |b|), and 0 when either norm
is 0.  "-inf" marks "no candidate".  Every index tie goes to the lowest index.
"""
from __future__ import annotations

import numpy as np

NEG_INF = float("-inf")


class CapacityError(ValueError):
    """The cache cap M cannot hold one chunk (M < Nq)."""


# The floating-point type every array of the oracle is computed in (see the header).
FLOAT = np.float64


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=FLOAT)


# ----------------------------------------------------------------------------------
# primitives
# ----------------------------------------------------------------------------------

def cosine_matrix(A, B) -> np.ndarray:
    """[na, nb] cosines between the rows of A and the rows of B (0 on a zero norm)."""
    A = _f64(A)
    B = _f64(B)
    na = np.linalg.norm(A, axis=1)
    nb = np.linalg.norm(B, axis=1)
    dots = A @ B.T
    den = np.outer(na, nb)
    out = np.zeros_like(dots)
    np.divide(dots, den, out=out, where=den > 0)
    return out


def cosine_rows(A, B) -> np.ndarray:
    """[n] cosines between A[i] and B[i]."""
    A = _f64(A)
    B = _f64(B)
    den = np.linalg.norm(A, axis=1) * np.linalg.norm(B, axis=1)
    dots = np.einsum("nd,nd->n", A, B)
    out = np.zeros_like(dots)
    np.divide(dots, den, out=out, where=den > 0)
    return out


def order_desc(scores: np.ndarray) -> np.ndarray:
    """Indices sorted by (score descending, index ascending), along the last axis."""
    return np.argsort(-_f64(scores), axis=-1, kind="stable")


# ----------------------------------------------------------------------------------
# ANN bucketing (AnnSA §2.C / AnnCA §2.B; method fixed by the spec)
# ----------------------------------------------------------------------------------

def centroid_scores(X, C) -> np.ndarray:
    """[n, B] dot products <C[c], x> (the bucketing score; dot, not cosine)."""
    return _f64(X) @ _f64(C).T


def key_buckets(K, C) -> np.ndarray:
    """b(k) = argmax_c <C[c], k>, lowest c on ties.  int64 [n]."""
    S = centroid_scores(K, C)
    if S.shape[0] == 0:
        return np.zeros(0, np.int64)
    return order_desc(S)[:, 0].astype(np.int64)


def query_buckets(Q, C, r: int) -> np.ndarray:
    """R(q) = the r centroids with the largest <C[c], q>, ordered by (score desc, c asc).
    int64 [n, r]."""
    S = centroid_scores(Q, C)
    if r > S.shape[1]:
        raise ValueError("r > B")
    return order_desc(S)[:, :r].astype(np.int64)


def bucket_order(ids, B: int, n_valid=None):
    """Tokens grouped by bucket (technical summary §2.C: each query attends to the keys of
    its own buckets; the spec fixes the grouping as a stable counting sort).  ids [H, n, r]
    bucket ids of the (token, slot) elements, element e = token * r + slot; only the first
    n_valid[h] tokens of head h take part.  Returns perm [H, n*r]: the head's elements in
    bucket order, ascending element id inside a bucket (entries past the head's count are
    -1), and offsets [H, B+1]: where each bucket starts, offsets[h, B] = the count."""
    ids = np.asarray(ids)
    H, n, r = ids.shape
    perm = np.full((H, n * r), -1, dtype=np.int64)
    offsets = np.zeros((H, B + 1), dtype=np.int64)
    for h in range(H):
        nv = n if n_valid is None else int(n_valid[h])
        flat = ids[h, :nv].reshape(-1)
        order = np.argsort(flat, kind="stable")
        perm[h, :order.size] = order
        offsets[h, 1:] = np.cumsum(np.bincount(flat, minlength=B)[:B])
    return perm, offsets


# ----------------------------------------------------------------------------------
# TempCache (technical summary §2.A)
# ----------------------------------------------------------------------------------

def tempcache_match(Q, K_cache):
    """Top-1 temporal correspondence of each current query among the cached keys.

    Q [nq, d]; K_cache [n, d] in age order (oldest first).
    Returns (top1 int64 [nq], s1 [nq], s2 [nq]):
      top1[i] = argmax_j cos(q_i, k_j), lowest j (oldest) on ties; -1 if n == 0
      s1[i]   = the best cosine; s2[i] = the best cosine over j != top1[i]
                (-inf when there is no such j).
    """
    Q = _f64(Q)
    K = _f64(K_cache)
    nq, n = Q.shape[0], K.shape[0]
    if n == 0:
        return (np.full(nq, -1, np.int64), np.full(nq, NEG_INF, FLOAT), np.full(nq, NEG_INF, FLOAT))
    S = cosine_matrix(Q, K)
    top1 = np.argmax(S, axis=1).astype(np.int64)       # first maximum = lowest j
    rows = np.arange(nq)
    s1 = S[rows, top1].copy()
    if n > 1:
        S[rows, top1] = NEG_INF
        s2 = S.max(axis=1)
    else:
        s2 = np.full(nq, NEG_INF, FLOAT)
    return top1, s1, s2


def tempcache_match_ann(Q, R, K_cache, kb_cache):
    """The ANN-restricted variant of the match: each current query is compared only
    with the cached keys that fall in one of its own buckets (technical summary §2.A:
    a lightweight approximate nearest-neighbour search instead of full attention
    matrices; the buckets are the ones AnnSA and AnnCA share).

    Q [nq, d]; R [nq, r] the query bucket sets; K_cache [n, d] in age order with
    key buckets kb_cache [n].  Returns (top1 int64 [nq], s1 [nq]):
      top1[i] = argmax over {j : kb_cache[j] in R[i]} of cos(q_i, k_j), lowest j on
                ties; -1 when no cached key shares a bucket with q_i
      s1[i]   = that cosine (-inf when top1[i] = -1).
    """
    Q = _f64(Q)
    K = _f64(K_cache)
    R = np.asarray(R, np.int64).reshape(Q.shape[0], -1)
    kb = np.asarray(kb_cache, np.int64)
    nq, n = Q.shape[0], K.shape[0]
    top1 = np.full(nq, -1, np.int64)
    s1 = np.full(nq, NEG_INF, FLOAT)
    if n == 0:
        return top1, s1
    S = cosine_matrix(Q, K)
    allowed = (kb[None, :, None] == R[:, None, :]).any(axis=2)   # [nq, n]
    S = np.where(allowed, S, NEG_INF)
    has = allowed.any(axis=1)
    best = np.argmax(S, axis=1).astype(np.int64)                # first maximum = lowest j
    top1[has] = best[has]
    s1[has] = S[np.arange(nq), best][has]
    return top1, s1


# ----------------------------------------------------------------------------------
# product quantization (technical summary §2.A / §2.B: "LSH or Quantization")
# ----------------------------------------------------------------------------------
# A key of dimension d is split into m consecutive sub-vectors of d/m dimensions; each
# sub-vector is replaced by the nearest (Euclidean) of the Kc codewords of its sub-space.
# Readings: codebooks are per head and given (an input, like the centroids); the
# nearest codeword is the one with the smallest squared distance, lowest index on ties;
# the quantised match ranks the cached keys by cos(q, decode(code(k))) and its eviction
# test uses the true key, as the exact match's does.

def pq_distances(X, codebooks) -> np.ndarray:
    """dist[t, s, c] = |x_t[s-th sub-vector] - codebooks[s, c]|^2.  X [n, d];
    codebooks [m, Kc, d/m].  [n, m, Kc]."""
    X = _f64(X)
    Cb = _f64(codebooks)
    m, Kc, ds = Cb.shape
    dist = np.zeros((X.shape[0], m, Kc), FLOAT)
    for s in range(m):
        sub = X[:, s * ds:(s + 1) * ds]
        dist[:, s, :] = ((sub[:, None, :] - Cb[s][None, :, :]) ** 2).sum(axis=2)
    return dist


def pq_encode(X, codebooks) -> np.ndarray:
    """codes[t, s] = argmin_c |x_t[s-th sub-vector] - codebooks[s, c]|^2 (lowest c on
    ties).  int64 [n, m]."""
    dist = pq_distances(X, codebooks)
    if dist.shape[0] == 0:
        return np.zeros((0, dist.shape[1]), np.int64)
    return np.argmin(dist, axis=2).astype(np.int64)


def pq_decode(codes, codebooks) -> np.ndarray:
    """The reconstruction: the chosen codewords concatenated.  [n, d]."""
    Cb = _f64(codebooks)
    codes = np.asarray(codes, np.int64)
    m = Cb.shape[0]
    if codes.shape[0] == 0:
        return np.zeros((0, m * Cb.shape[2]), FLOAT)
    return np.concatenate([Cb[s][codes[:, s]] for s in range(m)], axis=1)


def tempcache_match_pq(Q, codes_cache, codebooks):
    """The quantised TempCache match: top1[i] = argmax_j cos(q_i, k^_j) over the decoded
    cached keys k^_j (lowest j on ties; -1 if the cache is empty); s1 = that cosine."""
    K_hat = pq_decode(codes_cache, codebooks)
    top1, s1, _ = tempcache_match(Q, K_hat)
    return top1, s1


def evict_flags(top1, K_cur, K_cache, tau: float):
    """e_j = 1 iff some query i has top1[i] = j and cos(kcur_i, k_j) >= tau.

    kcur_i is the current key at query i's token position (the key that becomes the
    "most recent representative" of the content the query tracks).  Returns
    (evict bool [n], cos_evict [nq]) where cos_evict[i] = cos(kcur_i, k_top1[i]) (-inf
    when top1[i] < 0)."""
    top1 = np.asarray(top1, np.int64)
    n = np.asarray(K_cache).shape[0]
    e = np.zeros(n, bool)
    ce = np.full(top1.shape[0], NEG_INF, FLOAT)
    ok = top1 >= 0
    if ok.any():
        ce[ok] = cosine_rows(np.asarray(K_cur)[ok], np.asarray(K_cache)[top1[ok]])
        hit = ok.copy()
        hit[ok] = ce[ok] >= tau
        e[top1[hit]] = True
    return e, ce


def compact_plan(evict, n: int, nq: int, M: int):
    """The post-step cache order.

    Survivors (old entries with e_j = 0) in age order, then the nq current entries in
    token order; while longer than M, drop from the front (oldest).  Returns
    (index_map int64 [M], length): index_map[s] = j for an old entry, n + i for the
    current token i, -1 for s >= length.
    """
    if M < nq:
        raise CapacityError(f"M={M} < Nq={nq}")
    ev = np.asarray(evict, bool)[:n]
    order = np.concatenate([np.flatnonzero(~ev), n + np.arange(nq)]).astype(np.int64)
    if order.shape[0] > M:
        order = order[order.shape[0] - M:]
    imap = np.full(M, -1, np.int64)
    imap[: order.shape[0]] = order
    return imap, int(order.shape[0])


def gather_rows(index_map, length: int, old_rows, cur_rows) -> np.ndarray:
    """Rows of the compacted cache: old_rows[j] for j < n, cur_rows[j - n] otherwise."""
    old = np.asarray(old_rows)
    cur = np.asarray(cur_rows)
    n = old.shape[0]
    src = np.asarray(index_map, np.int64)[:length]
    out = np.empty((length,) + cur.shape[1:], dtype=np.result_type(old, cur))
    is_old = src < n
    out[is_old] = old[src[is_old]]
    out[~is_old] = cur[src[~is_old] - n]
    return out


# ----------------------------------------------------------------------------------
# the merge variant (technical summary §2.A, Theoretical Basis: Lemma 5.1)
# ----------------------------------------------------------------------------------
# Every cache entry stands for a group of g >= 1 keys.  When current entry i evicts
# cached entry j (its top-1 match with cos(kcur_i, k_j) >= tau), j is not dropped but
# folded into i: i's value becomes the mean over both groups and its count their sum;
# i's key stays (the most recent representative).  Attention gives every entry the
# logit q.k*scale + ln g.  Readings: a cached entry evicted by several current entries
# is folded into the lowest such i only (every other i keeps g = 1 and its own value);
# the FIFO cap drops the oldest entries with their whole groups.

def evict_owner(top1, cos_evict, tau: float, n: int) -> np.ndarray:
    """owner[j] = the lowest current index i with top1[i] = j and cos_evict[i] >= tau,
    -1 when no current entry evicts j.  int64 [n].  owner[j] >= 0 iff e_j = 1."""
    top1 = np.asarray(top1, np.int64)
    ce = _f64(cos_evict)
    owner = np.full(n, -1, np.int64)
    for i in range(top1.shape[0] - 1, -1, -1):     # descending, so the lowest i wins
        j = int(top1[i])
        if j >= 0 and ce[i] >= tau:
            owner[j] = i
    return owner


def merge_current(owner, top1, v_cur, cache_v, g_cache):
    """Value and count of each current entry after it absorbs the entry it owns.

    For current i, with j = top1[i] if owner[j] == i:
        g_i = 1 + g_j,   v_i <- (v_i + g_j * v_j) / g_i      (mean over both groups)
    otherwise g_i = 1 and v_i is unchanged.  Returns (v [nq, dv], g int64 [nq])."""
    owner = np.asarray(owner, np.int64)
    top1 = np.asarray(top1, np.int64)
    v = _f64(v_cur).copy()
    cv = _f64(cache_v)
    gc = np.asarray(g_cache, np.int64)
    g = np.ones(v.shape[0], np.int64)
    for i in range(v.shape[0]):
        j = int(top1[i])
        if j >= 0 and owner[j] == i:
            g[i] = 1 + gc[j]
            v[i] = (v[i] + gc[j] * cv[j]) / g[i]
    return v, g


def compact_merge(evict, owner, top1, cache_k, cache_v, g_cache, k_cur, v_cur, M: int):
    """The merge variant of the compaction: the plan of `compact_plan` (survivors in
    age order, then the current chunk, oldest dropped past M), with each current
    entry's value and count taken from `merge_current`.
    Returns (new_k, new_v, new_g int64, index_map, length)."""
    n, nq = np.asarray(cache_k).shape[0], np.asarray(k_cur).shape[0]
    imap, length = compact_plan(evict, n, nq, M)
    v_m, g_m = merge_current(owner, top1, v_cur, cache_v, g_cache)
    new_k = gather_rows(imap, length, cache_k, k_cur)
    new_v = gather_rows(imap, length, _f64(cache_v), v_m)
    new_g = gather_rows(imap, length, np.asarray(g_cache, np.int64), g_m)
    return new_k, new_v, new_g, imap, length


# ----------------------------------------------------------------------------------
# attention (AnnSA §2.C, AnnCA §2.B, dense baseline)
# ----------------------------------------------------------------------------------

def masked_softmax_attention(Q, K, V, allowed, scale: float, log_g=None):
    """o_i = sum_{s allowed} softmax_s(q_i.k_s * scale + log_g[s]) v_s, max-subtracted.

    allowed: bool [nq, nk] (None = all).  log_g: [nk] per-key logit shift (None = 0;
    the merge variant passes ln g, -inf for an empty group).  A row with nothing
    allowed gets o = 0 and lse = -inf.  Returns (O [nq, dv], lse [nq]) with
    lse = log sum exp(logits)."""
    Q = _f64(Q)
    K = _f64(K)
    V = _f64(V)
    nq, nk = Q.shape[0], K.shape[0]
    O = np.zeros((nq, V.shape[1]), FLOAT)
    lse = np.full(nq, NEG_INF, FLOAT)
    if nk == 0 or nq == 0:
        return O, lse
    step = max(1, (1 << 24) // max(nk, 1))           # row blocks bound the memory
    for a in range(0, nq, step):
        b = min(nq, a + step)
        S = (Q[a:b] @ K.T) * scale
        if log_g is not None:
            S = S + _f64(log_g)[None, :]
        if allowed is not None:
            S = np.where(allowed[a:b], S, NEG_INF)
        m = S.max(axis=1)
        live = np.isfinite(m)
        if not live.any():
            continue
        Pm = np.exp(S[live] - m[live, None])
        l = Pm.sum(axis=1)
        O[a:b][live] = (Pm @ V) / l[:, None]
        lse[a:b][live] = m[live] + np.log(l)
    return O, lse


def group_log(g) -> np.ndarray:
    """ln g per entry of the merge variant (-inf for g = 0: an empty group)."""
    g = _f64(g)
    out = np.full(g.shape, NEG_INF, FLOAT)
    np.log(g, out=out, where=g > 0)
    return out


def annsa_attention(Q, R, K, V, kb, scale: float, g=None):
    """Bucket-restricted self-attention: query i sees the keys s with kb[s] in R(i).

    Q [nq, d]; R [nq, r]; K, V [L, d] (the post-compaction cache, which holds the
    current chunk); kb [L]; g [L] the group counts of the merge variant (None: every
    entry is one key).  Returns (O, lse, n_empty)."""
    R = np.asarray(R, np.int64)
    kb = np.asarray(kb, np.int64)
    allowed = (kb[None, :, None] == R[:, None, :]).any(axis=2)
    O, lse = masked_softmax_attention(Q, K, V, allowed, scale, None if g is None else group_log(g))
    return O, lse, int((~allowed.any(axis=1)).sum())


def dense_attention(Q, K, V, scale: float, g=None):
    """Full softmax attention (the dense baseline); with group counts g, the dense
    attention over a merged cache."""
    return masked_softmax_attention(Q, K, V, None, scale, None if g is None else group_log(g))


def annca_select(Q, R, Kp, pb, F: int, Tf: int, tau_ca: float, topk: int, gate: bool = True):
    """Frame-relevant prompt tokens (technical summary §2.B).

    For frame f (queries i in [f*Tf, (f+1)*Tf)) and prompt token p:
      score[f, p] = max over the frame's queries i with pb[p] in R(i) of cos(q_i, kp_p)
                    (gate=False drops the bucket condition); -inf if there is none.
      rank = position in the order (score desc, p asc), -inf after every finite score.
      keep[f, p] = score >= tau_ca  or  rank < min(topk, P).
    Returns (keep bool [F, P], kidx list of int64 arrays (kept p ascending),
             kcnt int64 [F], score [F, P])."""
    Kp = _f64(Kp)
    P = Kp.shape[0]
    R = np.asarray(R, np.int64)
    pb = np.asarray(pb, np.int64)
    score = np.full((F, P), NEG_INF, FLOAT)
    keep = np.zeros((F, P), bool)
    kidx, kcnt = [], np.zeros(F, np.int64)
    for f in range(F):
        Qf = _f64(Q)[f * Tf:(f + 1) * Tf]
        if P > 0 and Qf.shape[0] > 0:
            Cf = cosine_matrix(Qf, Kp)
            if gate:
                shared = (R[f * Tf:(f + 1) * Tf, :, None] == pb[None, None, :]).any(axis=1)
                Cf = np.where(shared, Cf, NEG_INF)
            score[f] = Cf.max(axis=0)
        order = order_desc(score[f])
        rank = np.empty(P, np.int64)
        rank[order] = np.arange(P)
        keep[f] = (score[f] >= tau_ca) | (rank < min(topk, P))
        idx = np.flatnonzero(keep[f]).astype(np.int64)
        kidx.append(idx)
        kcnt[f] = idx.shape[0]
    return keep, kidx, kcnt, score


def cross_attention_subset(Q, Kp, Vp, kidx, F: int, Tf: int, scale: float):
    """Cross-attention of each frame's queries over its kept prompt tokens only."""
    Q = _f64(Q)
    O = np.zeros((Q.shape[0], np.asarray(Vp).shape[1]), FLOAT)
    lse = np.full(Q.shape[0], NEG_INF, FLOAT)
    for f in range(F):
        idx = np.asarray(kidx[f], np.int64)
        o, l = masked_softmax_attention(Q[f * Tf:(f + 1) * Tf], _f64(Kp)[idx], _f64(Vp)[idx], None, scale)
        O[f * Tf:(f + 1) * Tf] = o
        lse[f * Tf:(f + 1) * Tf] = l
    return O, lse


# ----------------------------------------------------------------------------------
# one head, one chunk
# ----------------------------------------------------------------------------------

def head_step(q, k_cur, v_cur, cache_k, cache_v, C, kp, vp, *, F, Tf, tau, M, r, tau_ca,
              topk, scale, gate=True, decisions=None, merge=False, g_cache=None):
    """The whole per-chunk step for one head.

    cache_k/cache_v [n, d]: the cache entering the step, oldest first.
    decisions: optional dict of discrete choices to take instead of the oracle's own
    (keys 'qb', 'kb_cur', 'kb_cache', 'pb', 'top1', 'evict', 'owner', 'keep'); the
    tests use it only with choices they have first checked to be valid alternatives
    (near-ties).
    merge: the Lemma 5.1 variant (evicted entries fold into their owner; attention
    with a ln g logit shift); g_cache [n] the incoming group counts (None: all 1).
    Returns a dict of every intermediate and output.
    """
    dec = decisions or {}
    n, nq = np.asarray(cache_k).shape[0], np.asarray(q).shape[0]
    qb = dec.get("qb")
    qb = query_buckets(q, C, r) if qb is None else np.asarray(qb, np.int64)
    kb_cur = dec.get("kb_cur")
    kb_cur = key_buckets(k_cur, C) if kb_cur is None else np.asarray(kb_cur, np.int64)
    kb_cache = dec.get("kb_cache")
    kb_cache = key_buckets(cache_k, C) if kb_cache is None else np.asarray(kb_cache, np.int64)
    pb = dec.get("pb")
    pb = key_buckets(kp, C) if pb is None else np.asarray(pb, np.int64)

    top1, s1, s2 = tempcache_match(q, cache_k)
    if dec.get("top1") is not None:
        top1 = np.asarray(dec["top1"], np.int64)
    evict, cos_evict = evict_flags(top1, k_cur, cache_k, tau)
    if dec.get("evict") is not None:
        evict = np.asarray(dec["evict"], bool)
    owner, new_g = None, None
    if merge:
        owner = evict_owner(top1, cos_evict, tau, n)
        if dec.get("owner") is not None:
            owner = np.asarray(dec["owner"], np.int64)
        gc = np.ones(n, np.int64) if g_cache is None else np.asarray(g_cache, np.int64)
        new_k, new_v, new_g, imap, length = compact_merge(evict, owner, top1, cache_k, cache_v, gc, k_cur,
                                                          v_cur, M)
    else:
        imap, length = compact_plan(evict, n, nq, M)
        new_k = gather_rows(imap, length, cache_k, k_cur)
        new_v = gather_rows(imap, length, cache_v, v_cur)
    new_kb = gather_rows(imap, length, kb_cache, kb_cur)

    o_self, lse_self, n_empty = annsa_attention(q, qb, new_k, new_v, new_kb, scale, new_g)

    keep, kidx, kcnt, score = annca_select(q, qb, kp, pb, F, Tf, tau_ca, topk, gate)
    if dec.get("keep") is not None:
        keep = np.asarray(dec["keep"], bool)
        kidx = [np.flatnonzero(keep[f]).astype(np.int64) for f in range(F)]
        kcnt = np.array([len(x) for x in kidx], np.int64)
    o_cross, lse_cross = cross_attention_subset(q, kp, vp, kidx, F, Tf, scale)

    return dict(qb=qb, kb_cur=kb_cur, kb_cache=kb_cache, pb=pb, top1=top1, s1=s1, s2=s2,
                cos_evict=cos_evict, evict=evict, owner=owner, new_g=new_g, index_map=imap, length=length,
                new_k=new_k, new_v=new_v, new_kb=new_kb, o_self=o_self, lse_self=lse_self,
                n_empty=n_empty, keep=keep, kidx=kidx, kcnt=kcnt, score=score,
                o_cross=o_cross, lse_cross=lse_cross)


def head_dense_step(q, history_k, history_v, k_cur, v_cur, kp, vp, scale):
    """The dense baseline for one head: attention over every past key plus the
    current chunk (append-only cache), and cross-attention over the whole prompt."""
    K = np.concatenate([_f64(history_k), _f64(k_cur)], axis=0)
    V = np.concatenate([_f64(history_v), _f64(v_cur)], axis=0)
    o_self, lse_self = dense_attention(q, K, V, scale)
    o_cross, lse_cross = dense_attention(q, kp, vp, scale)
    return dict(o_self=o_self, lse_self=lse_self, o_cross=o_cross, lse_cross=lse_cross)


def tempcache_only_advance(q, k_cur, v_cur, cache_k, cache_v, *, tau, M):
    """The TempCache part alone (match, evict, compact): advances a cache by one chunk.
    Used to warm a cache through earlier chunks.  Returns (new_k, new_v, info)."""
    top1, _, _ = tempcache_match(q, cache_k)
    evict, _ = evict_flags(top1, k_cur, cache_k, tau)
    imap, length = compact_plan(evict, np.asarray(cache_k).shape[0], np.asarray(q).shape[0], M)
    return (gather_rows(imap, length, cache_k, k_cur), gather_rows(imap, length, cache_v, v_cur),
            dict(evicted=int(evict.sum()), length=length, index_map=imap))
