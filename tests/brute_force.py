"""Exhaustive, loop-by-loop restatement of the FAST-AR step for tiny inputs.

Pure Python floats (double precision), explicit loops, no vectorisation and no code
shared with the oracle: every decision is taken by enumerating all candidates, the
compaction is simulated on a Python list, and attention is formed from an explicit
mask matrix.  Used to pin the oracle on 64-token inputs.
"""
import math


def dot(a, b):
    s = 0.0
    for x, y in zip(a, b):
        s += float(x) * float(y)
    return s


def norm(a):
    return math.sqrt(dot(a, a))


def cos(a, b):
    na, nb = norm(a), norm(b)
    if na == 0.0 or nb == 0.0:
        return 0.0
    return dot(a, b) / (na * nb)


def sorted_desc(scores):
    """Indices sorted by (score desc, index asc), by sorting explicit tuples."""
    return [i for _, i in sorted(((-s, i) for i, s in enumerate(scores)))]


def argmax_first(scores):
    best, arg = None, -1
    for i, s in enumerate(scores):
        if best is None or s > best:
            best, arg = s, i
    return arg


def step(q, k_cur, v_cur, cache_k, cache_v, C, kp, vp, *, F, Tf, tau, M, r, tau_ca, topk, scale):
    nq, n, P, B = len(q), len(cache_k), len(kp), len(C)
    # buckets
    kbucket = lambda x: argmax_first([dot(c, x) for c in C])
    qb = [sorted_desc([dot(c, x) for c in C])[:r] for x in q]
    kb_cur = [kbucket(x) for x in k_cur]
    kb_cache = [kbucket(x) for x in cache_k]
    pb = [kbucket(x) for x in kp]
    # match over every pair
    top1 = []
    for i in range(nq):
        top1.append(argmax_first([cos(q[i], cache_k[j]) for j in range(n)]) if n else -1)
    # evict
    evict = [False] * n
    for i in range(nq):
        j = top1[i]
        if j >= 0 and cos(k_cur[i], cache_k[j]) >= tau:
            evict[j] = True
    # compaction simulated on a list
    entries = []
    for j in range(n):
        if not evict[j]:
            entries.append(("old", j))
    for i in range(nq):
        entries.append(("cur", i))
    while len(entries) > M:
        entries.pop(0)
    index_map = [(j if kind == "old" else n + j) for kind, j in entries] + [-1] * (M - len(entries))
    ck = [cache_k[j] if kind == "old" else k_cur[j] for kind, j in entries]
    cv = [cache_v[j] if kind == "old" else v_cur[j] for kind, j in entries]
    cb = [kb_cache[j] if kind == "old" else kb_cur[j] for kind, j in entries]
    L = len(entries)
    # bucket-restricted attention from a mask matrix
    mask = [[cb[s] in qb[i] for s in range(L)] for i in range(nq)]

    def attend(qi, keys, vals, allowed):
        sc = [dot(qi, keys[s]) * scale if allowed[s] else -math.inf for s in range(len(keys))]
        m = max(sc) if sc else -math.inf
        if m == -math.inf:
            return [0.0] * len(vals[0] if vals else qi)
        w = [math.exp(x - m) if x != -math.inf else 0.0 for x in sc]
        z = sum(w)
        dv = len(vals[0])
        return [sum(w[s] * float(vals[s][c]) for s in range(len(vals))) / z for c in range(dv)]

    o_self = [attend(q[i], ck, cv, mask[i]) for i in range(nq)]
    # AnnCA by enumeration
    keep = []
    for f in range(F):
        sc = []
        for p in range(P):
            best = -math.inf
            for i in range(f * Tf, (f + 1) * Tf):
                if pb[p] in qb[i]:
                    best = max(best, cos(q[i], kp[p]))
            sc.append(best)
        order = sorted_desc(sc)
        rank = [0] * P
        for pos, p in enumerate(order):
            rank[p] = pos
        keep.append([sc[p] >= tau_ca or rank[p] < min(topk, P) for p in range(P)])
    o_cross = []
    for i in range(nq):
        f = i // Tf
        idx = [p for p in range(P) if keep[f][p]]
        o_cross.append(attend(q[i], [kp[p] for p in idx], [vp[p] for p in idx], [True] * len(idx)))
    return dict(qb=qb, kb_cur=kb_cur, kb_cache=kb_cache, pb=pb, top1=top1, evict=evict,
                index_map=index_map, length=L, o_self=o_self, keep=keep, o_cross=o_cross)


def ann_match(q, R, cache_k, kb):
    """Bucket-restricted top-1 by enumeration: for each query, every cached key whose
    bucket is one of the query's buckets is scored by cosine; the first (oldest) key
    with the largest score wins; (-1, -inf) when no key qualifies."""
    top1, s1 = [], []
    for i in range(len(q)):
        best_j, best = -1, float("-inf")
        for j in range(len(cache_k)):
            if kb[j] not in list(R[i]):
                continue
            c = cos(q[i], cache_k[j])
            if best_j < 0 or c > best:
                best_j, best = j, c
        top1.append(best_j)
        s1.append(best)
    return top1, s1


def merge_step(q, k_cur, v_cur, cache, *, tau, M):
    """The merge variant of one TempCache step by enumeration.

    cache: list of entries [k, v, g] (oldest first).  Every query is matched over all
    cached keys (first maximum), an entry is evicted when a query whose top-1 it is
    has cos(kcur_i, k_j) >= tau, and it is folded into the FIRST such query's entry:
    that entry's value becomes the count-weighted mean and its count the sum.  The new
    cache is the survivors then the current entries, oldest dropped past M.
    Returns (new cache, top1, owner)."""
    nq, n = len(q), len(cache)
    top1 = [argmax_first([cos(q[i], cache[j][0]) for j in range(n)]) if n else -1 for i in range(nq)]
    owner = [-1] * n
    for i in range(nq):
        j = top1[i]
        if j >= 0 and owner[j] < 0 and cos(k_cur[i], cache[j][0]) >= tau:
            owner[j] = i
    cur = []
    for i in range(nq):
        k, v, g = list(k_cur[i]), [float(x) for x in v_cur[i]], 1
        j = top1[i]
        if j >= 0 and owner[j] == i:
            gj = cache[j][2]
            v = [(v[c] + gj * float(cache[j][1][c])) / (1 + gj) for c in range(len(v))]
            g = 1 + gj
        cur.append([k, v, g])
    new = [cache[j] for j in range(n) if owner[j] < 0] + cur
    while len(new) > M:
        new.pop(0)
    return new, top1, owner


def grouped_attention(qi, entries, scale):
    """Attention of one query over entries [k, v, g], each weighted by its count:
    w_s = g_s * exp(q.k_s * scale - m)."""
    if not entries:
        return [0.0] * len(qi)
    sc = [dot(qi, e[0]) * scale for e in entries]
    m = max(sc)
    w = [e[2] * math.exp(x - m) for e, x in zip(entries, sc)]
    z = sum(w)
    dv = len(entries[0][1])
    return [sum(w[s] * float(entries[s][1][c]) for s in range(len(entries))) / z for c in range(dv)]


def pq_encode(X, codebooks):
    """Nearest codeword per sub-space by enumerating every codeword's squared distance."""
    m, Kc, ds = len(codebooks), len(codebooks[0]), len(codebooks[0][0])
    out = []
    for x in X:
        row = []
        for s in range(m):
            best, arg = None, -1
            for c in range(Kc):
                dist = 0.0
                for t in range(ds):
                    diff = float(x[s * ds + t]) - float(codebooks[s][c][t])
                    dist += diff * diff
                if best is None or dist < best:
                    best, arg = dist, c
            row.append(arg)
        out.append(row)
    return out


def pq_match(q, codes, codebooks):
    """Top-1 over the decoded cached keys by enumeration (first maximum of the cosine)."""
    ds = len(codebooks[0][0])
    dec = [[float(codebooks[s][cd][t]) for s, cd in enumerate(row) for t in range(ds)] for row in codes]
    top1 = []
    for qi in q:
        top1.append(argmax_first([cos(qi, k) for k in dec]) if dec else -1)
    return top1
