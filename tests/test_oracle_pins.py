"""Pins of the CPU oracle against things other than itself: hand-worked closed forms,
a library attention routine, exhaustive enumeration, exact ties and invariants the
definitions fix.  CPU only."""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import fastar_oracle as O
import brute_force

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as fh:
        return json.load(fh)


def _ev(x):
    if isinstance(x, str):
        return float(eval(x, {"__builtins__": {}}, {"sqrt": math.sqrt, "inf": math.inf}))
    return float(x)


# ----------------------------------------------------------------------------------
# hand-worked cases
# ----------------------------------------------------------------------------------

def test_golden_tempcache_2d():
    g = _load("tempcache_2d.json")
    top1, s1, s2 = O.tempcache_match(g["q"], g["cache_k"])
    assert top1.tolist() == g["top1"]
    np.testing.assert_allclose(s1, [_ev(x) for x in g["s1"]], rtol=0, atol=1e-12)
    np.testing.assert_allclose(s2, [_ev(x) for x in g["s2"]], rtol=0, atol=1e-12)
    e, ce = O.evict_flags(top1, g["k_cur"], g["cache_k"], g["tau"])
    np.testing.assert_allclose(ce, [_ev(x) for x in g["cos_evict"]], rtol=0, atol=1e-12)
    assert e.astype(int).tolist() == g["evict"]
    imap, L = O.compact_plan(e, len(g["cache_k"]), len(g["q"]), g["M"])
    assert L == g["length"]
    assert imap[:L].tolist() == g["index_map"]


def test_golden_buckets_2d():
    g = _load("buckets_2d.json")
    assert O.key_buckets(g["keys"], g["C"]).tolist() == g["key_buckets"]
    assert O.query_buckets(g["queries"], g["C"], g["r"]).tolist() == g["query_buckets"]


def test_golden_annca_2d():
    g = _load("annca_2d.json")
    R = O.query_buckets(g["q"], g["C"], g["r"])
    pb = O.key_buckets(g["kp"], g["C"])
    assert pb.tolist() == g["pb"]
    for case in g["cases"]:
        keep, kidx, kcnt, score = O.annca_select(g["q"], R, g["kp"], pb, g["F"], g["Tf"],
                                                 case["tau_ca"], case["topk"])
        want = np.array([[_ev(x) for x in row] for row in g["score"]])
        assert np.array_equal(np.isinf(score), np.isinf(want))
        fin = np.isfinite(want)
        np.testing.assert_allclose(score[fin], want[fin], rtol=0, atol=1e-12)
        assert keep.astype(int).tolist() == case["keep"]
        for f in range(g["F"]):
            assert kidx[f].tolist() == [p for p in range(len(g["kp"])) if case["keep"][f][p]]
            assert kcnt[f] == sum(case["keep"][f])


def test_attention_two_key_closed_form():
    # q=(1,0), k0=(1,0), k1=(0,1), scale 1/sqrt2: scores a=1/sqrt2 and 0.
    a = 1 / math.sqrt(2)
    o, lse = O.dense_attention([[1, 0]], [[1, 0], [0, 1]], [[1, 0], [0, 1]], 1 / math.sqrt(2))
    z = math.exp(a) + 1
    np.testing.assert_allclose(o[0], [math.exp(a) / z, 1 / z], rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse[0], math.log(z), rtol=0, atol=1e-14)
    # a third key outside the query's buckets changes nothing
    o2, lse2, _ = O.annsa_attention([[1, 0]], [[0]], [[1, 0], [0, 1], [5, 5]],
                                    [[1, 0], [0, 1], [100, 100]], [0, 0, 1], 1 / math.sqrt(2))
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse2, lse, rtol=0, atol=1e-14)


def test_attention_identical_keys_average_values():
    # g identical keys: every weight is 1/g, the output is the plain mean of the values.
    rng = np.random.default_rng(3)
    k = rng.standard_normal(8)
    V = rng.standard_normal((5, 8))
    o, lse = O.dense_attention(rng.standard_normal((2, 8)), np.tile(k, (5, 1)), V, 0.3)
    np.testing.assert_allclose(o, np.tile(V.mean(axis=0), (2, 1)), rtol=0, atol=1e-13)


def test_empty_bucket_gives_zero_row_and_neg_inf_lse():
    o, lse, n_empty = O.annsa_attention([[1.0, 2.0], [0.5, 0.5]], [[3], [0]], [[1.0, 0.0]], [[7.0, 7.0]],
                                        [0], 0.5)
    assert n_empty == 1
    assert np.all(o[0] == 0) and lse[0] == -np.inf
    np.testing.assert_allclose(o[1], [7.0, 7.0])


# ----------------------------------------------------------------------------------
# reduction to textbook attention (B=1, r=1, tau>1, tau_ca=-1, M >= n+Nq)
# ----------------------------------------------------------------------------------

def _rand_case(rng, n, nq, P, d, B, F=1):
    Tf = nq // F
    C = rng.standard_normal((B, d))
    C /= np.linalg.norm(C, axis=1, keepdims=True)
    return dict(q=rng.standard_normal((nq, d)), k_cur=rng.standard_normal((nq, d)),
                v_cur=rng.standard_normal((nq, d)), cache_k=rng.standard_normal((n, d)),
                cache_v=rng.standard_normal((n, d)), C=C, kp=rng.standard_normal((P, d)),
                vp=rng.standard_normal((P, d)), F=F, Tf=Tf)


@pytest.mark.parametrize("seed", [0, 1])
def test_textbook_reduction_matches_library_attention(seed):
    rng = np.random.default_rng(seed)
    n, nq, P, d = 40, 24, 20, 16
    c = _rand_case(rng, n, nq, P, d, B=1, F=2)
    scale = 1 / math.sqrt(d)
    out = O.head_step(c["q"], c["k_cur"], c["v_cur"], c["cache_k"], c["cache_v"], c["C"], c["kp"], c["vp"],
                      F=c["F"], Tf=c["Tf"], tau=2.0, M=n + nq, r=1, tau_ca=-1.0, topk=16, scale=scale)
    assert not out["evict"].any()
    assert out["length"] == n + nq
    assert out["index_map"].tolist() == list(range(n + nq))
    assert out["keep"].all()
    t = lambda x: torch.tensor(np.asarray(x), dtype=torch.float64)
    K = t(np.concatenate([c["cache_k"], c["k_cur"]]))
    V = t(np.concatenate([c["cache_v"], c["v_cur"]]))
    ref_self = torch.nn.functional.scaled_dot_product_attention(t(c["q"])[None], K[None], V[None], scale=scale)[0]
    ref_cross = torch.nn.functional.scaled_dot_product_attention(t(c["q"])[None], t(c["kp"])[None],
                                                                 t(c["vp"])[None], scale=scale)[0]
    np.testing.assert_allclose(out["o_self"], ref_self.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(out["o_cross"], ref_cross.numpy(), rtol=0, atol=1e-12)
    lse_ref = torch.logsumexp(t(c["q"]) @ K.T * scale, dim=1).numpy()
    np.testing.assert_allclose(out["lse_self"], lse_ref, rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------------
# convex hull of the query's own buckets
# ----------------------------------------------------------------------------------

def test_output_is_convex_combination_of_own_buckets():
    rng = np.random.default_rng(7)
    n, nq, d, B, r = 60, 20, 12, 6, 2
    C = rng.standard_normal((B, d))
    C /= np.linalg.norm(C, axis=1, keepdims=True)
    Q = rng.standard_normal((nq, d))
    K = rng.standard_normal((n, d))
    R = O.query_buckets(Q, C, r)
    kb = O.key_buckets(K, C)
    # one-hot value per bucket plus a uniform coordinate: mass may land only on R(i)
    V = np.zeros((n, B + 1))
    V[np.arange(n), kb] = 1.0
    V[:, B] = rng.uniform(0, 1, n)
    o, _, _ = O.annsa_attention(Q, R, K, V, kb, 0.25)
    for i in range(nq):
        outside = np.setdiff1d(np.arange(B), R[i])
        assert np.all(o[i, outside] == 0.0)
        if np.isin(kb, R[i]).any():
            np.testing.assert_allclose(o[i, :B].sum(), 1.0, rtol=0, atol=1e-12)
        assert 0.0 <= o[i, B] <= 1.0
    # sentinel form: keys outside R(q_0) carry 1e3, inside U[0,1]
    inside = np.isin(kb, R[0])
    Vs = np.where(inside[:, None], rng.uniform(0, 1, (n, 4)), 1e3)
    o0, _, _ = O.annsa_attention(Q[:1], R[:1], K, Vs, kb, 0.25)
    assert np.all((o0 >= 0) & (o0 <= 1))


# ----------------------------------------------------------------------------------
# cache cap over a rollout
# ----------------------------------------------------------------------------------

@pytest.mark.parametrize("M", [16, 40, 64])
def test_cache_length_law_over_rollout(M):
    rng = np.random.default_rng(11)
    nq, d = 16, 8
    base = rng.standard_normal((nq, d))
    ck = np.zeros((0, d))
    cv = np.zeros((0, d))
    for t in range(12):
        k_cur = base + 0.05 * t * rng.standard_normal((nq, d))
        q = k_cur + 0.1 * rng.standard_normal((nq, d))
        top1, _, _ = O.tempcache_match(q, ck)
        e, _ = O.evict_flags(top1, k_cur, ck, 0.9)
        imap, L = O.compact_plan(e, ck.shape[0], nq, M)
        assert L == min(M, ck.shape[0] - int(e.sum()) + nq)
        assert L <= M
        ck2, cv2, info = O.tempcache_only_advance(q, k_cur, k_cur * 2, ck, cv, tau=0.9, M=M)
        assert info["length"] == L and info["evicted"] == int(e.sum())
        ck, cv = ck2, cv2
        # the newest chunk is always the tail of the cache
        np.testing.assert_array_equal(ck[-nq:], k_cur)


def test_capacity_error():
    with pytest.raises(O.CapacityError):
        O.compact_plan(np.zeros(4, bool), 4, 10, 8)


# ----------------------------------------------------------------------------------
# permutation invariance
# ----------------------------------------------------------------------------------

def test_permutation_invariance():
    rng = np.random.default_rng(5)
    n, nq, P, d, B = 48, 16, 24, 8, 4
    c = _rand_case(rng, n, nq, P, d, B=B, F=1)
    kw = dict(F=1, Tf=nq, tau=0.8, M=n + nq, r=2, tau_ca=0.3, topk=4, scale=1 / math.sqrt(d))
    base = O.head_step(c["q"], c["k_cur"], c["v_cur"], c["cache_k"], c["cache_v"], c["C"], c["kp"], c["vp"], **kw)
    pi = rng.permutation(nq)
    pq = O.head_step(c["q"][pi], c["k_cur"][pi], c["v_cur"][pi], c["cache_k"], c["cache_v"], c["C"], c["kp"],
                     c["vp"], **kw)
    np.testing.assert_allclose(pq["o_self"], base["o_self"][pi], rtol=0, atol=1e-12)
    np.testing.assert_allclose(pq["o_cross"], base["o_cross"][pi], rtol=0, atol=1e-12)
    sigma = rng.permutation(n)
    pc = O.head_step(c["q"], c["k_cur"], c["v_cur"], c["cache_k"][sigma], c["cache_v"][sigma], c["C"], c["kp"],
                     c["vp"], **kw)
    assert pc["evict"].sum() == base["evict"].sum()
    np.testing.assert_allclose(pc["o_self"], base["o_self"], rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------------
# exhaustive enumeration on 64-token inputs
# ----------------------------------------------------------------------------------

@pytest.mark.parametrize("seed", [0, 1, 2])
def test_matches_exhaustive_enumeration(seed):
    rng = np.random.default_rng(100 + seed)
    n, nq, P, d, B, r = 48, 16, 24, 8, 4, 2
    F, Tf = 2, 8
    # drifting keys so that some entries are evicted and the FIFO drops some
    ck = rng.standard_normal((n, d))
    k_cur = ck[-nq:] + 0.05 * rng.standard_normal((nq, d))
    q = k_cur + 0.1 * rng.standard_normal((nq, d))
    cv = rng.standard_normal((n, d))
    v_cur = rng.standard_normal((nq, d))
    C = rng.standard_normal((B, d))
    C /= np.linalg.norm(C, axis=1, keepdims=True)
    kp = rng.standard_normal((P, d)) / math.sqrt(d)
    vp = rng.standard_normal((P, d))
    kw = dict(F=F, Tf=Tf, tau=0.95, M=56, r=r, tau_ca=0.4, topk=5, scale=1 / math.sqrt(d))
    got = O.head_step(q, k_cur, v_cur, ck, cv, C, kp, vp, **kw)
    want = brute_force.step(q.tolist(), k_cur.tolist(), v_cur.tolist(), ck.tolist(), cv.tolist(), C.tolist(),
                            kp.tolist(), vp.tolist(), **kw)
    assert got["evict"].sum() > 0, "case should exercise eviction"
    for key in ("kb_cur", "kb_cache", "pb", "top1"):
        assert got[key].tolist() == want[key], key
    assert got["qb"].tolist() == want["qb"]
    assert got["evict"].tolist() == want["evict"]
    assert got["index_map"].tolist() == want["index_map"]
    assert got["length"] == want["length"]
    assert got["keep"].tolist() == want["keep"]
    np.testing.assert_allclose(got["o_self"], np.array(want["o_self"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(got["o_cross"], np.array(want["o_cross"]), rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------------
# exact ties and duplicate eviction
# ----------------------------------------------------------------------------------

def test_exact_ties_take_lowest_index():
    # integer-valued duplicated keys: cosines tie exactly
    ck = np.array([[1, 2, 0, 0], [3, 0, 1, 0], [1, 2, 0, 0], [2, 4, 0, 0], [3, 0, 1, 0]], float)
    q = np.array([[1, 2, 0, 0], [3, 0, 1, 0], [0, 0, 0, 1]], float)
    top1, s1, s2 = O.tempcache_match(q, ck)
    assert top1.tolist() == [0, 1, 0]
    assert s1[0] == s2[0] and abs(s1[0] - 1.0) < 1e-15   # k0, k2, k3 tie exactly
    # duplicated centroids: argmax and the top-r order go to the lower index
    C = np.array([[1, 0, 0, 0], [0, 1, 0, 0], [1, 0, 0, 0], [0, 1, 0, 0]], float)
    assert O.key_buckets([[2, 1, 0, 0], [1, 2, 0, 0], [1, 1, 0, 0]], C).tolist() == [0, 1, 0]
    assert O.query_buckets([[2, 1, 0, 0], [1, 1, 0, 0]], C, 3).tolist() == [[0, 2, 1], [0, 1, 2]]


def test_duplicate_current_key_evicts_matched_entry():
    rng = np.random.default_rng(2)
    ck = rng.standard_normal((10, 6))
    k_cur = ck[[3, 7]].copy()
    q = k_cur.copy()
    top1, _, _ = O.tempcache_match(q, ck)
    assert top1.tolist() == [3, 7]
    e, ce = O.evict_flags(top1, k_cur, ck, 0.999999)
    np.testing.assert_allclose(ce, [1.0, 1.0], rtol=0, atol=1e-14)
    assert np.flatnonzero(e).tolist() == [3, 7]
    # inclusive threshold: tau exactly equal to the cosine still evicts
    e2, _ = O.evict_flags([0], [[1.0, 0.0]], [[1.0, 0.0]], 1.0)
    assert e2.tolist() == [True]


def test_first_chunk_empty_cache():
    q = np.ones((4, 3))
    top1, s1, s2 = O.tempcache_match(q, np.zeros((0, 3)))
    assert top1.tolist() == [-1] * 4 and np.all(s1 == -np.inf)
    e, _ = O.evict_flags(top1, q, np.zeros((0, 3)), 0.5)
    imap, L = O.compact_plan(e, 0, 4, 6)
    assert L == 4 and imap.tolist() == [0, 1, 2, 3, -1, -1]


def test_annca_all_unmatched_keeps_first_topk_by_index():
    # no prompt token shares a bucket with any query: every score is -inf, the
    # always-keep rule keeps the topk lowest indices.
    C = np.eye(3)
    q = np.array([[1.0, 0, 0]] * 4)
    kp = np.array([[0, 1.0, 0]] * 10)
    R = O.query_buckets(q, C, 1)
    pb = O.key_buckets(kp, C)
    keep, kidx, kcnt, score = O.annca_select(q, R, kp, pb, 1, 4, 0.1, 3)
    assert np.all(score == -np.inf)
    assert kidx[0].tolist() == [0, 1, 2] and kcnt.tolist() == [3]
    # ungated: every token has a finite (zero) cosine and only topk are kept
    keep2, kidx2, _, score2 = O.annca_select(q, R, kp, pb, 1, 4, 0.1, 3, gate=False)
    assert np.all(score2 == 0.0) and kidx2[0].tolist() == [0, 1, 2]


# ----------------------------------------------------------------------------------
# planted mistakes: each pin above must catch a slip of the kind it targets
# ----------------------------------------------------------------------------------

def test_pins_catch_planted_mistakes(monkeypatch):
    g = _load("tempcache_2d.json")
    # (1) ties to the newest instead of the oldest
    monkeypatch.setattr(O, "tempcache_match", lambda Q, K: _newest_tie_match(Q, K))
    with pytest.raises(AssertionError):
        test_golden_tempcache_2d()
    monkeypatch.undo()
    # (2) an exclusive threshold
    real = O.evict_flags

    def strict(top1, kc, ck, tau):
        e, ce = real(top1, kc, ck, tau)
        return (e & False) | _strict_evict(top1, ce, len(ck), tau), ce
    monkeypatch.setattr(O, "evict_flags", strict)
    with pytest.raises(AssertionError):
        test_duplicate_current_key_evicts_matched_entry()
    monkeypatch.undo()
    # (3) FIFO drop from the back instead of the front
    real_plan = O.compact_plan

    def back_drop(e, n, nq, M):
        order = np.concatenate([np.flatnonzero(~np.asarray(e, bool)[:n]), n + np.arange(nq)])[:M]
        imap = np.full(M, -1, np.int64)
        imap[:len(order)] = order
        return imap, len(order)
    monkeypatch.setattr(O, "compact_plan", back_drop)
    with pytest.raises(AssertionError):
        test_golden_tempcache_2d()
    monkeypatch.setattr(O, "compact_plan", real_plan)


def _newest_tie_match(Q, K):
    S = O.cosine_matrix(Q, K)
    n = S.shape[1]
    top1 = (n - 1 - np.argmax(S[:, ::-1], axis=1)).astype(np.int64)
    rows = np.arange(S.shape[0])
    s1 = S[rows, top1].copy()
    S[rows, top1] = -np.inf
    return top1, s1, S.max(axis=1)


def _strict_evict(top1, ce, n, tau):
    e = np.zeros(n, bool)
    for i, j in enumerate(np.asarray(top1)):
        if j >= 0 and ce[i] > tau:
            e[j] = True
    return e


def test_bucket_order_against_a_bucket_by_bucket_scan():
    # the grouping written out as loops: bucket 0's elements in ascending element id,
    # then bucket 1's, ...; offsets are where each bucket's run starts
    rng = np.random.default_rng(5)
    H, n, r, B = 3, 37, 2, 6
    ids = rng.integers(0, B, size=(H, n, r))
    n_valid = np.array([37, 20, 0])
    perm, off = O.bucket_order(ids, B, n_valid)
    for h in range(H):
        flat = [int(ids[h, i, s]) for i in range(int(n_valid[h])) for s in range(r)]
        want, starts = [], []
        for b in range(B):
            starts.append(len(want))
            want += [e for e, bb in enumerate(flat) if bb == b]
        assert perm[h, :len(want)].tolist() == want
        assert (perm[h, len(want):] == -1).all()
        assert off[h].tolist() == starts + [len(want)]
    # a plausible mistake, descending element ids inside each bucket, differs from it
    flat0 = ids[0].reshape(-1)
    bad = (flat0.size - 1) - np.argsort(flat0[::-1], kind="stable")
    assert np.array_equal(np.sort(bad), np.arange(flat0.size))
    assert bad.tolist() != perm[0, :flat0.size].tolist()


@pytest.mark.parametrize("seed", [0, 1])
def test_dense_baseline_step_matches_library_attention(seed):
    # the dense baseline is plain softmax attention over every past key plus the chunk,
    # and over the whole prompt: the library routine (float64) gives the same numbers
    rng = np.random.default_rng(seed)
    n_hist, nq, P, d = 57, 19, 13, 16
    q, k_cur, v_cur = rng.standard_normal((3, nq, d))
    hk, hv = rng.standard_normal((2, n_hist, d))
    kp, vp = rng.standard_normal((2, P, d))
    scale = 0.7 / math.sqrt(d)
    out = O.head_dense_step(q, hk, hv, k_cur, v_cur, kp, vp, scale)
    t = lambda x: torch.tensor(np.asarray(x), dtype=torch.float64)
    K, V = t(np.concatenate([hk, k_cur])), t(np.concatenate([hv, v_cur]))
    sdpa = torch.nn.functional.scaled_dot_product_attention
    np.testing.assert_allclose(out["o_self"], sdpa(t(q)[None], K[None], V[None], scale=scale)[0].numpy(),
                               rtol=0, atol=1e-12)
    np.testing.assert_allclose(out["o_cross"], sdpa(t(q)[None], t(kp)[None], t(vp)[None], scale=scale)[0].numpy(),
                               rtol=0, atol=1e-12)
    np.testing.assert_allclose(out["lse_self"], torch.logsumexp(t(q) @ K.T * scale, dim=1).numpy(), rtol=0,
                               atol=1e-12)
    np.testing.assert_allclose(out["lse_cross"], torch.logsumexp(t(q) @ t(kp).T * scale, dim=1).numpy(), rtol=0,
                               atol=1e-12)
    # a plausible mistake, the current chunk left out of the self-attention keys, differs
    miss, _ = O.dense_attention(q, hk, hv, scale)
    assert np.abs(miss - out["o_self"]).max() > 1e-3
