"""Pins of the merge variant of TempCache (technical summary §2.A, Theoretical Basis:
Lemma 5.1 — identical keys merge with no error when their values are averaged and
their logit is shifted by the group size).

The pins: the lemma's closed form against a plain softmax over the unmerged keys; a
rollout whose chunks re-send cached keys, whose merged cache must attend exactly like
the whole history; enumeration on tiny random cases (ties, several current entries
evicting one cached entry, the FIFO cap); the reduction to the replace step when
nothing is evicted; conservation of the group counts; and planted mistakes that the
pins must catch."""
import numpy as np
import pytest
from scipy.special import logsumexp, softmax

from oracle import fastar_oracle as O
import brute_force


def _plain_attention(Q, K, V, scale):
    """softmax(Q K^T * scale) V and its log-sum-exp, with SciPy's routines."""
    S = (Q @ K.T) * scale
    return softmax(S, axis=1) @ V, logsumexp(S, axis=1)


def _duplicates(seed, m=20, d=16, gmax=5, nq=12):
    rng = np.random.default_rng(500 + seed)
    Ku = rng.standard_normal((m, d))
    g = rng.integers(1, gmax + 1, m)
    rows = np.repeat(np.arange(m), g)
    Kx = Ku[rows]                       # every unique key g times
    Vx = rng.standard_normal((rows.shape[0], d))
    Vm = np.stack([Vx[rows == u].mean(axis=0) for u in range(m)])
    Q = rng.standard_normal((nq, d))
    return Q, Ku, g, Kx, Vx, Vm


def _pin_lemma(seed):
    Q, Ku, g, Kx, Vx, Vm = _duplicates(seed)
    scale = 1.0 / np.sqrt(Q.shape[1])
    want_o, want_l = _plain_attention(Q, Kx, Vx, scale)
    got_o, got_l = O.dense_attention(Q, Ku, Vm, scale, g=g)
    np.testing.assert_allclose(got_o, want_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(got_l, want_l, rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_lemma_exact_merge_of_duplicate_keys(seed):
    _pin_lemma(seed)


def test_lemma_holds_under_bucket_masks():
    # AnnSA with one bucket holding every key reduces to the dense merged attention
    Q, Ku, g, Kx, Vx, Vm = _duplicates(7)
    scale = 0.25
    R = np.zeros((Q.shape[0], 1), np.int64)
    o, lse, n_empty = O.annsa_attention(Q, R, Ku, Vm, np.zeros(Ku.shape[0], np.int64), scale, g=g)
    want_o, want_l = _plain_attention(Q, Kx, Vx, scale)
    assert n_empty == 0
    np.testing.assert_allclose(o, want_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, want_l, rtol=0, atol=1e-12)


def test_empty_group_contributes_nothing():
    rng = np.random.default_rng(3)
    Q, K, V = rng.standard_normal((4, 8)), rng.standard_normal((6, 8)), rng.standard_normal((6, 8))
    g = np.array([1, 0, 2, 1, 0, 3])
    keep = g > 0
    o, l = O.dense_attention(Q, K, V, 0.3, g=g)
    o2, l2 = O.dense_attention(Q, K[keep], V[keep], 0.3, g=g[keep])
    np.testing.assert_allclose(o, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l, l2, rtol=0, atol=1e-13)


def _merge_chunk(q, k_cur, v_cur, ck, cv, cg, tau, M):
    top1, _, _ = O.tempcache_match(q, ck)
    evict, ce = O.evict_flags(top1, k_cur, ck, tau)
    owner = O.evict_owner(top1, ce, tau, ck.shape[0])
    nk, nv, ng, imap, length = O.compact_merge(evict, owner, top1, ck, cv, cg, k_cur, v_cur, M)
    return nk, nv, ng, dict(top1=top1, evict=evict, owner=owner, imap=imap, length=length)


def _pin_rollout(seed, chunks=5, nq=10, d=16):
    """Chunks that re-send cached keys (query = key, so the match finds them) next to
    fresh keys; with no FIFO drop, the merged cache attends exactly like the whole
    history of keys and values."""
    rng = np.random.default_rng(900 + seed)
    tau, M = 0.999, 10_000
    ck, cv, cg = np.zeros((0, d)), np.zeros((0, d)), np.zeros(0, np.int64)
    hk, hv = [], []
    merged_any = doubled = False
    for t in range(chunks):
        k_cur = rng.standard_normal((nq, d))
        if t > 0:
            # re-send some cached keys; twice the same one in one chunk now and then
            pick = rng.choice(ck.shape[0], size=nq // 2, replace=False)
            if t % 2 == 0:
                pick[1] = pick[0]
                doubled = True
            k_cur[: nq // 2] = ck[pick]
        v_cur = rng.standard_normal((nq, d))
        q = k_cur.copy()
        ck, cv, cg, info = _merge_chunk(q, k_cur, v_cur, ck, cv, cg, tau, M)
        merged_any |= bool(info["evict"].any())
        hk.append(k_cur)
        hv.append(v_cur)
    assert merged_any and doubled
    assert cg.sum() == chunks * nq
    Kh, Vh = np.concatenate(hk), np.concatenate(hv)
    Qt = rng.standard_normal((8, d))
    want_o, want_l = _plain_attention(Qt, Kh, Vh, 0.2)
    got_o, got_l = O.dense_attention(Qt, ck, cv, 0.2, g=cg)
    np.testing.assert_allclose(got_o, want_o, rtol=0, atol=1e-10)
    np.testing.assert_allclose(got_l, want_l, rtol=0, atol=1e-10)


@pytest.mark.parametrize("seed", [0, 1])
def test_rollout_with_resent_keys_equals_full_history(seed):
    _pin_rollout(seed)


def _tiny(seed, n=14, nq=6, d=4):
    rng = np.random.default_rng(1300 + seed)
    ck = rng.standard_normal((n, d))
    cv = rng.standard_normal((n, d))
    cg = rng.integers(1, 4, n)
    # current keys near cached ones (several near the same one), queries near the keys
    src = rng.integers(0, n // 2, nq)
    k_cur = ck[src] + 0.15 * rng.standard_normal((nq, d))
    q = k_cur + 0.1 * rng.standard_normal((nq, d))
    v_cur = rng.standard_normal((nq, d))
    return q, k_cur, v_cur, ck, cv, cg


def _pin_enumeration(seed, M):
    q, k_cur, v_cur, ck, cv, cg = _tiny(seed)
    tau = 0.9
    nk, nv, ng, info = _merge_chunk(q, k_cur, v_cur, ck, cv, cg, tau, M)
    cache = [[list(ck[j]), list(cv[j]), int(cg[j])] for j in range(ck.shape[0])]
    new, top1, owner = brute_force.merge_step(q.tolist(), k_cur.tolist(), v_cur.tolist(), cache, tau=tau, M=M)
    assert info["top1"].tolist() == top1
    assert info["owner"].tolist() == owner
    assert info["length"] == len(new)
    np.testing.assert_allclose(nk, np.array([e[0] for e in new]), rtol=0, atol=0)
    np.testing.assert_allclose(nv, np.array([e[1] for e in new]), rtol=0, atol=1e-13)
    assert ng.tolist() == [e[2] for e in new]
    qt = np.random.default_rng(seed).standard_normal((3, ck.shape[1]))
    got, _ = O.dense_attention(qt, nk, nv, 0.5, g=ng)
    want = np.array([brute_force.grouped_attention(x.tolist(), new, 0.5) for x in qt])
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)
    return info


@pytest.mark.parametrize("seed", range(6))
def test_merge_step_equals_enumeration(seed):
    info = _pin_enumeration(seed, M=64)
    assert (info["owner"] >= 0).sum() == info["evict"].sum()


def test_enumeration_covers_a_shared_match_and_the_fifo_cap():
    shared = False
    for seed in range(6):
        info = _pin_enumeration(seed, M=12)      # 14 + 6 entries at most: the cap bites
        t = info["top1"][info["top1"] >= 0]
        ce_hits = np.isin(t, np.flatnonzero(info["evict"]))
        shared |= np.unique(t[ce_hits]).shape[0] < ce_hits.sum()
    assert shared, "no case had two current entries evicting one cached entry"


def test_owner_is_the_lowest_evicting_query():
    top1 = np.array([2, 0, 2, 2, -1])
    ce = np.array([0.5, 0.95, 0.97, 0.99, -np.inf])
    owner = O.evict_owner(top1, ce, 0.9, 4)
    assert owner.tolist() == [1, -1, 2, -1]       # query 0 does not evict (0.5 < 0.9)
    v, g = O.merge_current(owner, top1, np.ones((5, 2)), np.full((4, 2), 4.0), np.array([3, 1, 5, 1]))
    assert g.tolist() == [1, 4, 6, 1, 1]
    np.testing.assert_allclose(v[2], [(1 + 5 * 4.0) / 6] * 2)
    np.testing.assert_allclose(v[3], [1.0, 1.0])


def test_without_evictions_the_merge_step_is_the_replace_step():
    rng = np.random.default_rng(11)
    d, n, nq, B = 8, 30, 12, 4
    C = rng.standard_normal((B, d))
    C /= np.linalg.norm(C, axis=1, keepdims=True)
    args = [rng.standard_normal((nq, d)), rng.standard_normal((nq, d)), rng.standard_normal((nq, d)),
            rng.standard_normal((n, d)), rng.standard_normal((n, d)), C, rng.standard_normal((5, d)),
            rng.standard_normal((5, d))]
    kw = dict(F=2, Tf=6, M=36, r=2, tau_ca=0.5, topk=2, scale=0.35)
    a = O.head_step(*args, tau=1.5, **kw)
    b = O.head_step(*args, tau=1.5, merge=True, **kw)
    assert not b["evict"].any() and (b["new_g"] == 1).all()
    np.testing.assert_array_equal(a["index_map"], b["index_map"])
    np.testing.assert_allclose(b["o_self"], a["o_self"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(b["new_v"], a["new_v"], rtol=0, atol=0)


def test_merge_keeps_the_replace_order_and_conserves_counts():
    q, k_cur, v_cur, ck, cv, cg = _tiny(2)
    nk, nv, ng, info = _merge_chunk(q, k_cur, v_cur, ck, cv, cg, 0.9, 64)
    imap, length = O.compact_plan(info["evict"], ck.shape[0], q.shape[0], 64)
    np.testing.assert_array_equal(info["imap"], imap)
    np.testing.assert_array_equal(nk, O.gather_rows(imap, length, ck, k_cur))
    assert info["evict"].any()
    assert ng.sum() == cg.sum() + q.shape[0]                  # nothing dropped: every count survives
    # rows that absorbed nothing keep their values
    src = imap[:length]
    for s, j in enumerate(src):
        if j < ck.shape[0]:
            np.testing.assert_array_equal(nv[s], cv[j])
        elif info["owner"][info["top1"][j - ck.shape[0]]] != j - ck.shape[0]:
            np.testing.assert_array_equal(nv[s], v_cur[j - ck.shape[0]])


# ---- planted mistakes (in the oracle, on the CPU): each pin above must catch one ----

def _fails(pin, monkeypatch, name, fn):
    with monkeypatch.context() as mp:
        mp.setattr(O, name, fn)
        with pytest.raises(AssertionError):
            pin()


def test_planted_mistakes_are_caught(monkeypatch):
    # a log in the wrong base for the logit shift
    _fails(lambda: _pin_lemma(0), monkeypatch, "group_log", lambda g: np.log2(np.asarray(g, float)))
    # the shift with the wrong sign
    _fails(lambda: _pin_lemma(1), monkeypatch, "group_log", lambda g: -np.log(np.asarray(g, float)))
    real_owner, real_merge = O.evict_owner, O.merge_current

    def highest_owner(top1, ce, tau, n):
        owner = np.full(n, -1, np.int64)
        for i, j in enumerate(np.asarray(top1)):
            if j >= 0 and ce[i] >= tau:
                owner[j] = i
        return owner

    _fails(lambda: [_pin_enumeration(s, 64) for s in range(6)], monkeypatch, "evict_owner", highest_owner)

    def plain_mean(owner, top1, v_cur, cache_v, g_cache):
        v, g = real_merge(owner, top1, v_cur, cache_v, np.ones_like(np.asarray(g_cache)))
        return v, g

    _fails(lambda: _pin_rollout(0), monkeypatch, "merge_current", plain_mean)

    def owner_ignores_tau(top1, ce, tau, n):
        return real_owner(top1, np.full(np.asarray(ce).shape, 1.0), tau, n)

    _fails(lambda: [_pin_enumeration(s, 64) for s in range(6)], monkeypatch, "evict_owner", owner_ignores_tau)
