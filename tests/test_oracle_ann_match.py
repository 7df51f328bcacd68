"""Pins of the ANN-restricted TempCache match (the match variant that compares each
query only with the cached keys in its own buckets): exhaustive enumeration, the
one-bucket reduction to the exact match, the restriction, empty buckets, ties, and
planted mistakes that these pins must catch."""
import numpy as np
import pytest

from oracle import fastar_oracle as O
import brute_force


def _case(seed, n=48, nq=16, d=8, B=4, r=2):
    rng = np.random.default_rng(300 + seed)
    ck = rng.standard_normal((n, d))
    q = ck[rng.integers(0, n, nq)] + 0.3 * rng.standard_normal((nq, d))
    C = rng.standard_normal((B, d))
    C /= np.linalg.norm(C, axis=1, keepdims=True)
    kb = O.key_buckets(ck, C)
    R = O.query_buckets(q, C, r)
    return q, R, ck, kb


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_ann_match_equals_enumeration(seed):
    q, R, ck, kb = _case(seed)
    top1, s1 = O.tempcache_match_ann(q, R, ck, kb)
    want_t, want_s = brute_force.ann_match(q.tolist(), R.tolist(), ck.tolist(), kb.tolist())
    assert top1.tolist() == want_t
    np.testing.assert_allclose(s1, np.array(want_s), rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed", [0, 1])
def test_one_bucket_reduces_to_exact_match(seed):
    q, _, ck, _ = _case(seed)
    R = np.zeros((q.shape[0], 1), np.int64)
    kb = np.zeros(ck.shape[0], np.int64)
    top1, s1 = O.tempcache_match_ann(q, R, ck, kb)
    t_exact, s_exact, _ = O.tempcache_match(q, ck)
    assert top1.tolist() == t_exact.tolist()
    np.testing.assert_array_equal(s1, s_exact)


def test_key_outside_the_buckets_is_not_chosen():
    # query (1, 0): key 0 (bucket 0) has cosine 0.8, key 1 (bucket 1) cosine 1
    q = np.array([[1.0, 0.0]])
    ck = np.array([[0.8, 0.6], [2.0, 0.0]])
    kb = np.array([0, 1])
    top1, s1 = O.tempcache_match_ann(q, np.array([[0]]), ck, kb)
    assert top1.tolist() == [0] and s1[0] == pytest.approx(0.8)
    top1, s1 = O.tempcache_match_ann(q, np.array([[1]]), ck, kb)
    assert top1.tolist() == [1] and s1[0] == pytest.approx(1.0)


def test_empty_buckets_give_no_match():
    q = np.array([[1.0, 0.0], [0.0, 1.0]])
    ck = np.array([[1.0, 0.0], [0.0, 1.0]])
    kb = np.array([0, 0])
    top1, s1 = O.tempcache_match_ann(q, np.array([[1, 2], [0, 3]]), ck, kb)
    assert top1.tolist() == [-1, 1]
    assert s1[0] == -np.inf and s1[1] == pytest.approx(1.0)
    top1, s1 = O.tempcache_match_ann(q, np.array([[0], [0]]), np.zeros((0, 2)), np.zeros(0, np.int64))
    assert top1.tolist() == [-1, -1]


def test_ties_take_the_oldest_key_in_the_buckets():
    # keys 1, 2 and 3 are the same vector; key 1 is in another bucket
    q = np.array([[1.0, 1.0]])
    ck = np.array([[1.0, -1.0], [1.0, 1.0], [1.0, 1.0], [2.0, 2.0]])
    kb = np.array([0, 1, 0, 0])
    top1, _ = O.tempcache_match_ann(q, np.array([[0]]), ck, kb)
    assert top1.tolist() == [2]


def test_pins_catch_planted_mistakes(monkeypatch):
    real = O.tempcache_match_ann

    def unrestricted(Q, R, K, kb):   # forgets the bucket condition
        t, s, _ = O.tempcache_match(Q, K)
        return t, s
    monkeypatch.setattr(O, "tempcache_match_ann", unrestricted)
    with pytest.raises(AssertionError):
        test_key_outside_the_buckets_is_not_chosen()

    def newest_tie(Q, R, K, kb):     # takes the newest of equal keys
        Qr, Kr = np.asarray(Q)[:, :], np.asarray(K)[::-1]
        t, s = real(Qr, R, Kr, np.asarray(kb)[::-1])
        return np.where(t >= 0, len(K) - 1 - t, -1), s
    monkeypatch.setattr(O, "tempcache_match_ann", newest_tie)
    with pytest.raises(AssertionError):
        test_ties_take_the_oldest_key_in_the_buckets()
