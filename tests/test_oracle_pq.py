"""Pins of the quantization variant of the TempCache match (technical summary §2.A: the
ANN is "LSH or Quantization"): product-quantization encoding by enumeration, exact
reconstruction of codewords, the one-sub-space reduction to the nearest unit centroid
(the bucketing rule), the lossless-codebook reduction to the exact match, the match by
enumeration, ties, and planted mistakes."""
import numpy as np
import pytest

from oracle import fastar_oracle as O
import brute_force


def _case(seed, n=40, d=16, m=4, Kc=6, nq=12):
    rng = np.random.default_rng(700 + seed)
    X = rng.standard_normal((n, d))
    # codewords of very different sizes, so that nearest-by-distance differs from
    # largest-inner-product
    Cb = rng.standard_normal((m, Kc, d // m)) * rng.uniform(0.2, 2.5, size=(m, Kc, 1))
    Q = X[rng.integers(0, n, nq)] + 0.3 * rng.standard_normal((nq, d))
    return X, Cb, Q


def _pin_encode(seed):
    X, Cb, _ = _case(seed)
    got = O.pq_encode(X, Cb)
    want = brute_force.pq_encode(X.tolist(), Cb.tolist())
    assert got.tolist() == want


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_encode_equals_enumeration(seed):
    _pin_encode(seed)


def test_codewords_reconstruct_exactly():
    _, Cb, _ = _case(3)
    m, Kc, ds = Cb.shape
    rng = np.random.default_rng(5)
    pick = rng.integers(0, Kc, size=(25, m))
    X = np.concatenate([Cb[s][pick[:, s]] for s in range(m)], axis=1)
    codes = O.pq_encode(X, Cb)
    assert np.array_equal(codes, pick)
    np.testing.assert_array_equal(O.pq_decode(codes, Cb), X)


def test_one_subspace_of_unit_codewords_is_the_bucketing_rule():
    # with unit-norm codewords, the nearest codeword is the arg-max inner product
    rng = np.random.default_rng(8)
    C = rng.standard_normal((10, 32))
    C /= np.linalg.norm(C, axis=1, keepdims=True)
    X = rng.standard_normal((200, 32)) * 3.0
    codes = O.pq_encode(X, C[None])
    assert np.array_equal(codes[:, 0], O.key_buckets(X, C))


def test_lossless_codebook_reduces_to_the_exact_match():
    # one sub-space whose codewords are the cached keys themselves: k^ = k
    X, _, Q = _case(4)
    codes = O.pq_encode(X, X[None])
    assert np.array_equal(codes[:, 0], np.arange(X.shape[0]))
    top1, s1 = O.tempcache_match_pq(Q, codes, X[None])
    t_ex, s_ex, _ = O.tempcache_match(Q, X)
    assert np.array_equal(top1, t_ex)
    np.testing.assert_array_equal(s1, s_ex)


def _pin_match(seed):
    X, Cb, Q = _case(seed)
    codes = O.pq_encode(X, Cb)
    top1, s1 = O.tempcache_match_pq(Q, codes, Cb)
    assert top1.tolist() == brute_force.pq_match(Q.tolist(), codes.tolist(), Cb.tolist())
    K_hat = np.concatenate([Cb[s][codes[:, s]] for s in range(Cb.shape[0])], axis=1)
    want = (K_hat[top1] * Q).sum(axis=1) / (np.linalg.norm(K_hat[top1], axis=1) * np.linalg.norm(Q, axis=1))
    np.testing.assert_allclose(s1, want, rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_match_equals_enumeration(seed):
    _pin_match(seed)


def test_ties_and_empty_cache():
    Cb = np.array([[[1.0, 0.0], [0.0, 1.0]]])          # m = 1, Kc = 2
    X = np.array([[0.5, 0.5], [3.0, -1.0]])               # equidistant from both codewords, then nearer 0
    assert O.pq_encode(X, Cb)[:, 0].tolist() == [0, 0]
    # two cached keys decode to the same codeword: the oldest wins
    top1, _ = O.tempcache_match_pq(np.array([[1.0, 0.2]]), np.array([[1], [0], [0]]), Cb)
    assert top1.tolist() == [1]
    top1, s1 = O.tempcache_match_pq(np.ones((3, 2)), np.zeros((0, 1), np.int64), Cb)
    assert top1.tolist() == [-1, -1, -1] and np.all(s1 == -np.inf)


# ---- planted mistakes (in the oracle, on the CPU) ----

def test_planted_mistakes_are_caught(monkeypatch):
    real_encode = O.pq_encode

    def by_inner_product(X, codebooks):     # largest inner product instead of the nearest
        X, Cb = np.asarray(X, float), np.asarray(codebooks, float)
        m, Kc, ds = Cb.shape
        return np.stack([np.argmax(X[:, s * ds:(s + 1) * ds] @ Cb[s].T, axis=1) for s in range(m)], axis=1)

    def shifted_subspace(X, codebooks):     # sub-vectors taken one dimension off
        return real_encode(np.roll(np.asarray(X, float), 1, axis=1), codebooks)

    for fn in (by_inner_product, shifted_subspace):
        with monkeypatch.context() as mp:
            mp.setattr(O, "pq_encode", fn)
            with pytest.raises(AssertionError):
                for seed in range(3):
                    _pin_encode(seed)

    def decode_wrong_order(codes, codebooks):   # sub-spaces concatenated in reverse
        Cb = np.asarray(codebooks, float)
        codes = np.asarray(codes)
        return np.concatenate([Cb[s][codes[:, s]] for s in range(Cb.shape[0] - 1, -1, -1)], axis=1)

    with monkeypatch.context() as mp:
        mp.setattr(O, "pq_decode", decode_wrong_order)
        with pytest.raises(AssertionError):
            for seed in range(3):
                _pin_match(seed)
