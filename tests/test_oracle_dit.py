"""Pins of the transformer oracle (the DiT around the attention step): the GEMM with its
epilogues against a loop-by-loop product, identity and zero-gate reductions, and the
activations against their textbook definitions and known values."""
import math

import numpy as np
import pytest
from scipy.special import erf

from oracle import dit_oracle as D


def _loops(A, W, bias, act, R, gate):
    M, K = A.shape
    N = W.shape[0]
    out = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            s = 0.0
            for k in range(K):
                s += float(A[m, k]) * float(W[n, k])
            if bias is not None:
                s += float(bias[n])
            if act == 1:
                s = 0.5 * s * (1.0 + math.tanh(math.sqrt(2.0 / math.pi) * (s + 0.044715 * s ** 3)))
            elif act == 2:
                s = s / (1.0 + math.exp(-s))
            if R is not None:
                s = float(R[m, n]) + (1.0 if gate is None else float(gate[n])) * s
            out[m, n] = s
    return out


@pytest.mark.parametrize("act", [0, 1, 2])
@pytest.mark.parametrize("with_res", [False, True])
def test_gemm_equals_loops(act, with_res):
    rng = np.random.default_rng(10 * act + with_res)
    A, W = rng.standard_normal((5, 7)), rng.standard_normal((6, 7))
    bias, R, gate = rng.standard_normal(6), rng.standard_normal((5, 6)), rng.standard_normal(6)
    got = D.gemm(A, W, bias, act, R if with_res else None, gate if with_res else None)
    want = _loops(A, W, bias, act, R if with_res else None, gate if with_res else None)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_gemm_reductions():
    rng = np.random.default_rng(3)
    A = rng.standard_normal((9, 8))
    np.testing.assert_array_equal(D.gemm(A, np.eye(8)), A)                       # identity weight
    R = rng.standard_normal((9, 8))
    np.testing.assert_array_equal(D.gemm(A, np.eye(8), R=R, gate=np.zeros(8)), R)  # zero gate
    np.testing.assert_allclose(D.gemm(A, np.eye(8), R=R), R + A, rtol=0, atol=1e-15)


def test_activations():
    x = np.linspace(-6, 6, 241)
    exact_gelu = 0.5 * x * (1 + erf(x / np.sqrt(2)))
    assert np.max(np.abs(D.gelu_tanh(x) - exact_gelu)) < 1e-3      # the tanh form is within 1e-3 of erf
    np.testing.assert_allclose(D.gelu_tanh(x) - D.gelu_tanh(-x), x, atol=1e-14)
    assert D.gelu_tanh(0.0) == 0.0
    np.testing.assert_allclose(D.silu(x), x * (1 / (1 + np.exp(-x))), atol=1e-15)
    assert abs(D.silu(1.0) - 0.7310585786300049) < 1e-15           # 1 / (1 + e^-1)


def test_layer_norm_and_modulation():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((20, 48)) * 3 + 5
    y = D.layer_norm(x, 1e-12)
    np.testing.assert_allclose(y.mean(axis=1), 0, atol=1e-12)
    np.testing.assert_allclose(y.std(axis=1), 1, atol=1e-9)
    w, b = rng.standard_normal(48), rng.standard_normal(48)
    np.testing.assert_allclose(D.layer_norm(x, 1e-12, w, b), y * w + b, atol=1e-12)
    # zero modulation is the identity; scale -1 leaves the shift alone
    np.testing.assert_array_equal(D.modulate(y, np.zeros(48), np.zeros(48)), y)
    np.testing.assert_allclose(D.modulate(y, b, -np.ones(48)), np.broadcast_to(b, y.shape), atol=0)


def test_rms_norm():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((10, 64)) * 7
    y = D.rms_norm(x, np.ones(64), 1e-12)
    np.testing.assert_allclose(np.sqrt((y ** 2).mean(axis=1)), 1, atol=1e-9)
    np.testing.assert_allclose(D.rms_norm(2 * x, np.ones(64), 1e-12), y, atol=1e-12)   # scale invariant


def test_rope_properties():
    rng = np.random.default_rng(6)
    d, H, n = 36, 2, 40
    q, k = rng.standard_normal((n, H * d)), rng.standard_normal((n, H * d))
    pos = D.token_positions(n, 3, 4, 5)
    assert D.rope_split(128) == (44, 42, 42)
    # position 0 is the identity; every pair keeps its length
    np.testing.assert_array_equal(D.rope(q, d, np.zeros((n, 3))), q)
    r = D.rope(q, d, pos)
    np.testing.assert_allclose((r.reshape(n, -1, 2) ** 2).sum(-1), (q.reshape(n, -1, 2) ** 2).sum(-1), atol=1e-12)
    # the score of a rotated pair depends only on the difference of positions
    shift = np.array([2, 1, 3])
    qa, ka = D.rope(q, d, pos), D.rope(k, d, pos)
    qb, kb = D.rope(q, d, pos + shift), D.rope(k, d, pos + shift)
    for h in range(H):
        s = slice(h * d, (h + 1) * d)
        np.testing.assert_allclose(qa[:, s] @ ka[:, s].T, qb[:, s] @ kb[:, s].T, atol=1e-9)
    # one pair by hand: frame axis, pair 0 turns by the frame index (theta^0 = 1)
    x = np.zeros((1, d))
    x[0, 0] = 1.0
    got = D.rope(x, d, np.array([[0.7, 0, 0]]))
    np.testing.assert_allclose(got[0, :2], [np.cos(0.7), np.sin(0.7)], atol=1e-15)
    np.testing.assert_array_equal(D.token_positions(7, 2, 2, 3)[5], [2, 1, 2])
    np.testing.assert_array_equal(D.token_positions(7, 2, 2, 3)[6], [3, 0, 0])


def test_sinusoidal():
    e = D.sinusoidal([0.0, 1.0], 8)
    np.testing.assert_array_equal(e[0], [1, 1, 1, 1, 0, 0, 0, 0])
    np.testing.assert_allclose(e[1, 0], np.cos(1.0), atol=1e-15)
    np.testing.assert_allclose(e[1, 4 + 2], np.sin(1.0 * 10000.0 ** (-2 / 4)), atol=1e-15)
