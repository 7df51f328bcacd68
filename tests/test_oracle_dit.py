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
