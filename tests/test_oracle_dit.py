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


def test_heads_attention_matches_the_step_oracle():
    from oracle import fastar_oracle as O
    rng = np.random.default_rng(12)
    H, d = 3, 16
    Q, K, V = rng.standard_normal((9, H * d)), rng.standard_normal((14, H * d)), rng.standard_normal((14, H * d))
    got = D.heads_attention(Q, K, V, H)
    for h in range(H):
        s = slice(h * d, (h + 1) * d)
        want, _ = O.dense_attention(Q[:, s], K[:, s], V[:, s], 1 / np.sqrt(d))
        np.testing.assert_allclose(got[:, s], want, atol=1e-12)


class _Cfg:
    dim, heads, eps, freq_dim, grid_h, grid_w, theta = 16, 2, 1e-6, 8, 2, 3, 10000.0


def _params(rng, zero_blocks):
    Dm, f = 16, 32
    z = (lambda *s: np.zeros(s)) if zero_blocks else (lambda *s: rng.standard_normal(s) * 0.3)
    blocks = [dict(mod=z(6, Dm), qkv_w=z(3 * Dm, Dm), qkv_b=z(3 * Dm), norm_q=np.ones(Dm), norm_k=np.ones(Dm),
                   o_w=z(Dm, Dm), o_b=z(Dm), norm3_w=np.ones(Dm), norm3_b=z(Dm), cq_w=z(Dm, Dm), cq_b=z(Dm),
                   norm_cq=np.ones(Dm), co_w=z(Dm, Dm), co_b=z(Dm), f1_w=z(f, Dm), f1_b=z(f), f2_w=z(Dm, f),
                   f2_b=z(Dm)) for _ in range(2)]
    r = lambda *s: rng.standard_normal(s) * 0.3
    return dict(time_w1=r(Dm, 8), time_b1=r(Dm), time_w2=r(Dm, Dm), time_b2=r(Dm), proj_w=r(6 * Dm, Dm),
                proj_b=r(6 * Dm), patch_w=r(Dm, 4), patch_b=r(Dm), head_mod=r(2, Dm), head_w=r(4, Dm),
                head_b=r(4), blocks=blocks)


def test_dit_step_with_silent_blocks_is_the_head_alone():
    rng = np.random.default_rng(13)
    p = _params(rng, zero_blocks=True)
    lat = rng.standard_normal((6, 4))
    hist = [(np.zeros((0, 16)), np.zeros((0, 16)))] * 2
    tkv = [(rng.standard_normal((5, 16)), rng.standard_normal((5, 16)))] * 2
    got, _ = D.dit_step(p, _Cfg, lat, 0.75, 0.5, 0, hist, tkv)
    # by hand: the embedding MLP, the patch map, then LN + modulation + the head map
    emb = np.concatenate([np.cos(750.0 * 10000.0 ** (-np.arange(4) / 4)), np.sin(750.0 * 10000.0 ** (-np.arange(4) / 4))])
    s1 = emb @ p["time_w1"].T + p["time_b1"]
    e = (s1 / (1 + np.exp(-s1))) @ p["time_w2"].T + p["time_b2"]
    x = lat @ p["patch_w"].T + p["patch_b"]
    xn = (x - x.mean(1, keepdims=True)) / np.sqrt(x.var(1, keepdims=True) + 1e-6)
    h = xn * (1 + p["head_mod"][1] + e) + p["head_mod"][0] + e
    want = lat - 0.25 * (h @ p["head_w"].T + p["head_b"])
    np.testing.assert_allclose(got, want, atol=1e-12)


def test_text_context_and_cross_kv_reduce_with_identity_weights():
    # identity projections without bias: the text context is the tanh-form GELU of the
    # text itself (known values at 0 and for large |x|), and a block's cross keys are the
    # RMS-normed context rows (unit mean square), its values the context itself
    rng = np.random.default_rng(4)
    n, c = 9, 12
    text = rng.standard_normal((n, c)) * 3
    eye, zero = np.eye(c), np.zeros(c)
    p = dict(text_w1=eye, text_b1=zero, text_w2=eye, text_b2=zero)
    ctx = D.text_context(p, text)
    x = text
    np.testing.assert_allclose(ctx, 0.5 * x * (1 + np.tanh(math.sqrt(2 / math.pi) * (x + 0.044715 * x ** 3))),
                               rtol=0, atol=1e-12)
    edge = D.text_context(p, np.array([[0.0] * (c - 2) + [40.0, -40.0]]))
    np.testing.assert_allclose(edge[0, -2:], [40.0, 0.0], atol=1e-12)
    b = dict(ck_w=eye, ck_b=zero, cv_w=eye, cv_b=zero, norm_ck=np.ones(c))
    k, v = D.block_text_kv(b, ctx, 4, 0.0)
    np.testing.assert_allclose((k ** 2).mean(axis=1), 1.0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(k * np.sqrt((ctx ** 2).mean(axis=1, keepdims=True)), ctx, rtol=0, atol=1e-12)
    np.testing.assert_allclose(v, ctx, rtol=0, atol=1e-12)
