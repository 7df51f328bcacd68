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


# ----------------------------------------------------------------------------------
# the block body, worked by hand (tests/golden/dit_block_2d.json)
# ----------------------------------------------------------------------------------

def _golden_block():
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "dit_block_2d.json")))
    c = g["config"]

    class Cfg:
        pass

    for k, v in c.items():
        setattr(Cfg, k, v)
    p = {k: np.asarray(v, np.float64) for k, v in g["params"].items() if k != "block"}
    p["blocks"] = [{k: np.asarray(v, np.float64) for k, v in g["params"]["block"].items()}]
    tk = np.array([[float(x) if x != "ln3" else math.log(3.0) for x in row] for row in g["text_k"]])
    tv = np.asarray(g["text_v"], np.float64)
    return g, Cfg, p, tk, tv


def _run_golden(p, Cfg, g, tk, tv):
    hist = [(np.zeros((0, 2)), np.zeros((0, 2)))]
    return D.dit_step(p, Cfg, np.asarray(g["lat"], np.float64), g["t"], g["t_next"], g["frame0"], hist, [(tk, tv)])


def _block_only(p, Cfg, g, tk, tv, m):
    """dit_block on the golden's single token with the given modulation rows."""
    x = np.asarray(g["lat"], np.float64)            # identity patch map, zero patch bias
    pos = D.token_positions(1, g["frame0"], 1, 1)
    sa = lambda q, k, v: D.heads_attention(q, k, v, 1)
    ca = lambda qc: D.heads_attention(qc, tk, tv, 1)
    return D.dit_block(p["blocks"][0], Cfg, x, np.asarray(m, np.float64), pos, sa, ca)


def test_dit_block_hand_worked():
    g, Cfg, p, tk, tv = _golden_block()
    x3, (k, v) = _block_only(p, Cfg, g, tk, tv, g["modulation"])
    np.testing.assert_allclose(x3, g["expected"]["x_after_block"], rtol=0, atol=1e-9)
    np.testing.assert_allclose(v, g["expected"]["v"], rtol=0, atol=1e-9)
    kd = np.asarray(g["expected"]["k_direction"], np.float64)
    np.testing.assert_allclose(k, kd / np.sqrt((kd ** 2).mean()), rtol=0, atol=1e-9)   # RMS-normed, frame 0
    # the cross-attention and feed-forward branches off: what the self-attention branch leaves
    zero_ca = lambda qc: np.zeros_like(qc)
    m = np.asarray(g["modulation"], np.float64).copy()
    m[5] = 0.0
    x1, _ = D.dit_block(p["blocks"][0], Cfg, np.asarray(g["lat"], np.float64), m, D.token_positions(1, 0, 1, 1),
                        lambda q, k_, v_: D.heads_attention(q, k_, v_, 1), zero_ca)
    np.testing.assert_allclose(x1, g["expected"]["x_after_self_attention"], rtol=0, atol=1e-9)


def test_dit_step_hand_worked():
    # the whole step: timestep projection added to the block table, the block, the head
    g, Cfg, p, tk, tv = _golden_block()
    lat, kv = _run_golden(p, Cfg, g, tk, tv)
    np.testing.assert_allclose(lat, g["expected"]["lat_next"], rtol=0, atol=1e-9)
    np.testing.assert_allclose(kv[0][1], g["expected"]["v"], rtol=0, atol=1e-9)


@pytest.mark.parametrize("swap", [(0, 1), (3, 4), (2, 5), (0, 3), (1, 4)])
def test_dit_block_golden_tells_modulation_rows_apart(swap):
    # each plausible misreading of the six modulation rows (shift <-> scale, the gates of
    # the two branches, the two branches' shifts or scales) moves the hand-worked result
    g, Cfg, p, tk, tv = _golden_block()
    m = np.asarray(g["modulation"], np.float64).copy()
    a, b = swap
    m[[a, b]] = m[[b, a]]
    x3, _ = _block_only(p, Cfg, g, tk, tv, m)
    assert np.abs(x3 - np.asarray(g["expected"]["x_after_block"])).max() > 0.1


def test_dit_block_golden_catches_planted_mistakes(monkeypatch):
    g, Cfg, p, tk, tv = _golden_block()
    want = np.asarray(g["expected"]["x_after_block"])
    run = lambda: _block_only(p, Cfg, g, tk, tv, g["modulation"])[0]
    ln = D.layer_norm
    # (1) the cross-attention's layer norm without its affine map
    monkeypatch.setattr(D, "layer_norm", lambda x, eps, weight=None, bias=None: ln(x, eps))
    assert np.abs(run() - want).max() > 0.5
    monkeypatch.setattr(D, "layer_norm", ln)
    # (2) adaLN with shift and scale exchanged inside the modulation
    mod = D.modulate
    monkeypatch.setattr(D, "modulate", lambda y, shift, scale: mod(y, scale, shift))
    assert np.abs(run() - want).max() > 0.5
    monkeypatch.setattr(D, "modulate", mod)
    # (3) the feed-forward's activation left out
    gelu = D.ACTS[1]
    monkeypatch.setitem(D.ACTS, 1, lambda v: v)
    assert np.abs(run() - want).max() > 0.5
    monkeypatch.setitem(D.ACTS, 1, gelu)
    # (4) a gate on the cross-attention branch (the self-attention's)
    gemm = D.gemm
    co_w = p["blocks"][0]["co_w"]

    def gated_cross(A, W, bias=None, act=0, R=None, gate=None):
        if W is co_w:      # the cross-attention's output map, given the self-attention's gate
            gate = np.asarray(g["modulation"][2], np.float64)
        return gemm(A, W, bias, act, R, gate)

    monkeypatch.setattr(D, "gemm", gated_cross)
    assert np.abs(run() - want).max() > 0.5
    monkeypatch.setattr(D, "gemm", gemm)
    np.testing.assert_allclose(run(), want, rtol=0, atol=1e-9)


# ----------------------------------------------------------------------------------
# FAST-AR attention inside the DiT oracle
# ----------------------------------------------------------------------------------

def test_dit_fastar_textbook_reduction_equals_dense():
    # one bucket, r = 1, tau > 1 (nothing evicted), tau_ca = -1 (every text token kept),
    # M large enough for every chunk: each block's FAST-AR attention is dense attention
    # over its whole history, so the step equals the dense step chunk after chunk
    rng = np.random.default_rng(31)
    p = _params(rng, zero_blocks=False)
    for b in p["blocks"]:
        b["mod"][2] += 1.0
    H, d, frames = 2, 8, 2
    cent = [np.ones((H, 1, d)) / np.sqrt(d) for _ in p["blocks"]]
    fa = D.FastARAttention(cent, F=frames, Tf=3, M=64, r=1, tau=2.0, tau_ca=-1.0, topk=16)
    tkv = [(rng.standard_normal((5, 16)), rng.standard_normal((5, 16))) for _ in p["blocks"]]
    hist = [(np.zeros((0, 16)), np.zeros((0, 16))) for _ in p["blocks"]]
    for chunk in range(3):
        lat = rng.standard_normal((6, 4))
        want, kv = D.dit_step(p, _Cfg, lat, 0.5, 0.25, chunk * frames, hist, tkv)
        got, caches = D.dit_step(p, _Cfg, lat, 0.5, 0.25, chunk * frames, None, tkv, fastar=fa)
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)
        fa.caches = caches
        hist = [(np.concatenate([hk, k]), np.concatenate([hv, v])) for (hk, hv), (k, v) in zip(hist, kv)]
        for i, (k, v) in enumerate(hist):
            for h in range(H):
                np.testing.assert_allclose(caches[i][h][0], k[:, h * d:(h + 1) * d], atol=1e-15)


def test_dit_fastar_restricts_and_bounds():
    # with real buckets and a cap the FAST-AR step differs from the dense one, keeps at
    # most M entries per head, and a replayed decision set reproduces its own result
    rng = np.random.default_rng(32)
    p = _params(rng, zero_blocks=False)
    H, d, B = 2, 8, 4
    cent = []
    for _ in p["blocks"]:
        c = rng.standard_normal((H, B, d))
        cent.append(c / np.linalg.norm(c, axis=2, keepdims=True))
    tkv = [(rng.standard_normal((20, 16)), rng.standard_normal((20, 16))) for _ in p["blocks"]]
    fa = D.FastARAttention(cent, F=2, Tf=3, M=8, r=2, tau=0.3, tau_ca=0.5, topk=2)
    lat = rng.standard_normal((6, 4))
    for chunk in range(3):
        out, caches = D.dit_step(p, _Cfg, lat, 0.5, 0.25, chunk * 2, None, tkv, fastar=fa)
        fa.caches = caches
        assert all(c[0].shape[0] <= 8 for blk in caches for c in blk)
    dense, _ = D.dit_step(p, _Cfg, lat, 0.5, 0.25, 6, [(np.zeros((0, 16)), np.zeros((0, 16)))] * 2, tkv)
    fast, _ = D.dit_step(p, _Cfg, lat, 0.5, 0.25, 6, None, tkv, fastar=fa)
    assert np.abs(fast - dense).max() > 1e-3
