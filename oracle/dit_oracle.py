"""Plain CPU oracle of the diffusion transformer around the FAST-AR attention step.
TEST INFRASTRUCTURE.

Only the tests, the package's smoke check and the benchmark's CPU-baseline arm may
import or run this module.  It shares no code with the CUDA path and imports nothing
from it; the product path never calls it.

The pages describe FAST-AR as a drop-in replacement for the attention layers of an
autoregressive video diffusion transformer (blog, Significance; technical summary, Key
Results: Rolling-Forcing and LongVie2 on Wan-family backbones); the transformer itself is
not on the pages.  This module writes out, in float64 NumPy, a Wan2.1-shaped block with
the plainest reading of each operation (the readings are listed in the design notes):
layer norm with adaptive shift/scale/gate modulation (adaLN), fused QKV projection, RMS
norm of q and k, rotary positions over (frame, row, column), self-attention, a second
normed cross-attention over the text, a GELU(tanh) feed-forward, and the flow-matching
Euler update of the denoising loop.  The attention of every block is either dense or
FAST-AR (TempCache + AnnSA for the self-attention, AnnCA for the cross-attention), the
latter composed from the per-chunk step oracle's functions in the pages' order.

Pins: the block body against a case worked by hand (tests/golden/dit_block_2d.json), the
GEMM against loop-by-loop products, the norms, rotary map and embedding against their
definitions and closed forms, FAST-AR inside the DiT against the dense DiT in the
textbook reduction.
"""
from __future__ import annotations

import numpy as np


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


# ----------------------------------------------------------------------------------
# elementwise and GEMM
# ----------------------------------------------------------------------------------

def gelu_tanh(x) -> np.ndarray:
    """0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))."""
    x = _f64(x)
    return 0.5 * x * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * (x + 0.044715 * x ** 3)))


def silu(x) -> np.ndarray:
    """x / (1 + exp(-x))."""
    x = _f64(x)
    return x / (1.0 + np.exp(-x))


ACTS = {0: lambda v: v, 1: gelu_tanh, 2: silu}


def gemm(A, W, bias=None, act: int = 0, R=None, gate=None) -> np.ndarray:
    """R + gate * act(A @ W^T + bias); without R: act(A @ W^T + bias).
    A [M, K]; W [N, K] (a Linear weight); bias, gate [N]."""
    Y = _f64(A) @ _f64(W).T
    if bias is not None:
        Y = Y + _f64(bias)[None, :]
    Y = ACTS[act](Y)
    if R is not None:
        g = np.ones(Y.shape[1]) if gate is None else _f64(gate)
        Y = _f64(R) + g[None, :] * Y
    return Y


# ----------------------------------------------------------------------------------
# norms, rotary positions, timestep embedding
# ----------------------------------------------------------------------------------

def layer_norm(x, eps: float, weight=None, bias=None) -> np.ndarray:
    """(x - mean) / sqrt(var + eps) over the last axis (biased variance) [* weight + bias]."""
    x = _f64(x)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    y = (x - mu) / np.sqrt(var + eps)
    if weight is not None:
        y = y * _f64(weight) + (0.0 if bias is None else _f64(bias))
    return y


def modulate(y, shift, scale) -> np.ndarray:
    """adaLN: y * (1 + scale) + shift (per channel)."""
    return _f64(y) * (1.0 + _f64(scale)) + _f64(shift)


def rms_norm(x, weight, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * weight over the last axis."""
    x = _f64(x)
    return x / np.sqrt((x ** 2).mean(axis=-1, keepdims=True) + eps) * _f64(weight)


def rope_split(d: int):
    """Channels of a head given to the frame, row and column positions."""
    part = 2 * (d // 6)
    return d - 2 * part, part, part


def token_positions(n: int, t0: int, gh: int, gw: int) -> np.ndarray:
    """(frame, row, column) of the n tokens of a chunk, frame-major: [n, 3]."""
    i = np.arange(n)
    return np.stack([t0 + i // (gh * gw), (i // gw) % gh, i % gw], axis=1)


def rope(x, d: int, pos, theta: float = 10000.0) -> np.ndarray:
    """Rotary positions on x [n, H*d] (token-major): in each head, the channels split
    into frame / row / column parts (rope_split); in a part of width da the pair
    (2j, 2j + 1) is turned by pos_axis * theta^(-2j / da)."""
    x = _f64(x).copy()
    n, C = x.shape
    pos = np.asarray(pos, np.float64)
    widths = rope_split(d)
    for h in range(C // d):
        base = h * d
        for axis, da in enumerate(widths):
            for j in range(da // 2):
                c = base + sum(widths[:axis]) + 2 * j
                ang = pos[:, axis] * theta ** (-2.0 * j / da)
                a0, a1 = x[:, c].copy(), x[:, c + 1].copy()
                x[:, c] = a0 * np.cos(ang) - a1 * np.sin(ang)
                x[:, c + 1] = a0 * np.sin(ang) + a1 * np.cos(ang)
    return x


def sinusoidal(t, dim: int) -> np.ndarray:
    """[cos(t f_i), sin(t f_i)], f_i = 10000^(-i / (dim/2)), for each t: [len(t), dim]."""
    t = _f64(np.atleast_1d(t))
    half = dim // 2
    ang = t[:, None] * 10000.0 ** (-np.arange(half) / half)[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1)


# ----------------------------------------------------------------------------------
# the denoising step of the transformer (dense attention over the oracle's history, or
# FAST-AR attention over the oracle's bounded caches)
# ----------------------------------------------------------------------------------

def softmax_attention(Q, K, V, scale: float) -> np.ndarray:
    """Row softmax(Q K^T * scale) V, max-subtracted.  Q [n, d], K, V [m, d]."""
    S = _f64(Q) @ _f64(K).T * scale
    S = S - S.max(axis=1, keepdims=True)
    P = np.exp(S)
    return (P / P.sum(axis=1, keepdims=True)) @ _f64(V)


def heads_attention(Q, K, V, H: int) -> np.ndarray:
    """Multi-head attention on token-major [n, H*d] tensors, scale 1/sqrt(d)."""
    d = Q.shape[1] // H
    out = np.zeros((Q.shape[0], H * d))
    for h in range(H):
        s = slice(h * d, (h + 1) * d)
        out[:, s] = softmax_attention(Q[:, s], K[:, s], V[:, s], 1.0 / np.sqrt(d))
    return out


def text_context(p, text) -> np.ndarray:
    """The text encoder output projected to the model width: GELU MLP."""
    return gemm(gemm(text, p["text_w1"], p["text_b1"], act=1), p["text_w2"], p["text_b2"])


def block_text_kv(b, ctx, d: int, eps: float):
    """A block's cross-attention keys (RMS-normed) and values over the text."""
    return rms_norm(gemm(ctx, b["ck_w"], b["ck_b"]), b["norm_ck"], eps), gemm(ctx, b["cv_w"], b["cv_b"])


def dit_block(b, cfg, x, m, pos, self_attention, cross_attention, rope_on: bool = True):
    """One block on the residual stream x [tokens, D].  m [6, D]: the block's modulation
    rows (shift, scale, gate of the self-attention branch; shift, scale, gate of the
    feed-forward branch).  self_attention(q, k, v) and cross_attention(qc) return the
    attention outputs (token-major [tokens, D]) over the block's history and the text.
    Returns (x after the block, (k, v) of the chunk: keys normed and rotated)."""
    D, d, eps = cfg.dim, cfg.dim // cfg.heads, cfg.eps
    h = modulate(layer_norm(x, eps), m[0], m[1])
    qkv = gemm(h, b["qkv_w"], b["qkv_b"])
    q = rms_norm(qkv[:, :D], b["norm_q"], eps)
    k = rms_norm(qkv[:, D:2 * D], b["norm_k"], eps)
    v = qkv[:, 2 * D:]
    if rope_on:
        q, k = rope(q, d, pos, cfg.theta), rope(k, d, pos, cfg.theta)
    x = gemm(self_attention(q, k, v), b["o_w"], b["o_b"], R=x, gate=m[2])
    qc = rms_norm(gemm(layer_norm(x, eps, b["norm3_w"], b["norm3_b"]), b["cq_w"], b["cq_b"]), b["norm_cq"], eps)
    x = gemm(cross_attention(qc), b["co_w"], b["co_b"], R=x)
    h = modulate(layer_norm(x, eps), m[3], m[4])
    x = gemm(gemm(h, b["f1_w"], b["f1_b"], act=1), b["f2_w"], b["f2_b"], R=x, gate=m[5])
    return x, (k, v)


class FastARAttention:
    """FAST-AR in place of every block's attention (blog: a drop-in replacement for the
    attention layers): TempCache + AnnSA for the self-attention over a bounded per-head
    cache, AnnCA for the cross-attention over the text, each step as the per-chunk step
    oracle defines it.  AnnSA's buckets come from the self-attention queries, AnnCA's
    from the cross-attention queries (each attention its own queries).

    centroids[i] [H, B, d] of block i; caches[i][h] = (K, V, key buckets) of block i,
    head h, oldest first (empty at the start of a rollout).  A denoising step reads the
    caches and returns the caches it would leave (dit_step's second result); the
    rollout keeps those of a chunk's last step (commit)."""

    def __init__(self, centroids, *, F, Tf, M, r, tau, tau_ca, topk):
        self.C = [np.asarray(c, np.float64) for c in centroids]
        self.F, self.Tf, self.M, self.r = F, Tf, M, r
        self.tau, self.tau_ca, self.topk = tau, tau_ca, topk
        H, _, d = self.C[0].shape
        self.caches = [[(np.zeros((0, d)), np.zeros((0, d)), np.zeros(0, np.int64)) for _ in range(H)]
                       for _ in self.C]

    def self_attention(self, i, q, k, v, decisions=None):
        """Block i's TempCache + AnnSA on token-major q, k, v.  decisions[h]: optional
        discrete choices of head h ('qb', 'kb_cur', 'top1', 'evict') taken instead of
        the oracle's own.  Returns (o, the block's new caches)."""
        from . import fastar_oracle as O
        C = self.C[i]
        H, _, d = C.shape
        out = np.zeros((q.shape[0], H * d))
        new = []
        for h in range(H):
            s = slice(h * d, (h + 1) * d)
            qh, kh, vh = _f64(q[:, s]), _f64(k[:, s]), _f64(v[:, s])
            ck, cv, ckb = self.caches[i][h]
            dec = decisions[h] if decisions else {}
            qb = dec.get("qb")
            qb = O.query_buckets(qh, C[h], self.r) if qb is None else np.asarray(qb, np.int64)
            kb = dec.get("kb_cur")
            kb = O.key_buckets(kh, C[h]) if kb is None else np.asarray(kb, np.int64)
            top1 = dec.get("top1")
            top1 = O.tempcache_match(qh, ck)[0] if top1 is None else np.asarray(top1, np.int64)
            evict = dec.get("evict")
            evict = O.evict_flags(top1, kh, ck, self.tau)[0] if evict is None else np.asarray(evict, bool)
            imap, length = O.compact_plan(evict, ck.shape[0], qh.shape[0], self.M)
            nk, nv = O.gather_rows(imap, length, ck, kh), O.gather_rows(imap, length, cv, vh)
            nkb = O.gather_rows(imap, length, ckb, kb)
            out[:, s] = O.annsa_attention(qh, qb, nk, nv, nkb, 1.0 / np.sqrt(d))[0]
            new.append((nk, nv, nkb))
        return out, new

    def cross_attention(self, i, qc, tk, tv, decisions=None):
        """Block i's AnnCA on token-major queries qc over the text keys/values tk, tv.
        decisions[h]: optional 'qb', 'pb', 'keep' of head h."""
        from . import fastar_oracle as O
        C = self.C[i]
        H, _, d = C.shape
        out = np.zeros((qc.shape[0], H * d))
        for h in range(H):
            s = slice(h * d, (h + 1) * d)
            qh, kh, vh = _f64(qc[:, s]), _f64(tk[:, s]), _f64(tv[:, s])
            dec = decisions[h] if decisions else {}
            qb = dec.get("qb")
            qb = O.query_buckets(qh, C[h], self.r) if qb is None else np.asarray(qb, np.int64)
            pb = dec.get("pb")
            pb = O.key_buckets(kh, C[h]) if pb is None else np.asarray(pb, np.int64)
            keep = dec.get("keep")
            if keep is None:
                kidx = O.annca_select(qh, qb, kh, pb, self.F, self.Tf, self.tau_ca, self.topk)[1]
            else:
                kidx = [np.flatnonzero(np.asarray(keep[f], bool)) for f in range(self.F)]
            out[:, s] = O.cross_attention_subset(qh, kh, vh, kidx, self.F, self.Tf, 1.0 / np.sqrt(d))[0]
        return out


def dit_step(p, cfg, lat, t: float, t_next: float, frame0: int, history, text_kv, rope_on: bool = True,
             fastar: "FastARAttention | None" = None, decisions=None):
    """One denoising step of the chunk.  p: parameters (float arrays; blocks a list of
    dicts); lat [tokens, patch_ch] the latent; text_kv[i] = (K, V) of block i over the
    text.  Dense attention (fastar None): history[i] = (K, V) of block i's earlier chunks
    (token-major, keys already rotated); returns (the updated latent, [(k, v) of the
    chunk for every block]).  FAST-AR attention: history is not used, the caches are
    fastar's; decisions[i] = {'self': [per head], 'cross': [per head]} optional replayed
    choices; returns (the updated latent, the caches the step leaves)."""
    D, H = cfg.dim, cfg.heads
    emb = sinusoidal([t * 1000.0], cfg.freq_dim)
    e1 = gemm(emb, p["time_w1"], p["time_b1"], act=2)
    e = gemm(e1, p["time_w2"], p["time_b2"])[0]
    e0 = gemm(silu(e)[None, :], p["proj_w"], p["proj_b"])[0].reshape(6, D)
    x = gemm(lat, p["patch_w"], p["patch_b"])
    pos = token_positions(x.shape[0], frame0, cfg.grid_h, cfg.grid_w)
    kv_out, caches = [], []
    for i, (b, (tk, tv)) in enumerate(zip(p["blocks"], text_kv)):
        if fastar is None:
            hk, hv = history[i]
            sa = lambda q, k, v, hk=hk, hv=hv: heads_attention(q, np.concatenate([hk, k]), np.concatenate([hv, v]), H)
            ca = lambda qc, tk=tk, tv=tv: heads_attention(qc, tk, tv, H)
        else:
            dec = decisions[i] if decisions else {}

            def sa(q, k, v, i=i, dec=dec):
                o, new = fastar.self_attention(i, q, k, v, dec.get("self"))
                caches.append(new)
                return o

            ca = lambda qc, i=i, tk=tk, tv=tv, dec=dec: fastar.cross_attention(i, qc, tk, tv, dec.get("cross"))
        x, kv = dit_block(b, cfg, x, b["mod"] + e0, pos, sa, ca, rope_on)
        kv_out.append(kv)
    hm = p["head_mod"] + e
    h = modulate(layer_norm(x, cfg.eps), hm[0], hm[1])
    vel = gemm(h, p["head_w"], p["head_b"])
    return _f64(lat) + (t_next - t) * vel, (kv_out if fastar is None else caches)
