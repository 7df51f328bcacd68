"""Seeded synthetic inputs for the FAST-AR per-chunk attention step.

This module only draws random numbers and rounds them to the storage type; it holds
none of the method's arithmetic (no bucketing, matching, compaction or attention).
Both the CUDA path (through the benchmark and the tests) and the CPU oracle consume
what it produces.

Workload shape (FAST-AR, "Fast Autoregressive Video Diffusion and World Models with
Temporal Cache Compression and Sparse Attention", Problem Statement and §2.A–C):
an autoregressive video model produces one chunk of F latent frames per step; each
frame has T_f = h*w tokens. Keys drift slowly from frame to frame (the pages'
"near-duplicate cached keys across frames" and "slowly evolving queries/keys"), a
fraction of positions is re-drawn every frame, queries sit near their keys, and
the prompt is an unstructured set of P tokens.

Drift process, per head:
  * cluster means mu_c = normalise(N(0, I_d)), c < C
  * frame 0: k_t = mu_{c(t)} + sigma_mix * N(0, I_d), c(t) uniform
  * frame t > 0: k <- k + drift * N(0, I_d); round(rho * T_f) positions (shared by
    all heads) are re-drawn from the mixture with a fresh uniform cluster
  * queries q = k + qnoise * N(0, I_d); values V ~ N(0, I_d)
  * prompt keys Kp ~ N(0, I_d) / sqrt(d), prompt values Vp ~ N(0, I_d)
  * bucket centroids: B rows of N(0, I_d), each scaled to unit length (the random
    unit-centroid ANN the spec fixes for AnnSA/AnnCA bucketing)

bf16 configurations are rounded once, round-to-nearest-even, here; everything
downstream (CUDA path and oracle) sees exactly the rounded values.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import numpy as np


# ----------------------------------------------------------------------------------
# storage rounding
# ----------------------------------------------------------------------------------

def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); return float32."""
    a = np.ascontiguousarray(x, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).reshape(a.shape)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """The upper 16 bits of float32 values that are already bf16-exact."""
    a = np.ascontiguousarray(x, dtype=np.float32)
    return (a.view(np.uint32) >> 16).astype(np.uint16)


# ----------------------------------------------------------------------------------
# workload configurations
# ----------------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class LayerConfig:
    name: str
    H: int            # heads
    d: int            # head dimension
    Tf: int           # tokens per latent frame (h*w)
    F: int            # latent frames per chunk
    prior_frames: int  # frames generated before the measured chunk
    P: int            # prompt tokens
    C: int            # mixture clusters per head
    sigma_mix: float  # per-coordinate std of the mixture
    rho: float        # fraction of positions re-drawn per frame
    drift: float      # per-coordinate std of the per-frame key drift
    qnoise: float     # per-coordinate std of query noise around the key
    tau: float        # TempCache eviction threshold (cosine)
    M: int            # cache capacity (entries per head)
    B: int            # ANN buckets per head
    r: int            # buckets per query
    tau_ca: float     # AnnCA keep threshold (cosine)
    topk: int         # AnnCA always-keep count
    dtype: str        # "f32" or "bf16": storage type of every tensor input

    @property
    def Nq(self) -> int:
        return self.F * self.Tf

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.d))

    def replace(self, **kw) -> "LayerConfig":
        return dataclasses.replace(self, **kw)


# The tiny fp32 parity workload: 1 head, d=64, 16x16-token frames, 3 prior frames,
# 1-frame chunks, 8-cluster mixture, 32 prompt tokens.
TINY_FP32 = LayerConfig(
    name="tiny_fp32", H=1, d=64, Tf=256, F=1, prior_frames=3, P=32, C=8,
    sigma_mix=0.3, rho=0.1, drift=0.05, qnoise=0.1, tau=0.95, M=768, B=8, r=2,
    tau_ca=0.2, topk=16, dtype="f32")

# A Wan2.1-1.3B-shaped attention layer: 12 heads x d=128 (hidden 1536), chunks of 3
# latent frames of 30x52 tokens, 21 prior frames, 32-cluster mixture, 512 prompt tokens.
WAN13B_LAYER = LayerConfig(
    name="wan13b_layer", H=12, d=128, Tf=30 * 52, F=3, prior_frames=21, P=512, C=32,
    sigma_mix=0.3, rho=0.1, drift=0.05, qnoise=0.1, tau=0.95, M=9360, B=64, r=2,
    tau_ca=0.2, topk=16, dtype="bf16")

# The same layer stepped through a 200-frame rollout from an empty cache (67 chunks of
# 3 frames = 201 frames, so every step has the same shape).
WAN13B_ROLLOUT_CHUNKS = 67

# A HunyuanVideo-shaped 720p layer: 24 heads x d=128 (hidden 3072), chunks of 4 latent
# frames of 45x80 tokens, 16 prior frames, 64-cluster mixture, 5% re-drawn per frame.
HUNYUAN720P_LAYER = LayerConfig(
    name="hunyuan720p_layer", H=24, d=128, Tf=45 * 80, F=4, prior_frames=16, P=256, C=64,
    sigma_mix=0.3, rho=0.05, drift=0.05, qnoise=0.1, tau=0.9, M=28800, B=128, r=2,
    tau_ca=0.25, topk=16, dtype="bf16")

CONFIGS: Dict[str, LayerConfig] = {c.name: c for c in (TINY_FP32, WAN13B_LAYER, HUNYUAN720P_LAYER)}


# ----------------------------------------------------------------------------------
# the drifting-mixture generator
# ----------------------------------------------------------------------------------

class DriftingMixture:
    """Stateful per-head generator of frames for one rollout.

    Streams (all derived from one SeedSequence):
      * per head, a "static" stream: centroids, then cluster means, then the prompt;
      * per head, a "frame" stream: frame-0 clusters and noise, then per frame the
        drift noise, the re-drawn clusters and noise, query noise and values;
      * one shared stream for the re-drawn positions (shared by all heads).
    """

    def __init__(self, cfg: LayerConfig, seed: int = 0):
        self.cfg = cfg
        ss = np.random.SeedSequence(seed)
        kids = ss.spawn(2 * cfg.H + 1)
        self._static = [np.random.default_rng(k) for k in kids[: cfg.H]]
        self._frames = [np.random.default_rng(k) for k in kids[cfg.H: 2 * cfg.H]]
        self._pos = np.random.default_rng(kids[-1])
        H, d, B, C, P = cfg.H, cfg.d, cfg.B, cfg.C, cfg.P
        self._centroids = np.empty((H, B, d), np.float32)
        self._means = np.empty((H, C, d), np.float32)
        self._kp = np.empty((H, P, d), np.float32)
        self._vp = np.empty((H, P, d), np.float32)
        for h in range(H):
            g = self._static[h]
            c = g.standard_normal((B, d), dtype=np.float32)
            self._centroids[h] = c / np.linalg.norm(c, axis=1, keepdims=True)
            m = g.standard_normal((C, d), dtype=np.float32)
            self._means[h] = m / np.linalg.norm(m, axis=1, keepdims=True)
            self._kp[h] = g.standard_normal((P, d), dtype=np.float32) / np.float32(np.sqrt(d))
            self._vp[h] = g.standard_normal((P, d), dtype=np.float32)
        self._k: Optional[np.ndarray] = None   # unrounded key state [H, Tf, d]
        self.frames_emitted = 0

    # -- storage rounding -----------------------------------------------------------
    def _store(self, x: np.ndarray) -> np.ndarray:
        x = np.array(x, dtype=np.float32, copy=True)        # never alias the key state
        return bf16_round(x) if self.cfg.dtype == "bf16" else x

    # -- static inputs --------------------------------------------------------------
    @property
    def centroids(self) -> np.ndarray:
        """[H, B, d] unit centroids (rounded to the storage type)."""
        return self._store(self._centroids)

    @property
    def prompt(self):
        """(Kp, Vp), each [H, P, d]."""
        return self._store(self._kp), self._store(self._vp)

    # -- frames ----------------------------------------------------------------------
    def next_frame(self):
        """Advance one latent frame; return (K, V, Q), each [H, Tf, d]."""
        cfg = self.cfg
        H, Tf, d = cfg.H, cfg.Tf, cfg.d
        if self._k is None:
            k = np.empty((H, Tf, d), np.float32)
            for h in range(H):
                g = self._frames[h]
                cl = g.integers(0, cfg.C, size=Tf)
                k[h] = self._means[h][cl] + np.float32(cfg.sigma_mix) * g.standard_normal((Tf, d), dtype=np.float32)
            self._k = k
        else:
            nres = int(round(cfg.rho * Tf))
            pos = self._pos.choice(Tf, size=nres, replace=False) if nres > 0 else np.zeros(0, np.int64)
            for h in range(H):
                g = self._frames[h]
                self._k[h] += np.float32(cfg.drift) * g.standard_normal((Tf, d), dtype=np.float32)
                cl = g.integers(0, cfg.C, size=nres)
                self._k[h][pos] = self._means[h][cl] + np.float32(cfg.sigma_mix) * g.standard_normal((nres, d), dtype=np.float32)
        q = np.empty((H, Tf, d), np.float32)
        v = np.empty((H, Tf, d), np.float32)
        for h in range(H):
            g = self._frames[h]
            q[h] = self._k[h] + np.float32(cfg.qnoise) * g.standard_normal((Tf, d), dtype=np.float32)
            v[h] = g.standard_normal((Tf, d), dtype=np.float32)
        self.frames_emitted += 1
        return self._store(self._k), self._store(v), self._store(q)

    def next_chunk(self):
        """Advance F frames; return (K, V, Q), each [H, F*Tf, d], frame-major."""
        ks, vs, qs = [], [], []
        for _ in range(self.cfg.F):
            k, v, q = self.next_frame()
            ks.append(k)
            vs.append(v)
            qs.append(q)
        return (np.concatenate(ks, axis=1), np.concatenate(vs, axis=1), np.concatenate(qs, axis=1))


def pq_codebooks(keys: np.ndarray, m: int, Kc: int, seed: int = 0, dtype: str = "bf16") -> np.ndarray:
    """Product-quantization codebooks [H, m, Kc, d/m] drawn from data: per head and
    sub-space, the sub-vectors of Kc distinct rows of `keys` [H, n, d] picked at random
    (a common codebook initialisation; no training)."""
    H, n, d = keys.shape
    ds = d // m
    rng = np.random.default_rng(seed)
    cb = np.empty((H, m, Kc, ds), np.float32)
    for h in range(H):
        for s in range(m):
            rows = rng.choice(n, size=Kc, replace=False)
            cb[h, s] = keys[h, rows, s * ds:(s + 1) * ds]
    return bf16_round(cb) if dtype == "bf16" else cb


def layer_step_inputs(cfg: LayerConfig, seed: int = 0, prior_frames: Optional[int] = None) -> dict:
    """Inputs of one layer step after `prior_frames` frames of history.

    Returns a dict of float32 arrays (bf16-exact for bf16 configs):
      history_k, history_v  [H, prior*Tf, d]  every past key/value, oldest first
      q, k_cur, v_cur       [H, Nq, d]        the current chunk, frame-major
      centroids             [H, B, d]
      kp, vp                [H, P, d]
    """
    pf = cfg.prior_frames if prior_frames is None else prior_frames
    gen = DriftingMixture(cfg, seed)
    hk, hv = [], []
    for _ in range(pf):
        k, v, _q = gen.next_frame()
        hk.append(k)
        hv.append(v)
    q_list, k_list, v_list = [], [], []
    for _ in range(cfg.F):
        k, v, q = gen.next_frame()
        k_list.append(k)
        v_list.append(v)
        q_list.append(q)
    H, d = cfg.H, cfg.d
    empty = np.zeros((H, 0, d), np.float32)
    kp, vp = gen.prompt
    return dict(
        history_k=np.concatenate(hk, axis=1) if hk else empty,
        history_v=np.concatenate(hv, axis=1) if hv else empty,
        q=np.concatenate(q_list, axis=1),
        k_cur=np.concatenate(k_list, axis=1),
        v_cur=np.concatenate(v_list, axis=1),
        centroids=gen.centroids,
        kp=kp,
        vp=vp,
    )
