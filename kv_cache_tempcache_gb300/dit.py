"""A Wan2.1-1.3B-shaped diffusion transformer with random weights around the FAST-AR
attention step, for whole-chunk denoising on one GPU.

The pages describe FAST-AR as a drop-in replacement for the attention layers of an
autoregressive video diffusion transformer (technical summary, Key Results: Rolling-
Forcing / LongVie2 on Wan-family backbones).  This module supplies that transformer's
shape so that a chunk can be denoised end to end: every block is
    h  = LN(x) * (1 + scale1) + shift1                      (adaLN)
    q, k, v = h W_qkv^T + b;  q, k <- RMSNorm, rotary positions (frame, row, column)
    x += gate1 * (SelfAttn(q, k, v) W_o^T + b)               (FAST-AR: TempCache + AnnSA, or dense)
    x += CrossAttn(RMSNorm(LN_affine(x) W_q^T + b), text) W_o^T + b   (FAST-AR: AnnCA, or dense)
    x += gate2 * (GELU(LN(x) * (1 + scale2) + shift2) W_1^T + b) W_2^T + b)
with (shift, scale, gate) x 2 = the block's modulation + a projection of the timestep
embedding; the head is LN + modulation + a linear map to the latent patch channels.
Latents live in patch-token layout ([tokens, 16 channels x 1 x 2 x 2 = 64], rows padded
to 256 channels), so patchifying is a layout, not a kernel; the flow-matching Euler step
x <- x + (t_next - t) v is the head GEMM's gated-residual epilogue.

Every operation runs in libfastar's kernels (GEMMs on the tensor cores, row kernels,
the attention step); PyTorch supplies memory, random initialisation at set-up, and the
CUDA graphs that replay one denoising step (one graph per cache half).
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import torch

from . import _lib as L
from .layer import DenseLayer, FastARLayer


@dataclasses.dataclass(frozen=True)
class DiTConfig:
    dim: int = 1536
    heads: int = 12
    ffn: int = 8960
    layers: int = 30
    freq_dim: int = 256
    text_dim: int = 4096
    text_len: int = 512
    patch_ch: int = 64          # 16 latent channels x 1 x 2 x 2
    frames: int = 3             # latent frames per chunk
    grid_h: int = 30
    grid_w: int = 52
    steps: int = 4              # denoising steps per chunk
    eps: float = 1e-6
    theta: float = 10000.0
    # FAST-AR attention (the Wan-1.3B layer of the benchmark)
    M: int = 9360
    B: int = 64
    r: int = 2
    tau: float = 0.95
    tau_ca: float = 0.2
    topk: int = 16
    name: str = "wan13b_dit"

    @property
    def d(self) -> int:
        return self.dim // self.heads

    @property
    def tokens(self) -> int:
        return self.frames * self.grid_h * self.grid_w

    def replace(self, **kw) -> "DiTConfig":
        return dataclasses.replace(self, **kw)


WAN13B_DIT = DiTConfig()
LAT_LD = 256    # padded row length of the latent buffer (the head GEMM's N)


def timesteps(steps: int) -> List[float]:
    """Flow-matching times of a chunk's denoising steps, from 1 (noise) to 0."""
    return [1.0 - i / steps for i in range(steps + 1)]


class _Block:
    pass


class DiT:
    """Parameters, buffers and the denoising step of the transformer.  attention is
    "fastar" (TempCache + AnnSA + AnnCA per block) or "dense" (append-only caches)."""

    def __init__(self, cfg: DiTConfig, attention: str = "fastar", seed: int = 0, device="cuda",
                 dense_capacity: int = 0):
        L.load()
        if cfg.dim % 256 or cfg.ffn % 256 or cfg.text_dim % 64 or cfg.dim % cfg.heads:
            raise ValueError("dimensions must suit the GEMM tiles (multiples of 256 / 64)")
        self.cfg, self.attention = cfg, attention
        dev = torch.device(device)
        self.dev = dev
        # random initialisation on the device (a seeded generator there)
        g = torch.Generator(device=dev).manual_seed(seed)
        bf = torch.bfloat16

        def w(n, k):      # a Linear weight [n, k], N(0, 1/k), bf16
            return (torch.randn(n, k, generator=g, device=dev) / math.sqrt(k)).to(bf)

        def vec(n, s=0.02):
            return torch.randn(n, generator=g, device=dev) * s

        D, N = cfg.dim, cfg.tokens
        self.patch_w = torch.zeros(D, LAT_LD, dtype=bf, device=dev)
        self.patch_w[:, :cfg.patch_ch] = w(D, cfg.patch_ch)
        self.patch_b = vec(D)
        self.time_w1, self.time_b1 = w(D, cfg.freq_dim), vec(D)
        self.time_w2, self.time_b2 = w(D, D), vec(D)
        self.proj_w, self.proj_b = w(6 * D, D), vec(6 * D)
        self.text_w1, self.text_b1 = w(D, cfg.text_dim), vec(D)
        self.text_w2, self.text_b2 = w(D, D), vec(D)
        self.blocks = []
        for _ in range(cfg.layers):
            b = _Block()
            b.mod = torch.randn(6, D, generator=g, device=dev) / math.sqrt(D)
            b.qkv_w, b.qkv_b = w(3 * D, D), vec(3 * D)
            b.norm_q, b.norm_k = (1 + vec(D, 0.1)), (1 + vec(D, 0.1))
            b.o_w, b.o_b = w(D, D), vec(D)
            b.norm3_w, b.norm3_b = (1 + vec(D, 0.1)), vec(D)
            b.cq_w, b.cq_b = w(D, D), vec(D)
            b.ck_w, b.ck_b = w(D, D), vec(D)
            b.cv_w, b.cv_b = w(D, D), vec(D)
            b.norm_cq, b.norm_ck = (1 + vec(D, 0.1)), (1 + vec(D, 0.1))
            b.co_w, b.co_b = w(D, D), vec(D)
            b.f1_w, b.f1_b = w(cfg.ffn, D), vec(cfg.ffn)
            b.f2_w, b.f2_b = w(D, cfg.ffn), vec(D)
            self.blocks.append(b)
        self.head_mod = torch.randn(2, D, generator=g, device=dev) / math.sqrt(D)
        self.head_w = torch.zeros(LAT_LD, D, dtype=bf, device=dev)
        self.head_w[:cfg.patch_ch] = w(cfg.patch_ch, D)
        self.head_b = torch.zeros(LAT_LD, dtype=torch.float32, device=dev)
        self.head_b[:cfg.patch_ch] = vec(cfg.patch_ch)
        # buffers
        self.lat = torch.zeros(N, LAT_LD, dtype=bf, device=dev)
        self.x = torch.zeros(N, D, dtype=bf, device=dev)
        self.h = torch.zeros(N, D, dtype=bf, device=dev)
        self.qkv = torch.zeros(N, 3 * D, dtype=bf, device=dev)
        self.o = torch.zeros(N, D, dtype=bf, device=dev)
        self.qc = torch.zeros(N, D, dtype=bf, device=dev)
        self.f = torch.zeros(N, cfg.ffn, dtype=bf, device=dev)
        self.t_dev = torch.zeros(1, dtype=torch.float32, device=dev)
        self.frame_dev = torch.zeros(1, dtype=torch.int32, device=dev)   # the chunk's first frame
        self.dt_vec = torch.zeros(LAT_LD, dtype=torch.float32, device=dev)
        self.sin = torch.zeros(1, cfg.freq_dim, dtype=bf, device=dev)
        self.e1 = torch.zeros(1, D, dtype=bf, device=dev)
        self.e = torch.zeros(1, D, dtype=torch.float32, device=dev)
        self.e_silu = torch.zeros(1, D, dtype=bf, device=dev)
        self.e0 = torch.zeros(1, 6 * D, dtype=torch.float32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        # attention layers
        H, d = cfg.heads, cfg.d
        if attention == "fastar":
            self.attn = [FastARLayer(H=H, d=d, Tf=cfg.grid_h * cfg.grid_w, F=cfg.frames, M=cfg.M, B=cfg.B, r=cfg.r,
                                     P=cfg.text_len, tau=cfg.tau, tau_ca=cfg.tau_ca, topk=cfg.topk, dtype=bf,
                                     device=dev) for _ in range(cfg.layers)]
            for a in self.attn:
                a.set_centroids(torch.nn.functional.normalize(torch.randn(H, cfg.B, d, generator=g, device=dev),
                                                              dim=-1).to(bf))
        else:
            cap = max(dense_capacity, N)
            self.attn = [DenseLayer(H, d, N, cap, cfg.text_len, dtype=bf, device=dev) for _ in range(cfg.layers)]
        self.frame0 = 0
        self._graphs = {}

    # ---- views ---------------------------------------------------------------------------
    def _heads(self, t2d):
        """[N, H*d] token-major -> [H, N, d] view."""
        N = t2d.shape[0]
        return t2d.view(N, self.cfg.heads, self.cfg.d).transpose(0, 1)

    # ---- set-up ----------------------------------------------------------------------------
    def set_text(self, text: torch.Tensor):
        """Projects the text encoder output [text_len, text_dim] (bf16) to each block's
        cross-attention keys and values (once per rollout)."""
        cfg = self.cfg
        P, D = cfg.text_len, cfg.dim
        t1 = torch.empty(P, D, dtype=torch.bfloat16, device=self.dev)
        ctx = torch.empty(P, D, dtype=torch.bfloat16, device=self.dev)
        L.fastar_gemm(text, self.text_w1, t1, bias=self.text_b1, act=L.ACT_GELU_TANH, dev_status=self.status)
        L.fastar_gemm(t1, self.text_w2, ctx, bias=self.text_b2, dev_status=self.status)
        k = torch.empty(P, D, dtype=torch.bfloat16, device=self.dev)
        v = torch.empty(P, D, dtype=torch.bfloat16, device=self.dev)
        for b, a in zip(self.blocks, self.attn):
            L.fastar_gemm(ctx, b.ck_w, k, bias=b.ck_b, dev_status=self.status)
            L.fastar_rmsnorm_rope(k, cfg.d, weight=b.norm_ck, eps=cfg.eps)
            L.fastar_gemm(ctx, b.cv_w, v, bias=b.cv_b, dev_status=self.status)
            a.set_prompt(self._heads(k).contiguous(), self._heads(v).contiguous())

    # ---- the denoising step ------------------------------------------------------------------
    def _enqueue_step(self, advance: bool, probe=None):
        """One denoising step of the current chunk (reads self.t_dev, self.dt_vec and the
        latent; updates the latent in place).  probe (eager steps only): called as
        probe("self", i, layer, q, k, v, out) after block i's self-attention and
        probe("cross", i, layer, qc, out) after its cross-attention, with [H, N, d] views
        of the block's attention inputs and output, for inspection between kernels."""
        cfg, D, N = self.cfg, self.cfg.dim, self.cfg.tokens
        st = self.status
        # timestep embedding -> e (head) and the blocks' modulation e0
        L.fastar_sinusoidal_embedding(self.t_dev, self.sin)
        L.fastar_gemm(self.sin, self.time_w1, self.e1, bias=self.time_b1, act=L.ACT_SILU, dev_status=st)
        L.fastar_gemm(self.e1, self.time_w2, self.e, bias=self.time_b2, dev_status=st)
        L.fastar_gemm(self.e1, self.time_w2, self.e_silu, bias=self.time_b2, act=L.ACT_SILU, dev_status=st)
        L.fastar_gemm(self.e_silu, self.proj_w, self.e0, bias=self.proj_b, dev_status=st)
        e0 = [self.e0[0, i * D:(i + 1) * D] for i in range(6)]
        # patch embedding (K = 256 padded channels; the padding weights are zero)
        L.fastar_gemm(self.lat, self.patch_w, self.x, bias=self.patch_b, dev_status=st)
        q, k, v = (self._heads(self.qkv[:, i * D:(i + 1) * D]) for i in range(3))
        o = self._heads(self.o)
        for i, (b, a) in enumerate(zip(self.blocks, self.attn)):
            L.fastar_layernorm_mod(self.x, self.h, eps=cfg.eps, shift_a=b.mod[0], shift_b=e0[0], scale_a=b.mod[1],
                                   scale_b=e0[1])
            L.fastar_gemm(self.h, b.qkv_w, self.qkv, bias=b.qkv_b, dev_status=st)
            L.fastar_rmsnorm_rope(self.qkv[:, :D], cfg.d, weight=b.norm_q, rope=True, t0_dev=self.frame_dev,
                                  grid=(cfg.grid_h, cfg.grid_w), eps=cfg.eps, theta=cfg.theta)
            L.fastar_rmsnorm_rope(self.qkv[:, D:2 * D], cfg.d, weight=b.norm_k, rope=True, t0_dev=self.frame_dev,
                                  grid=(cfg.grid_h, cfg.grid_w), eps=cfg.eps, theta=cfg.theta)
            a.step_self(q, k, v, out=o, advance=advance)
            if probe is not None:
                probe("self", i, a, q, k, v, o)
            L.fastar_gemm(self.o, b.o_w, self.x, bias=b.o_b, R=self.x, gate_a=b.mod[2], gate_b=e0[2], dev_status=st)
            L.fastar_layernorm_mod(self.x, self.h, eps=cfg.eps, weight=b.norm3_w, bias=b.norm3_b)
            L.fastar_gemm(self.h, b.cq_w, self.qc, bias=b.cq_b, dev_status=st)
            L.fastar_rmsnorm_rope(self.qc, cfg.d, weight=b.norm_cq, eps=cfg.eps)
            a.step_cross(self._heads(self.qc), out=o)
            if probe is not None:
                probe("cross", i, a, self._heads(self.qc), o)
            L.fastar_gemm(self.o, b.co_w, self.x, bias=b.co_b, R=self.x, dev_status=st)
            L.fastar_layernorm_mod(self.x, self.h, eps=cfg.eps, shift_a=b.mod[3], shift_b=e0[3], scale_a=b.mod[4],
                                   scale_b=e0[4])
            L.fastar_gemm(self.h, b.f1_w, self.f, bias=b.f1_b, act=L.ACT_GELU_TANH, dev_status=st)
            L.fastar_gemm(self.f, b.f2_w, self.x, bias=b.f2_b, R=self.x, gate_a=b.mod[5], gate_b=e0[5],
                          dev_status=st)
        # head: LN + modulation (its own table + e), velocity, Euler update of the latent
        L.fastar_layernorm_mod(self.x, self.h, eps=cfg.eps, shift_a=self.head_mod[0], shift_b=self.e[0],
                               scale_a=self.head_mod[1], scale_b=self.e[0])
        L.fastar_gemm(self.h, self.head_w, self.lat, bias=self.head_b, R=self.lat, gate_a=self.dt_vec, dev_status=st)

    def set_time(self, t: float, t_next: float):
        self.t_dev.fill_(float(t) * 1000.0)          # the embedding sees t in [0, 1000]
        self.dt_vec.fill_(float(t_next) - float(t))

    def step(self, t: float, t_next: float, commit: bool):
        """One denoising step, eagerly (FAST-AR: the caches advance only when commit)."""
        self.set_time(t, t_next)
        self._enqueue_step(advance=False)
        if commit:
            self._commit()

    def _commit(self):
        cfg = self.cfg
        for a in self.attn:
            if self.attention == "fastar":
                a.cur = 1 - a.cur
            else:
                a.n += cfg.tokens
        self.frame0 += cfg.frames
        self.frame_dev.fill_(self.frame0)

    # ---- graphs ----------------------------------------------------------------------------------
    def _graph_key(self):
        if self.attention == "fastar":
            return ("fastar", self.attn[0].cur)
        return ("dense", self.attn[0].n)

    def capture(self):
        """The current denoising step as a CUDA graph (FAST-AR: one per cache half, kept;
        dense: one per cache length)."""
        key = self._graph_key()
        if key in self._graphs:
            return self._graphs[key]
        torch.cuda.synchronize(self.dev)
        s = torch.cuda.Stream(device=self.dev)
        s.wait_stream(torch.cuda.current_stream(self.dev))
        saved = self.lat.clone()
        with torch.cuda.stream(s):
            self._enqueue_step(advance=False)          # warm-up outside the capture
        torch.cuda.synchronize(self.dev)
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=s):
            self._enqueue_step(advance=False)
        torch.cuda.synchronize(self.dev)
        self.lat.copy_(saved)
        if self.attention == "dense":
            self._graphs = {}                          # the dense graph is only good for this length
        self._graphs[key] = gr
        return gr

    def denoise_chunk(self, noise: torch.Tensor, use_graph: bool = True, timer=None, probe=None):
        """Denoises one chunk from noise (patch-token layout [tokens, 64]) in cfg.steps
        Euler steps, commits its keys and values to the caches, and returns the latent.
        probe: see _enqueue_step (eager steps only)."""
        cfg = self.cfg
        if probe is not None and use_graph:
            raise ValueError("a probe needs eager steps (use_graph=False)")
        self.lat.zero_()
        self.lat[:, :cfg.patch_ch].copy_(noise)
        ts = timesteps(cfg.steps)
        gr = self.capture() if use_graph else None
        for i in range(cfg.steps):
            self.set_time(ts[i], ts[i + 1])
            if timer:
                timer("begin")
            if gr is not None:
                gr.replay()
            else:
                self._enqueue_step(advance=False, probe=probe)
            if timer:
                timer("end")
        self._commit()
        return self.lat[:, :cfg.patch_ch]

    def status_word(self) -> int:
        st = int(self.status.item())
        for a in self.attn:
            if self.attention == "fastar":
                st |= a.status()
        return st
