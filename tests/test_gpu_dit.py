"""GPU parity of the DiT around the attention step (the Wan-1.3B-shaped transformer with
random weights) against the oracle's denoising step, through the C ABI: two chunks (the
second attends to the first through the cache), two denoising steps each, eager and as
replayed CUDA graphs, with FAST-AR attention in its textbook reduction (one bucket,
r = 1, tau > 1, tau_ca = -1, no FIFO drop: exactly dense attention, so no discrete
decision can differ) and with the dense path.

Tolerance: every GEMM and row operation rounds its output to bf16 (relative 2^-9), about
a dozen times per block along the residual stream, and the latent is stored in bf16
between steps; the update (latent - noise) must be within 4 % of its norm (relative
Frobenius) and the same comparison must rule out a plausible mistake (the rotary
positions left out), which moves the update by several times that (the test opens the
self-attention gate, so that attention carries weight in the output)."""
import numpy as np
import pytest
import torch

from kv_cache_tempcache_gb300 import synth
from kv_cache_tempcache_gb300.dit import DiT, DiTConfig, timesteps
from oracle import dit_oracle as D

pytestmark = pytest.mark.gpu

SMALL = DiTConfig(dim=256, heads=2, ffn=512, layers=2, text_dim=256, text_len=64, frames=2, grid_h=4, grid_w=20,
                  steps=2, M=512, B=1, r=1, tau=2.0, tau_ca=-1.0, topk=16, name="dit_small")


def _np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _params(dit):
    c = dit.cfg
    p = dict(time_w1=_np(dit.time_w1), time_b1=_np(dit.time_b1), time_w2=_np(dit.time_w2), time_b2=_np(dit.time_b2),
             proj_w=_np(dit.proj_w), proj_b=_np(dit.proj_b), text_w1=_np(dit.text_w1), text_b1=_np(dit.text_b1),
             text_w2=_np(dit.text_w2), text_b2=_np(dit.text_b2), patch_w=_np(dit.patch_w[:, :c.patch_ch]),
             patch_b=_np(dit.patch_b), head_mod=_np(dit.head_mod), head_w=_np(dit.head_w[:c.patch_ch]),
             head_b=_np(dit.head_b[:c.patch_ch]))
    keys = ["mod", "qkv_w", "qkv_b", "norm_q", "norm_k", "o_w", "o_b", "norm3_w", "norm3_b", "cq_w", "cq_b", "ck_w",
            "ck_b", "cv_w", "cv_b", "norm_cq", "norm_ck", "co_w", "co_b", "f1_w", "f1_b", "f2_w", "f2_b"]
    p["blocks"] = [{k: _np(getattr(b, k)) for k in keys} for b in dit.blocks]
    return p


def _rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


@pytest.mark.parametrize("attention", ["fastar", "dense"])
def test_dit_chunks_match_the_oracle(attention):
    cfg = SMALL
    rng = np.random.default_rng(21)
    dit = DiT(cfg, attention, seed=3, dense_capacity=2 * cfg.tokens)
    for b in dit.blocks:          # self-attention at full strength in the residual stream
        b.mod[2] += 1.0
    text = synth.bf16_round(rng.standard_normal((cfg.text_len, cfg.text_dim)).astype(np.float32))
    dit.set_text(torch.from_numpy(text).cuda().to(torch.bfloat16))
    p = _params(dit)
    ctx = D.text_context(p, text)
    text_kv = [D.block_text_kv(b, ctx, cfg.d, cfg.eps) for b in p["blocks"]]
    hist = [(np.zeros((0, cfg.dim)), np.zeros((0, cfg.dim)))] * cfg.layers
    ts = timesteps(cfg.steps)
    for chunk, use_graph in ((0, False), (1, True)):
        noise = synth.bf16_round(rng.standard_normal((cfg.tokens, cfg.patch_ch)).astype(np.float32))
        out = dit.denoise_chunk(torch.from_numpy(noise).cuda().to(torch.bfloat16), use_graph=use_graph)
        torch.cuda.synchronize()
        assert dit.status_word() == 0
        got = _np(out)
        lat, lat_norope = noise.astype(np.float64), noise.astype(np.float64)
        for i in range(cfg.steps):
            lat, kv = D.dit_step(p, cfg, lat, ts[i], ts[i + 1], chunk * cfg.frames, hist, text_kv)
            lat_norope, _ = D.dit_step(p, cfg, lat_norope, ts[i], ts[i + 1], chunk * cfg.frames, hist, text_kv,
                                       rope_on=False)
        err = _rel(got - noise, lat - noise)
        wrong = _rel(lat_norope - noise, lat - noise)
        assert err < 4e-2, f"chunk {chunk}: relative error {err:.3e}"
        assert wrong > 3 * err, f"the comparison cannot tell a missing rotary map ({wrong:.3e} vs {err:.3e})"
        hist = [(np.concatenate([hk, k]), np.concatenate([hv, v])) for (hk, hv), (k, v) in zip(hist, kv)]
