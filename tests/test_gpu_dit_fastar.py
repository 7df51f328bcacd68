"""GPU parity of FAST-AR inside the DiT at non-trivial settings (16 buckets, r = 2,
tau = 0.95, tau_ca = 0.2, a cache cap that drops entries from the third chunk on),
through the C ABI.

Every block's attention step is checked on the GPU's own inputs (its q, k, v, its
incoming cache, its cross-attention queries and text keys/values), stage by stage, with
the layer tests' rules: bucket ids, top-1 indices, eviction flags and kept-prompt sets
must be correct answers under the near-tie margin; the compaction is exact given the
flags; the attention outputs are within the bf16 tolerance of the oracle evaluated on
those validated choices.  Then the whole rollout is compared with the oracle's DiT run
on the same validated choices (replayed): its bf16 GEMMs and row operations make the
continuous values differ slightly, so the discrete choices are replayed, never
recomputed, and the latent update must be within 4 % of its norm, a comparison that a
missing rotary map visibly fails.  The near-tie counts are reported."""
import numpy as np
import pytest
import torch

import parity
from kv_cache_tempcache_gb300 import synth
from kv_cache_tempcache_gb300.dit import DiT, DiTConfig, timesteps
from oracle import dit_oracle as D
from oracle import fastar_oracle as O

pytestmark = pytest.mark.gpu

CFG = DiTConfig(dim=256, heads=2, ffn=512, layers=2, text_dim=256, text_len=64, frames=2, grid_h=4, grid_w=20,
                steps=2, M=320, B=16, r=2, tau=0.95, tau_ca=0.2, topk=16, name="dit_small_fastar")


def _np(t):
    return t.detach().float().contiguous().cpu().numpy().astype(np.float64)


def _i(t):
    return t.detach().contiguous().cpu().numpy().astype(np.int64)


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


class Recorder:
    """Copies every block's attention inputs, decisions and outputs between kernels."""

    def __init__(self):
        self.rec = []

    def __call__(self, kind, i, a, *t):
        if kind == "self":
            q, k, v, o = t
            cin, cout = a.caches[a.cur], a.caches[1 - a.cur]
            self.rec.append(dict(block=i, q=_np(q), k=_np(k), v=_np(v), o_self=_np(o), qb=_i(a.qb),
                                 kb_cur=_i(a.kb_cur)[..., 0], top1=_i(a.top1), evict=_i(a.evict),
                                 imap=_i(a.index_map), len_in=_i(cin.len), len_out=_i(cout.len), ck=_np(cin.k),
                                 cv=_np(cin.v), ckb=_i(cin.kb)[..., 0], status=a.status()))
        else:
            qc, o = t
            r = self.rec[-1]
            assert r["block"] == i
            r.update(qc=_np(qc), o_cross=_np(o), qb_c=_i(a.qb), pb=_i(a.pb)[..., 0], keep=_i(a.keep),
                     kidx=_i(a.kidx), kcnt=_i(a.kcnt), score=_np(a.score), kp=_np(a.kp), vp=_np(a.vp))


def _check_block(r, C, cfg, counts):
    """All stage checks of one block's attention step, head by head, on the GPU's inputs."""
    assert r["status"] == 0
    H, d, F, Tf, M = cfg.heads, cfg.d, cfg.frames, cfg.grid_h * cfg.grid_w, cfg.M
    scale = 1.0 / np.sqrt(d)
    tol = parity.TOL["bf16"]
    for h in range(H):
        q, k, v = r["q"][h], r["k"][h], r["v"][h]
        nq, n = q.shape[0], int(r["len_in"][h])
        ck, cv, ckb = r["ck"][h][:n], r["cv"][h][:n], r["ckb"][h][:n]
        counts["topr"] += parity.check_topr(O.centroid_scores(q, C[h]), r["qb"][h], "self query buckets")
        counts["key"] += parity.check_argmax(O.centroid_scores(k, C[h]), r["kb_cur"][h], "current key buckets")
        top1 = r["top1"][h]
        if n:
            counts["key"] += parity.check_argmax(O.centroid_scores(ck, C[h]), ckb, "cache key buckets")
            counts["top1"] += parity.check_argmax(O.cosine_matrix(q, ck), top1, "tempcache top-1")
            counts["evict"] += parity.check_evict(O.cosine_rows(k, ck[top1]), top1, r["evict"][h], n, cfg.tau)
        else:
            assert np.all(top1 == -1)
        e = r["evict"][h][:n].astype(bool)
        counts["evicted"] += int(e.sum())
        imap, length = O.compact_plan(e, n, nq, M)
        counts["dropped"] += n - int(e.sum()) + nq - length
        assert int(r["len_out"][h]) == length
        assert np.array_equal(r["imap"][h], imap), "index map"
        new_k, new_v = O.gather_rows(imap, length, ck, k), O.gather_rows(imap, length, cv, v)
        new_kb = O.gather_rows(imap, length, ckb, r["kb_cur"][h])
        o, _, n_empty = O.annsa_attention(q, r["qb"][h], new_k, new_v, new_kb, scale)
        counts["empty"] += n_empty
        parity.close(r["o_self"][h], o, *tol, f"o_self block {r['block']} head {h}")
        # AnnCA on the block's own cross-attention queries
        qc, kp, vp = r["qc"][h], r["kp"][h], r["vp"][h]
        counts["topr"] += parity.check_topr(O.centroid_scores(qc, C[h]), r["qb_c"][h], "cross query buckets")
        counts["key"] += parity.check_argmax(O.centroid_scores(kp, C[h]), r["pb"][h], "text key buckets")
        _, _, _, score_o = O.annca_select(qc, r["qb_c"][h], kp, r["pb"][h], F, Tf, cfg.tau_ca, cfg.topk)
        fin = np.isfinite(score_o)
        assert np.array_equal(np.isfinite(r["score"][h]), fin), "AnnCA gating"
        np.testing.assert_allclose(r["score"][h][fin], score_o[fin], rtol=0, atol=2e-5)
        kept = []
        for f in range(F):
            counts["keep"] += parity.check_keep(score_o[f], r["keep"][h][f], cfg.tau_ca, cfg.topk, f"keep frame {f}")
            idx = np.flatnonzero(r["keep"][h][f])
            assert int(r["kcnt"][h][f]) == len(idx)
            assert np.array_equal(r["kidx"][h][f][:len(idx)], idx)
            kept.append(idx)
            counts["kept"] += len(idx)
        oc, _ = O.cross_attention_subset(qc, kp, vp, kept, F, Tf, scale)
        parity.close(r["o_cross"][h], oc, *tol, f"o_cross block {r['block']} head {h}")


def _decisions(recs, cfg):
    """The validated discrete choices of one denoising step, per block, for replay."""
    out = []
    for r in recs:
        n = r["len_in"]
        out.append({"self": [dict(qb=r["qb"][h], kb_cur=r["kb_cur"][h], top1=r["top1"][h],
                                  evict=r["evict"][h][:int(n[h])].astype(bool)) for h in range(cfg.heads)],
                    "cross": [dict(qb=r["qb_c"][h], pb=r["pb"][h], keep=r["keep"][h].astype(bool))
                              for h in range(cfg.heads)]})
    return out


def _rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


@pytest.mark.parametrize("tau", [0.95, 0.6])
def test_dit_fastar_blocks_and_rollout_match_the_oracle(tau):
    # tau = 0.95 is the benchmarked setting; at 0.6 the random-weight transformer's keys of
    # consecutive chunks are similar enough that entries are evicted as well as dropped
    cfg = CFG.replace(tau=tau)
    rng = np.random.default_rng(22)
    dit = DiT(cfg, "fastar", seed=5)
    for b in dit.blocks:          # self-attention at full strength in the residual stream
        b.mod[2] += 1.0
    text = synth.bf16_round(rng.standard_normal((cfg.text_len, cfg.text_dim)).astype(np.float32))
    dit.set_text(torch.from_numpy(text).cuda().to(torch.bfloat16))
    p = _params(dit)
    ctx = D.text_context(p, text)
    text_kv = [D.block_text_kv(b, ctx, cfg.d, cfg.eps) for b in p["blocks"]]
    cents = [_np(a.centroids) for a in dit.attn]
    fa = D.FastARAttention(cents, F=cfg.frames, Tf=cfg.grid_h * cfg.grid_w, M=cfg.M, r=cfg.r, tau=cfg.tau,
                           tau_ca=cfg.tau_ca, topk=cfg.topk)
    fa_norope = D.FastARAttention(cents, F=cfg.frames, Tf=cfg.grid_h * cfg.grid_w, M=cfg.M, r=cfg.r, tau=cfg.tau,
                                  tau_ca=cfg.tau_ca, topk=cfg.topk)
    counts = dict(topr=0, key=0, top1=0, evict=0, keep=0, empty=0, evicted=0, dropped=0, kept=0)
    ts = timesteps(cfg.steps)
    base = rng.standard_normal((cfg.tokens, cfg.patch_ch)).astype(np.float32)
    for chunk in range(3):
        # chunks that resemble one another, as consecutive video chunks do
        noise = synth.bf16_round(base + 0.3 * rng.standard_normal(base.shape).astype(np.float32))
        rec = Recorder()
        out = dit.denoise_chunk(torch.from_numpy(noise).cuda().to(torch.bfloat16), use_graph=False, probe=rec)
        torch.cuda.synchronize()
        assert dit.status_word() == 0
        assert len(rec.rec) == cfg.steps * cfg.layers
        for r in rec.rec:
            _check_block(r, cents[r["block"]], cfg, counts)
        got = _np(out)
        lat, lat_norope = noise.astype(np.float64), noise.astype(np.float64)
        for s in range(cfg.steps):
            dec = _decisions(rec.rec[s * cfg.layers:(s + 1) * cfg.layers], cfg)
            for i, blk in enumerate(dec):   # the oracle's caches are the GPU's lengths
                for h in range(cfg.heads):
                    assert fa.caches[i][h][0].shape[0] == len(blk["self"][h]["evict"])
            lat, caches = D.dit_step(p, cfg, lat, ts[s], ts[s + 1], chunk * cfg.frames, None, text_kv, fastar=fa,
                                     decisions=dec)
            lat_norope, caches_nr = D.dit_step(p, cfg, lat_norope, ts[s], ts[s + 1], chunk * cfg.frames, None,
                                               text_kv, rope_on=False, fastar=fa_norope, decisions=dec)
        fa.caches, fa_norope.caches = caches, caches_nr
        err = _rel(got - noise, lat - noise)
        wrong = _rel(lat_norope - noise, lat - noise)
        assert err < 4e-2, f"chunk {chunk}: relative error {err:.3e}"
        assert wrong > 3 * err, f"the comparison cannot tell a missing rotary map ({wrong:.3e} vs {err:.3e})"
    assert counts["dropped"] > 0, "the cache cap was never reached"
    if tau < 0.9:
        assert counts["evicted"] > 0, "nothing was evicted"
    parity.report(f"DiT FAST-AR (B=16, r=2, tau={tau}; 3 chunks x 2 steps x 2 blocks x 2 heads)", counts)
