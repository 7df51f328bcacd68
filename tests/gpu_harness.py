"""Runs one FAST-AR layer step through the C ABI on the GPU and checks every stage
against the CPU oracle (see parity.py for the comparison rules)."""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

from kv_cache_tempcache_gb300 import synth
from kv_cache_tempcache_gb300.layer import FastARLayer, DenseLayer
from oracle import fastar_oracle as O
import parity


def torch_dtype(cfg):
    return torch.bfloat16 if cfg.dtype == "bf16" else torch.float32


def to_dev(x, cfg, dev="cuda"):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(dev).to(torch_dtype(cfg))


def raw_window(inputs, cfg):
    """The most recent min(M, history) history entries as a cache (oldest first)."""
    hk, hv = inputs["history_k"], inputs["history_v"]
    n = min(cfg.M, hk.shape[1])
    return hk[:, hk.shape[1] - n:], hv[:, hv.shape[1] - n:]


def make_layer(cfg, gate=True, diagnostics=True):
    return FastARLayer(H=cfg.H, d=cfg.d, Tf=cfg.Tf, F=cfg.F, M=cfg.M, B=cfg.B, r=cfg.r, P=cfg.P, tau=cfg.tau,
                       tau_ca=cfg.tau_ca, topk=cfg.topk, dtype=torch_dtype(cfg), gate=gate,
                       diagnostics=diagnostics)


def np_(t):
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.detach().cpu().numpy()


def gpu_step(cfg, inputs, cache_k, cache_v, gate=True, q_layout="HND", diagnostics=True):
    """Runs one step; returns a dict of every GPU intermediate as NumPy."""
    layer = make_layer(cfg, gate, diagnostics)
    layer.set_centroids(to_dev(inputs["centroids"], cfg))
    layer.set_prompt(to_dev(inputs["kp"], cfg), to_dev(inputs["vp"], cfg))
    layer.load_cache(to_dev(cache_k, cfg), to_dev(cache_v, cfg))
    if q_layout == "NHD":   # [N, H, d] storage, viewed as [H, N, d]
        q = to_dev(inputs["q"].transpose(1, 0, 2), cfg).transpose(0, 1)
        k = to_dev(inputs["k_cur"].transpose(1, 0, 2), cfg).transpose(0, 1)
        v = to_dev(inputs["v_cur"].transpose(1, 0, 2), cfg).transpose(0, 1)
    else:
        q, k, v = (to_dev(inputs[x], cfg) for x in ("q", "k_cur", "v_cur"))
    cin, cout = layer.caches[layer.cur], layer.caches[1 - layer.cur]
    kb_in = np_(cin.kb)[..., 0].copy()
    knorm_in = np_(cin.knorm).copy()
    layer.step(q, k, v, advance=False)
    torch.cuda.synchronize()
    out = dict(
        qb=np_(layer.qb), kb_cur=np_(layer.kb_cur)[..., 0], kcur_norm=np_(layer.kcur_norm), kb_in=kb_in,
        knorm_in=knorm_in, pb=np_(layer.pb)[..., 0], top1=np_(layer.top1), s1=np_(layer.s1), s2=np_(layer.s2) if diagnostics else None,
        evict=np_(layer.evict), index_map=np_(layer.index_map), len_out=np_(cout.len), k_out=np_(cout.k),
        v_out=np_(cout.v), kb_out=np_(cout.kb)[..., 0], knorm_out=np_(cout.knorm), kperm=np_(layer.kperm),
        koff=np_(layer.koff), qperm=np_(layer.qperm), qoff=np_(layer.qoff), o_self=np_(layer.o_self),
        lse_self=np_(layer.lse_self), keep=np_(layer.keep), kidx=np_(layer.kidx), kcnt=np_(layer.kcnt),
        score=np_(layer.score), o_cross=np_(layer.o_cross), status=layer.status())
    return out, layer


@dataclasses.dataclass
class Counts:
    topr_ties: int = 0
    key_ties: int = 0
    top1_ties: int = 0
    evict_amb: int = 0
    keep_amb: int = 0
    empty_queries: int = 0


def check_head(cfg, inputs, cache_k, cache_v, g, h, gate=True, counts=None, check_sort=True):
    """All stage checks for head h.  cache_k/cache_v: the cache entering the step."""
    c = counts or Counts()
    tol = parity.TOL[cfg.dtype]
    C = inputs["centroids"][h]
    q, kc, vc = inputs["q"][h], inputs["k_cur"][h], inputs["v_cur"][h]
    ck, cv = cache_k[h], cache_v[h]
    kp, vp = inputs["kp"][h], inputs["vp"][h]
    n, Nq, M, B, r = ck.shape[0], q.shape[0], cfg.M, cfg.B, cfg.r
    # 1. buckets
    c.topr_ties += parity.check_topr(O.centroid_scores(q, C), g["qb"][h], "query buckets")
    c.key_ties += parity.check_argmax(O.centroid_scores(kc, C), g["kb_cur"][h], "current key buckets")
    if n:
        c.key_ties += parity.check_argmax(O.centroid_scores(ck, C), g["kb_in"][h][:n], "cache key buckets")
        np.testing.assert_allclose(g["knorm_in"][h][:n], np.linalg.norm(ck.astype(np.float64), axis=1), rtol=1e-5)
    if cfg.P:
        c.key_ties += parity.check_argmax(O.centroid_scores(kp, C), g["pb"][h], "prompt buckets")
    np.testing.assert_allclose(g["kcur_norm"][h], np.linalg.norm(kc.astype(np.float64), axis=1), rtol=1e-5)
    # 2. match
    top1 = g["top1"][h].astype(np.int64)
    if n:
        S = O.cosine_matrix(q, ck)
        c.top1_ties += parity.check_argmax(S, top1, "tempcache top-1")
        o_top1, o_s1, o_s2 = O.tempcache_match(q, ck)
        np.testing.assert_allclose(g["s1"][h], o_s1, rtol=0, atol=2e-5)
        if g["s2"] is not None:
            fin = np.isfinite(o_s2)
            assert np.array_equal(np.isfinite(g["s2"][h]), fin)
            np.testing.assert_allclose(g["s2"][h][fin], o_s2[fin], rtol=0, atol=2e-5)
    else:
        assert np.all(top1 == -1)
    # 3. eviction (from the GPU's validated top-1)
    if n:
        cos_at = O.cosine_rows(kc, ck[top1])
        c.evict_amb += parity.check_evict(cos_at, top1, g["evict"][h], n, cfg.tau)
    e_gpu = g["evict"][h][:n].astype(bool)
    # 4. compaction: exact given the flags
    imap, L = O.compact_plan(e_gpu, n, Nq, M)
    assert int(g["len_out"][h]) == L
    assert np.array_equal(g["index_map"][h].astype(np.int64), imap), "index map"
    np.testing.assert_array_equal(g["k_out"][h][:L], O.gather_rows(imap, L, ck, kc))
    np.testing.assert_array_equal(g["v_out"][h][:L], O.gather_rows(imap, L, cv, vc))
    kb_new = O.gather_rows(imap, L, g["kb_in"][h][:n], g["kb_cur"][h])
    np.testing.assert_array_equal(g["kb_out"][h][:L], kb_new)
    np.testing.assert_allclose(g["knorm_out"][h][:L], O.gather_rows(imap, L, g["knorm_in"][h][:n], g["kcur_norm"][h]),
                               rtol=0, atol=0)
    # 5. sort (stable counting sort == stable argsort)
    if check_sort:
        koff = np.concatenate([[0], np.cumsum(np.bincount(kb_new, minlength=B))])
        assert np.array_equal(g["koff"][h], koff)
        assert np.array_equal(g["kperm"][h][:L], np.argsort(kb_new, kind="stable"))
        qflat = g["qb"][h].reshape(-1)
        qoff = np.concatenate([[0], np.cumsum(np.bincount(qflat, minlength=B))])
        assert np.array_equal(g["qoff"][h], qoff)
        assert np.array_equal(g["qperm"][h], np.argsort(qflat, kind="stable"))
    # 6. AnnSA attention on the GPU's validated decisions
    new_k = O.gather_rows(imap, L, ck, kc)
    new_v = O.gather_rows(imap, L, cv, vc)
    o, lse, n_empty = O.annsa_attention(q, g["qb"][h], new_k, new_v, kb_new, cfg.scale)
    c.empty_queries += n_empty
    parity.close(g["o_self"][h], o, *tol, f"o_self head {h}")
    fin = np.isfinite(lse)
    assert np.array_equal(np.isfinite(g["lse_self"][h]), fin)
    np.testing.assert_allclose(g["lse_self"][h][fin], lse[fin], rtol=0, atol=1e-3)
    # 7. AnnCA selection
    keep_o, _, _, score_o = O.annca_select(q, g["qb"][h], kp, g["pb"][h], cfg.F, cfg.Tf, cfg.tau_ca, cfg.topk, gate)
    fin = np.isfinite(score_o)
    assert np.array_equal(np.isfinite(g["score"][h]), fin), "AnnCA gating"
    np.testing.assert_allclose(g["score"][h][fin], score_o[fin], rtol=0, atol=2e-5)
    kept = []
    for f in range(cfg.F):
        c.keep_amb += parity.check_keep(score_o[f], g["keep"][h][f], cfg.tau_ca, cfg.topk, f"keep head {h} frame {f}")
        idx = np.flatnonzero(g["keep"][h][f])
        assert int(g["kcnt"][h][f]) == len(idx)
        assert np.array_equal(g["kidx"][h][f][:len(idx)], idx)
        assert np.all(g["kidx"][h][f][len(idx):] == -1)
        kept.append(idx)
    # 8. cross-attention over the GPU's kept sets
    oc, lc = O.cross_attention_subset(q, kp, vp, kept, cfg.F, cfg.Tf, cfg.scale)
    parity.close(g["o_cross"][h], oc, *tol, f"o_cross head {h}")
    return c


def check_head_sampled(cfg, inputs, cache_k, cache_v, g, h, rows, counts=None):
    """check_head for a head whose per-query outputs are checked on the query rows `rows`
    only (top-1 and its score, AnnSA and cross-attention outputs); everything whose oracle
    is cheap at any size stays complete: every bucket id, the eviction flags from the GPU's
    top-1, the compaction, both sorts and the AnnCA selection."""
    c = counts or Counts()
    tol = parity.TOL[cfg.dtype]
    rows = np.asarray(rows)
    C = inputs["centroids"][h]
    q, kc, vc = inputs["q"][h], inputs["k_cur"][h], inputs["v_cur"][h]
    ck, cv = cache_k[h], cache_v[h]
    kp, vp = inputs["kp"][h], inputs["vp"][h]
    n, Nq, M, B = ck.shape[0], q.shape[0], cfg.M, cfg.B
    c.topr_ties += parity.check_topr(O.centroid_scores(q, C), g["qb"][h], "query buckets")
    c.key_ties += parity.check_argmax(O.centroid_scores(kc, C), g["kb_cur"][h], "current key buckets")
    c.key_ties += parity.check_argmax(O.centroid_scores(ck, C), g["kb_in"][h][:n], "cache key buckets")
    c.key_ties += parity.check_argmax(O.centroid_scores(kp, C), g["pb"][h], "prompt buckets")
    # the match on the sampled queries, each against the whole incoming cache
    top1 = g["top1"][h].astype(np.int64)
    c.top1_ties += parity.check_argmax(O.cosine_matrix(q[rows], ck), top1[rows], "tempcache top-1 (sampled)")
    _, o_s1, _ = O.tempcache_match(q[rows], ck)
    np.testing.assert_allclose(g["s1"][h][rows], o_s1, rtol=0, atol=2e-5)
    assert ((top1 >= 0) & (top1 < n)).all()
    # eviction from the GPU's top-1 of every query, then the compaction and the sorts exactly
    c.evict_amb += parity.check_evict(O.cosine_rows(kc, ck[top1]), top1, g["evict"][h], n, cfg.tau)
    e_gpu = g["evict"][h][:n].astype(bool)
    imap, L = O.compact_plan(e_gpu, n, Nq, M)
    assert int(g["len_out"][h]) == L
    assert np.array_equal(g["index_map"][h].astype(np.int64), imap), "index map"
    np.testing.assert_array_equal(g["k_out"][h][:L], O.gather_rows(imap, L, ck, kc))
    np.testing.assert_array_equal(g["v_out"][h][:L], O.gather_rows(imap, L, cv, vc))
    kb_new = O.gather_rows(imap, L, g["kb_in"][h][:n], g["kb_cur"][h])
    np.testing.assert_array_equal(g["kb_out"][h][:L], kb_new)
    koff = np.concatenate([[0], np.cumsum(np.bincount(kb_new, minlength=B))])
    assert np.array_equal(g["koff"][h], koff)
    assert np.array_equal(g["kperm"][h][:L], np.argsort(kb_new, kind="stable"))
    qflat = g["qb"][h].reshape(-1)
    assert np.array_equal(g["qoff"][h], np.concatenate([[0], np.cumsum(np.bincount(qflat, minlength=B))]))
    assert np.array_equal(g["qperm"][h], np.argsort(qflat, kind="stable"))
    # AnnSA on the sampled queries (each over its own buckets' keys of the new cache)
    new_k, new_v = O.gather_rows(imap, L, ck, kc), O.gather_rows(imap, L, cv, vc)
    o, lse, n_empty = O.annsa_attention(q[rows], g["qb"][h][rows], new_k, new_v, kb_new, cfg.scale)
    c.empty_queries += n_empty
    parity.close(g["o_self"][h][rows], o, *tol, f"o_self head {h} (sampled)")
    # the AnnCA selection on every prompt token and frame
    keep_o, _, _, score_o = O.annca_select(q, g["qb"][h], kp, g["pb"][h], cfg.F, cfg.Tf, cfg.tau_ca, cfg.topk, True)
    fin = np.isfinite(score_o)
    assert np.array_equal(np.isfinite(g["score"][h]), fin), "AnnCA gating"
    np.testing.assert_allclose(g["score"][h][fin], score_o[fin], rtol=0, atol=2e-5)
    for f in range(cfg.F):
        c.keep_amb += parity.check_keep(score_o[f], g["keep"][h][f], cfg.tau_ca, cfg.topk, f"keep head {h} frame {f}")
        idx = np.flatnonzero(g["keep"][h][f])
        assert int(g["kcnt"][h][f]) == len(idx)
        assert np.array_equal(g["kidx"][h][f][:len(idx)], idx)
        # cross-attention of the frame's sampled queries over the GPU's kept set
        rf = rows[rows // cfg.Tf == f]
        if len(rf):
            oc, _ = O.cross_attention_subset(q[rf], kp, vp, [idx], 1, len(rf), cfg.scale)
            parity.close(g["o_cross"][h][rf], oc, *tol, f"o_cross head {h} frame {f} (sampled)")
    return c


def check_step(cfg, inputs, cache_k, cache_v, g, heads=None, gate=True):
    assert g["status"] == 0, f"device status {g['status']}"
    counts = Counts()
    for h in (range(cfg.H) if heads is None else heads):
        check_head(cfg, inputs, cache_k, cache_v, g, h, gate, counts)
    return counts


def small_bf16():
    return synth.LayerConfig(name="small_bf16", H=2, d=128, Tf=200, F=3, prior_frames=6, P=100, C=8,
                             sigma_mix=0.3, rho=0.1, drift=0.05, qnoise=0.1, tau=0.95, M=1000, B=16, r=2,
                             tau_ca=0.2, topk=16, dtype="bf16")
