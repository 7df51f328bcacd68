"""GPU parity of the merge variant of TempCache (technical summary §2.A, Theoretical
Basis: Lemma 5.1) against the oracle: the match's owners, the merging compaction, and
attention with the ln g logit shift (bucket-restricted and dense), through the C ABI.

Protocol as for the replace step: the GPU's discrete decisions (buckets, top-1,
eviction, owners) are validated first, up to near-ties; the oracle is then evaluated
on them and the merged cache and the outputs are compared."""
import numpy as np
import pytest
import torch

from kv_cache_tempcache_gb300 import _lib as L, synth
from kv_cache_tempcache_gb300.layer import FastARLayer
from oracle import fastar_oracle as O
import gpu_harness as GH
import parity

pytestmark = pytest.mark.gpu


def _layer(cfg):
    return FastARLayer(H=cfg.H, d=cfg.d, Tf=cfg.Tf, F=cfg.F, M=cfg.M, B=cfg.B, r=cfg.r, P=cfg.P, tau=cfg.tau,
                       tau_ca=cfg.tau_ca, topk=cfg.topk, dtype=GH.torch_dtype(cfg), merge=True)


def _counts(seed, H, n):
    return np.random.default_rng(4000 + seed).integers(1, 6, size=(H, n)).astype(np.int32)


def _merge_step(cfg, inputs, ck, cv, gin):
    layer = _layer(cfg)
    layer.set_centroids(GH.to_dev(inputs["centroids"], cfg))
    layer.set_prompt(GH.to_dev(inputs["kp"], cfg), GH.to_dev(inputs["vp"], cfg))
    layer.load_cache(GH.to_dev(ck, cfg), GH.to_dev(cv, cfg), torch.from_numpy(gin).cuda())
    cin, cout = layer.caches[layer.cur], layer.caches[1 - layer.cur]
    kb_in = GH.np_(cin.kb)[..., 0].copy()
    q, k, v = (GH.to_dev(inputs[x], cfg) for x in ("q", "k_cur", "v_cur"))
    layer.step(q, k, v, advance=False)
    torch.cuda.synchronize()
    return dict(qb=GH.np_(layer.qb), kb_cur=GH.np_(layer.kb_cur)[..., 0], kb_in=kb_in, top1=GH.np_(layer.top1),
                evict=GH.np_(layer.evict), owner=GH.np_(layer.owner), index_map=GH.np_(layer.index_map),
                len_out=GH.np_(cout.len), k_out=GH.np_(cout.k), v_out=GH.np_(cout.v), g_out=GH.np_(cout.g),
                kb_out=GH.np_(cout.kb)[..., 0], o_self=GH.np_(layer.o_self), lse_self=GH.np_(layer.lse_self),
                o_cross=GH.np_(layer.o_cross), status=layer.status())


def _check_head(cfg, inputs, ck, cv, gin, g, h):
    q, kc, vc = inputs["q"][h], inputs["k_cur"][h], inputs["v_cur"][h]
    C = inputs["centroids"][h]
    n, Nq = ck.shape[1], cfg.Nq
    parity.check_topr(O.centroid_scores(q, C), g["qb"][h], "query buckets")
    parity.check_argmax(O.centroid_scores(kc, C), g["kb_cur"][h], "current key buckets")
    top1 = g["top1"][h].astype(np.int64)
    if n:
        parity.check_argmax(O.centroid_scores(ck[h], C), g["kb_in"][h][:n], "cache key buckets")
        parity.check_argmax(O.cosine_matrix(q, ck[h]), top1, "top-1")
        cos_at = O.cosine_rows(kc, ck[h][top1])
        parity.check_evict(cos_at, top1, g["evict"][h], n, cfg.tau)
        parity.check_owner(cos_at, top1, g["evict"][h], g["owner"][h], n, cfg.tau)
    else:
        assert np.all(top1 == -1) and np.all(g["owner"][h] == -1)
    # the merged cache on the GPU's validated decisions
    ev = g["evict"][h][:n].astype(bool)
    owner = g["owner"][h][:n].astype(np.int64)
    nk, nv, ng, imap, length = O.compact_merge(ev, owner, top1, ck[h], cv[h], gin[h], kc, vc, cfg.M)
    assert int(g["len_out"][h]) == length
    assert np.array_equal(g["index_map"][h].astype(np.int64), imap)
    np.testing.assert_array_equal(g["k_out"][h][:length], nk)
    assert np.array_equal(g["g_out"][h][:length], ng), "group counts"
    # values: exact copies where nothing merged, one bf16 rounding of the mean where it did
    np.testing.assert_allclose(g["v_out"][h][:length], nv, rtol=2.0 ** -8, atol=1e-6)
    merged = int((ng > 1).sum() - (gin[h][imap[:length][imap[:length] < n]] > 1).sum())
    kb_new = O.gather_rows(imap, length, g["kb_in"][h][:n], g["kb_cur"][h])
    assert np.array_equal(g["kb_out"][h][:length], kb_new)
    # AnnSA over grouped keys
    o, lse, _ = O.annsa_attention(q, g["qb"][h], nk, nv, kb_new, cfg.scale, g=ng)
    parity.close(g["o_self"][h], o, *parity.TOL[cfg.dtype], f"grouped o_self head {h}")
    fin = np.isfinite(lse)
    assert np.array_equal(np.isfinite(g["lse_self"][h]), fin)
    np.testing.assert_allclose(g["lse_self"][h][fin], lse[fin], rtol=0, atol=1e-3)
    return merged


@pytest.mark.parametrize("seed", [0, 1])
def test_merge_step_small(seed):
    cfg = GH.small_bf16()
    inputs = synth.layer_step_inputs(cfg, seed=seed)
    ck, cv = GH.raw_window(inputs, cfg)
    gin = _counts(seed, cfg.H, ck.shape[1])
    g = _merge_step(cfg, inputs, ck, cv, gin)
    assert g["status"] == 0
    merged = sum(_check_head(cfg, inputs, ck, cv, gin, g, h) for h in range(cfg.H))
    assert g["evict"].sum() > 0 and merged > 0


def test_merge_step_d64_partial_cache_and_empty_cache():
    cfg = GH.small_bf16().replace(d=64, M=2400)
    inputs = synth.layer_step_inputs(cfg, seed=2)
    ck, cv = inputs["history_k"][:, :500], inputs["history_v"][:, :500]
    gin = _counts(2, cfg.H, 500)
    g = _merge_step(cfg, inputs, ck, cv, gin)
    assert g["status"] == 0 and (g["len_out"] < cfg.M).all()
    for h in range(cfg.H):
        _check_head(cfg, inputs, ck, cv, gin, g, h)
    empty = np.zeros((cfg.H, 0, cfg.d), np.float32)
    g = _merge_step(cfg, inputs, empty, empty, np.zeros((cfg.H, 0), np.int32))
    for h in range(cfg.H):
        _check_head(cfg, inputs, empty, empty, np.zeros((cfg.H, 0), np.int64), g, h)
    assert (g["g_out"][:, :cfg.Nq] == 1).all()


def test_merge_step_full_size_layer():
    cfg = synth.WAN13B_LAYER
    inputs = synth.layer_step_inputs(cfg, seed=0)
    ck, cv = GH.raw_window(inputs, cfg)
    gin = _counts(0, cfg.H, ck.shape[1])
    g = _merge_step(cfg, inputs, ck, cv, gin)
    assert g["status"] == 0
    for h in (0, cfg.H - 1):
        _check_head(cfg, inputs, ck, cv, gin, g, h)
    # every head: the counts add up (nothing is lost but what the FIFO cap drops)
    assert (g["g_out"].sum(axis=1) <= gin.sum(axis=1) + cfg.Nq).all()


def _dense_grouped(cfg, q, k, v, gcnt):
    out = torch.zeros_like(q)
    lse = torch.zeros(q.shape[:2], dtype=torch.float32, device="cuda")
    L.fastar_dense_attn_grouped(q, k, v, k.shape[1], gcnt, cfg.scale, out, lse)
    torch.cuda.synchronize()
    return GH.np_(out), GH.np_(lse)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("bf16", 64), ("f32", 128)])
def test_dense_grouped_matches_oracle_with_empty_groups(dtype, d):
    cfg = GH.small_bf16().replace(dtype=dtype, d=d)
    rng = np.random.default_rng(17)
    H, nq, nk = 2, 300, 1001
    rnd = lambda *s: synth.bf16_round(rng.standard_normal(s).astype(np.float32))
    q, k, v = rnd(H, nq, d), rnd(H, nk, d), rnd(H, nk, d)
    gcnt = rng.integers(0, 7, size=(H, nk)).astype(np.int32)      # zeros: empty groups
    o, lse = _dense_grouped(cfg, GH.to_dev(q, cfg), GH.to_dev(k, cfg), GH.to_dev(v, cfg),
                            torch.from_numpy(gcnt).cuda())
    for h in range(H):
        want_o, want_l = O.dense_attention(q[h], k[h], v[h], cfg.scale, g=gcnt[h])
        parity.close(o[h], want_o, *parity.TOL[dtype], f"dense grouped head {h}")
        np.testing.assert_allclose(lse[h], want_l, rtol=0, atol=1e-3)


def test_unit_counts_give_the_ungrouped_result_bit_for_bit():
    cfg = GH.small_bf16()
    rng = np.random.default_rng(23)
    H, nq, nk, d = 2, 257, 700, 128
    q, k, v = (GH.to_dev(rng.standard_normal(s).astype(np.float32), cfg) for s in ((H, nq, d), (H, nk, d), (H, nk, d)))
    ones = torch.ones((H, nk), dtype=torch.int32, device="cuda")
    o_g, l_g = _dense_grouped(cfg, q, k, v, ones)
    o_u = torch.zeros_like(q)
    l_u = torch.zeros((H, nq), dtype=torch.float32, device="cuda")
    L.fastar_dense_attn(q, k, v, nk, cfg.scale, o_u, l_u)
    torch.cuda.synchronize()
    assert np.array_equal(o_g, GH.np_(o_u)) and np.array_equal(l_g, GH.np_(l_u))


def test_lemma_on_gpu_resent_keys_rollout_equals_full_history():
    """Chunks that re-send cached keys (queries equal to keys): the merged cache, with
    its counts, attends like the whole history (the Lemma's exactness, up to bf16)."""
    cfg = GH.small_bf16().replace(H=2, Tf=96, F=2, M=4000, tau=0.99, B=8, r=2)
    rng = np.random.default_rng(31)
    layer = _layer(cfg)
    layer.set_centroids(GH.to_dev(synth.bf16_round(rng.standard_normal((cfg.H, cfg.B, cfg.d)).astype(np.float32)),
                                  cfg))
    layer.set_prompt(GH.to_dev(np.zeros((cfg.H, cfg.P, cfg.d), np.float32), cfg),
                     GH.to_dev(np.zeros((cfg.H, cfg.P, cfg.d), np.float32), cfg))
    hist_k, hist_v, cache_k = [], [], None
    for t in range(5):
        k = synth.bf16_round(rng.standard_normal((cfg.H, cfg.Nq, cfg.d)).astype(np.float32))
        if t:
            pick = rng.choice(cache_k.shape[1], size=cfg.Nq // 2, replace=False)
            k[:, : cfg.Nq // 2] = cache_k[:, pick]
        v = synth.bf16_round(rng.standard_normal((cfg.H, cfg.Nq, cfg.d)).astype(np.float32))
        layer.step(*(GH.to_dev(x, cfg) for x in (k, k, v)))
        torch.cuda.synchronize()
        assert layer.status() == 0
        if t:
            assert GH.np_(layer.evict).sum() > 0
        c = layer.cache
        n = int(c.len[0].item())
        cache_k = GH.np_(c.k[:, :n])
        hist_k.append(k)
        hist_v.append(v)
    c = layer.cache
    n = int(c.len[0].item())
    assert (GH.np_(c.len) == n).all() and n < 5 * cfg.Nq
    assert (GH.np_(c.g[:, :n]).sum(axis=1) == 5 * cfg.Nq).all()
    Qt = synth.bf16_round(rng.standard_normal((cfg.H, 200, cfg.d)).astype(np.float32))
    o, _ = _dense_grouped(cfg, GH.to_dev(Qt, cfg), c.k[:, :n].contiguous(), c.v[:, :n].contiguous(),
                          c.g[:, :n].contiguous())
    Kh, Vh = np.concatenate(hist_k, axis=1), np.concatenate(hist_v, axis=1)
    for h in range(cfg.H):
        want, _ = O.dense_attention(Qt[h], Kh[h], Vh[h], cfg.scale)
        parity.close(o[h], want, *parity.TOL["bf16"], f"merged cache vs full history, head {h}")
