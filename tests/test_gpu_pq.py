"""GPU parity of the quantization variant of the TempCache match (technical summary §2.A:
"LSH or Quantization"; product quantization of the cached keys) against the oracle:
the codes (up to near-ties in distance), the top-1 over the decoded keys, the eviction
flags and owners on the true keys, the codes moved through the compaction, and the
step's AnnSA output, through the C ABI and the layer."""
import numpy as np
import pytest
import torch

from kv_cache_tempcache_gb300 import synth
from kv_cache_tempcache_gb300.layer import FastARLayer
from oracle import fastar_oracle as O
import gpu_harness as GH
import parity

pytestmark = pytest.mark.gpu


def _pq_step(cfg, inputs, ck, cv, cb, m, Kc):
    layer = FastARLayer(H=cfg.H, d=cfg.d, Tf=cfg.Tf, F=cfg.F, M=cfg.M, B=cfg.B, r=cfg.r, P=cfg.P, tau=cfg.tau,
                        tau_ca=cfg.tau_ca, topk=cfg.topk, dtype=GH.torch_dtype(cfg), pq=(m, Kc))
    layer.set_centroids(GH.to_dev(inputs["centroids"], cfg))
    layer.set_prompt(GH.to_dev(inputs["kp"], cfg), GH.to_dev(inputs["vp"], cfg))
    layer.set_codebooks(GH.to_dev(cb, cfg))
    layer.load_cache(GH.to_dev(ck, cfg), GH.to_dev(cv, cfg))
    cin, cout = layer.caches[layer.cur], layer.caches[1 - layer.cur]
    codes_in = GH.np_(cin.codes).copy()
    kb_in = GH.np_(cin.kb)[..., 0].copy()
    q, k, v = (GH.to_dev(inputs[x], cfg) for x in ("q", "k_cur", "v_cur"))
    layer.step(q, k, v, advance=False)
    torch.cuda.synchronize()
    n = GH.np_
    return dict(codes_in=codes_in, codes_cur=n(layer.codes_cur), top1=n(layer.top1), s1=n(layer.s1),
                evict=n(layer.evict), owner=n(layer.owner), index_map=n(layer.index_map), len_out=n(cout.len),
                codes_out=n(cout.codes), k_out=n(cout.k), qb=n(layer.qb), kb_in=kb_in,
                kb_cur=n(layer.kb_cur)[..., 0], o_self=n(layer.o_self), status=layer.status())


def _check_codes(X, cbh, got, what):
    """Every (key, sub-space) code must be a nearest codeword up to a near-tie."""
    dist = O.pq_distances(X, cbh)                       # [n, m, Kc]
    n, m, Kc = dist.shape
    return parity.check_argmax(-dist.reshape(n * m, Kc), got.reshape(-1).astype(np.int64), what)


def _check_head(cfg, inputs, ck, cv, cb, g, h):
    q, kc, vc = inputs["q"][h], inputs["k_cur"][h], inputs["v_cur"][h]
    n, Nq = ck.shape[1], cfg.Nq
    ties = 0
    if n:
        ties += _check_codes(ck[h], cb[h], g["codes_in"][h][:n], f"cache codes h{h}")
    ties += _check_codes(kc, cb[h], g["codes_cur"][h], f"current codes h{h}")
    top1 = g["top1"][h].astype(np.int64)
    if n:
        K_hat = O.pq_decode(g["codes_in"][h][:n], cb[h])
        S = O.cosine_matrix(q, K_hat)
        ties += parity.check_argmax(S, top1, f"quantised top-1 h{h}")
        np.testing.assert_allclose(g["s1"][h], S[np.arange(Nq), top1], rtol=0, atol=2e-5)
        cos_at = O.cosine_rows(kc, ck[h][top1])         # the eviction test uses the true keys
        parity.check_evict(cos_at, top1, g["evict"][h], n, cfg.tau)
        parity.check_owner(cos_at, top1, g["evict"][h], g["owner"][h], n, cfg.tau)
    else:
        assert np.all(top1 == -1)
    ev = g["evict"][h][:n].astype(bool)
    imap, length = O.compact_plan(ev, n, Nq, cfg.M)
    assert int(g["len_out"][h]) == length and np.array_equal(g["index_map"][h].astype(np.int64), imap)
    want_codes = O.gather_rows(imap, length, g["codes_in"][h][:n], g["codes_cur"][h])
    assert np.array_equal(g["codes_out"][h][:length], want_codes), "codes through the compaction"
    new_k = O.gather_rows(imap, length, ck[h], kc)
    np.testing.assert_array_equal(g["k_out"][h][:length], new_k)
    kb_new = O.gather_rows(imap, length, g["kb_in"][h][:n], g["kb_cur"][h])
    o, _, _ = O.annsa_attention(q, g["qb"][h], new_k, O.gather_rows(imap, length, cv[h], vc), kb_new, cfg.scale)
    parity.close(g["o_self"][h], o, *parity.TOL[cfg.dtype], f"o_self h{h}")
    return ties


@pytest.mark.parametrize("seed", [0, 1])
def test_pq_step_small(seed):
    cfg = GH.small_bf16()
    inputs = synth.layer_step_inputs(cfg, seed=seed)
    ck, cv = GH.raw_window(inputs, cfg)
    cb = synth.pq_codebooks(inputs["history_k"], 32, 16, seed=seed)
    g = _pq_step(cfg, inputs, ck, cv, cb, 32, 16)
    assert g["status"] == 0
    for h in range(cfg.H):
        _check_head(cfg, inputs, ck, cv, cb, g, h)
    assert g["evict"].sum() > 0


def test_pq_d64_eight_dim_subspaces_partial_and_empty_cache():
    cfg = GH.small_bf16().replace(d=64, M=2400)
    inputs = synth.layer_step_inputs(cfg, seed=2)
    ck, cv = inputs["history_k"][:, :500], inputs["history_v"][:, :500]
    cb = synth.pq_codebooks(inputs["history_k"], 8, 64, seed=2)        # d/m = 8, 64 codewords
    g = _pq_step(cfg, inputs, ck, cv, cb, 8, 64)
    assert g["status"] == 0
    for h in range(cfg.H):
        _check_head(cfg, inputs, ck, cv, cb, g, h)
    empty = np.zeros((cfg.H, 0, cfg.d), np.float32)
    g = _pq_step(cfg, inputs, empty, empty, cb, 8, 64)
    for h in range(cfg.H):
        _check_head(cfg, inputs, empty, empty, cb, g, h)


def test_pq_full_size_layer_sampled_heads():
    cfg = synth.WAN13B_LAYER
    inputs = synth.layer_step_inputs(cfg, seed=0)
    ck, cv = GH.raw_window(inputs, cfg)
    cb = synth.pq_codebooks(inputs["history_k"][:, :cfg.Tf], 32, 16, seed=0)
    g = _pq_step(cfg, inputs, ck, cv, cb, 32, 16)
    assert g["status"] == 0
    for h in (0, cfg.H - 1):
        _check_head(cfg, inputs, ck, cv, cb, g, h)
    assert (g["len_out"] == cfg.M).all()
