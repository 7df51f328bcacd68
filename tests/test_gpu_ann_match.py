"""GPU parity of the ANN-restricted TempCache match (each query compared only with the
incoming cache's keys in its own buckets) against the oracle.

Protocol: the GPU's bucket decisions are checked first (argmax / top-r within the
near-tie margin); the oracle is then evaluated on those decisions, and the GPU's
top-1 must reach the restricted row maximum within the margin, s1 must match it, and
the eviction flags must follow from the GPU's (validated) choices."""
import numpy as np
import pytest
import torch

from oracle import fastar_oracle as O
from kv_cache_tempcache_gb300 import _lib as L, synth
import gpu_harness as GH
import parity

pytestmark = pytest.mark.gpu


def _run(cfg, seed, cache_len=None):
    inp = synth.layer_step_inputs(cfg, seed=seed)
    ck, _ = GH.raw_window(inp, cfg)
    H, d, nq, M, B, r = cfg.H, cfg.d, cfg.Nq, cfg.M, cfg.B, cfg.r
    dev = torch.device("cuda")
    q = GH.to_dev(inp["q"], cfg)
    kc = GH.to_dev(inp["k_cur"], cfg)
    C = GH.to_dev(inp["centroids"], cfg)
    cache = torch.zeros((H, M, d), dtype=q.dtype, device=dev)
    n = ck.shape[1]
    cache[:, :n] = GH.to_dev(ck, cfg)
    lens = np.full(H, n, np.int64) if cache_len is None else np.asarray(cache_len, np.int64)
    clen = torch.tensor(lens, dtype=torch.int32, device=dev)
    i32 = lambda *s: torch.zeros(s, dtype=torch.int32, device=dev)
    qb, kb = i32(H, nq, r), i32(H, M, 1)
    knorm = torch.zeros((H, M, 1), dtype=torch.float32, device=dev)
    L.fastar_bucket_assign(q, C, r, qb)
    L.fastar_bucket_assign(cache, C, 1, kb, None, knorm)
    qperm, qoff, kperm, koff = i32(H, nq * r), i32(H, B + 1), i32(H, M), i32(H, B + 1)
    status = i32(1)
    L.fastar_bucket_sort(qb, B, qperm, qoff, None, status)
    L.fastar_bucket_sort(kb, B, kperm, koff, clen, status)
    ws = torch.zeros(L.workspace_bytes(L.OP_MATCH_ANN, H, nq, M, d, B, r), dtype=torch.uint8, device=dev)
    top1, s1 = i32(H, nq), torch.zeros((H, nq), dtype=torch.float32, device=dev)
    evict = torch.ones((H, M), dtype=torch.uint8, device=dev)
    owner = torch.full((H, M), 7, dtype=torch.int32, device=dev)
    L.fastar_tempcache_match_ann(q, kc, r, B, qperm, qoff, cache, knorm, clen, kperm, koff, cfg.tau, top1, s1,
                                 evict, status, ws, owner=owner)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return inp, ck, lens, dict(qb=GH.np_(qb), kb=GH.np_(kb)[..., 0], top1=GH.np_(top1), s1=GH.np_(s1),
                               evict=GH.np_(evict), owner=GH.np_(owner))


def _check(cfg, inp, ck, lens, g):
    stats = dict(ties=0, ambiguous=0, matched=0)
    for h in range(cfg.H):
        n = int(lens[h])
        Ch = inp["centroids"][h]
        Kh = ck[h][:n]
        # the GPU's buckets must be correct answers (near-ties either way)
        parity.check_topr(O.centroid_scores(inp["q"][h], Ch), g["qb"][h], f"query buckets h{h}")
        if n:
            parity.check_argmax(O.centroid_scores(Kh, Ch), g["kb"][h][:n], f"key buckets h{h}")
        R, kb = g["qb"][h].astype(np.int64), g["kb"][h][:n].astype(np.int64)
        # restricted cosines on the GPU's buckets; the oracle's decision for reference
        S = O.cosine_matrix(inp["q"][h], Kh) if n else np.zeros((cfg.Nq, 0))
        allowed = (kb[None, :, None] == R[:, None, :]).any(axis=2)
        Sm = np.where(allowed, S, -np.inf)
        want_t, want_s = O.tempcache_match_ann(inp["q"][h], R, Kh, kb)
        got_t = g["top1"][h].astype(np.int64)
        has = want_t >= 0
        assert np.array_equal(got_t < 0, ~has), f"h{h}: queries with / without a candidate differ"
        if has.any():
            stats["ties"] += parity.check_argmax(Sm[has], got_t[has], f"ann top1 h{h}")
            np.testing.assert_allclose(g["s1"][h][has], Sm[has].max(axis=1), rtol=0, atol=2e-3)
        assert np.all(np.isneginf(g["s1"][h][~has]))
        _, ce = O.evict_flags(got_t, inp["k_cur"][h], Kh, cfg.tau)
        stats["ambiguous"] += parity.check_evict(ce, got_t, g["evict"][h], n, cfg.tau)
        parity.check_owner(ce, got_t, g["evict"][h], g["owner"][h], n, cfg.tau)
        assert not g["evict"][h][n:].any(), "flags beyond the cache length"
        stats["matched"] += int(has.sum())
    return stats


@pytest.mark.parametrize("seed", [0, 1])
def test_ann_match_small(seed):
    cfg = GH.small_bf16()
    inp, ck, lens, g = _run(cfg, seed)
    st = _check(cfg, inp, ck, lens, g)
    assert st["matched"] > 0


def test_ann_match_partial_cache_and_d64():
    cfg = GH.small_bf16().replace(d=64)
    inp, ck, lens, g = _run(cfg, 3, cache_len=[700, 0])
    _check(cfg, inp, ck, lens, g)
    assert (g["top1"][1] == -1).all()


def test_ann_match_full_size_layer():
    cfg = synth.WAN13B_LAYER
    inp, ck, lens, g = _run(cfg, 0)
    st = _check(cfg, inp, ck, lens, g)
    assert st["matched"] > 0.9 * cfg.H * cfg.Nq
