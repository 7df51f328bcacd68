"""GPU parity of the whole FAST-AR layer step against the CPU oracle, stage by stage,
through the C ABI.  Sizes span several tiles with ragged tails."""
import math

import numpy as np
import pytest
import torch

from kv_cache_tempcache_gb300 import synth
from oracle import fastar_oracle as O
import gpu_harness as GH
import parity

pytestmark = pytest.mark.gpu


def _run(cfg, seed=0, gate=True, q_layout="HND", cache=None):
    inputs = synth.layer_step_inputs(cfg, seed=seed)
    ck, cv = GH.raw_window(inputs, cfg) if cache is None else cache(inputs)
    g, _ = GH.gpu_step(cfg, inputs, ck, cv, gate=gate, q_layout=q_layout)
    counts = GH.check_step(cfg, inputs, ck, cv, g, gate=gate)
    return inputs, g, counts


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tiny_fp32_step(seed):
    _, g, counts = _run(synth.TINY_FP32, seed)
    assert g["evict"].sum() > 0, "the tiny workload should evict"
    parity.report(f"tiny_fp32 layer step, seed {seed}", counts)


@pytest.mark.parametrize("seed", [0, 1])
def test_small_bf16_step(seed):
    cfg = GH.small_bf16()
    _, g, counts = _run(cfg, seed)
    assert g["evict"].sum() > 0
    assert (g["len_out"] == cfg.M).all()
    parity.report(f"small_bf16 layer step, seed {seed}", counts)


@pytest.mark.parametrize("r", [3, 4])
def test_more_buckets_per_query(r):
    # r > 2: AnnSA merges more than two slot partials per query, AnnCA gates on more ids
    _, g, _ = _run(GH.small_bf16().replace(r=r, name=f"bf16_r{r}"))
    assert g["evict"].sum() > 0


def test_bf16_d64_and_f32_d128():
    _run(GH.small_bf16().replace(d=64, name="bf16_d64"))
    _run(GH.small_bf16().replace(dtype="f32", name="f32_d128", H=1, Tf=130, prior_frames=4, M=600))


def test_token_major_layout():
    cfg = GH.small_bf16().replace(H=3)
    _run(cfg, q_layout="NHD")


def test_empty_cache_first_chunk():
    cfg = GH.small_bf16()
    inputs = synth.layer_step_inputs(cfg, seed=3)
    H, d = cfg.H, cfg.d
    empty = np.zeros((H, 0, d), np.float32)
    g, _ = GH.gpu_step(cfg, inputs, empty, empty)
    GH.check_step(cfg, inputs, empty, empty, g)
    assert (g["top1"] == -1).all() and (g["len_out"] == cfg.Nq).all()


def test_partial_cache_no_fifo_drop():
    cfg = GH.small_bf16().replace(M=2400)
    _, g, _ = _run(cfg, cache=lambda inp: (inp["history_k"][:, :500], inp["history_v"][:, :500]))
    assert (g["len_out"] < cfg.M).all()


def test_threshold_extremes():
    # tau = -1: a cosine is never below -1, so every cache entry that is some current key's
    # top-1 match is evicted; tau_ca above 1: no score reaches it, so each frame keeps
    # exactly its top-k floor
    cfg = GH.small_bf16().replace(tau=-1.0, tau_ca=1.5, name="bf16_extremes")
    _, g, _ = _run(cfg)
    n = min(cfg.M, cfg.prior_frames * cfg.Tf)
    for h in range(cfg.H):
        t1 = g["top1"][h]
        matched = np.unique(t1[t1 >= 0])
        assert len(matched) > 0
        assert g["evict"][h, :n].sum() == len(matched) and g["evict"][h, matched].all()
    assert (g["kcnt"] == cfg.topk).all()


def test_largest_bucket_and_prompt_counts():
    # the largest sizes the interface accepts for the ANN parts: B = 256 buckets, r = 8
    # buckets per query, P = 1024 prompt tokens
    cfg = GH.small_bf16().replace(B=256, r=8, P=1024, name="bf16_max_sizes")
    _, g, _ = _run(cfg)
    assert g["qb"].max() < 256 and (g["kcnt"] >= cfg.topk).all()


def test_prompt_smaller_than_topk_and_ungated():
    cfg = GH.small_bf16().replace(P=8, topk=16)
    _, g, _ = _run(cfg)
    assert (g["kcnt"] == 8).all()
    _run(GH.small_bf16(), gate=False)


def test_textbook_reduction_on_gpu():
    # B=1, r=1, tau>1, tau_ca=-1, M >= n+Nq: sparse == dense, nothing evicted, all prompt kept
    cfg = GH.small_bf16().replace(B=1, r=1, tau=2.0, tau_ca=-1.0, M=2000, prior_frames=4)
    inputs, g, _ = _run(cfg, cache=lambda inp: (inp["history_k"], inp["history_v"]))
    assert g["evict"].sum() == 0 and (g["len_out"] == 800 + cfg.Nq).all()
    assert g["keep"].all()
    tol = parity.TOL[cfg.dtype]
    for h in range(cfg.H):
        K = np.concatenate([inputs["history_k"][h], inputs["k_cur"][h]])
        V = np.concatenate([inputs["history_v"][h], inputs["v_cur"][h]])
        o, _ = O.dense_attention(inputs["q"][h], K, V, cfg.scale)
        parity.close(g["o_self"][h], o, *tol, "reduced AnnSA vs dense")


def test_exact_ties_lowest_index():
    # integer-valued, bf16-exact duplicated keys: every dot product is exact in fp32
    cfg = synth.LayerConfig(name="ties", H=1, d=64, Tf=64, F=1, prior_frames=0, P=16, C=1, sigma_mix=0, rho=0,
                            drift=0, qnoise=0, tau=0.999, M=256, B=4, r=2, tau_ca=0.5, topk=4, dtype="bf16")
    rng = np.random.default_rng(0)
    base = rng.integers(-3, 4, size=(8, 64)).astype(np.float32)
    ck = np.concatenate([base, base, 2 * base, base])[None]           # 32 entries, 4 copies of each direction
    cv = rng.standard_normal((1, 32, 64)).astype(np.float32)
    q = base[rng.integers(0, 8, size=64)][None]
    cent = np.zeros((1, 4, 64), np.float32)
    cent[0, 0, 0] = cent[0, 2, 0] = 1.0                               # duplicated centroids
    cent[0, 1, 1] = cent[0, 3, 1] = 1.0
    inputs = dict(q=q, k_cur=q.copy(), v_cur=rng.standard_normal((1, 64, 64)).astype(np.float32),
                  centroids=cent, kp=base[rng.integers(0, 8, size=16)][None],
                  vp=rng.standard_normal((1, 16, 64)).astype(np.float32))
    inputs = {k: synth.bf16_round(v) for k, v in inputs.items()}
    ck, cv = synth.bf16_round(ck), synth.bf16_round(cv)
    g, _ = GH.gpu_step(cfg, inputs, ck, cv)
    # exact: the oldest copy wins every tie, duplicated centroids resolve to the lower index
    o_top1, _, _ = O.tempcache_match(inputs["q"][0], ck[0])
    assert np.array_equal(g["top1"][0], o_top1)
    assert np.array_equal(g["qb"][0], O.query_buckets(inputs["q"][0], cent[0], 2))
    assert np.array_equal(g["kb_in"][0][:32], O.key_buckets(ck[0], cent[0]))
    assert set(np.unique(g["kb_in"][0][:32]).tolist()) <= {0, 1}
    GH.check_step(cfg, inputs, ck, cv, g)


def test_dense_baseline_matches_oracle():
    cfg = GH.small_bf16()
    inputs = synth.layer_step_inputs(cfg, seed=4)
    H, d, Nq = cfg.H, cfg.d, cfg.Nq
    hist = inputs["history_k"].shape[1]
    dense = GH.DenseLayer(H, d, Nq, hist + Nq, cfg.P, dtype=torch.bfloat16)
    dense.load_history(GH.to_dev(inputs["history_k"], cfg), GH.to_dev(inputs["history_v"], cfg))
    dense.set_prompt(GH.to_dev(inputs["kp"], cfg), GH.to_dev(inputs["vp"], cfg))
    o_s, o_c = dense.step(*(GH.to_dev(inputs[x], cfg) for x in ("q", "k_cur", "v_cur")))
    torch.cuda.synchronize()
    tol = parity.TOL["bf16"]
    for h in range(H):
        want = O.head_dense_step(inputs["q"][h], inputs["history_k"][h], inputs["history_v"][h], inputs["k_cur"][h],
                                 inputs["v_cur"][h], inputs["kp"][h], inputs["vp"][h], cfg.scale)
        parity.close(GH.np_(o_s[h]), want["o_self"], *tol, "dense self")
        parity.close(GH.np_(o_c[h]), want["o_cross"], *tol, "dense cross")


def test_top1_only_match_equals_top2_match():
    """The step without the second-best diagnostic (the benchmark's configuration)
    takes exactly the same decisions and produces the same outputs."""
    cfg = GH.small_bf16().replace(H=3)
    inputs = synth.layer_step_inputs(cfg, seed=8)
    ck, cv = GH.raw_window(inputs, cfg)
    g1, _ = GH.gpu_step(cfg, inputs, ck, cv, diagnostics=True)
    g0, _ = GH.gpu_step(cfg, inputs, ck, cv, diagnostics=False)
    for key in ("top1", "s1", "evict", "index_map", "len_out", "o_self", "o_cross", "keep"):
        assert np.array_equal(g0[key], g1[key]), key
    GH.check_step(cfg, inputs, ck, cv, g0)


def test_graph_replay_equals_eager():
    cfg = GH.small_bf16()
    inputs = synth.layer_step_inputs(cfg, seed=5)
    ck, cv = GH.raw_window(inputs, cfg)
    g, layer = GH.gpu_step(cfg, inputs, ck, cv)
    q, k, v = (GH.to_dev(inputs[x], cfg) for x in ("q", "k_cur", "v_cur"))
    layer.capture(q, k, v)
    layer.o_self.zero_()
    layer.o_cross.zero_()
    layer.replay()
    torch.cuda.synchronize()
    assert np.array_equal(GH.np_(layer.o_self), g["o_self"])
    assert np.array_equal(GH.np_(layer.o_cross), g["o_cross"])
    assert np.array_equal(GH.np_(layer.index_map), g["index_map"])


def test_rollout_matches_oracle_chunk_by_chunk():
    """From an empty cache, chunk after chunk: GPU and oracle evolve independently and
    must agree on every cache decision until a validated near-tie (if any)."""
    cfg = GH.small_bf16().replace(M=900)
    gen = synth.DriftingMixture(cfg, seed=7)
    layer = GH.make_layer(cfg)
    layer.set_centroids(GH.to_dev(gen.centroids, cfg))
    kp, vp = gen.prompt
    layer.set_prompt(GH.to_dev(kp, cfg), GH.to_dev(vp, cfg))
    ck = [np.zeros((0, cfg.d), np.float32) for _ in range(cfg.H)]
    cv = [np.zeros((0, cfg.d), np.float32) for _ in range(cfg.H)]
    bytes0 = torch.cuda.memory_allocated()
    for t in range(8):
        k, v, q = gen.next_chunk()
        layer.step(*(GH.to_dev(x, cfg) for x in (q, k, v)))
        torch.cuda.synchronize()
        assert layer.status() == 0
        c = layer.cache
        for h in range(cfg.H):
            nk, nv, info = O.tempcache_only_advance(q[h], k[h], v[h], ck[h], cv[h], tau=cfg.tau, M=cfg.M)
            L = int(c.len[h].item())
            assert L == info["length"] <= cfg.M
            np.testing.assert_array_equal(GH.np_(c.k[h, :L]), nk)
            np.testing.assert_array_equal(GH.np_(c.v[h, :L]), nv)
            ck[h], cv[h] = nk, nv
        assert torch.cuda.memory_allocated() == bytes0, "the step must not allocate"


@pytest.mark.parametrize("P,d", [(100, 128), (8, 64), (512, 128)])
def test_cross_attention_paths_agree_bit_for_bit(P, d):
    """The kept prompt rows read in place (no workspace), gathered into contiguous planes
    and read by the tensor engine (workspace), or read from the planes the selection's
    ranking launch wrote (fastar_cross_attn_kept, the layer's path): same rows, same order,
    so the same bits; against the oracle.  The planes hold exactly the kept rows, then
    zero rows to the next 64-row boundary."""
    from kv_cache_tempcache_gb300 import _lib as L
    cfg = GH.small_bf16().replace(P=P, d=d, topk=min(16, P))
    inputs = synth.layer_step_inputs(cfg, seed=6)
    ck, cv = GH.raw_window(inputs, cfg)
    g, layer = GH.gpu_step(cfg, inputs, ck, cv)
    q = GH.to_dev(inputs["q"], cfg)
    outs = []
    ws = torch.zeros(L.workspace_bytes(L.OP_CROSS_ATTN, cfg.H, n=0, d=d, P=P, F=cfg.F), dtype=torch.uint8,
                     device="cuda")
    for path in ("in_place", "workspace", "planes"):
        o = torch.zeros_like(q)
        lse = torch.zeros(q.shape[:2], dtype=torch.float32, device="cuda")
        if path == "planes":
            L.fastar_cross_attn_kept(q, cfg.F, layer.kp_kept, layer.vp_kept, layer.kcnt, cfg.scale, o, lse)
        else:
            L.fastar_cross_attn_subset(q, cfg.F, layer.kp, layer.vp, layer.kidx, layer.kcnt, cfg.scale, o, lse,
                                       workspace=ws if path == "workspace" else None)
        torch.cuda.synchronize()
        outs.append((GH.np_(o), GH.np_(lse)))
    for i in (1, 2):
        assert np.array_equal(outs[0][0], outs[i][0]) and np.array_equal(outs[0][1], outs[i][1])
    assert np.array_equal(outs[2][0], g["o_cross"])
    kp, vp = GH.np_(layer.kp), GH.np_(layer.vp)
    kpk, vpk = GH.np_(layer.kp_kept), GH.np_(layer.vp_kept)
    for h in range(cfg.H):
        for f in range(cfg.F):
            idx = np.flatnonzero(g["keep"][h][f])
            n, lim = len(idx), min(P, -(-len(idx) // 64) * 64)
            assert np.array_equal(kpk[h, f, :n], kp[h, idx]) and np.array_equal(vpk[h, f, :n], vp[h, idx])
            assert not kpk[h, f, n:lim].any() and not vpk[h, f, n:lim].any()
    tol = parity.TOL[cfg.dtype]
    for h in range(cfg.H):
        kept = [np.flatnonzero(g["keep"][h][f]) for f in range(cfg.F)]
        oc, _ = O.cross_attention_subset(inputs["q"][h], inputs["kp"][h], inputs["vp"][h], kept, cfg.F, cfg.Tf,
                                         cfg.scale)
        parity.close(outs[1][0][h], oc, *tol, f"o_cross head {h}")


@pytest.mark.parametrize("r,layout", [(2, "HND"), (3, "HND"), (2, "NHD")])
def test_fused_assignment_equals_two_calls(r, layout):
    # fastar_bucket_assign_qk: the queries' top-r sets and norms and the current keys'
    # buckets and norms in one launch, bit for bit the two separate calls
    from kv_cache_tempcache_gb300 import _lib as L
    cfg = GH.small_bf16()
    inp = synth.layer_step_inputs(cfg, seed=3)
    if layout == "NHD":
        q = GH.to_dev(inp["q"].transpose(1, 0, 2), cfg).transpose(0, 1)
        k = GH.to_dev(inp["k_cur"].transpose(1, 0, 2), cfg).transpose(0, 1)
    else:
        q, k = GH.to_dev(inp["q"], cfg), GH.to_dev(inp["k_cur"], cfg)
    C = GH.to_dev(inp["centroids"], cfg)
    H, n = cfg.H, cfg.Nq
    i32 = lambda *s: torch.full(s, -5, dtype=torch.int32, device="cuda")
    qb1, kb1, qb2, kb2 = i32(H, n, r), i32(H, n, 1), i32(H, n, r), i32(H, n, 1)
    kn1 = torch.zeros((H, n), dtype=torch.float32, device="cuda")
    kn2, qn1, qn2 = torch.zeros_like(kn1), torch.zeros_like(kn1), torch.zeros_like(kn1)
    L.fastar_bucket_assign(q, C, r, qb1, None, qn1)
    L.fastar_bucket_assign(k, C, 1, kb1, None, kn1)
    L.fastar_bucket_assign_qk(q, k, C, r, qb2, kb2, kn2, q_norms=qn2)
    torch.cuda.synchronize()
    assert torch.equal(qb1, qb2) and torch.equal(kb1, kb2) and torch.equal(kn1, kn2) and torch.equal(qn1, qn2)
    # the norms of the bf16 rows, against float64
    qf = GH.to_dev(inp["q"], cfg).float().cpu().numpy().astype(np.float64)
    np.testing.assert_allclose(GH.np_(qn2), np.linalg.norm(qf, axis=-1), rtol=1e-5)
    parity.check_topr(O.centroid_scores(inp["q"][0], inp["centroids"][0]), GH.np_(qb2)[0], "fused query buckets")


def test_annca_with_the_assignment_norms():
    # fastar_annca_select given the queries' norms from the assignment: the cosines agree with
    # the call that forms the norms itself to fp32 rounding, and both selections are correct
    # answers for the oracle's
    from kv_cache_tempcache_gb300 import _lib as L
    cfg = GH.small_bf16()
    inp = synth.layer_step_inputs(cfg, seed=6)
    q, k, kp = GH.to_dev(inp["q"], cfg), GH.to_dev(inp["k_cur"], cfg), GH.to_dev(inp["kp"], cfg)
    C = GH.to_dev(inp["centroids"], cfg)
    H, n, P, F = cfg.H, cfg.Nq, cfg.P, cfg.F
    dev = torch.device("cuda")
    qb = torch.zeros((H, n, cfg.r), dtype=torch.int32, device=dev)
    kb = torch.zeros((H, n, 1), dtype=torch.int32, device=dev)
    pb = torch.zeros((H, P, 1), dtype=torch.int32, device=dev)
    kn, qn = (torch.zeros((H, n), dtype=torch.float32, device=dev) for _ in range(2))
    L.fastar_bucket_assign_qk(q, k, C, cfg.r, qb, kb, kn, q_norms=qn)
    L.fastar_bucket_assign(kp, C, 1, pb)
    res = []
    for norms in (None, qn):
        keep = torch.zeros((H, F, P), dtype=torch.uint8, device=dev)
        kidx = torch.zeros((H, F, P), dtype=torch.int32, device=dev)
        kcnt = torch.zeros((H, F), dtype=torch.int32, device=dev)
        score = torch.zeros((H, F, P), dtype=torch.float32, device=dev)
        L.fastar_annca_select(q, F, qb, kp, pb, cfg.tau_ca, cfg.topk, 1, keep, kidx, kcnt, score, B=cfg.B,
                              q_norms=norms)
        torch.cuda.synchronize()
        res.append((GH.np_(keep), GH.np_(kcnt), GH.np_(score)))
    s0, s1 = res[0][2], res[1][2]
    fin = np.isfinite(s0)
    assert np.array_equal(fin, np.isfinite(s1))
    np.testing.assert_allclose(s1[fin], s0[fin], rtol=2e-6, atol=1e-7)
    qbn, pbn = GH.np_(qb), GH.np_(pb)[..., 0]
    for keep, kcnt, _ in res:
        for h in range(H):
            _, _, _, ref = O.annca_select(inp["q"][h], qbn[h], inp["kp"][h], pbn[h], F, cfg.Tf, cfg.tau_ca, cfg.topk)
            for f in range(F):
                parity.check_keep(ref[f], keep[h, f], cfg.tau_ca, cfg.topk, f"keep head {h} frame {f}")
                assert int(kcnt[h, f]) == int(keep[h, f].sum())
