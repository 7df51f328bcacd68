"""The AnnCA failure rule on the GPU, through the C ABI.

A (head, frame) whose selection could not be formed is marked kcnt = -1 with nothing kept;
the cross-attention (which takes no status word) attends to no prompt token for that frame
(O = 0, lse = -inf), exactly as for kcnt = 0, on every path: the kept rows read in place,
gathered into a workspace, or read from the kept-row planes; the other frames keep the step's
own results."""
import numpy as np
import pytest
import torch

from kv_cache_tempcache_gb300 import _lib as L, synth
import gpu_harness as GH

pytestmark = pytest.mark.gpu


def _layer_after_step():
    cfg = GH.small_bf16()
    inputs = synth.layer_step_inputs(cfg, seed=11)
    ck, cv = GH.raw_window(inputs, cfg)
    g, layer = GH.gpu_step(cfg, inputs, ck, cv)
    assert g["status"] == 0
    return cfg, inputs, layer


def test_cross_attention_skips_failed_and_empty_frames_on_every_path():
    cfg, inputs, layer = _layer_after_step()
    q = GH.to_dev(inputs["q"], cfg)
    kcnt = layer.kcnt.clone()
    kcnt[0, 1] = -1   # a failed selection
    kcnt[1, 2] = 0    # an empty one
    ws = torch.zeros(L.workspace_bytes(L.OP_CROSS_ATTN, cfg.H, n=0, d=cfg.d, P=cfg.P, F=cfg.F), dtype=torch.uint8,
                     device="cuda")
    ref = None
    for path in ("in_place", "workspace", "planes"):
        o = torch.full_like(q, 7.0)
        lse = torch.zeros(q.shape[:2], dtype=torch.float32, device="cuda")
        if path == "planes":
            L.fastar_cross_attn_kept(q, cfg.F, layer.kp_kept, layer.vp_kept, kcnt, cfg.scale, o, lse)
        else:
            L.fastar_cross_attn_subset(q, cfg.F, layer.kp, layer.vp, layer.kidx, kcnt, cfg.scale, o, lse,
                                       workspace=ws if path == "workspace" else None)
        torch.cuda.synchronize()
        on, ln = GH.np_(o), GH.np_(lse)
        Tf = cfg.Tf
        for h, f in ((0, 1), (1, 2)):
            assert not on[h, f * Tf:(f + 1) * Tf].any(), f"{path}: frame ({h}, {f}) attended to something"
            assert np.isneginf(ln[h, f * Tf:(f + 1) * Tf]).all()
        if ref is None:
            ref = (on, ln)
        else:   # the three paths agree bit for bit, failed frames included
            assert np.array_equal(on, ref[0]) and np.array_equal(ln, ref[1])
    # the untouched frames are the layer's own results
    g_cross = GH.np_(layer.o_cross)
    for h in range(cfg.H):
        for f in range(cfg.F):
            if (h, f) not in ((0, 1), (1, 2)):
                rows = slice(f * cfg.Tf, (f + 1) * cfg.Tf)
                assert np.array_equal(ref[0][h, rows], g_cross[h, rows])
