"""The allocation-free AnnCA selection entry point against the regular one.

Some callers cannot allocate device memory while they run the step (a server that
reserves all device memory at start-up, a process under a fixed shared budget);
fastar_annca_select_noalloc serves them from a fixed scratch array inside the
library.  Its results must equal the regular entry point's on the same inputs, on
consecutive calls (the shared scratch keeps the previous call's contents).
This file is collected last on purpose."""
import numpy as np
import pytest
import torch

from kv_cache_tempcache_gb300 import synth

pytestmark = pytest.mark.gpu


def _case(seed):
    from kv_cache_tempcache_gb300 import _lib as L
    cfg = synth.LayerConfig(name="noalloc", H=3, d=128, Tf=300, F=3, prior_frames=0, P=200, C=8, sigma_mix=0.3,
                            rho=0.1, drift=0.05, qnoise=0.1, tau=0.95, M=900, B=16, r=2, tau_ca=0.2, topk=16,
                            dtype="bf16")
    inp = synth.layer_step_inputs(cfg, seed=seed)
    dev = torch.device("cuda")
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev).to(torch.bfloat16)
    q, kp, C = t(inp["q"]), t(inp["kp"]), t(inp["centroids"])
    qb = torch.zeros((cfg.H, cfg.Nq, cfg.r), dtype=torch.int32, device=dev)
    pb = torch.zeros((cfg.H, cfg.P, 1), dtype=torch.int32, device=dev)
    L.fastar_bucket_assign(q, C, cfg.r, qb)
    L.fastar_bucket_assign(kp, C, 1, pb)
    return cfg, q, kp, qb, pb


def _outputs(cfg, dev):
    return (torch.full((cfg.H, cfg.F, cfg.P), 7, dtype=torch.uint8, device=dev),
            torch.full((cfg.H, cfg.F, cfg.P), -7, dtype=torch.int32, device=dev),
            torch.full((cfg.H, cfg.F), -7, dtype=torch.int32, device=dev))


def test_noalloc_selection_equals_regular_on_two_calls_in_a_row():
    from kv_cache_tempcache_gb300 import _lib as L
    from kv_cache_tempcache_gb300.build_lib import build
    build()
    L.load()
    dev = torch.device("cuda")
    for seed, tau_ca in ((0, 0.2), (1, 0.35)):
        cfg, q, kp, qb, pb = _case(seed)
        keep_r, kidx_r, kcnt_r = _outputs(cfg, dev)
        ws = torch.zeros(L.workspace_bytes(L.OP_ANNCA, cfg.H, 0, 0, cfg.d, cfg.B, cfg.r, cfg.P, cfg.F),
                         dtype=torch.uint8, device=dev)
        L.fastar_annca_select(q, cfg.F, qb, kp, pb, tau_ca, cfg.topk, 1, keep_r, kidx_r, kcnt_r, None, ws)
        keep_n, kidx_n, kcnt_n = _outputs(cfg, dev)
        torch.cuda.synchronize()
        before = torch.cuda.memory_allocated()
        L.fastar_annca_select_noalloc(q, cfg.F, qb, kp, pb, tau_ca, cfg.topk, 1, keep_n, kidx_n, kcnt_n)
        torch.cuda.synchronize()
        assert torch.cuda.memory_allocated() == before
        # integer outputs of the same kernels on the same inputs: identical
        assert torch.equal(keep_n, keep_r)
        assert torch.equal(kidx_n, kidx_r)
        assert torch.equal(kcnt_n, kcnt_r)
        assert int(kcnt_r.min()) >= cfg.topk


def test_noalloc_rejects_sizes_beyond_its_scratch():
    from kv_cache_tempcache_gb300 import _lib as L
    lib = L.load()
    # H * F * P = 4 * 100 * 1000 > 262144: refused before any device work
    rc = lib.fastar_annca_select_noalloc(0x10000, L.BF16, 4, 100, 64, 128, 8192, 128, 0x10000, 2, 0x10000, 0x10000,
                                         1000, 0.2, 16, 1, 0x10000, 0x10000, 0x10000, None)
    assert rc == L.ECAPACITY
