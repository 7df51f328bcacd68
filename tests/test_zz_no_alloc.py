"""The allocation-free AnnCA selection entry point against the regular one and the oracle.

Some callers cannot allocate device memory while they run the step (a server that
reserves all device memory at start-up, a process under a fixed shared budget);
fastar_annca_select_noalloc serves them from a fixed scratch array inside the
library.  Its results must equal the regular entry point's on the same inputs, on
consecutive calls of different sizes (the shared scratch keeps the previous call's
contents, which a smaller call must never read), and must be correct answers for the
oracle's selection on the same inputs.  No device memory may be allocated by a call.
This file is collected last on purpose."""
import numpy as np
import pytest
import torch

import parity
from kv_cache_tempcache_gb300 import synth
from oracle import fastar_oracle as O

pytestmark = pytest.mark.gpu


def _case(seed, F, Tf, P):
    from kv_cache_tempcache_gb300 import _lib as L
    cfg = synth.LayerConfig(name="noalloc", H=3, d=128, Tf=Tf, F=F, prior_frames=0, P=P, C=8, sigma_mix=0.3,
                            rho=0.1, drift=0.05, qnoise=0.1, tau=0.95, M=F * Tf, B=16, r=2, tau_ca=0.2, topk=16,
                            dtype="bf16")
    inp = synth.layer_step_inputs(cfg, seed=seed)
    dev = torch.device("cuda")
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev).to(torch.bfloat16)
    q, kp, C = t(inp["q"]), t(inp["kp"]), t(inp["centroids"])
    qb = torch.zeros((cfg.H, cfg.Nq, cfg.r), dtype=torch.int32, device=dev)
    pb = torch.zeros((cfg.H, cfg.P, 1), dtype=torch.int32, device=dev)
    L.fastar_bucket_assign(q, C, cfg.r, qb)
    L.fastar_bucket_assign(kp, C, 1, pb)
    return cfg, inp, q, kp, qb, pb


def _outputs(cfg, dev):
    return (torch.full((cfg.H, cfg.F, cfg.P), 7, dtype=torch.uint8, device=dev),
            torch.full((cfg.H, cfg.F, cfg.P), -7, dtype=torch.int32, device=dev),
            torch.full((cfg.H, cfg.F), -7, dtype=torch.int32, device=dev))


def _check_against_oracle(cfg, inp, qb, pb, keep, kidx, kcnt, tau_ca, counts):
    """The buckets the GPU assigned are validated first, then the selection is checked
    against the oracle's on those buckets (near-ties at the threshold or the top-k edge
    may go either way)."""
    qb, pb = qb.cpu().numpy(), pb.cpu().numpy()[..., 0]
    keep, kidx, kcnt = keep.cpu().numpy(), kidx.cpu().numpy(), kcnt.cpu().numpy()
    for h in range(cfg.H):
        C, q, kp = inp["centroids"][h], inp["q"][h], inp["kp"][h]
        counts["topr"] += parity.check_topr(O.centroid_scores(q, C), qb[h], "query buckets")
        counts["key"] += parity.check_argmax(O.centroid_scores(kp, C), pb[h], "prompt buckets")
        _, _, _, score = O.annca_select(q, qb[h], kp, pb[h], cfg.F, cfg.Tf, tau_ca, cfg.topk)
        for f in range(cfg.F):
            counts["keep"] += parity.check_keep(score[f], keep[h, f], tau_ca, cfg.topk, f"keep head {h} frame {f}")
            idx = np.flatnonzero(keep[h, f])
            assert int(kcnt[h, f]) == len(idx)
            assert np.array_equal(kidx[h, f, :len(idx)], idx)
            assert np.all(kidx[h, f, len(idx):] == -1)


def test_noalloc_selection_equals_regular_on_consecutive_calls():
    from kv_cache_tempcache_gb300 import _lib as L
    from kv_cache_tempcache_gb300.build_lib import build
    build()
    L.load()
    dev = torch.device("cuda")
    counts = dict(topr=0, key=0, keep=0)
    # a large call, then smaller ones (fewer frames, fewer prompt tokens) on the same
    # scratch, then the large shape again with other data
    for i, (seed, F, Tf, P, tau_ca) in enumerate(((0, 3, 300, 200, 0.2), (1, 2, 250, 120, 0.35),
                                                  (2, 1, 300, 64, 0.2), (3, 3, 300, 200, 0.25))):
        cfg, inp, q, kp, qb, pb = _case(seed, F, Tf, P)
        keep_r, kidx_r, kcnt_r = _outputs(cfg, dev)
        ws = torch.zeros(L.workspace_bytes(L.OP_ANNCA, cfg.H, 0, 0, cfg.d, cfg.B, cfg.r, cfg.P, cfg.F),
                         dtype=torch.uint8, device=dev)
        L.fastar_annca_select(q, cfg.F, qb, kp, pb, tau_ca, cfg.topk, 1, keep_r, kidx_r, kcnt_r, None, ws)
        keep_n, kidx_n, kcnt_n = _outputs(cfg, dev)
        torch.cuda.synchronize()
        before = torch.cuda.memory_allocated()
        free_before = torch.cuda.mem_get_info()[0]
        L.fastar_annca_select_noalloc(q, cfg.F, qb, kp, pb, tau_ca, cfg.topk, 1, keep_n, kidx_n, kcnt_n)
        torch.cuda.synchronize()
        # neither the caching allocator nor the driver handed out memory for the call (the
        # first call of the process may load the library's module, array included)
        assert torch.cuda.memory_allocated() == before
        if i > 0:
            assert torch.cuda.mem_get_info()[0] == free_before
        # integer outputs of the same kernels on the same inputs: identical
        assert torch.equal(keep_n, keep_r)
        assert torch.equal(kidx_n, kidx_r)
        assert torch.equal(kcnt_n, kcnt_r)
        assert int(kcnt_r.min()) >= min(cfg.topk, cfg.P)
        _check_against_oracle(cfg, inp, qb, pb, keep_n, kidx_n, kcnt_n, tau_ca, counts)
    parity.report("AnnCA selection without allocation (4 consecutive calls)", counts)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    from kv_cache_tempcache_gb300 import _lib as L
    lib = L.load()
    # H * F * P = 4 * 100 * 1000 > 262144: refused before any device work
    rc = lib.fastar_annca_select_noalloc(0x10000, L.BF16, 4, 100, 64, 128, 8192, 128, 0x10000, 2, 0x10000, 0x10000,
                                         1000, 0.2, 16, 1, 0x10000, 0x10000, 0x10000, None)
    assert rc == L.ECAPACITY
