"""GPU parity of the compaction that also leaves AnnSA's input ready (the new cache, its
keys grouped by bucket, and a bucket-ordered copy of its K/V rows), through the C ABI,
against the oracle bit for bit: the cache order from compact_plan / gather_rows, the
bucket order from bucket_order, and every sorted row equal to the new cache's row at
its kperm entry.  The step's (query, slot) pairs, sorted in the same planning launch,
must be bucket_order's too, and equal to the stand-alone sort's.  The attention that
reads the caller's sorted copy must give exactly what the entry that makes its own copy
gives."""
import numpy as np
import pytest
import torch

from kv_cache_tempcache_gb300 import _lib as L, synth
from oracle import fastar_oracle as O

pytestmark = pytest.mark.gpu


def _i32(a):
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a, np.int32))).cuda()


def _np(t):
    return t.detach().float().cpu().numpy() if t.dtype == torch.bfloat16 else t.detach().cpu().numpy()


@pytest.mark.parametrize("H,M,nq,B,lens,d,dtype", [
    (3, 1000, 600, 16, [1000, 700, 0], 128, "bf16"),     # full, partial and empty incoming caches
    (2, 9360, 4680, 64, [9360, 9000], 128, "bf16"),      # the Wan-1.3B layer's cap and chunk
    (2, 700, 300, 8, [650, 700], 64, "f32"),             # fp32 rows, d = 64 (the SIMT attention path)
])
def test_sorted_compaction_matches_oracle(H, M, nq, B, lens, d, dtype):
    rng = np.random.default_rng(M + B)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    rnd = synth.bf16_round if dtype == "bf16" else (lambda a: a.astype(np.float32))

    def _rows(a):
        return torch.from_numpy(np.ascontiguousarray(rnd(a.astype(np.float32)))).cuda().to(tdt)

    k_in, v_in = rng.standard_normal((2, H, M, d)).astype(np.float32)
    k_cur, v_cur = rng.standard_normal((2, H, nq, d)).astype(np.float32)
    kb_in = rng.integers(0, B, size=(H, M))
    kb_cur = rng.integers(0, B, size=(H, nq))
    knorm_in = rng.random((H, M)).astype(np.float32) + 0.5
    knorm_cur = rng.random((H, nq)).astype(np.float32) + 0.5
    evict = (rng.random((H, M)) < 0.2).astype(np.uint8)
    len_in = np.array(lens)
    dev = dict(
        k_cur=_rows(k_cur), v_cur=_rows(v_cur), kcur_norm=torch.from_numpy(knorm_cur).cuda(),
        kcur_bucket=_i32(kb_cur[..., None]), k_in=_rows(k_in), v_in=_rows(v_in),
        knorm_in=torch.from_numpy(knorm_in).cuda(), kb_in=_i32(kb_in[..., None]), len_in=_i32(len_in),
        evict=torch.from_numpy(evict).cuda())
    out = dict(k_out=torch.zeros((H, M, d), dtype=tdt, device="cuda"),
               v_out=torch.zeros((H, M, d), dtype=tdt, device="cuda"),
               knorm_out=torch.zeros((H, M), dtype=torch.float32, device="cuda"),
               kb_out=torch.zeros((H, M, 1), dtype=torch.int32, device="cuda"),
               len_out=torch.zeros(H, dtype=torch.int32, device="cuda"),
               index_map=torch.zeros((H, M), dtype=torch.int32, device="cuda"))
    kperm = torch.zeros((H, M), dtype=torch.int32, device="cuda")
    koff = torch.zeros((H, B + 1), dtype=torch.int32, device="cuda")
    kpos = torch.zeros((H, M), dtype=torch.int32, device="cuda")
    k_sorted = torch.zeros((H, M, d), dtype=tdt, device="cuda")
    v_sorted = torch.zeros((H, M, d), dtype=tdt, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    r = 2
    qb_h = rng.integers(0, B, size=(H, nq, r))
    qb = _i32(qb_h)
    qperm_c = torch.full((H, nq * r), -5, dtype=torch.int32, device="cuda")
    qoff_c = torch.full((H, B + 1), -5, dtype=torch.int32, device="cuda")
    L.fastar_cache_compact_sorted(dev["k_cur"], dev["v_cur"], dev["kcur_norm"], dev["kcur_bucket"], dev["k_in"],
                                  dev["v_in"], dev["knorm_in"], dev["kb_in"], dev["len_in"], dev["evict"],
                                  out["k_out"], out["v_out"], out["knorm_out"], out["kb_out"], out["len_out"],
                                  out["index_map"], B, kperm, koff, kpos, k_sorted, v_sorted, status, qb=qb,
                                  qperm=qperm_c, qoff=qoff_c)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    want_qperm, want_qoff = O.bucket_order(qb_h, B)
    np.testing.assert_array_equal(_np(qperm_c), want_qperm)
    np.testing.assert_array_equal(_np(qoff_c), want_qoff)
    g = {k: _np(v) for k, v in out.items()}
    kperm_g, koff_g, ks_g, vs_g = _np(kperm), _np(koff), _np(k_sorted), _np(v_sorted)
    kin_b, vin_b = rnd(k_in), rnd(v_in)
    kcur_b, vcur_b = rnd(k_cur), rnd(v_cur)
    kb_new = []
    for h in range(H):
        n = int(len_in[h])
        imap, length = O.compact_plan(evict[h], n, nq, M)
        assert int(g["len_out"][h]) == length
        np.testing.assert_array_equal(g["index_map"][h], imap)
        np.testing.assert_array_equal(g["k_out"][h, :length], O.gather_rows(imap, length, kin_b[h, :n], kcur_b[h]))
        np.testing.assert_array_equal(g["v_out"][h, :length], O.gather_rows(imap, length, vin_b[h, :n], vcur_b[h]))
        np.testing.assert_array_equal(g["knorm_out"][h, :length],
                                      O.gather_rows(imap, length, knorm_in[h, :n], knorm_cur[h]))
        kb = O.gather_rows(imap, length, kb_in[h, :n], kb_cur[h])
        np.testing.assert_array_equal(g["kb_out"][h, :length, 0], kb)
        kb_new.append(np.pad(kb, (0, M - length)))
    want_perm, want_off = O.bucket_order(np.stack(kb_new)[..., None], B, g["len_out"])
    np.testing.assert_array_equal(koff_g, want_off)
    for h in range(H):
        length = int(g["len_out"][h])
        np.testing.assert_array_equal(kperm_g[h, :length], want_perm[h, :length])
        # the sorted copy is the new cache's rows in bucket order
        np.testing.assert_array_equal(ks_g[h, :length], g["k_out"][h, want_perm[h, :length]])
        np.testing.assert_array_equal(vs_g[h, :length], g["v_out"][h, want_perm[h, :length]])

    # the attention that reads this copy equals the one that makes its own, bit for bit
    q = _rows(rng.standard_normal((H, nq, d)).astype(np.float32))
    qperm = torch.zeros((H, nq * r), dtype=torch.int32, device="cuda")
    qoff = torch.zeros((H, B + 1), dtype=torch.int32, device="cuda")
    L.fastar_bucket_sort(qb, B, qperm, qoff, None, status)
    torch.cuda.synchronize()
    assert torch.equal(qperm, qperm_c) and torch.equal(qoff, qoff_c)
    ws = torch.zeros(L.workspace_bytes(L.OP_SPARSE_ATTN, H, n=nq, M=M, d=d, B=B, r=r), dtype=torch.uint8,
                     device="cuda")
    res = []
    for presorted in (False, True):
        o = torch.zeros((H, nq, d), dtype=tdt, device="cuda")
        lse = torch.zeros((H, nq), dtype=torch.float32, device="cuda")
        if presorted:
            L.fastar_sparse_attn_presorted(q, r, B, qperm, qoff, out["k_out"], out["v_out"], kperm, koff, k_sorted,
                                           v_sorted, d ** -0.5, o, lse, status, ws)
        else:
            L.fastar_sparse_attn(q, r, B, qperm, qoff, out["k_out"], out["v_out"], kperm, koff, d ** -0.5, o, lse,
                                 status, ws)
        torch.cuda.synchronize()
        res.append((_np(o), _np(lse)))
    assert int(status.item()) == 0
    np.testing.assert_array_equal(res[0][0], res[1][0])
    np.testing.assert_array_equal(res[0][1], res[1][1])
