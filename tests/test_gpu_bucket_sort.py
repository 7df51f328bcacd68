"""GPU parity of the stable counting sort that groups (token, slot) elements by bucket,
through the C ABI, against the oracle's bucket order, bit for bit: at the layer's sizes,
at sizes past the per-CTA staging bound, with partial lengths, an empty head, several
slots per token and the largest bucket count."""
import numpy as np
import pytest
import torch

from kv_cache_tempcache_gb300 import _lib as L
from oracle import fastar_oracle as O

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("H,n,r,B,partial", [
    (12, 9360, 1, 64, True),      # the layer's cache keys
    (12, 4680, 2, 64, False),     # the layer's (query, slot) pairs
    (3, 90000, 1, 256, True),     # chunks past the per-CTA staging bound: ids read from global
    (2, 14400, 2, 128, False),    # 28800 pairs per head
    (4, 777, 3, 5, True),         # ragged, few buckets
])
def test_bucket_sort_matches_oracle(H, n, r, B, partial):
    rng = np.random.default_rng(n + B)
    # skewed bucket sizes: a few heavy buckets and a long tail
    p = rng.dirichlet(np.full(B, 0.3))
    ids = rng.choice(B, size=(H, n, r), p=p).astype(np.int32)
    n_valid = rng.integers(0, n + 1, size=H).astype(np.int32) if partial else None
    if partial:
        n_valid[0] = 0
        n_valid[-1] = n
    want_perm, want_off = O.bucket_order(ids, B, n_valid)
    perm = torch.full((H, n * r), -1, dtype=torch.int32, device="cuda")
    off = torch.zeros((H, B + 1), dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    nv = torch.from_numpy(n_valid).cuda() if partial else None
    L.fastar_bucket_sort(torch.from_numpy(ids).cuda(), B, perm, off, nv, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    np.testing.assert_array_equal(off.cpu().numpy(), want_off)
    got = perm.cpu().numpy()
    for h in range(H):
        cnt = int(want_off[h, B])
        np.testing.assert_array_equal(got[h, :cnt], want_perm[h, :cnt])
