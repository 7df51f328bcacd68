"""GPU parity of the row-wise operations of the DiT around the attention step (layer norm
with adaptive modulation, RMS norm with rotary positions, the sinusoidal timestep
embedding) against the oracle, through the C ABI.  Outputs are rounded once to bf16:
|got - want| <= 2^-8 |want| + 1e-3 max|want|."""
import numpy as np
import pytest
import torch

from kv_cache_tempcache_gb300 import _lib as L, synth
from oracle import dit_oracle as D

pytestmark = pytest.mark.gpu


def _bf(a):
    return torch.from_numpy(np.ascontiguousarray(synth.bf16_round(a.astype(np.float32)))).cuda().to(torch.bfloat16)


def _f32(a):
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a, np.float32))).cuda()


def _check(got, want):
    got = got.float().cpu().numpy().astype(np.float64)
    bound = 2.0 ** -8 * np.abs(want) + 1e-3 * np.abs(want).max()
    bad = np.abs(got - want) > bound
    assert not bad.any(), f"{int(bad.sum())} of {bad.size} outside the bound; worst {np.abs(got - want).max():.3e}"


@pytest.mark.parametrize("C", [64, 1536, 4096])
@pytest.mark.parametrize("affine,mod", [(False, False), (True, False), (False, True), (True, True)])
def test_layernorm_mod(C, affine, mod):
    rng = np.random.default_rng(C + 2 * affine + mod)
    n = 301
    x = synth.bf16_round((rng.standard_normal((n, C)) * 2 + 0.5).astype(np.float32))
    w, b = rng.standard_normal(C), rng.standard_normal(C)
    sha, shb, sca, scb = (rng.standard_normal(C) * 0.3 for _ in range(4))
    out = torch.empty((n, C), dtype=torch.bfloat16, device="cuda")
    kw = dict(weight=_f32(w), bias=_f32(b)) if affine else {}
    if mod:
        kw.update(shift_a=_f32(sha), shift_b=_f32(shb), scale_a=_f32(sca), scale_b=_f32(scb))
    L.fastar_layernorm_mod(_bf(x), out, eps=1e-6, **kw)
    torch.cuda.synchronize()
    want = D.layer_norm(x, 1e-6, w if affine else None, b if affine else None)
    if mod:
        want = D.modulate(want, sha + shb, sca + scb)
    _check(out, want)


@pytest.mark.parametrize("norm,rope", [(True, False), (False, True), (True, True)])
def test_rmsnorm_rope_on_a_qkv_slice(norm, rope):
    rng = np.random.default_rng(10 + 2 * norm + rope)
    n, H, d = 4680, 12, 128
    C = H * d
    qkv = synth.bf16_round(rng.standard_normal((n, 3 * C)).astype(np.float32))
    w = rng.standard_normal(C) * 0.5 + 1
    buf = _bf(qkv)
    view = buf[:, C:2 * C]                      # the k part of a fused projection, in place
    L.fastar_rmsnorm_rope(view, d, weight=_f32(w) if norm else None, rope=rope, t0=9, grid=(30, 52))
    torch.cuda.synchronize()
    want = qkv[:, C:2 * C].astype(np.float64)
    if norm:
        want = D.rms_norm(want, w, 1e-6)
    if rope:
        want = D.rope(want, d, D.token_positions(n, 9, 30, 52))
    _check(view, want)
    # the neighbouring slices are untouched
    np.testing.assert_array_equal(buf[:, :C].float().cpu().numpy(), qkv[:, :C])
    np.testing.assert_array_equal(buf[:, 2 * C:].float().cpu().numpy(), qkv[:, 2 * C:])


def test_rmsnorm_rope_head_dim_64():
    rng = np.random.default_rng(3)
    n, H, d = 517, 4, 64
    x = synth.bf16_round(rng.standard_normal((n, H * d)).astype(np.float32))
    w = rng.standard_normal(H * d)
    t = _bf(x)
    L.fastar_rmsnorm_rope(t, d, weight=_f32(w), rope=True, t0=2, grid=(11, 13))
    torch.cuda.synchronize()
    _check(t, D.rope(D.rms_norm(x, w, 1e-6), d, D.token_positions(n, 2, 11, 13)))


def test_sinusoidal_embedding():
    t = np.array([0.0, 1.0, 250.0, 999.0], np.float32)
    out = torch.empty((4, 256), dtype=torch.bfloat16, device="cuda")
    L.fastar_sinusoidal_embedding(_f32(t), out)
    torch.cuda.synchronize()
    want = D.sinusoidal(t, 256)
    np.testing.assert_allclose(out.float().cpu().numpy(), want, rtol=0, atol=2 ** -8 + 1e-4)
