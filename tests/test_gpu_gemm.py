"""GPU parity of the tensor-core GEMM (the projections and feed-forward of the DiT around
the attention step) against the oracle, through the C ABI: every epilogue, ragged M,
the DiT's shapes, in-place residual updates, and the argument checks.

Tolerance: inputs are bf16-exact; the product accumulates in fp32 (relative error far
below 1e-5 here) and the output is rounded once to bf16 (relative 2^-9), so
|got - want| <= 2^-8 |want| + 1e-3 max|want| covers it with margin."""
import numpy as np
import pytest
import torch

from kv_cache_tempcache_gb300 import _lib as L, synth
from oracle import dit_oracle as D

pytestmark = pytest.mark.gpu


def _bf(a):
    return torch.from_numpy(np.ascontiguousarray(synth.bf16_round(a.astype(np.float32)))).cuda().to(torch.bfloat16)


def _f32(a):
    return torch.from_numpy(np.ascontiguousarray(a.astype(np.float32))).cuda()


def _check(got, want):
    got = got.float().cpu().numpy().astype(np.float64)
    bound = 2.0 ** -8 * np.abs(want) + 1e-3 * np.abs(want).max()
    bad = np.abs(got - want) > bound
    assert not bad.any(), f"{int(bad.sum())} of {bad.size} outside the bound; worst {np.abs(got - want).max():.3e}"


@pytest.mark.parametrize("M,N,K", [(1, 256, 64), (129, 512, 128), (300, 256, 1536), (4680, 1536, 64)])
@pytest.mark.parametrize("act", [L.ACT_NONE, L.ACT_GELU_TANH, L.ACT_SILU])
def test_gemm_shapes_and_activations(M, N, K, act):
    rng = np.random.default_rng(M + N + K + act)
    A = synth.bf16_round(rng.standard_normal((M, K)).astype(np.float32))
    W = synth.bf16_round((rng.standard_normal((N, K)) / np.sqrt(K)).astype(np.float32))
    bias = rng.standard_normal(N).astype(np.float32)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    L.fastar_gemm(_bf(A), _bf(W), C, bias=_f32(bias), act=act)
    torch.cuda.synchronize()
    _check(C, D.gemm(A, W, bias, act))


def test_fp32_output():
    rng = np.random.default_rng(11)
    M, N, K = 3, 9216, 1536                       # the shape of the modulation vectors
    A = synth.bf16_round(rng.standard_normal((M, K)).astype(np.float32))
    W = synth.bf16_round((rng.standard_normal((N, K)) / np.sqrt(K)).astype(np.float32))
    bias = rng.standard_normal(N).astype(np.float32)
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    L.fastar_gemm(_bf(A), _bf(W), C, bias=_f32(bias), act=L.ACT_SILU)
    torch.cuda.synchronize()
    want = D.gemm(A, W, bias, L.ACT_SILU)
    np.testing.assert_allclose(C.cpu().numpy(), want, rtol=1e-4, atol=1e-4 * np.abs(want).max())


def test_gated_residual_in_place_and_strided_views():
    rng = np.random.default_rng(7)
    M, N, K = 700, 1536, 512
    A = synth.bf16_round(rng.standard_normal((M, K)).astype(np.float32))
    W = synth.bf16_round((rng.standard_normal((N, K)) / np.sqrt(K)).astype(np.float32))
    R = synth.bf16_round(rng.standard_normal((M, N)).astype(np.float32))
    ga, gb = rng.standard_normal(N).astype(np.float32), rng.standard_normal(N).astype(np.float32)
    # A as a column slice of a wider buffer (leading dimension > K); C written over R
    Abig = torch.zeros((M, K + 256), dtype=torch.bfloat16, device="cuda")
    Abig[:, 128:128 + K] = _bf(A)
    Rt = _bf(R)
    L.fastar_gemm(Abig[:, 128:128 + K], _bf(W), Rt, R=Rt, gate_a=_f32(ga), gate_b=_f32(gb))
    torch.cuda.synchronize()
    _check(Rt, D.gemm(A, W, None, 0, R, ga + gb))
    # gate_a alone, no bias; then no gate (gate 1)
    Rt = _bf(R)
    L.fastar_gemm(_bf(A), _bf(W), Rt, R=Rt, gate_a=_f32(ga))
    torch.cuda.synchronize()
    _check(Rt, D.gemm(A, W, None, 0, R, ga))
    Rt = _bf(R)
    L.fastar_gemm(_bf(A), _bf(W), Rt, R=Rt)
    torch.cuda.synchronize()
    _check(Rt, D.gemm(A, W, None, 0, R, None))


@pytest.mark.parametrize("N,K,act", [(4608, 1536, L.ACT_NONE), (8960, 1536, L.ACT_GELU_TANH), (1536, 8960, L.ACT_NONE)])
def test_dit_shapes_sampled_rows(N, K, act):
    rng = np.random.default_rng(N + K)
    M = 4680
    A = synth.bf16_round(rng.standard_normal((M, K)).astype(np.float32))
    W = synth.bf16_round((rng.standard_normal((N, K)) / np.sqrt(K)).astype(np.float32))
    bias = rng.standard_normal(N).astype(np.float32) * 0.1
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    L.fastar_gemm(_bf(A), _bf(W), C, bias=_f32(bias), act=act)
    torch.cuda.synchronize()
    rows = np.concatenate([np.arange(0, 130), rng.choice(M, 200, replace=False), np.arange(M - 60, M)])
    _check(C[torch.from_numpy(rows).cuda()], D.gemm(A[rows], W, bias, act))


def test_argument_checks():
    x = torch.zeros((128, 256), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((300, 256), dtype=torch.bfloat16, device="cuda")
    c = torch.zeros((128, 300), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(L.FastarError) as e:
        L.fastar_gemm(x, w, c)                      # N = 300 is not a multiple of 256
    assert e.value.code == L.EUNSUPPORTED
    y = torch.zeros((256, 256), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(L.FastarError) as e:
        L.fastar_gemm(y, y, y)                      # C over A
    assert e.value.code == L.EINVAL
