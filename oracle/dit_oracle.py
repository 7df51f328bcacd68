"""Plain CPU oracle of the diffusion transformer around the FAST-AR attention step.
TEST INFRASTRUCTURE.

Only the tests, the package's smoke check and the benchmark's CPU-baseline arm may
import or run this module.  It shares no code with the CUDA path and imports nothing
from it; the product path never calls it.

The pages describe FAST-AR as a drop-in replacement for the attention layers of an
autoregressive video diffusion transformer (blog, Significance; technical summary, Key
Results: Rolling-Forcing and LongVie2 on Wan-family backbones); the transformer itself is
not on the pages.  This module writes out, in float64 NumPy, a Wan2.1-shaped block with
the plainest reading of each operation (the readings are listed in the design notes):
layer norm with adaptive shift/scale/gate modulation (adaLN), fused QKV projection, RMS
norm of q and k, rotary positions over (frame, row, column), self-attention, a second
normed cross-attention over the text, a GELU(tanh) feed-forward, and the flow-matching
Euler update of the denoising loop.
"""
from __future__ import annotations

import numpy as np


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


# ----------------------------------------------------------------------------------
# elementwise and GEMM
# ----------------------------------------------------------------------------------

def gelu_tanh(x) -> np.ndarray:
    """0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))."""
    x = _f64(x)
    return 0.5 * x * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * (x + 0.044715 * x ** 3)))


def silu(x) -> np.ndarray:
    """x / (1 + exp(-x))."""
    x = _f64(x)
    return x / (1.0 + np.exp(-x))


ACTS = {0: lambda v: v, 1: gelu_tanh, 2: silu}


def gemm(A, W, bias=None, act: int = 0, R=None, gate=None) -> np.ndarray:
    """R + gate * act(A @ W^T + bias); without R: act(A @ W^T + bias).
    A [M, K]; W [N, K] (a Linear weight); bias, gate [N]."""
    Y = _f64(A) @ _f64(W).T
    if bias is not None:
        Y = Y + _f64(bias)[None, :]
    Y = ACTS[act](Y)
    if R is not None:
        g = np.ones(Y.shape[1]) if gate is None else _f64(gate)
        Y = _f64(R) + g[None, :] * Y
    return Y
