"""EvoFusion oracles -- test infrastructure only.

Plain float64 CPU statements of the operator stacks around triangle
attention.  Upstream: LayerNorm of the pair representation over its channel
axis, then one linear projection without a bias term whose output columns
are the queries, keys, values and gate of every head and the pair bias of
every head.  Downstream: the SwiGLU transition of the pair representation
with its residual add.

MegaFold technical summary, "Methodik" section 3 "EvoFusion", Umfang and
Mechanismus: EvoFusion restructures layer normalisation and the linear
projections that follow it so that the normalised N x N tensor is never
written to HBM between the two.  The pages print no formula; this module
takes the plainest reading (LayerNorm with per-channel scale and shift and a
variance without Bessel's correction, epsilon added to the variance; a single
bias-free weight matrix whose output columns are laid out q | k | v | g |
pair bias, heads major within each of q, k, v, g).  The fused kernel must
compute exactly this up to its stated rounding.

Only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  The product library never does, and
this module imports nothing from the product.

The downstream stack is named in the same passage (Umfang: layer
normalisation, linear projections and SwiGLU activations).  The pages print
no formula for it either; the plainest reading, taken here, is what follows
the gated attention in AlphaFold3-style pair stacks: the attention's
bias-free output projection from H*D back to C channels and its residual add,
then the transition block -- LayerNorm as above, two bias-free projections to
F hidden units (a SiLU branch and a linear branch), their product, a
bias-free projection back to C channels, and the residual add of the
block's input.

Parity status: pinned (tests/test_fusion_oracle_pins.py).
"""
from __future__ import annotations

import numpy as np


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        import torch
        x = x.detach().to(torch.float64).cpu().contiguous().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def layer_norm(z, gamma, beta, eps=1e-5):
    """LayerNorm over the last axis: (z - mean) / sqrt(var + eps) * gamma + beta,
    var the mean squared deviation (no Bessel correction)."""
    z = _f64(z)
    mean = z.mean(axis=-1, keepdims=True)
    dev = z - mean
    var = (dev * dev).mean(axis=-1, keepdims=True)
    return dev / np.sqrt(var + eps) * _f64(gamma) + _f64(beta)


def ln_proj(z, gamma, beta, w, H, D, eps=1e-5):
    """The fused upstream stack of triangle attention.

    z     : [B, N, N, C] pair representation.
    gamma, beta : [C] LayerNorm scale and shift.
    w     : [4*H*D + H, C] projection weights (row o produces output column o).
    Returns float64 arrays q, k, v, g of shape [B, N, N, H, D] (the pair
    projections in the layout the attention reads as starting- or ending-node
    views) and pair_bias of shape [B, H, N, N] (indexed [b, h, i, j]).
    """
    y = layer_norm(z, gamma, beta, eps)
    w = _f64(w)
    B, N, N2, C = y.shape
    assert N2 == N and w.shape == (4 * H * D + H, C)
    out = y.reshape(-1, C) @ w.T          # [B*N*N, 4HD + H]
    hd = H * D
    parts = [out[:, i * hd:(i + 1) * hd].reshape(B, N, N, H, D) for i in range(4)]
    bias = out[:, 4 * hd:].reshape(B, N, N, H).transpose(0, 3, 1, 2).copy()
    return parts[0], parts[1], parts[2], parts[3], bias


def silu(x):
    """x * sigmoid(x) = x / (1 + exp(-x)), written so that it does not
    overflow for large negative x."""
    x = _f64(x)
    e = np.exp(-np.abs(x))
    return np.where(x >= 0, x / (1.0 + e), x * e / (1.0 + e))


def transition(z, gamma, beta, w1, w2, eps=1e-5, o=None, w_o=None):
    """The output projection of the gated attention with its residual add
    (when o is given), then the SwiGLU transition with its residual add.

    z      : [B, N, N, C] pair representation.
    o      : [B, N, N, HD] gated attention output of the same rows (optional).
    w_o    : [C, HD] output projection (given exactly when o is).
    gamma, beta : [C] LayerNorm scale and shift.
    w1     : [2F, C]: rows 0..F-1 the SiLU branch, rows F..2F-1 the linear branch.
    w2     : [C, F].
    Returns float64 out [B, N, N, C] = z1 + (silu(y w1a^T) * (y w1b^T)) w2^T,
    y = LayerNorm(z1), z1 = z + o w_o^T (z1 = z without o).
    """
    z = _f64(z)
    assert (o is None) == (w_o is None)
    if o is not None:
        z = z + _f64(o) @ _f64(w_o).T
    y = layer_norm(z, gamma, beta, eps)
    w1, w2 = _f64(w1), _f64(w2)
    F = w1.shape[0] // 2
    assert w1.shape == (2 * F, z.shape[-1]) and w2.shape == (z.shape[-1], F)
    a = y @ w1[:F].T
    b = y @ w1[F:].T
    h = silu(a) * b
    return z + h @ w2.T
