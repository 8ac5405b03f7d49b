"""EvoFusion upstream oracle -- test infrastructure only.

A plain float64 CPU statement of the operator stack that feeds triangle
attention: LayerNorm of the pair representation over its channel axis, then
one linear projection without a bias term whose output columns are the
queries, keys, values and gate of every head and the pair bias of every head.

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
