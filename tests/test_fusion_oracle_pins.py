"""Pins for the EvoFusion upstream oracle (oracle/fusion.py): LayerNorm of the
pair representation over its channels followed by one bias-free projection
into q, k, v, g and the pair bias.  Checked without re-typing the oracle's
formula:
* a worked LayerNorm example small enough to do by hand;
* closed-form invariants: every normalised row has mean 0 and variance
  var/(var + eps); LayerNorm ignores a per-row shift and a positive per-row
  scale of its input;
* the projection is linear in the weights, and a weight matrix that copies
  channels returns those channels of the normalised input in the documented
  q | k | v | g | bias column order and [b, h, i, j] bias layout;
* an independent library: torch's float64 layer_norm and matmul.
"""
import numpy as np
import pytest
import torch

from oracle import fusion


def _rand(shape, seed, scale=1.0):
    g = np.random.default_rng(seed)
    return g.standard_normal(shape) * scale


def test_worked_example_from_the_definition():
    """Two rows worked by hand: [1, 2, 3, 4] has mean 2.5 and (population)
    variance 1.25; [2, 2, 2, 6] has mean 3 and variance 3."""
    z = np.array([[1.0, 2.0, 3.0, 4.0], [2.0, 2.0, 2.0, 6.0]])
    r1, r3 = 1.25 ** -0.5, 3.0 ** -0.5
    expected = np.array([[-1.5 * r1, -0.5 * r1, 0.5 * r1, 1.5 * r1],
                         [-1.0 * r3, -1.0 * r3, -1.0 * r3, 3.0 * r3]])
    out = fusion.layer_norm(z, np.ones(4), np.zeros(4), eps=0.0)
    np.testing.assert_allclose(out, expected, rtol=0, atol=1e-12)
    # gamma and beta act per channel after the standardisation
    gamma, beta = np.array([1.0, 2.0, -1.0, 0.5]), np.array([0.0, 1.0, 2.0, -3.0])
    np.testing.assert_allclose(fusion.layer_norm(z, gamma, beta, eps=0.0),
                               expected * gamma + beta, rtol=0, atol=1e-12)


def test_rows_are_standardised():
    z = _rand((2, 5, 5, 16), 1, 3.0) + 7.0
    eps = 1e-5
    y = fusion.layer_norm(z, np.ones(16), np.zeros(16), eps)
    var = z.var(axis=-1)
    np.testing.assert_allclose(y.mean(axis=-1), 0.0, atol=1e-12)
    np.testing.assert_allclose((y * y).mean(axis=-1), var / (var + eps), rtol=1e-12)


def test_invariant_to_row_shift_and_scale():
    z = _rand((1, 4, 4, 32), 2)
    gamma, beta = 1 + 0.1 * _rand(32, 3), 0.1 * _rand(32, 4)
    shift = _rand((1, 4, 4, 1), 5, 10.0)
    scale = np.exp(_rand((1, 4, 4, 1), 6))
    a = fusion.layer_norm(z, gamma, beta, eps=0.0)
    b = fusion.layer_norm(z * scale + shift, gamma, beta, eps=0.0)
    np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-10)


def test_projection_column_order_and_bias_layout():
    B, N, C, H, D = 1, 3, 8, 2, 2
    z = _rand((B, N, N, C), 7)
    gamma, beta = 1 + 0.2 * _rand(C, 8), 0.3 * _rand(C, 9)
    y = fusion.layer_norm(z, gamma, beta)
    # weight row o copies channel o % C
    w = np.zeros((4 * H * D + H, C))
    for o in range(w.shape[0]):
        w[o, o % C] = 1.0
    q, k, v, g, bias = fusion.ln_proj(z, gamma, beta, w, H, D)
    cols = [y[..., [o % C for o in range(i * H * D, (i + 1) * H * D)]].reshape(B, N, N, H, D)
            for i in range(4)]
    for got, want in zip((q, k, v, g), cols):
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-14)
    for h in range(H):
        np.testing.assert_allclose(bias[:, h], y[..., (4 * H * D + h) % C], rtol=0, atol=1e-14)


def test_projection_is_linear_in_the_weights():
    B, N, C, H, D = 1, 4, 16, 2, 4
    z = _rand((B, N, N, C), 10)
    gamma, beta = np.ones(C), np.zeros(C)
    w1, w2 = _rand((4 * H * D + H, C), 11), _rand((4 * H * D + H, C), 12)
    a = fusion.ln_proj(z, gamma, beta, w1, H, D)
    b = fusion.ln_proj(z, gamma, beta, w2, H, D)
    c = fusion.ln_proj(z, gamma, beta, w1 + 2.0 * w2, H, D)
    for x, y, s in zip(a, b, c):
        np.testing.assert_allclose(s, x + 2.0 * y, rtol=1e-12, atol=1e-12)


def test_matches_torch_layer_norm_and_matmul():
    B, N, C, H, D = 2, 6, 32, 2, 8
    z = _rand((B, N, N, C), 13, 2.0)
    gamma, beta = 1 + 0.1 * _rand(C, 14), 0.1 * _rand(C, 15)
    w = _rand((4 * H * D + H, C), 16, C ** -0.5)
    q, k, v, g, bias = fusion.ln_proj(z, gamma, beta, w, H, D, eps=1e-5)
    zt = torch.tensor(z)
    yt = torch.nn.functional.layer_norm(zt, (C,), torch.tensor(gamma), torch.tensor(beta), 1e-5)
    out = torch.matmul(yt, torch.tensor(w).T)
    hd = H * D
    for i, got in enumerate((q, k, v, g)):
        np.testing.assert_allclose(got, out[..., i * hd:(i + 1) * hd].reshape(B, N, N, H, D).numpy(),
                                   rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(bias, out[..., 4 * hd:].permute(0, 3, 1, 2).numpy(), rtol=1e-12,
                               atol=1e-12)
