"""Pins for the EvoFusion downstream oracle (oracle/fusion.py `transition`,
`silu`): the attention's output projection with its residual add, then the
SwiGLU transition of the pair representation with its residual add.  Checked
without re-typing the oracle's formula:
* SiLU against its closed-form values (silu(0) = 0, silu(1) = e / (1 + e),
  silu(-1) = -1 / (1 + e)), the identity silu(x) - silu(-x) = x, and its
  limits (x for large x, 0 for large negative x, no overflow);
* a transition worked by hand on a two-channel row;
* special cases: zero output weights, or a zero linear branch, return z
  exactly; the update out - z is linear in w2, ignores a per-row shift of z
  (the LayerNorm removes it), and rows are independent;
* the output projection: a zero w_o changes nothing, a zero linear branch
  leaves z + o w_o^T (checked against torch's float64 matmul), and a worked
  row by hand;
* an independent library: torch's float64 layer_norm, silu and matmul.
"""
import math

import numpy as np
import pytest
import torch

from oracle import fusion


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _inputs(seed, B=1, N=3, C=8, F=16):
    z = _rand((B, N, N, C), seed) * 1.5 + 0.3
    gamma = 1.0 + 0.1 * _rand(C, seed + 1)
    beta = 0.1 * _rand(C, seed + 2)
    w1 = _rand((2 * F, C), seed + 3, C ** -0.5)
    w2 = _rand((C, F), seed + 4, F ** -0.5)
    return z, gamma, beta, w1, w2


def test_silu_closed_forms():
    e = math.e
    got = fusion.silu(np.array([0.0, 1.0, -1.0, 2.0]))
    np.testing.assert_allclose(got, [0.0, e / (1 + e), -1 / (1 + e), 2 * e * e / (1 + e * e)],
                               rtol=1e-15, atol=0)
    x = _rand(50, 7, 4.0)
    np.testing.assert_allclose(fusion.silu(x) - fusion.silu(-x), x, rtol=0, atol=1e-12)
    big = fusion.silu(np.array([40.0, -40.0, 800.0, -800.0]))
    assert np.all(np.isfinite(big))
    np.testing.assert_allclose(big, [40.0, -40.0 * math.exp(-40.0), 800.0, 0.0],
                               rtol=1e-14, atol=1e-300)


def test_worked_example_by_hand():
    """z = [1, 3]: mean 2, variance 1, so y = [-1, 1] (gamma 1, beta 0, eps
    0).  With w1 rows a = [0, 1] and b = [0, 3]: a = 1, b = 3,
    h = 3 silu(1) = 3 e / (1 + e); w2 = [[1], [-2]] adds h and -2h."""
    z = np.array([[[[1.0, 3.0]]]])
    w1 = np.array([[0.0, 1.0], [0.0, 3.0]])
    w2 = np.array([[1.0], [-2.0]])
    h = 3 * math.e / (1 + math.e)
    out = fusion.transition(z, np.ones(2), np.zeros(2), w1, w2, eps=0.0)
    np.testing.assert_allclose(out.reshape(2), [1.0 + h, 3.0 - 2 * h], rtol=0, atol=1e-14)


def test_zero_output_weights_or_linear_branch_return_z():
    z, gamma, beta, w1, w2 = _inputs(11)
    assert np.array_equal(fusion.transition(z, gamma, beta, w1, np.zeros_like(w2)), z)
    F = w2.shape[1]
    w1b0 = w1.copy()
    w1b0[F:] = 0.0
    assert np.array_equal(fusion.transition(z, gamma, beta, w1b0, w2), z)


def test_update_is_linear_in_w2_and_ignores_a_row_shift():
    z, gamma, beta, w1, w2 = _inputs(12)
    t1 = fusion.transition(z, gamma, beta, w1, w2) - z
    t2 = fusion.transition(z, gamma, beta, w1, -2.5 * w2) - z
    np.testing.assert_allclose(t2, -2.5 * t1, rtol=1e-12, atol=1e-12)
    shift = _rand(z.shape[:-1] + (1,), 13, 3.0)
    t3 = fusion.transition(z + shift, gamma, beta, w1, w2) - (z + shift)
    np.testing.assert_allclose(t3, t1, rtol=1e-9, atol=1e-9)


def test_rows_are_independent():
    z, gamma, beta, w1, w2 = _inputs(14, N=4)
    out = fusion.transition(z, gamma, beta, w1, w2)
    perm = np.random.default_rng(15).permutation(16)
    zp = z.reshape(1, 16, 1, -1)[:, perm].reshape(z.shape)
    outp = fusion.transition(zp, gamma, beta, w1, w2)
    np.testing.assert_allclose(outp.reshape(16, -1), out.reshape(16, -1)[perm], rtol=0,
                               atol=1e-13)


@pytest.mark.parametrize("eps", [1e-5, 1e-3])
def test_matches_torch_layer_norm_silu_and_matmul(eps):
    z, gamma, beta, w1, w2 = _inputs(16, B=2, N=5, C=16, F=64)
    t = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float64))
    F = w2.shape[1]
    y = torch.nn.functional.layer_norm(t(z), (z.shape[-1],), t(gamma), t(beta), eps)
    h = torch.nn.functional.silu(y @ t(w1[:F]).T) * (y @ t(w1[F:]).T)
    ref = (t(z) + h @ t(w2).T).numpy()
    np.testing.assert_allclose(fusion.transition(z, gamma, beta, w1, w2, eps), ref, rtol=1e-12,
                               atol=1e-12)


def test_output_projection_by_hand():
    """z = [1, 2], o = [1], w_o = [[0], [1]]: z1 = [1, 3], then the worked
    transition above (y = [-1, 1], h = 3 e / (1 + e))."""
    z = np.array([[[[1.0, 2.0]]]])
    o = np.array([[[[1.0]]]])
    w_o = np.array([[0.0], [1.0]])
    w1 = np.array([[0.0, 1.0], [0.0, 3.0]])
    w2 = np.array([[1.0], [-2.0]])
    h = 3 * math.e / (1 + math.e)
    out = fusion.transition(z, np.ones(2), np.zeros(2), w1, w2, eps=0.0, o=o, w_o=w_o)
    np.testing.assert_allclose(out.reshape(2), [1.0 + h, 3.0 - 2 * h], rtol=0, atol=1e-14)


def test_output_projection_special_cases():
    z, gamma, beta, w1, w2 = _inputs(21, C=8, F=16)
    o = _rand(z.shape[:-1] + (12,), 22)
    w_o = _rand((8, 12), 23, 12 ** -0.5)
    base = fusion.transition(z, gamma, beta, w1, w2)
    assert np.array_equal(fusion.transition(z, gamma, beta, w1, w2, o=o, w_o=np.zeros_like(w_o)),
                          base)
    F = w2.shape[1]
    w1b0 = w1.copy()
    w1b0[F:] = 0.0
    got = fusion.transition(z, gamma, beta, w1b0, w2, o=o, w_o=w_o)
    ref = (torch.from_numpy(z) + torch.from_numpy(o) @ torch.from_numpy(w_o).T).numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-13)


def test_with_output_projection_matches_torch():
    z, gamma, beta, w1, w2 = _inputs(24, B=1, N=4, C=16, F=64)
    o = _rand(z.shape[:-1] + (16,), 25, 0.5)
    w_o = _rand((16, 16), 26, 0.25)
    t = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float64))
    F = w2.shape[1]
    z1 = t(z) + t(o) @ t(w_o).T
    y = torch.nn.functional.layer_norm(z1, (16,), t(gamma), t(beta), 1e-5)
    ref = (z1 + (torch.nn.functional.silu(y @ t(w1[:F]).T) * (y @ t(w1[F:]).T)) @ t(w2).T)
    np.testing.assert_allclose(fusion.transition(z, gamma, beta, w1, w2, o=o, w_o=w_o),
                               ref.numpy(), rtol=1e-12, atol=1e-12)
