"""Parity of the fused downstream stack (evoattn_transition: the attention's
output projection with its residual add, then the SwiGLU transition; the
EvoFusion downstream stack) against the float64 oracle (oracle/fusion.py), on
the GPU, through the C ABI, with and without the output projection.

Tolerance, derived from the arithmetic: the kernel rounds the normalised row
to bf16 before the first projection, the activation h to bf16 before the
second, and the output to bf16 (each a relative error up to 2^-9, about
2^-9/sqrt(3) = 1.1e-3 relative L2), with fp32 sums in between.  The output
z + update is held to relative L2 <= 5e-3 and to four bf16 ulps of its
largest magnitude per element; the update alone (out - z, which the output
rounding dominates where |z| > |update|) to relative L2 <= 2e-2."""
import numpy as np
import pytest
import torch

from oracle import fusion
from protein_folding_attention_gb300 import evoattn, synthetic

from helpers import as_np, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda"
C, F = 128, 512


def _check(got, ref, z):
    g, r, z = as_np(got), np.asarray(ref), as_np(z)
    assert np.isfinite(g).all()
    e = rel_l2(g, r)
    a = float(np.abs(g - r).max())
    lim = 4 * 2.0 ** -8 * float(np.abs(r).max())
    assert e <= 5e-3 and a <= lim, f"out: rel-L2 {e:.3e} max-abs {a:.3e} (limit {lim:.3e})"
    eu = rel_l2(g - z, r - z)
    assert eu <= 2e-2, f"update: rel-L2 {eu:.3e}"
    return e, eu


def _run(B, N, seed, HD=0):
    x = synthetic.make_transition_inputs(B, N, C, F, seed=seed, HD=HD)
    xd = {k: (None if v is None else v.to(DEV)) for k, v in x.items()}
    out = evoattn.transition(xd["z"], xd["gamma"], xd["beta"], xd["w1"], xd["w2"], eps=1e-5,
                             o=xd["o"], w_o=xd["w_o"])
    assert evoattn.device_status() == evoattn.OK
    return x, out


def _oracle(x, rows=None):
    pick = (lambda t: t) if rows is None else rows
    o = None if x["o"] is None else pick(x["o"])
    return fusion.transition(pick(x["z"]), x["gamma"], x["beta"], x["w1"], x["w2"], eps=1e-5,
                             o=o, w_o=x["w_o"])


@pytest.mark.parametrize("HD", [0, 128])
@pytest.mark.parametrize("B,N", [(1, 40),    # 1600 rows: a ragged last tile
                                 (2, 24),    # two batches
                                 (1, 11),    # fewer rows than a tile
                                 (1, 128),   # 128 whole tiles
                                 (1, 200)])  # more tiles than SMs: several tiles per CTA
def test_transition_matches_oracle(B, N, HD):
    x, out = _run(B, N, seed=B * 1000 + N + HD, HD=HD)
    _check(out, _oracle(x), x["z"])


@pytest.mark.parametrize("HD", [0, 128])
def test_transition_repeats_bit_for_bit(HD):
    """Every output element is one row's fixed-order computation: two calls
    give identical bits."""
    _, a = _run(1, 64, seed=3, HD=HD)
    a = a.clone()
    _, b = _run(1, 64, seed=3, HD=HD)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_transition_zero_w2_returns_z():
    """With w2 = 0 the update is exactly zero: the output equals z to the bit
    (z + 0 rounds back to z)."""
    x = synthetic.make_transition_inputs(1, 48, C, F, seed=5, HD=128)
    xd = {k: v.to(DEV) for k, v in x.items()}
    out = evoattn.transition(xd["z"], xd["gamma"], xd["beta"], xd["w1"],
                             torch.zeros_like(xd["w2"]))
    assert evoattn.device_status() == evoattn.OK
    assert torch.equal(out.view(torch.int16), xd["z"].view(torch.int16))
    # and with a zero output projection as well
    out = evoattn.transition(xd["z"], xd["gamma"], xd["beta"], xd["w1"],
                             torch.zeros_like(xd["w2"]), o=xd["o"],
                             w_o=torch.zeros_like(xd["w_o"]))
    assert evoattn.device_status() == evoattn.OK
    assert torch.equal(out.view(torch.int16), xd["z"].view(torch.int16))


@pytest.mark.parametrize("HD", [0, 128])
@pytest.mark.parametrize("N", [384, 768])
def test_transition_full_size_sampled(N, HD):
    """The pair representation of the N = 384 and N = 768 workloads: rows are
    independent, so the oracle recomputes a random sample of 64 rows."""
    x, out = _run(1, N, seed=N, HD=HD)
    gen = torch.Generator().manual_seed(23)
    ii = torch.randint(0, N, (64,), generator=gen)
    jj = torch.randint(0, N, (64,), generator=gen)
    rows = lambda t: t[0, ii, jj].reshape(1, 8, 8, t.shape[-1])
    _check(rows(out.cpu()), _oracle(x, rows), rows(x["z"]))
