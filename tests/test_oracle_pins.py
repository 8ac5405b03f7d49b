"""Pins for the float64 oracle: facts the mathematics fixes, checked without
re-typing the oracle's own formula.

The pages (MegaFold, technical summary, "Methodik" section 1 "EvoFlash-3D")
print no worked numeric example, so the oracle is pinned by
* special cases with a closed form (zero logits -> column mean, one kept key
  -> that key's value row, a dominant bias -> that key's value row, a two-key
  softmax -> a logistic function, a constant bias -> shifted log-sum-exp);
* invariants (probabilities sum to one, shift invariance of softmax gives
  zero-sum gradients, key permutation invariance, s-permutation and
  row-duplication behaviour of the s-reduction of the bias gradient);
* the backward against central finite differences of the forward;
* an independent library: torch's float64 scaled_dot_product_attention with
  an additive float mask, and torch autograd for every gradient.
Each test is chosen so that a plausible slip (a dropped bias term, a bias with
j and k swapped, a mask on the wrong axis or the wrong s, a wrong scale, a
sigmoid left out of the gate, a missing sum over s) fails at least one.
"""
import math

import numpy as np
import pytest
import torch

from protein_folding_attention_gb300 import synthetic

pytestmark = pytest.mark.filterwarnings("ignore")


def _case(B=1, S=3, N=5, H=2, D=4, mask="none", gate=False, seed=7, **kw):
    w = synthetic.small(B=B, S=S, N=N, H=H, D=D, dtype="f32", node="dense",
                        mask=mask, gate=gate, seed=seed, **kw)
    x = synthetic.make_inputs(w)
    return {k: (None if v is None else (v.double() if v.is_floating_point() else v))
            for k, v in x.items()}


def test_zero_logits_give_column_mean_of_v(oracle_mod):
    x = _case(S=2, N=7, D=3, mask="tail", mask_tail=2)
    q = torch.zeros_like(x["q"])
    bias = torch.zeros_like(x["bias"])
    out, lse = oracle_mod.fwd(q, x["k"], x["v"], bias, x["mask"], None)
    kept = x["v"][:, :, :, :5, :].numpy()
    expect = kept.mean(axis=3, keepdims=True)
    np.testing.assert_allclose(out, np.broadcast_to(expect, out.shape), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, math.log(5.0), rtol=0, atol=1e-13)


def test_single_kept_key_selects_its_value_row(oracle_mod):
    x = _case(S=4, N=6, mask="none")
    mask = torch.zeros(1, 4, 6, dtype=torch.uint8)
    kstar = [3, 0, 5, 2]                     # a different kept key for every s
    for s, kk in enumerate(kstar):
        mask[0, s, kk] = 1
    out, _ = oracle_mod.fwd(x["q"], x["k"], x["v"], x["bias"], mask, None)
    for s, kk in enumerate(kstar):
        expect = x["v"][0, s, :, kk, :].numpy()[:, None, :]
        np.testing.assert_allclose(out[0, s], np.broadcast_to(expect, out[0, s].shape),
                                   rtol=0, atol=1e-12)


def test_dominant_bias_selects_key_per_query_row(oracle_mod):
    x = _case(S=2, N=6, H=3)
    bias = x["bias"].clone()
    # query row j gets a +1e4 bias on key (2j+1) mod N: pins bias[b,h,j,k] orientation
    kstar = [(2 * j + 1) % 6 for j in range(6)]
    for j, kk in enumerate(kstar):
        bias[:, :, j, kk] += 1e4
    out, _ = oracle_mod.fwd(x["q"], x["k"], x["v"], bias, None, None)
    for j, kk in enumerate(kstar):
        np.testing.assert_allclose(out[:, :, :, j, :], x["v"][:, :, :, kk, :].numpy(),
                                   rtol=0, atol=1e-12)


def test_probabilities_sum_to_one(oracle_mod):
    x = _case(S=3, N=9, mask="bernoulli", mask_p=0.3, gate=True)
    ones = torch.ones_like(x["v"])
    out, _ = oracle_mod.fwd(x["q"], x["k"], ones, x["bias"], x["mask"], None)
    np.testing.assert_allclose(out, 1.0, rtol=0, atol=1e-14)
    out_g, _ = oracle_mod.fwd(x["q"], x["k"], ones, x["bias"], x["mask"], x["gate"])
    np.testing.assert_allclose(out_g, torch.sigmoid(x["gate"]).numpy(), rtol=0, atol=1e-14)


def test_constant_bias_shifts_lse(oracle_mod):
    x = _case(S=2, N=8, mask="tail", mask_tail=3)
    q = torch.zeros_like(x["q"])
    c = torch.linspace(-2.0, 3.0, 2 * 8, dtype=torch.float64).reshape(1, 2, 8, 1)
    bias = c.expand(1, 2, 8, 8).contiguous()
    _, lse = oracle_mod.fwd(q, x["k"], x["v"], bias, x["mask"], None)
    expect = (c[..., 0] + math.log(5.0)).numpy()[:, None, :, :]   # [B,1,H,N]
    np.testing.assert_allclose(lse, np.broadcast_to(expect, lse.shape), rtol=0, atol=1e-13)


def test_two_key_softmax_is_logistic(oracle_mod):
    # D = 1, N = 2: x_k = q*k_k + bias_k, p_0 = 1 / (1 + exp(x_1 - x_0))
    q = torch.tensor([0.7, -1.3], dtype=torch.float64).reshape(1, 1, 1, 2, 1)
    k = torch.tensor([1.5, -0.25], dtype=torch.float64).reshape(1, 1, 1, 2, 1)
    v = torch.tensor([2.0, -3.0], dtype=torch.float64).reshape(1, 1, 1, 2, 1)
    bias = torch.tensor([[0.1, -0.4], [0.9, 0.3]], dtype=torch.float64).reshape(1, 1, 2, 2)
    out, lse = oracle_mod.fwd(q, k, v, bias, None, None)
    for j, (qj, b0, b1) in enumerate([(0.7, 0.1, -0.4), (-1.3, 0.9, 0.3)]):
        x0, x1 = qj * 1.5 + b0, qj * -0.25 + b1
        p0 = 1.0 / (1.0 + math.exp(x1 - x0))
        assert abs(out[0, 0, 0, j, 0] - (p0 * 2.0 + (1 - p0) * -3.0)) < 1e-14
        assert abs(lse[0, 0, 0, j] - (max(x0, x1) + math.log1p(math.exp(-abs(x0 - x1))))) < 1e-14


def test_zero_gate_halves_output(oracle_mod):
    x = _case(S=2, N=6, mask="tail", mask_tail=1)
    plain, _ = oracle_mod.fwd(x["q"], x["k"], x["v"], x["bias"], x["mask"], None)
    gated, _ = oracle_mod.fwd(x["q"], x["k"], x["v"], x["bias"], x["mask"],
                              torch.zeros_like(x["q"]))
    np.testing.assert_allclose(gated, 0.5 * plain, rtol=0, atol=1e-15)


def _torch_reference(x, mask_keep):
    """Independent statement via torch: per-s scaled_dot_product_attention
    (float64, math backend on CPU) with the pair bias plus the mask as its
    additive float mask; gradients by autograd."""
    q, k, v = (x[n].clone().requires_grad_(True) for n in ("q", "k", "v"))
    bias = x["bias"].clone().requires_grad_(True)
    gate = x["gate"].clone().requires_grad_(True) if x["gate"] is not None else None
    B, S, H, N, D = q.shape
    outs = []
    for s in range(S):
        add = bias
        if mask_keep is not None:
            mb = torch.where(mask_keep[:, s].bool(), 0.0, -1e9).to(torch.float64)
            add = bias + mb[:, None, None, :]
        o = torch.nn.functional.scaled_dot_product_attention(q[:, s], k[:, s], v[:, s],
                                                             attn_mask=add)
        outs.append(o)
    o = torch.stack(outs, dim=1)
    if gate is not None:
        o = torch.sigmoid(gate) * o
    (o * x["dout"]).sum().backward()
    grads = {"dq": q.grad, "dk": k.grad, "dv": v.grad, "dbias": bias.grad,
             "dgate": gate.grad if gate is not None else None}
    return o.detach(), grads


@pytest.mark.parametrize("mask,gate", [("none", False), ("tail", True), ("bernoulli", True)])
def test_matches_torch_sdpa_and_autograd(oracle_mod, mask, gate):
    x = _case(B=2, S=3, N=7, H=3, D=8, mask=mask, mask_tail=2, mask_p=0.3, gate=gate, seed=11)
    ref_out, ref = _torch_reference(x, x["mask"])
    out, _ = oracle_mod.fwd(x["q"], x["k"], x["v"], x["bias"], x["mask"], x["gate"])
    np.testing.assert_allclose(out, ref_out.numpy(), rtol=1e-12, atol=1e-12)
    g = oracle_mod.bwd(x["q"], x["k"], x["v"], x["bias"], x["mask"], x["gate"], x["dout"])
    for name in ("dq", "dk", "dv", "dbias") + (("dgate",) if gate else ()):
        np.testing.assert_allclose(g[name], ref[name].numpy(), rtol=1e-10, atol=1e-11,
                                   err_msg=name)


def test_backward_matches_central_differences(oracle_mod):
    x = _case(B=1, S=3, N=5, H=2, D=4, mask="bernoulli", mask_p=0.25, gate=True, seed=3)
    dout = x["dout"].numpy()
    g = oracle_mod.bwd(x["q"], x["k"], x["v"], x["bias"], x["mask"], x["gate"], x["dout"])
    base = {n: x[n].numpy().copy() for n in ("q", "k", "v", "bias", "gate")}

    def loss(arrs):
        out, _ = oracle_mod.fwd(arrs["q"], arrs["k"], arrs["v"], arrs["bias"], x["mask"],
                                arrs["gate"])
        return float((out * dout).sum())

    h = 1e-6
    for name, grad in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("bias", "dbias"),
                       ("gate", "dgate")):
        fd = np.zeros_like(base[name])
        it = np.nditer(base[name], flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            arrs = {n: a.copy() for n, a in base.items()}
            arrs[name][idx] += h
            lp = loss(arrs)
            arrs[name][idx] -= 2 * h
            lm = loss(arrs)
            fd[idx] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(g[grad], fd, rtol=1e-6, atol=1e-8, err_msg=grad)


def test_gradient_invariants(oracle_mod):
    x = _case(B=1, S=4, N=8, H=2, D=4, mask="tail", mask_tail=3, gate=True, seed=5)
    g = oracle_mod.bwd(x["q"], x["k"], x["v"], x["bias"], x["mask"], x["gate"], x["dout"])
    # softmax is shift invariant along k: every row of ds sums to zero
    np.testing.assert_allclose(g["dbias"].sum(axis=-1), 0.0, atol=1e-12)
    np.testing.assert_allclose(g["dk"].sum(axis=3), 0.0, atol=1e-12)
    # keys masked for every s get no probability mass: zero dbias and dv there
    np.testing.assert_array_equal(g["dbias"][..., 5:], 0.0)
    np.testing.assert_array_equal(g["dv"][:, :, :, 5:, :], 0.0)


def test_key_permutation_invariance(oracle_mod):
    x = _case(S=2, N=9, mask="bernoulli", mask_p=0.3, gate=True, seed=8)
    perm = torch.randperm(9, generator=torch.Generator().manual_seed(1))
    out, _ = oracle_mod.fwd(x["q"], x["k"], x["v"], x["bias"], x["mask"], x["gate"])
    out_p, _ = oracle_mod.fwd(x["q"], x["k"][:, :, :, perm], x["v"][:, :, :, perm],
                              x["bias"][..., perm], x["mask"][..., perm], x["gate"])
    np.testing.assert_allclose(out_p, out, rtol=0, atol=1e-13)


def test_s_reduction_of_bias_gradient(oracle_mod):
    x = _case(S=4, N=6, mask="bernoulli", mask_p=0.2, gate=True, seed=9)
    g = oracle_mod.bwd(x["q"], x["k"], x["v"], x["bias"], x["mask"], x["gate"], x["dout"])
    # permuting s permutes the per-s outputs and leaves dbias unchanged
    perm = torch.tensor([2, 0, 3, 1])
    xp = {n: (t[:, perm] if (t is not None and n != "bias") else t) for n, t in x.items()}
    gp = oracle_mod.bwd(xp["q"], xp["k"], xp["v"], xp["bias"], xp["mask"], xp["gate"],
                        xp["dout"])
    np.testing.assert_allclose(gp["dbias"], g["dbias"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(gp["dq"], g["dq"][:, perm.numpy()], rtol=0, atol=1e-15)
    # a duplicated s row contributes twice: S=2 of identical rows == 2 x S=1
    one = {n: (t[:, :1] if (t is not None and n != "bias") else t) for n, t in x.items()}
    two = {n: (torch.cat([t, t], dim=1) if (t is not None and n != "bias") else t)
           for n, t in one.items()}
    g1 = oracle_mod.bwd(one["q"], one["k"], one["v"], one["bias"], one["mask"], one["gate"],
                        one["dout"])
    g2 = oracle_mod.bwd(two["q"], two["k"], two["v"], two["bias"], two["mask"], two["gate"],
                        two["dout"])
    np.testing.assert_allclose(g2["dbias"], 2.0 * g1["dbias"], rtol=0, atol=1e-14)


def test_slip_detection_sanity(oracle_mod):
    """The SDPA comparison is sensitive to a bias with j and k swapped: a
    non-symmetric bias makes the swapped reading differ measurably."""
    x = _case(S=1, N=6, H=2, D=4, seed=12)
    out, _ = oracle_mod.fwd(x["q"], x["k"], x["v"], x["bias"], None, None)
    swapped, _ = oracle_mod.fwd(x["q"], x["k"], x["v"], x["bias"].transpose(2, 3), None, None)
    assert np.abs(out - swapped).max() > 1e-2
