"""Backward parity of the CUDA path against the float64 oracle (GPU)."""
import numpy as np
import pytest
import torch

import oracle
from protein_folding_attention_gb300 import evoattn, synthetic

from helpers import F32_REL, GRAD_REL, as_np, rel_l2, to_device

pytestmark = pytest.mark.gpu
DEV = "cuda"
GRADS = ("dq", "dk", "dv", "dbias", "dgate")


def run_fwd_bwd(x, flags=evoattn.DBIAS_DETERMINISTIC):
    xd = {k: to_device(v, DEV) for k, v in x.items()}
    out, lse = evoattn.fwd(xd["q"], xd["k"], xd["v"], xd["bias"], xd["mask"], xd["gate"])
    g = evoattn.bwd(xd["q"], xd["k"], xd["v"], xd["bias"], xd["mask"], xd["gate"], out, lse,
                    xd["dout"], flags=flags)
    assert evoattn.device_status() == evoattn.OK
    return g


def check_bwd(x, g, tol):
    ref = oracle.bwd(x["q"], x["k"], x["v"], x["bias"], x["mask"], x["gate"], x["dout"])
    errs = {}
    for n in GRADS:
        if ref[n] is None:
            assert g[n] is None
            continue
        assert np.isfinite(as_np(g[n])).all(), n
        errs[n] = rel_l2(g[n], ref[n])
    bad = {n: e for n, e in errs.items() if e > tol}
    assert not bad, f"rel-L2 over {tol}: {errs}"
    return errs


def test_fp32_tiny_start_n32():
    w = synthetic.WORKLOADS["tiny_start_n32_fp32"]
    x = synthetic.make_inputs(w)
    check_bwd(x, run_fwd_bwd(x), F32_REL)


def test_fp32_gated_ending_node():
    w = synthetic.small("f32e", B=1, S=6, N=40, H=2, D=32, dtype="f32", node="ending",
                        mask="bernoulli", mask_p=0.25, gate=True, seed=31)
    x = synthetic.make_inputs(w)
    check_bwd(x, run_fwd_bwd(x), F32_REL)


CASES = [
    # (S, N, H, D, node, mask, gate)
    (1, 128, 1, 32, "dense", "none", False),
    (3, 128, 2, 32, "starting", "tail", True),
    (5, 200, 2, 32, "starting", "tail", True),      # ragged key/query tail
    (4, 256, 2, 32, "ending", "tail", True),        # transposed views + j-contiguous bias
    (7, 96, 3, 32, "msa", "bernoulli", True),       # N < one tile, odd S
    (2, 384, 1, 32, "starting", "bernoulli", False),
    (6, 136, 2, 16, "starting", "tail", True),      # D = 16
    (9, 64, 2, 16, "ending", "bernoulli", True),
    (1, 8, 1, 32, "dense", "tail", True),           # tiny N
]


@pytest.mark.parametrize("S,N,H,D,node,mask,gate", CASES)
@pytest.mark.parametrize("flags", [evoattn.DBIAS_DETERMINISTIC, evoattn.DBIAS_ATOMIC,
                                   evoattn.DBIAS_FUSED])
def test_bf16_bwd_small(S, N, H, D, node, mask, gate, flags):
    w = synthetic.small("c", B=1, S=S, N=N, H=H, D=D, dtype="bf16", node=node, mask=mask,
                        mask_tail=max(1, N // 10), mask_p=0.2, gate=gate, seed=S * 1000 + N + 7)
    x = synthetic.make_inputs(w)
    check_bwd(x, run_fwd_bwd(x, flags), GRAD_REL)


@pytest.mark.parametrize("bias_std", [8.0, 12.0])
def test_bf16_bwd_large_pair_bias(bias_std):
    """Gradients with a pair bias of standard deviation 8-12 (the bias term
    dominates the logits), both bias layouts.  The softmax is then nearly one
    key per row and dS = P (dP - delta) cancels: the bf16 rounding of out
    (which delta is computed from) and of the gated output gradient (an MMA
    operand) bring the gradients' relative L2 error to about 8e-3 at standard
    deviation 12 and 1e-2 at 16 (a float64 emulation of those roundings gives
    the same figures), so the sweep stops at 12."""
    for node in ("starting", "ending"):
        w = synthetic.small("lb", B=1, S=5, N=200, H=2, D=32, dtype="bf16", node=node,
                            mask="tail", mask_tail=13, gate=True, bias_std=bias_std,
                            seed=int(bias_std) * 10 + (node == "ending"))
        x = synthetic.make_inputs(w)
        check_bwd(x, run_fwd_bwd(x), GRAD_REL)


def test_bf16_bwd_batch2():
    w = synthetic.small("b2", B=2, S=4, N=160, H=2, D=32, dtype="bf16", node="starting",
                        mask="bernoulli", mask_p=0.3, gate=True, seed=78)
    x = synthetic.make_inputs(w)
    check_bwd(x, run_fwd_bwd(x), GRAD_REL)


def test_deterministic_dbias_is_bit_identical():
    w = synthetic.small("det", B=1, S=40, N=256, H=2, D=32, dtype="bf16", node="starting",
                        mask="bernoulli", mask_p=0.2, gate=True, seed=4)
    x = synthetic.make_inputs(w)
    a = run_fwd_bwd(x)["dbias"].clone()
    b = run_fwd_bwd(x)["dbias"].clone()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    # the atomic variant meets the tolerance but need not be bit-identical
    c = run_fwd_bwd(x, evoattn.DBIAS_ATOMIC)["dbias"]
    assert rel_l2(c, a) < 1e-5


def test_gradients_are_bit_identical_run_to_run():
    """dk and dv accumulate in tensor memory, dgate is per element and the
    deterministic dbias sums fixed slots in order: they repeat bit for bit.
    dq (fp32 vector atomics across key tiles) is checked against the oracle
    only."""
    w = synthetic.small("rep", B=1, S=24, N=520, H=2, D=32, dtype="bf16", node="ending",
                        mask="tail", mask_tail=40, gate=True, seed=9)
    x = synthetic.make_inputs(w)
    a = {k: v.clone() for k, v in run_fwd_bwd(x).items()}
    b = run_fwd_bwd(x)
    for k in ("dk", "dv", "dgate", "dbias"):
        assert torch.equal(a[k].view(torch.int16 if a[k].element_size() == 2 else torch.int32),
                           b[k].view(torch.int16 if b[k].element_size() == 2 else torch.int32)), k


def _full_size_all_rows(name, flags):
    """Every gradient of a full-size workload, over every s row, against the
    oracle, in the benchmark's launch configuration.  This covers the
    production s-slot walk of the dbias reduction (several slots of many s
    rows each) element by element."""
    w = synthetic.WORKLOADS[name]
    xd = synthetic.make_inputs(w, device=DEV)
    out, lse = evoattn.fwd(xd["q"], xd["k"], xd["v"], xd["bias"], xd["mask"], xd["gate"])
    g = evoattn.bwd(xd["q"], xd["k"], xd["v"], xd["bias"], xd["mask"], xd["gate"], out, lse,
                    xd["dout"], flags=flags)
    assert evoattn.device_status() == evoattn.OK
    host = {k: (None if v is None else v.cpu()) for k, v in xd.items()}
    del xd
    ref = oracle.bwd(host["q"], host["k"], host["v"], host["bias"], host["mask"], host["gate"],
                     host["dout"])
    errs = {n: rel_l2(g[n], ref[n]) for n in GRADS if ref[n] is not None}
    bad = {n: e for n, e in errs.items() if e > GRAD_REL}
    assert not bad, f"{name}: rel-L2 over {GRAD_REL}: {errs}"


@pytest.mark.parametrize("name", ["pairformer_start_n384", "msa_row_s512_n384"])
def test_bf16_bwd_full_size_every_row(name):
    _full_size_all_rows(name, evoattn.DBIAS_DETERMINISTIC)


@pytest.mark.slow
def test_bf16_bwd_full_size_every_row_end_n768():
    """The benchmark workload itself (about a minute of oracle time)."""
    _full_size_all_rows("pairformer_end_n768", evoattn.DBIAS_DETERMINISTIC)


def test_bf16_bwd_full_size_every_row_atomic_dbias():
    _full_size_all_rows("pairformer_start_n384", evoattn.DBIAS_ATOMIC)


def test_bf16_bwd_full_size_every_row_fused_dbias():
    """dbias summed inside the dK/dV pass: the MSA-row workload (S = 512,
    three key tiles, Bernoulli key mask), every gradient over every s row."""
    _full_size_all_rows("msa_row_s512_n384", evoattn.DBIAS_FUSED)


def test_fused_dbias_leaves_the_other_gradients_unchanged():
    """The fused mode only adds the dbias atomics to the dK/dV pass: dk, dv
    and dgate are the default mode's bits, dq differs by the order of its
    fp32 additions at most, and dbias agrees with the deterministic sum to
    fp32 reordering."""
    w = synthetic.small("fz", B=1, S=10, N=296, H=2, D=32, dtype="bf16", node="ending",
                        mask="bernoulli", mask_p=0.2, gate=True, seed=123)
    x = synthetic.make_inputs(w)
    a = run_fwd_bwd(x)
    b = run_fwd_bwd(x, evoattn.DBIAS_FUSED)
    for k in ("dk", "dv", "dgate"):
        assert torch.equal(a[k].view(torch.int16), b[k].view(torch.int16)), k
    assert rel_l2(b["dq"], a["dq"]) < 2e-3
    assert rel_l2(b["dbias"], a["dbias"]) < 1e-4


@pytest.mark.parametrize("name", ["pairformer_start_n384", "pairformer_end_n768",
                                  "msa_row_s512_n384", "long_start_n1536"])
def test_bf16_bwd_full_size_sampled(name):
    """Full-size workload in the benchmark's launch configuration.  dq, dk, dv
    and dgate of a sample of s rows are recomputed by the oracle (each s slice
    is independent); dbias, a sum over every s, is checked through properties
    that hold at any size (rows sum to zero; keys masked for every s receive
    nothing) and, at full N, against the oracle on a gathered subset of rows."""
    w = synthetic.WORKLOADS[name]
    xd = synthetic.make_inputs(w, device=DEV)
    out, lse = evoattn.fwd(xd["q"], xd["k"], xd["v"], xd["bias"], xd["mask"], xd["gate"])
    g = evoattn.bwd(xd["q"], xd["k"], xd["v"], xd["bias"], xd["mask"], xd["gate"], out, lse,
                    xd["dout"])
    assert evoattn.device_status() == evoattn.OK
    gen = torch.Generator().manual_seed(7)
    picks = sorted(set(torch.randint(0, w.S, (2,), generator=gen).tolist()) | {0, w.S - 1})
    sl = lambda t, s: None if t is None else t[:, s:s + 1].cpu()
    for s in picks:
        ref = oracle.bwd(sl(xd["q"], s), sl(xd["k"], s), sl(xd["v"], s), xd["bias"].cpu(),
                         sl(xd["mask"], s), sl(xd["gate"], s), sl(xd["dout"], s))
        for n in ("dq", "dk", "dv", "dgate"):
            e = rel_l2(g[n][:, s:s + 1], ref[n])
            assert e <= GRAD_REL, f"{n} s={s}: rel-L2 {e:.3e}"
    db = g["dbias"].double()
    assert torch.isfinite(db).all()
    rowsum = db.sum(-1).abs().max().item()
    assert rowsum <= 1e-3 * db.abs().max().item() * w.N ** 0.5
    if w.mask == "tail" and w.mask_tail > 0:
        assert torch.count_nonzero(g["dbias"][..., w.N - w.mask_tail:]) == 0
    # dbias at full N on 12 gathered rows, against the oracle
    rows = torch.tensor(picks + [1, 2, 3, 5, 8, 13, 21, 34][: 12 - len(picks)])
    sub = {k: (None if v is None else
               (v if k == "bias" else v.index_select(1, rows.to(v.device))))
           for k, v in xd.items()}
    sub = {k: (None if v is None else v.contiguous()) for k, v in sub.items()}
    sub["bias"] = xd["bias"]
    o2, l2 = evoattn.fwd(sub["q"], sub["k"], sub["v"], sub["bias"], sub["mask"], sub["gate"])
    g2 = evoattn.bwd(sub["q"], sub["k"], sub["v"], sub["bias"], sub["mask"], sub["gate"], o2,
                     l2, sub["dout"])
    ref = oracle.bwd(*(None if sub[n] is None else sub[n].cpu()
                       for n in ("q", "k", "v", "bias", "mask", "gate", "dout")))
    e = rel_l2(g2["dbias"], ref["dbias"])
    assert e <= GRAD_REL, f"dbias (gathered rows) rel-L2 {e:.3e}"
