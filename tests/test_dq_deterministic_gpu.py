"""The deterministic-dQ backward mode (EVOATTN_DQ_DETERMINISTIC) on the GPU.

By default the BF16 backward adds the dQ partial of every 128-key tile into
one fp32 buffer with vector atomics, so the rounding of dq depends on the
order in which the key tiles finish.  With the flag each key tile stores its
partial into a slice of its own and the slices are summed in key-tile order:
dq must then repeat bit for bit whatever the workspace held before, meet the
same tolerance against the float64 oracle, and agree closely with the
default mode (the two differ only in the order of fp32 additions)."""
import pytest
import torch

from protein_folding_attention_gb300 import evoattn, synthetic

from helpers import GRAD_REL, rel_l2, to_device
from test_parity_bwd_gpu import GRADS, check_bwd

pytestmark = pytest.mark.gpu
DEV = "cuda"
DET = evoattn.DQ_DETERMINISTIC


def _bwd(xd, out, lse, flags, fill=None):
    ws = torch.empty(max(evoattn.workspace_size(*xd["q"].shape, flags=flags), 1),
                     device=DEV, dtype=torch.uint8)
    if fill is not None:
        ws.fill_(fill)  # e.g. 0xFF: every fp32 word a NaN
    g = evoattn.bwd(xd["q"], xd["k"], xd["v"], xd["bias"], xd["mask"], xd["gate"], out, lse,
                    xd["dout"], flags=flags, workspace=ws)
    assert evoattn.device_status() == evoattn.OK
    return {k: (None if v is None else v.clone()) for k, v in g.items()}


def _fwd(x):
    xd = {k: to_device(v, DEV) for k, v in x.items()}
    out, lse = evoattn.fwd(xd["q"], xd["k"], xd["v"], xd["bias"], xd["mask"], xd["gate"])
    return xd, out, lse


CASES = [
    # (S, N, H, D, node, mask, gate)
    (3, 128, 2, 32, "starting", "tail", True),      # one key tile: one slice
    (5, 200, 2, 32, "starting", "tail", True),      # ragged tail, two slices
    (4, 296, 2, 32, "ending", "bernoulli", True),   # three slices, transposed views
    (6, 136, 2, 16, "starting", "tail", True),      # D = 16
    (7, 96, 3, 32, "msa", "bernoulli", False),
]


@pytest.mark.parametrize("S,N,H,D,node,mask,gate", CASES)
@pytest.mark.parametrize("dbias", [evoattn.DBIAS_DETERMINISTIC, evoattn.DBIAS_ATOMIC])
def test_det_dq_matches_oracle(S, N, H, D, node, mask, gate, dbias):
    w = synthetic.small("dqd", B=1, S=S, N=N, H=H, D=D, dtype="bf16", node=node, mask=mask,
                        mask_tail=max(1, N // 10), mask_p=0.2, gate=gate, seed=S * 77 + N)
    x = synthetic.make_inputs(w)
    xd, out, lse = _fwd(x)
    check_bwd(x, _bwd(xd, out, lse, dbias | DET), GRAD_REL)


def test_det_dq_is_bit_identical_whatever_the_workspace_held():
    """Two runs, the second over a workspace filled with NaN bit patterns:
    every gradient (dq included) is identical to the bit."""
    w = synthetic.small("dqrep", B=1, S=24, N=520, H=2, D=32, dtype="bf16", node="ending",
                        mask="tail", mask_tail=40, gate=True, seed=9)
    x = synthetic.make_inputs(w)
    xd, out, lse = _fwd(x)
    a = _bwd(xd, out, lse, DET)
    b = _bwd(xd, out, lse, DET, fill=0xFF)
    for n in GRADS:
        t, u = a[n], b[n]
        iv = torch.int16 if t.element_size() == 2 else torch.int32
        assert torch.equal(t.view(iv), u.view(iv)), n
    # the default (atomic dQ) mode gives the same dk, dv, dgate, dbias bits and
    # a dq that differs only through the order of the fp32 additions
    c = _bwd(xd, out, lse, evoattn.DBIAS_DETERMINISTIC)
    for n in ("dk", "dv", "dgate", "dbias"):
        iv = torch.int16 if a[n].element_size() == 2 else torch.int32
        assert torch.equal(a[n].view(iv), c[n].view(iv)), n
    assert rel_l2(c["dq"], a["dq"]) < 2e-3


def test_det_dq_full_size_every_row():
    """The N = 384 pair-stack workload (S = 384, three key tiles) in the
    benchmark's launch configuration: every gradient against the oracle, and
    dq repeated bit for bit."""
    import oracle
    w = synthetic.WORKLOADS["pairformer_start_n384"]
    xd = synthetic.make_inputs(w, device=DEV)
    out, lse = evoattn.fwd(xd["q"], xd["k"], xd["v"], xd["bias"], xd["mask"], xd["gate"])
    g = _bwd(xd, out, lse, DET)
    again = _bwd(xd, out, lse, DET, fill=0x7F)
    assert torch.equal(g["dq"].view(torch.int16), again["dq"].view(torch.int16))
    del again
    host = {k: (None if v is None else v.cpu()) for k, v in xd.items()}
    del xd, out, lse
    ref = oracle.bwd(host["q"], host["k"], host["v"], host["bias"], host["mask"], host["gate"],
                     host["dout"])
    errs = {n: rel_l2(g[n], ref[n]) for n in GRADS if ref[n] is not None}
    assert all(e <= GRAD_REL for e in errs.values()), errs
