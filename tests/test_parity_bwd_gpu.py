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
