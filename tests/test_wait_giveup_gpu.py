"""The bounded-wait failure path of the tcgen05 kernels, on the GPU, without a
fault or a hang: the testing hook evoattn_debug_set_wait makes the compute
warps' first wait in every kernel wait for an event that nothing signals,
with a limit of 50 microseconds.  Each CTA must then give up, let the copies
and MMAs it already issued finish, free its tensor memory and exit; the
device status must read EVOATTN_ERR_TIMEOUT; and the next normal call in the
same process must run and match the oracle (the context stays usable and the
earlier give-up does not leak into later launches)."""
import pytest
import torch

import oracle
from protein_folding_attention_gb300 import evoattn, synthetic

from helpers import FWD_REL, GRAD_REL, rel_l2, to_device

pytestmark = pytest.mark.gpu

LIMIT_NS = 50_000


def _inputs(node):
    w = synthetic.small("to", B=1, S=6, N=200, H=2, D=32, dtype="bf16", node=node,
                        mask="tail", mask_tail=11, gate=True, seed=314)
    x = synthetic.make_inputs(w)
    return x, {k: to_device(v, "cuda") for k, v in x.items()}


def _stalled(fn):
    assert evoattn.device_status() == evoattn.OK
    evoattn.debug_set_wait(LIMIT_NS, stall=True)
    try:
        fn()
        status = evoattn.device_status()
    finally:
        evoattn.debug_set_wait(0, stall=False)
    return status


@pytest.mark.parametrize("node", ["starting", "ending"])
def test_forward_gives_up_and_recovers(node):
    x, xd = _inputs(node)
    args = (xd["q"], xd["k"], xd["v"], xd["bias"], xd["mask"], xd["gate"])
    assert _stalled(lambda: evoattn.fwd(*args)) == evoattn.ERR_TIMEOUT
    out, lse = evoattn.fwd(*args)
    assert evoattn.device_status() == evoattn.OK
    ref_out, ref_lse = oracle.fwd(x["q"], x["k"], x["v"], x["bias"], x["mask"], x["gate"])
    assert rel_l2(out, ref_out) <= FWD_REL
    assert rel_l2(lse, ref_lse) <= FWD_REL


@pytest.mark.parametrize("flags", [evoattn.DBIAS_DETERMINISTIC, evoattn.DBIAS_ATOMIC,
                                   evoattn.DBIAS_FUSED])
def test_backward_gives_up_and_recovers(flags):
    x, xd = _inputs("ending")
    args = (xd["q"], xd["k"], xd["v"], xd["bias"], xd["mask"], xd["gate"])
    out, lse = evoattn.fwd(*args)
    assert evoattn.device_status() == evoattn.OK
    status = _stalled(lambda: evoattn.bwd(*args, out, lse, xd["dout"], flags=flags))
    assert status == evoattn.ERR_TIMEOUT
    g = evoattn.bwd(*args, out, lse, xd["dout"], flags=flags)
    assert evoattn.device_status() == evoattn.OK
    ref = oracle.bwd(x["q"], x["k"], x["v"], x["bias"], x["mask"], x["gate"], x["dout"])
    for n in ("dq", "dk", "dv", "dbias", "dgate"):
        assert torch.isfinite(g[n]).all(), n
        assert rel_l2(g[n], ref[n]) <= GRAD_REL, n


def test_default_limit_is_restored():
    """After the stalled launches, a default-limit call on a full tile set
    completes normally (no launch aborts on an earlier launch's give-up)."""
    x, xd = _inputs("starting")
    args = (xd["q"], xd["k"], xd["v"], xd["bias"], xd["mask"], xd["gate"])
    assert _stalled(lambda: evoattn.fwd(*args)) == evoattn.ERR_TIMEOUT
    for _ in range(3):
        evoattn.fwd(*args)
    assert evoattn.device_status() == evoattn.OK


def test_ln_proj_gives_up_and_recovers():
    """The fused LayerNorm + projection kernel: its LayerNorm warps' first
    wait stalls, every CTA gives up, the status reads ERR_TIMEOUT, and the
    next call matches the oracle."""
    from oracle import fusion
    from helpers import rel_l2
    x = synthetic.make_fusion_inputs(1, 40, 128, 4, 32, seed=8)
    xd = {k: v.to("cuda") for k, v in x.items()}
    run = lambda: evoattn.ln_proj(xd["z"], xd["gamma"], xd["beta"], xd["w"], 4, 32)
    assert _stalled(run) == evoattn.ERR_TIMEOUT
    out = run()
    assert evoattn.device_status() == evoattn.OK
    ref = fusion.ln_proj(x["z"], x["gamma"], x["beta"], x["w"], 4, 32)
    for got, r in zip(out, ref):
        assert rel_l2(got, r) <= 5e-3


def test_transition_gives_up_and_recovers():
    """The fused transition kernel: its LayerNorm warps' first wait stalls,
    every CTA gives up, the status reads ERR_TIMEOUT, and the next call
    matches the oracle."""
    from oracle import fusion
    for HD in (0, 128):
        x = synthetic.make_transition_inputs(1, 40, 128, 512, seed=8, HD=HD)
        xd = {k: (None if v is None else v.to("cuda")) for k, v in x.items()}
        run = lambda: evoattn.transition(xd["z"], xd["gamma"], xd["beta"], xd["w1"], xd["w2"],
                                         o=xd["o"], w_o=xd["w_o"])
        assert _stalled(run) == evoattn.ERR_TIMEOUT
        out = run()
        assert evoattn.device_status() == evoattn.OK
        ref = fusion.transition(x["z"], x["gamma"], x["beta"], x["w1"], x["w2"], o=x["o"],
                                w_o=x["w_o"])
        assert rel_l2(out, ref) <= 5e-3
