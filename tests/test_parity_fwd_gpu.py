"""Forward parity of the CUDA path against the float64 oracle (GPU)."""
import numpy as np
import pytest
import torch

import oracle
from protein_folding_attention_gb300 import evoattn, synthetic

from helpers import FWD_ABS, FWD_REL, F32_REL, as_np, max_abs, rel_l2, to_device

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_fwd(x):
    xd = {k: to_device(v, DEV) for k, v in x.items()}
    out, lse = evoattn.fwd(xd["q"], xd["k"], xd["v"], xd["bias"], xd["mask"], xd["gate"])
    assert evoattn.device_status() == evoattn.OK
    return out, lse


def check_fwd(x, out, lse, rel=FWD_REL, abs_=FWD_ABS):
    ref_out, ref_lse = oracle.fwd(x["q"], x["k"], x["v"], x["bias"], x["mask"], x["gate"])
    r, a = rel_l2(out, ref_out), max_abs(out, ref_out)
    assert np.isfinite(as_np(out)).all()
    assert r <= rel and a <= abs_, f"out rel-L2 {r:.3e} max-abs {a:.3e}"
    rl, al = rel_l2(lse, ref_lse), max_abs(lse, ref_lse)
    assert rl <= rel and al <= abs_, f"lse rel-L2 {rl:.3e} max-abs {al:.3e}"
    return r, a


def test_fp32_tiny_start_n32():
    w = synthetic.WORKLOADS["tiny_start_n32_fp32"]
    x = synthetic.make_inputs(w)
    out, lse = run_fwd(x)
    check_fwd(x, out, lse, rel=F32_REL, abs_=F32_REL)


CASES = [
    # (S, N, H, D, node, mask, gate)
    (1, 128, 1, 32, "dense", "none", False),
    (3, 128, 2, 32, "starting", "tail", True),
    (5, 200, 2, 32, "starting", "tail", True),      # ragged key/query tail
    (4, 256, 2, 32, "ending", "tail", True),        # transposed views + j-contiguous bias
    (7, 96, 3, 32, "msa", "bernoulli", True),       # N < one tile, odd S
    (2, 384, 1, 32, "starting", "bernoulli", False),
    (6, 136, 2, 16, "starting", "tail", True),      # D = 16
    (3, 192, 2, 64, "ending", "bernoulli", True),   # D = 64
    (1, 8, 1, 32, "dense", "tail", True),           # tiny N
]


# More work items (query tile x head x row group) than SMs, and S not a
# multiple of the row group, so partial groups (fewer rows, one warpgroup
# idle) sit between full ones in the same launch.
MULTI_ITEM = [
    # (S, N, H, D, node, mask, gate)
    (7, 704, 16, 32, "ending", "bernoulli", True),     # 192 items, groups of 4 and 3
    (5, 520, 16, 16, "starting", "tail", False),      # 160 items, groups of 4 and 1
    (3, 640, 16, 64, "msa", "bernoulli", True),        # 160 items, groups of 2 and 1
]


@pytest.mark.parametrize("S,N,H,D,node,mask,gate", MULTI_ITEM)
def test_bf16_fwd_many_items(S, N, H, D, node, mask, gate):
    w = synthetic.small("mi", B=1, S=S, N=N, H=H, D=D, dtype="bf16", node=node, mask=mask,
                        mask_tail=max(1, N // 10), mask_p=0.2, gate=gate, seed=S * 100 + N + D)
    x = synthetic.make_inputs(w)
    out, lse = run_fwd(x)
    check_fwd(x, out, lse)
    # the same call again gives the same bits (no state carried between
    # launches)
    out2, lse2 = run_fwd(x)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lse2.view(torch.int32))


@pytest.mark.parametrize("S,N,H,D,node,mask,gate", CASES)
def test_bf16_fwd_small(S, N, H, D, node, mask, gate):
    w = synthetic.small("c", B=1, S=S, N=N, H=H, D=D, dtype="bf16", node=node, mask=mask,
                        mask_tail=max(1, N // 10), mask_p=0.2, gate=gate, seed=S * 1000 + N)
    x = synthetic.make_inputs(w)
    out, lse = run_fwd(x)
    check_fwd(x, out, lse)


@pytest.mark.parametrize("bias_std", [8.0, 16.0])
def test_bf16_fwd_large_pair_bias(bias_std):
    """A pair bias of standard deviation 8-16 makes the bias dominate the
    logits, so any error in the coefficient with which it enters the logit
    tile grows in proportion; both layouts of the bias tile are covered."""
    for node in ("starting", "ending"):
        w = synthetic.small("lb", B=1, S=3, N=200, H=2, D=32, dtype="bf16", node=node,
                            mask="tail", mask_tail=13, gate=True, bias_std=bias_std,
                            seed=int(bias_std) * 10 + (node == "ending"))
        x = synthetic.make_inputs(w)
        out, lse = run_fwd(x)
        check_fwd(x, out, lse)


def test_bf16_fwd_batch2():
    w = synthetic.small("b2", B=2, S=3, N=160, H=2, D=32, dtype="bf16", node="starting",
                        mask="bernoulli", mask_p=0.3, gate=True, seed=77)
    x = synthetic.make_inputs(w)
    out, lse = run_fwd(x)
    check_fwd(x, out, lse)


def test_bf16_fwd_fully_masked_row_is_finite():
    w = synthetic.small("fm", B=1, S=2, N=64, H=1, D=32, dtype="bf16", node="dense",
                        mask="none", gate=False, seed=5)
    x = synthetic.make_inputs(w)
    x["mask"] = torch.ones(1, 2, 64, dtype=torch.uint8)
    x["mask"][0, 1] = 0        # row s=1 masks every key: uniform softmax
    out, lse = run_fwd(x)
    o = as_np(out)
    assert np.isfinite(o).all()
    v = as_np(x["v"])
    np.testing.assert_allclose(o[0, 1], np.broadcast_to(v[0, 1].mean(axis=1, keepdims=True),
                                                        o[0, 1].shape), atol=2e-2)


@pytest.mark.parametrize("name", ["pairformer_start_n384", "pairformer_end_n768",
                                  "msa_row_s512_n384", "long_start_n1536"])
def test_bf16_fwd_full_size_sampled(name):
    """Full-size workload in the benchmark's launch configuration; the oracle
    recomputes a sample of s rows (each s slice is independent)."""
    w = synthetic.WORKLOADS[name]
    xd = synthetic.make_inputs(w, device=DEV)
    out, lse = evoattn.fwd(xd["q"], xd["k"], xd["v"], xd["bias"], xd["mask"], xd["gate"])
    assert evoattn.device_status() == evoattn.OK
    gen = torch.Generator().manual_seed(99)
    picks = sorted(set(torch.randint(0, w.S, (3,), generator=gen).tolist()) | {0, w.S - 1})
    for s in picks:
        sl = lambda t: None if t is None else t[:, s:s + 1].cpu()
        ref_out, ref_lse = oracle.fwd(sl(xd["q"]), sl(xd["k"]), sl(xd["v"]), xd["bias"].cpu(),
                                      sl(xd["mask"]), sl(xd["gate"]))
        r, a = rel_l2(out[:, s:s + 1], ref_out), max_abs(out[:, s:s + 1], ref_out)
        assert r <= FWD_REL and a <= FWD_ABS, f"s={s}: rel {r:.3e} abs {a:.3e}"
        rl, al = rel_l2(lse[:, s:s + 1], ref_lse), max_abs(lse[:, s:s + 1], ref_lse)
        assert rl <= FWD_REL and al <= FWD_ABS, f"s={s}: lse rel {rl:.3e} abs {al:.3e}"
