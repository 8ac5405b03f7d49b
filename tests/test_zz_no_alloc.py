"""evoattn_bwd_noalloc: the backward for callers that cannot allocate device
memory (a plugin inside a framework that owns every device allocation, or a
hot path that must not call cudaMalloc).  Its scratch is a fixed array inside
the library instead of a caller workspace.

Called through the C ABI and checked against evoattn_bwd (caller workspace)
on the same inputs, twice in a row, since consecutive calls share the array.
This file is collected last so that a run stopping at the first failure has
already run every other test."""
import ctypes

import pytest
import torch

from protein_folding_attention_gb300 import evoattn, synthetic

from helpers import GRAD_REL, rel_l2, to_device

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 << 20  # EVOATTN_NOALLOC_SCRATCH_BYTES in include/evoattn.h


def _noalloc_fn():
    lib = evoattn.load()
    fn = lib.evoattn_bwd_noalloc
    fn.argtypes = lib.evoattn_bwd.argtypes[:-3] + [ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


def _call_noalloc(fn, x, out, lse, grads, dbias, flags=evoattn.DBIAS_DETERMINISTIC):
    s5 = lambda t: None if t is None else (ctypes.c_int64 * 5)(*t.stride())
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    B, S, H, N, D = x["q"].shape
    return fn(p(x["q"]), s5(x["q"]), p(x["k"]), s5(x["k"]), p(x["v"]), s5(x["v"]),
              p(x["bias"]), (ctypes.c_int64 * 4)(*x["bias"].stride()),
              p(x["mask"]), (ctypes.c_int64 * 3)(*x["mask"].stride()),
              p(x["gate"]), s5(x["gate"]), p(out), s5(out), p(lse),
              p(x["dout"]), s5(x["dout"]), p(grads["dq"]), s5(grads["dq"]),
              p(grads["dk"]), s5(grads["dk"]), p(grads["dv"]), s5(grads["dv"]), p(dbias),
              p(grads["dgate"]), s5(grads["dgate"]), B, S, H, N, D, evoattn.BF16,
              flags, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _problem(node, S, N, seed):
    w = synthetic.small("na", B=1, S=S, N=N, H=2, D=32, dtype="bf16", node=node,
                        mask="bernoulli", mask_p=0.2, gate=True, seed=seed)
    assert evoattn.workspace_size(w.B, w.S, w.H, w.N, w.D) <= SCRATCH_BYTES
    x = {k: to_device(v, "cuda") for k, v in synthetic.make_inputs(w).items()}
    out, lse = evoattn.fwd(x["q"], x["k"], x["v"], x["bias"], x["mask"], x["gate"])
    return x, out, lse


def _noalloc_grads(fn, x, out, lse, flags):
    grads = {n: torch.full_like(x["q"], float("nan")) for n in ("dq", "dk", "dv", "dgate")}
    B, S, H, N, D = x["q"].shape
    dbias = torch.full((B, H, N, N), float("nan"), device="cuda")
    assert _call_noalloc(fn, x, out, lse, grads, dbias, flags) == evoattn.OK
    assert evoattn.device_status() == evoattn.OK
    grads["dbias"] = dbias
    return grads


def _bits(t):
    return t.view(torch.int16 if t.element_size() == 2 else torch.int32)


@pytest.mark.parametrize("node", ["starting", "ending"])
def test_noalloc_matches_workspace_backward_twice(node):
    """Two calls in a row, each after the shared scratch was left dirty by a
    different problem (other seed, other N and S, so another dbias slot
    count and layout).  dk, dv, dgate and the deterministic dbias come from
    the same kernels in the same order as with a caller workspace, so they
    must agree bit for bit; a kernel that read a scratch byte it had not
    written would break that.  dq is summed with fp32 atomics (order not
    fixed) and is compared by relative L2 error."""
    fn = _noalloc_fn()
    x, out, lse = _problem(node, S=16, N=200, seed=21)
    ref = evoattn.bwd(x["q"], x["k"], x["v"], x["bias"], x["mask"], x["gate"], out, lse,
                      x["dout"])
    other, o_out, o_lse = _problem(node, S=24, N=256, seed=5)
    for _ in range(2):
        _noalloc_grads(fn, other, o_out, o_lse, evoattn.DBIAS_DETERMINISTIC)  # dirty scratch
        g = _noalloc_grads(fn, x, out, lse, evoattn.DBIAS_DETERMINISTIC)
        for n in ("dk", "dv", "dgate", "dbias"):
            assert torch.equal(_bits(g[n]), _bits(ref[n])), n
        assert torch.isfinite(g["dq"]).all()
        assert rel_l2(g["dq"], ref["dq"]) <= GRAD_REL


def test_noalloc_atomic_dbias_twice():
    """The atomic dbias variant through the no-alloc entry point, twice, after
    dirtying the scratch: dk, dv, dgate bit for bit, dbias and dq within the
    rounding of a different summation order."""
    fn = _noalloc_fn()
    x, out, lse = _problem("starting", S=16, N=200, seed=22)
    ref = evoattn.bwd(x["q"], x["k"], x["v"], x["bias"], x["mask"], x["gate"], out, lse,
                      x["dout"])
    other, o_out, o_lse = _problem("ending", S=24, N=256, seed=6)
    for _ in range(2):
        _noalloc_grads(fn, other, o_out, o_lse, evoattn.DBIAS_DETERMINISTIC)
        g = _noalloc_grads(fn, x, out, lse, evoattn.DBIAS_ATOMIC)
        for n in ("dk", "dv", "dgate"):
            assert torch.equal(_bits(g[n]), _bits(ref[n])), n
        assert rel_l2(g["dbias"], ref["dbias"]) <= 1e-5
        assert rel_l2(g["dq"], ref["dq"]) <= GRAD_REL


def test_noalloc_deterministic_dq_bit_for_bit():
    """With EVOATTN_DQ_DETERMINISTIC every gradient, dq included, is fixed by
    the problem: the no-alloc entry point, after the scratch was dirtied by
    another problem, must give the workspace call's bits for all five."""
    fn = _noalloc_fn()
    flags = evoattn.DBIAS_DETERMINISTIC | evoattn.DQ_DETERMINISTIC
    x, out, lse = _problem("ending", S=12, N=200, seed=23)
    assert evoattn.workspace_size(1, 12, 2, 200, 32, flags=flags) <= SCRATCH_BYTES
    ref = evoattn.bwd(x["q"], x["k"], x["v"], x["bias"], x["mask"], x["gate"], out, lse,
                      x["dout"], flags=flags)
    ref = {k: v.clone() for k, v in ref.items()}
    other, o_out, o_lse = _problem("starting", S=24, N=256, seed=7)
    for _ in range(2):
        _noalloc_grads(fn, other, o_out, o_lse, evoattn.DBIAS_ATOMIC)  # dirty scratch
        g = _noalloc_grads(fn, x, out, lse, flags)
        for n in ("dq", "dk", "dv", "dgate", "dbias"):
            assert torch.equal(_bits(g[n]), _bits(ref[n])), n


def test_noalloc_rejects_problems_beyond_its_scratch():
    w = synthetic.small("big", B=1, S=64, N=384, H=4, D=32, dtype="bf16", node="starting",
                        mask="none", gate=False, seed=1)
    assert evoattn.workspace_size(w.B, w.S, w.H, w.N, w.D) > SCRATCH_BYTES
    x = {k: (None if v is None else to_device(v, "cuda"))
         for k, v in synthetic.make_inputs(w).items()}
    x["mask"] = torch.ones(w.B, w.S, w.N, dtype=torch.uint8, device="cuda")
    out, lse = evoattn.fwd(x["q"], x["k"], x["v"], x["bias"], x["mask"], None)
    grads = {n: torch.empty_like(x["q"]) for n in ("dq", "dk", "dv")}
    grads["dgate"] = None
    dbias = torch.empty(w.B, w.H, w.N, w.N, device="cuda")
    assert _call_noalloc(_noalloc_fn(), x, out, lse, grads, dbias) == evoattn.ERR_WORKSPACE
