"""The C ABI without a GPU: the library loads, exports every entry point that
include/evoattn.h declares, and rejects bad arguments on the host with the
documented status before touching the device (fake pointers are never
dereferenced because validation fails first)."""
import ctypes
import os
import re

import pytest

from protein_folding_attention_gb300 import build_lib, evoattn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_lib.build()
    return evoattn.load()


def declared_entry_points():
    text = open(os.path.join(ROOT, "include", "evoattn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(evoattn_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_entry_points()
    assert {"evoattn_fwd", "evoattn_bwd", "evoattn_bwd_workspace_size",
            "evoattn_get_device_status", "evoattn_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/evoattn.h but not exported"


def test_status_strings(lib):
    for code in range(7):
        s = evoattn.status_string(code)
        assert s and s != "unknown status"
    assert evoattn.status_string(99) == "unknown status"
    assert lib.evoattn_version() >= 100


S5 = ctypes.c_int64 * 5
S4 = ctypes.c_int64 * 4
S3 = ctypes.c_int64 * 3
FAKE = ctypes.c_void_p(1 << 20)  # 16-byte aligned, never dereferenced


def dense5(B, S, H, N, D):
    return S5(S * H * N * D, H * N * D, N * D, D, 1)


def call_fwd(lib, *, q=FAKE, qs=None, bias=FAKE, bs=None, mask=None, ms=None, gate=None,
             gs=None, out=FAKE, lse=FAKE, shape=(1, 4, 2, 64, 32), dtype=evoattn.BF16):
    B, S, H, N, D = shape
    qs = qs or dense5(*shape)
    bs = bs or S4(H * N * N, N * N, N, 1)
    return lib.evoattn_fwd(q, qs, FAKE, qs, FAKE, qs, bias, bs, mask, ms, gate, gs or qs,
                           out, qs, lse, B, S, H, N, D, dtype, None)


def test_fwd_rejects_bad_arguments(lib):
    assert call_fwd(lib, q=None) == evoattn.ERR_INVALID_ARG
    assert call_fwd(lib, bias=None) == evoattn.ERR_INVALID_ARG
    assert call_fwd(lib, lse=None) == evoattn.ERR_INVALID_ARG
    assert call_fwd(lib, shape=(1, 0, 2, 64, 32)) == evoattn.ERR_INVALID_ARG
    assert call_fwd(lib, mask=FAKE, ms=None) == evoattn.ERR_INVALID_ARG
    assert call_fwd(lib, shape=(1, 4, 2, 64, 48)) == evoattn.ERR_UNSUPPORTED
    assert call_fwd(lib, shape=(1, 4, 2, 64, 128)) == evoattn.ERR_UNSUPPORTED  # bf16 D<=64
    assert call_fwd(lib, dtype=7) == evoattn.ERR_UNSUPPORTED
    neg = S5(-1, 1, 1, 1, 1)
    assert call_fwd(lib, qs=neg) == evoattn.ERR_INVALID_ARG


def test_fwd_bf16_alignment_rules(lib):
    shape = (1, 4, 2, 64, 32)
    # d stride must be 1
    assert call_fwd(lib, qs=S5(2 * 4 * 2 * 64 * 32, 2 * 2 * 64 * 32, 2 * 64 * 32, 64, 2)) == \
        evoattn.ERR_ALIGNMENT
    # other strides multiples of 8 elements
    assert call_fwd(lib, qs=S5(4 * 2 * 64 * 36, 2 * 64 * 36, 64 * 36, 36, 1)) == \
        evoattn.ERR_ALIGNMENT
    # 16-byte aligned base
    assert call_fwd(lib, q=ctypes.c_void_p((1 << 20) + 8)) == evoattn.ERR_ALIGNMENT
    # bias: unit stride along k or j, not neither
    assert call_fwd(lib, bs=S4(2 * 64 * 64 * 8, 64 * 64 * 8, 64 * 8, 8)) == evoattn.ERR_ALIGNMENT
    # bias row stride not a multiple of 8
    assert call_fwd(lib, bs=S4(2 * 64 * 68, 64 * 68, 66, 1)) == evoattn.ERR_ALIGNMENT
    # lse must be 16-byte aligned
    assert call_fwd(lib, lse=ctypes.c_void_p((1 << 20) + 4)) == evoattn.ERR_ALIGNMENT
    del shape


def call_bwd(lib, *, gate=None, dgate=None, ws=FAKE, ws_bytes=1 << 40, flags=0,
             shape=(1, 4, 2, 64, 32), dtype=evoattn.BF16, dq=FAKE):
    B, S, H, N, D = shape
    s = dense5(*shape)
    bs = S4(H * N * N, N * N, N, 1)
    return lib.evoattn_bwd(FAKE, s, FAKE, s, FAKE, s, FAKE, bs, None, None, gate, s, FAKE, s,
                           FAKE, FAKE, s, dq, s, FAKE, s, FAKE, s, FAKE, dgate, s,
                           B, S, H, N, D, dtype, flags, ws, ws_bytes, None)


def test_bwd_rejects_bad_arguments(lib):
    assert call_bwd(lib, dq=None) == evoattn.ERR_INVALID_ARG
    assert call_bwd(lib, gate=FAKE, dgate=None) == evoattn.ERR_INVALID_ARG
    assert call_bwd(lib, gate=None, dgate=FAKE) == evoattn.ERR_INVALID_ARG
    assert call_bwd(lib, flags=8) == evoattn.ERR_INVALID_ARG
    assert call_bwd(lib, flags=14) == evoattn.ERR_INVALID_ARG
    assert call_bwd(lib, ws=None) == evoattn.ERR_WORKSPACE
    assert call_bwd(lib, ws_bytes=16) == evoattn.ERR_WORKSPACE
    assert call_bwd(lib, ws=ctypes.c_void_p((1 << 20) + 16)) == evoattn.ERR_WORKSPACE
    assert call_bwd(lib, shape=(1, 4, 2, 64, 24)) == evoattn.ERR_UNSUPPORTED


def call_bwd_noalloc(lib, *, shape=(1, 4, 2, 64, 32), dtype=evoattn.BF16, flags=0):
    B, S, H, N, D = shape
    s = dense5(*shape)
    bs = S4(H * N * N, N * N, N, 1)
    fn = lib.evoattn_bwd_noalloc
    fn.argtypes = lib.evoattn_bwd.argtypes[:-3] + [ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn(FAKE, s, FAKE, s, FAKE, s, FAKE, bs, None, None, None, s, FAKE, s,
              FAKE, FAKE, s, FAKE, s, FAKE, s, FAKE, s, FAKE, None, s,
              B, S, H, N, D, dtype, flags, None)


def test_bf16_backward_d64_is_unsupported(lib):
    """The BF16 forward takes D = 64, the BF16 backward does not: every
    backward entry point says so with ERR_UNSUPPORTED (not a CUDA or
    workspace error), and the workspace query returns 0."""
    shape = (1, 4, 2, 64, 64)
    assert call_bwd(lib, shape=shape) == evoattn.ERR_UNSUPPORTED
    assert call_bwd(lib, shape=shape, flags=1) == evoattn.ERR_UNSUPPORTED
    assert call_bwd_noalloc(lib, shape=shape) == evoattn.ERR_UNSUPPORTED
    assert evoattn.workspace_size(1, 4, 2, 64, 64) == 0
    # fp32 inputs have a D = 64 backward
    assert evoattn.workspace_size(1, 4, 2, 64, 64, torch_f32()) > 0
    # the forward accepts BF16 D = 64 (validation passes up to the alignment checks)
    assert call_fwd(lib, shape=shape, q=ctypes.c_void_p((1 << 20) + 8)) == evoattn.ERR_ALIGNMENT


def test_fused_dbias_workspace(lib):
    """EVOATTN_DBIAS_FUSED keeps no slot partials: its workspace equals the
    atomic mode's (both modes of dQ), below the deterministic mode's."""
    B, S, H, N, D = 1, 8, 2, 300, 32
    for dq in (0, evoattn.DQ_DETERMINISTIC):
        fused = evoattn.workspace_size(B, S, H, N, D, flags=evoattn.DBIAS_FUSED | dq)
        assert fused == evoattn.workspace_size(B, S, H, N, D, flags=evoattn.DBIAS_ATOMIC | dq)
        assert fused < evoattn.workspace_size(B, S, H, N, D, flags=dq)
        assert fused == evoattn.workspace_size(
            B, S, H, N, D, flags=evoattn.DBIAS_FUSED | evoattn.DBIAS_ATOMIC | dq)


def test_deterministic_dq_workspace(lib):
    """EVOATTN_DQ_DETERMINISTIC combines with either dbias mode; its BF16
    workspace holds one fp32 dQ slice per 128-key tile instead of one, the
    F32 workspace does not change, and an unknown bit makes the size query
    return 0."""
    B, S, H, N, D = 1, 8, 2, 300, 32
    L = B * S * H * N * D
    nkt = (N + 127) // 128
    for dbias in (evoattn.DBIAS_DETERMINISTIC, evoattn.DBIAS_ATOMIC):
        base = evoattn.workspace_size(B, S, H, N, D, flags=dbias)
        det = evoattn.workspace_size(B, S, H, N, D, flags=dbias | evoattn.DQ_DETERMINISTIC)
        assert det - base == (nkt - 1) * L * 4
        assert call_bwd(lib, shape=(B, S, H, N, D), flags=dbias | evoattn.DQ_DETERMINISTIC,
                        ws_bytes=det - 256) == \
            evoattn.ERR_WORKSPACE
    f32 = torch_f32()
    assert evoattn.workspace_size(B, S, H, N, D, f32, flags=evoattn.DQ_DETERMINISTIC) == \
        evoattn.workspace_size(B, S, H, N, D, f32)
    assert evoattn.workspace_size(B, S, H, N, D, flags=8) == 0
    assert call_bwd_noalloc(lib, flags=8) == evoattn.ERR_INVALID_ARG


def test_debug_wait_hook_round_trips(lib):
    assert lib.evoattn_debug_set_wait(50_000, 1) == evoattn.OK
    assert lib.evoattn_debug_set_wait(0, 0) == evoattn.OK


def test_workspace_is_linear_not_cubic(lib):
    for dt in (torch_bf16(), torch_f32()):
        small = evoattn.workspace_size(1, 64, 4, 256, 32, dt)
        assert small > 0
        big = evoattn.workspace_size(1, 768, 4, 768, 32, dt)
        cubic = 1 * 768 * 4 * 768 * 768 * 2  # bf16 logits of the whole problem
        assert big < cubic / 4
    assert evoattn.workspace_size(1, 8, 2, 64, 48) == 0


def torch_bf16():
    import torch
    return torch.bfloat16


def torch_f32():
    import torch
    return torch.float32


def call_ln_proj(lib, *, z=FAKE, w=FAKE, q=FAKE, eps=1e-5, B=1, N=8, C=128, H=4, D=32):
    return lib.evoattn_ln_proj(z, FAKE, FAKE, w, eps, q, FAKE, FAKE, FAKE, FAKE,
                               B, N, C, H, D, None)


def test_ln_proj_rejects_bad_arguments(lib):
    assert call_ln_proj(lib, z=None) == evoattn.ERR_INVALID_ARG
    assert call_ln_proj(lib, q=None) == evoattn.ERR_INVALID_ARG
    assert call_ln_proj(lib, N=0) == evoattn.ERR_INVALID_ARG
    assert call_ln_proj(lib, eps=0.0) == evoattn.ERR_INVALID_ARG
    assert call_ln_proj(lib, eps=float("nan")) == evoattn.ERR_INVALID_ARG
    assert call_ln_proj(lib, C=64) == evoattn.ERR_UNSUPPORTED
    assert call_ln_proj(lib, H=4, D=16) == evoattn.ERR_UNSUPPORTED   # H*D != 128
    assert call_ln_proj(lib, H=16, D=8) == evoattn.ERR_UNSUPPORTED   # more than 8 heads
    assert call_ln_proj(lib, B=1, N=50000) == evoattn.ERR_UNSUPPORTED  # B*N*N >= 2^31
    assert call_ln_proj(lib, z=ctypes.c_void_p((1 << 20) + 8)) == evoattn.ERR_ALIGNMENT
    assert call_ln_proj(lib, w=ctypes.c_void_p((1 << 20) + 2)) == evoattn.ERR_ALIGNMENT


def call_transition(lib, *, z=FAKE, o=None, w_o=None, w1=FAKE, w2=FAKE, out=FAKE, eps=1e-5,
                    B=1, N=8, C=128, HD=128, F=512):
    return lib.evoattn_transition(z, o, w_o, FAKE, FAKE, w1, w2, eps, out, B, N, C, HD, F, None)


def test_transition_rejects_bad_arguments(lib):
    assert call_transition(lib, z=None) == evoattn.ERR_INVALID_ARG
    assert call_transition(lib, w2=None) == evoattn.ERR_INVALID_ARG
    assert call_transition(lib, out=None) == evoattn.ERR_INVALID_ARG
    assert call_transition(lib, o=FAKE) == evoattn.ERR_INVALID_ARG        # o without w_o
    assert call_transition(lib, w_o=FAKE) == evoattn.ERR_INVALID_ARG      # w_o without o
    assert call_transition(lib, N=0) == evoattn.ERR_INVALID_ARG
    assert call_transition(lib, eps=0.0) == evoattn.ERR_INVALID_ARG
    assert call_transition(lib, eps=float("inf")) == evoattn.ERR_INVALID_ARG
    assert call_transition(lib, C=64, F=256) == evoattn.ERR_UNSUPPORTED
    assert call_transition(lib, F=256) == evoattn.ERR_UNSUPPORTED    # F != 4C
    assert call_transition(lib, o=FAKE, w_o=FAKE, HD=64) == evoattn.ERR_UNSUPPORTED
    assert call_transition(lib, B=1, N=50000) == evoattn.ERR_UNSUPPORTED  # B*N*N >= 2^31
    assert call_transition(lib, z=ctypes.c_void_p((1 << 20) + 8)) == evoattn.ERR_ALIGNMENT
    assert call_transition(lib, w1=ctypes.c_void_p((1 << 20) + 2)) == evoattn.ERR_ALIGNMENT
    assert call_transition(lib, out=ctypes.c_void_p((1 << 20) + 4)) == evoattn.ERR_ALIGNMENT
    assert call_transition(lib, o=ctypes.c_void_p((1 << 20) + 8), w_o=FAKE) == \
        evoattn.ERR_ALIGNMENT
