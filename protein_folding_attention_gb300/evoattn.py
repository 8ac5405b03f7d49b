"""Python binding of the EvoAttention C ABI (``include/evoattn.h``).

Argument marshalling only: every step of the computation runs in the CUDA
library ``libevoattn.so`` built in-tree by ``build_lib.build()``.  PyTorch
provides device memory and the current stream; tensors are passed as raw
pointers plus element strides.  There is no fallback: if the library is
missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libevoattn.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_ALIGNMENT, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT = range(7)
BF16, F32 = 0, 1
DBIAS_DETERMINISTIC, DBIAS_ATOMIC = 0, 1
DQ_DETERMINISTIC = 2  # OR-ed with either: dq bit-identical too
DBIAS_FUSED = 4  # dbias summed in the dK/dV pass (fp32 atomics)

_lib = None
_I64_5 = ctypes.c_int64 * 5
_I64_4 = ctypes.c_int64 * 4
_I64_3 = ctypes.c_int64 * 3


class EvoAttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


def load(path: str = LIB_PATH):
    """Load the CUDA library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"EvoAttention CUDA library not built: {path} is missing "
                           "(run __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    vp, i64p, u8p, fp = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int64), ctypes.c_void_p, ctypes.c_void_p
    i, u, sz = ctypes.c_int, ctypes.c_uint, ctypes.c_size_t
    lib.evoattn_fwd.argtypes = [vp, i64p, vp, i64p, vp, i64p, vp, i64p, u8p, i64p, vp, i64p,
                                vp, i64p, fp, i, i, i, i, i, i, vp]
    lib.evoattn_fwd.restype = i
    lib.evoattn_bwd_workspace_size.argtypes = [i, i, i, i, i, i, u]
    lib.evoattn_bwd_workspace_size.restype = sz
    lib.evoattn_bwd.argtypes = [vp, i64p, vp, i64p, vp, i64p, vp, i64p, u8p, i64p, vp, i64p,
                                vp, i64p, fp, vp, i64p, vp, i64p, vp, i64p, vp, i64p, fp,
                                vp, i64p, i, i, i, i, i, i, u, vp, sz, vp]
    lib.evoattn_bwd.restype = i
    lib.evoattn_bwd_profiled.argtypes = lib.evoattn_bwd.argtypes + [ctypes.POINTER(vp)]
    lib.evoattn_bwd_profiled.restype = i
    lib.evoattn_get_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_int)]
    lib.evoattn_get_device_status.restype = i
    lib.evoattn_status_string.argtypes = [i]
    lib.evoattn_status_string.restype = ctypes.c_char_p
    lib.evoattn_version.argtypes = []
    lib.evoattn_version.restype = i
    lib.evoattn_ln_proj.argtypes = [vp, fp, fp, vp, ctypes.c_float, vp, vp, vp, vp, vp,
                                    i, i, i, i, i, vp]
    lib.evoattn_ln_proj.restype = i
    lib.evoattn_transition.argtypes = [vp, vp, vp, fp, fp, vp, vp, ctypes.c_float, vp,
                                       i, i, i, i, i, vp]
    lib.evoattn_transition.restype = i
    lib.evoattn_debug_set_wait.argtypes = [ctypes.c_ulonglong, i]
    lib.evoattn_debug_set_wait.restype = i
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().evoattn_status_string(int(status)).decode()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {t.dtype} (bf16 or fp32)")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _s5(t):
    return None if t is None else _I64_5(*t.stride())


def _s4(t):
    return None if t is None else _I64_4(*t.stride())


def _s3(t):
    return None if t is None else _I64_3(*t.stride())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status: int, what: str):
    if status != OK:
        raise EvoAttnError(status, what)


def fwd(q, k, v, pair_bias, mask=None, gate=None, out=None, lse=None, stream=None):
    """out = sigmoid(gate) * softmax(q k^T / sqrt(D) + pair_bias + mask_bias) v.

    q, k, v, gate: [B,S,H,N,D] (any strides; bf16 needs unit stride along D);
    pair_bias: [B,H,N,N]; mask: [B,S,N] uint8/bool (nonzero = keep) or None.
    Returns (out, lse); out defaults to a dense tensor like q, lse is fp32
    [B,S,H,N] contiguous.
    """
    lib = load()
    B, S, H, N, D = q.shape
    if out is None:
        out = torch.empty((B, S, H, N, D), device=q.device, dtype=q.dtype)
    if lse is None:
        lse = torch.empty((B, S, H, N), device=q.device, dtype=torch.float32)
    if mask is not None and mask.dtype != torch.uint8:
        mask = mask.to(torch.uint8)
    st = lib.evoattn_fwd(_ptr(q), _s5(q), _ptr(k), _s5(k), _ptr(v), _s5(v),
                         _ptr(pair_bias), _s4(pair_bias), _ptr(mask), _s3(mask),
                         _ptr(gate), _s5(gate), _ptr(out), _s5(out), _ptr(lse),
                         B, S, H, N, D, _dtype_code(q), _stream(stream))
    _check(st, "evoattn_fwd")
    return out, lse


def workspace_size(B, S, H, N, D, dtype=torch.bfloat16, flags=DBIAS_DETERMINISTIC) -> int:
    code = BF16 if dtype == torch.bfloat16 else F32
    return int(load().evoattn_bwd_workspace_size(B, S, H, N, D, code, flags))


def bwd(q, k, v, pair_bias, mask, gate, out, lse, dout, flags=DBIAS_DETERMINISTIC,
        dq=None, dk=None, dv=None, dbias=None, dgate=None, workspace=None, stream=None,
        stage_events=None):
    """Gradients of sum(out * dout).  Returns dict dq, dk, dv (like q), dbias
    (fp32 [B,H,N,N]) and dgate (None without a gate).  `stage_events`: five
    torch.cuda.Event recorded around the backward's kernels (see
    evoattn_bwd_profiled)."""
    lib = load()
    B, S, H, N, D = q.shape
    mk = lambda t: t if t is not None else torch.empty((B, S, H, N, D), device=q.device,
                                                       dtype=q.dtype)
    dq, dk, dv = mk(dq), mk(dk), mk(dv)
    if gate is not None:
        dgate = mk(dgate)
    else:
        dgate = None
    if dbias is None:
        dbias = torch.empty((B, H, N, N), device=q.device, dtype=torch.float32)
    if mask is not None and mask.dtype != torch.uint8:
        mask = mask.to(torch.uint8)
    need = workspace_size(B, S, H, N, D, q.dtype, flags)
    if workspace is None:
        workspace = torch.empty(max(need, 1), device=q.device, dtype=torch.uint8)
    args = (_ptr(q), _s5(q), _ptr(k), _s5(k), _ptr(v), _s5(v),
            _ptr(pair_bias), _s4(pair_bias), _ptr(mask), _s3(mask),
            _ptr(gate), _s5(gate), _ptr(out), _s5(out), _ptr(lse),
            _ptr(dout), _s5(dout), _ptr(dq), _s5(dq), _ptr(dk), _s5(dk),
            _ptr(dv), _s5(dv), _ptr(dbias), _ptr(dgate), _s5(dgate),
            B, S, H, N, D, _dtype_code(q), flags, _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream(stream))
    if stage_events is None:
        st = lib.evoattn_bwd(*args)
    else:
        if len(stage_events) != 5:
            raise ValueError("stage_events needs 5 events")
        cur = stream if stream is not None else torch.cuda.current_stream()
        for e in stage_events:           # torch creates events lazily on first record
            if not getattr(e, "cuda_event", 0):
                e.record(cur)
        handles = (ctypes.c_void_p * 5)(*[ctypes.c_void_p(e.cuda_event) for e in stage_events])
        st = lib.evoattn_bwd_profiled(*args, handles)
    _check(st, "evoattn_bwd")
    return {"dq": dq, "dk": dk, "dv": dv, "dbias": dbias, "dgate": dgate}


def ln_proj(z, gamma, beta, w, H, D, eps=1e-5, out=None, stream=None):
    """EvoFusion upstream stack: LayerNorm of z [B, N, N, C] (bf16, dense) with
    gamma, beta [C] (fp32), then the bias-free projection w [4*H*D + H, C]
    (bf16).  Returns (q, k, v, g, pair_bias): q..g [B, N, N, H, D] bf16 and
    pair_bias [B, H, N, N] bf16 (see evoattn_ln_proj).  `out` may supply the
    five output tensors."""
    lib = load()
    B, N, N2, C = z.shape
    if N2 != N:
        raise ValueError("z must be [B, N, N, C]")
    if out is None:
        mk = lambda: torch.empty((B, N, N, H, D), device=z.device, dtype=torch.bfloat16)
        out = (mk(), mk(), mk(), mk(),
               torch.empty((B, H, N, N), device=z.device, dtype=torch.bfloat16))
    q, k, v, g, bias = out
    st = lib.evoattn_ln_proj(_ptr(z), _ptr(gamma), _ptr(beta), _ptr(w), float(eps),
                             _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(bias),
                             B, N, C, H, D, _stream(stream))
    _check(st, "evoattn_ln_proj")
    return q, k, v, g, bias


def transition(z, gamma, beta, w1, w2, eps=1e-5, o=None, w_o=None, out=None, stream=None):
    """EvoFusion downstream stack: z1 = z + o w_o^T (when o is given), then
    out = z1 + SwiGLU transition of LayerNorm(z1), for z [B, N, N, C] (bf16,
    dense), o [B, N, N, HD] and w_o [C, HD] (bf16), gamma, beta [C] (fp32),
    w1 [2F, C] and w2 [C, F] (bf16).  Returns out [B, N, N, C] bf16 (see
    evoattn_transition)."""
    lib = load()
    B, N, N2, C = z.shape
    if N2 != N:
        raise ValueError("z must be [B, N, N, C]")
    F = w2.shape[1]
    HD = o.shape[-1] if o is not None else 0
    if out is None:
        out = torch.empty_like(z)
    st = lib.evoattn_transition(_ptr(z), _ptr(o), _ptr(w_o), _ptr(gamma), _ptr(beta),
                                _ptr(w1), _ptr(w2), float(eps), _ptr(out), B, N, C, HD, F,
                                _stream(stream))
    _check(st, "evoattn_transition")
    return out


def debug_set_wait(limit_ns: int = 0, stall: bool = False) -> None:
    """Testing hook (evoattn_debug_set_wait): the wait limit of the kernels
    enqueued from now on (0 = the default 2 s) and whether their compute warps'
    first wait stalls until it gives up."""
    _check(load().evoattn_debug_set_wait(int(limit_ns), 1 if stall else 0),
           "evoattn_debug_set_wait")


def device_status(stream=None) -> int:
    """Synchronise the stream, then read and clear the device status word."""
    out = ctypes.c_int(-1)
    _check(load().evoattn_get_device_status(_stream(stream), ctypes.byref(out)),
           "evoattn_get_device_status")
    return out.value
