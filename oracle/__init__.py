"""EvoAttention oracle -- test infrastructure only.

A plain float64 CPU statement of the attention over the pair representation
that MegaFold's EvoFlash-3D kernel computes (MegaFold technical summary,
"Methodik" section 1 "EvoFlash-3D": online numerically stable softmax, logits
with an additively broadcast pair-bias term) and of its analytic backward.
The arithmetic lives in ``evoattn_oracle.c`` (plain C, float64, OpenMP over
independent slices); this module compiles it and marshals arrays.

Only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does, and
this package imports nothing from the product.

Parity status of every function here: pinned (see tests/test_oracle_pins.py).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "evoattn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/liboracle.so`` with gcc (-O2, IEEE math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        dp = ctypes.POINTER(ctypes.c_double)
        u8 = ctypes.POINTER(ctypes.c_uint8)
        i = ctypes.c_int
        lib.oracle_fwd.argtypes = [dp, dp, dp, dp, u8, dp, dp, dp, i, i, i, i, i]
        lib.oracle_fwd.restype = i
        lib.oracle_bwd.argtypes = [dp, dp, dp, dp, u8, dp, dp, dp, dp, dp, dp, dp, i, i, i, i, i]
        lib.oracle_bwd.restype = i
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = i
        _lib = lib
    return _lib


def _f64(x):
    """Dense float64 copy of a numpy array or torch tensor (exact for bf16/fp32)."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: widen on its own device, then move
        import torch
        x = x.detach().to(torch.float64).cpu().contiguous().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _u8(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu().contiguous().numpy()
    return np.ascontiguousarray(np.asarray(x).astype(np.uint8))


def _ptr(a, kind=ctypes.c_double):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(kind))


def num_threads() -> int:
    """OpenMP threads one oracle call uses."""
    return int(_load().oracle_num_threads())


def fwd(q, k, v, bias, mask=None, gate=None):
    """Forward of the pair-biased gated attention.

    q, k, v, gate: [B,S,H,N,D]; bias: [B,H,N,N] (indexed [b,h,j,k], j = query
    row, k = key); mask: [B,S,N], nonzero = keep.  Any strides are accepted
    here; the C code sees dense copies.  Returns (out [B,S,H,N,D], lse
    [B,S,H,N]) as float64 numpy arrays.
    """
    q, k, v, bias, gate = map(_f64, (q, k, v, bias, gate))
    mask = _u8(mask)
    B, S, H, N, D = q.shape
    assert k.shape == q.shape and v.shape == q.shape and bias.shape == (B, H, N, N)
    assert mask is None or mask.shape == (B, S, N)
    assert gate is None or gate.shape == q.shape
    out = np.empty_like(q)
    lse = np.empty((B, S, H, N))
    rc = _load().oracle_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(bias), _ptr(mask, ctypes.c_uint8),
                            _ptr(gate), _ptr(out), _ptr(lse), B, S, H, N, D)
    if rc != 0:
        raise RuntimeError("oracle_fwd failed")
    return out, lse


def bwd(q, k, v, bias, mask, gate, dout):
    """Backward: returns dict with dq, dk, dv ([B,S,H,N,D]), dbias ([B,H,N,N],
    summed over s in ascending order) and dgate ([B,S,H,N,D], None without a
    gate), all float64.  The forward is recomputed from the inputs."""
    q, k, v, bias, gate, dout = map(_f64, (q, k, v, bias, gate, dout))
    mask = _u8(mask)
    B, S, H, N, D = q.shape
    assert dout.shape == q.shape and bias.shape == (B, H, N, N)
    dq, dk, dv = np.empty_like(q), np.empty_like(q), np.empty_like(q)
    dbias = np.empty((B, H, N, N))
    dgate = np.empty_like(q) if gate is not None else None
    rc = _load().oracle_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(bias), _ptr(mask, ctypes.c_uint8),
                            _ptr(gate), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dbias),
                            _ptr(dgate), B, S, H, N, D)
    if rc != 0:
        raise RuntimeError("oracle_bwd failed")
    return {"dq": dq, "dk": dk, "dv": dv, "dbias": dbias, "dgate": dgate}
