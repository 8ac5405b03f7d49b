"""Shared helpers for the GPU parity tests (no attention arithmetic here)."""
import numpy as np
import torch


def to_device(x, dev):
    """Copy keeping the exact strides (the layouts under test are views)."""
    if x is None:
        return None
    y = torch.empty_strided(x.size(), x.stride(), dtype=x.dtype, device=dev)
    y.copy_(x)
    return y


def as_np(t):
    return t.detach().to(torch.float64).cpu().numpy() if hasattr(t, "detach") else np.asarray(t)


def rel_l2(gpu, ref):
    g, r = as_np(gpu), as_np(ref)
    return float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-300))


def max_abs(gpu, ref):
    return float(np.abs(as_np(gpu) - as_np(ref)).max())


# Tolerances of the method's parity bar: forward rel-L2 <= 5e-3 and max-abs
# <= 2e-2 for bf16, gradients rel-L2 <= 1e-2 for bf16, everything <= 1e-5
# for fp32 inputs.
FWD_REL, FWD_ABS, GRAD_REL, F32_REL = 5e-3, 2e-2, 1e-2, 1e-5
