"""Seeded synthetic inputs for EvoAttention (triangle and MSA-row attention).

This module only draws random tensors and lays them out; it holds none of the
attention arithmetic.  Both the CUDA path's tests/benchmark and the oracle's
tests take their inputs from here.

Layouts follow how the pair-representation projections arrive in an
AlphaFold3-style trunk (MegaFold technical summary, "Methodik" section 2: the
pair tensor is [N_token, N_token, h_pair] and successive layers alternate the
attention axis, row-wise then column-wise):

* the projected pair tensor is stored [B, N_i, N_j, H, D] (dense);
* starting node (row-wise): s = i, n = j  -> view permute(0, 1, 3, 2, 4);
* ending node (column-wise): s = j, n = i -> view permute(0, 2, 3, 1, 4), a
  strided transpose with no copy;
* MSA-row attention: the MSA projection [B, S_msa, N, H, D] with s = MSA row;
* pair bias: stored [B, H, N, N] dense; the ending node passes its (j, k)
  transpose as a view (j becomes the contiguous axis).

Every view has unit stride along D, which the tensor-memory-accelerator loads
of the CUDA path require.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    S: int
    N: int
    H: int
    D: int
    dtype: str = "bf16"          # "bf16" or "f32"
    node: str = "starting"       # "starting", "ending", "msa", or "dense"
    mask: str = "tail"           # "none", "tail" or "bernoulli"
    mask_tail: int = 0           # keys k >= N - mask_tail are masked for every s
    mask_p: float = 0.0          # probability that an (s, k) entry is masked
    gate: bool = True
    bias_std: float = 1.0
    seed: int = 0

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def logits(self) -> int:
        return self.B * self.S * self.H * self.N * self.N

    @property
    def fwd_flops(self) -> int:
        return 4 * self.logits * self.D

    @property
    def bwd_flops(self) -> int:
        return 10 * self.logits * self.D


# The five workloads of the method's evaluation space, named by what they are.
WORKLOADS = {
    w.name: w for w in [
        Workload("tiny_start_n32_fp32", B=1, S=32, N=32, H=2, D=16, dtype="f32",
                 node="starting", mask="tail", mask_tail=4, gate=False, seed=0),
        Workload("pairformer_start_n384", B=1, S=384, N=384, H=4, D=32,
                 node="starting", mask="tail", mask_tail=16, gate=True, seed=1),
        Workload("pairformer_end_n768", B=1, S=768, N=768, H=4, D=32,
                 node="ending", mask="tail", mask_tail=math.floor(0.05 * 768), gate=True, seed=2),
        Workload("msa_row_s512_n384", B=1, S=512, N=384, H=8, D=32,
                 node="msa", mask="bernoulli", mask_p=0.2, gate=True, bias_std=2.0, seed=3),
        Workload("long_start_n1536", B=1, S=1536, N=1536, H=4, D=32,
                 node="starting", mask="tail", mask_tail=math.floor(0.10 * 1536), gate=True, seed=4),
    ]
}
WORKLOAD_ORDER = list(WORKLOADS)


def _pair_view(base: torch.Tensor, node: str) -> torch.Tensor:
    """[B, X, Y, H, D] storage -> [B, S, H, N, D] view for the given axis."""
    if node in ("starting", "msa"):
        return base.permute(0, 1, 3, 2, 4)
    if node == "ending":
        return base.permute(0, 2, 3, 1, 4)
    if node == "dense":
        return base
    raise ValueError(node)


def empty_view(w: Workload, device, dtype=None) -> torch.Tensor:
    """An uninitialised [B,S,H,N,D] tensor in the workload's layout."""
    dtype = dtype or w.torch_dtype
    if w.node == "dense":
        return torch.empty(w.B, w.S, w.H, w.N, w.D, device=device, dtype=dtype)
    if w.node == "ending":
        base = torch.empty(w.B, w.N, w.S, w.H, w.D, device=device, dtype=dtype)
    else:
        base = torch.empty(w.B, w.S, w.N, w.H, w.D, device=device, dtype=dtype)
    return _pair_view(base, w.node)


def make_inputs(w: Workload, device="cpu", seed=None):
    """Draw the workload's inputs on ``device`` from a seeded generator.

    Returns a dict with q, k, v, gate (None without a gate), dout ([B,S,H,N,D]
    views in the workload layout), bias ([B,H,N,N] view) and mask ([B,S,N]
    uint8, 1 = keep, or None).  Draw order: q, k, v, bias, gate, dout, mask.
    """
    seed = w.seed if seed is None else seed
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    dt = w.torch_dtype

    def pair():
        v = empty_view(w, device, torch.float32)
        base = v
        while base._base is not None:
            base = base._base
        base.normal_(0.0, 1.0, generator=gen)
        return v.to(dt) if dt != torch.float32 else v

    def keep_layout(x):
        # .to() of a permuted view keeps strides (preserve_format); force the
        # same physical layout as the workload's pair storage regardless.
        out = empty_view(w, device, dt)
        out.copy_(x)
        return out

    q = keep_layout(pair())
    k = keep_layout(pair())
    v = keep_layout(pair())
    bias_base = torch.empty(w.B, w.H, w.N, w.N, device=device, dtype=torch.float32)
    bias_base.normal_(0.0, w.bias_std, generator=gen)
    bias_base = bias_base.to(dt)
    bias = bias_base.transpose(2, 3) if w.node == "ending" else bias_base
    gate = keep_layout(pair()) if w.gate else None
    dout = keep_layout(pair())
    mask = None
    if w.mask == "tail":
        mask = torch.ones(w.B, w.S, w.N, device=device, dtype=torch.uint8)
        if w.mask_tail > 0:
            mask[:, :, w.N - w.mask_tail:] = 0
    elif w.mask == "bernoulli":
        u = torch.rand(w.B, w.S, w.N, device=device, generator=gen)
        mask = (u >= w.mask_p).to(torch.uint8)
        dead = mask.sum(-1) == 0          # keep at least one key per row
        if bool(dead.any()):
            mask[..., 0] = torch.where(dead, torch.ones_like(mask[..., 0]), mask[..., 0])
    elif w.mask != "none":
        raise ValueError(w.mask)
    return {"q": q, "k": k, "v": v, "bias": bias, "gate": gate, "dout": dout, "mask": mask}


def small(name="case", B=1, S=3, N=5, H=2, D=4, **kw) -> Workload:
    """A small workload for tests (default: the finite-difference shape)."""
    return Workload(name, B=B, S=S, N=N, H=H, D=D, **kw)


def make_fusion_inputs(B, N, C, H, D, seed=0, device="cpu"):
    """Seeded inputs of the EvoFusion upstream stack (LayerNorm + projection):
    z [B, N, N, C] bf16 with a per-channel offset and scale (so the
    normalisation has a mean and a spread to remove), gamma ~ 1 + 0.1 N(0,1)
    and beta ~ 0.1 N(0,1) in fp32, and w [4*H*D + H, C] bf16 ~ N(0, 1/C) (so
    every projected value is of order one).  Draw order: channel offsets,
    channel scales, z, gamma, beta, w."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    f32 = dict(device=device, dtype=torch.float32)
    mu = torch.randn(C, generator=gen, **f32)
    sd = torch.rand(C, generator=gen, **f32) * 1.5 + 0.5
    z = (torch.randn(B, N, N, C, generator=gen, **f32) * sd + mu).to(torch.bfloat16)
    gamma = 1.0 + 0.1 * torch.randn(C, generator=gen, **f32)
    beta = 0.1 * torch.randn(C, generator=gen, **f32)
    w = (torch.randn(4 * H * D + H, C, generator=gen, **f32) * C ** -0.5).to(torch.bfloat16)
    return {"z": z, "gamma": gamma, "beta": beta, "w": w}


def make_transition_inputs(B, N, C, F, seed=0, device="cpu", HD=0):
    """Seeded inputs of the EvoFusion downstream stack (the SwiGLU transition
    with its residual add, optionally preceded by the attention's output
    projection): z [B, N, N, C] bf16 with a per-channel offset and scale,
    gamma ~ 1 + 0.1 N(0,1) and beta ~ 0.1 N(0,1) in fp32, w1 [2F, C] bf16
    ~ N(0, 1/C) (so the SiLU and linear branches are of order one), w2 [C, F]
    bf16 ~ N(0, 1/F) and, when HD > 0, the gated attention output o
    [B, N, N, HD] bf16 ~ N(0, 1/4) (the size of a gated, averaged value) and
    w_o [C, HD] bf16 ~ N(0, 1/HD).  Draw order: channel offsets, channel
    scales, z, gamma, beta, w1, w2, o, w_o."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    f32 = dict(device=device, dtype=torch.float32)
    mu = torch.randn(C, generator=gen, **f32)
    sd = torch.rand(C, generator=gen, **f32) * 1.5 + 0.5
    z = (torch.randn(B, N, N, C, generator=gen, **f32) * sd + mu).to(torch.bfloat16)
    gamma = 1.0 + 0.1 * torch.randn(C, generator=gen, **f32)
    beta = 0.1 * torch.randn(C, generator=gen, **f32)
    w1 = (torch.randn(2 * F, C, generator=gen, **f32) * C ** -0.5).to(torch.bfloat16)
    w2 = (torch.randn(C, F, generator=gen, **f32) * F ** -0.5).to(torch.bfloat16)
    x = {"z": z, "gamma": gamma, "beta": beta, "w1": w1, "w2": w2, "o": None, "w_o": None}
    if HD > 0:
        x["o"] = (torch.randn(B, N, N, HD, generator=gen, **f32) * 0.5).to(torch.bfloat16)
        x["w_o"] = (torch.randn(C, HD, generator=gen, **f32) * HD ** -0.5).to(torch.bfloat16)
    return x
