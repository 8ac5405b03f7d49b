#!/usr/bin/env python3
"""EvoAttention forward + backward benchmark on GB300.

One step = evoattn_fwd + evoattn_bwd (every kernel of the path) over the
ending-node triangle attention of the N=768 pair representation
(B=1, S=N=768, H=4, D=32, bf16, 5 % trailing key mask, sigmoid gate), with
the inputs already resident in HBM.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Throughput counts 4*B*S*H*N^2*D FLOP for the forward and 2.5x that for the
backward.  With N>1 (torchrun) every rank runs its own replica of the
workload (the path has no cross-GPU exchange); the value is the total FLOP of
all ranks over the slowest rank's time.  `--impl reference` times the float64
CPU oracle on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "EvoAttention fwd+bwd TFLOP/s and % of GB300 BF16 dense peak (N=768 triangle attn)"
WORKLOAD = "pairformer_end_n768"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# ex2.approx.f32 results per clock per SM on GB300: the XU pipe takes a warp
# instruction every 2 clocks per sub-partition (16 per sub-partition); a
# register-only run of the softmax inner loop reached 55.6 per clock per SM.
# The third roofline of the path, beside HBM and tensor cores.
EX2_PER_CLK_PER_SM = 64


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        loaded = [x for x in sm if x > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def max_over_ranks(seconds: float, dist=None, device=None) -> float:
    """Slowest rank's time (the job's time); identity without a process group."""
    if dist is None:
        return seconds
    import torch
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_rank: float, world_size: int, seconds_per_step: float) -> float:
    """Whole-job throughput: every rank's FLOP over the slowest rank's step time."""
    return flops_per_rank * world_size / seconds_per_step / 1e12


def config_block(w):
    return {"workload": w.name, "B": w.B, "S": w.S, "N": w.N, "H": w.H, "D": w.D,
            "node": w.node, "mask": f"{w.mask_tail} trailing keys masked" if w.mask == "tail"
            else w.mask, "gate": w.gate, "global_batch": w.B * w.S, "seq_len": w.N,
            "parallelism": "replicas", "l2": "inputs larger than L2 (no flush needed)"}


PER_CONFIG = ("pairformer_start_n384", "pairformer_end_n768", "msa_row_s512_n384",
              "long_start_n1536")


def algorithmic_bytes(w):
    """HBM bytes the forward and the backward must move at least, the logits
    never counted (they stay on chip): forward reads q, k, v, g, the pair
    bias and the mask and writes out and lse; backward reads q, k, v, g, out
    and dout, the pair bias, the mask, lse and delta, and writes dq, dk, dv,
    dgate and dbias (fp32).  Returns (forward, backward)."""
    L = w.B * w.S * w.H * w.N * w.D
    R = w.B * w.S * w.H * w.N
    n2 = w.B * w.H * w.N * w.N
    e = 2 if w.dtype == "bf16" else 4
    gl = 1 if w.gate else 0
    mask = w.B * w.S * w.N if w.mask != "none" else 0
    fwd = (3 + gl) * L * e + n2 * e + mask + L * e + R * 4
    bwd = (5 + gl) * L * e + (3 + gl) * L * e + n2 * e + n2 * 4 + mask + 3 * R * 4
    return fwd, bwd


def measure_config(w, dev, peak, steps=5, warmup=3, hbm_peak=None, ex2_peak=None):
    """Forward and backward of one workload on its own inputs: CUDA-event
    times (median over `steps`), TFLOP/s, fraction of the bf16 peak, the
    rate of the algorithmic HBM bytes against the measured copy bandwidth
    (`hbm_peak`, GB/s), logits per second against the exponential unit
    (`ex2_peak`, ex2/s; one ex2 per logit in each pass), and the device bytes
    the caller holds for the call (inputs, outputs and the backward
    workspace: the library allocates nothing itself).  Returns a dict; every
    tensor it allocated is freed on return."""
    import torch

    from protein_folding_attention_gb300 import evoattn, synthetic
    torch.cuda.synchronize(dev)
    base = torch.cuda.memory_allocated(dev)
    x = synthetic.make_inputs(w, device=dev)
    # the input generator's own temporaries (e.g. the fp32 draw behind a
    # Bernoulli mask) are not part of the call: count from here
    torch.cuda.synchronize(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    B, S, H, N, D = w.B, w.S, w.H, w.N, w.D
    out = synthetic.empty_view(w, dev)
    lse = torch.empty(B, S, H, N, device=dev, dtype=torch.float32)
    g = {n: synthetic.empty_view(w, dev) for n in ("dq", "dk", "dv")}
    g["dgate"] = synthetic.empty_view(w, dev) if w.gate else None
    dbias = torch.empty(B, H, N, N, device=dev, dtype=torch.float32)
    wsp = torch.empty(evoattn.workspace_size(B, S, H, N, D, w.torch_dtype), device=dev,
                      dtype=torch.uint8)

    def fwd():
        evoattn.fwd(x["q"], x["k"], x["v"], x["bias"], x["mask"], x["gate"], out=out, lse=lse)

    def bwd(ev=None):
        evoattn.bwd(x["q"], x["k"], x["v"], x["bias"], x["mask"], x["gate"], out, lse,
                    x["dout"], dq=g["dq"], dk=g["dk"], dv=g["dv"], dbias=dbias,
                    dgate=g["dgate"], workspace=wsp, stage_events=ev)

    for _ in range(warmup):
        fwd()
        bwd()
    ef = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    eb = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
    for i in range(steps):
        ef[i][0].record()
        fwd()
        ef[i][1].record()
        bwd(eb[i])
    torch.cuda.synchronize(dev)
    if evoattn.device_status() != evoattn.OK:
        raise RuntimeError(f"device status set on {w.name}")
    t_f = statistics.median(a.elapsed_time(b) for a, b in ef) * 1e-3
    t_b = statistics.median(e[0].elapsed_time(e[4]) for e in eb) * 1e-3
    held = int(torch.cuda.max_memory_allocated(dev) - base)
    res = {"fwd_ms": t_f * 1e3, "fwd_tflops": w.fwd_flops / t_f / 1e12,
           "fwd_frac_of_peak": w.fwd_flops / t_f / 1e12 / peak,
           "bwd_ms": t_b * 1e3, "bwd_tflops": w.bwd_flops / t_b / 1e12,
           "bwd_frac_of_peak": w.bwd_flops / t_b / 1e12 / peak,
           "L": w.B * w.S * w.H * w.N * w.D, "BHN2": w.B * w.H * w.N * w.N,
           "device_bytes": held,
           "formula_bytes": held_bytes(B, S, H, N, D, gate=w.gate, mask=w.mask != "none"),
           "bwd_workspace_bytes": int(wsp.numel()),
           "logits_bytes_if_materialized_bf16": int(w.logits * 2)}
    fb, bb = algorithmic_bytes(w)
    res["fwd_hbm_bytes"], res["bwd_hbm_bytes"] = fb, bb
    res["fwd_hbm_gbs"], res["bwd_hbm_gbs"] = fb / t_f / 1e9, bb / t_b / 1e9
    if hbm_peak:
        res["fwd_hbm_frac"] = fb / t_f / 1e9 / hbm_peak
        res["bwd_hbm_frac"] = bb / t_b / 1e9 / hbm_peak
    res["fwd_logits_per_s"], res["bwd_logits_per_s"] = w.logits / t_f, w.logits / t_b
    if ex2_peak:
        res["fwd_ex2_frac"] = w.logits / t_f / ex2_peak
    del x, out, lse, g, dbias, wsp
    torch.cuda.synchronize(dev)
    return res


def measure_ln_proj(N, dev, peaks, steps=10, warmup=3, B=1, C=128, H=4, D=32):
    """The EvoFusion upstream stack (LayerNorm + q/k/v/g/pair-bias projection)
    on the [B, N, N, C] pair representation: CUDA-event time, algorithmic HBM
    bytes (z read, weights read, five outputs written) against the measured
    copy bandwidth, and the projection's TFLOP/s."""
    import torch

    from protein_folding_attention_gb300 import evoattn, synthetic
    x = synthetic.make_fusion_inputs(B, N, C, H, D, seed=N, device=dev)
    out = evoattn.ln_proj(x["z"], x["gamma"], x["beta"], x["w"], H, D)
    for _ in range(warmup):
        evoattn.ln_proj(x["z"], x["gamma"], x["beta"], x["w"], H, D, out=out)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for a, b in ev:
        a.record()
        evoattn.ln_proj(x["z"], x["gamma"], x["beta"], x["w"], H, D, out=out)
        b.record()
    torch.cuda.synchronize(dev)
    if evoattn.device_status() != evoattn.OK:
        raise RuntimeError("device status set by evoattn_ln_proj")
    t = statistics.median(a.elapsed_time(b) for a, b in ev) * 1e-3
    rows = B * N * N
    nout = 4 * H * D + H
    bytes_ = rows * C * 2 + nout * C * 2 + rows * nout * 2
    flops = 2 * rows * C * nout
    gbs = bytes_ / t / 1e9
    return {"workload": f"pair_ln_proj_n{N}", "B": B, "N": N, "C": C, "H": H, "D": D,
            "ms": t * 1e3, "hbm_bytes": bytes_, "hbm_gbs": gbs,
            "frac_of_hbm_peak": gbs / peaks["hbm_gbs"], "tflops": flops / t / 1e12,
            "traffic": profiled_traffic("evoattn_ln_proj_kernel", f"pair_ln_proj_n{N}"),
            "normalised_tensor_bytes_not_written": rows * C * 2}


def measure_transition(N, dev, peaks, steps=10, warmup=3, B=1, C=128, F=512, HD=0):
    """The EvoFusion downstream stack (the SwiGLU transition with its residual
    add) on the [B, N, N, C] pair representation: CUDA-event time, TFLOP/s of
    the two projections against the measured bf16 peak, and the HBM rate of
    its algorithmic bytes (z read, out written; the 384 KB of weights come
    from L2)."""
    import torch

    from protein_folding_attention_gb300 import evoattn, synthetic
    x = synthetic.make_transition_inputs(B, N, C, F, seed=N, device=dev, HD=HD)
    run = lambda out=None: evoattn.transition(x["z"], x["gamma"], x["beta"], x["w1"], x["w2"],
                                              o=x["o"], w_o=x["w_o"], out=out)
    out = run()
    for _ in range(warmup):
        run(out)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for a, b in ev:
        a.record()
        run(out)
        b.record()
    torch.cuda.synchronize(dev)
    if evoattn.device_status() != evoattn.OK:
        raise RuntimeError("device status set by evoattn_transition")
    t = statistics.median(a.elapsed_time(b) for a, b in ev) * 1e-3
    rows = B * N * N
    flops = 6 * rows * C * F + 2 * rows * C * HD
    bytes_ = 2 * rows * C * 2 + rows * HD * 2 + (3 * F + HD) * C * 2
    name = f"pair_outproj_transition_n{N}" if HD else f"pair_transition_n{N}"
    return {"workload": name, "B": B, "N": N, "C": C, "F": F, "HD": HD,
            "ms": t * 1e3, "tflops": flops / t / 1e12,
            "frac_of_bf16_peak": flops / t / 1e12 / peaks["bf16_tflops"],
            "hbm_bytes": bytes_, "hbm_gbs": bytes_ / t / 1e9,
            "traffic": profiled_traffic("evoattn_transition_kernel", name),
            "intermediate_bytes_not_written": rows * ((2 if HD else 1) * C + 3 * F) * 2}


def held_bytes(B, S, H, N, D, gate=True, mask=True, flags=0):
    """Device bytes a caller holds for one bf16 forward + backward: q, k, v,
    dout (+ gate) and out, dq, dk, dv (+ dgate) [B,S,H,N,D]; the pair bias
    (bf16) and dbias (fp32) [B,H,N,N]; the mask [B,S,N] (uint8); lse [B,S,H,N]
    (fp32); the backward workspace the library asks for.  The library itself
    allocates nothing."""
    from protein_folding_attention_gb300 import evoattn
    L, R, n2 = B * S * H * N * D, B * S * H * N, B * H * N * N
    per_row_tensors = 4 + int(gate)
    return (2 * per_row_tensors * L * 2 + n2 * 2 + n2 * 4 + (B * S * N if mask else 0) + R * 4
            + evoattn.workspace_size(B, S, H, N, D, flags=flags))


def dbias_slot_elems(B, S, H, N):
    """Elements of the dbias slot partials in the backward workspace: the
    slot count is about 4 * 152 / (B * H * tiles^2), at most S, so this term
    stays below ~(608 + B*H*tiles^2) * 128^2 elements whatever S."""
    nt = (N + 127) // 128
    slots = min(S, max(1, -(-4 * 152 // (B * H * nt * nt))))
    return slots * B * H * N * N


def memory_fit(points):
    """Least-squares fit of held bytes = a*L + r*R + b*BHN2 + c*BSN + p*P + d*X
    + e over {"L", "R", "BHN2", "BSN", "P", "X", "device_bytes"} points
    (L = B*S*H*N*D, R = B*S*H*N rows, BHN2 = B*H*N*N, BSN = B*S*N, P = the
    dbias slot-partial elements, X = B*S*H*N*N the logits).  A footprint linear in the inputs gives d = 0
    and a zero residual.  Columns are scaled to unit norm before the solve."""
    import numpy as np
    A = np.array([[p["L"], p["R"], p["BHN2"], p["BSN"], p["P"], p["X"], 1.0] for p in points],
                 dtype=np.float64)
    y = np.array([p["device_bytes"] for p in points], dtype=np.float64)
    scale = np.linalg.norm(A, axis=0)
    coef, *_ = np.linalg.lstsq(A / scale, y, rcond=None)
    coef = coef / scale
    resid = A @ coef - y
    return {"bytes_per_L": float(coef[0]), "bytes_per_row": float(coef[1]),
            "bytes_per_BHN2": float(coef[2]), "bytes_per_BSN": float(coef[3]),
            "bytes_per_slot_partial": float(coef[4]), "bytes_per_logit": float(coef[5]),
            "const_bytes": float(coef[6]),
            "max_rel_residual": float(np.max(np.abs(resid) / y)),
            "points": len(points)}


def memory_model(B=1):
    """held_bytes over a grid of S, N (S = N and S != N, N off and on the
    128-key tile size), H and D, and its fit: the linear footprint of the
    library (bytes per L, per B*H*N^2, per mask byte, per dbias slot-partial
    element) and the coefficient of the logits count, which must be zero."""
    pts = []
    for S in (16, 64, 256, 768, 1536):
        for N in (64, 200, 384, 768, 1536):
            for H, D in ((4, 32), (1, 16), (2, 32)):
                pts.append({"L": B * S * H * N * D, "R": B * S * H * N,
                            "BHN2": B * H * N * N, "BSN": B * S * N,
                            "P": dbias_slot_elems(B, S, H, N), "X": B * S * H * N * N,
                            "device_bytes": held_bytes(B, S, H, N, D)})
    return memory_fit(pts)


def oracle_sample_time(w, n_rows, device_inputs=None):
    """Time the float64 oracle (fwd + bwd) on n_rows of the workload's s rows.
    Returns (seconds, flops_of_sample, threads)."""
    import torch

    import oracle
    from protein_folding_attention_gb300 import synthetic
    x = device_inputs if device_inputs is not None else synthetic.make_inputs(
        synthetic.Workload(w.name + "_sample", B=w.B, S=n_rows, N=w.N, H=w.H, D=w.D,
                           dtype=w.dtype, node=w.node, mask=w.mask, mask_tail=w.mask_tail,
                           mask_p=w.mask_p, gate=w.gate, bias_std=w.bias_std, seed=w.seed))
    sub = {k: (None if v is None else (v.cpu() if k == "bias" else v[:, :n_rows].cpu()))
           for k, v in x.items()}
    oracle.build()
    t0 = time.perf_counter()
    oracle.fwd(sub["q"], sub["k"], sub["v"], sub["bias"], sub["mask"], sub["gate"])
    oracle.bwd(sub["q"], sub["k"], sub["v"], sub["bias"], sub["mask"], sub["gate"], sub["dout"])
    dt = time.perf_counter() - t0
    flops = 14 * w.B * n_rows * w.H * w.N * w.N * w.D
    del torch
    return dt, flops, oracle.num_threads()


def run_reference(args, w):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    rows = args.ref_rows
    times = []
    flops = threads = 0
    if args.warmup > 0:          # one untimed sample builds the oracle and warms caches
        oracle_sample_time(w, rows)
    for _ in range(args.steps):
        dt, flops, threads = oracle_sample_time(w, rows)
        times.append(dt)
    t = statistics.mean(times)
    value = flops / t / 1e12
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_block(w), "impl": "reference",
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads,
                             "kind": "oracle",
                             "sample": f"{rows} of {w.S} s rows (fwd+bwd incl. dbias over them), "
                                       f"full N={w.N}, H={w.H}, D={w.D}"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, w):
    import torch

    from protein_folding_attention_gb300 import evoattn, synthetic

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    evoattn.load()
    peaks, peak_src = load_peaks()

    x = synthetic.make_inputs(w, device=dev)
    B, S, H, N, D = w.B, w.S, w.H, w.N, w.D
    out = synthetic.empty_view(w, dev)
    lse = torch.empty(B, S, H, N, device=dev, dtype=torch.float32)
    grads = {n: synthetic.empty_view(w, dev) for n in ("dq", "dk", "dv", "dgate")}
    dbias = torch.empty(B, H, N, N, device=dev, dtype=torch.float32)
    wsp = torch.empty(evoattn.workspace_size(B, S, H, N, D, w.torch_dtype), device=dev,
                      dtype=torch.uint8)
    stream = torch.cuda.current_stream(dev)

    def fwd():
        evoattn.fwd(x["q"], x["k"], x["v"], x["bias"], x["mask"], x["gate"], out=out, lse=lse)

    def bwd(events=None, flags=evoattn.DBIAS_DETERMINISTIC, workspace=None):
        evoattn.bwd(x["q"], x["k"], x["v"], x["bias"], x["mask"], x["gate"], out, lse,
                    x["dout"], flags=flags, dq=grads["dq"], dk=grads["dk"], dv=grads["dv"],
                    dbias=dbias, dgate=grads["dgate"],
                    workspace=wsp if workspace is None else workspace, stage_events=events)

    def barrier():
        if pg is not None:
            pg.barrier()
        torch.cuda.synchronize(dev)

    mem0 = torch.cuda.memory_allocated(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    for _ in range(args.warmup):
        fwd()
        bwd()
    barrier()
    status = evoattn.device_status()
    if status != evoattn.OK:
        raise RuntimeError(f"device status {status} after warm-up")
    # The library allocates nothing: everything on the device is the caller's
    # inputs, outputs and the backward workspace (linear in B*S*H*N*D plus
    # O(B*H*N^2)); the logits are never stored.
    memory = {"device_bytes_in_use": int(torch.cuda.max_memory_allocated(dev)),
              "growth_during_steps_bytes": int(torch.cuda.max_memory_allocated(dev) - mem0),
              "bwd_workspace_bytes": int(wsp.numel()),
              "logits_bytes_if_materialized_bf16": int(w.logits * 2)}

    # ---- timed region: K steps, per-kernel events on the launching stream ----
    n_ev = 5
    ev_f = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(args.steps)]
    ev_b = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
            for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        barrier()
        t0.record(stream)
        for i in range(args.steps):
            ev_f[i][0].record(stream)
            fwd()
            ev_f[i][1].record(stream)
            bwd(ev_b[i])
        t1.record(stream)
        barrier()
    elapsed = max_over_ranks(t0.elapsed_time(t1) * 1e-3, pg, dev)
    status = evoattn.device_status()
    if status != evoattn.OK:
        raise RuntimeError(f"device status {status} in timed region")

    t_fwd = statistics.mean(a.elapsed_time(b) for a, b in ev_f) * 1e-3
    stage = [statistics.mean(e[k].elapsed_time(e[k + 1]) for e in ev_b) * 1e-3
             for k in range(n_ev - 1)]
    t_bwd = sum(stage)
    step = elapsed / args.steps
    total_flops = (w.fwd_flops + w.bwd_flops) * ws
    value = job_tflops(w.fwd_flops + w.bwd_flops, ws, step)
    peak = peaks["bf16_tflops"]
    peak_sus = peaks.get("bf16_tflops_sustained", peak)

    # ---- dbias: the atomic variant timed beside the deterministic one --------
    # (same workspace: the deterministic one needs the larger)
    ev_a = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
            for _ in range(max(3, args.steps // 2))]
    for _ in range(2):
        bwd(None, evoattn.DBIAS_ATOMIC)
    for e in ev_a:
        bwd(e, evoattn.DBIAS_ATOMIC)
    barrier()
    stage_a = [statistics.mean(e[k].elapsed_time(e[k + 1]) for e in ev_a) * 1e-3
               for k in range(n_ev - 1)]
    # and the fused mode: dbias summed with atomics inside the dK/dV pass
    ev_z = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
            for _ in range(max(3, args.steps // 2))]
    for _ in range(2):
        bwd(None, evoattn.DBIAS_FUSED)
    for e in ev_z:
        bwd(e, evoattn.DBIAS_FUSED)
    barrier()
    stage_z = [statistics.mean(e[k].elapsed_time(e[k + 1]) for e in ev_z) * 1e-3
               for k in range(n_ev - 1)]
    # HBM bytes of the deterministic reduce stage: slot partials read + dbias
    # written (k_dbias_sum), fp32 dQ read + bf16 dq written (k_dq_convert)
    nt = (w.N + 127) // 128
    slots = min(w.S, max(1, -(-4 * 152 // (w.B * w.H * nt * nt))))
    n2 = w.B * w.H * w.N * w.N
    lin = w.B * w.S * w.H * w.N * w.D
    reduce_bytes = (slots + 1) * n2 * 4 + lin * 4 + lin * 2
    dbias_variants = {
        "deterministic": {"dbias_ms": stage[2] * 1e3, "reduce_ms": stage[3] * 1e3,
                          "bwd_ms": sum(stage) * 1e3, "slots": slots,
                          "reduce_hbm_gbs": reduce_bytes / stage[3] / 1e9},
        "atomic": {"dbias_ms": stage_a[2] * 1e3, "reduce_ms": stage_a[3] * 1e3,
                   "bwd_ms": sum(stage_a) * 1e3},
        "fused": {"dkdv_with_dbias_ms": stage_z[1] * 1e3, "reduce_ms": stage_z[3] * 1e3,
                  "bwd_ms": sum(stage_z) * 1e3},
    }

    # ---- dQ: the deterministic mode (per-key-tile slices, ordered sum) timed
    # beside the default atomic accumulation; its larger workspace is
    # allocated here, outside the measured steps
    wsp_det = torch.empty(evoattn.workspace_size(B, S, H, N, D, w.torch_dtype,
                                                 flags=evoattn.DQ_DETERMINISTIC),
                          device=dev, dtype=torch.uint8)
    ev_d = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
            for _ in range(max(3, args.steps // 2))]
    for _ in range(2):
        bwd(None, evoattn.DQ_DETERMINISTIC, wsp_det)
    for e in ev_d:
        bwd(e, evoattn.DQ_DETERMINISTIC, wsp_det)
    barrier()
    stage_d = [statistics.mean(e[k].elapsed_time(e[k + 1]) for e in ev_d) * 1e-3
               for k in range(n_ev - 1)]
    dq_modes = {
        "atomic": {"dkdv_ms": stage[1] * 1e3, "reduce_ms": stage[3] * 1e3,
                   "bwd_ms": sum(stage) * 1e3, "workspace_bytes": int(wsp.numel())},
        "deterministic": {"dkdv_ms": stage_d[1] * 1e3, "reduce_ms": stage_d[3] * 1e3,
                          "bwd_ms": sum(stage_d) * 1e3,
                          "workspace_bytes": int(wsp_det.numel())},
    }
    del wsp_det
    if evoattn.device_status() != evoattn.OK:
        raise RuntimeError("device status after the dQ-mode timing")

    # ---- exponential unit: the forward, dK/dV and dbias kernels each
    # evaluate exactly one ex2 per logit; peak = EX2_PER_CLK_PER_SM x SMs x
    # the maximum SM clock
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    sm_mhz = float(peaks.get("sm_max_mhz", 2070.0))
    ex2_peak = EX2_PER_CLK_PER_SM * n_sm * sm_mhz * 1e6
    sfu = {"ex2_per_clk_per_sm": EX2_PER_CLK_PER_SM, "sms": n_sm, "sm_mhz": sm_mhz,
           "peak_ex2_per_s": ex2_peak, "logits": w.logits}
    for name, t in (("evoattn_fwd_kernel", t_fwd), ("k_dkdv", stage[1]), ("k_dbias", stage[2])):
        sfu[name] = {"logits_per_s": w.logits / t, "frac": w.logits / t / ex2_peak}

    # ---- end to end: pinned host inputs -> device, fwd+bwd, results -> host
    e2e = None
    if not args.no_e2e:
        host_in = {k: (None if v is None else torch.empty_strided(
            v.size(), v.stride(), dtype=v.dtype, pin_memory=True).copy_(v))
            for k, v in x.items()}
        outs = {"out": out, "dbias": dbias, **grads}
        host_out = {k: torch.empty_strided(v.size(), v.stride(), dtype=v.dtype,
                                           pin_memory=True) for k, v in outs.items()}
        h2d = sum(v.numel() * v.element_size() for v in host_in.values() if v is not None)
        d2h = sum(v.numel() * v.element_size() for v in host_out.values())

        # Steps are pipelined the way a training loop prefetches its next
        # batch: two sets of device inputs and outputs alternate, so step
        # i+1's inputs go up (stream `up`) while step i computes, and step
        # i's results come down (stream `dn`) as soon as the kernel that
        # writes each of them has finished (the forward's end and the
        # backward's stage events).  Every step still uploads all of its
        # inputs and downloads all of its results inside the timed region.
        def make_set():
            xs = {k: (None if v is None else torch.empty_strided(
                v.size(), v.stride(), dtype=v.dtype, device=dev)) for k, v in x.items()}
            ys = {"out": synthetic.empty_view(w, dev),
                  "lse": torch.empty(B, S, H, N, device=dev, dtype=torch.float32),
                  "dbias": torch.empty(B, H, N, N, device=dev, dtype=torch.float32)}
            for n in ("dq", "dk", "dv", "dgate"):
                ys[n] = synthetic.empty_view(w, dev) if grads.get(n) is not None else None
            return xs, ys

        sets = [make_set(), make_set()]
        up, dn = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        e_up = [torch.cuda.Event() for _ in range(2)]
        e_done = [torch.cuda.Event() for _ in range(2)]
        e_dl = [torch.cuda.Event() for _ in range(2)]
        e_f = [torch.cuda.Event() for _ in range(2)]
        bevs = [[torch.cuda.Event() for _ in range(5)] for _ in range(2)]
        used = [False, False]

        def e2e_step(i):
            sb = i % 2
            xs, ys = sets[sb]
            with torch.cuda.stream(up):
                if used[sb]:
                    up.wait_event(e_done[sb])  # step i-2 no longer reads these inputs
                for k, v in host_in.items():
                    if v is not None:
                        xs[k].copy_(v, non_blocking=True)
                e_up[sb].record(up)
            stream.wait_event(e_up[sb])
            if used[sb]:
                stream.wait_event(e_dl[sb])  # step i-2's results have left these buffers
            evoattn.fwd(xs["q"], xs["k"], xs["v"], xs["bias"], xs["mask"], xs["gate"],
                        out=ys["out"], lse=ys["lse"])
            e_f[sb].record(stream)
            ev = bevs[sb]
            evoattn.bwd(xs["q"], xs["k"], xs["v"], xs["bias"], xs["mask"], xs["gate"],
                        ys["out"], ys["lse"], xs["dout"], dq=ys["dq"], dk=ys["dk"],
                        dv=ys["dv"], dbias=ys["dbias"], dgate=ys["dgate"], workspace=wsp,
                        stage_events=ev)
            e_done[sb].record(stream)
            with torch.cuda.stream(dn):
                dn.wait_event(e_f[sb])
                host_out["out"].copy_(ys["out"], non_blocking=True)
                if "dgate" in host_out:
                    dn.wait_event(ev[1])  # after k_pre
                    host_out["dgate"].copy_(ys["dgate"], non_blocking=True)
                dn.wait_event(ev[2])  # after k_dkdv
                host_out["dk"].copy_(ys["dk"], non_blocking=True)
                host_out["dv"].copy_(ys["dv"], non_blocking=True)
                dn.wait_event(e_done[sb])
                host_out["dq"].copy_(ys["dq"], non_blocking=True)
                host_out["dbias"].copy_(ys["dbias"], non_blocking=True)
                e_dl[sb].record(dn)
            used[sb] = True

        for i in range(2):
            e2e_step(i)
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ksteps = max(4, args.steps // 2)
        barrier()
        e0.record(stream)
        up.wait_event(e0)
        dn.wait_event(e0)
        for i in range(ksteps):
            e2e_step(i)
        stream.wait_stream(up)
        stream.wait_stream(dn)
        e1.record(stream)
        barrier()
        if evoattn.device_status() != evoattn.OK:
            raise RuntimeError("device status set during the end-to-end steps")
        # the results that came down are the ones the device-resident steps
        # computed from the same inputs (bit for bit: out, dk, dv, dgate)
        for k in ("out", "dk", "dv", "dgate"):
            if k in host_out and not torch.equal(host_out[k], outs[k].cpu()):
                raise RuntimeError(f"end-to-end {k} differs from the device-resident result")
        te = max_over_ranks(e0.elapsed_time(e1) * 1e-3 / ksteps, pg, dev)
        e2e = {"value": total_flops / te / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": te * 1e3}

    # ---- roofline of the dominant kernel --------------------------------------
    kernels = {
        "evoattn_fwd_kernel": (t_fwd, w.fwd_flops),
        "k_pre": (stage[0], 0),
        "k_dkdv": (stage[1], w.bwd_flops),
        "k_dbias": (stage[2], 0),
        "k_dbias_sum+k_dq_convert": (stage[3], 0),
    }
    dom = max(kernels, key=lambda k: kernels[k][0])
    dt_dom, fl_dom = kernels[dom]
    traffic = profiled_traffic(dom, w.name)
    if fl_dom > 0:
        achieved = fl_dom / dt_dom / 1e12
        roof = {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_source": f"{peak_src} bf16 burst", "traffic": traffic}
    else:
        roof = {"kernel": dom, "bound": "alu", "achieved": None, "peak": None,
                "unit": None, "frac": None, "traffic": traffic}

    # ---- every synthetic configuration: fwd / bwd times and held memory ----
    per_config = None
    if rank == 0 and not args.no_per_config:
        per_config = {}
        n_sm_cfg = torch.cuda.get_device_properties(dev).multi_processor_count
        ex2_cfg = EX2_PER_CLK_PER_SM * n_sm_cfg * float(peaks.get("sm_max_mhz", 2070.0)) * 1e6
        for name in PER_CONFIG:
            per_config[name] = measure_config(synthetic.WORKLOADS[name], dev, peak,
                                              hbm_peak=peaks["hbm_gbs"], ex2_peak=ex2_cfg)
        per_config["memory_fit"] = memory_model()
    evofusion = None
    if rank == 0 and not args.no_per_config:
        evofusion = {f"n{n}": measure_ln_proj(n, dev, peaks) for n in (384, 768)}
        evofusion.update({f"transition_n{n}": measure_transition(n, dev, peaks)
                          for n in (384, 768)})
        evofusion.update({f"outproj_transition_n{n}": measure_transition(n, dev, peaks, HD=128)
                          for n in (384, 768)})

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu:
        dt, fl, thr = oracle_sample_time(w, args.cpu_rows)
        cpu = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
               "sample": f"{args.cpu_rows} of {w.S} s rows (fwd+bwd incl. dbias over them), "
                         f"full N={w.N}, H={w.H}, D={w.D}; {dt:.1f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": config_block(w),
            "fwd": {"ms": t_fwd * 1e3, "tflops": w.fwd_flops / t_fwd / 1e12,
                    "frac_of_peak": w.fwd_flops / t_fwd / 1e12 / peak,
                    "frac_of_sustained_peak": w.fwd_flops / t_fwd / 1e12 / peak_sus},
            "bwd": {"ms": t_bwd * 1e3, "tflops": w.bwd_flops / t_bwd / 1e12,
                    "frac_of_peak": w.bwd_flops / t_bwd / 1e12 / peak,
                    "frac_of_sustained_peak": w.bwd_flops / t_bwd / 1e12 / peak_sus,
                    "stages_ms": dict(zip(["pre", "dkdv", "dbias", "reduce"],
                                          [s * 1e3 for s in stage]))},
            "peak_tflops": peak, "peak_source": peak_src,
            "frac_of_peak": value / ws / peak,
            "sustained_peak_tflops": peak_sus,
            "frac_of_sustained_peak": value / ws / peak_sus,
            "memory": memory,
            "dbias_variants": dbias_variants,
            "dq_modes": dq_modes,
            "roofline": roof, "sfu": sfu, "cpu_baseline": cpu, "e2e": e2e,
            "per_config": per_config, "evofusion": evofusion,
            "clocks": clocks.summary(),
            "gpu_launches": args.steps * 6,
        }
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()
    return 0


def profiled_traffic(kernel, workload):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if one
    exists for this kernel and workload (profiles/traffic.txt lines:
    kernel workload bytes_per_launch)."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        for line in open(p):
            f = line.split()
            if len(f) >= 3 and f[0] == kernel and f[1] == workload:
                return float(f[2])
    except OSError:
        pass
    return None


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--ref-rows", type=int, default=16,
                    help="s rows per step of the --impl reference arm")
    ap.add_argument("--cpu-rows", type=int, default=192,
                    help="s rows of the cpu_baseline sample")
    ap.add_argument("--s-rows", type=int, default=0,
                    help="profiling only: truncate the workload to this many s rows")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-per-config", action="store_true")
    ap.add_argument("--evofusion-only", type=int, default=0, metavar="N",
                    help="profiling only: time the LayerNorm + projection kernel on the "
                         "[1, N, N, 128] pair representation and print its JSON")
    ap.add_argument("--transition-only", type=int, default=0, metavar="N",
                    help="profiling only: time the fused SwiGLU transition kernel on the "
                         "[1, N, N, 128] pair representation and print its JSON")
    args = ap.parse_args()
    if args.transition_only:
        import torch
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        peaks, _ = load_peaks()
        print(json.dumps(measure_transition(args.transition_only, dev, peaks)))
        print(json.dumps(measure_transition(args.transition_only, dev, peaks, HD=128)))
        return 0
    if args.evofusion_only:
        import torch
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        peaks, _ = load_peaks()
        print(json.dumps(measure_ln_proj(args.evofusion_only, dev, peaks)))
        return 0
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be at least 3")
    from protein_folding_attention_gb300 import synthetic
    w = synthetic.WORKLOADS[args.workload]
    if args.s_rows:
        import dataclasses
        w = dataclasses.replace(w, name=f"{w.name}_s{args.s_rows}", S=args.s_rows)
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
