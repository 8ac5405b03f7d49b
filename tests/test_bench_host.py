"""Host-side logic of bench.py without a GPU: clock-sample parsing, the
committed traffic table, the whole-job aggregation over ranks (world size 2
on gloo), and the JSON line of the --impl reference arm on the tiny workload."""
import json
import os
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_clock_summary_parses_nvidia_smi_lines():
    c = bench.ClockSampler(0)
    c.lines = ["0, 1950, 2070, 1200.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
               "0, 2070, 2070, 1300.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
               "0, 345, 2070, 300.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active"]
    s = c.summary()
    assert s["sm_max_mhz"] == 2070.0
    assert s["sm_mhz"] == pytest.approx(2010.0)   # median of the loaded samples
    assert s["reasons"] == ["sw_power_cap"]


def test_traffic_table_lookup():
    assert bench.profiled_traffic("k_dkdv", "pairformer_end_n768") > 1e8
    assert bench.profiled_traffic("k_dkdv", "no_such_workload") is None


def _ranks(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t = bench.max_over_ranks(1.0 + rank, dist)        # rank 1 is the slowest
    q.put((rank, t, bench.job_tflops(2e12, world, t)))
    dist.destroy_process_group()


def test_job_time_is_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_ranks, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    out = sorted(q.get() for _ in range(2))
    assert [t for _, t, _ in out] == [2.0, 2.0]
    assert out[0][2] == pytest.approx(2e12 * 2 / 2.0 / 1e12)


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_start_n32_fp32", "--steps", "1", "--warmup", "0",
                        "--ref-rows", "4"], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_memory_fit_recovers_a_linear_footprint():
    """The fit of held device bytes returns the coefficients of a footprint
    that is linear in its inputs and a zero residual; a term in the logits
    count X = B*S*H*N^2 shows up as its own coefficient."""
    pts = []
    for B, S, H, N, D in ((1, 8, 2, 64, 32), (1, 64, 4, 200, 16), (2, 16, 1, 384, 32),
                          (1, 300, 4, 96, 32), (1, 5, 2, 768, 16), (3, 40, 2, 128, 32),
                          (1, 1, 8, 1000, 16), (1, 77, 3, 333, 32)):
        p = {"L": B * S * H * N * D, "R": B * S * H * N, "BHN2": B * H * N * N,
             "BSN": B * S * N, "P": bench.dbias_slot_elems(B, S, H, N),
             "X": B * S * H * N * N}
        p["device_bytes"] = (26 * p["L"] + 8 * p["R"] + 6 * p["BHN2"] + p["BSN"]
                             + 4 * p["P"] + 1000)
        pts.append(p)
    f = bench.memory_fit(pts)
    assert f["bytes_per_L"] == pytest.approx(26.0)
    assert f["bytes_per_BHN2"] == pytest.approx(6.0)
    assert abs(f["bytes_per_logit"]) < 1e-9
    assert f["max_rel_residual"] < 1e-9
    cubic = [dict(p, device_bytes=p["device_bytes"] + 2 * p["X"]) for p in pts]
    assert bench.memory_fit(cubic)["bytes_per_logit"] == pytest.approx(2.0)


def test_library_footprint_has_no_logit_term():
    """What a caller holds for one forward + backward (inputs, outputs and the
    workspace the library asks for; the library allocates nothing), over a
    grid of S, N, H and D: exactly 26 bytes per element of q (ten bf16
    tensors, the bf16 gated output gradient, the fp32 dQ accumulator), 8 per
    query row (lse, delta), 6 per pair-bias entry (bf16 bias, fp32 dbias), 1
    per mask byte and 4 per dbias slot-partial element, and nothing per
    logit."""
    f = bench.memory_model()
    assert f["max_rel_residual"] < 1e-9
    assert f["bytes_per_L"] == pytest.approx(26.0)
    assert f["bytes_per_row"] == pytest.approx(8.0)
    assert f["bytes_per_BHN2"] == pytest.approx(6.0)
    assert f["bytes_per_BSN"] == pytest.approx(1.0)
    assert f["bytes_per_slot_partial"] == pytest.approx(4.0)
    assert abs(f["bytes_per_logit"]) < 1e-9


def test_algorithmic_bytes_of_the_workloads():
    """The HBM bytes each pass must move (logits never counted), per workload,
    in MB: forward and backward of the four bf16 configurations."""
    from protein_folding_attention_gb300 import synthetic
    expect = {"pairformer_start_n384": (192.4, 388.3), "pairformer_end_n768": (769.7, 1553.0),
              "msa_row_s512_n384": (512.2, 1032.8), "long_start_n1536": (3078.9, 6212.0)}
    for name, (f, b) in expect.items():
        fb, bb = bench.algorithmic_bytes(synthetic.WORKLOADS[name])
        assert fb / 1e6 == pytest.approx(f, abs=0.1) and bb / 1e6 == pytest.approx(b, abs=0.1)
