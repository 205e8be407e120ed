"""Host-side logic of bench.py on the CPU: algorithmic work counts, roofline
arithmetic, the JSON line, the reference (oracle) arm, and the max-over-ranks
reduction with two gloo ranks."""
import json
import os
import socket
import subprocess
import sys

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_work_counts_mamba130m():
    w = bench.work_counts(2, 2048, 1536, 16, 4)
    assert w["elems"] == 6_291_456
    assert w["bytes"] == 76_120_064          # x, delta, y + B, C + A
    assert w["mufu"] == 6_291_456 * 16 + 2 * 6_291_456
    assert w["fp32"] == 4 * 6_291_456 * 16


def test_work_counts_bf16_and_state():
    w = bench.work_counts(8, 2048, 2048, 16, 2)
    assert w["bytes"] == 202_506_240
    w4 = bench.work_counts(1, 131072, 1536, 16, 4, hT=True)
    assert w4["bytes"] == 2_432_892_928          # includes the final state hT


def test_decode_step_work_counts():
    w = bench.step_work_counts(256, 2560, 16)
    assert w["bytes"] == 91_947_008          # state read + write dominates (83.9 MB)
    assert w["elems"] == 655_360


def test_reference_arm_decode_workload():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "5", "--steps", "2", "--warmup", "1", "--ref-chains", "4"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0


def test_roofline_arithmetic():
    """frac is against the benchmark statement's bound, max(t_HBM, t_MUFU + t_FP32);
    frac_strict against max(t_HBM, t_MUFU, t_FP32)."""
    pk = bench.peaks(148, 2032.0, 6484.3)
    assert pk["mufu_per_s"] == pytest.approx(148 * 32 * 2.032e9)
    w = bench.work_counts(2, 2048, 1536, 16, 4)
    t_mufu = w["mufu"] / pk["mufu_per_s"]
    t_fp32 = w["fp32"] / pk["fp32_per_s"]
    t = 2 * (t_mufu + t_fp32)
    r = bench.roofline(w, pk, seconds=t)
    assert r["bound"] == "alu"
    assert r["frac"] == pytest.approx(0.5)
    assert r["frac_strict"] == pytest.approx(max(t_mufu, t_fp32) / t)
    assert r["frac_strict"] < r["frac"]
    assert r["achieved"] == pytest.approx(w["updates"] / t / 1e12)
    assert r["peak"] * r["frac"] == pytest.approx(r["achieved"])


def test_measured_alu_peaks_replace_the_derived_ones():
    alu = {"ex2_per_s": 8.0e12, "fp32_per_s": 30.0e12, "ffma_per_s": 30.0e12, "ffma2_per_s": 29.0e12}
    pk = bench.peaks(148, 2032.0, 6484.3, alu)
    assert pk["mufu_per_s"] == 8.0e12 and pk["fp32_per_s"] == 30.0e12
    assert "measured" in bench.peak_source("measured", alu, 148, 2032.0)
    assert "derived" in bench.peak_source("measured", None, 148, 2032.0)


def test_roofline_hbm_bound_in_bytes():
    """An HBM-bound call (the decode step) reports bytes per second against the
    measured copy bandwidth; frac is the same ratio either way."""
    pk = bench.peaks(148, 2032.0, 6484.3)
    w = bench.step_work_counts(256, 2560, 16)
    assert w["bytes"] == 2 * 256 * 2560 * 16 * 4 + 3 * 256 * 2560 * 4 + 2 * 256 * 16 * 4 + 2560 * 16 * 4
    t = 2 * w["bytes"] / pk["hbm_bytes_per_s"]
    r = bench.roofline(w, pk, seconds=t)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["peak"] == pytest.approx(6484.3)
    assert r["frac"] == pytest.approx(0.5)
    assert r["achieved"] == pytest.approx(0.5 * 6484.3)


def test_result_line_has_contract_keys():
    line = bench.result_line(value=1.0, n_gpus=1, steps=3, warmup=3, ms_per_step=1.0,
                             config={"workload": "w"}, roof={}, cpu={}, e2e={}, launches=3,
                             clocks={}, dtype="f32")
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert k in line
    json.dumps(line)


def test_reference_arm_runs_on_cpu():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "1", "--steps", "3", "--warmup", "1"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        v = bench.max_over_ranks(float(rank + 1) * 1.5, world)
        bench.barrier(world)
        q.put((rank, v))
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 3.0), (1, 3.0)]


def test_single_process_is_identity():
    assert bench.max_over_ranks(2.5, 1) == 2.5


def test_gated_work_counts_add_z_and_silu():
    w0 = bench.work_counts(2, 2048, 1536, 16, 4)
    w1 = bench.work_counts(2, 2048, 1536, 16, 4, gated=True)
    E = 2 * 2048 * 1536
    assert w1["bytes"] - w0["bytes"] == E * 4 + 1536 * 4
    assert w1["mufu"] - w0["mufu"] == 2 * E and w1["fp32"] - w0["fp32"] == 3 * E
    assert w1["updates"] == w0["updates"]


def test_reference_arm_runs_gated_workload():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "6", "--steps", "1", "--warmup", "0", "--ref-chains", "4"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and "gate" in line["config"]["workload"]


def test_backward_work_counts():
    w = bench.bwd_work_counts(2, 2048, 1536, 16)
    E, S = 2 * 2048 * 1536, 2 * 2048 * 16
    assert w["bytes"] == 5 * E * 4 + 4 * S * 4 + 2 * 1536 * 16 * 4 == 127_074_304
    assert w["mufu"] == E * 16 + 4 * E and w["fp32"] == 21 * E * 16
    roof = bench.roofline(w, bench.peaks(148, 2032.0, 6484.3), 389e-6)
    assert roof["bound"] == "alu"                     # the adjoint's FP32 work binds, not the bytes
    assert roof["frac_strict"] == pytest.approx(roof["t_roof_us"]["fp32"] / 389.0)
    assert roof["frac"] == pytest.approx((roof["t_roof_us"]["fp32"] + roof["t_roof_us"]["mufu"]) / 389.0)


def test_traffic_is_null_when_the_kernel_changed(monkeypatch):
    """profiled_traffic returns the stored bytes only while the digest of the
    kernel's sources matches the one stored with them."""
    from selective_state_space_157_b300 import build as bld
    monkeypatch.setattr(bld, "source_digest", lambda kernel="fwd": "0000000000000000")
    assert bench.profiled_traffic(2) is None and bench.profiled_traffic(9) is None


def test_reference_arm_runs_backward_workload():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "9", "--steps", "1", "--warmup", "0"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and "backward" in line["config"]["workload"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
