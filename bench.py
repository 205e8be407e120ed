#!/usr/bin/env python
"""Benchmark of libselscan's selective scan on B300 GPUs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 2] [--impl reference]

One step is one selscan_fwd call over one batch of the workload (default:
the Mamba-130M-like layer scan, Bsz=2 L=2048 D=1536 N=16 fp32, softplus on),
with its inputs already in device memory. Several copies of the inputs are
rotated so that every step reads from HBM, not from L2. W untimed warm-up
steps, then exactly K steps between a barrier and a synchronisation, timed
with CUDA events on the launching stream; the maximum over ranks is taken.
Rank 0 prints one JSON line.

Several GPUs run independent replicas (the scan has no cross-GPU exchange):
every rank processes the same workload on its own GPU and `value` counts
the elements all ranks processed.

`--impl reference` times the fp64 CPU oracle, the only other implementation
of the method, on the host cores, on a bounded sample of the same workload
per step.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "selective-scan B·L·D elems/s and HBM GB/s as % of roofline (1 B300)"
UNIT = "elem/s"

# Per-SM unit counts of the B300 (sm_103) used for the arithmetic roofline:
# the special-function unit issues 32 base-2 exponentials per clock per SM
# (measured: 29.7/clk at the nominal clock, 8.9 T/s on 148 SMs), the FP32
# pipe 128 lanes per clock per SM.
MUFU_EX2_PER_CLK_SM = 32
FP32_PER_CLK_SM = 128
FALLBACK_HBM_GBS = 6400.0   # used only if the measured peak file is absent


# --------------------------------------------------------------- roofline

def work_counts(Bsz, L, D, N, elem_bytes, softplus=True, h0=False, hT=False):
    """Algorithmic work of one forward call.

    bytes: x, delta, y streams (3 * B*L*D elements) + B, C (2 * B*L*N) + A (D*N fp32)
    (+ h0 / hT, B*D*N fp32 each when used); the (B, L, D, N) intermediates
    are never formed, so they do not count.
    mufu: one exponential per (t, d, n), plus exp and log per (t, d) for softplus.
    fp32: four per (t, d, n): dl*A, (dl*x)*B, the state FMA and the read-out FMA.
    """
    E = Bsz * L * D
    S = Bsz * L * N
    nbytes = 3 * E * elem_bytes + 2 * S * elem_bytes + D * N * 4
    nbytes += Bsz * D * N * 4 * (int(bool(h0)) + int(bool(hT)))
    return {"elems": E, "updates": E * N, "bytes": nbytes,
            "mufu": E * N + (2 * E if softplus else 0), "fp32": 4 * E * N}


def peaks(sms: int, sm_mhz: float, hbm_gbs: float):
    return {"mufu_per_s": sms * MUFU_EX2_PER_CLK_SM * sm_mhz * 1e6,
            "fp32_per_s": sms * FP32_PER_CLK_SM * sm_mhz * 1e6,
            "hbm_bytes_per_s": hbm_gbs * 1e9}


def roofline(work: dict, pk: dict, seconds: float, traffic=None, kernel="selscan_fwd"):
    """Roofline of one call: strict bound max(t_HBM, t_MUFU, t_FP32), and the
    summed form max(t_HBM, t_MUFU + t_FP32) as the benchmark statement words it."""
    t_hbm = work["bytes"] / pk["hbm_bytes_per_s"]
    t_mufu = work["mufu"] / pk["mufu_per_s"]
    t_fp32 = work["fp32"] / pk["fp32_per_s"]
    t_roof = max(t_hbm, t_mufu, t_fp32)
    t_sum = max(t_hbm, t_mufu + t_fp32)
    bound = "hbm" if t_hbm >= max(t_mufu, t_fp32) else "alu"
    return {
        "bound": bound,
        "achieved": work["updates"] / seconds / 1e12,
        "peak": work["updates"] / t_roof / 1e12,
        "unit": "Tupdate/s",
        "frac": t_roof / seconds,
        "frac_summed_bound": t_sum / seconds,
        "hbm_gbs": work["bytes"] / seconds / 1e9,
        "hbm_frac": t_hbm / seconds,
        "t_roof_us": {"hbm": t_hbm * 1e6, "mufu": t_mufu * 1e6, "fp32": t_fp32 * 1e6},
        "traffic": traffic,
        "kernel": kernel,
        "peak_source": pk.get("source", ""),
    }


def read_measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d.get("sm_max_mhz", 2032.0)), "measured (MEASURED_PEAKS.json)"
    return FALLBACK_HBM_GBS, 2032.0, "fallback"


def profiled_traffic(workload_id: int):
    """DRAM bytes per call from the committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        from selective_state_space_157_b300.build import source_digest
        entry = d.get(str(workload_id))
        if entry and entry.get("sources") == source_digest():
            return entry["dram_bytes_per_call"]
    except Exception:
        return None
    return None


def result_line(*, value, n_gpus, steps, warmup, ms_per_step, config, roof, cpu, e2e, launches,
                clocks, dtype):
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": n_gpus, "steps": steps,
        "warmup": warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dtype, "data": "synthetic",
        "config": config, "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": launches, "clocks": clocks,
    }


# --------------------------------------------------------------- clocks

class ClockSampler:
    """Samples SM clock and throttle reasons through NVML while running."""

    REASONS = {
        0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
        0x4: "sw_power_cap", 0x80: "hw_power_brake_slowdown", 0x2: "applications_clocks_setting",
    }

    def __init__(self, index: int, period_s: float = 0.001):
        self.index, self.period = index, period_s
        self.samples, self.reasons = [], set()
        self._stop = threading.Event()
        self._thread = None
        self.max_mhz = None
        try:
            import pynvml
            pynvml.nvmlInit()
            self.nv = pynvml
            self.h = self._handle(pynvml, index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
            self._reasons = getattr(pynvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                pynvml.nvmlDeviceGetCurrentClocksThrottleReasons
        except Exception:
            self.nv = None

    @staticmethod
    def _handle(pynvml, index):
        """NVML numbers GPUs on its own; find the CUDA device by PCI address."""
        try:
            import torch
            p = torch.cuda.get_device_properties(index)
            bus = f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
            return pynvml.nvmlDeviceGetHandleByPciBusId(bus.encode())
        except Exception:
            return pynvml.nvmlDeviceGetHandleByIndex(index)

    def _run(self):
        while not self._stop.is_set():
            try:
                self.samples.append(self.nv.nvmlDeviceGetClockInfo(self.h, self.nv.NVML_CLOCK_SM))
                r = self._reasons(self.h)
                for bit, name in self.REASONS.items():
                    if r & bit:
                        self.reasons.add(name)
            except Exception:
                pass
            time.sleep(self.period)

    def __enter__(self):
        if self.nv is not None:
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()
        return self

    def __exit__(self, *exc):
        if self._thread is not None:
            self._stop.set()
            self._thread.join()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
                    "source": "unavailable"}
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons), "samples": len(self.samples), "source": "NVML, 1 ms"}


# --------------------------------------------------------------- distributed

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Maximum of a float over all ranks (identity for one process)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# --------------------------------------------------------------- CPU oracle

def cpu_oracle_run(inp, chains=None, nthreads=0):
    """Times the fp64 oracle on the given chains (all when None). Returns
    (seconds, elements processed, threads used)."""
    import numpy as np
    import oracle
    Bsz, L, D = inp.x.shape
    nthreads = nthreads or len(os.sched_getaffinity(0))
    o = oracle.default()
    x, dl, A, B, C = inp.f32("x"), inp.f32("delta"), inp.A, inp.f32("B"), inp.f32("C")
    t0 = time.perf_counter()
    if chains is None:
        o.selscan_fwd(x, dl, A, B, C, inp.delta_softplus, nthreads=nthreads)
        n = Bsz * D
    else:
        o.selscan_fwd_chains(x, dl, A, B, C, np.asarray(chains), inp.delta_softplus, nthreads=nthreads)
        n = len(chains)
    return time.perf_counter() - t0, n * L, nthreads


def sample_chains(Bsz, D, count):
    import numpy as np
    return np.unique(np.linspace(0, Bsz * D - 1, count).astype(np.int64))


# --------------------------------------------------------------- GPU runs

def run_gpu(args, world, rank, local):
    import torch
    import selective_state_space_157_b300 as ss
    from selective_state_space_157_b300 import workloads as W

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    w = W.WORKLOADS[args.workload]
    if w.steps:
        raise SystemExit("bench.py times the forward workloads 1-4; the decode workload is a parity case")
    inp = W.workload_inputs(args.workload)
    bf16 = w.dtype == W.BF16
    es = 2 if bf16 else 4

    def dev_t(a, kind):
        if bf16 and kind == "io":
            return torch.from_numpy(a.view("int16")).view(torch.bfloat16).to(dev)
        return torch.from_numpy(a).to(dev)

    Bsz, L, D = inp.x.shape
    N = inp.A.shape[1]
    want_hT = w.return_state
    foot = (3 * Bsz * L * D + 2 * Bsz * L * N) * es
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    copies = max(1, -(-(2 * l2) // foot))          # rotate until > 2x L2 is touched between reuses
    base = [dev_t(inp.x, "io"), dev_t(inp.delta, "io"), dev_t(inp.A, "f"),
            dev_t(inp.B, "io"), dev_t(inp.C, "io")]
    sets = [base] + [[t.clone() for t in base] for _ in range(copies - 1)]
    ys = [torch.empty_like(base[0]) for _ in range(copies)]
    hT = torch.empty(Bsz, D, N, device=dev) if want_hT else None

    def step(i):
        x, dl, A, B, C = sets[i % copies]
        ss.selscan_fwd(x, dl, A, B, C, True, None, y=ys[i % copies], hT=hT)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    ss.check_device_error()

    plan = ss.fwd_plan(Bsz, L, D, N, bf16=bf16)
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world, dev)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        e0.record(stream)
        for i in range(args.steps):
            step(i)
        e1.record(stream)
        torch.cuda.synchronize()
    barrier(world, dev)
    ss.check_device_error()
    sec = e0.elapsed_time(e1) / 1e3
    sec = max_over_ranks(sec, world, dev)
    per_step = sec / args.steps
    elems = Bsz * L * D
    value = world * elems * args.steps / sec

    # end to end through the public API from pinned host buffers
    e2e = None
    if rank == 0 or world > 1:
        host = [torch.from_numpy(inp.x.view("int16")).view(torch.bfloat16) if bf16 else torch.from_numpy(inp.x),
                torch.from_numpy(inp.delta.view("int16")).view(torch.bfloat16) if bf16 else torch.from_numpy(inp.delta),
                torch.from_numpy(inp.A),
                torch.from_numpy(inp.B.view("int16")).view(torch.bfloat16) if bf16 else torch.from_numpy(inp.B),
                torch.from_numpy(inp.C.view("int16")).view(torch.bfloat16) if bf16 else torch.from_numpy(inp.C)]
        host = [t.pin_memory() for t in host]
        y_host = torch.empty(ys[0].shape, dtype=ys[0].dtype, pin_memory=True)
        e2e_steps = max(1, min(args.steps, 20))
        ss.selscan_fwd(*host, True, y=y_host)            # warm the copy path
        barrier(world, dev)
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            ss.selscan_fwd(*host, True, y=y_host)      # H2D, kernels, D2H, synchronise
        t_e2e = max_over_ranks(time.perf_counter() - t0, world, dev)
        h2d = sum(t.numel() * t.element_size() for t in host)
        e2e = {"value": world * elems * e2e_steps / t_e2e, "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": y_host.numel() * y_host.element_size()}

    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank != 0:
        return None

    hbm_gbs, max_mhz, src = read_measured_peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    pk = peaks(sms, max_mhz, hbm_gbs)
    pk["source"] = f"HBM {src}; MUFU/FP32 derived: {sms} SMs x (32 ex2, 128 fp32)/clk x {max_mhz:.0f} MHz"
    work = work_counts(Bsz, L, D, N, es, softplus=True, hT=want_hT)
    roof = roofline(work, pk, per_step, traffic=profiled_traffic(args.workload),
                    kernel=f"selscan_fwd call ({plan['launches']} launches, {plan['chunks']} chunks)")

    cpu = None
    if not args.no_cpu_baseline:
        chains = None if Bsz * D * L <= 8_000_000 else sample_chains(Bsz, D, 256)
        secs, n_el, thr = cpu_oracle_run(inp, chains)
        cpu = {"value": n_el / secs, "unit": UNIT, "cores": thr, "kind": "oracle",
               "sample": ("the whole workload" if chains is None else f"{len(chains)} of {Bsz * D} chains over all L")
               + f" ({n_el} elements, {secs:.2f} s, fp64)"}

    config = {"workload": f"{w.name}: Bsz={Bsz} L={L} D={D} N={N} {w.dtype}, softplus on"
                          + (", returns hT" if want_hT else ""),
              "global_batch": Bsz * world, "seq_len": L, "parallelism": f"replicas x{world}",
              "l2": f"{copies} rotating input sets ({copies * foot / 1e6:.0f} MB) > 2x L2 ({l2 / 1e6:.0f} MB)"
                    if copies > 1 else f"inputs {foot / 1e6:.0f} MB > 2x L2",
              "plan": plan}
    return result_line(value=value, n_gpus=world, steps=args.steps, warmup=args.warmup,
                       ms_per_step=per_step * 1e3, config=config, roof=roof, cpu=cpu, e2e=e2e,
                       launches=plan["launches"] * args.steps, clocks=clk.summary(),
                       dtype="bf16 io, f32 math" if bf16 else "f32")


def run_reference(args, world, rank):
    """The oracle as the reference arm: each step is one oracle run over a
    bounded sample of the workload's chains, on the host cores."""
    if rank != 0:
        return None
    from selective_state_space_157_b300 import workloads as W
    w = W.WORKLOADS[args.workload]
    inp = W.workload_inputs(args.workload)
    Bsz, L, D = inp.x.shape
    chains = sample_chains(Bsz, D, args.ref_chains)
    for _ in range(args.warmup):
        cpu_oracle_run(inp, chains)
    tot, n_total, thr = 0.0, 0, 0
    for _ in range(args.steps):
        s, n, thr = cpu_oracle_run(inp, chains)
        tot += s
        n_total += n
    value = n_total / tot
    sample = f"{len(chains)} of {Bsz * D} chains over all L={L} per step (fp64)"
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{w.name}: Bsz={Bsz} L={L} D={D} N={inp.A.shape[1]} {w.dtype}, softplus on",
                   "seq_len": L, "parallelism": "host threads"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": thr, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", type=int, default=2, choices=[1, 2, 3, 4])
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-chains", type=int, default=192, help="chains per reference step")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        out = run_reference(args, world, rank)
    else:
        out = run_gpu(args, world, rank, local)
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
