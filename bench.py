#!/usr/bin/env python
"""Benchmark of libselscan's selective scan on B300 GPUs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 2] [--impl reference]

One step is one selscan_fwd call over one batch of the workload (default:
the long-context scan, Bsz=1 L=131072 D=1536 N=16 fp32, softplus on, final
state returned -- the largest configuration the benchmark statement names),
with its inputs already in device memory. Inputs larger than L2 are read
from HBM on every step; smaller ones are rotated over several copies so that
they are. W untimed warm-up steps, then exactly K steps between a barrier and
a synchronisation, timed with CUDA events on the launching stream; the
maximum over ranks is taken. Rank 0 prints one JSON line. With the default
workload the line also carries ``per_config``: the same measurement, shorter,
of the 130M-like (2), 370M-like bf16 (3) and decode (5) workloads.

The roofline is the benchmark statement's: the slower of the HBM time
(algorithmic bytes over the measured copy bandwidth) and the MUFU time plus
the FP32 time (exponentials over the measured ex2 rate, plus FP32 operations
over the measured FMA rate; both rates from the committed probe
csrc/probe/alu_peaks.cu, run at the start of every bench). ``frac`` is
measured against that bound; ``frac_strict`` against max(HBM, MUFU, FP32).

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

# Per-SM unit counts of the B300 (sm_103), used for the arithmetic roofline
# only when the peak probe cannot run (the line then says "derived"): 32
# base-2 exponentials and 128 FP32 lanes per clock per SM.
MUFU_EX2_PER_CLK_SM = 32
FP32_PER_CLK_SM = 128
FALLBACK_HBM_GBS = 6400.0   # used only if the measured peak file is absent
DEFAULT_WORKLOAD = 4
PER_CONFIG = (2, 3, 5)


# --------------------------------------------------------------- roofline

def work_counts(Bsz, L, D, N, elem_bytes, softplus=True, h0=False, hT=False, gated=False, zoh=False):
    """Algorithmic work of one forward call.

    bytes: x, delta, y streams (3 * B*L*D elements) + B, C (2 * B*L*N) + A (D*N fp32)
    (+ h0 / hT, B*D*N fp32 each when used; + the gate's z stream and Dskip
    (D fp32) for the gated form); the (B, L, D, N) intermediates are never
    formed, so they do not count.
    mufu: one exponential per (t, d, n), plus exp and log per (t, d) for
    softplus, plus exp and reciprocal per (t, d) for silu(z).
    fp32: four per (t, d, n): dl*A, (dl*x)*B, the state FMA and the read-out
    FMA; the gated form adds the skip FMA, 1 + e^-z and the product per (t, d).
    The zero-order-hold form adds per (t, d, n) one division (a MUFU
    reciprocal) and three FP32 operations for (e^w - 1) / A * x * B.
    """
    E = Bsz * L * D
    S = Bsz * L * N
    nbytes = 3 * E * elem_bytes + 2 * S * elem_bytes + D * N * 4
    nbytes += Bsz * D * N * 4 * (int(bool(h0)) + int(bool(hT)))
    mufu = E * N + (2 * E if softplus else 0)
    fp32 = 4 * E * N
    if gated:
        nbytes += E * elem_bytes + D * 4
        mufu += 2 * E
        fp32 += 3 * E
    if zoh:
        mufu += E * N
        fp32 += 3 * E * N
    return {"elems": E, "updates": E * N, "bytes": nbytes, "mufu": mufu, "fp32": fp32}


def bwd_work_counts(Bsz, L, D, N, gated=False):
    """Algorithmic work of one backward call (fp32, softplus on, no h0/dhT).

    bytes: x, delta, dy read and dx, ddelta written (5 * B*L*D fp32), B, C read
    and dB, dC written (4 * B*L*N), A read and dA written (2 * D*N).
    mufu: the decay exp(dl*A) once per (t, d, n), which the recomputed
    forward and the adjoint share; per (t, d) exp and log for softplus and
    exp and reciprocal for its derivative.
    fp32: 21 per (t, d, n): 4 for the recomputed state update (as in the
    forward), 13 for the adjoint step (g += gy*C, gy*h, g*h*a, (.)*A + g*B*x,
    dA += (.)*dl, g*dl*x, g*dl*B, g *= a), and one addition for each of the
    four sums (dx and ddelta over n, dB and dC over d).
    gated (the block's skip and gate): z read and dz written, Dskip read and
    dDskip written; per (t, d) sigmoid(z) (exp and reciprocal) and 12 fp32
    operations (silu, silu', dz, the skip's share of dx and dDskip); per
    (t, d, n) 2 more for the scan's read-out s_t that dz needs.
    """
    E = Bsz * L * D
    S = Bsz * L * N
    nbytes = 5 * E * 4 + 4 * S * 4 + 2 * D * N * 4
    mufu, fp32 = E * N + 4 * E, 21 * E * N
    if gated:
        nbytes += 2 * E * 4 + 2 * D * 4
        mufu += 2 * E
        fp32 += 2 * E * N + 12 * E
    return {"elems": E, "updates": E * N, "bytes": nbytes, "mufu": mufu, "fp32": fp32}


def step_work_counts(Bsz, D, N):
    """Algorithmic work of one decode step: the state is read and written once
    (2 * B*D*N fp32), x, delta and y move once (3 * B*D), B and C once per batch
    row (2 * B*N), A once (D*N)."""
    E = Bsz * D
    nbytes = 2 * E * N * 4 + 3 * E * 4 + 2 * Bsz * N * 4 + D * N * 4
    return {"elems": E, "updates": E * N, "bytes": nbytes, "mufu": E * N, "fp32": 4 * E * N}


def peaks(sms: int, sm_mhz: float, hbm_gbs: float, alu=None):
    """Roofline denominators: the measured HBM copy rate, and the ex2 and FP32
    rates from the probe (``alu``, ops/s) or, failing that, derived from the
    unit counts at the maximum SM clock."""
    if alu:
        mufu, fp32 = alu["ex2_per_s"], alu["fp32_per_s"]
    else:
        mufu, fp32 = sms * MUFU_EX2_PER_CLK_SM * sm_mhz * 1e6, sms * FP32_PER_CLK_SM * sm_mhz * 1e6
    return {"mufu_per_s": mufu, "fp32_per_s": fp32, "hbm_bytes_per_s": hbm_gbs * 1e9}


def roofline(work: dict, pk: dict, seconds: float, traffic=None, kernel="selscan_fwd"):
    """Roofline of one call. The bound is the benchmark statement's: the
    slower of t_HBM and t_MUFU + t_FP32 (``frac``); the stricter
    max(t_HBM, t_MUFU, t_FP32) is reported as ``frac_strict``."""
    t_hbm = work["bytes"] / pk["hbm_bytes_per_s"]
    t_mufu = work["mufu"] / pk["mufu_per_s"]
    t_fp32 = work["fp32"] / pk["fp32_per_s"]
    t_strict = max(t_hbm, t_mufu, t_fp32)
    t_sum = max(t_hbm, t_mufu + t_fp32)
    bound = "hbm" if t_hbm >= t_mufu + t_fp32 else "alu"
    if bound == "hbm":   # bytes moved per second against the measured copy bandwidth
        achieved, peak, unit = work["bytes"] / seconds / 1e9, pk["hbm_bytes_per_s"] / 1e9, "GB/s"
    else:                # state updates per second against the MUFU + FP32 bound
        achieved, peak, unit = work["updates"] / seconds / 1e12, work["updates"] / t_sum / 1e12, "Tupdate/s"
    return {
        "bound": bound,
        "achieved": achieved,
        "peak": peak,
        "unit": unit,
        "frac": t_sum / seconds,
        "frac_strict": t_strict / seconds,
        "hbm_gbs": work["bytes"] / seconds / 1e9,
        "hbm_frac": t_hbm / seconds,
        "t_roof_us": {"hbm": t_hbm * 1e6, "mufu": t_mufu * 1e6, "fp32": t_fp32 * 1e6},
        "traffic": traffic,
        "kernel": kernel,
        "peak_source": pk.get("source", ""),
    }


def measure_alu_peaks():
    """Runs the committed probe (libselscan_probe.so): ex2 results per second
    and FP32 lane-operations per second (the larger of the scalar and packed
    FMA rates). None if the probe is missing or fails."""
    import ctypes
    path = os.path.join(ROOT, "selective_state_space_157_b300", "libselscan_probe.so")
    if not os.path.exists(path):
        return None
    try:
        lib = ctypes.CDLL(path)
        e, f, f2 = ctypes.c_double(0), ctypes.c_double(0), ctypes.c_double(0)
        if lib.selscan_probe_alu_peaks(ctypes.byref(e), ctypes.byref(f), ctypes.byref(f2)) != 0:
            return None
        return {"ex2_per_s": e.value, "ffma_per_s": f.value, "ffma2_per_s": f2.value,
                "fp32_per_s": max(f.value, f2.value)}
    except OSError:
        return None


def peak_source(src_hbm: str, alu, sms: int, mhz: float) -> str:
    if alu:
        return (f"HBM {src_hbm}; MUFU {alu['ex2_per_s'] / 1e12:.2f} T ex2/s and FP32 "
                f"{alu['fp32_per_s'] / 1e12:.2f} T op/s measured by csrc/probe/alu_peaks.cu "
                f"(scalar FMA {alu['ffma_per_s'] / 1e12:.2f}, packed {alu['ffma2_per_s'] / 1e12:.2f} T op/s)")
    return (f"HBM {src_hbm}; MUFU/FP32 derived (probe unavailable): {sms} SMs x "
            f"({MUFU_EX2_PER_CLK_SM} ex2, {FP32_PER_CLK_SM} fp32)/clk x {mhz:.0f} MHz")


def read_measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d.get("sm_max_mhz", 2032.0)), "measured (MEASURED_PEAKS.json)"
    return FALLBACK_HBM_GBS, 2032.0, "fallback"


def kernel_family(w) -> str:
    """The kernel family a workload times (the key of its sources' digest)."""
    if w.ssd_heads:
        return "ssd"
    if w.backward:
        return "bwd"
    if w.steps:
        return "step"
    if w.conv_K:
        return "conv1d"
    return "fwd"


def profiled_traffic(workload_id: int):
    """DRAM bytes per call from the committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        from selective_state_space_157_b300 import workloads as W
        from selective_state_space_157_b300.build import source_digest
        entry = d.get(str(workload_id))
        if entry and entry.get("sources") == source_digest(kernel_family(W.WORKLOADS[workload_id])):
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

class _Nvml:
    """Minimal ctypes binding to the driver's NVML library (libnvidia-ml.so.1)."""
    CLOCK_SM = 1

    def __init__(self):
        import ctypes
        self.c = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")

    def handle(self, cuda_index: int):
        """NVML numbers GPUs on its own: find the CUDA device by PCI address."""
        c = self.c
        h = c.c_void_p()
        try:
            import torch
            p = torch.cuda.get_device_properties(cuda_index)
            bus = f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0".encode()
            if self.lib.nvmlDeviceGetHandleByPciBusId_v2(c.c_char_p(bus), c.byref(h)) == 0:
                return h
        except Exception:
            pass
        if self.lib.nvmlDeviceGetHandleByIndex_v2(c.c_uint(cuda_index), c.byref(h)) != 0:
            raise RuntimeError("no NVML handle")
        return h

    def clock(self, h, maximum=False):
        v = self.c.c_uint()
        fn = self.lib.nvmlDeviceGetMaxClockInfo if maximum else self.lib.nvmlDeviceGetClockInfo
        return v.value if fn(h, self.CLOCK_SM, self.c.byref(v)) == 0 else None

    def reasons(self, h):
        v = self.c.c_ulonglong()
        for name in ("nvmlDeviceGetCurrentClocksEventReasons", "nvmlDeviceGetCurrentClocksThrottleReasons"):
            fn = getattr(self.lib, name, None)
            if fn is not None and fn(h, self.c.byref(v)) == 0:
                return v.value
        return 0


class ClockSampler:
    """Samples the SM clock and the clock-event (throttle) reasons through NVML
    every millisecond while running."""

    REASONS = {
        0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
        0x4: "sw_power_cap", 0x80: "hw_power_brake_slowdown", 0x2: "applications_clocks_setting",
    }

    def __init__(self, index: int, period_s: float = 0.001):
        self.period = period_s
        self.samples, self.reasons = [], set()
        self._stop = threading.Event()
        self._thread = None
        self.max_mhz = None
        self.error = None
        try:
            self.nv = _Nvml()
            self.h = self.nv.handle(index)
            self.max_mhz = self.nv.clock(self.h, maximum=True)
        except Exception as e:   # no NVML: the line says so
            self.nv = None
            self.error = str(e)

    def _run(self):
        while not self._stop.is_set():
            mhz = self.nv.clock(self.h)
            if mhz is not None:
                self.samples.append(mhz)
            r = self.nv.reasons(self.h)
            for bit, name in self.REASONS.items():
                if r & bit:
                    self.reasons.add(name)
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
                    "source": "unavailable" + (f" ({self.error})" if self.error else "")}
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons), "samples": len(self.samples),
                "source": "NVML every 1 ms during the timed region"}


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

def cpu_oracle_run(inp, chains=None, nthreads=0, gate=None, zoh=False):
    """Times the fp64 oracle on the given chains (all when None), with the
    block's skip and gate when ``gate`` = (Dskip, z fp32). Returns
    (seconds, elements processed, threads used)."""
    import numpy as np
    import oracle
    Bsz, L, D = inp.x.shape
    nthreads = nthreads or len(os.sched_getaffinity(0))
    o = oracle.default()
    x, dl, A, B, C = inp.f32("x"), inp.f32("delta"), inp.A, inp.f32("B"), inp.f32("C")
    Dskip, z = gate if gate is not None else (None, None)
    t0 = time.perf_counter()
    if chains is None:
        o.selscan_fwd(x, dl, A, B, C, inp.delta_softplus, nthreads=nthreads, Dskip=Dskip, z=z, zoh=zoh)
        n = Bsz * D
    else:
        o.selscan_fwd_chains(x, dl, A, B, C, np.asarray(chains), inp.delta_softplus, nthreads=nthreads,
                             Dskip=Dskip, z=z, zoh=zoh)
        n = len(chains)
    return time.perf_counter() - t0, n * L, nthreads


def sample_chains(Bsz, D, count):
    import numpy as np
    return np.unique(np.linspace(0, Bsz * D - 1, count).astype(np.int64))


# --------------------------------------------------------------- GPU runs

class _FwdBench:
    """Device inputs of a forward workload, rotated over enough copies that
    more than 2x L2 is touched between reuses, and its step function."""

    def __init__(self, wid, dev, seq_len=None):
        import dataclasses
        import torch
        import selective_state_space_157_b300 as ss
        from selective_state_space_157_b300 import workloads as W
        self.w = w = W.WORKLOADS[wid]
        if seq_len:
            # A shorter sequence of the same workload (same kernels, same
            # distributions): the small case a full profiler capture runs on.
            if w.gated:
                raise SystemExit("--seq-len is not offered for the gated workload")
            self.w = w = dataclasses.replace(w, L=seq_len)
            self.inp = inp = W.fwd_inputs(w.Bsz, w.L, w.D, w.N, seed=w.seed, dtype=w.dtype, u_mean=w.u_mean,
                                          a_init=w.a_init, delta_softplus=True)
        else:
            self.inp = inp = W.workload_inputs(wid)
        self.bf16 = bf16 = w.dtype == W.BF16
        self.es = es = 2 if bf16 else 4
        self.gate = W.workload_gate_inputs(wid) if w.gated else None

        def dev_t(a, kind):
            if bf16 and kind == "io":
                return torch.from_numpy(a.view("int16")).view(torch.bfloat16).to(dev)
            return torch.from_numpy(a).to(dev)

        self.Bsz, self.L, self.D = Bsz, L, D = inp.x.shape
        self.N = N = inp.A.shape[1]
        self.foot = ((4 if w.gated else 3) * Bsz * L * D + 2 * Bsz * L * N) * es
        self.l2 = l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.copies = copies = max(1, -(-(2 * l2) // self.foot))
        base = [dev_t(inp.x, "io"), dev_t(inp.delta, "io"), dev_t(inp.A, "f"), dev_t(inp.B, "io"),
                dev_t(inp.C, "io")]
        if w.gated:
            base += [dev_t(self.gate[1], "io")]
            self.Dskip_dev = dev_t(self.gate[0], "f")
        self.sets = [base] + [[t.clone() for t in base] for _ in range(copies - 1)]
        self.ys = [torch.empty_like(base[0]) for _ in range(copies)]
        self.hT = torch.empty(Bsz, D, N, device=dev) if w.return_state else None
        self.ss = ss

    def step(self, i):
        k = i % self.copies
        x, dl, A, B, C = self.sets[k][:5]
        if self.w.zoh:
            self.ss.selscan_fwd(x, dl, A, B, C, True, None, y=self.ys[k], hT=self.hT, zoh=True)
        elif self.w.gated:
            self.ss.selscan_fwd(x, dl, A, B, C, True, None, y=self.ys[k], hT=self.hT,
                                D_skip=self.Dskip_dev, z=self.sets[k][5])
        else:
            self.ss.selscan_fwd(x, dl, A, B, C, True, None, y=self.ys[k], hT=self.hT)

    def l2_note(self):
        if self.copies > 1:
            return (f"{self.copies} rotating input sets ({self.copies * self.foot / 1e6:.0f} MB) "
                    f"> 2x L2 ({self.l2 / 1e6:.0f} MB)")
        return f"inputs {self.foot / 1e6:.0f} MB > 2x L2 ({self.l2 / 1e6:.0f} MB)"

    def workload_name(self):
        w = self.w
        return (f"{w.name}: Bsz={self.Bsz} L={self.L} D={self.D} N={self.N} {w.dtype}, softplus on"
                + (", returns hT" if w.return_state else "")
                + (", skip and SiLU gate fused (y = (scan + Dskip x) silu(z))" if w.gated else "")
                + (", zero-order-hold Bbar" if w.zoh else ""))

    def work(self):
        return work_counts(self.Bsz, self.L, self.D, self.N, self.es, softplus=True, hT=self.w.return_state,
                           gated=self.w.gated, zoh=self.w.zoh)


def timed_steps(step, steps, warmup, world, dev, local):
    """W warm-up steps, then K steps between a barrier and a synchronisation,
    timed with CUDA events on the launching stream, clocks sampled meanwhile.
    Returns (seconds over all K steps, max over ranks; clock summary)."""
    import torch
    import selective_state_space_157_b300 as ss
    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    ss.check_device_error()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world, dev)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        e0.record(stream)
        for i in range(steps):
            step(i)
        e1.record(stream)
        torch.cuda.synchronize()
    barrier(world, dev)
    ss.check_device_error()
    return max_over_ranks(e0.elapsed_time(e1) / 1e3, world, dev), clk.summary()


def run_gpu(args, world, rank, local):
    import torch
    import selective_state_space_157_b300 as ss
    from selective_state_space_157_b300 import workloads as W

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    alu = measure_alu_peaks()
    w = W.WORKLOADS[args.workload]
    if w.ssd_heads:
        return run_ssd(args, world, rank, local, dev, w)
    if w.steps:
        return run_decode(args, world, rank, local, dev, w, alu)
    if w.conv_K:
        return run_conv(args, world, rank, local, dev, w, alu)
    if w.backward:
        return run_bwd(args, world, rank, local, dev, w, alu)

    fb = _FwdBench(args.workload, dev, args.seq_len)
    w = fb.w
    Bsz, L, D, N, bf16 = fb.Bsz, fb.L, fb.D, fb.N, fb.bf16
    sec, clocks = timed_steps(fb.step, args.steps, args.warmup, world, dev, local)
    per_step = sec / args.steps
    elems = Bsz * L * D
    value = world * elems * args.steps / sec
    plan = ss.fwd_plan(Bsz, L, D, N, bf16=bf16)
    config = {"workload": fb.workload_name(), "global_batch": Bsz * world, "seq_len": L,
              "parallelism": f"replicas x{world}", "l2": fb.l2_note(), "plan": plan}
    work = fb.work()
    inp, gate = fb.inp, fb.gate
    del fb
    torch.cuda.empty_cache()

    e2e = fwd_e2e(args, world, dev, w, inp, gate, bf16, elems)

    per_config = None
    if args.workload == DEFAULT_WORKLOAD and not args.no_per_config and not args.seq_len:
        per_config = {}
        for wid in PER_CONFIG:
            per_config[str(wid)] = measure_config(wid, args, world, local, dev, alu)
            torch.cuda.empty_cache()

    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank != 0:
        return None

    hbm_gbs, max_mhz, src = read_measured_peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    pk = peaks(sms, max_mhz, hbm_gbs, alu)
    pk["source"] = peak_source(src, alu, sms, max_mhz)
    roof = roofline(work, pk, per_step, traffic=None if args.seq_len else profiled_traffic(args.workload),
                    kernel=f"selscan_fwd call ({plan['launches']} launches, {plan['chunks']} chunks)")

    cpu = None
    if not args.no_cpu_baseline:
        chains = None if Bsz * D * L <= 8_000_000 else sample_chains(Bsz, D, 256)
        secs, n_el, thr = cpu_oracle_run(inp, chains, gate=gate, zoh=w.zoh)
        cpu = {"value": n_el / secs, "unit": UNIT, "cores": thr, "kind": "oracle",
               "sample": ("the whole workload" if chains is None else f"{len(chains)} of {Bsz * D} chains over all L")
               + f" ({n_el} elements, {secs:.2f} s, fp64)"}
    line = result_line(value=value, n_gpus=world, steps=args.steps, warmup=args.warmup,
                       ms_per_step=per_step * 1e3, config=config, roof=roof, cpu=cpu, e2e=e2e,
                       launches=plan["launches"] * args.steps, clocks=clocks,
                       dtype="bf16 io, f32 math" if bf16 else "f32")
    if per_config is not None:
        line["per_config"] = per_config
    return line


def host_like(t):
    """A copy of host tensor ``t`` in page-locked memory from the library's
    host allocator (``selscan_host_alloc``), whose buffers the DMA engines
    read at the link's rate."""
    import selective_state_space_157_b300 as ss
    h = ss.host_empty(tuple(t.shape), t.dtype)
    h.copy_(t)
    return h


def host_zeros(shape, dtype=None):
    import selective_state_space_157_b300 as ss
    h = ss.host_empty(shape, dtype)
    h.zero_()
    return h


def evict_host_caches(nbytes=512 << 20):
    """Writes and reads a host buffer larger than the CPU's caches, so that
    host inputs written shortly before sit in DRAM, as inputs a loader wrote
    earlier would. On the B300 machines a DMA read of pinned memory whose lines
    were still dirty in the CPU cache ran at 15-17 GB/s instead of 55."""
    import numpy as np
    scratch = np.ones(nbytes // 8)
    float(scratch.sum())
    del scratch


def pcie_rates(dev, nbytes=256 << 20, reps=4):
    """Copy rates between page-locked host memory (the library's host
    allocator, written and then evicted from the CPU caches, as the end-to-end
    legs' buffers are) and this GPU (GB/s), timed with CUDA events: host to
    device, device to host, and both directions at once on two streams (their
    sum; the link does not carry both directions at their one-way rates
    together). The bound the end-to-end leg's copies can approach."""
    import torch
    h = host_zeros((nbytes,), torch.uint8)
    h2 = host_zeros((nbytes,), torch.uint8)
    evict_host_caches()
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d2 = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    st, st2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    rates = []
    for pairs in (((d, h),), ((h, d),), ((d, h), (h2, d2))):
        streams = (st, st2)[:len(pairs)]
        for (dst, src), s_ in zip(pairs, streams):
            with torch.cuda.stream(s_):
                dst.copy_(src, non_blocking=True)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        if len(pairs) > 1:
            st2.wait_event(e0)
        for (dst, src), s_ in zip(pairs, streams):
            with torch.cuda.stream(s_):
                for _ in range(reps):
                    dst.copy_(src, non_blocking=True)
        if len(pairs) > 1:
            st.wait_stream(st2)
        e1.record(st)
        torch.cuda.synchronize(dev)
        rates.append(len(pairs) * reps * nbytes / (e0.elapsed_time(e1) / 1e3) / 1e9)
    del h, h2, d, d2
    return rates[0], rates[1], rates[2]


def copy_bound_s(h2d, d2h, rates):
    """The least time the copies of one step can take: each direction at its
    own rate, and both together at the two-way rate."""
    h2d_gbs, d2h_gbs, both_gbs = rates
    return max(h2d / (h2d_gbs * 1e9), d2h / (d2h_gbs * 1e9), (h2d + d2h) / (both_gbs * 1e9))


def fwd_e2e(args, world, dev, w, inp, gate, bf16, elems):
    """End to end through the public API: the step's inputs copied in from
    pinned host memory, the scan, y copied out, inside the timed region."""
    import torch
    import selective_state_space_157_b300 as ss
    host = [torch.from_numpy(inp.x.view("int16")).view(torch.bfloat16) if bf16 else torch.from_numpy(inp.x),
            torch.from_numpy(inp.delta.view("int16")).view(torch.bfloat16) if bf16 else torch.from_numpy(inp.delta),
            torch.from_numpy(inp.A),
            torch.from_numpy(inp.B.view("int16")).view(torch.bfloat16) if bf16 else torch.from_numpy(inp.B),
            torch.from_numpy(inp.C.view("int16")).view(torch.bfloat16) if bf16 else torch.from_numpy(inp.C)]
    y_host = host_zeros(tuple(inp.x.shape), torch.bfloat16 if bf16 else torch.float32)
    hT_host = host_zeros((inp.x.shape[0], inp.x.shape[2], inp.A.shape[1])) \
        if w.return_state else None
    e2e_steps = max(1, min(args.steps, 20 if elems < 50_000_000 else 5))
    kw = {}
    if w.gated:
        # The block's skip and gate: Dskip and z from host memory as well.
        host += [torch.from_numpy(gate[1]), torch.from_numpy(gate[0])]
    host = [host_like(t) for t in host]
    if w.gated:
        kw = {"z": host[5], "D_skip": host[6]}
    if w.zoh:
        kw["zoh"] = True

    def e2e_call():
        # selscan_fwd_host(_ex): H2D, kernels, D2H, synchronise
        ss.selscan_fwd(*host[:5], True, y=y_host, hT=hT_host, **kw)
    e2e_call()                                       # warm the copy path
    evict_host_caches()
    barrier(world, dev)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_call()
    t_e2e = max_over_ranks(time.perf_counter() - t0, world, dev)
    h2d = sum(t.numel() * t.element_size() for t in host)
    d2h = y_host.numel() * y_host.element_size() + (hT_host.numel() * 4 if hT_host is not None else 0)
    rates = pcie_rates(dev)
    bound = copy_bound_s(h2d, d2h, rates)
    per_step = t_e2e / e2e_steps
    return {"value": world * elems * e2e_steps / t_e2e, "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": per_step * 1e3,
            "pcie": {"h2d_gbs": rates[0], "d2h_gbs": rates[1], "both_ways_gbs": rates[2],
                     "copy_bound_ms": bound * 1e3, "frac_of_copy_bound": bound / per_step,
                     "note": "rates of 256 MB page-locked copies measured in this run (one way each, and both "
                             "ways at once); host buffers from selscan_host_alloc, inputs evicted from the CPU "
                             "caches before the timed calls"}}


def measure_config(wid, args, world, local, dev, alu):
    """A shorter measurement of another workload for ``per_config``: per-step
    time, throughput and roofline fractions (no end-to-end or CPU legs). The
    timed region is taken three times and the median reported, with all
    three, so that one stall of the shared machine does not stand for the
    workload."""
    import torch
    import selective_state_space_157_b300 as ss
    from selective_state_space_157_b300 import workloads as W
    w = W.WORKLOADS[wid]
    steps = max(1, min(args.steps, 50))
    warmup = max(3, min(args.warmup, 10))
    hbm_gbs, max_mhz, src = read_measured_peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    pk = peaks(sms, max_mhz, hbm_gbs, alu)
    reps = []
    if w.steps:
        for _ in range(3):
            per_step, clocks, note = decode_time(w, steps, warmup, world, dev, local)
            reps.append((per_step, clocks))
        work = step_work_counts(w.Bsz, w.D, w.N)
        name = f"{w.name}: Bsz={w.Bsz} D={w.D} N={w.N} f32 decode step, state updated in place ({note})"
        elems = w.Bsz * w.D
    else:
        fb = _FwdBench(wid, dev)
        for _ in range(3):
            sec, clocks = timed_steps(fb.step, steps, warmup, world, dev, local)
            reps.append((sec / steps, clocks))
        work = fb.work()
        plan = ss.fwd_plan(fb.Bsz, fb.L, fb.D, fb.N, bf16=fb.bf16)
        name = fb.workload_name() + f" ({plan['chunks']} chunks; {fb.l2_note()})"
        elems = fb.Bsz * fb.L * fb.D
        del fb
    per_step, clocks = sorted(reps, key=lambda r: r[0])[len(reps) // 2]
    roof = roofline(work, pk, per_step)
    return {"workload": name, "ms_per_step": per_step * 1e3, "value": world * elems / per_step, "unit": UNIT,
            "frac": roof["frac"], "frac_strict": roof["frac_strict"], "bound": roof["bound"],
            "hbm_gbs": roof["hbm_gbs"], "t_roof_us": roof["t_roof_us"], "steps": steps, "warmup": warmup,
            "repeats_ms_per_step": [r[0] * 1e3 for r in reps], "reported": "median of the 3 timed regions",
            "clocks": clocks}


def run_conv(args, world, rank, local, dev, w, alu=None):
    """The conv1d workload: one step = one selscan_conv1d (K taps, SiLU) over
    (Bsz, L, D), a carried state handed in and out. Input sets rotate past
    2x L2. HBM-bound: x read and out written once."""
    import torch
    import selective_state_space_157_b300 as ss
    from selective_state_space_157_b300 import workloads as W

    K = w.conv_K
    x, wt, bias, state = W.conv_inputs(w.Bsz, w.L, w.D, K, seed=w.seed, with_state=True)
    es = 4
    foot = 2 * w.Bsz * w.L * w.D * es
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    copies = max(1, -(-(2 * l2) // foot))
    xs = [torch.from_numpy(x).to(dev) for _ in range(copies)]
    outs = [torch.empty_like(xs[0]) for _ in range(copies)]
    wd, bd, sd = (torch.from_numpy(a).to(dev) for a in (wt, bias, state))
    so = torch.empty_like(sd)

    def step(i):
        ss.conv1d(xs[i % copies], wd, bd, state_in=sd, out=outs[i % copies], state_out=so)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    # The steps are replayed from CUDA graphs (as in the decode workload):
    # the Python call per step takes longer than the kernel.
    per_graph = 4 * copies
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)

    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                for i in range(n):
                    step(i)
        return g

    full = capture(per_graph)
    rest = capture(args.steps % per_graph) if args.steps % per_graph else None
    stream.wait_stream(side)
    full.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world, dev)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        e0.record(stream)
        for _ in range(args.steps // per_graph):
            full.replay()
        if rest is not None:
            rest.replay()
        e1.record(stream)
        torch.cuda.synchronize()
    barrier(world, dev)
    ss.check_device_error()
    sec = max_over_ranks(e0.elapsed_time(e1) / 1e3, world, dev)
    per_step = sec / args.steps
    elems = w.Bsz * w.L * w.D
    value = world * elems * args.steps / sec

    hx = host_like(torch.from_numpy(x))
    hy = host_zeros(tuple(hx.shape), hx.dtype)
    e2e_steps = max(1, min(args.steps, 20))
    evict_host_caches()
    barrier(world, dev)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        yd, _ = ss.conv1d(hx.to(dev, non_blocking=True), wd, bd, state_in=sd, state_out=so)
        hy.copy_(yd, non_blocking=True)
        torch.cuda.current_stream().synchronize()
    t_e2e = max_over_ranks(time.perf_counter() - t0, world, dev)
    e2e = {"value": world * elems * e2e_steps / t_e2e, "unit": UNIT,
           "h2d_bytes_per_step": hx.numel() * 4, "d2h_bytes_per_step": hy.numel() * 4}
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank != 0:
        return None

    hbm_gbs, max_mhz, src = read_measured_peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    pk = peaks(sms, max_mhz, hbm_gbs, alu)
    pk["source"] = peak_source(src, alu, sms, max_mhz)
    nbytes = 2 * elems * es + w.D * (K + 1) * 4 + 2 * w.Bsz * w.D * (K - 1) * 4
    work = {"elems": elems, "updates": elems * K, "bytes": nbytes, "mufu": 2 * elems, "fp32": (K + 2) * elems}
    roof = roofline(work, pk, per_step, traffic=profiled_traffic(args.workload), kernel="selscan_conv1d (1 launch)")
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        thr = 1
        t0 = time.perf_counter()
        oracle.default().conv1d(x, wt, bias, state_in=state)
        secs = time.perf_counter() - t0
        cpu = {"value": elems / secs, "unit": UNIT, "cores": thr, "kind": "oracle",
               "sample": f"the whole workload ({elems} elements, {secs:.2f} s, fp64, one thread)"}
    config = {"workload": f"{w.name}: Bsz={w.Bsz} L={w.L} D={w.D} K={K} f32, causal depthwise conv1d + SiLU",
              "global_batch": w.Bsz * world, "seq_len": w.L, "parallelism": f"replicas x{world}",
              "l2": f"{copies} rotating input sets ({copies * foot / 1e6:.0f} MB) > 2x L2",
              "launch": f"CUDA graph replay of {per_graph} captured selscan_conv1d calls"}
    return result_line(value=value, n_gpus=world, steps=args.steps, warmup=args.warmup,
                       ms_per_step=per_step * 1e3, config=config, roof=roof, cpu=cpu, e2e=e2e,
                       launches=args.steps, clocks=clk.summary(), dtype="f32")


def run_bwd(args, world, rank, local, dev, w, alu=None):
    """The backward workload: one step = one selscan_bwd over (Bsz, L, D, N)
    with softplus on and upstream gradient dy (no dhT). Input sets rotate past
    2x L2."""
    import torch
    import selective_state_space_157_b300 as ss
    from selective_state_space_157_b300 import workloads as W

    inp = W.workload_inputs(args.workload)
    dy, _ = W.bwd_grads(w.Bsz, w.L, w.D, w.N, seed=w.seed, with_dhT=False)
    host = {k: inp.f32(k) for k in ("x", "delta", "B", "C")}
    host["dy"] = dy
    Dsk = None
    if w.gated:   # the block's skip and gate: z with the inputs, Dskip once
        Dskip, host["z"] = W.gate_inputs(w.Bsz, w.L, w.D, seed=w.seed)
        Dsk = torch.from_numpy(Dskip).to(dev)
    foot = sum(a.nbytes for a in host.values())
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    copies = max(1, -(-(2 * l2) // foot))
    sets = [{k: torch.from_numpy(a).to(dev) for k, a in host.items()} for _ in range(copies)]
    A = torch.from_numpy(inp.A).to(dev)

    def step(i):
        s = sets[i % copies]
        return ss.selscan_bwd(s["x"], s["delta"], A, s["B"], s["C"], s["dy"], True, want_dh0=False,
                              D_skip=Dsk, z=s.get("z"))

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
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
    sec = max_over_ranks(e0.elapsed_time(e1) / 1e3, world, dev)
    per_step = sec / args.steps
    elems = w.Bsz * w.L * w.D
    value = world * elems * args.steps / sec

    hin = {k: host_like(torch.from_numpy(a)) for k, a in host.items()}
    outs = {"dx": (w.Bsz, w.L, w.D), "ddelta": (w.Bsz, w.L, w.D), "dA": (w.D, w.N), "dB": (w.Bsz, w.L, w.N),
            "dC": (w.Bsz, w.L, w.N)}
    if w.gated:
        outs.update({"dz": (w.Bsz, w.L, w.D), "dD_skip": (w.D,)})
    hout = {k: host_zeros(shape) for k, shape in outs.items()}
    e2e_steps = max(1, min(args.steps, 10))
    evict_host_caches()
    barrier(world, dev)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        d = {k: t.to(dev, non_blocking=True) for k, t in hin.items()}
        g = ss.selscan_bwd(d["x"], d["delta"], A, d["B"], d["C"], d["dy"], True, want_dh0=False,
                           D_skip=Dsk, z=d.get("z"))
        for k in outs:
            hout[k].copy_(g[k], non_blocking=True)
        torch.cuda.current_stream().synchronize()
    t_e2e = max_over_ranks(time.perf_counter() - t0, world, dev)
    e2e = {"value": world * elems * e2e_steps / t_e2e, "unit": UNIT,
           "h2d_bytes_per_step": sum(t.numel() * 4 for t in hin.values()),
           "d2h_bytes_per_step": sum(t.numel() * 4 for t in hout.values())}
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank != 0:
        return None

    hbm_gbs, max_mhz, src = read_measured_peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    pk = peaks(sms, max_mhz, hbm_gbs, alu)
    pk["source"] = peak_source(src, alu, sms, max_mhz)
    work = bwd_work_counts(w.Bsz, w.L, w.D, w.N, gated=w.gated)
    roof = roofline(work, pk, per_step, traffic=profiled_traffic(args.workload),
                    kernel="bwd_local + bwd_main kernels (2 launches)")
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        t0 = time.perf_counter()
        oracle.default().selscan_bwd(host["x"], host["delta"], inp.A, host["B"], host["C"], dy, True,
                                     **({"Dskip": Dskip, "z": host["z"]} if w.gated else {}))
        secs = time.perf_counter() - t0
        cpu = {"value": elems / secs, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"the whole workload ({elems} elements, {secs:.2f} s, fp64 reverse sweep, one thread)"}
    config = {"workload": f"{w.name}: Bsz={w.Bsz} L={w.L} D={w.D} N={w.N} f32, softplus on, backward "
                          + ("of the block's gated output (dx, ddelta, dA, dB, dC, dz, dDskip from dy)" if w.gated
                             else "(dx, ddelta, dA, dB, dC from dy)"),
              "global_batch": w.Bsz * world, "seq_len": w.L, "parallelism": f"replicas x{world}",
              "l2": f"{copies} rotating input sets ({copies * foot / 1e6:.0f} MB) > 2x L2"}
    return result_line(value=value, n_gpus=world, steps=args.steps, warmup=args.warmup,
                       ms_per_step=per_step * 1e3, config=config, roof=roof, cpu=cpu, e2e=e2e,
                       launches=2 * args.steps, clocks=clk.summary(), dtype="f32")


def decode_time(w, steps, warmup, world, dev, local, eager=True):
    """Times K decode steps. Eight independent decode streams (state and
    per-step inputs each) are rotated so that every step reads its 42 MB
    state from HBM rather than L2, as a server interleaving several sequences
    would. The steps are captured in CUDA graphs and the timed steps replay
    them, as a decode loop launches a fixed step sequence. Returns (seconds
    per step, clock summary, a note with the launch form and, when ``eager``,
    the time of the same steps launched one Python call at a time)."""
    import torch
    import selective_state_space_157_b300 as ss
    from selective_state_space_157_b300 import workloads as W

    streams = 8
    A = torch.from_numpy(W.decode_A(w)).to(dev)
    states = [torch.from_numpy(W.decode_state(w)).to(dev) for _ in range(streams)]
    inputs = [[torch.from_numpy(a).to(dev) for a in W.decode_step_inputs(w, k)] for k in range(streams)]
    ys = [torch.empty(w.Bsz, w.D, device=dev) for _ in range(streams)]

    def step(i):
        x, dl, B, C = inputs[i % streams]
        ss.selscan_step(states[i % streams], x, dl, A, B, C, y=ys[i % streams])

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    ss.check_device_error()
    stream = torch.cuda.current_stream()
    # One graph holds `per_graph` consecutive steps (the streams in turn); K
    # steps replay it K // per_graph times, then a graph of the K % per_graph
    # steps that remain.
    per_graph = 4 * streams
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)

    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                for i in range(n):
                    step(i)
        return g

    full = capture(per_graph)
    rest = capture(steps % per_graph) if steps % per_graph else None
    stream.wait_stream(side)
    for _ in range(max(1, warmup // per_graph)):
        full.replay()
    torch.cuda.synchronize()

    def replay_all(_):
        for _ in range(steps // per_graph):
            full.replay()
        if rest is not None:
            rest.replay()

    note = f"CUDA graph replay of {per_graph} captured selscan_step calls (the {streams} decode streams in turn)"
    if eager:
        sec_eager, _ = timed_steps(step, steps, 0, world, dev, local)
        note += f"; one Python call per step: {sec_eager / steps * 1e6:.1f} us per step"
    sec, clocks = timed_steps(replay_all, 1, 0, world, dev, local)
    decode_time.state = (A, states, ys)
    return sec / steps, clocks, note


def run_decode(args, world, rank, local, dev, w, alu=None):
    """The decode workload: one step = one selscan_step over (Bsz, D, N),
    graph-replayed over eight rotating decode streams (decode_time)."""
    import torch
    import selective_state_space_157_b300 as ss
    from selective_state_space_157_b300 import workloads as W

    per_step, clocks, note = decode_time(w, args.steps, args.warmup, world, dev, local)
    A, states, ys = decode_time.state
    elems = w.Bsz * w.D
    value = world * elems / per_step

    # end to end: host inputs of the step in, y out, state kept on the device
    # The step's inputs packed in one page-locked host buffer and copied in
    # with one transfer into a device buffer the loop reuses, as a decode
    # loop would.
    parts = W.decode_step_inputs(w, 0)
    sizes = [a.size for a in parts]
    hx = ss.host_empty((sum(sizes),))
    dx = torch.empty(sum(sizes), device=dev)
    views, o = [], 0
    for a, n in zip(parts, sizes):
        hx[o:o + n].copy_(torch.from_numpy(a.reshape(-1)))
        views.append(dx[o:o + n].view(a.shape))
        o += n
    x, dl, B, C = views
    hy = host_zeros((w.Bsz, w.D))
    e2e_steps = max(1, min(args.steps, 50))
    evict_host_caches()
    barrier(world, dev)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        dx.copy_(hx, non_blocking=True)
        ss.selscan_step(states[0], x, dl, A, B, C, y=ys[0])
        hy.copy_(ys[0], non_blocking=True)
        torch.cuda.current_stream().synchronize()
    t_e2e = max_over_ranks(time.perf_counter() - t0, world, dev)
    e2e = {"value": world * elems * e2e_steps / t_e2e, "unit": UNIT,
           "h2d_bytes_per_step": hx.numel() * hx.element_size(),
           "d2h_bytes_per_step": hy.numel() * hy.element_size()}
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank != 0:
        return None

    hbm_gbs, max_mhz, src = read_measured_peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    pk = peaks(sms, max_mhz, hbm_gbs, alu)
    pk["source"] = peak_source(src, alu, sms, max_mhz)
    roof = roofline(step_work_counts(w.Bsz, w.D, w.N), pk, per_step, traffic=profiled_traffic(args.workload),
                    kernel="selscan_step (1 launch)")
    cpu = None
    if not args.no_cpu_baseline:
        import numpy as np
        import oracle
        chains = sample_chains(w.Bsz, w.D, 4096)
        st = W.decode_state(w).reshape(-1, w.N)[chains].astype(np.float64)
        Ah = W.decode_A(w)
        steps_h = 32
        hin = [W.decode_step_inputs(w, k) for k in range(steps_h)]
        t0 = time.perf_counter()
        for k in range(steps_h):
            oracle.selscan_step(st, *hin[k][:2], Ah, *hin[k][2:], chains=chains)
        secs = time.perf_counter() - t0
        cpu = {"value": len(chains) * steps_h / secs, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"{len(chains)} of {w.Bsz * w.D} chains x {steps_h} steps ({secs:.2f} s, fp64, one thread)"}
    config = {"workload": f"{w.name}: Bsz={w.Bsz} D={w.D} N={w.N} f32 decode step, state updated in place",
              "global_batch": w.Bsz * world, "seq_len": 1, "parallelism": f"replicas x{world}",
              "l2": f"8 rotating decode streams ({8 * w.Bsz * w.D * w.N * 4 / 1e6:.0f} MB of state) > 2x L2",
              "launch": note}
    return result_line(value=value, n_gpus=world, steps=args.steps, warmup=args.warmup,
                       ms_per_step=per_step * 1e3, config=config, roof=roof, cpu=cpu, e2e=e2e,
                       launches=args.steps, clocks=clocks, dtype="f32")


def ssd_work_counts(Bsz, L, H, P, N, elem_bytes):
    """Algorithmic work of one SSD call (chunks of Q = 64 steps).

    bytes: x read and y written (2 * B*L*H*P elements), B and C read
    (2 * B*L*N), dt (B*L*H fp32) and A (H fp32).
    tensor flops: per batch row and chunk, C B^T once (2 Q Q N, shared by the
    heads); per head and chunk the masked dual product with X (2 Q Q P), the
    incoming state's contribution C H (2 Q N P) and the chunk's state
    (B o w)^T X (2 N Q P). (The kernel recomputes C B^T for every head; that
    repeat is not counted.)"""
    Q = 64
    nch = -(-L // Q)
    nbytes = 2 * Bsz * L * H * P * elem_bytes + 2 * Bsz * L * N * elem_bytes + Bsz * L * H * 4 + H * 4
    flops = Bsz * nch * (2 * Q * Q * N + H * (2 * Q * Q * P + 4 * Q * N * P))
    return {"elems": Bsz * L * H * P, "bytes": nbytes, "flops": flops}


def run_ssd(args, world, rank, local, dev, w):
    """The Mamba-2 SSD workload: one step = one selscan_ssd_fwd over the
    pages' layer (bf16 I/O). Input sets rotate past 2x L2."""
    import numpy as np
    import torch
    import selective_state_space_157_b300 as ss
    from selective_state_space_157_b300 import workloads as W

    (x, dt, A, B, C), (Bsz, L, H, P, N) = W.ssd_workload_inputs(args.workload)
    bf16 = w.dtype == W.BF16
    tdt = torch.bfloat16 if bf16 else torch.float32
    es = 2 if bf16 else 4
    t = lambda a, d=torch.float32: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev).to(d)
    foot = 2 * Bsz * L * H * P * es + 2 * Bsz * L * N * es + Bsz * L * H * 4
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    copies = max(1, -(-(2 * l2) // foot))
    sets = [[t(x, tdt), t(dt), t(A), t(B, tdt), t(C, tdt)] for _ in range(copies)]
    ys = [torch.empty_like(s_[0]) for s_ in sets]

    def step(i):
        xs, dts, As, Bs, Cs = sets[i % copies]
        ss.ssd_fwd(xs, dts, As, Bs, Cs, True, y=ys[i % copies])

    sec, clocks = timed_steps(step, args.steps, args.warmup, world, dev, local)
    per_step = sec / args.steps
    elems = Bsz * L * H * P
    value = world * elems * args.steps / sec

    host = [host_like(torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(d))
            for a, d in ((x, tdt), (dt, torch.float32), (A, torch.float32), (B, tdt), (C, tdt))]
    hy = host_zeros(tuple(x.shape), tdt)
    e2e_steps = max(1, min(args.steps, 20))
    evict_host_caches()
    barrier(world, dev)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        d = [h_.to(dev, non_blocking=True) for h_ in host]
        yd = ss.ssd_fwd(*d, True)
        hy.copy_(yd, non_blocking=True)
        torch.cuda.current_stream().synchronize()
    t_e2e = max_over_ranks(time.perf_counter() - t0, world, dev)
    e2e = {"value": world * elems * e2e_steps / t_e2e, "unit": UNIT,
           "h2d_bytes_per_step": sum(h_.numel() * h_.element_size() for h_ in host),
           "d2h_bytes_per_step": hy.numel() * hy.element_size()}
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank != 0:
        return None

    hbm_gbs, max_mhz, src = read_measured_peaks()
    work = ssd_work_counts(Bsz, L, H, P, N, es)
    tf = read_measured_tensor_peak()
    t_hbm = work["bytes"] / (hbm_gbs * 1e9)
    t_tc = work["flops"] / (tf["tflops"] * 1e12)
    bound = "hbm" if t_hbm >= t_tc else "tensor"
    if bound == "hbm":
        achieved, peak, unit = work["bytes"] / per_step / 1e9, hbm_gbs, "GB/s"
    else:
        achieved, peak, unit = work["flops"] / per_step / 1e12, tf["tflops"], "TFLOP/s"
    roof = {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": max(t_hbm, t_tc) / per_step,
            "hbm_gbs": work["bytes"] / per_step / 1e9, "tensor_tflops": work["flops"] / per_step / 1e12,
            "t_roof_us": {"hbm": t_hbm * 1e6, "tensor": t_tc * 1e6},
            "traffic": profiled_traffic(args.workload),
            "kernel": "selscan_ssd_fwd call (3 launches: chunk states, carries, outputs)",
            "peak_source": f"HBM {src}; tensor {tf['source']}"}
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        hs = 4   # a sample of heads: the oracle's time is linear in the heads
        t0 = time.perf_counter()
        oracle.default().ssd_fwd(x[:, :, :hs], dt[:, :, :hs], A[:hs], B, C, True)
        secs = time.perf_counter() - t0
        cpu = {"value": Bsz * L * hs * P / secs, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"{hs} of {H} heads over all L ({Bsz * L * hs * P} elements, {secs:.2f} s, fp64, one thread)"}
    config = {"workload": f"{w.name}: Bsz={Bsz} L={L} H={H} P={P} N={N} {w.dtype} I/O, softplus on "
                          "(Mamba-2 SSD, fp16 tensor-core operands)",
              "global_batch": Bsz * world, "seq_len": L, "parallelism": f"replicas x{world}",
              "l2": f"{copies} rotating input sets ({copies * foot / 1e6:.0f} MB) > 2x L2"}
    return result_line(value=value, n_gpus=world, steps=args.steps, warmup=args.warmup,
                       ms_per_step=per_step * 1e3, config=config, roof=roof, cpu=cpu, e2e=e2e,
                       launches=3 * args.steps, clocks=clocks, dtype="bf16 io, f16 tensor operands, f32 accumulate"
                       if bf16 else "f32 io, f16 tensor operands, f32 accumulate")


def read_measured_tensor_peak():
    """Dense fp16 tensor throughput: MEASURED_PEAKS.json's cuBLAS bf16 burst
    figure (fp16 and bf16 share one rate on this part: nominal ratio 1)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"tflops": float(d["bf16_tflops"]), "source": "measured bf16 burst (MEASURED_PEAKS.json) x 1 for fp16"}
    return {"tflops": 1800.0, "source": "fallback 1.8 PFLOP/s bf16 burst x 1 for fp16"}


def run_reference(args, world, rank):
    """The oracle as the reference arm: each step is one oracle run over a
    bounded sample of the workload's chains, on the host cores."""
    if rank != 0:
        return None
    from selective_state_space_157_b300 import workloads as W
    w = W.WORKLOADS[args.workload]
    if w.ssd_heads:
        return run_reference_ssd(args, world, w)
    if w.steps:
        return run_reference_decode(args, world, w)
    if w.conv_K:
        return run_reference_conv(args, world, w)
    if w.backward:
        return run_reference_bwd(args, world, w)
    inp = W.workload_inputs(args.workload)
    gate = W.workload_gate_inputs(args.workload) if w.gated else None
    Bsz, L, D = inp.x.shape
    chains = sample_chains(Bsz, D, args.ref_chains)
    for _ in range(args.warmup):
        cpu_oracle_run(inp, chains, gate=gate, zoh=w.zoh)
    tot, n_total, thr = 0.0, 0, 0
    for _ in range(args.steps):
        s, n, thr = cpu_oracle_run(inp, chains, gate=gate, zoh=w.zoh)
        tot += s
        n_total += n
    value = n_total / tot
    sample = f"{len(chains)} of {Bsz * D} chains over all L={L} per step (fp64)"
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{w.name}: Bsz={Bsz} L={L} D={D} N={inp.A.shape[1]} {w.dtype}, softplus on"
                               + (", skip and SiLU gate" if w.gated else "")
                               + (", zero-order hold" if w.zoh else ""),
                   "seq_len": L, "parallelism": "host threads"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": thr, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_reference_ssd(args, world, w):
    """Reference arm for the SSD workload: each step is one oracle run over a
    sample of the heads, on the host."""
    import oracle
    from selective_state_space_157_b300 import workloads as W
    (x, dt, A, B, C), (Bsz, L, H, P, N) = W.ssd_workload_inputs(args.workload)
    hs = 4
    o = oracle.default()
    a = (x[:, :, :hs], dt[:, :, :hs], A[:hs], B, C, True)
    for _ in range(args.warmup):
        o.ssd_fwd(*a)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        o.ssd_fwd(*a)
    tot = time.perf_counter() - t0
    elems = Bsz * L * hs * P
    value = elems * args.steps / tot
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{w.name}: Bsz={Bsz} L={L} H={H} P={P} N={N}, Mamba-2 SSD", "seq_len": L,
                   "parallelism": "host thread"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{hs} of {H} heads per step ({elems} elements, fp64)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_reference_conv(args, world, w):
    """Reference arm for the conv1d workload: each step is one oracle
    convolution over the whole workload, on the host."""
    import oracle
    from selective_state_space_157_b300 import workloads as W
    x, wt, bias, state = W.conv_inputs(w.Bsz, w.L, w.D, w.conv_K, seed=w.seed, with_state=True)
    o = oracle.default()
    for _ in range(args.warmup):
        o.conv1d(x, wt, bias, state_in=state)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        o.conv1d(x, wt, bias, state_in=state)
    tot = time.perf_counter() - t0
    elems = w.Bsz * w.L * w.D
    value = elems * args.steps / tot
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{w.name}: Bsz={w.Bsz} L={w.L} D={w.D} K={w.conv_K} f32, causal depthwise conv1d + SiLU",
                   "seq_len": w.L, "parallelism": "host thread"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"the whole workload per step ({elems} elements, fp64)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_reference_bwd(args, world, w):
    """Reference arm for the backward workload: each step is one oracle
    reverse sweep over the whole workload, on the host."""
    import oracle
    from selective_state_space_157_b300 import workloads as W
    inp = W.workload_inputs(args.workload)
    dy, _ = W.bwd_grads(w.Bsz, w.L, w.D, w.N, seed=w.seed, with_dhT=False)
    a = (inp.f32("x"), inp.f32("delta"), inp.A, inp.f32("B"), inp.f32("C"), dy, True)
    kw = {}
    if w.gated:
        Dskip, z = W.gate_inputs(w.Bsz, w.L, w.D, seed=w.seed)
        kw = {"Dskip": Dskip, "z": z}
    o = oracle.default()
    for _ in range(args.warmup):
        o.selscan_bwd(*a, **kw)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        o.selscan_bwd(*a, **kw)
    tot = time.perf_counter() - t0
    elems = w.Bsz * w.L * w.D
    value = elems * args.steps / tot
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{w.name}: Bsz={w.Bsz} L={w.L} D={w.D} N={w.N} f32, softplus on, backward",
                   "seq_len": w.L, "parallelism": "host thread"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"the whole workload per step ({elems} elements, fp64)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_reference_decode(args, world, w):
    """Reference arm for the decode workload: each step is one oracle decode
    step over a sample of the chains, on the host."""
    import numpy as np
    import oracle
    from selective_state_space_157_b300 import workloads as W
    chains = sample_chains(w.Bsz, w.D, args.ref_chains * 64)
    st = W.decode_state(w).reshape(-1, w.N)[chains].astype(np.float64)
    A = W.decode_A(w)
    ins = [W.decode_step_inputs(w, k) for k in range(max(1, min(args.steps, 8)))]
    for i in range(args.warmup):
        x, dl, B, C = ins[i % len(ins)]
        oracle.selscan_step(st, x, dl, A, B, C, chains=chains)
    t0 = time.perf_counter()
    for i in range(args.steps):
        x, dl, B, C = ins[i % len(ins)]
        oracle.selscan_step(st, x, dl, A, B, C, chains=chains)
    tot = time.perf_counter() - t0
    value = len(chains) * args.steps / tot
    sample = f"{len(chains)} of {w.Bsz * w.D} chains per step (fp64, one thread)"
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{w.name}: Bsz={w.Bsz} D={w.D} N={w.N} f32 decode step", "seq_len": 1,
                   "parallelism": "host"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", type=int, default=DEFAULT_WORKLOAD, choices=list(range(1, 12)))
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true", help="skip the per_config measurements")
    ap.add_argument("--seq-len", type=int, default=None,
                    help="run a forward workload at this sequence length instead (profiling a small case)")
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
