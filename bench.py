#!/usr/bin/env python
"""Benchmark of the forward selective scan on GB300.

One step = one call of the hot path (ssm_scan_fwd through the C ABI) over one
batch of the synthetic workload, inputs resident in HBM.  Prints ONE JSON
line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--variant auto|fused|chunked|twopass] [--impl ours|reference]
                  [--op fwd|step|bwd|conv|convscan]

``--op step`` times the single-token decode step (ssm_scan_step) on the
decode workload instead: one step = one token for every sequence of the
batch, the state resident in HBM, reported against the HBM roofline.
``--op bwd`` times the backward (ssm_scan_bwd: chunk-start states, then the
reverse walk with chunk recomputation) on the forward workload.
``--op conv`` times the causal depthwise convolution + SiLU in front of the
scan (ssm_conv1d_fwd, 4 taps) on the forward workload's x, against the HBM
roofline.  ``--op convscan`` times convolution and scan in one call
(ssm_scan_fwd_conv): the convolution fused into the scan kernel, with the
separate two-kernel chain timed beside it.

N > 1 runs under torch.distributed.run, one rank per GPU: every rank scans its
own batch of the same shape (weak scaling, no data-path collective); the
elapsed time is the maximum over ranks.  ``--impl reference`` times the fp64
CPU oracle (the deliberately slow reference arm) on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "selective-scan Gelem/s (B·D·L/s) and achieved HBM GB/s as % of GB300 roofline"
UNIT = "Gelem/s"
DEFAULT_WORKLOAD = "long_seq_f32"
SMS = 152                      # GB300 streaming multiprocessors
SM_MAX_MHZ = 2070.0            # maximum SM clock
UPDATES_PER_CLK_SM = 32        # (t,d,n) updates per clock per SM: 128 FP32 lanes / 4 ops, 32 ex2/clk
HBM_FALLBACK_GBS = 6800.0
# kernels this library launches per step: fused = B/C re-layout + scan;
# two-pass = re-layout + pass 1 + segment carry + pass 2; chunked = B/C chunk
# re-layout + scan
KERNELS_PER_STEP = {"fused": 2, "chunked": 2, "twopass": 4}
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "dram_traffic.json")
_FUSED_SOURCES = ["selective_state_space_02_gb300/csrc/scan_fused_impl.cuh",
                  "selective_state_space_02_gb300/csrc/scan_fused_dispatch.cuh",
                  "selective_state_space_02_gb300/csrc/scan_fused.cu",
                  "selective_state_space_02_gb300/csrc/scan_device.cuh",
                  "selective_state_space_02_gb300/csrc/scan_tma.cuh"]
KERNEL_SOURCES = {
    "fused": _FUSED_SOURCES,
    "twopass": _FUSED_SOURCES,
    "chunked": ["selective_state_space_02_gb300/csrc/scan_chunked.cu",
                "selective_state_space_02_gb300/csrc/scan_device.cuh",
                "selective_state_space_02_gb300/csrc/scan_tma.cuh"],
}


# ----------------------------------------------------------------- helpers
def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--variant", default="auto")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--flush-mib", type=int, default=512, help="L2 flush buffer written between timed steps")
    ap.add_argument("--soak-s", type=float, default=1.0, help="untimed load before the timed region (clock sampling)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-parity", action="store_true", help="skip the all-element check against the oracle")
    ap.add_argument("--op", default="fwd", choices=["fwd", "step", "bwd", "conv", "convscan"])
    ap.add_argument("--seqlen", type=int, default=None,
                    help="run the workload's shape with this sequence length instead (smaller cases for profiler "
                         "captures; the line's config reports it)")
    a = ap.parse_args(argv)
    if a.warmup < 3:
        ap.error("--warmup must be at least 3")
    return a


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Largest `value` over all ranks (the job's elapsed time)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(base_seed: int, rank: int) -> int:
    """Each rank scans its own batch: same shape, different seeded data."""
    return base_seed + 1000003 * rank


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    except Exception:
        return HBM_FALLBACK_GBS, "fallback"


def alu_peak_updates_per_s() -> float:
    return SMS * SM_MAX_MHZ * 1e6 * UPDATES_PER_CLK_SM


def source_hash(variant: str) -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES.get(variant, []):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, variant: str):
    """DRAM bytes per step (all of the step's kernels) from the committed ncu
    summary, or None when the kernel sources changed since the counters were
    taken."""
    try:
        with open(PROFILE_TRAFFIC) as f:
            j = json.load(f)
        e = j[workload][variant]
        if e.get("source_hash") != source_hash(variant):
            return None
        return e["dram_bytes_per_step"]
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples while the GPU is busy."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None
        try:
            import torch
            pr = torch.cuda.get_device_properties(device_index)
            self.pci = f"{pr.pci_domain_id:08X}:{pr.pci_bus_id:02X}:{pr.pci_device_id:02X}.0"
        except Exception:
            self.pci = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if self.pci:
            cmd += ["-i", self.pci]
        try:
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        # wait for the first sample so the load phase is covered
        deadline = time.time() + 3.0
        while self.proc and time.time() < deadline and os.path.getsize(self.path) == 0:
            time.sleep(0.05)
        self.t0 = time.time()

    def stop(self):
        self.t1 = time.time()
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        rows = []
        try:
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 8:
                    rows.append(parts)
            os.unlink(self.path)
        except Exception:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        sm = [float(r[0]) for r in rows if r[0].replace(".", "", 1).isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "", 1).isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].lower() == "active"})
        pw = [float(r[2]) for r in rows if r[2].replace(".", "", 1).isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons,
                "power_w_max": max(pw) if pw else None,
                "samples": len(rows)}


# Bytes of L2 per GPU (GB300: 129 MB) when the device does not report it.
L2_FALLBACK_BYTES = 129 * 10**6

L2_NOTE = ("flushed between timed steps: a {mib} MiB write, then a read of the same buffer so that no "
           "dirty line of it is left to be written back during the timed kernel; outside the timed events")


def flush_l2(buf):
    """Evict the workload from L2: write a buffer larger than L2, then read
    it back so that L2 ends up holding clean lines of that buffer (the write
    alone would leave ~129 MB of dirty lines whose write-back lands inside
    the next timed step)."""
    buf.zero_()
    buf.view(-1).max()


# --seqlen: the workloads' shapes with another sequence length
SEQLEN_OVERRIDE = None


def workload_problem(name: str, rank: int):
    from selective_state_space_02_gb300 import synth
    cfg = dict(synth.WORKLOADS[name])
    cfg["seed"] = rank_seed(cfg["seed"], rank)
    if SEQLEN_OVERRIDE:
        cfg["seqlen"] = SEQLEN_OVERRIDE
    return synth.make_problem(**cfg), cfg


def _oracle_arrays(p):
    return dict(x=p.f32("x"), delta=p.f32("delta"), A=p.A.numpy(), B=p.f32("B"), C=p.f32("C"),
                D=None if p.D is None else p.D.numpy(), z=p.f32("z"),
                dt_bias=None if p.dt_bias is None else p.dt_bias.numpy())


def oracle_full(p):
    """The fp64 oracle over every channel of the workload on all host cores:
    (y, final_state, seconds, threads)."""
    import oracle
    oracle.build()
    a = _oracle_arrays(p)
    threads = oracle.max_threads()
    t = time.perf_counter()
    y, fs = oracle.fwd(a["x"], a["delta"], a["A"], a["B"], a["C"], a["D"], a["z"], a["dt_bias"], p.delta_softplus,
                       return_final_state=True)
    return y, fs, time.perf_counter() - t, threads


def _single_thread_oracle(p, arrs, budget_s: float = 5.0):
    """The fp64 oracle on one host thread over a bounded sample of whole
    channels (every step)."""
    import numpy as np
    import oracle
    nch = p.batch * p.dim
    probe = list(range(min(nch, 2)))
    t = time.perf_counter()
    oracle.fwd(arrs["x"], arrs["delta"], arrs["A"], arrs["B"], arrs["C"], arrs["D"], arrs["z"],
               arrs["dt_bias"], p.delta_softplus, channels=probe, nthreads=1, return_final_state=False)
    per_chan = (time.perf_counter() - t) / len(probe)
    k = int(min(nch, max(len(probe), budget_s / max(per_chan, 1e-9))))
    chans = list(range(k)) if k == nch else sorted(np.random.default_rng(1).choice(nch, k, replace=False).tolist())
    t = time.perf_counter()
    oracle.fwd(arrs["x"], arrs["delta"], arrs["A"], arrs["B"], arrs["C"], arrs["D"], arrs["z"],
               arrs["dt_bias"], p.delta_softplus, channels=chans, nthreads=1, return_final_state=False)
    dt = time.perf_counter() - t
    return {"value": k * p.seqlen / dt / 1e9, "unit": UNIT, "cores": 1,
            "sample": ("whole workload" if k == nch else f"{k} of {nch} channels") + f", all {p.seqlen} steps ({dt:.2f} s)"}


def cpu_baseline(p, max_seconds: float = 20.0, full=None):
    """Time the fp64 oracle on the host cores over a bounded sample of the
    workload (whole channels, every step), and on one thread beside it.
    ``full`` is a finished pass over the whole workload (from the parity
    check), used when it stayed within the time bound."""
    import numpy as np
    import oracle
    oracle.build()
    nch = p.batch * p.dim
    arrs = _oracle_arrays(p)
    one = _single_thread_oracle(p, arrs)
    if full is not None and full[2] <= 1.5 * max_seconds:
        dt, threads = full[2], full[3]
        return {"value": p.elems / dt / 1e9, "unit": UNIT, "cores": threads, "kind": "oracle",
                "sample": f"whole workload, all {p.seqlen} steps, one pass ({dt:.2f} s)", "single_thread": one}
    threads = oracle.max_threads()
    # calibrate on a few channels, then size the sample to ~max_seconds / 2
    probe = list(range(min(nch, max(threads, 8))))
    t = time.perf_counter()
    oracle.fwd(arrs["x"], arrs["delta"], arrs["A"], arrs["B"], arrs["C"], arrs["D"], arrs["z"],
               arrs["dt_bias"], p.delta_softplus, channels=probe, return_final_state=False)
    per_chan = (time.perf_counter() - t) / len(probe)
    k = int(min(nch, max(len(probe), (max_seconds / 2) / max(per_chan, 1e-9))))
    chans = list(range(k)) if k == nch else sorted(np.random.default_rng(0).choice(nch, k, replace=False).tolist())
    t = time.perf_counter()
    oracle.fwd(arrs["x"], arrs["delta"], arrs["A"], arrs["B"], arrs["C"], arrs["D"], arrs["z"],
               arrs["dt_bias"], p.delta_softplus, channels=chans, return_final_state=False)
    dt = time.perf_counter() - t
    elems = k * p.seqlen
    sample = ("whole workload" if k == nch else f"{k} of {nch} channels") + \
        f", all {p.seqlen} steps, one pass ({dt:.2f} s)"
    return {"value": elems / dt / 1e9, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample,
            "single_thread": one}


PARITY_TOL = {"f32": 1e-4, "bf16": 2e-2}


def parity_check(p, y_dev, fs_dev, full):
    """Every element of y (and of the final state, when returned) against the
    oracle: the largest |got - ref| / (1 + |ref|), against the tolerance."""
    import numpy as np
    yr, fr = full[0], full[1]
    nch = p.batch * p.dim
    yg = y_dev.float().cpu().numpy().reshape(nch, p.seqlen).astype(np.float64)
    err = float(np.max(np.abs(yg - yr) / (1.0 + np.abs(yr)))) if yr.size else 0.0
    out = {"oracle": "fp64 CPU recurrence, every element", "elements": int(yr.size),
           "y_max_scaled_err": err, "y_tol": PARITY_TOL[p.dtype]}
    ok = err <= PARITY_TOL[p.dtype]
    if fs_dev is not None:
        fg = fs_dev.cpu().numpy().reshape(nch, p.dstate).astype(np.float64)
        ferr = float(np.max(np.abs(fg - fr) / (1.0 + np.abs(fr)))) if fr.size else 0.0
        out.update({"final_state_max_scaled_err": ferr, "final_state_tol": 1e-4})
        ok = ok and ferr <= 1e-4
    out["ok"] = bool(ok)
    return out


# ------------------------------------------------------------- our arm
def run_ours(args):
    import torch
    import selective_state_space_02_gb300 as ssm
    from selective_state_space_02_gb300 import synth

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    dev = torch.device("cuda", local)
    p, cfg = workload_problem(args.workload, rank)
    g = lambda t: None if t is None else t.to(dev)
    x, dl, z, B, C, A, D, bias = (g(p.x), g(p.delta), g(p.z), g(p.B), g(p.C), g(p.A), g(p.D), g(p.dt_bias))
    variant = args.variant if args.variant != "auto" else ssm.select_variant(
        p.batch, p.dim, p.dstate, p.seqlen, p.torch_dtype)
    y = torch.empty_like(x)
    fs = torch.empty(p.batch, p.dim, p.dstate, device=dev) if p.final_state else None
    wsb = ssm.workspace_size(p.batch, p.dim, p.dstate, p.seqlen, p.torch_dtype, variant)
    ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev)
    flush = torch.empty(args.flush_mib << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        ssm.scan_fwd(x, dl, A, B, C, D=D, z=z, dt_bias=bias, delta_softplus=p.delta_softplus,
                     return_final_state=fs is not None, variant=variant, y=y, final_state=fs, workspace=ws)

    for _ in range(args.warmup):
        flush_l2(flush)
        step()
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    t_end = time.time() + args.soak_s
    while time.time() < t_end:          # untimed load: clocks settle, sampler sees the load
        for _ in range(20):
            flush_l2(flush)
            step()
        torch.cuda.synchronize()

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush_l2(flush)                 # L2 flush, outside the timed events
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]     # ms per step (device)
    total_ms = max_over_ranks(sum(per), world, dev)
    ms_per_step = total_ms / args.steps
    elems = p.elems
    value = world * elems * args.steps / (total_ms / 1e3) / 1e9

    hbm_peak, peak_kind = measured_peaks()
    mb = synth.min_bytes(p)
    kern_s = statistics.mean(per) / 1e3
    hbm_gbs = mb / kern_s / 1e9
    updates = elems * p.dstate
    alu_achieved = updates / kern_s
    alu_peak = alu_peak_updates_per_s()
    traffic = None if SEQLEN_OVERRIDE else profiled_traffic(args.workload, variant)
    roofline = {
        "bound": "alu",
        "achieved": round(alu_achieved / 1e12, 4),
        "peak": round(alu_peak / 1e12, 4),
        "unit": "Tupdate/s",
        "frac": round(alu_achieved / alu_peak, 4),
        "traffic": traffic,
        "kernel": {"fused": "fused scan step: B/C re-layout (~3%) and the scan kernel",
                   "twopass": "two-pass scan step: B/C re-layout, totals pass, segment carry, seeded pass "
                              "(all four launches; achieved and traffic per step)",
                   "chunked": "chunked scan step: B/C chunk re-layout and the scan kernel"}[variant],
        "traffic_note": "DRAM bytes of all the step's kernels from one ncu capture; y lines still dirty in L2 "
                        "when the last kernel ends are written back after it and are not counted",
        "peak_basis": f"{SMS} SMs x {SM_MAX_MHZ:.0f} MHz x {UPDATES_PER_CLK_SM} (t,d,n) updates/clk/SM "
                      "(1 ex2 + 4 FP32 ops per update; 32 ex2 and 128 FP32 lanes per clk per SM)",
        "hbm": {"achieved": round(hbm_gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(hbm_gbs / hbm_peak, 4), "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
                "algorithmic_bytes_per_launch": mb},
    }

    e2e = None
    if not args.no_e2e:
        pin = lambda t: None if t is None else t.pin_memory()
        hx, hdl, hz, hB, hC, hA, hD, hb = (pin(p.x), pin(p.delta), pin(p.z), pin(p.B), pin(p.C), pin(p.A),
                                           pin(p.D), pin(p.dt_bias))
        hy = torch.empty_like(hx).pin_memory()
        hfs = torch.empty(p.batch, p.dim, p.dstate).pin_memory() if p.final_state else None
        need = ssm.host_buffer_size(p.batch, p.dim, p.dstate, p.seqlen, p.torch_dtype, hD is not None,
                                    hz is not None, hb is not None, hfs is not None, variant)
        dbuf = torch.empty(need, dtype=torch.uint8, device=dev)

        def hstep():
            ssm.scan_fwd_host(hx, hdl, hA, hB, hC, D=hD, z=hz, dt_bias=hb, delta_softplus=p.delta_softplus,
                              y=hy, final_state=hfs, device_buffer=dbuf, variant=variant, stream=stream)

        for _ in range(args.warmup):
            hstep()
        barrier(world)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            hstep()
        t_e2e = max_over_ranks(time.perf_counter() - t0, world, dev)
        h2d = sum(t.numel() * t.element_size() for t in (hx, hdl, hz, hB, hC, hA, hD, hb) if t is not None)
        d2h = hy.numel() * hy.element_size() + (hfs.numel() * 4 if hfs is not None else 0)
        e2e = {"value": world * elems * args.steps / t_e2e / 1e9, "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "api": "ssm_scan_fwd_host (pinned host buffers, copies inside the timed region)"}

    full = None
    parity = None
    if rank == 0 and (not args.no_parity or (world == 1 and not args.no_cpu_baseline)):
        full = oracle_full(p)
    if rank == 0 and not args.no_parity:
        # rank 0's y (and final state) of the last timed step, checked outside the timed region
        parity = parity_check(p, y, fs, full)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(p, full=full)

    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload, "batch": p.batch, "dim": p.dim, "dstate": p.dstate,
                   "seqlen": p.seqlen, "io_dtype": p.dtype, "gate": p.z is not None,
                   "final_state": p.final_state, "variant": variant,
                   "l2": L2_NOTE.format(mib=args.flush_mib),
                   "parallelism": f"{world} independent replicas, one batch each" if world > 1 else "single GPU"},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "parity": parity,
        "clocks": {k: clocks.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons", "samples", "power_w_max")},
        "gpu_launches": args.steps * KERNELS_PER_STEP[variant],
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------ reference arm
def run_reference(args):
    rank, world, local = dist_env()
    if rank != 0:
        return
    import oracle
    from selective_state_space_02_gb300 import synth
    oracle.build()
    p, cfg = workload_problem(args.workload, 0)
    import numpy as np
    nch = p.batch * p.dim
    arrs = (p.f32("x"), p.f32("delta"), p.A.numpy(), p.f32("B"), p.f32("C"),
            None if p.D is None else p.D.numpy(), p.f32("z"),
            None if p.dt_bias is None else p.dt_bias.numpy())
    threads = oracle.max_threads()
    # size one step to about 1 s of host work so K + W steps stay within minutes
    probe = list(range(min(nch, max(threads, 8))))
    t = time.perf_counter()
    oracle.fwd(*arrs, p.delta_softplus, channels=probe, return_final_state=False)
    per_chan = (time.perf_counter() - t) / len(probe)
    k = int(min(nch, max(len(probe), 1.0 / max(per_chan, 1e-9))))
    rng = np.random.default_rng(1)
    steps = []
    for i in range(args.warmup + args.steps):
        chans = sorted(rng.choice(nch, k, replace=False).tolist()) if k < nch else None
        t = time.perf_counter()
        oracle.fwd(*arrs, p.delta_softplus, channels=chans, return_final_state=False)
        if i >= args.warmup:
            steps.append(time.perf_counter() - t)
    total = sum(steps)
    value = k * p.seqlen * args.steps / total / 1e9
    sample = f"{k} of {nch} channels per step (all {p.seqlen} steps each)"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": args.workload, "batch": p.batch, "dim": p.dim, "dstate": p.dstate,
                   "seqlen": p.seqlen, "io_dtype": p.dtype, "gate": p.z is not None},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------ decode step
STEP_METRIC = "decode step: channel-tokens/s (B·D per step) and achieved HBM GB/s as % of GB300 roofline"
STEP_UNIT = "Gtoken-channels/s"


def step_problem(name: str, rank: int):
    from selective_state_space_02_gb300 import synth
    cfg = dict(synth.STEP_WORKLOADS[name])
    cfg["seed"] = rank_seed(cfg["seed"], rank)
    p = synth.make_problem(**cfg)
    return p, synth.make_state(p.batch, p.dim, p.dstate, seed=cfg["seed"] + 1)


def step_cpu_baseline(p, h0, reps: int = 3):
    """The fp64 oracle step over the whole decode batch, a few times."""
    import oracle
    from selective_state_space_02_gb300 import synth
    oracle.build()
    s = synth.step_inputs(p, 0)
    f = lambda v: None if v is None else v.float().numpy()
    h = h0.numpy().astype("float64")
    t = time.perf_counter()
    for _ in range(reps):
        h, _ = oracle.step(h, f(s["x"]), f(s["delta"]), p.A.numpy(), f(s["B"]), f(s["C"]),
                           None if p.D is None else p.D.numpy(), f(s["z"]),
                           None if p.dt_bias is None else p.dt_bias.numpy(), p.delta_softplus)
    dt = (time.perf_counter() - t) / reps
    return {"value": p.batch * p.dim / dt / 1e9, "unit": STEP_UNIT, "cores": 1, "kind": "oracle",
            "sample": f"whole decode batch ({p.batch} x {p.dim} channels), {reps} steps, serial"}


def run_step(args):
    import torch
    import selective_state_space_02_gb300 as ssm
    from selective_state_space_02_gb300 import synth

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    dev = torch.device("cuda", local)
    name = args.workload if args.workload in synth.STEP_WORKLOADS else "decode_bf16"
    p, h0 = step_problem(name, rank)
    # one token through `copies` layers: every step has its own state and
    # token inputs, together more than twice the L2, so no step finds its
    # data in L2 and the steps run back to back between one pair of events
    one = {k: v for k, v in synth.step_inputs(p, 0).items()}
    per_copy = h0.numel() * 4 + sum(v.numel() * v.element_size() for k, v in one.items()
                                    if v is not None and k in ("x", "delta", "z"))
    L2_BYTES = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or L2_FALLBACK_BYTES
    copies = max(2, -(-(2 * L2_BYTES) // per_copy))
    ins = [{k: (v.to(dev) if v is not None else None) for k, v in one.items()} for _ in range(copies)]
    states = [h0.to(dev) for _ in range(copies)]
    ys = [torch.empty_like(ins[0]["x"]) for _ in range(copies)]
    s, state, y = ins[0], states[0], ys[0]
    stream = torch.cuda.current_stream(dev)

    def layer(i):
        c = ins[i]
        ssm.scan_step(states[i], c["x"], c["delta"], c["A"], c["B"], c["C"], D=c["D"], z=c["z"], dt_bias=c["dt_bias"],
                      delta_softplus=p.delta_softplus, y=ys[i])

    def step():
        layer(0)

    for i in range(max(args.warmup, 3) * copies):
        layer(i % copies)
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    t_end = time.time() + args.soak_s
    while time.time() < t_end:
        for i in range(20 * copies):
            layer(i % copies)
        torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(args.steps):
        layer(i % copies)
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    total_ms = max_over_ranks(start.elapsed_time(end), world, dev)
    per = [total_ms / args.steps]
    # the same layers captured once in a CUDA graph (one token through all of
    # them) and replayed: the launch-free form of a decode loop
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for i in range(copies):
            layer(i)
    stream.wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(copies):
            layer(i)
    replays = max(1, args.steps // copies)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(replays):
        graph.replay()
    g1.record(stream)
    torch.cuda.synchronize()
    graph_ms = g0.elapsed_time(g1) / (replays * copies)
    chans = p.batch * p.dim
    value = world * chans * args.steps / (total_ms / 1e3) / 1e9
    hbm_peak, peak_kind = measured_peaks()
    mb = synth.step_min_bytes(p)
    kern_s = statistics.mean(per) / 1e3
    roofline = {"bound": "hbm", "achieved": round(mb / kern_s / 1e9, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(mb / kern_s / 1e9 / hbm_peak, 4), "traffic": None,
                "kernel": "decode step (ssm_scan_step)", "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
                "algorithmic_bytes_per_launch": mb}
    e2e = None
    if not args.no_e2e:
        pin = lambda t: None if t is None else t.pin_memory()
        hs = {k: pin(v) for k, v in synth.step_inputs(p, 0).items()
              if k in ("x", "delta", "z", "B", "C") and v is not None}
        hy = torch.empty_like(hs["x"]).pin_memory()

        def hstep():
            for k, v in hs.items():
                s[k].copy_(v, non_blocking=True)
            step()
            hy.copy_(y, non_blocking=True)
            stream.synchronize()

        for _ in range(args.warmup):
            hstep()
        barrier(world)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            hstep()
        t_e2e = max_over_ranks(time.perf_counter() - t0, world, dev)
        e2e = {"value": world * chans * args.steps / t_e2e / 1e9, "unit": STEP_UNIT,
               "h2d_bytes_per_step": sum(v.numel() * v.element_size() for v in hs.values()),
               "d2h_bytes_per_step": hy.numel() * hy.element_size(),
               "api": "scan_step with the token's inputs copied from pinned host memory and y copied back"}
    cpu = step_cpu_baseline(p, h0) if rank == 0 and world == 1 and not args.no_cpu_baseline else None
    line = {
        "metric": STEP_METRIC, "value": round(value, 3), "unit": STEP_UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": name, "batch": p.batch, "dim": p.dim, "dstate": p.dstate, "io_dtype": p.dtype,
                   "gate": p.z is not None,
                   "l2": f"inputs larger than L2: the timed steps cycle over {copies} state and token-input sets "
                         f"({copies * per_copy / 2**20:.0f} MiB in all, {2 * L2_BYTES / 2**20:.0f} MiB = twice the "
                         "L2 at least), back to back between one pair of CUDA events",
                   "parallelism": f"{world} independent replicas" if world > 1 else "single GPU"},
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        "clocks": {k: clocks.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons", "samples", "power_w_max")},
        "gpu_launches": args.steps,
        "graph": {"ms_per_step": round(graph_ms, 5),
                  "achieved_gbs": round(synth.step_min_bytes(p) / (graph_ms / 1e3) / 1e9, 1),
                  "note": f"the {copies} layers of one token captured once in a CUDA graph and replayed "
                          f"{replays} times (launch-free decode loop); the line's value is the direct calls"},
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------------ backward
BWD_METRIC = "selective-scan backward Gelem/s (B·D·L/s)"


def bwd_min_bytes(p) -> int:
    """Bytes the backward must move at least: the forward's inputs (x, delta,
    z, B, C in the I/O dtype; A, D, dt_bias) and dy read once; dx, ddelta,
    dz written in the I/O dtype, dB and dC in float32, dA, dD, ddt_bias."""
    e = 2 if p.dtype == "bf16" else 4
    z = 1 if p.z is not None else 0
    n = p.batch * p.dim * p.seqlen * e * ((3 + z) + (2 + z))   # x, delta, dy, (z) in; dx, ddelta, (dz) out
    n += 2 * p.batch * p.dstate * p.seqlen * e + 2 * p.batch * p.dstate * p.seqlen * 4
    n += 2 * p.dim * p.dstate * 4 + 4 * p.dim * 4
    return n


def run_bwd(args):
    import torch
    import numpy as np
    import selective_state_space_02_gb300 as ssm
    from selective_state_space_02_gb300 import synth

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    dev = torch.device("cuda", local)
    p, cfg = workload_problem(args.workload, rank)
    g = lambda t: None if t is None else t.to(dev)
    x, dl, z, B, C, A, D, bias = (g(p.x), g(p.delta), g(p.z), g(p.B), g(p.C), g(p.A), g(p.D), g(p.dt_bias))
    dy = torch.from_numpy(np.random.default_rng(cfg["seed"] + 7).standard_normal(
        (p.batch, p.dim, p.seqlen)).astype(np.float32)).to(p.torch_dtype)
    ddy = dy.to(dev)
    wsb = ssm._native.load().ssm_scan_bwd_workspace_size(p.batch, p.dim, p.dstate, p.seqlen,
                                                          ssm._dtype_code(p.torch_dtype))
    ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev)
    flush = torch.empty(args.flush_mib << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        return ssm.scan_bwd(x, dl, A, B, C, ddy, D=D, z=z, dt_bias=bias, delta_softplus=p.delta_softplus,
                            workspace=ws)

    for _ in range(args.warmup):
        flush_l2(flush)
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    t_end = time.time() + args.soak_s
    while time.time() < t_end:
        for _ in range(5):
            flush_l2(flush)
            step()
        torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush_l2(flush)
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    per = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    total_ms = max_over_ranks(sum(per), world, dev)
    elems = p.elems
    value = world * elems * args.steps / (total_ms / 1e3) / 1e9
    hbm_peak, peak_kind = measured_peaks()
    kern_s = statistics.mean(per) / 1e3
    mb = bwd_min_bytes(p)
    bwd_kernels = ssm._native.load().ssm_scan_bwd_kernel_count(p.batch, p.dim, p.dstate, p.seqlen)
    updates = elems * p.dstate
    alu_peak = alu_peak_updates_per_s()
    roofline = {"bound": "alu", "achieved": round(updates / kern_s / 1e12, 4), "peak": round(alu_peak / 1e12, 4),
                "unit": "Tupdate/s", "frac": round(updates / kern_s / alu_peak, 4), "traffic": None,
                "kernel": "backward (B/C re-layout, chunk-start states, reverse walk)",
                "peak_basis": f"{SMS} SMs x {SM_MAX_MHZ:.0f} MHz x {UPDATES_PER_CLK_SM} (t,d,n) updates/clk/SM, "
                              "one ex2 per update (the backward evaluates three: the chunk-start states pass, "
                              "the chunk recomputation and the adjoint)",
                "hbm": {"achieved": round(mb / kern_s / 1e9, 1), "peak": hbm_peak, "unit": "GB/s",
                        "frac": round(mb / kern_s / 1e9 / hbm_peak, 4),
                        "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
                        "algorithmic_bytes_per_launch": mb}}
    e2e = None
    if not args.no_e2e:
        pin = lambda t: None if t is None else t.pin_memory()
        hin = {"x": (pin(p.x), x), "delta": (pin(p.delta), dl), "z": (pin(p.z), z), "B": (pin(p.B), B),
               "C": (pin(p.C), C), "dy": (pin(dy), ddy)}
        hin = {k: v for k, v in hin.items() if v[0] is not None}
        outs = {}

        def hstep():
            for hsrc, ddst in hin.values():
                ddst.copy_(hsrc, non_blocking=True)
            grads = step()
            for k in ("dx", "ddelta", "dz", "dB", "dC"):
                if grads.get(k) is not None:
                    if k not in outs:
                        outs[k] = torch.empty(grads[k].shape, dtype=grads[k].dtype).pin_memory()
                    outs[k].copy_(grads[k], non_blocking=True)
            stream.synchronize()

        for _ in range(args.warmup):
            hstep()
        barrier(world)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            hstep()
        t_e2e = max_over_ranks(time.perf_counter() - t0, world, dev)
        e2e = {"value": world * elems * args.steps / t_e2e / 1e9, "unit": UNIT,
               "h2d_bytes_per_step": sum(v[0].numel() * v[0].element_size() for v in hin.values()),
               "d2h_bytes_per_step": sum(v.numel() * v.element_size() for v in outs.values()),
               "api": "scan_bwd with its inputs copied from pinned host memory and the gradients copied back"}
    # The training pair, timed after the line's own region: a forward that
    # stores the chunk-start states with the backward from them
    # (ssm_scan_fwd_ckpt + ssm_scan_bwd_ckpt), against the forward followed by
    # the backward that computes them again; L2 flushed before each pair.
    lib = ssm._native.load()
    code = ssm._dtype_code(p.torch_dtype)
    sizes = (p.batch, p.dim, p.dstate, p.seqlen, code)
    u8 = lambda n: torch.empty(max(n, 1), dtype=torch.uint8, device=dev)
    fws, fwc, bwc = (u8(lib.ssm_scan_fwd_workspace_size(*sizes, 0)), u8(lib.ssm_scan_fwd_ckpt_workspace_size(*sizes, 0)),
                     u8(lib.ssm_scan_bwd_ckpt_workspace_size(*sizes)))
    fkw = dict(D=D, z=z, dt_bias=bias, delta_softplus=p.delta_softplus, y=torch.empty_like(x))
    bkw = dict(D=D, z=z, dt_bias=bias, delta_softplus=p.delta_softplus, workspace=bwc)

    def pair_plain():
        ssm.scan_fwd(x, dl, A, B, C, workspace=fws, **fkw)
        step()

    def pair_ckpt():
        _, ck = ssm.scan_fwd(x, dl, A, B, C, workspace=fwc, return_ckpt=True, **fkw)
        ssm.scan_bwd(x, dl, A, B, C, ddy, ckpt=ck, **bkw)

    _, ck0 = ssm.scan_fwd(x, dl, A, B, C, workspace=fwc, return_ckpt=True, **fkw)
    t_plain = statistics.mean(_timed_steps(pair_plain, args, flush, stream, world))
    t_ckpt = statistics.mean(_timed_steps(pair_ckpt, args, flush, stream, world))
    t_bwd_ckpt = statistics.mean(_timed_steps(lambda: ssm.scan_bwd(x, dl, A, B, C, ddy, ckpt=ck0, **bkw),
                                              args, flush, stream, world))
    training = {"fwd_then_bwd_ms": round(t_plain, 5), "fwd_ckpt_then_bwd_ckpt_ms": round(t_ckpt, 5),
                "bwd_from_ckpt_ms": round(t_bwd_ckpt, 5),
                "note": "ms per pair (CUDA events, rank 0); the forward with checkpoints stores the state at every "
                        "32-step chunk start and the backward from them skips its chunk-start states pass"}
    line = {
        "metric": BWD_METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload, "batch": p.batch, "dim": p.dim, "dstate": p.dstate,
                   "seqlen": p.seqlen, "io_dtype": p.dtype, "gate": p.z is not None,
                   "l2": L2_NOTE.format(mib=args.flush_mib),
                   "parallelism": f"{world} independent replicas" if world > 1 else "single GPU"},
        "roofline": roofline, "cpu_baseline": None, "e2e": e2e,
        "clocks": {k: clocks.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons", "samples", "power_w_max")},
        "gpu_launches": args.steps * bwd_kernels,
        "training_step": training,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------- convolution
CONV_METRIC = "causal depthwise conv1d + SiLU: Gelem/s (B·D·L/s) and achieved HBM GB/s as % of GB300 roofline"
CONV_WIDTH = 4


def run_conv(args):
    import torch
    import selective_state_space_02_gb300 as ssm
    from selective_state_space_02_gb300 import synth

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    dev = torch.device("cuda", local)
    p, cfg = workload_problem(args.workload, rank)
    w, b = synth.make_conv(p.dim, CONV_WIDTH, seed=cfg["seed"] + 11)
    w, b = w.to(dev), b.to(dev)
    # the timed calls cycle over input and output sets that together exceed
    # twice the L2, back to back between one pair of events (a short call
    # timed alone sits within the events' resolution of about 2 us)
    per_copy = 2 * p.x.numel() * p.x.element_size()
    L2_BYTES = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or L2_FALLBACK_BYTES
    copies = max(2, -(-(2 * L2_BYTES) // per_copy))
    xs = [p.x.to(dev) for _ in range(copies)]
    ys = [torch.empty_like(xs[0]) for _ in range(copies)]
    souts = [torch.empty((p.batch, p.dim, CONV_WIDTH - 1), dtype=xs[0].dtype, device=dev) for _ in range(copies)]
    x, y = xs[0], ys[0]
    stream = torch.cuda.current_stream(dev)

    def call(i):
        ssm.conv1d(xs[i], w, b, silu=True, y=ys[i], state_out=souts[i])

    def step():
        call(0)

    for i in range(max(args.warmup, 3) * copies):
        call(i % copies)
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    t_end = time.time() + args.soak_s
    while time.time() < t_end:
        for i in range(5 * copies):
            call(i % copies)
        torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(args.steps):
        call(i % copies)
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    total_ms = max_over_ranks(start.elapsed_time(end), world, dev)
    per = [total_ms / args.steps]
    elems = p.elems
    value = world * elems * args.steps / (total_ms / 1e3) / 1e9
    hbm_peak, peak_kind = measured_peaks()
    e = x.element_size()
    mb = 2 * elems * e + p.dim * (CONV_WIDTH + 1) * 4 + p.batch * p.dim * (CONV_WIDTH - 1) * e
    kern_s = statistics.mean(per) / 1e3
    roofline = {"bound": "hbm", "achieved": round(mb / kern_s / 1e9, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(mb / kern_s / 1e9 / hbm_peak, 4), "traffic": None,
                "kernel": "conv1d (ssm_conv1d_fwd)", "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
                "algorithmic_bytes_per_launch": mb}
    e2e = None
    if not args.no_e2e:
        hx = p.x.pin_memory()
        hy = torch.empty_like(hx).pin_memory()

        def hstep():
            x.copy_(hx, non_blocking=True)
            step()
            hy.copy_(y, non_blocking=True)
            stream.synchronize()

        for _ in range(args.warmup):
            hstep()
        barrier(world)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            hstep()
        t_e2e = max_over_ranks(time.perf_counter() - t0, world, dev)
        e2e = {"value": world * elems * args.steps / t_e2e / 1e9, "unit": UNIT,
               "h2d_bytes_per_step": hx.numel() * hx.element_size(),
               "d2h_bytes_per_step": hy.numel() * hy.element_size(),
               "api": "conv1d with x copied from pinned host memory and y copied back"}
    line = {
        "metric": CONV_METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload, "batch": p.batch, "dim": p.dim, "seqlen": p.seqlen,
                   "width": CONV_WIDTH, "io_dtype": p.dtype, "silu": True,
                   "l2": f"inputs larger than L2: the timed calls cycle over {copies} sets of x and y "
                         f"({copies * per_copy / 2**20:.0f} MiB in all), back to back between one pair of CUDA events",
                   "parallelism": f"{world} independent replicas" if world > 1 else "single GPU"},
        "roofline": roofline, "cpu_baseline": None, "e2e": e2e,
        "clocks": {k: clocks.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons", "samples", "power_w_max")},
        "gpu_launches": args.steps,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


CONVSCAN_METRIC = ("convolution + selective scan Gelem/s (B·D·L/s), the 4-tap causal conv and SiLU "
                   "fused into the scan kernel, with the separate two-kernel chain timed beside it")


def _timed_steps(step, args, flush, stream, world):
    """Warm-up, then args.steps steps each after an L2 flush, timed with CUDA
    events on `stream` (ms per step)."""
    import torch
    for _ in range(args.warmup):
        flush_l2(flush)
        step()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush_l2(flush)
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    return [a.elapsed_time(b_) for a, b_ in zip(starts, ends)]


def run_convscan(args):
    """The convolution + scan call (ssm_scan_fwd_conv) on the workload's shape
    with a 4-tap filter: the fused mode is the line's value; the separate mode
    (ssm_conv1d_fwd into the workspace, then the scan) is timed beside it."""
    import torch
    import selective_state_space_02_gb300 as ssm
    from selective_state_space_02_gb300 import synth

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    dev = torch.device("cuda", local)
    p, cfg = workload_problem(args.workload, rank)
    g = lambda t: None if t is None else t.to(dev)
    x, dl, z, B, C, A, D, bias = (g(p.x), g(p.delta), g(p.z), g(p.B), g(p.C), g(p.A), g(p.D), g(p.dt_bias))
    w, cb = synth.make_conv(p.dim, CONV_WIDTH, seed=cfg["seed"] + 11)
    w, cb = w.to(dev), cb.to(dev)
    y = torch.empty_like(x)
    flush = torch.empty(args.flush_mib << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    per = {}
    for mode in ("fused", "separate"):
        wsb = ssm.conv_scan_workspace_size(p.batch, p.dim, p.dstate, p.seqlen, CONV_WIDTH, p.torch_dtype, mode)
        ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev)

        def step(mode=mode, ws=ws):
            ssm.scan_fwd_conv(x, w, dl, A, B, C, conv_bias=cb, D=D, z=z, dt_bias=bias,
                              delta_softplus=p.delta_softplus, mode=mode, y=y, workspace=ws)

        if mode == "fused":
            sampler = ClockSampler(local)
            sampler.start()
            t_end = time.time() + args.soak_s
            while time.time() < t_end:
                for _ in range(20):
                    flush_l2(flush)
                    step()
                torch.cuda.synchronize()
            per[mode] = _timed_steps(step, args, flush, stream, world)
            clocks = sampler.stop()
        else:
            per[mode] = _timed_steps(step, args, flush, stream, world)
        del ws
    total_ms = max_over_ranks(sum(per["fused"]), world, dev)
    sep_ms = max_over_ranks(sum(per["separate"]), world, dev)
    elems = p.elems
    value = world * elems * args.steps / (total_ms / 1e3) / 1e9
    updates = elems * p.dstate
    kern_s = statistics.mean(per["fused"]) / 1e3
    alu_peak = alu_peak_updates_per_s()
    line = {
        "metric": CONVSCAN_METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload, "batch": p.batch, "dim": p.dim, "dstate": p.dstate,
                   "seqlen": p.seqlen, "width": CONV_WIDTH, "io_dtype": p.dtype, "gate": p.z is not None,
                   "mode": "fused", "l2": L2_NOTE.format(mib=args.flush_mib),
                   "parallelism": f"{world} independent replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "alu", "achieved": round(updates / kern_s / 1e12, 4),
                     "peak": round(alu_peak / 1e12, 4), "unit": "Tupdate/s",
                     "frac": round(updates / kern_s / alu_peak, 4), "traffic": None,
                     "kernel": "fused conv + scan step (B/C re-layout plus the scan kernel with the convolution)"},
        "separate": {"ms_per_step": round(sep_ms / args.steps, 5),
                     "value": round(world * elems * args.steps / (sep_ms / 1e3) / 1e9, 3), "unit": UNIT,
                     "kernels": "ssm_conv1d_fwd, then the scan (B/C re-layout plus the scan kernel)"},
        "cpu_baseline": None, "e2e": None,
        "clocks": {k: clocks.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons", "samples", "power_w_max")},
        "gpu_launches": args.steps * 2,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main(argv=None):
    global SEQLEN_OVERRIDE
    args = parse_args(argv)
    SEQLEN_OVERRIDE = args.seqlen
    if args.impl == "reference":
        run_reference(args)
    elif args.op == "step":
        run_step(args)
    elif args.op == "bwd":
        run_bwd(args)
    elif args.op == "conv":
        run_conv(args)
    elif args.op == "convscan":
        run_convscan(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
