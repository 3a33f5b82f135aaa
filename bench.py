"""Throughput of the fused attention forward pass on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]
    python bench.py --sweep [--sweep-seconds S]
    python bench.py --paired [--a-flags F] [--b-flags F] [--b-lib PATH]
    python bench.py --aa-runs 10

A step is one forward pass (every step of the hot path) over one batch of
synthetic input already resident in HBM.  The default workload is
B=4, H=16, Sq=Skv=4096, D=128, bf16, non-causal.  Rank 0 prints one JSON line.
For prefill the line's value times back-to-back fa_fwd_ex calls with
FA_FLAG_OVERLAP_PREVIOUS (programmatic dependent launch: a step starts on
the SMs the previous one has run out of work for and waits for it before
its first write); the same K steps as plain fa_fwd calls, timed step by
step, are its `plain` entry.  --no-overlap times the plain calls only.

Multi-GPU (torchrun, one process per GPU): every rank runs its own batch of
the same shape (independent heads, no data-path collective), so scaling is
weak; the time is the max over ranks and the value is all ranks' FLOPs over
that time.

--impl reference times the CPU oracle (oracle/, fp64 three-step attention) on
the host cores, on a bounded row sample of the same workload per step.

--sweep prints one line per configured workload (the small parity case, the
B2 H8 S1024 workloads, the headline, the long causal ones, the B*S = 16384
sweep and decode), each with its roofline, clocks and a short oracle sample.

--paired is the measurement protocol of "The FA5090 Optimization Journey"
(section 2.8): two arms of the same workload timed in alternation inside one
process (order reversed every other alternation), each alternation giving
one margin t_A / t_B; the line reports the median margin, its spread and the
AB / BA halves.  Arms differ by fa_fwd_ex flags or by another build of the
library (_build.build(variant=...)).  --aa-runs N runs the A/A null (both
arms the same build) in N fresh processes: t_noise = p95 of |margin - 1|,
and a change is kept only at a margin >= 1 + t_noise.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from attention_forward_gb300 import inputs  # noqa: E402

METRIC = "attention fwd TFLOP/s (4*B*H*Sq*Skv*D, 1/2 causal)"
UNIT = "TFLOP/s"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0,
                  "bf16_tflops_sustained": 1700.0}


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=inputs.HEADLINE.name,
                    choices=sorted(inputs.BY_NAME))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-gemm-ceiling", action="store_true")
    ap.add_argument("--no-overlap", action="store_true",
                    help="time plain fa_fwd steps only (no programmatic dependent launch)")
    ap.add_argument("--prefill-kernel", default="auto", choices=["auto", "single", "pair"],
                    help="prefill kernel: the library's choice (default), single CTAs "
                         "(FA_FLAG_SINGLE_CTA) or CTA pairs (FA_FLAG_PAIR)")
    ap.add_argument("--extra-flags", type=lambda x: int(x, 0), default=0,
                    help="FA_FLAG_* bits added to every call of this run (e.g. 0x20 for "
                         "the correction-warpgroup form)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="--impl reference: total oracle time over all steps")
    ap.add_argument("--sweep", action="store_true",
                    help="one line per configured workload")
    ap.add_argument("--sweep-only", default="", help="comma-separated workload names")
    ap.add_argument("--sweep-seconds", type=float, default=0.3,
                    help="--sweep: GPU time of each workload's timed region")
    ap.add_argument("--sweep-cpu-seconds", type=float, default=1.5,
                    help="--sweep: oracle time of each workload's CPU baseline")
    ap.add_argument("--paired", action="store_true", help="paired A/B of two arms")
    ap.add_argument("--aa-runs", type=int, default=0,
                    help="A/A null over this many fresh processes")
    ap.add_argument("--a-flags", type=lambda x: int(x, 0), default=0)
    ap.add_argument("--b-flags", type=lambda x: int(x, 0), default=0)
    ap.add_argument("--a-lib", default="", help="another build of the library for arm A")
    ap.add_argument("--b-lib", default="", help="another build of the library for arm B")
    ap.add_argument("--a-tag", default="A")
    ap.add_argument("--b-tag", default="B")
    ap.add_argument("--alternations", type=int, default=120)
    ap.add_argument("--pwarm", type=int, default=25)
    ap.add_argument("--pmeasure", type=int, default=100)
    return ap.parse_args(argv)


# ----------------------------------------------------------------- helpers

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def shard_seed(seed: int, rank: int) -> int:
    """Each rank draws its own batch (weak scaling)."""
    return seed + 1000 * rank


def job_throughput(flops_per_step: float, steps: int, world: int,
                   max_seconds: float) -> float:
    """Whole-job TFLOP/s: every rank ran `steps` steps of its own batch (weak
    scaling), the job took as long as the slowest rank."""
    return flops_per_step * steps * world / max_seconds / 1e12


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# Host-side dispatch (argument checks, the choice of kernel and split,
# workspaces) and the device self-check: not part of what the attention
# kernels' counters depend on.
_HOST_ONLY = {"fa_api.cu", "fa_noalloc.cu", "fa_host.h", "fa_diag.cu"}


_COMMENT = re.compile(r"//[^\n]*|/\*.*?\*/", re.S)


def kernel_fingerprint() -> str:
    """sha256 (16 hex digits) of the device code and launch wrappers under
    attention_forward_gb300/csrc: every file but the host-side dispatch,
    with comments removed and white space collapsed (an edit of a comment
    or of the layout changes no kernel)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "attention_forward_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name in _HOST_ONLY:
            continue
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            code = " ".join(_COMMENT.sub(" ", f.read()).split())
        h.update(name.encode() + code.encode())
    return h.hexdigest()[:16]


def profiled_traffic(kind: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources and this workload; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(kind, {})
    if e.get("kernel_fingerprint") != kernel_fingerprint() or e.get("workload") != workload:
        return None
    return e.get("dram_bytes_per_launch")


class NvmlClocks:
    """SM clock, power and clock-event reasons of one GPU, read in-process
    through NVML (read-only queries, nothing is set) about every half
    millisecond by a background thread, each sample stamped on arrival.
    Fast enough for timed regions of a few milliseconds."""
    # nvmlClocksEventReasons bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    NVML_CLOCK_SM = 1

    def __init__(self, pci_bus_id: str, period_s: float = 0.0005):
        import ctypes
        self.ct = ctypes
        self.samples = []
        self.ok = False
        self.period = period_s
        self._stop = threading.Event()
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return
        if nv.nvmlInit_v2() != 0:
            return
        h = ctypes.c_void_p()
        if nv.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(), ctypes.byref(h)) != 0:
            return
        self.nv, self.h = nv, h
        mx = ctypes.c_uint(0)
        self.max_mhz = (float(mx.value) if nv.nvmlDeviceGetMaxClockInfo(
            h, self.NVML_CLOCK_SM, ctypes.byref(mx)) == 0 else None)
        self.reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons", None)
        self.ok = True
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()

    def _run(self):
        ct, nv, h = self.ct, self.nv, self.h
        mhz, mw, rs = ct.c_uint(0), ct.c_uint(0), ct.c_ulonglong(0)
        while not self._stop.is_set():
            if nv.nvmlDeviceGetClockInfo(h, self.NVML_CLOCK_SM, ct.byref(mhz)) == 0:
                w = mw.value / 1e3 if nv.nvmlDeviceGetPowerUsage(h, ct.byref(mw)) == 0 else None
                r = rs.value if (self.reasons_fn and self.reasons_fn(h, ct.byref(rs)) == 0) else 0
                self.samples.append((time.time(), float(mhz.value), w, r))
            time.sleep(self.period)

    def stop(self):
        self._stop.set()
        if self.ok:
            self.thread.join(timeout=2)

    def summary(self, t0: float, t1: float):
        inside = [x for x in self.samples if t0 <= x[0] <= t1]
        out = {"sm_mhz": None, "sm_max_mhz": self.max_mhz if self.ok else None,
               "reasons": [], "samples": len(inside), "source": "nvml, in-process"}
        if not inside:
            out["note"] = "no clock sample inside the timed region"
            return out
        reasons = set()
        for _, _, _, r in inside:
            reasons |= {n for bit, n in self.REASONS.items() if r & bit}
        pw = [x[2] for x in inside if x[2] is not None]
        out.update(sm_mhz=statistics.median(x[1] for x in inside),
                   sm_mhz_min=min(x[1] for x in inside),
                   power_w_median=statistics.median(pw) if pw else None,
                   reasons=sorted(reasons))
        if len(inside) < 3:
            out["note"] = "fewer than 3 samples inside the timed region"
        return out


class SmiClocks:
    """Fallback without NVML: nvidia-smi clocks / throttle reasons every
    20 ms, stamped on arrival; only samples inside the timed region count."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20", "-i", gpu_id],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        inside = [s for t, s in self.samples if t0 <= t <= t1]
        out = {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": len(inside),
               "source": "nvidia-smi -lms 20"}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        mhz, mx, pw = [], [], []
        for s in inside:
            try:
                mhz.append(float(s[0]))
                mx.append(float(s[1]))
                pw.append(float(s[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, s[4:8]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        if not mhz:
            out["note"] = "no clock sample inside the timed region"
            return out
        out.update(sm_mhz=statistics.median(mhz), sm_max_mhz=max(mx),
                   power_w_median=statistics.median(pw) if pw else None,
                   reasons=sorted(reasons))
        if len(mhz) < 3:
            out["note"] = "fewer than 3 samples inside the timed region"
        return out


def clock_sampler(device):
    """NVML in-process sampler, else nvidia-smi."""
    c = NvmlClocks(gpu_id_for_smi(device))
    if c.ok:
        return c
    return SmiClocks(gpu_id_for_smi(device))


def gpu_id_for_smi(device) -> str:
    props = torch.cuda.get_device_properties(device)
    bus = getattr(props, "pci_bus_id", None)
    dom = getattr(props, "pci_domain_id", None)
    dev = getattr(props, "pci_device_id", None)
    if bus is not None and dom is not None and dev is not None:
        return f"{dom:08X}:{bus:02X}:{dev:02X}.0"
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids = [x for x in vis.split(",") if x.strip()]
    if ids and ids[device.index if device.index is not None else 0].strip().isdigit():
        return ids[device.index or 0].strip()
    return str(device.index or 0)


def gemm_ceiling(device) -> float:
    """Dense bf16 GEMM throughput in this run (torch.matmul 8192^3, best of
    10): the ceiling the attention kernel is compared with."""
    n = 8192
    a = torch.randn(n, n, device=device, dtype=torch.bfloat16)
    b = torch.randn(n, n, device=device, dtype=torch.bfloat16)
    for _ in range(3):
        torch.matmul(a, b)
    torch.cuda.synchronize(device)
    best = float("inf")
    for _ in range(10):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        torch.matmul(a, b)
        e.record()
        e.synchronize()
        best = min(best, s.elapsed_time(e) / 1e3)
    del a, b
    return 2.0 * n ** 3 / best / 1e12


# ------------------------------------------------------------ CPU (oracle)

class OracleSample:
    """The fp64 oracle timed on a row sample of the workload (host cores).
    The per-row cost is 4*Skv*D FLOPs (the visible keys for causal rows)."""

    def __init__(self, w: inputs.Workload, seed: int = 0, nthreads: int = 0):
        import oracle
        self.oracle = oracle
        self.w = w
        self.nthreads = nthreads or oracle.default_threads()
        self.rng = np.random.default_rng(seed)
        heads = sorted(set(int(x) for x in self.rng.integers(0, w.B * w.H, size=4)))
        self.nh = len(heads)
        q, k, v = w.make(heads=heads)
        self.q, self.k, self.v = (t.float().numpy()[None] for t in (q, k, v))

    def _flops(self, rows):
        w = self.w
        i = rows % w.Sq
        if w.causal:
            vis = np.minimum(w.Skv, i + (w.Skv - w.Sq) + 1).clip(min=0)
        else:
            vis = np.full(rows.shape, w.Skv)
        return float((4.0 * vis * w.D).sum())

    def run(self, n: int):
        rows = self.rng.integers(0, self.nh * self.w.Sq, size=n)
        t = time.perf_counter()
        self.oracle.attention(self.q, self.k, self.v, self.w.scale, self.w.causal,
                              rows=rows, nthreads=self.nthreads)
        return time.perf_counter() - t, self._flops(rows)

    def rows_for(self, target_s: float) -> int:
        n = max(self.nthreads, 8)
        self.run(n)  # the first call pays one-time costs: not a calibration point
        dt, _ = self.run(n)
        while dt < 0.25 and n < (1 << 20):
            n *= 4
            dt, _ = self.run(n)
        return max(self.nthreads, int(n * target_s / max(dt, 1e-6)))

    def describe(self, n: int) -> str:
        return (f"{n} query rows (all their visible keys) drawn from {self.nh} heads of "
                f"{self.w.name}, fp64, {self.nthreads} threads")


def oracle_rate(w: inputs.Workload, target_s: float, nthreads: int = 0):
    """(TFLOP/s, cores, sample, seconds) of the oracle on about target_s of
    work, on nthreads host threads (0: all cores)."""
    smp = OracleSample(w, nthreads=nthreads)
    n = smp.rows_for(target_s)
    dt, fl = smp.run(n)
    return fl / dt / 1e12, smp.nthreads, smp.describe(n), dt


# ------------------------------------------------------------------ arms

def bench_reference(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    # each step: a bounded row sample, sized so the whole run stays near a
    # couple of minutes
    smp = OracleSample(w)
    per_step = min(10.0, max(0.02, args.ref_seconds / max(1, args.steps + args.warmup)))
    n = smp.rows_for(per_step)
    for _ in range(args.warmup):
        smp.run(n)
    secs, flops = 0.0, 0.0
    for _ in range(args.steps):
        dt, fl = smp.run(n)
        secs += dt
        flops += fl
    value = flops / secs / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, 1),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": smp.nthreads,
                         "kind": "oracle", "sample": "each step: " + smp.describe(n)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w, n_gpus):
    return {"workload": w.name, "B": w.B, "H": w.H, "Sq": w.Sq, "Skv": w.Skv, "D": w.D,
            "causal": w.causal, "global_batch": w.B * n_gpus, "seq_len": w.Skv,
            "parallelism": f"independent batches x{n_gpus}"}


def launches_per_step(fa, w) -> int:
    """Kernel launches of one fa_fwd call: the fused kernel, plus the
    combine kernel when the keys are split (decode, and prefill whose items
    do not fill the SMs)."""
    return 2 if fa.fa_workspace_bytes(w.B, w.H, w.Sq, w.Skv, w.D) > 0 else 1


def algorithmic_bytes(w) -> int:
    """Q, K, V read once, O and LSE written once."""
    return (w.B * w.H * (w.Sq + 2 * w.Skv) * w.D * 2 + w.B * w.H * w.Sq * w.D * 2
            + w.B * w.H * w.Sq * 4)


def roofline(fa, w, launch_s, kflags):
    """The roofline object of the step's dominant kernel."""
    peaks, peak_src = load_peaks()
    if w.Sq == 1:
        achieved = algorithmic_bytes(w) / launch_s / 1e9
        peak = float(peaks["hbm_gbs"])
        return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": profiled_traffic("decode", w.name),
                "peak_source": f"{peak_src} hbm_gbs",
                "kernel": "fa_decode_kernel + fa_decode_combine_kernel (one step)"}
    achieved = w.flops() / launch_s / 1e12
    peak = float(peaks["bf16_tflops"])
    pairs = fa.fa_prefill_uses_pairs(w.B, w.H, w.Sq, w.Skv, w.D, w.causal, kflags)
    kern = "fa_prefill_pair_kernel (two-CTA clusters)" if pairs else "fa_prefill_kernel"
    if pairs:
        tail = fa.fa_prefill_tail_items(w.B, w.H, w.Sq, w.Skv, w.D, w.causal,
                                        inputs.DTYPES[w.dtype], kflags)
        if tail:
            kern += f", its last {tail} items split into key quarters (merged in the kernel)"
    if launches_per_step(fa, w) > 1 and not pairs:
        kern += " with split keys + fa_decode_combine_kernel (one step)"
    return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak,
            "traffic": profiled_traffic("prefill_pair" if pairs else "prefill_single", w.name),
            "peak_source": f"{peak_src} bf16_tflops (burst; dense fp16 has the same rate)",
            "kernel": kern}


class Problem:
    """One workload's device inputs and outputs, and its step (one fa_fwd or
    fa_fwd_ex call on `stream`)."""

    def __init__(self, w, device, stream, seed=None, kflags=0, lib=None):
        from attention_forward_gb300 import fa
        self.fa, self.w, self.device, self.stream = fa, w, device, stream
        q, k, v = inputs.make_qkv(w.B, w.H, w.Sq, w.Skv, w.D, w.dtype,
                                  w.seed if seed is None else seed, w.qk_mult)
        self.host = (q, k, v)
        self.dq, self.dk, self.dv = (t.to(device) for t in (q, k, v))
        self.o = torch.empty_like(self.dq)
        self.lse = torch.empty((w.B, w.H, w.Sq), dtype=torch.float32, device=device)
        self.kflags, self.lib = kflags, lib

    def step(self, kflags=None, lib=None):
        kflags = self.kflags if kflags is None else kflags
        lib = lib or self.lib
        if kflags or lib is not None:
            self.fa.fa_fwd_ex(self.dq, self.dk, self.dv, causal=self.w.causal, flags=kflags,
                              out=self.o, lse=self.lse, stream=self.stream, lib=lib)
        else:
            self.fa.fa_fwd(self.dq, self.dk, self.dv, causal=self.w.causal, out=self.o,
                           lse=self.lse, stream=self.stream)


def timed_steps(prob, K, warmup, world=1, sampler=None, per_step=True):
    """W untimed steps, then exactly K steps bracketed by a barrier and a
    synchronize on both sides, with CUDA events on the launching stream
    around the whole region and (per_step) around every step.  Without
    per-step events consecutive steps may overlap (an event between two
    launches would serialise them); every step's time is then the region's
    over K.  Returns (seconds of the region, sorted per-step ms, clocks)."""
    fa, device, stream = prob.fa, prob.device, prob.stream
    for _ in range(max(3, warmup)):
        prob.step()
    torch.cuda.synchronize(device)
    if fa.fa_get_device_status() != fa.FA_OK:
        raise RuntimeError("kernel watchdog fired during warm-up")
    own = sampler is None
    if own:
        sampler = clock_sampler(device)
        time.sleep(0.05)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world, device)
    torch.cuda.synchronize(device)
    wall0 = time.time()
    t_start.record(stream)
    for i in range(K):
        if per_step:
            ev[i][0].record(stream)
        prob.step()
        if per_step:
            ev[i][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize(device)
    wall1 = time.time()
    barrier(world, device)
    clocks = sampler.summary(wall0, wall1)
    if own:
        sampler.stop()
    if fa.fa_get_device_status() != fa.FA_OK:
        raise RuntimeError("kernel watchdog fired in the timed region")
    total_s = t_start.elapsed_time(t_end) / 1e3
    if per_step:
        launch_ms = sorted(a.elapsed_time(b) for a, b in ev)
    else:
        launch_ms = [total_s * 1e3 / K] * K
    return total_s, launch_ms, clocks


def result_line(prob, K, warmup, world, total_max, launch_ms, clocks):
    """The JSON line of one timed run (without e2e and the CPU baseline)."""
    fa, w = prob.fa, prob.w
    launch_s = statistics.mean(launch_ms) / 1e3
    pct = lambda f: launch_ms[min(K - 1, int(f * K))]
    roof = roofline(fa, w, launch_s, prob.kflags)
    n_in = 3 * prob.dq.numel() * 2 if w.Sq == w.Skv else (prob.dq.numel() + 2 * prob.dk.numel()) * 2
    return {
        "metric": METRIC, "value": job_throughput(w.flops(), K, world, total_max),
        "unit": UNIT, "n_gpus": world, "steps": K, "warmup": warmup,
        "ms_per_step": total_max / K * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic (seeded N(0,1), per-rank batches)",
        "config": dict(workload_config(w, world),
                       l2=f"inputs {n_in / 2**20:.0f} MiB "
                          f"{'>' if n_in > L2_BYTES else '<='} L2 129 MiB; no flush"),
        "roofline": roof,
        "gpu_launches": K * launches_per_step(fa, w),
        "step_ms": {"mean": launch_s * 1e3, "median": statistics.median(launch_ms),
                    "p10": pct(0.10), "p90": pct(0.90),
                    "source": ("CUDA events around each step" if len(set(launch_ms)) > 1 or K == 1
                               else "CUDA events around the region, over K (steps overlap)")},
        "clocks": clocks,
    }


def kernel_flags(fa, name, extra=0):
    return {"auto": 0, "single": fa.FA_FLAG_SINGLE_CTA, "pair": fa.FA_FLAG_PAIR}[name] | extra


OVERLAP_NOTE = ("back-to-back fa_fwd_ex calls with FA_FLAG_OVERLAP_PREVIOUS (CUDA programmatic "
                "dependent launch): a step's CTAs start on the SMs the previous step has run out "
                "of work for, read the resident inputs at once and wait for the previous step "
                "before their first write; every step computes the whole forward pass; timed "
                "with events around the region only")


def measure(prob, K, warmup, world, device, overlap):
    """The line of one workload: with overlap (prefill), K overlapped steps
    are the line's value and K plain fa_fwd steps, timed with per-step
    events, its `plain` entry; without (or for decode, which the flag does
    not change), the plain steps alone."""
    fa = prob.fa
    base = prob.kflags
    total_p, ms_p, clocks_p = timed_steps(prob, K, warmup, world)
    total_p = max_over_ranks(total_p, world, device)
    plain = result_line(prob, K, warmup, world, total_p, ms_p, clocks_p)
    if not overlap or prob.w.Sq == 1:
        plain["launch"] = "back-to-back fa_fwd calls, CUDA events around each step"
        return plain
    prob.kflags = base | fa.FA_FLAG_OVERLAP_PREVIOUS
    try:
        total_o, ms_o, clocks_o = timed_steps(prob, K, warmup, world, per_step=False)
    finally:
        prob.kflags = base
    total_o = max_over_ranks(total_o, world, device)
    line = result_line(prob, K, warmup, world, total_o, ms_o, clocks_o)
    line["launch"] = OVERLAP_NOTE
    # the roofline is the kernel's: flops of a launch over the launch's own
    # duration, which only the plain steps (an event pair around each) give;
    # the overlapped steps' rate is kept beside it
    ov = line["roofline"]
    line["roofline"] = dict(plain["roofline"], achieved_overlapped_steps=ov["achieved"],
                            frac_overlapped_steps=ov["frac"],
                            duration_source="CUDA events around each plain launch")
    line["plain"] = {"value": plain["value"], "ms_per_step": plain["ms_per_step"],
                     "roofline_frac": plain["roofline"]["frac"], "step_ms": plain["step_ms"],
                     "clocks": plain["clocks"],
                     "launch": "back-to-back fa_fwd calls, CUDA events around each step"}
    return line


def bench_ours(args, w):
    from attention_forward_gb300 import fa
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    fa.load()
    stream = torch.cuda.current_stream(device)
    prob = Problem(w, device, stream, seed=shard_seed(w.seed, rank),
                   kflags=kernel_flags(fa, args.prefill_kernel, args.extra_flags))
    K = args.steps
    line = measure(prob, K, args.warmup, world, device, not args.no_overlap)
    decode = w.Sq == 1

    if not args.no_e2e:
        line["e2e"] = e2e(w, *prob.host, device, stream, min(K, 40))
    if rank == 0 and world == 1 and not args.no_gemm_ceiling:
        g = gemm_ceiling(device)
        line["gemm_ceiling_tflops_same_run"] = g
        line["frac_of_same_run_gemm"] = line["roofline"]["achieved"] / g if not decode else None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def cpu_baseline(w, seconds, one_core=True):
    r, cores, sample, dt = oracle_rate(w, seconds)
    out = {"value": r, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample,
           "seconds": dt}
    if one_core:
        r1, _, sample1, dt1 = oracle_rate(w, seconds / 2, nthreads=1)
        out["one_core"] = {"value": r1, "unit": UNIT, "sample": sample1, "seconds": dt1}
    return out


def bench_sweep(args):
    """One JSON line per configured workload on this GPU: as many steps as
    fill about --sweep-seconds of GPU time (at least 20), the same timing,
    clock sampling and roofline as the default run, and a short oracle
    sample on the host cores."""
    from attention_forward_gb300 import fa
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    fa.load()
    stream = torch.cuda.current_stream(device)
    gemm = None if args.no_gemm_ceiling else gemm_ceiling(device)
    names = args.sweep_only.split(",") if args.sweep_only else None
    for w in inputs.CONFIGURED:
        if names and w.name not in names:
            continue
        prob = Problem(w, device, stream, kflags=kernel_flags(fa, args.prefill_kernel, args.extra_flags))
        # size the run: a few probe steps first
        for _ in range(3):
            prob.step()
        torch.cuda.synchronize(device)
        t0 = time.perf_counter()
        for _ in range(5):
            prob.step()
        torch.cuda.synchronize(device)
        per = (time.perf_counter() - t0) / 5
        K = int(min(5000, max(20, args.sweep_seconds / max(per, 1e-6))))
        line = measure(prob, K, args.warmup, 1, device, not args.no_overlap)
        if gemm is not None:
            line["gemm_ceiling_tflops_same_run"] = gemm
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(w, args.sweep_cpu_seconds, one_core=False)
        print(json.dumps(line), flush=True)
        del prob
        torch.cuda.empty_cache()
    return 0


def paired_margins(prob, arms, alternations, pwarm, pmeasure):
    """The FA5090 paired protocol: per alternation, each arm runs pwarm
    untimed then pmeasure timed launches (CUDA events per launch) and gives
    its median; the order is AB on even and BA on odd alternations.
    Returns the per-alternation (median A ms, median B ms, order)."""
    out = []
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(pmeasure)]
    for i in range(alternations):
        order = (0, 1) if i % 2 == 0 else (1, 0)
        med = [0.0, 0.0]
        for a in order:
            kflags, lib = arms[a]
            for _ in range(pwarm):
                prob.step(kflags, lib)
            for e0, e1 in evs:
                e0.record(prob.stream)
                prob.step(kflags, lib)
                e1.record(prob.stream)
            torch.cuda.synchronize(prob.device)
            med[a] = statistics.median(e0.elapsed_time(e1) for e0, e1 in evs)
        out.append((med[0], med[1], "AB" if order == (0, 1) else "BA"))
    return out


def paired_summary(res):
    """Statistics of paired alternations [(median_A_ms, median_B_ms, "AB"|"BA")]:
    the per-alternation margin t_A / t_B (> 1: B faster), its median,
    geometric mean and p10/p90, the median of each order half, B's wins."""
    m = np.array([a / b for a, b, _ in res])
    half = lambda o: float(np.median([a / b for a, b, oo in res if oo == o]))
    return {
        "margin": float(np.median(m)),
        "margin_gmean": float(np.exp(np.mean(np.log(m)))),
        "paired_lo": float(np.percentile(m, 10)), "paired_hi": float(np.percentile(m, 90)),
        "ab_half": half("AB"), "ba_half": half("BA"),
        "b_wins": int((m > 1).sum()), "alternations": len(res),
        "t_a_ms": float(np.median([a for a, _, _ in res])),
        "t_b_ms": float(np.median([b for _, b, _ in res])),
    }


def aa_noise(margins):
    """The A/A null's noise floor: p95 of |margin - 1| (and its maximum)."""
    dev = np.abs(np.asarray(margins, dtype=np.float64) - 1.0)
    return float(np.percentile(dev, 95)), float(dev.max())


def bench_paired(args, w):
    """Paired, interleaved A/B of two arms on one workload (see the module
    docstring); prints one JSON line."""
    from attention_forward_gb300 import fa
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    fa.load()
    stream = torch.cuda.current_stream(device)
    # both arms call fa_fwd_ex (the in-tree build unless another is given)
    libs = [fa.load_path(p) if p else fa.load() for p in (args.a_lib, args.b_lib)]
    arms = [(args.a_flags, libs[0]), (args.b_flags, libs[1])]
    prob = Problem(w, device, stream)
    # both arms must compute the same attention: compare their outputs
    outs = []
    for kflags, lib in arms:
        prob.step(kflags, lib)
        torch.cuda.synchronize(device)
        outs.append((prob.o.clone(), prob.lse.clone()))
    bitwise = bool(torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1]))
    sampler = clock_sampler(device)
    time.sleep(0.05)
    wall0 = time.time()
    res = paired_margins(prob, arms, args.alternations, args.pwarm, args.pmeasure)
    wall1 = time.time()
    clocks = sampler.summary(wall0, wall1)
    sampler.stop()
    if fa.fa_get_device_status() != fa.FA_OK:
        raise RuntimeError("kernel watchdog fired in a paired run")
    line = {
        "mode": "paired", "workload": w.name,
        "a": {"flags": args.a_flags, "lib": args.a_lib or "in-tree", "tag": args.a_tag},
        "b": {"flags": args.b_flags, "lib": args.b_lib or "in-tree", "tag": args.b_tag},
        **paired_summary(res),
        "protocol": f"{args.alternations} alternations x ({args.pwarm} warm-up + "
                    f"{args.pmeasure} timed launches per arm), order AB/BA alternating; "
                    "margin = median_A / median_B per alternation (> 1: B faster)",
        "outputs_bitwise_equal": bitwise, "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    return 0


def bench_aa(args, w):
    """The A/A null: the paired protocol with both arms the same build, in
    --aa-runs fresh processes; t_noise = p95 of |margin - 1|."""
    margins, lines = [], []
    for _ in range(args.aa_runs):
        cmd = [sys.executable, os.path.abspath(__file__), "--paired", "--workload", w.name,
               "--alternations", str(args.alternations), "--pwarm", str(args.pwarm),
               "--pmeasure", str(args.pmeasure), "--a-tag", "A", "--b-tag", "A'"]
        r = subprocess.run(cmd, capture_output=True, text=True, timeout=1800)
        if r.returncode != 0:
            raise RuntimeError(r.stderr[-2000:])
        d = json.loads([x for x in r.stdout.splitlines() if x.strip()][-1])
        margins.append(d["margin"])
        lines.append({k: d[k] for k in ("margin", "ab_half", "ba_half", "b_wins",
                                        "t_a_ms", "t_b_ms")} | {"sm_mhz": d["clocks"]["sm_mhz"]})
    t_noise, t_max = aa_noise(margins)
    print(json.dumps({"mode": "aa_null", "workload": w.name, "runs": len(margins),
                      "margins": margins, "t_noise": t_noise,
                      "t_noise_max": t_max, "t_keep": 1.0 + t_noise,
                      "protocol": f"{args.alternations} alternations x ({args.pwarm} + "
                                  f"{args.pmeasure} launches per arm), each run a fresh "
                                  "process, both arms the in-tree build",
                      "per_run": lines}), flush=True)
    return 0


def e2e(w, q, k, v, device, stream, n_steps):
    """Same metric through the host-buffer C-ABI call: every step copies Q,
    K, V from pinned host memory, runs, and copies O and LSE back.  Steps
    alternate between two streams with a staging buffer each (double
    buffering), so one step's copies overlap the other step's kernel."""
    from attention_forward_gb300 import fa
    qh, kh, vh = (t.pin_memory() for t in (q, k, v))
    streams = [stream, torch.cuda.Stream(device)]
    ohs = [torch.empty_like(qh).pin_memory() for _ in range(2)]
    lhs = [torch.empty((w.B, w.H, w.Sq), dtype=torch.float32).pin_memory() for _ in range(2)]
    nbytes = fa.fa_host_staging_bytes(w.B, w.H, w.Sq, w.Skv, w.D)
    stagings = [torch.empty(nbytes, dtype=torch.uint8, device=device) for _ in range(2)]

    def step(i):
        b = i % 2
        fa.fa_fwd_host(qh, kh, vh, stagings[b], causal=w.causal, out_h=ohs[b],
                       lse_h=lhs[b], stream=streams[b])

    for i in range(4):
        step(i)
    torch.cuda.synchronize(device)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(streams[0])
    streams[1].wait_event(s)
    for i in range(n_steps):
        step(i)
    done = torch.cuda.Event()
    done.record(streams[1])
    streams[0].wait_event(done)
    e.record(streams[0])
    torch.cuda.synchronize(device)
    sec = s.elapsed_time(e) / 1e3 / n_steps
    h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh))
    d2h = ohs[0].numel() * ohs[0].element_size() + lhs[0].numel() * 4
    return {"value": w.flops() / sec / 1e12, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": sec * 1e3, "steps": n_steps,
            "api": "fa_fwd_host (pinned host buffers, copies inside the timed region; "
                   "steps alternate between two streams, double-buffered)"}


def main(argv=None):
    args = parse_args(argv)
    w = inputs.BY_NAME[args.workload]
    if args.impl == "reference":
        return bench_reference(args, w)
    if args.sweep:
        return bench_sweep(args)
    if args.aa_runs:
        return bench_aa(args, w)
    if args.paired:
        return bench_paired(args, w)
    return bench_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
