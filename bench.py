"""Benchmark of the selected-token log-probability hot path on GB300.

One step = forward (logp, lse) + backward (dlogits) over the long-CoT workload
(N = 32768 rows, V = 151936, BF16 logits ~ N(0, 2^2) plus a +8 spike per row,
5% ignore rows, g = +-1/N), inputs resident in HBM.  The logits (9.96 GB) and
dlogits (9.96 GB) are far larger than L2 (129 MB), so no L2 flush is needed
between steps.

Metric: effective HBM GB/s of forward + backward, counting the algorithmic
6 bytes per logit (forward: one 2-byte read; backward: one 2-byte read and one
2-byte write), plus ms per step.  Prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
    python bench.py --path linear      # fused LM head + logp forward (tensor cores)

--path linear times the fused LM-head forward instead (BF16 hidden states
[32768, 4096] against BF16 LM-head weights [151936, 4096], logits never
materialised) and reports dense TFLOP/s (2 N V D per call) against the
measured bf16 tensor peak.

--impl reference times the FP64 CPU oracle on the host cores (a bounded
sample of rows per step) on the same metric; under torchrun only rank 0 runs
it.  For N > 1 (torchrun) the ranks split the rows of one global batch of
N x 32768 rows (rank r's block drawn from seed r): rows are independent and
each row's bits are batch-invariant, so every rank runs the same kernels on
its own rows with no collective on the data path (weak scaling).
"""

from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fwd+bwd ms & HBM GB/s (% roofline) at N=32768, V=151936 BF16"
UNIT = "GB/s"
BYTES_PER_LOGIT = 6          # fwd read 2 + bwd read 2 + bwd write 2
BWD_BYTES_PER_LOGIT = 4
FWD_BYTES_PER_LOGIT = 2
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0
LIN_METRIC = "fused LM-head + logp forward TFLOP/s at N=32768, D=4096, V=151936 BF16"
LIN_DESC = ("fused LM head: hidden [N, D] BF16 ~ N(0,1), weight [V, D] BF16 ~ N(0,(2/sqrt D)^2), "
            "targets uniform, 5% ignore_index (synthetic)")
# Pages' fused kernel, forward + backward at 32768 x 151936 (B200, BF16):
# 27.2 ms (RL-Kernel PR #495, Results table).  Context only: another GPU.
PAGES_FWD_BWD_MS = 27.2
WORKLOAD_DESC = ("long-CoT: N=32768, V=151936, BF16 logits ~ N(0,2^2) + 8 spike/row, "
                 "5% ignore_index, g=+-1/N (synthetic)")


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, copy)"
    return FALLBACK_HBM_GBS, "fallback 6.8 TB/s"


def _tensor_peaks():
    """(burst, sustained, source) dense bf16 TFLOP/s."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return (float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "measured (MEASURED_PEAKS.json bf16_tflops, cuBLAS burst)")
    return FALLBACK_BF16_TFLOPS, FALLBACK_BF16_TFLOPS_SUSTAINED, "fallback 1.9 PFLOP/s"


# Device sources of each profiled kernel (a profile's traffic is reported only
# while these files are unchanged since its capture).
KERNEL_SOURCES = {
    "k_logp_bwd": ("logp_kernels.cuh", "logp_prims.cuh"),
    "k_logp_fwd_bulk": ("logp_kernels.cuh", "logp_prims.cuh"),
    "k_linear_logp_tiles": ("linear_logp.cuh", "logp_kernels.cuh", "logp_prims.cuh"),
}


def _kernel_hash(kernel: str = "k_logp_bwd") -> str:
    h = hashlib.sha256()
    for fn in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "selected_token_logprob_gb300", "csrc", fn), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _profiled_traffic(kernel: str, parts: bool = False):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if it
    was taken on the current kernel source; else None.  With parts: a dict of
    the read, write and total bytes (and the method's bytes, when recorded)."""
    p = os.path.join(ROOT, "profiles", f"{kernel}_long.md")
    if not os.path.exists(p):
        return None
    txt = open(p).read()
    m_hash = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", txt)
    m_bytes = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    if not m_hash or not m_bytes or m_hash.group(1) != _kernel_hash(kernel):
        return None
    if not parts:
        return float(m_bytes.group(1))
    out = {"total": float(m_bytes.group(1))}
    for key, name in (("read", "dram_read_bytes_per_launch"), ("write", "dram_write_bytes_per_launch"),
                      ("algorithmic_active", "algorithmic_bytes_active")):
        m = re.search(name + r":\s*([0-9.eE+]+)", txt)
        out[key] = float(m.group(1)) if m else None
    return out


class ClockSampler:
    """SM clock, its maximum, power and the clock-event reasons during the
    timed region (mark() is called at its start and end).

    Read-only queries.  Preferred: NVML through ctypes, polled every 10 ms in
    a thread, so that even a timed region of a few tens of milliseconds holds
    several samples.  Fallback: `nvidia-smi -lms 200`.  Only samples whose
    time stamp falls inside the marked window are summarised."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # NVML clock-event reason bits (nvml.h: nvmlClocksEventReason*)
    REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                   0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    PERIOD_S = 0.010

    def __init__(self, gpu_index: int, uuid: str | None = None):
        self.gpu = gpu_index
        self.uuid = uuid
        self.proc = None
        self.out = ""
        self.window = None
        self.samples = []          # (time, sm_mhz, sm_max_mhz, set of reasons, watts)
        self.source = None
        self._thread = None
        self._stop = None

    # ---- NVML
    def _nvml_start(self) -> bool:
        import ctypes
        import threading

        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return False
        if nv.nvmlInit_v2() != 0:
            return False
        h = ctypes.c_void_p()
        ok = False
        if self.uuid:
            ok = nv.nvmlDeviceGetHandleByUUID(self.uuid.encode(), ctypes.byref(h)) == 0
        if not ok:
            ok = nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.gpu), ctypes.byref(h)) == 0
        if not ok:
            return False
        reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        self._stop = threading.Event()

        def loop():
            mhz, mx, pw = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint()
            rs = ctypes.c_ulonglong()
            while not self._stop.is_set():
                t = time.time()
                a = nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz))          # NVML_CLOCK_SM
                b = nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
                c = reasons_fn(h, ctypes.byref(rs))
                d = nv.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw))
                if a == 0 and b == 0 and c == 0:
                    names = {n for bit, n in self.REASON_BITS.items() if rs.value & bit}
                    self.samples.append((t, float(mhz.value), float(mx.value), names,
                                         pw.value / 1000.0 if d == 0 else None))
                self._stop.wait(self.PERIOD_S)

        self._thread = threading.Thread(target=loop, daemon=True)
        self._thread.start()
        self.source = "nvml, every 10 ms"
        return True

    def __enter__(self):
        if self._nvml_start():
            time.sleep(0.05)
            return self
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi, every 200 ms"
            time.sleep(0.5)                  # let it start sampling before the timed region
        except (OSError, ValueError):
            self.proc = None
        return self

    def mark(self):
        """Call at the start and at the end of the timed region."""
        now = time.time()
        self.window = (now, None) if self.window is None or self.window[1] is not None else (self.window[0], now)

    def __exit__(self, *exc):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(2)
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()
        return False

    @staticmethod
    def _stamp(text: str):
        import datetime

        try:
            return datetime.datetime.strptime(text.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def _smi_samples(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        out = []
        for r in csv.reader(io.StringIO(self.out or "")):
            if len(r) < 10:
                continue
            ts = self._stamp(r[0])
            num = lambda x: float(x) if x.strip().replace(".", "").isdigit() else None  # noqa: E731
            reasons = {names[i] for i in range(4) if "Active" in r[6 + i] and "Not" not in r[6 + i]}
            out.append((ts, num(r[2]), num(r[3]), reasons, num(r[4])))
        return out

    def summary(self):
        rows = list(self.samples) if self.samples else self._smi_samples()
        if self.window and self.window[1] is not None:
            t0, t1 = self.window
            inside = [r for r in rows if r[0] is not None and t0 <= r[0] <= t1]
        else:
            inside = rows
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0,
                    "source": self.source}
        sm = [r[1] for r in inside if r[1] is not None]
        smax = [r[2] for r in inside if r[2] is not None]
        pw = [r[4] for r in inside if r[4] is not None]
        reasons = sorted(set().union(*[r[3] for r in inside]))
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": round(max(pw), 1) if pw else None,
                "reasons": reasons, "samples": len(inside), "source": self.source}


def _gpu_uuid(dev) -> str | None:
    """The CUDA device's UUID as NVML names it ("GPU-..."), if torch exposes it."""
    import torch

    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
    except (AttributeError, RuntimeError):
        return None
    return u if u.startswith("GPU-") else f"GPU-{u}"


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _max_over_ranks(val: float, world: int, device) -> float:
    if world == 1:
        return val
    import torch
    import torch.distributed as dist

    t = torch.tensor([val], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def run_ours(args):
    import torch

    import selected_token_logprob_gb300 as flp
    import workloads

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    flp._lib.load()

    wl = workloads.WORKLOADS[args.workload]
    n, v = wl.n, wl.v
    tdt = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[args.dtype]
    ebytes = 4 if args.dtype == "f32" else 2
    temp = args.temperature
    x, y, g = workloads.make(wl, device=dev, seed=wl.seed + rank, dtype=tdt)
    logp = torch.empty(n, dtype=torch.float32, device=dev)
    lse = torch.empty(n, dtype=torch.float32, device=dev)
    lse_lo = torch.empty(n, dtype=torch.float32, device=dev)
    dl = torch.empty((n, v), dtype=tdt, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        flp.fused_logp_forward(x, y, logp=logp, lse=lse, lse_lo=lse_lo, temperature=temp)
        flp.fused_logp_backward(x, y, lse, g, dlogits=dl, lse_lo=lse_lo, temperature=temp)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    # peak memory of a step beyond the resident inputs and outputs (the
    # library allocates nothing; the target is logits + dlogits + O(N))
    base = torch.cuda.memory_allocated(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    step()
    torch.cuda.synchronize(dev)
    step_extra = torch.cuda.max_memory_allocated(dev) - base
    memory = {"logits_bytes": x.numel() * x.element_size(), "dlogits_bytes": dl.numel() * dl.element_size(),
              "per_row_bytes": n * (8 + 4 + 4 + 4 + 4), "step_extra_bytes": int(step_extra),
              "note": "logits, dlogits, targets, grad, logp, lse, lse_lo resident before the step; "
                      "step_extra = max_memory_allocated during one step minus memory_allocated before it"}

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    sampler = ClockSampler(local, _gpu_uuid(dev))
    _barrier(world)
    torch.cuda.synchronize(dev)
    with sampler:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        sampler.mark()
        t0.record(stream)
        for k in range(args.steps):
            ev[k][0].record(stream)
            flp.fused_logp_forward(x, y, logp=logp, lse=lse, lse_lo=lse_lo, temperature=temp)
            ev[k][1].record(stream)
            flp.fused_logp_backward(x, y, lse, g, dlogits=dl, lse_lo=lse_lo, temperature=temp)
            ev[k][2].record(stream)
        t1.record(stream)
        torch.cuda.synchronize(dev)
        sampler.mark()
    _barrier(world)
    total_ms = _max_over_ranks(t0.elapsed_time(t1), world, dev)
    fwd_ms = [e[0].elapsed_time(e[1]) for e in ev]
    bwd_ms = [e[1].elapsed_time(e[2]) for e in ev]
    ms_per_step = total_ms / args.steps
    logits_per_rank = n * v
    bpl = BYTES_PER_LOGIT * ebytes // 2              # algorithmic bytes per logit, this dtype
    value = world * logits_per_rank * bpl / (ms_per_step * 1e-3) / 1e9

    # end to end through the public API from pinned host buffers
    e2e = run_e2e(args, flp, x, y, g, dev, stream, world, temp, bpl)

    peak, peak_src = _peaks()
    bwd_avg = statistics.mean(bwd_ms)
    fwd_avg = statistics.mean(fwd_ms)
    achieved = logits_per_rank * BWD_BYTES_PER_LOGIT * ebytes // 2 / (bwd_avg * 1e-3) / 1e9
    clocks = sampler.summary()
    prof = (_profiled_traffic("k_logp_bwd", parts=True)
            if args.dtype == "bf16" and args.workload == "long" else None)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": round(value / (logits_per_rank * BYTES_PER_LOGIT / (PAGES_FWD_BWD_MS * 1e-3) / 1e9), 3)
        if world == 1 and args.dtype == "bf16" and temp == 1.0 else None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC if args.workload == "long" else args.workload,
                   "n": n, "v": v, "logits_dtype": args.dtype, "temperature": temp,
                   "parallelism": (f"rows x{world}: rank r computes rows [r*{n}, (r+1)*{n}) of one global "
                                   f"batch of {world * n} rows (row block r drawn from seed r), no collective "
                                   f"on the data path" if world > 1 else "single GPU"),
                   "l2": "inputs (9.96 GB) exceed the 129 MB L2; no flush"},
        "fwd_ms": round(fwd_avg, 4), "bwd_ms": round(bwd_avg, 4),
        "fwd_gbs": round(logits_per_rank * FWD_BYTES_PER_LOGIT * ebytes // 2 / (fwd_avg * 1e-3) / 1e9, 1),
        "bwd_gbs": round(achieved, 1),
        "roofline": {"kernel": "k_logp_bwd", "bound": "hbm", "achieved": round(achieved, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_source": peak_src,
                     "traffic": prof["total"] if prof else None,
                     "traffic_read": prof["read"] if prof else None,
                     "traffic_write": prof["write"] if prof else None,
                     "algorithmic_bytes": logits_per_rank * BWD_BYTES_PER_LOGIT * ebytes // 2,
                     "algorithmic_bytes_active": prof["algorithmic_active"] if prof else None,
                     "traffic_note": "ncu dram__bytes_read/write.sum of a full launch (one-pass capture of this "
                                     "command, profiles/k_logp_bwd_long.md); inactive rows are not read, the "
                                     "writes still dirty in L2 at the kernel's end are not counted",
                     "fwd_frac": round(logits_per_rank * FWD_BYTES_PER_LOGIT * ebytes // 2
                                       / (fwd_avg * 1e-3) / 1e9 / peak, 4),
                     "step_frac": round(value / world / peak, 4)},
        "e2e": e2e,
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
        "memory": memory,
        "vs_baseline_note": "pages' fused kernel 27.2 ms fwd+bwd on one B200 (context only)",
    }
    if rank == 0:
        line["cpu_baseline"] = cpu_baseline(args, x, y, g, v)
    if world == 1 and args.side_paths != "none":
        del x, g, dl
        torch.cuda.empty_cache()
        line["side_paths"] = _side_paths(args)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def _side_paths(args):
    """The two other paths of the library, device-timed on the same GPU after
    the logits path's line is complete (its timed region is over): the fused
    LM-head forward (and its backward) at N = 32768, D = 4096, V = 151936, and
    the GRPO loss over 16.8M tokens.  Each keeps its own clock record; its own
    `--path` run adds the end-to-end leg and the oracle."""
    import copy

    out = {}
    for name in args.side_paths.split(","):
        sub = copy.copy(args)
        sub.warmup = 3
        if name == "linear":
            sub.steps, sub.linear_bwd_steps = 10, 3
            line = run_linear(sub, side=True)
            keep = ("metric", "value", "unit", "steps", "ms_per_step", "config", "roofline", "backward",
                    "gpu_launches", "clocks")
        elif name == "grpo":
            sub.steps = 20
            line = run_grpo(sub, side=True)
            keep = ("metric", "value", "unit", "steps", "ms_per_step", "config", "roofline",
                    "token_mean_with_normalizer", "counts_taken_beforehand", "small_call_us", "gpu_launches",
                    "clocks")
        else:
            raise SystemExit(f"--side-paths: unknown path {name!r}")
        out[name] = {k: line[k] for k in keep}
    return out


def run_linear(args, side=False):
    """The fused LM-head forward: one step = one fused_linear_logp_forward
    call (contraction kernel + partial merge) over the whole batch.  With
    `side` (one GPU, called after the logits path's measurement) only the
    device-timed forward and backward are taken and the line is returned."""
    import torch

    import selected_token_logprob_gb300 as flp
    import workloads

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1 and not side:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    flp._lib.load()
    n, d, v = args.linear_n, args.linear_d, workloads.QWEN3_VOCAB
    h, w, y = workloads.linear(n, d, v, seed=rank, device=dev)
    ws = torch.empty(flp.fused_linear_logp_workspace_size(n, v), dtype=torch.uint8, device=dev)
    logp = torch.empty(n, dtype=torch.float32, device=dev)
    lse = torch.empty(n, dtype=torch.float32, device=dev)
    lse_lo = torch.empty(n, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        flp.fused_linear_logp_forward(h, w, y, logp=logp, lse=lse, lse_lo=lse_lo, workspace=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    sampler = ClockSampler(local, _gpu_uuid(dev))
    _barrier(world)
    torch.cuda.synchronize(dev)
    with sampler:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        sampler.mark()
        t0.record(stream)
        for k in range(args.steps):
            ev[k][0].record(stream)
            step()
            ev[k][1].record(stream)
        t1.record(stream)
        torch.cuda.synchronize(dev)
        sampler.mark()
    _barrier(world)
    total_ms = _max_over_ranks(t0.elapsed_time(t1), world, dev)
    ms_per_step = total_ms / args.steps
    flops = 2.0 * n * v * d
    value = world * flops / (ms_per_step * 1e-3) / 1e12
    call_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    achieved = flops / (call_ms * 1e-3) / 1e12
    burst, sustained, src = _tensor_peaks()
    e2e = None if side else _linear_e2e(args, flp, h, w, y, ws, dev, stream, world)
    bwd = _linear_backward_timing(args, flp, h, w, y, lse, lse_lo, dev, stream)
    line = {
        "metric": LIN_METRIC if (n, d) == (32768, 4096) else f"fused LM-head + logp forward TFLOP/s "
                                                            f"at N={n}, D={d}, V={v} BF16",
        "value": round(value, 1), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": LIN_DESC, "n": n, "d": d, "v": v,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": f"inputs ({(n + v) * d * 2 / 1e9:.2f} GB) exceed the 129 MB L2; no flush"},
        "roofline": {"kernel": "k_linear_logp_tiles (+ k_linear_logp_merge in the timed call)",
                     "bound": "tensor", "achieved": round(achieved, 1), "peak": burst, "unit": "TFLOP/s",
                     "frac": round(achieved / burst, 4), "peak_source": src,
                     "frac_of_sustained": round(achieved / sustained, 4),
                     "traffic": _profiled_traffic("k_linear_logp_tiles")
                     if (n, d) == (32768, 4096) else None},
        "e2e": e2e,
        "gpu_launches": 2 * args.steps,
        "clocks": sampler.summary(),
        "backward": bwd,
    }
    if side:
        return line
    if rank == 0:
        line["cpu_baseline"] = _linear_cpu_baseline(args, h, w, y, v, d)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


GRPO_METRIC = "GRPO loss + d loss / d logp GB/s (% HBM roofline) at N=16777216 tokens, 16384 sequences"


def _grpo_inputs(n, nseq, seed, device):
    """Seeded GRPO inputs: logp in (-6, 0), old and ref near it, N(0,1)
    advantages, 10% inactive tokens, nseq packed sequences of random lengths."""
    import torch

    g = torch.Generator().manual_seed(seed)
    lp = -torch.rand(n, generator=g) * 6 - 0.05
    old = lp + (torch.rand(n, generator=g) - 0.5) * 1.2
    ref = lp + (torch.rand(n, generator=g) - 0.5) * 1.0
    adv = torch.randn(n, generator=g)
    mask = (torch.rand(n, generator=g) > 0.1).to(torch.uint8)
    cuts = torch.sort(torch.randint(0, n + 1, (nseq - 1,), generator=g)).values
    cu = torch.cat([torch.zeros(1, dtype=torch.int64), cuts, torch.full((1,), n, dtype=torch.int64)])
    return [t.to(device) for t in (lp, old, ref, adv, mask, cu)]


def run_grpo(args, side=False):
    """The GRPO loss on the logp path over a large RL batch: one call = the
    per-token terms with per-chunk sums, the fixed-order fold (with the
    sequences' folds), the per-sequence weights.  With `side` the end-to-end
    leg and the oracle are skipped and the line is returned."""
    import torch

    import selected_token_logprob_gb300 as flp

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    flp._lib.load()
    n, nseq = args.grpo_n, args.grpo_seqs
    lp, old, ref, adv, mask, cu = _grpo_inputs(n, nseq, 1 + rank, dev)
    ws = torch.empty(flp.logp_grpo_loss_workspace_size(n, nseq), dtype=torch.uint8, device=dev)
    kw = dict(ref_logp=ref, active_mask=mask, cu_seqlens=cu, mode="seq_mean_token_mean", eps_lo=0.2,
              eps_hi=0.28, beta=0.04, workspace=ws)

    def step():
        return flp.logp_grpo_loss(lp, old, adv, **kw)

    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    # a call takes well under a millisecond: time at least a second of them so
    # that the clock sampler (every 200 ms) sees the timed region (the count
    # comes from the wall time of 20 calls, host overhead included)
    t_probe = time.perf_counter()
    for _ in range(20):
        step()
    torch.cuda.synchronize(dev)
    per_call = (time.perf_counter() - t_probe) / 20
    steps = max(args.steps, int(1.0 / max(per_call, 1e-6)))
    sampler = ClockSampler(local, _gpu_uuid(dev))
    with sampler:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        sampler.mark()
        t0.record(stream)
        for _ in range(steps):
            step()
        t1.record(stream)
        torch.cuda.synchronize(dev)
        sampler.mark()
    ms = t0.elapsed_time(t1) / steps
    bpt = 4 * 4 + 1 + 4              # logp, old, ref, adv read + mask read + grad written
    alg = n * bpt + (nseq + 1) * 8
    gbs = alg / (ms * 1e-3) / 1e9
    peak, src = _peaks()
    # token mean with the caller's normaliser (e.g. a count over all
    # micro-batches): the weight is known up front, nothing is counted
    kw_tm = dict(ref_logp=ref, active_mask=mask, cu_seqlens=cu, mode="token_mean", eps_lo=0.2, eps_hi=0.28,
                 beta=0.04, normalizer=float(n), workspace=ws)
    for _ in range(3):
        flp.logp_grpo_loss(lp, old, adv, **kw_tm)
    a_ = torch.cuda.Event(enable_timing=True)
    b_ = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    a_.record(stream)
    for _ in range(args.steps):
        flp.logp_grpo_loss(lp, old, adv, **kw_tm)
    b_.record(stream)
    torch.cuda.synchronize(dev)
    tm_ms = a_.elapsed_time(b_) / args.steps
    # the same call with the batch layout's counts taken beforehand (once per
    # batch, e.g. on a second stream during the logp forward, or reused over
    # several epochs): the token pass alone
    flp.logp_grpo_loss_counts(n, active_mask=mask, cu_seqlens=cu, mode="seq_mean_token_mean", workspace=ws)
    for _ in range(3):
        flp.logp_grpo_loss(lp, old, adv, counted=True, **kw)
    torch.cuda.synchronize(dev)
    a_.record(stream)
    for _ in range(args.steps):
        flp.logp_grpo_loss(lp, old, adv, counted=True, **kw)
    b_.record(stream)
    torch.cuda.synchronize(dev)
    counted_ms = a_.elapsed_time(b_) / args.steps
    # GPU time of one call at the logits workloads' size (32768 tokens, 256
    # sequences): 20 calls captured in a CUDA graph and replayed, so that the
    # host's per-call overhead does not show
    lp2, old2, ref2, adv2, mask2, cu2 = _grpo_inputs(32768, 256, 7, dev)
    ws2 = torch.empty(flp.logp_grpo_loss_workspace_size(32768, 256), dtype=torch.uint8, device=dev)
    kw2 = dict(ref_logp=ref2, active_mask=mask2, cu_seqlens=cu2, mode="seq_mean_token_mean", beta=0.04,
               workspace=ws2)
    for _ in range(3):
        flp.logp_grpo_loss(lp2, old2, adv2, **kw2)
    torch.cuda.synchronize(dev)
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            for _ in range(20):
                flp.logp_grpo_loss(lp2, old2, adv2, **kw2)
    stream.wait_stream(cap)
    graph.replay()
    torch.cuda.synchronize(dev)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(5):
        graph.replay()
    b.record(stream)
    torch.cuda.synchronize(dev)
    small_us = a.elapsed_time(b) / 100 * 1e3
    if side:
        e2e_ms = None
    else:
        e2e_ms, h2d = _grpo_e2e(args, flp, (lp, old, ref, adv, mask, cu), ws, dev, stream)
    line = {
        "metric": GRPO_METRIC if (n, nseq) == (16777216, 16384) else f"GRPO loss GB/s at N={n}, {nseq} sequences",
        "value": round(gbs, 1), "unit": "GB/s", "n_gpus": 1, "steps": steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"GRPO clipped surrogate + k3 KL (beta 0.04), seq_mean_token_mean, {n} tokens in "
                               f"{nseq} packed sequences of random lengths, 10% inactive (synthetic)",
                   "n": n, "num_seqs": nseq, "parallelism": "single GPU",
                   "l2": f"inputs {n * 17 / 1e6:.0f} MB per step against a 129 MB L2 (no flush)"},
        "roofline": {"kernel": "k_grpo_count + k_grpo_fix + k_grpo_pass (the whole call)",
                     "bound": "hbm",
                     "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s", "frac": round(gbs / peak, 4),
                     "peak_source": src, "bytes_per_token": bpt, "traffic": None},
        "small_call_us": {"n": 32768, "num_seqs": 256, "us": round(small_us, 2), "timed": "CUDA graph of 20 calls"},
        "token_mean_with_normalizer": {"ms_per_step": round(tm_ms, 4),
                                       "GB/s": round(alg / (tm_ms * 1e-3) / 1e9, 1),
                                       "frac": round(alg / (tm_ms * 1e-3) / 1e9 / peak, 4)},
        "counts_taken_beforehand": {"ms_per_step": round(counted_ms, 4),
                                    "GB/s": round(alg / (counted_ms * 1e-3) / 1e9, 1),
                                    "frac": round(alg / (counted_ms * 1e-3) / 1e9 / peak, 4),
                                    "note": "logp_grpo_loss(counted=True) after one logp_grpo_loss_counts for "
                                            "the batch layout: the token pass alone"},
        "e2e": None if e2e_ms is None else
        {"value": round(alg / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s", "ms_per_step": round(e2e_ms, 3),
         "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": 4},
        "gpu_launches": 3 * steps,
        "clocks": sampler.summary(),
    }
    if side:
        return line
    if rank == 0 and args.cpu_seconds > 0:
        import oracle

        rows = min(n, 1 << 20)
        hl = [t[:rows].double().cpu().numpy() for t in (lp, old, ref, adv)]
        hm = mask[:rows].cpu().numpy()
        cut = cu.cpu().numpy()
        cut = np.concatenate([cut[cut < rows], [rows]])
        t_start, done = time.perf_counter(), 0
        while True:
            oracle.grpo_loss(hl[0], hl[1], hl[3], ref_logp=hl[2], mask=hm, cu_seqlens=cut,
                             mode="seq_mean_token_mean", eps_lo=0.2, eps_hi=0.28, beta=0.04)
            done += 1
            el = time.perf_counter() - t_start
            if el >= min(args.cpu_seconds, 5.0):
                break
        line["cpu_baseline"] = {"value": round(done * (rows * bpt) / el / 1e9, 3), "unit": "GB/s",
                                "cores": oracle.num_threads(), "kind": "oracle",
                                "sample": f"{done} x {rows} tokens (the first {rows} of the batch), FP64, {el:.1f} s"}
    print(json.dumps(line), flush=True)


def _grpo_e2e(args, flp, inputs, ws, dev, stream):
    """End to end: the step's inputs copied from pinned host memory, the loss
    read back; returns (ms per step, host-to-device bytes per step)."""
    import torch

    host = [t.cpu().pin_memory() for t in inputs]
    devs = [torch.empty_like(t) for t in inputs]
    hloss = torch.empty(1, dtype=torch.float32).pin_memory()

    def e2e_step():
        for d_, h_ in zip(devs, host):
            d_.copy_(h_, non_blocking=True)
        loss, _ = flp.logp_grpo_loss(devs[0], devs[1], devs[3], ref_logp=devs[2], active_mask=devs[4],
                                     cu_seqlens=devs[5], mode="seq_mean_token_mean", eps_lo=0.2, eps_hi=0.28,
                                     beta=0.04, workspace=ws)
        hloss.copy_(loss, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize(dev)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(max(1, args.e2e_steps)):
        e2e_step()
    b.record(stream)
    torch.cuda.synchronize(dev)
    return a.elapsed_time(b) / max(1, args.e2e_steps), sum(t.numel() * t.element_size() for t in host)


def _linear_backward_timing(args, flp, h, w, y, lse, lse_lo, dev, stream):
    """The fused LM-head backward (dZ recomputed on the tensor cores per
    4096-row chunk, then dH = dZ W and dW = dZ^T H on the library's own
    tensor-core contraction kernel): 3 contractions of 2 N V D FLOP each,
    timed separately from the forward's metric."""
    import torch

    n, d = h.shape
    v = w.shape[0]
    if args.linear_bwd_steps <= 0:
        return None
    g = torch.full((n,), 1.0 / n, dtype=torch.float32, device=dev)
    wsb = torch.empty(flp.fused_linear_logp_backward_workspace_size(d, v), dtype=torch.uint8, device=dev)
    dh = torch.empty((n, d), dtype=torch.float32, device=dev)
    dw = torch.empty((v, d), dtype=torch.float32, device=dev)

    def call():
        flp.fused_linear_logp_backward(h, w, y, lse, g, lse_lo=lse_lo, dhidden=dh, dweight=dw, workspace=wsb)

    call()
    torch.cuda.synchronize(dev)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.linear_bwd_steps):
        call()
    b.record(stream)
    torch.cuda.synchronize(dev)
    ms = a.elapsed_time(b) / args.linear_bwd_steps
    burst, sustained, _ = _tensor_peaks()
    tf = 3 * 2.0 * n * v * d / (ms * 1e-3) / 1e12
    return {"ms": round(ms, 3), "tflops": round(tf, 1), "frac": round(tf / burst, 4),
            "frac_of_sustained": round(tf / sustained, 4), "steps": args.linear_bwd_steps,
            "flop_per_call": 3 * 2.0 * n * v * d,
            "kernels": "per 4096-row chunk: k_linear_logp_tiles<grad> (dZ, BF16), k_gemm_bf16_pair (dH, 5 K splits) + "
                        "k_gemm_split_sum, k_gemm_bf16_pair (dW, added over the chunks)"}


def _linear_e2e(args, flp, h, w, y, ws, dev, stream, world):
    """Through the public API with every input copied from pinned host memory
    each step (hidden, targets and the LM-head weight) and logp/lse read back.
    The weight goes over in vocabulary slices on the tile grid, on two copy
    streams, and each slice's tile partials are computed as soon as it lands
    (the vocabulary-sharded entry points: bitwise the same result as one call);
    the fixed-order merge follows."""
    import torch

    n, d = h.shape
    v = w.shape[0]
    hh = torch.empty(h.shape, dtype=h.dtype, pin_memory=True)
    hh.copy_(h)
    hw = torch.empty(w.shape, dtype=w.dtype, pin_memory=True)
    hw.copy_(w)
    hy = y.cpu().pin_memory()
    hlogp = torch.empty(n, dtype=torch.float32).pin_memory()
    hlse = torch.empty(n, dtype=torch.float32).pin_memory()
    dh, dw, dy = torch.empty_like(h), torch.empty_like(w), torch.empty_like(y)
    tiles = -(-v // 256)
    slices = max(1, min(args.e2e_chunks, tiles))
    per = -(-tiles // slices) * 256
    bounds = [(a, min(v, a + per)) for a in range(0, v, per)]
    copy_streams = [torch.cuda.Stream(dev) for _ in range(2)]
    h_landed = torch.cuda.Event()
    landed = [torch.cuda.Event() for _ in bounds]

    def step():
        for cs in copy_streams:
            cs.wait_stream(stream)             # the previous step is done with these buffers
        with torch.cuda.stream(copy_streams[0]):
            dh.copy_(hh, non_blocking=True)
            dy.copy_(hy, non_blocking=True)
            h_landed.record(copy_streams[0])
        for k, (a, b) in enumerate(bounds):
            cs = copy_streams[k % 2]
            with torch.cuda.stream(cs):
                dw[a:b].copy_(hw[a:b], non_blocking=True)
                landed[k].record(cs)
        stream.wait_event(h_landed)
        for k, (a, b) in enumerate(bounds):
            stream.wait_event(landed[k])
            flp.fused_linear_logp_shard_partials(dh, dw[a:b], a, v, dy, ws)
        logp, lse = flp.fused_linear_logp_merge(ws, v, dy)
        hlogp.copy_(logp, non_blocking=True)
        hlse.copy_(lse, non_blocking=True)

    steps = max(1, min(args.steps, args.e2e_steps))
    step()
    torch.cuda.synchronize(dev)
    _barrier(world)
    a_ev = torch.cuda.Event(enable_timing=True)
    b_ev = torch.cuda.Event(enable_timing=True)
    a_ev.record(stream)
    for _ in range(steps):
        step()
    b_ev.record(stream)
    torch.cuda.synchronize(dev)
    ms = _max_over_ranks(a_ev.elapsed_time(b_ev) / steps, world, dev)
    return {"value": round(world * 2.0 * n * v * d / (ms * 1e-3) / 1e12, 1), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 3), "steps": steps,
            "h2d_bytes_per_step": (n + v) * d * 2 + n * 8, "d2h_bytes_per_step": n * 4 * 2,
            "pipeline": f"weight in {len(bounds)} vocabulary slices on 2 copy streams, each slice's tile "
                        f"partials computed as it lands, then the merge"}

def _linear_cpu_baseline(args, h, w, y, v, d):
    """The FP64 oracle on a bounded row sample of the same workload."""
    import oracle
    import workloads

    if args.cpu_seconds <= 0:
        return None
    wb = workloads.bf16_bits(w)
    hb = workloads.bf16_bits(h[:64])
    yn = y[:64].cpu().numpy()
    rows, t0 = 0, time.perf_counter()
    while True:
        k = 16
        a = rows % 64
        oracle.linear_logp(hb[a:a + k], wb, yn[a:a + k], d=d)
        rows += k
        el = time.perf_counter() - t0
        if el >= args.cpu_seconds:
            break
    return {"value": round(2.0 * rows * v * d / el / 1e12, 5), "unit": "TFLOP/s",
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{rows} rows of the fused LM-head workload (first rows of the batch, full "
                      f"V x D contraction per row in FP64), {el:.1f} s"}


def run_e2e(args, flp, x, y, g, dev, stream, world, temp=1.0, bpl=BYTES_PER_LOGIT):
    """End to end through the public API: every step copies that step's
    logits, targets and upstream gradients from pinned host memory and reads
    logp and lse back.  The copy goes in row chunks on two copy streams, and
    each chunk's forward + backward starts as soon as its rows have landed
    (rows are independent and every row's result is batch-invariant, so the
    chunked step gives the same bits as one call over all rows)."""
    import torch

    n, v = x.shape
    hx = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
    hx.copy_(x)
    hy = y.cpu().pin_memory()
    hg = g.cpu().pin_memory()
    hlogp = torch.empty(n, dtype=torch.float32).pin_memory()
    hlse = torch.empty(n, dtype=torch.float32).pin_memory()
    dx = torch.empty_like(x)
    dy = torch.empty_like(y)
    dg = torch.empty_like(g)
    logp = torch.empty(n, dtype=torch.float32, device=dev)
    lse = torch.empty(n, dtype=torch.float32, device=dev)
    lse_lo = torch.empty(n, dtype=torch.float32, device=dev)
    dl = torch.empty_like(x)
    chunks = max(1, min(args.e2e_chunks, n))
    per = -(-n // chunks)
    ranges = [(a, min(n, a + per)) for a in range(0, n, per)]
    copy_streams = [torch.cuda.Stream(dev) for _ in range(2)]
    landed = [torch.cuda.Event() for _ in ranges]

    def step():
        for k, (a, b) in enumerate(ranges):
            cs = copy_streams[k % 2]
            cs.wait_stream(stream)          # the previous step is done with these rows
            with torch.cuda.stream(cs):
                dx[a:b].copy_(hx[a:b], non_blocking=True)
                dy[a:b].copy_(hy[a:b], non_blocking=True)
                dg[a:b].copy_(hg[a:b], non_blocking=True)
                landed[k].record(cs)
        for k, (a, b) in enumerate(ranges):
            stream.wait_event(landed[k])
            flp.fused_logp_forward(dx[a:b], dy[a:b], logp=logp[a:b], lse=lse[a:b], lse_lo=lse_lo[a:b],
                                   temperature=temp)
            flp.fused_logp_backward(dx[a:b], dy[a:b], lse[a:b], dg[a:b], dlogits=dl[a:b],
                                    lse_lo=lse_lo[a:b], temperature=temp)
        hlogp.copy_(logp, non_blocking=True)
        hlse.copy_(lse, non_blocking=True)

    steps = max(1, min(args.steps, args.e2e_steps))
    for _ in range(2):
        step()
    torch.cuda.synchronize(dev)
    _barrier(world)
    a_ev = torch.cuda.Event(enable_timing=True)
    b_ev = torch.cuda.Event(enable_timing=True)
    a_ev.record(stream)
    for _ in range(steps):
        step()
    b_ev.record(stream)
    torch.cuda.synchronize(dev)
    ms = _max_over_ranks(a_ev.elapsed_time(b_ev) / steps, world, dev)
    del hx
    return {"value": round(world * n * v * bpl / (ms * 1e-3) / 1e9, 2), "unit": UNIT,
            "ms_per_step": round(ms, 3), "steps": steps,
            "h2d_bytes_per_step": n * v * x.element_size() + n * 8 + n * 4,
            "d2h_bytes_per_step": n * 4 * 2,
            "pipeline": f"{len(ranges)} row chunks, 2 copy streams overlapping the compute"}

def _oracle_sample_rate(x_rows_u16, y_np, g_np, v, seconds: float):
    """GB/s-equivalent of the FP64 oracle (forward + dense backward) on a
    cycling row sample, for about `seconds` of wall time."""
    import numpy as np

    import oracle

    chunk = 64
    rows_done = 0
    t0 = time.perf_counter()
    t_fwd = t_bwd = 0.0
    i = 0
    nrows = x_rows_u16.shape[0]
    while True:
        a = (i * chunk) % nrows
        xb = np.ascontiguousarray(x_rows_u16[a:a + chunk])
        yb = y_np[a:a + chunk]
        gb = g_np[a:a + chunk]
        ta = time.perf_counter()
        oracle.forward(xb, yb)
        tb = time.perf_counter()
        oracle.backward(xb, yb, gb)
        t_fwd += tb - ta
        t_bwd += time.perf_counter() - tb
        rows_done += xb.shape[0]
        i += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return rows_done * v * BYTES_PER_LOGIT / el / 1e9, rows_done, el, t_fwd / rows_done, t_bwd / rows_done


def cpu_baseline(args, x, y, g, v):
    import oracle
    import workloads

    if args.cpu_seconds <= 0 or x.dtype != __import__("torch").bfloat16:
        return None
    rows = min(512, x.shape[0])
    xs = workloads.bf16_bits(x[:rows])
    rate, done, el, fwd_row, bwd_row = _oracle_sample_rate(xs, y[:rows].cpu().numpy(), g[:rows].cpu().numpy(), v,
                                                           args.cpu_seconds)
    n = x.shape[0]
    return {"value": round(rate, 4), "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{done} rows of the {getattr(args, 'workload', 'long')} workload (first {rows} rows, "
                      f"cycled), FP64 forward + dense backward, {el:.1f} s",
            "ms_extrapolated": {"fwd": round(fwd_row * n * 1e3, 1), "bwd": round(bwd_row * n * 1e3, 1),
                                "total": round((fwd_row + bwd_row) * n * 1e3, 1),
                                "note": f"per-row time of the sample times N = {n} rows (linear extrapolation)"}}


def run_reference(args):
    """The FP64 CPU oracle as the reference arm (rank 0 only)."""
    world, rank, _ = _dist()
    if rank != 0:
        return
    import oracle
    import workloads

    oracle.build()
    if args.path == "linear":
        return _run_reference_linear(args, world)
    if args.path == "grpo":
        return _run_reference_grpo(args, world)
    wl = workloads.WORKLOADS[args.workload]
    rows = args.ref_rows
    x, y, g = workloads.make(wl, n=rows)   # same recipe, a bounded row sample, on the host
    xb = workloads.bf16_bits(x)
    yn, gn = y.numpy(), g.numpy()
    for _ in range(args.warmup):
        oracle.forward(xb, yn)
        oracle.backward(xb, yn, gn)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.forward(xb, yn)
        oracle.backward(xb, yn, gn)
        times.append(time.perf_counter() - t0)
    sec = statistics.mean(times)
    value = rows * wl.v * BYTES_PER_LOGIT / sec / 1e9
    sample = (f"{rows} rows of the long-CoT workload per step (FP64 forward + dense backward); "
              f"GB/s counts the same 6 B/logit")
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": WORKLOAD_DESC, "n": wl.n, "v": wl.v, "rows_per_step": rows},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def _run_reference_linear(args, world):
    """The FP64 oracle of the fused LM head on a bounded row sample."""
    import oracle
    import workloads

    n, d, v = args.linear_n, args.linear_d, workloads.QWEN3_VOCAB
    rows = max(1, min(args.ref_rows // 8, n))
    h, w, y = workloads.linear(rows, d, v, seed=0)      # the recipe's first rows, on the host
    hb, wb, yn = workloads.bf16_bits(h), workloads.bf16_bits(w), y.numpy()
    for _ in range(min(args.warmup, 1)):
        oracle.linear_logp(hb, wb, yn, d=d)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.linear_logp(hb, wb, yn, d=d)
        times.append(time.perf_counter() - t0)
    sec = statistics.mean(times)
    value = 2.0 * rows * v * d / sec / 1e12
    sample = f"{rows} rows of the fused LM-head workload per step (FP64 contraction + log-softmax)"
    line = {
        "metric": LIN_METRIC, "value": round(value, 5), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": LIN_DESC, "n": n, "d": d, "v": v, "rows_per_step": rows},
        "cpu_baseline": {"value": round(value, 5), "unit": "TFLOP/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 5), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def _run_reference_grpo(args, world):
    """The FP64 oracle of the GRPO loss on a bounded sample of the GRPO
    workload: the sequences that lie in its first --ref-rows x 8192 tokens."""
    import oracle

    n, nseq = args.grpo_n, args.grpo_seqs
    lp, old, ref, adv, mask, cu = _grpo_inputs(n, nseq, 1, "cpu")
    rows = min(n, max(1, args.ref_rows) * 8192)
    cut = cu.numpy()
    cut = np.concatenate([cut[cut < rows], [rows]])
    hl = [t[:rows].double().numpy() for t in (lp, old, ref, adv)]
    hm = mask[:rows].numpy()
    kw = dict(ref_logp=hl[2], mask=hm, cu_seqlens=cut, mode="seq_mean_token_mean", eps_lo=0.2, eps_hi=0.28,
              beta=0.04)
    for _ in range(min(args.warmup, 1)):
        oracle.grpo_loss(hl[0], hl[1], hl[3], **kw)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.grpo_loss(hl[0], hl[1], hl[3], **kw)
        times.append(time.perf_counter() - t0)
    sec = statistics.mean(times)
    bpt = 4 * 4 + 1 + 4
    value = rows * bpt / sec / 1e9
    sample = f"the first {rows} tokens of the GRPO workload per step (FP64 loss and gradient); same 21 B/token"
    metric = GRPO_METRIC if (n, nseq) == (16777216, 16384) else f"GRPO loss GB/s at N={n}, {nseq} sequences"
    line = {
        "metric": metric, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": f"GRPO clipped surrogate + k3 KL (beta 0.04), seq_mean_token_mean, {n} tokens in "
                               f"{nseq} packed sequences of random lengths, 10% inactive (synthetic)",
                   "n": n, "num_seqs": nseq, "tokens_per_step": rows},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200,
                    help="timed steps (200 x 4.3 ms: long enough for several clock samples)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="long")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--e2e-chunks", type=int, default=8,
                    help="row chunks of the end-to-end step (host copies overlap the compute)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-rows", type=int, default=128)
    ap.add_argument("--dtype", choices=["bf16", "f16", "f32"], default="bf16",
                    help="logits dtype (the metric is quoted for bf16)")
    ap.add_argument("--temperature", type=float, default=1.0)
    ap.add_argument("--path", choices=["logits", "linear", "grpo"], default="logits",
                    help="logits: logp fwd+bwd over BF16 logits (the headline); "
                         "linear: fused LM head + logp forward")
    ap.add_argument("--side-paths", default="linear,grpo",
                    help="with the logits path on one GPU: also device-time these paths after its line is "
                         "complete and attach them under side_paths ('none' to skip)")
    ap.add_argument("--linear-n", type=int, default=32768)
    ap.add_argument("--linear-d", type=int, default=4096)
    ap.add_argument("--grpo-n", type=int, default=16777216)
    ap.add_argument("--grpo-seqs", type=int, default=16384)
    ap.add_argument("--linear-bwd-steps", type=int, default=5,
                    help="timed calls of the fused LM-head backward (0: skip)")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)   # at least 3 untimed warm-up steps
    if args.impl == "reference":
        run_reference(args)
    elif args.path == "linear":
        run_linear(args)
    elif args.path == "grpo":
        run_grpo(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
