#!/usr/bin/env python
"""Benchmark of the block-sparse spatio-temporal attention path on GB300.

Step = one pass of the per-layer hot path of the blog "Accelerating
Spatio-Temporal Attention for Video Diffusion on TPUs" (Figure 8) over one
batch of synthetic input, all on the GPU, two launches:
  flag-driven permutation of Q, K, V (one launch)  ->  block-sparse attention
  (exact mask, full / boundary tiles) whose stores put O back in (F,H,W) order
on 75,600 tokens (21 x 45 x 80 latent patches) x 10 heads x d = 128, bf16,
5 spatial heads (frame window 3 + first-frame sink) and 5 temporal heads
(raster window 612 + sink) picked by seeded flags.  The tile map is built once
before timing (it depends only on the geometry, as on the pages).

value = effective TFLOP/s = 4 * d * (retained query-key pairs, all heads) /
step time; ms_per_step is the step time.  Extra keys report the attention
kernel alone, its roofline against the measured bf16 peak (over the timed
steps, and again as a burst after idle and sustained for seconds at the
board's power limit, each against the peak measured in that regime), the
dense control, the tile-aligned (B3) and the no-permutation variants, the
permutation bandwidth, an end-to-end number through host buffers, and the fp64
oracle on the host cores.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "sparse-attn ms & TFLOP/s, 75.6K tok×10h×d128 bf16, % of BF16 TC peak"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
ATTN_SOURCES = ["block_sparse_spatio_gb300/csrc/bss_attention.cu", "block_sparse_spatio_gb300/csrc/bss_ptx.cuh"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "attn_fwd_mixed75k_dram_traffic.txt")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mixed_75600tok_10h_d128")
    ap.add_argument("--heads", type=int, default=0, help="override head count (profiling runs)")
    ap.add_argument("--no-extras", action="store_true", help="skip variants, e2e and cpu baseline")
    ap.add_argument("--rounding", type=int, default=0, choices=[0, 1, 2],
                    help="mask of the timed step: 0 exact (B2, default), 1 tile-aligned (B3), 2 every visited "
                         "tile masked (B1); profiling runs")
    ap.add_argument("--dense", action="store_true",
                    help="time the dense control (every tile, no permutation) instead of the sparse step; "
                         "profiling runs")
    ap.add_argument("--cpu-rows-per-head", type=int, default=6144,
                    help="oracle sample of the cpu_baseline entry (about 20 s on 16 cores)")
    ap.add_argument("--cpu-rows-per-head-1core", type=int, default=64,
                    help="oracle sample of the cpu_baseline's one-core figure")
    ap.add_argument("--ref-rows-per-head", type=int, default=256,
                    help="oracle sample per step of --impl reference")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


# ---- replicas: every rank runs its own batch, no data exchange (weak scaling)
def replica_seed(w, rank: int) -> int:
    """Seed of rank `rank`'s synthetic batch: a different batch on every rank."""
    return w.index + 1000 * rank


def max_over_ranks(x: float, world: int, device) -> float:
    """The slowest rank's figure (the timing rule: max over ranks)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank: float, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank's work over the slowest rank's time."""
    return flops_per_rank * world / (ms_per_step * 1e-3) / 1e12


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return {k: float(p[k]) for k in ("bf16_tflops", "bf16_tflops_sustained", "hbm_gbs")}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def _code_only(text: str) -> str:
    """C++ source without comments and with whitespace collapsed: what the
    compiler sees (a comment edit does not change the kernel)."""
    out, i, n = [], 0, len(text)
    while i < n:
        if text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif text[i] == '"':
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(text[i])
            i += 1
    return " ".join("".join(out).split())


def source_hash():
    """Hash of the attention kernel's code (comments and layout excluded)."""
    h = hashlib.sha256()
    for rel in ATTN_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def traffic_from_profile():
    """DRAM bytes per attention launch from the committed ncu summary, or None
    when the kernel source changed since the counters were taken."""
    try:
        kv = {}
        with open(TRAFFIC_FILE) as fh:
            for line in fh:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("source_sha256_16") != source_hash():
            return None
        return float(kv["dram_bytes_per_full_launch"])
    except Exception:
        return None


class NvmlClockSampler:
    """In-process NVML sampling (read-only queries through ctypes) of the SM
    clock, its maximum, the power draw and the clock-event reasons, every
    `period_s` seconds on a background thread; only samples taken between
    mark_begin() and mark_end() are kept."""
    # clock-event reason bits of nvmlDeviceGetCurrentClocksEventReasons (nvml.h)
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, uuid: str | None, pci_bus_id: str | None, period_s: float = 0.005):
        import ctypes
        self.ok = False
        self.period = period_s
        self.samples = []
        self.t_begin = self.t_end = None
        self._stop = threading.Event()
        self.thread = None
        self.power_instant = True  # cleared once the instantaneous field is refused
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            # NVML sees every GPU of the machine: find this process's GPU by its
            # UUID or PCI bus id (an index could name another GPU)
            h = ctypes.c_void_p()
            rc = 1
            if uuid:
                rc = lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h))
            if rc != 0 and pci_bus_id:
                rc = lib.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(), ctypes.byref(h))
            if rc != 0:
                return
            self.lib, self.h, self.ct = lib, h, ctypes
            mx = ctypes.c_uint()
            self.max_mhz = float(mx.value) if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0 else None
            self.reason_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self.ok = True
        except Exception:
            self.ok = False

    def _instant_power_w(self):
        """The instantaneous board power (field NVML_FI_DEV_POWER_INSTANT, mW),
        or None where the driver does not serve it.  nvmlDeviceGetPowerUsage
        averages over about a second, which lags a timed region of 0.1-0.4 s."""
        ct = self.ct

        class FieldValue(ct.Structure):  # nvmlFieldValue_t (nvml.h)
            _fields_ = [("fieldId", ct.c_uint), ("scopeId", ct.c_uint), ("timestamp", ct.c_longlong),
                        ("latencyUsec", ct.c_longlong), ("valueType", ct.c_int), ("nvmlReturn", ct.c_int),
                        ("value", ct.c_ulonglong)]

        fv = FieldValue(fieldId=186)
        try:
            if self.lib.nvmlDeviceGetFieldValues(self.h, 1, ct.byref(fv)) != 0 or fv.nvmlReturn != 0:
                return None
        except Exception:
            return None
        raw = fv.value
        if fv.valueType == 0:  # double
            mw = ct.c_double.from_buffer_copy(ct.c_ulonglong(raw)).value
        elif fv.valueType in (1, 5, 6):  # 32- or 16-bit integers
            mw = raw & (0xFFFF if fv.valueType == 6 else 0xFFFFFFFF)
        else:
            mw = raw
        return float(mw) / 1e3

    def _one(self):
        ct, lib, h = self.ct, self.lib, self.h
        mhz, mw, rs = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        if lib.nvmlDeviceGetClockInfo(h, 1, ct.byref(mhz)) != 0:
            return None
        power = self._instant_power_w() if self.power_instant else None
        if power is None:
            self.power_instant = False
            power = float(mw.value) / 1e3 if lib.nvmlDeviceGetPowerUsage(h, ct.byref(mw)) == 0 else None
        reasons = int(rs.value) if self.reason_fn(h, ct.byref(rs)) == 0 else 0
        return (time.monotonic(), float(mhz.value), power, reasons)

    def _loop(self):
        while not self._stop.is_set():
            smp = self._one()
            if smp is not None:
                self.samples.append(smp)
            time.sleep(self.period)

    def start(self):
        if self.ok:
            self.thread = threading.Thread(target=self._loop, daemon=True)
            self.thread.start()

    def mark_begin(self):
        self.t_begin = time.monotonic()

    def mark_end(self):
        self.t_end = time.monotonic()

    def stop(self):
        self._stop.set()
        if self.thread:
            self.thread.join(timeout=2)
        kept = [x for x in self.samples if self.t_begin is not None and self.t_begin <= x[0] <= self.t_end]
        return summarize_clocks([x[1] for x in kept], [self.max_mhz] if self.max_mhz else [],
                                [x[2] for x in kept if x[2] is not None],
                                {nm for x in kept for bit, nm in self.REASONS.items() if x[3] & bit},
                                f"in-process NVML every {self.period * 1e3:.0f} ms; power: "
                                + ("instantaneous" if self.power_instant else "NVML's one-second average"))


def summarize_clocks(sm, smax, power, reasons, how):
    return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
            "sm_mhz_min": min(sm) if sm else None, "power_w_max": max(power) if power else None,
            "reasons": sorted(reasons), "samples": len(sm),
            "window": f"samples taken between the start and the end of the timed region ({how})"}


def clock_sampler(torch, device_index: int):
    """The NVML sampler when the driver's library answers, else nvidia-smi."""
    uuid = bus = None
    try:
        prop = torch.cuda.get_device_properties(device_index)
    except Exception:
        prop = None
    try:
        u = str(prop.uuid)
        uuid = u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        uuid = None
    try:
        bus = f"{prop.pci_domain_id:08X}:{prop.pci_bus_id:02X}:{prop.pci_device_id:02X}.0"
    except Exception:
        bus = None
    s = NvmlClockSampler(uuid, bus)
    return s if s.ok else ClockSampler(device_index)


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed
    region (the fallback when NVML cannot be loaded in-process)."""
    QUERY = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None
        self.t_begin = self.t_end = None

    def mark_begin(self):
        self.t_begin = datetime.datetime.now()

    def mark_end(self):
        self.t_end = datetime.datetime.now()

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
                if self.t_begin is not None and not (self.t_begin <= ts <= self.t_end):
                    continue  # outside the timed region
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        return summarize_clocks(sm, smax, power, reasons, "nvidia-smi every 50 ms")


# --------------------------------------------------------------------------- oracle (host)
def oracle_sample(w, q, k, v, flags, rows_per_head, seed):
    """Time the fp64 oracle on seeded query rows of every head; return
    (seconds, rows evaluated, retained pairs of those rows)."""
    import oracle
    import workloads as W
    g = oracle.Geometry(w.F, w.Hs, w.Ws, wf=w.wf, ws=w.ws, bkv=128)
    t0 = time.perf_counter()
    nrows = 0
    for h in range(q.shape[0]):
        kind = oracle.TEMPORAL_PERMUTED if flags[h] else oracle.SPATIAL
        rows = W.sample_rows(w.N, rows_per_head, seed=seed + h)
        oracle.attention(W.bf16_bits(q[h]), W.bf16_bits(k[h]), W.bf16_bits(v[h]), kind, g, rows=rows)
        nrows += len(rows)
    return time.perf_counter() - t0, nrows


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return
    import oracle
    import workloads as W
    w = W.BY_NAME[args.workload]
    H = args.heads or w.H
    flags = w.head_flags()[:H]
    q, k, v = W.qkv(w, H=H)
    flops_total = 4.0 * w.d * retained_total(w, flags)
    rows_total = H * w.N
    rows_per_head = max(8, args.ref_rows_per_head)
    times = []
    for i in range(args.warmup + args.steps):
        dt, nrows = oracle_sample(w, q, k, v, flags, rows_per_head, seed=1000 + i)
        if i >= args.warmup:
            times.append(dt * rows_total / nrows)   # seconds for the whole workload
    step_s = statistics.median(times)
    val = flops_total / step_s / 1e12
    cores = oracle.num_threads()
    sample = (f"{rows_per_head} seeded query rows per head x {H} heads per step "
              f"({100.0 * rows_per_head * H / rows_total:.2f}% of rows), time scaled to all {rows_total} rows")
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "tokens": w.N, "heads": H, "head_dim": w.d, "mask": "exact"},
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def retained_total(w, flags):
    """Exact retained pairs summed over heads (closed forms of the two masks)."""
    F, S = w.F, w.S
    sp = S * S * sum(min(f + w.wf, F - 1) - max(f - w.wf, 0) + 1 + (1 if f > w.wf else 0) for f in range(F))
    tp = 0
    for s in range(S):
        b = min(s + w.ws, S - 1) - max(s - w.ws, 0) + 1
        tp += F * b + (S - b)
    tp *= F
    return sum(tp if fl else sp for fl in flags)


# --------------------------------------------------------------------------- GPU arm
def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
        return
    import torch
    import torch.distributed as dist

    import block_sparse_spatio_gb300 as bss
    import workloads as W

    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    bss.load()
    peaks, peak_src = load_peaks()

    w = W.BY_NAME[args.workload]
    H = args.heads or w.H
    flags = w.head_flags()[:H]
    # replicas: every rank runs its own batch (different seed), no data exchange
    Q, K, V = W.qkv_device(w, dev, seed=replica_seed(w, rank))
    if H != w.H:
        Q, K, V = (x[:H].contiguous() for x in (Q, K, V))
    O = torch.empty_like(Q)
    Qp, Kp, Vp = (torch.empty_like(Q) for _ in range(3))
    fl = torch.tensor(flags, dtype=torch.uint8, device=dev)
    params = bss.MaskParams(w.F, w.Hs, w.Ws, w.d, w.wf, w.ws, temporal_permuted=1, rounding=args.rounding)
    tm = bss.build_tile_map(params)
    st = (tm.stats(0), tm.stats(1))
    retained = sum(st[f]["retained_pairs"] for f in flags)
    if args.dense:
        retained = H * w.N * w.N
    flops = 4.0 * w.d * retained
    stream = torch.cuda.current_stream()
    attn_events = []

    def step(record=False):
        if args.dense:
            if record:
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
            bss.dense_attention(Q, K, V, O)
            if record:
                e1.record(stream)
                attn_events.append((e0, e1))
            return
        # temporal heads' Q, K, V permuted into the workspaces (one launch),
        # spatial heads used in place
        bss.permute_flagged_multi((Q, K, V), (Qp, Kp, Vp), fl, params)
        if record:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
        # the temporal heads' O rows are stored straight to their (F,H,W) rows
        bss.sparse_attention_split(Q, K, V, O, Qp, Kp, Vp, None, tm, fl)
        if record:
            e1.record(stream)
            attn_events.append((e0, e1))

    launches_per_step = 1 if args.dense else 2
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    status = bss.get_device_status()
    if status != 0:
        raise RuntimeError(f"device status {bss.status_string(status)} during warm-up")

    sampler = clock_sampler(torch, local_rank)
    sampler.start()
    time.sleep(0.3)
    sampler.mark_begin()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        step(record=True)
    t1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    sampler.mark_end()
    clocks = sampler.stop()
    elapsed_ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    status = bss.get_device_status()
    if status != 0:
        raise RuntimeError(f"device status {bss.status_string(status)} in the timed region")
    ms_per_step = elapsed_ms / args.steps
    attn_ms = statistics.mean(a.elapsed_time(b) for a, b in attn_events)
    value = whole_job_tflops(flops, world, ms_per_step)
    attn_tflops = flops / (attn_ms * 1e-3) / 1e12
    dense_ctl = None
    if not args.dense and not args.no_extras:
        dense_ctl = dense_control(bss, torch, Q, K, V, O, Qp, Kp, Vp, tm, fl, retained, peaks)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "tokens": w.N, "frames_x_h_x_w": [w.F, w.Hs, w.Ws], "heads": H,
                   "head_dim": w.d, "flags_temporal": flags, "spatial_frame_window": w.wf,
                   "temporal_raster_window": w.ws, "mask": ("dense control" if args.dense else
                            ["exact (full/boundary tiles, B2)", "tile-aligned (B3)",
                             "every visited tile masked (B1)"][args.rounding]), "tile": [tm.BQ, tm.BKV],
                   "step": ("dense attention" if args.dense else
                            "permute temporal heads' QKV (one launch) -> sparse attention storing their O rows in (F,H,W) order"),
                   "l2": f"inputs larger than L2 (Q+K+V = {3 * Q.numel() * 2 / 1e6:.0f} MB)",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "retained_pairs": retained,
                   "retained_fraction": retained / (H * w.N * w.N)},
        "attention": {"ms": attn_ms, "tflops": attn_tflops,
                      "frac_of_peak": attn_tflops / peaks["bf16_tflops"],
                      "frac_of_sustained_peak": attn_tflops / peaks["bf16_tflops_sustained"],
                      "tile_stats": {"spatial": st[0], "temporal": st[1]}},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    if dense_ctl is not None:
        line["dense_control"] = dense_ctl
    traffic = traffic_from_profile()
    if H != w.H and traffic is not None:
        traffic = traffic * H / w.H
    line["roofline"] = {"bound": "tensor", "achieved": attn_tflops, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                        "frac": attn_tflops / peaks["bf16_tflops"], "traffic": traffic,
                        "peak_source": f"{peak_src} bf16 burst (cuBLAS 8192^3)", "kernel": "attn_fwd_kernel<128, false, 2>"}
    if not args.dense and not args.no_extras and rank == 0:
        # the timed region above sits on the power ramp (the board reaches its
        # limit after ~0.1-0.5 s of load); these two legs time the kernel at
        # either end of it, each against the peak measured in the same regime
        line["roofline"].update(power_regimes(bss, torch, Q, K, V, O, Qp, Kp, Vp, tm, fl, flops, peaks, local_rank))

    if not args.no_extras and rank == 0:
        line["variants"] = variants(bss, torch, W, w, H, Q, K, V, dev, peaks, flags)
        line["e2e"] = e2e(bss, torch, params, tm, flags, Q, K, V, flops, args)
    if not args.no_extras and rank == 0 and world == 1:
        line["cpu_baseline"] = cpu_baseline(w, Q, K, V, flags, args, flops)
    tm.destroy()
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def _time(torch, fn, reps=5, warm=3):
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    ev = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        fn()
        b.record(s)
        ev.append((a, b))
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in ev)


def _time_batched(torch, fn, reps=20, warm=3):
    """Mean device time of a short launch: `reps` launches back to back between
    one pair of events, so that the host's per-call work (argument checks,
    ctypes marshalling) overlaps the device work instead of sitting between an
    event and the launch it brackets."""
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s)
    for _ in range(reps):
        fn()
    b.record(s)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def _time_interleaved(torch, fns, rounds=9, warm=2):
    """Median time of each of several launches compared with one another: every
    round times each once, in an order rotated from round to round, so clock
    drift under the power cap falls on all of them alike."""
    names = list(fns)
    for _ in range(warm):
        for n in names:
            fns[n]()
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    ev = {n: [] for n in names}
    for r in range(rounds):
        for i in range(len(names)):
            n = names[(i + r) % len(names)]
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            fns[n]()
            b.record(s)
            ev[n].append((a, b))
    torch.cuda.synchronize()
    return {n: statistics.median(a.elapsed_time(b) for a, b in ev[n]) for n in names}


def power_regimes(bss, torch, Q, K, V, O, Qp, Kp, Vp, tm, fl, flops, peaks, local_rank, sustain_s=3.0):
    """The attention kernel in the two regimes the two measured peaks describe.

    burst: one launch after 0.5 s with the GPU idle (median of 3), against the
    burst peak (a short cuBLAS GEMM run).  sustained: launches back to back for
    about `sustain_s` seconds, the mean over the second half (after the power
    controller has settled at the board's limit), against the sustained peak
    (cuBLAS back to back for seconds), with the clocks of that half.  Qp, Kp, Vp
    already hold the step's permuted temporal heads."""
    def attn():
        bss.sparse_attention_split(Q, K, V, O, Qp, Kp, Vp, None, tm, fl)

    s = torch.cuda.current_stream()
    burst = []
    for _ in range(3):
        torch.cuda.synchronize()
        time.sleep(0.5)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        attn()
        b.record(s)
        torch.cuda.synchronize()
        burst.append(a.elapsed_time(b))
    burst_ms = statistics.median(burst)

    half = max(4, int(sustain_s / 2 / (burst_ms * 1e-3)))
    for _ in range(half):
        attn()
    torch.cuda.synchronize()
    sampler = clock_sampler(torch, local_rank)
    sampler.start()
    time.sleep(0.05)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler.mark_begin()
    a.record(s)
    for _ in range(half):
        attn()
    b.record(s)
    torch.cuda.synchronize()
    sampler.mark_end()
    clocks = sampler.stop()
    sus_ms = a.elapsed_time(b) / half
    status = bss.get_device_status()
    if status != 0:
        raise RuntimeError(f"device status {bss.status_string(status)} in the power-regime runs")
    bt, st = flops / (burst_ms * 1e-3) / 1e12, flops / (sus_ms * 1e-3) / 1e12
    return {"burst": {"ms": burst_ms, "achieved": bt, "peak": peaks["bf16_tflops"], "frac": bt / peaks["bf16_tflops"],
                      "how": "one launch after 0.5 s idle, median of 3; peak: cuBLAS bf16 burst"},
            "sustained": {"ms": sus_ms, "achieved": st, "peak": peaks["bf16_tflops_sustained"],
                          "frac": st / peaks["bf16_tflops_sustained"], "launches": half, "clocks": clocks,
                          "how": f"{2 * half} launches back to back (about {2 * half * sus_ms / 1e3:.1f} s), mean of "
                                 f"the second half; peak: cuBLAS bf16 back to back for seconds"}}


def dense_control(bss, torch, Q, K, V, O, Qp, Kp, Vp, tm, fl, retained, peaks, rounds=7):
    """The library's dense kernel on the step's shape against the step's sparse
    attention launch, timed interleaved (each round times both, in alternating
    order, so clock drift under the power cap falls on both): the speed-up and
    the retained-fraction target 1 / (retained pairs / all pairs)."""
    H, N, d = Q.shape
    Od = torch.empty_like(Q)
    ms = _time_interleaved(torch, {
        "sparse": lambda: bss.sparse_attention_split(Q, K, V, O, Qp, Kp, Vp, None, tm, fl),
        "dense": lambda: bss.dense_attention(Q, K, V, Od)}, rounds=rounds)
    frac = retained / (H * N * N)
    speedup = ms["dense"] / ms["sparse"]
    dense_flops = 4.0 * d * H * N * N
    return {"ms": ms["dense"], "tflops": dense_flops / ms["dense"] / 1e9,
            "frac_of_peak": dense_flops / ms["dense"] / 1e9 / peaks["bf16_tflops"],
            "sparse_attention_ms": ms["sparse"], "speedup": speedup, "retained_fraction": frac,
            "target_speedup": 1.0 / frac, "speedup_over_target": speedup * frac,
            "timing": f"median of {rounds} interleaved rounds, same inputs"}


def variants(bss, torch, W, w, H, Q, K, V, dev, peaks, flags):
    """Attention-kernel timings of the pages' other measurements, same inputs."""
    out = {}
    O = torch.empty_like(Q)
    dense_flops = 4.0 * w.d * H * w.N * w.N
    zeros = torch.zeros(H, dtype=torch.uint8, device=dev)
    # the pages' B0 (dense) -> B1 -> B2 -> B3 progression, timed interleaved
    bvars = (("spatial_naive_B1", 2), ("spatial_exact_B2", 0), ("spatial_tile_aligned_B3", 1))
    maps = {name: bss.build_tile_map(bss.MaskParams(w.F, w.Hs, w.Ws, w.d, w.wf, w.ws, temporal_permuted=1,
                                                    rounding=rnd)) for name, rnd in bvars}
    try:
        fns = {name: (lambda tm=tm: bss.sparse_attention(Q, K, V, O, tm, zeros)) for name, tm in maps.items()}
        fns["dense"] = lambda: bss.dense_attention(Q, K, V, O)
        bms = _time_interleaved(torch, fns)
        dense_ms = bms["dense"]
        out["dense_control"] = {"ms": dense_ms, "tflops": dense_flops / dense_ms / 1e9,
                                "frac_of_peak": dense_flops / dense_ms / 1e9 / peaks["bf16_tflops"]}
        for name, _ in bvars:
            s0 = maps[name].stats(0)
            ms = bms[name]
            fl_ = 4.0 * w.d * H * s0["retained_pairs"]
            frac = s0["retained_pairs"] / w.N ** 2
            out[name] = {"ms": ms, "tflops": fl_ / ms / 1e9, "frac_of_peak": fl_ / ms / 1e9 / peaks["bf16_tflops"],
                         "speedup_vs_dense": dense_ms / ms, "retained_fraction": frac,
                         "speedup_over_target": dense_ms / ms * frac, "tiles": s0}
    finally:
        for tm in maps.values():
            tm.destroy()
    out["tile_shape_sweep"] = tile_shape_sweep(bss, torch, w)
    # latency side of the sweep: the kernel at both query-tile heights it runs
    pe = bss.MaskParams(w.F, w.Hs, w.Ws, w.d, w.wf, w.ws, temporal_permuted=1, rounding=0)
    zeros_ = torch.zeros(H, dtype=torch.uint8, device=dev)
    lat = {}
    qmaps = {(bq, bkv): bss.build_tile_map(pe, BQ=bq, BKV=bkv)
             for bq in bss.ATTN_BQ_SUPPORTED for bkv in bss.ATTN_BKV_SUPPORTED}
    try:
        qms = _time_interleaved(torch, {key: (lambda tmq=tmq: bss.sparse_attention(Q, K, V, O, tmq, zeros_))
                                        for key, tmq in qmaps.items()})
        for (bq, bkv), tmq in qmaps.items():
            st0 = tmq.stats(0)
            ms = qms[(bq, bkv)]
            ex = st0["full"] + st0["boundary"] + st0["pad"] + st0["columns"]
            lat[f"BQ{bq}_BKV{bkv}"] = {"ms": ms, "tflops": 4.0 * w.d * H * st0["retained_pairs"] / ms / 1e9,
                                       "masked_share": (st0["boundary"] + st0["pad"] + st0["columns"]) / ex}
    finally:
        for tmq in qmaps.values():
            tmq.destroy()
    out["tile_shape_latency_spatial"] = lat
    ones = torch.ones(H, dtype=torch.uint8, device=dev)
    Qp, Kp, Vp, Op = (torch.empty_like(Q) for _ in range(4))
    p1 = bss.MaskParams(w.F, w.Hs, w.Ws, w.d, w.wf, w.ws, temporal_permuted=1, rounding=0)
    p0 = bss.MaskParams(w.F, w.Hs, w.Ws, w.d, w.wf, w.ws, temporal_permuted=0, rounding=0)
    with bss.build_tile_map(p1) as tm1, bss.build_tile_map(p0) as tm0:
        tp = tm1.stats(1)["retained_pairs"]
        fl_ = 4.0 * w.d * H * tp

        def with_perm():
            bss.attention_step(Q, K, V, O, tm1, ones, Qp, Kp, Vp)

        tms = _time_interleaved(torch, {
            "perm": with_perm,
            "attn": lambda: bss.sparse_attention(Qp, Kp, Vp, Op, tm1, ones),
            "noperm": lambda: bss.sparse_attention(Q, K, V, O, tm0, ones),
            "fused": lambda: bss.sparse_attention_fused(Q, K, V, O, tm1, ones)}, rounds=5)
        ms_perm, ms_attn, ms_noperm, ms_fused = tms["perm"], tms["attn"], tms["noperm"], tms["fused"]
        out["temporal_heads"] = {
            "with_permutation_ms": ms_perm, "attention_only_ms": ms_attn, "in_kernel_indexing_ms": ms_noperm,
            "fused_permutation_ms": ms_fused,
            "tflops_attention": fl_ / ms_attn / 1e9, "tflops_in_kernel_indexing": fl_ / ms_noperm / 1e9,
            "tflops_fused_permutation": fl_ / ms_fused / 1e9,
            "tiles_permuted": tm1.stats(1), "tiles_in_kernel_indexing": tm0.stats(1)}
        # the mixed-flag step as one launch: permutation fused into the attention kernel
        fl_mixed = torch.tensor(flags, dtype=torch.uint8, device=dev)
        mixed_fl = 4.0 * w.d * sum(tm1.stats(f)["retained_pairs"] for f in flags)

        def explicit_step():
            bss.attention_step(Q, K, V, O, tm1, fl_mixed, Qp, Kp, Vp)

        mms = _time_interleaved(torch, {"explicit": explicit_step,
                                        "fused": lambda: bss.sparse_attention_fused(Q, K, V, O, tm1, fl_mixed)},
                                rounds=5)
        ms_exp, ms_fst = mms["explicit"], mms["fused"]
        out["mixed_step_fused_permutation"] = {
            "explicit_step_ms": ms_exp, "fused_ms": ms_fst, "tflops_fused": mixed_fl / ms_fst / 1e9,
            "speedup": ms_exp / ms_fst,
            "note": "permute the temporal heads' QKV -> attention storing their O rows in (F,H,W) order (4 launches) vs one launch reading (F,H,W) memory"}
        rows = torch.tensor(W.sample_rows(w.N, 64, seed=w.index), dtype=torch.int32, device=dev)
        rflags = torch.empty(H, dtype=torch.uint8, device=dev)
        rerr = torch.empty(H, 2, dtype=torch.float32, device=dev)
        route_ms = _time_batched(torch, lambda: bss.route_heads(Q, K, V, p1, rows, rflags, rerr))
        out["routing"] = {"ms": route_ms, "sampled_rows": int(rows.numel()),
                          "flags": rflags.cpu().tolist(), "note": "dense/spatial/temporal outputs of the sampled rows"}
        perm_ms = _time_batched(torch, lambda: bss.permute(Q, Qp, ones, p1, False))
        nbytes = 2.0 * Q.numel() * 2
        half = torch.tensor([1, 0] * (H // 2) + [1] * (H % 2), dtype=torch.uint8, device=dev)
        nflag = int(half.sum().item())
        half_ms = _time_batched(torch, lambda: bss.permute(Q, Qp, half, p1, False, only_flagged=True))
        hbytes = 2.0 * nflag * w.N * w.d * 2
        # the step's launch: the flagged heads of Q, K and V in one launch
        qkv_ms = _time_batched(torch, lambda: bss.permute_flagged_multi((Q, K, V), (Qp, Kp, Vp), half, p1))
        out["permute"] = {"ms": perm_ms, "gbs": nbytes / perm_ms / 1e6, "frac_of_hbm_peak":
                          nbytes / perm_ms / 1e6 / peaks["hbm_gbs"],
                          "flagged_only_half_heads": {"ms": half_ms, "gbs": hbytes / half_ms / 1e6,
                                                      "frac_of_hbm_peak": hbytes / half_ms / 1e6 / peaks["hbm_gbs"]},
                          "flagged_half_heads_qkv_one_launch": {
                              "ms": qkv_ms, "gbs": 3 * hbytes / qkv_ms / 1e6,
                              "frac_of_hbm_peak": 3 * hbytes / qkv_ms / 1e6 / peaks["hbm_gbs"]},
                          "timing": "20 launches back to back between one pair of CUDA events"}
    out["p1440_step"] = p1440_step(bss, torch, W, dev, peaks)
    return out


def p1440_step(bss, torch, W, dev, peaks):
    """The 1440p-scale workload (21 x 90 x 160 = 302,400 tokens, 10 heads, 5
    spatial + 5 temporal, tile-aligned masks): the same step as the headline
    (temporal heads' permutes + attention) and the dense control at that size."""
    w2 = W.P1440_302K
    Q, K, V = W.qkv_device(w2, dev)
    O = torch.empty_like(Q)
    Qp, Kp, Vp = (torch.empty_like(Q) for _ in range(3))
    flags = w2.head_flags()
    fl = torch.tensor(flags, dtype=torch.uint8, device=dev)
    p = bss.MaskParams(w2.F, w2.Hs, w2.Ws, w2.d, w2.wf, w2.ws, temporal_permuted=1, rounding=1)
    with bss.build_tile_map(p) as tm:
        st = {kind: tm.stats(kind) for kind in (0, 1)}
        pairs = sum(st[f]["retained_pairs"] for f in flags)
        exact = sum(st[f]["exact_retained_pairs"] for f in flags)
        ms = _time(torch, lambda: bss.attention_step(Q, K, V, O, tm, fl, Qp, Kp, Vp))
    dense_ms = _time(torch, lambda: bss.dense_attention(Q, K, V, O), reps=3, warm=2)
    status = bss.get_device_status()
    if status != 0:
        raise RuntimeError(f"device status {bss.status_string(status)} in the 1440p variant")
    flops = 4.0 * w2.d * pairs
    dense_flops = 4.0 * w2.d * w2.H * w2.N * w2.N
    return {"workload": w2.name, "flags_temporal": flags, "step_ms": ms, "tflops": flops / ms / 1e9,
            "frac_of_peak": flops / ms / 1e9 / peaks["bf16_tflops"],
            "dense_ms": dense_ms, "dense_tflops": dense_flops / dense_ms / 1e9, "speedup_vs_dense": dense_ms / ms,
            "retained_fraction": pairs / (w2.H * w2.N * w2.N),
            "exact_retained_fraction": exact / (w2.H * w2.N * w2.N), "tiles": st,
            "flops": "4 d x pairs kept by the tile-aligned masks"}


def tile_shape_sweep(bss, torch, w):
    """Masking work against tile shape (the blog's Figure 7 axis), from the tile
    maps of both mask kinds of this workload's exact masks: the share of executed
    tiles that need an intra-tile mask (boundary + padding), and the executed
    pairs (tiles x tile area) per retained pair.  The attention kernel runs the
    256 x 128 shape; 3328 / 4864 / 1024 x 1536 are the pages' TPU shapes."""
    rows = []
    p = bss.MaskParams(w.F, w.Hs, w.Ws, w.d, w.wf, w.ws, temporal_permuted=1, rounding=0)
    for bq, bkv in ((128, 64), (128, 128), (256, 64), (256, 128), (256, 256), (512, 128), (1024, 1536),
                    (3328, 1536), (4864, 1536)):
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record()
        tm = bss.build_tile_map(p, BQ=bq, BKV=bkv)
        s1.record()
        torch.cuda.synchronize()
        row = {"BQ": bq, "BKV": bkv, "build_ms": s0.elapsed_time(s1)}
        for kind, name in ((0, "spatial"), (1, "temporal")):
            st = tm.stats(kind)
            ex = st["full"] + st["boundary"] + st["pad"] + st["columns"]
            row[name] = {"executed_tiles": ex,
                         "masked_share": (st["boundary"] + st["pad"] + st["columns"]) / max(ex, 1),
                         "executed_pairs_per_retained": ex * bq * bkv / st["retained_pairs"]}
        tm.destroy()
        rows.append(row)
    return rows


def e2e(bss, torch, params, tm, flags, Qd, Kd, Vd, flops, args):
    """The same step through the library's host-buffer call
    (bss_attention_step_host): every step copies its Q, K, V and flags host ->
    device and its O device -> host, pipelined by the library over consecutive
    steps (three workspace sets: the copies of one step overlap the kernels of
    another; heads in groups of two).  K consecutive steps are timed with one
    pair of events on the compute stream: the workspace's copy streams are
    ordered after the first event and the compute stream waits for the last
    step's D2H copy before the second, so every step's copies are inside the
    timed region."""
    H, N, d = Qd.shape
    hq, hk, hv = (torch.empty(H, N, d, dtype=torch.bfloat16, pin_memory=True) for _ in range(3))
    ho = torch.empty(H, N, d, dtype=torch.bfloat16, pin_memory=True)
    for x, src in ((hq, Qd), (hk, Kd), (hv, Vd)):
        x.copy_(src.cpu())
    ws = bss.step_workspace(params, H)
    fl_host = torch.tensor(flags, dtype=torch.uint8).pin_memory()
    main = torch.cuda.current_stream()
    # as many steps as the device timing: the pipeline's fill (the first H2D
    # copy) and drain (the last D2H copy) are spread over the same K steps
    steps = max(3, args.steps)

    def run(n):
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(main)
        ws.wait_stream(main)
        last = None
        for _ in range(n):
            last = bss.attention_step_host(hq, hk, hv, ho, tm, fl_host, ws)
        main.wait_event(last)
        t1.record(main)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / n

    run(3)
    # the copies alone, one step's worth each, on an idle GPU: how much time the
    # pipeline has to hide behind the kernels
    cs = torch.cuda.Stream()
    scratch = [torch.empty_like(Qd) for _ in range(3)]
    c0, c1, c2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    torch.cuda.synchronize()
    with torch.cuda.stream(cs):
        c0.record(cs)
        for src, dst in zip((hq, hk, hv), scratch):
            dst.copy_(src, non_blocking=True)
        c1.record(cs)
        ho.copy_(scratch[0], non_blocking=True)
        c2.record(cs)
    torch.cuda.synchronize()
    h2d_ms, d2h_ms = c0.elapsed_time(c1), c1.elapsed_time(c2)
    del scratch
    sampler = clock_sampler(torch, torch.cuda.current_device())
    sampler.start()
    time.sleep(0.3)
    sampler.mark_begin()
    ms = run(steps)
    sampler.mark_end()
    clocks = sampler.stop()
    ws.destroy()
    return {"value": flops / (ms * 1e-3) / 1e12, "unit": UNIT, "ms_per_step": ms, "steps": steps, "clocks": clocks,
            "copies_alone_ms": {"h2d_qkv": h2d_ms, "d2h_o": d2h_ms},
            "h2d_bytes_per_step": 3 * H * N * d * 2 + H, "d2h_bytes_per_step": H * N * d * 2,
            "api": "bss_attention_step_host (C ABI) from pinned host buffers",
            "pipelining": "three workspace sets: the H2D copy of step i+1 and the D2H copy of step i-1 "
                          "overlap the kernels of step i; heads copied in and computed in groups of two"}


def cpu_baseline(w, Q, K, V, flags, args, flops):
    import oracle
    H = Q.shape[0]
    q, k, v = (x.cpu() for x in (Q, K, V))
    cores = oracle.num_threads()
    dt, nrows = oracle_sample(w, q, k, v, flags, args.cpu_rows_per_head, seed=2000)
    rows_total = H * w.N
    full_s = dt * rows_total / nrows
    # the same oracle on one core, a smaller sample
    oracle.set_num_threads(1)
    try:
        dt1, nrows1 = oracle_sample(w, q, k, v, flags, args.cpu_rows_per_head_1core, seed=3000)
    finally:
        oracle.set_num_threads(cores)
    full_s1 = dt1 * rows_total / nrows1
    return {"value": flops / full_s / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{args.cpu_rows_per_head} seeded query rows per head x {H} heads "
                      f"({100.0 * nrows / rows_total:.2f}% of rows, {dt:.1f} s), time scaled to all rows",
            "seconds_full_workload_extrapolated": full_s,
            "single_core": {"value": flops / full_s1 / 1e12, "unit": UNIT, "cores": 1,
                            "sample": f"{args.cpu_rows_per_head_1core} seeded query rows per head x {H} heads "
                                      f"({dt1:.1f} s), time scaled to all rows",
                            "seconds_full_workload_extrapolated": full_s1}}


if __name__ == "__main__":
    main()
