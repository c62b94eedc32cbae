#!/usr/bin/env python
"""Throughput of the FP4 (E2M1) block-scaled decode path on one GB300 per rank.

One step = one pass of the whole path over one batch of synthetic input:
MXFP4 unpack of an MoE expert stack (gate+up [32, 5760, 2880] and down
[32, 2880, 2880] codes; two fp4_mx_unpack launches) plus an NVFP4 embedding
gather-dequant (vocab 200,000 x hidden 8,192, 16,384 Zipf(1.1) ids as [64, 256];
one fp4_nv_embedding_gather launch). ``--workload`` picks one of the other named
workloads instead (one entry point per step).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0). ``value`` is decoded elements per second over all
ranks with inputs resident in HBM; ``e2e`` is the same metric through the public
API with pinned host buffers, the host->device copies of each step's inputs and
the device->host copies of its outputs inside the timed region; ``roofline`` is
the dominant kernel (the MXFP4 unpack) against the measured HBM copy bandwidth;
``cpu_baseline`` is the CPU oracle on a bounded sample of the same workload.
With ``--impl reference`` the CPU oracle itself is timed on the same workload
(a bounded sample per step) and reported as the reference arm.

Under torchrun each rank runs the full workload on its own GPU (replicas: the
decode has no exchange step), timing is bracketed by barriers and the maximum
over ranks is reported.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decoded FP4 elements/sec and achieved HBM GB/s (% of GB300 peak), 1 GPU"
UNIT = "elements/s"
FALLBACK_HBM_GBS = 6800.0
WORKLOADS = ("step", "mx_moe", "mx_stress", "mx_exhaustive", "nv_embedding_200k",
             "nv_embedding_32k")
DOMINANT = "mx_unpack"  # kernel the roofline object describes


# ---------------------------------------------------------------------------
# distributed plumbing (replicas)
# ---------------------------------------------------------------------------

class Dist:
    def __init__(self):
        self.rank = int(os.environ.get("RANK", "0"))
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, backend: str):
        if self.world > 1:
            import torch.distributed as dist
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group(backend=backend, rank=self.rank, world_size=self.world)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, value: float, device=None) -> float:
        return reduce_max(self.pg, value, device)

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


def reduce_max(pg, value: float, device=None) -> float:
    """Maximum of a float over all ranks (identity without a process group)."""
    if pg is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region (read-only NVML queries; nvidia-smi fallback)
# ---------------------------------------------------------------------------

_REASONS = [(0x1, "gpu_idle"), (0x2, "applications_clocks_setting"), (0x4, "sw_power_cap"),
            (0x8, "hw_slowdown"), (0x10, "sync_boost"), (0x20, "sw_thermal_slowdown"),
            (0x40, "hw_thermal_slowdown"), (0x80, "hw_power_brake_slowdown"),
            (0x100, "display_clock_setting")]


class ClockSampler:
    """Polls SM clock, power and clock-event reasons every few ms in a thread."""

    def __init__(self, device_index: int, period_s: float = 0.002):
        self.period = period_s
        self.samples = []  # (t, sm_mhz, reasons_mask, power_w)
        self.max_mhz = None
        self.source = None
        self._stop = threading.Event()
        self._thread = None
        self._nvml = None
        self._handle = None
        try:
            self._open_nvml(device_index)
            self.source = "nvml"
        except Exception:  # noqa: BLE001 -- sampling is best effort
            self._nvml = None
            self.source = "nvidia-smi" if _which("nvidia-smi") else None

    def _open_nvml(self, device_index: int):
        import torch
        nvml = ctypes.CDLL("libnvidia-ml.so.1")
        if nvml.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        handle = ctypes.c_void_p()
        props = torch.cuda.get_device_properties(device_index)
        bus = None
        if hasattr(props, "pci_bus_id"):
            bus = "%08X:%02X:%02X.0" % (getattr(props, "pci_domain_id", 0), props.pci_bus_id,
                                        getattr(props, "pci_device_id", 0))
        ok = bus is not None and nvml.nvmlDeviceGetHandleByPciBusId_v2(
            bus.encode(), ctypes.byref(handle)) == 0
        if not ok and nvml.nvmlDeviceGetHandleByIndex_v2(device_index, ctypes.byref(handle)) != 0:
            raise RuntimeError("no NVML handle")
        self._nvml, self._handle = nvml, handle
        mhz = ctypes.c_uint()
        if nvml.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mhz)) == 0:
            self.max_mhz = int(mhz.value)
        self._reasons_fn = getattr(nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(nvml, "nvmlDeviceGetCurrentClocksThrottleReasons")

    def _sample_nvml(self):
        mhz, reasons, mw = ctypes.c_uint(), ctypes.c_ulonglong(), ctypes.c_uint()
        self._nvml.nvmlDeviceGetClockInfo(self._handle, 1, ctypes.byref(mhz))
        self._reasons_fn(self._handle, ctypes.byref(reasons))
        self._nvml.nvmlDeviceGetPowerUsage(self._handle, ctypes.byref(mw))
        return int(mhz.value), int(reasons.value), mw.value / 1000.0

    def _run(self):
        while not self._stop.is_set():
            try:
                self.samples.append((time.perf_counter(), *self._sample_nvml()))
            except Exception:  # noqa: BLE001
                return
            time.sleep(self.period)

    def start(self):
        if self._nvml is not None:
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()

    def stop(self):
        self._stop.set()
        if self._thread is not None:
            self._thread.join()

    def summary(self, t0: float, t1: float) -> dict:
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        if not inside and self.samples:
            # the region was shorter than one period: use the sample nearest its end
            inside = [min(self.samples, key=lambda s: abs(s[0] - t1))]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [],
                    "samples": 0, "source": self.source}
        mask = 0
        for s in inside:
            mask |= s[2]
        return {"sm_mhz": statistics.median(s[1] for s in inside), "sm_max_mhz": self.max_mhz,
                "reasons": [n for b, n in _REASONS if mask & b],
                "power_w_max": max(s[3] for s in inside), "samples": len(inside),
                "source": self.source}


def _which(name):
    for d in os.environ.get("PATH", "").split(os.pathsep):
        if os.path.exists(os.path.join(d, name)):
            return os.path.join(d, name)
    return None


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

def load_workload(name: str):
    from block_scaled_fp4_mx_gb300 import inputs
    mx, nv = [], []
    if name in ("step", "mx_moe"):
        mx = inputs.mx_moe()
    if name in ("step", "nv_embedding_200k"):
        nv = [inputs.nv_embedding_200k()]
    if name == "mx_stress":
        mx = [inputs.mx_stress()]
    if name == "mx_exhaustive":
        mx = [inputs.mx_exhaustive()]
    if name == "nv_embedding_32k":
        nv = [inputs.nv_embedding_32k()]
    return mx, nv


def workload_label(name: str, mx, nv) -> str:
    if name == "step":
        return ("mx_moe_unpack_32x(5760+2880)x2880 + "
                "nv_embedding_gather_200000x8192_zipf1.1_ids64x256")
    return name


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            peaks = json.load(fh)
        return float(peaks["hbm_gbs"]), "measured"
    except Exception:  # noqa: BLE001
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in ("block_scaled_fp4_mx_gb300/csrc/mx_unpack.cu",
                "block_scaled_fp4_mx_gb300/csrc/fp4_decode.cuh"):
        with open(os.path.join(ROOT, rel), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(elements_per_launch: float):
    """DRAM bytes per launch of the dominant kernel from the committed ncu capture,
    scaled to this launch size; None when the kernel source changed since."""
    path = os.path.join(ROOT, "profiles", "mx_unpack_dram_traffic.json")
    try:
        with open(path) as fh:
            rec = json.load(fh)
    except Exception:  # noqa: BLE001
        return None, None
    if rec.get("kernel_source_sha256_16") != kernel_source_hash():
        return None, "stale"
    return rec["dram_bytes_per_element"] * elements_per_launch, rec.get("capture")


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_ours(args, d: Dist):
    import torch

    import block_scaled_fp4_mx_gb300 as fp4

    dev = torch.device("cuda", d.local_rank)
    torch.cuda.set_device(dev)
    d.init("nccl")
    fp4.load()
    mx_in, nv_in = load_workload(args.workload)

    stream = torch.cuda.current_stream(dev)
    mx_dev = [(torch.from_numpy(x.packed).to(dev), torch.from_numpy(x.scales).to(dev),
               torch.empty(x.rows, x.k, dtype=torch.bfloat16, device=dev)) for x in mx_in]
    nv_dev = [(torch.from_numpy(x.ids).to(dev), torch.from_numpy(x.weight).to(dev),
               torch.from_numpy(x.scales).to(dev),
               torch.tensor([x.global_scale], dtype=torch.float32, device=dev),
               torch.empty(*x.ids.shape, x.hidden, dtype=torch.bfloat16, device=dev))
              for x in nv_in]
    torch.cuda.synchronize()

    mx_elems = sum(x.n_elems for x in mx_in)
    nv_elems = sum(x.n_elems for x in nv_in)
    step_elems = mx_elems + nv_elems
    mx_bytes = sum(x.algorithmic_bytes() for x in mx_in)
    nv_bytes = sum(x.algorithmic_bytes() for x in nv_in)
    nv_min_bytes = sum(x.distinct_row_bytes() for x in nv_in)
    launches_per_step = len(mx_in) + len(nv_in)

    def step(ev=None):
        for i, (p, s, o) in enumerate(mx_dev):
            if ev is not None:
                ev["mx"][i][0].record(stream)
            fp4.fp4_mx_unpack(p, s, out=o, stream=stream)
            if ev is not None:
                ev["mx"][i][1].record(stream)
        for i, (ids, w, sc, gs, o) in enumerate(nv_dev):
            if ev is not None:
                ev["nv"][i][0].record(stream)
            fp4.fp4_nv_embedding_gather(ids, w, sc, gs, out=o, stream=stream)
            if ev is not None:
                ev["nv"][i][1].record(stream)

    def new_events():
        mk = lambda: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        return {"mx": [mk() for _ in mx_dev], "nv": [mk() for _ in nv_dev]}

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    sampler = ClockSampler(dev.index)
    sampler.start()
    per_step_events = [new_events() for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    d.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    start.record(stream)
    for k in range(args.steps):
        step(per_step_events[k])
    end.record(stream)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    d.barrier()
    sampler.stop()
    elapsed_ms = start.elapsed_time(end)
    elapsed_ms = d.max(elapsed_ms, dev)

    mx_ms = sum(e[0].elapsed_time(e[1]) for ev in per_step_events for e in ev["mx"])
    nv_ms = sum(e[0].elapsed_time(e[1]) for ev in per_step_events for e in ev["nv"])
    k = args.steps
    value = step_elems * k * d.world / (elapsed_ms / 1e3)
    alg_gbs = (mx_bytes + nv_bytes) * k / (elapsed_ms / 1e3) / 1e9
    peak, peak_kind = measured_peak()
    clocks = sampler.summary(t0, t1)

    kernels = {}
    roofline = None
    if mx_in:
        mx_launch_s = mx_ms / 1e3 / (k * len(mx_in))
        bytes_per_launch = mx_bytes / len(mx_in)
        achieved = bytes_per_launch / mx_launch_s / 1e9
        traffic, capture = ncu_traffic(mx_elems / len(mx_in))
        kernels["mx_unpack"] = {"launches_per_step": len(mx_in), "avg_launch_us": mx_launch_s * 1e6,
                                "elements_per_launch": mx_elems / len(mx_in),
                                "algorithmic_bytes_per_launch": bytes_per_launch,
                                "gbs": achieved, "frac_of_peak": achieved / peak}
        roofline = {"kernel": "mx_unpack_words_kernel", "bound": "hbm", "achieved": achieved,
                    "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                    "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if
                    peak_kind == "measured" else "fallback 6.8 TB/s",
                    "traffic": traffic,
                    "traffic_source": capture}
    if nv_in:
        nv_launch_s = nv_ms / 1e3 / (k * len(nv_in))
        kernels["nv_embedding_gather"] = {
            "launches_per_step": len(nv_in), "avg_launch_us": nv_launch_s * 1e6,
            "elements_per_launch": nv_elems / len(nv_in),
            "logical_bytes_per_launch": nv_bytes / len(nv_in),
            "distinct_row_bytes_per_launch": nv_min_bytes / len(nv_in),
            "gbs_logical": nv_bytes / len(nv_in) / nv_launch_s / 1e9,
            "gbs_distinct_rows": nv_min_bytes / len(nv_in) / nv_launch_s / 1e9,
            "frac_of_peak_logical": nv_bytes / len(nv_in) / nv_launch_s / 1e9 / peak}
        if roofline is None:
            achieved = nv_bytes / len(nv_in) / nv_launch_s / 1e9
            roofline = {"kernel": "nv_gather_rows_kernel", "bound": "hbm", "achieved": achieved,
                        "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                        "peak_source": peak_kind, "traffic": None,
                        "traffic_source": None}

    e2e = None if args.no_e2e else run_e2e(args, d, dev, mx_in, nv_in, mx_dev, nv_dev, step_elems)
    cpu = None
    if d.rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(mx_in, nv_in, budget_s=args.cpu_budget)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": d.world, "steps": k,
        "warmup": args.warmup, "ms_per_step": elapsed_ms / k, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int16+fp32", "data": "synthetic",
        "config": {"workload": workload_label(args.workload, mx_in, nv_in),
                   "mx_elements_per_step": mx_elems, "nv_elements_per_step": nv_elems,
                   "algorithmic_bytes_per_step": mx_bytes + nv_bytes,
                   "l2": "inputs (398 MB packed MoE codes, 922 MB packed table) and outputs "
                         "(1.86 GB) larger than the 129 MB L2; no flush",
                   "parallelism": f"replicas x{d.world}"},
        "hbm_gbs_algorithmic": alg_gbs, "pct_of_peak_hbm": 100.0 * alg_gbs / peak,
        "roofline": roofline, "kernels": kernels, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": launches_per_step * k, "clocks": clocks,
        "device": torch.cuda.get_device_name(dev),
    }
    if d.rank == 0:
        emit(line, args)
    d.close()


def _row_chunks(n: int, chunks: int):
    step = max(1, -(-n // max(1, chunks)))
    return [(r, min(n, r + step)) for r in range(0, n, step)]


def run_e2e(args, d, dev, mx_in, nv_in, mx_dev, nv_dev, step_elems):
    """Same steps through the public API with pinned host buffers: every step
    copies its inputs host->device, decodes, and copies its outputs back. Each
    tensor is cut into row chunks issued round-robin on a few streams, so the
    host->device copies, the kernels and the device->host copies of different
    chunks overlap (the copy engines of both directions run at once)."""
    import torch

    import block_scaled_fp4_mx_gb300 as fp4

    main = torch.cuda.current_stream(dev)
    streams = [torch.cuda.Stream(dev) for _ in range(max(1, args.e2e_streams))]
    pin = lambda a: torch.from_numpy(a).pin_memory()
    mx_host = [(pin(x.packed), pin(x.scales),
                torch.empty(x.rows, x.k, dtype=torch.bfloat16).pin_memory()) for x in mx_in]
    nv_host = [(pin(x.ids.reshape(-1)),
                torch.empty(x.ids.size, x.hidden, dtype=torch.bfloat16).pin_memory())
               for x in nv_in]
    nv_flat = [(ids.view(-1), w, sc, gs, o.view(-1, o.shape[-1])) for ids, w, sc, gs, o in nv_dev]
    h2d = sum(p.numel() + s.numel() for p, s, _ in mx_host) + sum(i.numel() * 8 for i, _ in nv_host)
    d2h = sum(o.numel() * 2 for *_, o in mx_host) + sum(o.numel() * 2 for _, o in nv_host)
    jobs = []
    for (hp, hs, ho), (p, s, o) in zip(mx_host, mx_dev):
        for r0, r1 in _row_chunks(p.shape[0], args.e2e_chunks):
            jobs.append(("mx", (hp[r0:r1], hs[r0:r1], ho[r0:r1]), (p[r0:r1], s[r0:r1], o[r0:r1])))
    for (hi, ho), (ids, w, sc, gs, o) in zip(nv_host, nv_flat):
        for r0, r1 in _row_chunks(ids.shape[0], max(1, args.e2e_chunks // 2)):
            jobs.append(("nv", (hi[r0:r1], ho[r0:r1]), (ids[r0:r1], w, sc, gs, o[r0:r1])))

    def step():
        start = torch.cuda.Event()
        start.record(main)
        for st in streams:
            st.wait_event(start)
        for j, (kind, host, devb) in enumerate(jobs):
            st = streams[j % len(streams)]
            with torch.cuda.stream(st):
                if kind == "mx":
                    (hp, hs, ho), (p, s, o) = host, devb
                    p.copy_(hp, non_blocking=True)
                    s.copy_(hs, non_blocking=True)
                    fp4.fp4_mx_unpack(p, s, out=o, stream=st)
                    ho.copy_(o, non_blocking=True)
                else:
                    (hi, ho), (ids, w, sc, gs, o) = host, devb
                    ids.copy_(hi, non_blocking=True)
                    fp4.fp4_nv_embedding_gather(ids, w, sc, gs, out=o, stream=st)
                    ho.copy_(o, non_blocking=True)
        for st in streams:
            done = torch.cuda.Event()
            done.record(st)
            main.wait_event(done)

    steps = max(1, min(args.steps, args.e2e_steps))
    for _ in range(max(3, min(args.warmup, 5))):
        step()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    d.barrier()
    torch.cuda.synchronize()
    start.record(main)
    for _ in range(steps):
        step()
    end.record(main)
    torch.cuda.synchronize()
    d.barrier()
    ms = d.max(start.elapsed_time(end), dev)
    return {"value": step_elems * steps * d.world / (ms / 1e3), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": ms / steps, "gpu_launches_per_step": len(jobs),
            "host_link_gbs": (h2d + d2h) / (ms / steps / 1e3) / 1e9,
            "note": f"MXFP4 codes+scales and token ids copied in, all bf16 outputs copied out, "
                    f"{len(jobs)} row chunks on {len(streams)} streams; the NVFP4 table stays "
                    f"resident (model weights)"}


# ---------------------------------------------------------------------------
# CPU oracle timings
# ---------------------------------------------------------------------------

def _mx_sample(x, rows):
    return x.packed[:rows], x.scales[:rows]


def cpu_rates(mx_in, nv_in, seconds: float):
    """Oracle throughput (elements/s) on leading slices of the workload, sized to
    take about ``seconds`` each; returns (mx_rate, nv_rate, description, threads)."""
    import numpy as np

    import oracle

    o = oracle.get()
    threads = o.max_threads()
    desc = []
    mx_rate = nv_rate = None
    if mx_in:
        x = mx_in[0]
        rows = max(1, min(x.rows, 64))
        while True:
            p, s = _mx_sample(x, rows)
            t = time.perf_counter()
            o.mx_unpack(p, s, threads)
            dt = time.perf_counter() - t
            if dt >= seconds / 4 or rows == x.rows:
                break
            rows = min(x.rows, int(rows * max(2.0, seconds / 2 / max(dt, 1e-4))))
        reps, total = 0, 0.0
        while total < seconds and reps < 50:
            t = time.perf_counter()
            o.mx_unpack(p, s, threads)
            total += time.perf_counter() - t
            reps += 1
        mx_rate = rows * x.k * reps / total
        desc.append(f"MXFP4: first {rows} rows of {x.name} ({rows * x.k} codes) x{reps}")
    if nv_in:
        x = nv_in[0]
        flat = x.ids.reshape(-1)
        n = max(1, min(flat.size, 16))
        while True:
            t = time.perf_counter()
            o.nv_embedding_gather(flat[:n], x.weight, x.scales, x.global_scale, threads=threads)
            dt = time.perf_counter() - t
            if dt >= seconds / 4 or n == flat.size:
                break
            n = min(flat.size, int(n * max(2.0, seconds / 2 / max(dt, 1e-4))))
        reps, total = 0, 0.0
        while total < seconds and reps < 50:
            t = time.perf_counter()
            o.nv_embedding_gather(flat[:n], x.weight, x.scales, x.global_scale, threads=threads)
            total += time.perf_counter() - t
            reps += 1
        nv_rate = n * x.hidden * reps / total
        desc.append(f"NVFP4: first {n} ids of {x.name} ({n * x.hidden} codes) x{reps}")
    return mx_rate, nv_rate, "; ".join(desc), threads


def cpu_baseline(mx_in, nv_in, budget_s: float = 10.0) -> dict:
    parts = (1 if mx_in else 0) + (1 if nv_in else 0)
    mx_rate, nv_rate, desc, threads = cpu_rates(mx_in, nv_in, budget_s / max(1, parts))
    t_step = 0.0
    if mx_in:
        t_step += sum(x.n_elems for x in mx_in) / mx_rate
    if nv_in:
        t_step += sum(x.n_elems for x in nv_in) / nv_rate
    total = sum(x.n_elems for x in mx_in) + sum(x.n_elems for x in nv_in)
    return {"value": total / t_step, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": desc + "; rates combined in the step's element mix",
            "mx_elements_per_s": mx_rate, "nv_elements_per_s": nv_rate,
            "cpu": _cpu_model()}


def _cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True).stdout
        for line in out.splitlines():
            if line.startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except Exception:  # noqa: BLE001
        pass
    return os.uname().machine


def run_reference(args, d: Dist):
    """The CPU oracle as the reference arm: rank 0 only, a bounded sample per step."""
    if d.rank != 0:
        return
    import oracle

    oracle.build()
    mx_in, nv_in = load_workload(args.workload)
    per_step = max(0.5, min(20.0, args.reference_budget / max(1, args.steps + args.warmup)))
    mx_rate, nv_rate, desc, threads = cpu_rates(mx_in, nv_in, per_step / 2)
    # each step: the sampled slices once, timed
    o = oracle.get()
    times = []
    sample_elems = 0
    for i in range(args.warmup + args.steps):
        t = time.perf_counter()
        elems = 0
        if mx_in:
            x = mx_in[0]
            rows = max(1, min(x.rows, int(mx_rate * per_step / 2 / x.k)))
            o.mx_unpack(x.packed[:rows], x.scales[:rows], threads)
            elems += rows * x.k
        if nv_in:
            x = nv_in[0]
            n = max(1, min(x.ids.size, int(nv_rate * per_step / 2 / x.hidden)))
            o.nv_embedding_gather(x.ids.reshape(-1)[:n], x.weight, x.scales, x.global_scale,
                                  threads=threads)
            elems += n * x.hidden
        dt = time.perf_counter() - t
        if i >= args.warmup:
            times.append(dt)
            sample_elems = elems
    sec = sum(times)
    value = sample_elems * len(times) / sec
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": d.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sec / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int16+fp32",
        "data": "synthetic",
        "config": {"workload": workload_label(args.workload, mx_in, nv_in),
                   "parallelism": "rank 0 only (CPU)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"per step {sample_elems} codes: {desc}", "cpu": _cpu_model()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    emit(line, args)


def emit(line: dict, args):
    text = json.dumps(line)
    print(text, flush=True)
    if args.json_out:
        with open(args.json_out, "a") as fh:
            fh.write(text + "\n")


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=WORKLOADS, default="step")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--e2e-chunks", type=int, default=8,
                    help="row chunks per MXFP4 tensor in the e2e leg (half as many for NVFP4)")
    ap.add_argument("--e2e-streams", type=int, default=3)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle time for the cpu_baseline estimate")
    ap.add_argument("--reference-budget", type=float, default=120.0,
                    help="seconds of oracle time for the whole --impl reference run")
    ap.add_argument("--json-out", default=None)
    args = ap.parse_args(argv)
    if args.warmup < 0 or args.steps < 1:
        ap.error("need --steps >= 1 and --warmup >= 0")
    d = Dist()
    if args.impl == "reference":
        run_reference(args, d)
    else:
        run_ours(args, d)


if __name__ == "__main__":
    main()
