#!/usr/bin/env python
"""Throughput of the FP4 (E2M1) block-scaled decode path on one GB300 per rank.

One step = one pass of the whole path over the three large workloads: MXFP4
unpack of an MoE expert stack (gate+up [32, 5760, 2880] and down [32, 2880, 2880]
codes; two fp4_mx_unpack launches), an NVFP4 embedding gather-dequant (vocab
200,000 x hidden 8,192, 16,384 Zipf(1.1) ids as [64, 256]; one
fp4_nv_embedding_gather launch) and the MXFP4 stress stream (2^30 packed bytes,
30% zero codes, exponents from {0, 107, 127, 137, 255}; one fp4_mx_unpack
launch). The two small parity workloads (the exhaustive 256 x 256 unpack and the
32k-vocabulary gather) are launch-bound; they are timed in the same run outside
the step, and every workload is also timed alone (its launches back to back).
``--workload`` picks one of the other named workloads instead (one entry point
per step, e.g. ``nv_dequant_200k``: fp4_nv_dequant of the whole 200k x 8,192
table).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0). ``value`` is decoded elements per second over all
ranks with inputs resident in HBM; ``e2e`` is the same metric through the public
API with pinned host buffers, the host->device copies of each step's inputs and
the device->host copies of its outputs inside the timed region; ``roofline`` is
the dominant kernel (most device time per step; the MXFP4 unpack by default)
against the measured HBM copy bandwidth;
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decoded FP4 elements/sec and achieved HBM GB/s (% of GB300 peak), 1 GPU"
UNIT = "elements/s"
FALLBACK_HBM_GBS = 6800.0
WORKLOADS = ("step", "mx_moe", "mx_stress", "mx_exhaustive", "nv_embedding_200k",
             "nv_embedding_32k", "nv_dequant_200k", "nv_dequant_32k", "mx_quantize_moe",
             "mx_moe_gemm_8", "mx_moe_gemm_32", "mx_moe_gemm_128", "mx_moe_gemm_512",
             "mx_moe_forward", "mx_moe_forward_decode", "kv_pages")


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
# workloads: each op kind knows its launch, its bytes, its e2e chunks and its
# oracle sample
# ---------------------------------------------------------------------------

class MxOp:
    """fp4_mx_unpack of one [rows, k] tensor."""
    kind, kernel = "mx_unpack", "mx_unpack_words_kernel"

    def __init__(self, x):
        self.x = x
        self.elems = x.n_elems
        self.bytes = x.algorithmic_bytes()
        self.min_bytes = self.bytes
        self.units, self.elems_per_unit = x.rows, x.k

    def to_device(self, torch, dev):
        x = self.x
        self.p = torch.from_numpy(x.packed).to(dev)
        self.s = torch.from_numpy(x.scales).to(dev)
        self.o = torch.empty(x.rows, x.k, dtype=torch.bfloat16, device=dev)

    def launch(self, fp4, stream):
        fp4.fp4_mx_unpack(self.p, self.s, out=self.o, stream=stream)

    def e2e_jobs(self, torch, fp4, chunks):
        """[(h2d bytes, d2h bytes, fn(stream))] for row chunks, host buffers pinned."""
        hp, hs = torch.from_numpy(self.x.packed).pin_memory(), torch.from_numpy(self.x.scales).pin_memory()
        ho = torch.empty(self.o.shape, dtype=torch.bfloat16).pin_memory()
        jobs = []
        for r0, r1 in _row_chunks(self.x.rows, chunks):
            def fn(st, r0=r0, r1=r1):
                self.p[r0:r1].copy_(hp[r0:r1], non_blocking=True)
                self.s[r0:r1].copy_(hs[r0:r1], non_blocking=True)
                fp4.fp4_mx_unpack(self.p[r0:r1], self.s[r0:r1], out=self.o[r0:r1], stream=st)
                ho[r0:r1].copy_(self.o[r0:r1], non_blocking=True)
            jobs.append((hp[r0:r1].numel() + hs[r0:r1].numel(), ho[r0:r1].numel() * 2, fn))
        return jobs

    def oracle_units(self, o, n, threads):
        o.mx_unpack(self.x.packed[:n], self.x.scales[:n], threads)

    def sample_name(self):
        return f"rows of {self.x.name}"


class NvGatherOp:
    """fp4_nv_embedding_gather of a batch of ids."""
    kind, kernel = "nv_embedding_gather", "nv_gather_rows_kernel<true>"

    def __init__(self, x):
        self.x = x
        self.elems = x.n_elems
        self.bytes = x.algorithmic_bytes()
        self.min_bytes = x.distinct_row_bytes()
        self.units, self.elems_per_unit = x.ids.size, x.hidden

    def to_device(self, torch, dev):
        x = self.x
        self.ids = torch.from_numpy(x.ids).to(dev)
        self.w = torch.from_numpy(x.weight).to(dev)
        self.sc = torch.from_numpy(x.scales).to(dev)
        self.gs = torch.tensor([x.global_scale], dtype=torch.float32, device=dev)
        self.o = torch.empty(*x.ids.shape, x.hidden, dtype=torch.bfloat16, device=dev)

    def launch(self, fp4, stream):
        fp4.fp4_nv_embedding_gather(self.ids, self.w, self.sc, self.gs, out=self.o, stream=stream)

    def e2e_jobs(self, torch, fp4, chunks):
        hi = torch.from_numpy(self.x.ids.reshape(-1)).pin_memory()
        ids, o = self.ids.view(-1), self.o.view(-1, self.x.hidden)
        ho = torch.empty(o.shape, dtype=torch.bfloat16).pin_memory()
        jobs = []
        for r0, r1 in _row_chunks(ids.shape[0], max(1, chunks // 2)):
            def fn(st, r0=r0, r1=r1):
                ids[r0:r1].copy_(hi[r0:r1], non_blocking=True)
                fp4.fp4_nv_embedding_gather(ids[r0:r1], self.w, self.sc, self.gs, out=o[r0:r1],
                                            stream=st)
                ho[r0:r1].copy_(o[r0:r1], non_blocking=True)
            jobs.append(((r1 - r0) * 8, ho[r0:r1].numel() * 2, fn))
        return jobs

    def oracle_units(self, o, n, threads):
        x = self.x
        o.nv_embedding_gather(x.ids.reshape(-1)[:n], x.weight, x.scales, x.global_scale,
                              threads=threads)

    def sample_name(self):
        return f"ids of {self.x.name}"


class NvDenseOp:
    """fp4_nv_dequant of a whole table."""
    kind, kernel = "nv_dequant", "nv_gather_rows_kernel<false>"

    def __init__(self, x):
        self.x = x
        self.elems = x.vocab * x.hidden
        self.bytes = x.vocab * (x.hidden // 2 + x.hidden // x.group_size + 2 * x.hidden)
        self.min_bytes = self.bytes
        self.units, self.elems_per_unit = x.vocab, x.hidden

    def to_device(self, torch, dev):
        x = self.x
        self.w = torch.from_numpy(x.weight).to(dev)
        self.sc = torch.from_numpy(x.scales).to(dev)
        self.gs = torch.tensor([x.global_scale], dtype=torch.float32, device=dev)
        self.o = torch.empty(x.vocab, x.hidden, dtype=torch.bfloat16, device=dev)

    def launch(self, fp4, stream):
        fp4.fp4_nv_dequant(self.w, self.sc, self.gs, out=self.o, stream=stream)

    def e2e_jobs(self, torch, fp4, chunks):
        hw, hs = torch.from_numpy(self.x.weight).pin_memory(), torch.from_numpy(self.x.scales).pin_memory()
        ho = torch.empty(self.o.shape, dtype=torch.bfloat16).pin_memory()
        jobs = []
        for r0, r1 in _row_chunks(self.x.vocab, chunks):
            def fn(st, r0=r0, r1=r1):
                self.w[r0:r1].copy_(hw[r0:r1], non_blocking=True)
                self.sc[r0:r1].copy_(hs[r0:r1], non_blocking=True)
                fp4.fp4_nv_dequant(self.w[r0:r1], self.sc[r0:r1], self.gs, out=self.o[r0:r1],
                                   stream=st)
                ho[r0:r1].copy_(self.o[r0:r1], non_blocking=True)
            jobs.append((hw[r0:r1].numel() + hs[r0:r1].numel(), ho[r0:r1].numel() * 2, fn))
        return jobs

    def oracle_units(self, o, n, threads):
        x = self.x
        o.nv_dequant(x.weight[:n], x.scales[:n], x.global_scale, threads=threads)

    def sample_name(self):
        return f"rows of the {self.x.name} table"


class MxPagesOp:
    """fp4_mx_unpack_pages of a page table against an MXFP4 KV pool."""
    kind, kernel = "mx_unpack_pages", "mx_pages_rows_kernel"

    def __init__(self, kv):
        self.kv = kv
        self.elems = kv.n_elems
        self.bytes = kv.algorithmic_bytes()
        self.min_bytes = self.bytes
        self.units, self.elems_per_unit = kv.page_ids.size, kv.page_elems

    def to_device(self, torch, dev):
        self.ids = torch.from_numpy(self.kv.page_ids).to(dev)
        self.p = torch.from_numpy(self.kv.pool.packed).to(dev)
        self.s = torch.from_numpy(self.kv.pool.scales).to(dev)
        self.o = torch.empty(*self.kv.page_ids.shape, self.kv.page_elems, dtype=torch.bfloat16,
                             device=dev)

    def launch(self, fp4, stream):
        fp4.fp4_mx_unpack_pages(self.ids, self.p, self.s, out=self.o, stream=stream)

    def e2e_jobs(self, torch, fp4, chunks):
        hi = torch.from_numpy(self.kv.page_ids.reshape(-1)).pin_memory()
        ids, o = self.ids.view(-1), self.o.view(-1, self.kv.page_elems)
        ho = torch.empty(o.shape, dtype=torch.bfloat16).pin_memory()
        jobs = []
        for r0, r1 in _row_chunks(ids.shape[0], max(1, chunks // 2)):
            def fn(st, r0=r0, r1=r1):
                ids[r0:r1].copy_(hi[r0:r1], non_blocking=True)
                fp4.fp4_mx_unpack_pages(ids[r0:r1], self.p, self.s, out=o[r0:r1], stream=st)
                ho[r0:r1].copy_(o[r0:r1], non_blocking=True)
            jobs.append(((r1 - r0) * 8, ho[r0:r1].numel() * 2, fn))
        return jobs

    def oracle_units(self, o, n, threads):
        o.mx_unpack_pages(self.kv.page_ids.reshape(-1)[:n], self.kv.pool.packed,
                          self.kv.pool.scales, threads)

    def sample_name(self):
        return "pages of the KV page table"


class MxQuantOp:
    """fp4_mx_quantize of one bf16 [rows, k] tensor."""
    kind, kernel = "mx_quantize", "mx_quantize_words_kernel"

    def __init__(self, w):
        self.w = w
        self.elems = w.n_elems
        self.bytes = w.algorithmic_bytes()
        self.min_bytes = self.bytes
        self.out_bytes = self.elems // 2 + self.elems // 32  # codes + E8M0 scales
        self.units, self.elems_per_unit = w.rows, w.k

    def to_device(self, torch, dev):
        self.x = torch.from_numpy(self.w.x.view(np.int16)).to(dev).view(torch.bfloat16)
        self.p = torch.empty(self.w.rows, self.w.k // 2, dtype=torch.uint8, device=dev)
        self.s = torch.empty(self.w.rows, self.w.k // 32, dtype=torch.uint8, device=dev)

    def launch(self, fp4, stream):
        fp4.fp4_mx_quantize(self.x, self.p, self.s, stream=stream)

    def e2e_jobs(self, torch, fp4, chunks):
        hx = torch.from_numpy(self.w.x.view(np.int16)).pin_memory().view(torch.bfloat16)
        hp = torch.empty(self.p.shape, dtype=torch.uint8).pin_memory()
        hs = torch.empty(self.s.shape, dtype=torch.uint8).pin_memory()
        jobs = []
        for r0, r1 in _row_chunks(self.w.rows, chunks):
            def fn(st, r0=r0, r1=r1):
                self.x[r0:r1].copy_(hx[r0:r1], non_blocking=True)
                fp4.fp4_mx_quantize(self.x[r0:r1], self.p[r0:r1], self.s[r0:r1], stream=st)
                hp[r0:r1].copy_(self.p[r0:r1], non_blocking=True)
                hs[r0:r1].copy_(self.s[r0:r1], non_blocking=True)
            jobs.append((hx[r0:r1].numel() * 2, hp[r0:r1].numel() + hs[r0:r1].numel(), fn))
        return jobs

    def oracle_units(self, o, n, threads):
        o.mx_quantize(self.w.x[:n], threads)

    def sample_name(self):
        return f"rows of {self.w.name}"


class MoeGemmOp:
    """fp4_mx_moe_gemm: bf16 activations grouped by expert x MXFP4 expert weights."""
    kind, kernel = "mx_moe_gemm", "mx_moe_gemm_kernel"

    def __init__(self, w, rows_per_expert: int, seed: int = 6):
        from block_scaled_fp4_mx_gb300 import inputs
        self.experts = 32
        self.n = w.rows // self.experts
        self.k = w.k
        self.w = w
        self.rows = rows_per_expert
        t = self.experts * rows_per_expert
        self.a_bits = inputs.bf16_normal_bits(np.random.default_rng(seed), t * self.k,
                                              scale=1.0).reshape(t, self.k)
        self.offsets = np.arange(self.experts + 1, dtype=np.int64) * rows_per_expert
        self.elems = w.n_elems  # weights decoded per launch
        self.flops = 2.0 * t * self.n * self.k
        self.out_bytes = 2 * t * self.n
        self.bytes = w.packed.size + w.scales.size + 2 * t * self.k + self.out_bytes
        self.min_bytes = self.bytes
        self.units, self.elems_per_unit = self.experts, self.n * self.k
        self.label = f"mx_moe_gemm_{rows_per_expert}_tokens_per_expert_{self.n}x{self.k}"
        # up to 64 tokens per expert the weight stream (0.53 B per weight) takes longer
        # than the MMAs at the bf16 peak: the roofline is HBM bandwidth
        self.hbm_bound = self.bytes / 6.8e12 > self.flops / 1.9e15

    def to_device(self, torch, dev):
        self.a = torch.from_numpy(self.a_bits.view(np.int16)).to(dev).view(torch.bfloat16)
        self.off = torch.from_numpy(self.offsets).to(dev)
        self.wp = torch.from_numpy(self.w.packed.reshape(self.experts, self.n, self.k // 2)).to(dev)
        self.ws = torch.from_numpy(self.w.scales.reshape(self.experts, self.n, self.k // 32)).to(dev)
        self.o = torch.empty(self.a.shape[0], self.n, dtype=torch.bfloat16, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)

    def launch(self, fp4, stream):
        fp4.fp4_mx_moe_gemm(self.a, self.off, self.wp, self.ws, self.rows, out=self.o,
                            status=self.status, stream=stream)

    unfused_what = ("fp4_mx_unpack of the weights to bf16 + cuBLAS batched bf16 GEMM "
                    "(torch.bmm), same inputs")

    def unfused(self, torch, fp4, stream):
        """The two-step path for comparison: fp4_mx_unpack of all expert weights to
        bf16 in HBM, then a cuBLAS batched bf16 GEMM."""
        if not hasattr(self, "w_bf16"):
            self.w_bf16 = torch.empty(self.experts, self.n, self.k, dtype=torch.bfloat16,
                                      device=self.a.device)
        fp4.fp4_mx_unpack(self.wp, self.ws, out=self.w_bf16.view(self.experts, self.n, self.k),
                          stream=stream)
        a3 = self.a.view(self.experts, self.rows, self.k)
        torch.bmm(a3, self.w_bf16.transpose(1, 2), out=self.o.view(self.experts, self.rows, self.n))

    def e2e_jobs(self, torch, fp4, chunks):
        ha = torch.from_numpy(self.a_bits.view(np.int16)).pin_memory().view(torch.bfloat16)
        ho = torch.empty(self.o.shape, dtype=torch.bfloat16).pin_memory()

        def fn(st):
            self.a.copy_(ha, non_blocking=True)
            fp4.fp4_mx_moe_gemm(self.a, self.off, self.wp, self.ws, self.rows, out=self.o,
                                status=self.status, stream=st)
            ho.copy_(self.o, non_blocking=True)
        return [(ha.numel() * 2, ho.numel() * 2, fn)]

    def oracle_units(self, o, n, threads):
        r = n * self.rows
        o.mx_moe_gemm(self.a_bits[:r], self.offsets[:n + 1],
                      self.w.packed.reshape(self.experts, self.n, self.k // 2)[:n],
                      self.w.scales.reshape(self.experts, self.n, self.k // 32)[:n], threads)

    def sample_name(self):
        return f"experts of the MoE GEMM ({self.rows} tokens each)"


class MoeForwardOp:
    """fp4_mx_moe_forward: the whole MoE layer (routing, gate/up GEMM with
    silu(gate) * up, down GEMM, top-k weighted sum) on the MoE weights: 4,096 tokens,
    top-4 of 32 experts, hidden 2,880, intermediate 2,880."""
    kind, kernel = "mx_moe_forward", "mx_moe_forward (all kernels)"
    launches = 5  # route (count + scan), scatter, gate/up GEMM, down GEMM, combine

    def __init__(self, w1, w2, tokens: int = 4096, topk: int = 4, seed: int = 9):
        from block_scaled_fp4_mx_gb300 import inputs
        self.experts = 32
        self.n2, self.k = w1.rows // self.experts, w1.k  # 2N, K
        self.n = self.n2 // 2
        assert w2.rows // self.experts == self.k and w2.k == self.n
        self.w1, self.w2, self.tokens, self.topk = w1, w2, tokens, topk
        rng = np.random.default_rng(seed)
        self.a_bits = inputs.bf16_normal_bits(rng, tokens * self.k, scale=1.0).reshape(tokens, self.k)
        self.ids = np.stack([rng.permutation(self.experts)[:topk] for _ in range(tokens)]).astype(np.int32)
        wts = rng.random((tokens, topk)).astype(np.float32)
        self.wts = (wts / wts.sum(axis=1, keepdims=True)).astype(np.float32)
        slots = tokens * topk
        self.elems = w1.n_elems + w2.n_elems  # every expert weight decoded (at least once)
        self.flops = 2.0 * slots * (self.n2 * self.k + self.k * self.n)
        self.out_bytes = 2 * tokens * self.k
        self.bytes = (w1.packed.size + w1.scales.size + w2.packed.size + w2.scales.size
                      + 2 * tokens * self.k + 8 * slots + self.out_bytes)
        self.min_bytes = self.bytes
        self.units, self.elems_per_unit = self.experts, self.elems // self.experts
        self.label = f"mx_moe_forward_{tokens}_tokens_top{topk}"
        self.hbm_bound = self.bytes / 6.8e12 > self.flops / 1.9e15

    def to_device(self, torch, dev):
        import block_scaled_fp4_mx_gb300 as fp4
        e, k, n, n2 = self.experts, self.k, self.n, self.n2
        self.a = torch.from_numpy(self.a_bits.view(np.int16)).to(dev).view(torch.bfloat16)
        self.t_ids = torch.from_numpy(self.ids).to(dev)
        self.t_wts = torch.from_numpy(self.wts).to(dev)
        self.w1p = torch.from_numpy(self.w1.packed.reshape(e, n2, k // 2)).to(dev)
        self.w1s = torch.from_numpy(self.w1.scales.reshape(e, n2, k // 32)).to(dev)
        self.w2p = torch.from_numpy(self.w2.packed.reshape(e, k, n // 2)).to(dev)
        self.w2s = torch.from_numpy(self.w2.scales.reshape(e, k, n // 32)).to(dev)
        need = fp4.fp4_mx_moe_workspace_bytes(self.tokens, self.topk, e, n, k)
        self.work = torch.empty(need, dtype=torch.uint8, device=dev)
        self.o = torch.empty(self.tokens, k, dtype=torch.bfloat16, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)

    def launch(self, fp4, stream):
        fp4.fp4_mx_moe_forward(self.a, self.t_ids, self.t_wts, self.w1p, self.w1s, self.w2p,
                               self.w2s, out=self.o, workspace=self.work, status=self.status,
                               stream=stream)

    cpu_start_units = 1  # one expert of the oracle layer is already a few seconds
    unfused_what = ("fp4_mx_unpack of both weight stacks to bf16 + per-expert cuBLAS GEMMs, "
                    "torch silu * mul and index_add top-k sum (slot sort precomputed), same inputs")

    def unfused(self, torch, fp4, stream):
        """The same layer from fp4_mx_unpack of both weight stacks to bf16 in HBM and
        torch ops (cuBLAS GEMMs per expert, silu * mul, index_add for the top-k sum);
        the slot sort is done once, outside the timed region."""
        e, k, n, n2 = self.experts, self.k, self.n, self.n2
        if not hasattr(self, "w1_bf16"):
            dev = self.a.device
            self.w1_bf16 = torch.empty(e, n2, k, dtype=torch.bfloat16, device=dev)
            self.w2_bf16 = torch.empty(e, k, n, dtype=torch.bfloat16, device=dev)
            flat = self.ids.reshape(-1)
            order = np.argsort(flat, kind="stable")
            self.u_tok = torch.from_numpy(order // self.topk).to(dev)
            self.u_w = torch.from_numpy(self.wts.reshape(-1)[order]).to(dev)
            self.u_off = np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=e))])
            self.u_y = torch.empty(flat.size, k, dtype=torch.bfloat16, device=dev)
        fp4.fp4_mx_unpack(self.w1p, self.w1s, out=self.w1_bf16, stream=stream)
        fp4.fp4_mx_unpack(self.w2p, self.w2s, out=self.w2_bf16, stream=stream)
        xg = self.a.index_select(0, self.u_tok)
        for x in range(e):
            r0, r1 = int(self.u_off[x]), int(self.u_off[x + 1])
            if r1 > r0:
                h = xg[r0:r1] @ self.w1_bf16[x].T
                act = torch.nn.functional.silu(h[:, :n]) * h[:, n:]
                torch.matmul(act, self.w2_bf16[x].T, out=self.u_y[r0:r1])
        out = torch.zeros(self.tokens, k, dtype=torch.float32, device=self.a.device)
        out.index_add_(0, self.u_tok, self.u_y.float() * self.u_w[:, None])
        self.o.copy_(out)

    def e2e_jobs(self, torch, fp4, chunks):
        ha = torch.from_numpy(self.a_bits.view(np.int16)).pin_memory().view(torch.bfloat16)
        hi = torch.from_numpy(self.ids).pin_memory()
        hw = torch.from_numpy(self.wts).pin_memory()
        ho = torch.empty(self.o.shape, dtype=torch.bfloat16).pin_memory()

        def fn(st):
            self.a.copy_(ha, non_blocking=True)
            self.t_ids.copy_(hi, non_blocking=True)
            self.t_wts.copy_(hw, non_blocking=True)
            self.launch(fp4, st)
            ho.copy_(self.o, non_blocking=True)
        return [(ha.numel() * 2 + hi.numel() * 4 + hw.numel() * 4, ho.numel() * 2, fn)]

    def oracle_units(self, o, n, threads):
        """The layer restricted to the first n experts (slots on other experts are
        dropped): decode and GEMM work both scale with n."""
        e, k, nn, n2 = self.experts, self.k, self.n, self.n2
        ids = np.where(self.ids < n, self.ids, -1)
        o.mx_moe_forward(self.a_bits, ids, self.wts,
                         self.w1.packed.reshape(e, n2, k // 2)[:n], self.w1.scales.reshape(e, n2, k // 32)[:n],
                         self.w2.packed.reshape(e, k, nn // 2)[:n], self.w2.scales.reshape(e, k, nn // 32)[:n],
                         threads)

    def sample_name(self):
        return (f"experts of the MoE layer ({self.tokens} tokens, top-{self.topk}; "
                "slots on other experts dropped)")


def load_workload(name: str):
    """The ops of one step of the named workload, in launch order."""
    from block_scaled_fp4_mx_gb300 import inputs
    if name == "step":
        return ([MxOp(x) for x in inputs.mx_moe()] + [NvGatherOp(inputs.nv_embedding_200k())]
                + [MxOp(inputs.mx_stress())])
    table = {
        "mx_moe": lambda: [MxOp(x) for x in inputs.mx_moe()],
        "mx_stress": lambda: [MxOp(inputs.mx_stress())],
        "mx_exhaustive": lambda: [MxOp(inputs.mx_exhaustive())],
        "nv_embedding_200k": lambda: [NvGatherOp(inputs.nv_embedding_200k())],
        "nv_embedding_32k": lambda: [NvGatherOp(inputs.nv_embedding_32k())],
        "nv_dequant_200k": lambda: [NvDenseOp(inputs.nv_embedding_200k())],
        "nv_dequant_32k": lambda: [NvDenseOp(inputs.nv_embedding_32k())],
        "mx_quantize_moe": lambda: [MxQuantOp(w) for w in inputs.bf16_moe()],
        "kv_pages": lambda: [MxPagesOp(inputs.kv_pages())],
        "mx_moe_gemm_8": lambda: [MoeGemmOp(w, 8) for w in inputs.mx_moe()],
        "mx_moe_gemm_32": lambda: [MoeGemmOp(w, 32) for w in inputs.mx_moe()],
        "mx_moe_gemm_128": lambda: [MoeGemmOp(inputs.mx_moe()[0], 128)],
        "mx_moe_gemm_512": lambda: [MoeGemmOp(inputs.mx_moe()[0], 512)],
        "mx_moe_forward": lambda: [MoeForwardOp(*inputs.mx_moe())],
        "mx_moe_forward_decode": lambda: [MoeForwardOp(*inputs.mx_moe(), tokens=64)],
    }
    return table[name]()


def side_workload(name: str):
    """Small workloads timed in the same run outside the step (latency figures):
    the exhaustive 256 x 256 MXFP4 unpack and the 32k-vocabulary NVFP4 gather."""
    from block_scaled_fp4_mx_gb300 import inputs
    if name == "step":
        return [MxOp(inputs.mx_exhaustive()), NvGatherOp(inputs.nv_embedding_32k())]
    return []


def workload_label(name: str) -> str:
    if name == "step":
        return ("mx_moe_unpack_32x(5760+2880)x2880 + "
                "nv_embedding_gather_200000x8192_zipf1.1_ids64x256 + "
                "mx_stress_unpack_2^31_codes")
    return name


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            peaks = json.load(fh)
        return float(peaks["hbm_gbs"]), "measured"
    except Exception:  # noqa: BLE001
        return FALLBACK_HBM_GBS, "fallback"


def measured_tensor_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            peaks = json.load(fh)
        return float(peaks["bf16_tflops"]), "measured"
    except Exception:  # noqa: BLE001
        return 1900.0, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in ("block_scaled_fp4_mx_gb300/csrc/mx_unpack.cu",
                "block_scaled_fp4_mx_gb300/csrc/fp4_decode.cuh"):
        with open(os.path.join(ROOT, rel), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def workload_traffic(kind: str, workload: str, elements_per_launch: float):
    """DRAM bytes (read + write) per launch of one workload from the committed ncu
    captures in profiles/dram_traffic_by_workload.json, with the capture's command;
    (None, None) without a capture, (None, "stale") once a listed source changed."""
    path = os.path.join(ROOT, "profiles", "dram_traffic_by_workload.json")
    try:
        with open(path) as fh:
            recs = json.load(fh)
    except Exception:  # noqa: BLE001
        return None, None
    for rec in recs:
        if rec["kind"] != kind or rec["workload"] != workload:
            continue
        if abs(rec["launch_elements"] - elements_per_launch) > 0.5:
            return None, None
        h = hashlib.sha256()
        for rel in rec["sources"]:
            with open(os.path.join(ROOT, rel), "rb") as fh:
                h.update(fh.read())
        if h.hexdigest()[:16] != rec["source_sha256_16"]:
            return None, "stale"
        return rec["dram_bytes_read"] + rec["dram_bytes_write"], rec["capture"]
    return None, None


def ncu_traffic(kind: str, elements_per_launch: float):
    """DRAM bytes per launch of the MXFP4 kernel from the committed ncu capture,
    scaled to this launch size; None for other kernels or once the kernel source
    changed since the capture."""
    if kind != "mx_unpack":
        return None, None
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

def op_label(op) -> str:
    """Name of the workload an op runs on (the input's name)."""
    if hasattr(op, "label"):
        return op.label
    for attr in ("x", "w", "kv"):
        v = getattr(op, attr, None)
        if v is not None and hasattr(v, "name"):
            return v.name
    return op.kind


def per_launch_record(op, launch_s: float, peak: float, tensor_peak: float) -> dict:
    """Throughput figures of one launch of ``op`` that took ``launch_s`` seconds."""
    rec = {"avg_launch_us": launch_s * 1e6, "elements": op.elems,
           "elements_per_s": op.elems / launch_s, "algorithmic_bytes": op.bytes,
           "gbs": op.bytes / launch_s / 1e9, "frac_of_peak": op.bytes / launch_s / 1e9 / peak}
    if op.min_bytes != op.bytes:
        rec["distinct_row_bytes"] = op.min_bytes
        rec["gbs_distinct_rows"] = op.min_bytes / launch_s / 1e9
        rec["frac_of_peak_distinct_rows"] = rec["gbs_distinct_rows"] / peak
    if getattr(op, "flops", 0.0):
        rec["tflops"] = op.flops / launch_s / 1e12
        rec["frac_of_tensor_peak"] = rec["tflops"] / tensor_peak
    return rec


def time_alone(torch, fp4, op, stream, launches: int) -> float:
    """Mean seconds per launch of ``op`` run back to back (after 3 warm-up launches).
    The launches are captured once in a CUDA graph and the graph is replayed, so
    that short kernels are timed on the device, not at the host's launch rate."""
    for _ in range(3):
        op.launch(fp4, stream)
    torch.cuda.synchronize()
    graph = None
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            capture = torch.cuda.current_stream()
            for _ in range(launches):
                op.launch(fp4, capture)
        graph.replay()
        torch.cuda.synchronize()
    except Exception:  # noqa: BLE001 -- an op that cannot be captured is timed directly
        graph = None
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for _ in range(launches):
            op.launch(fp4, stream)
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / 1e3 / launches


def run_ours(args, d: Dist):
    import torch

    import block_scaled_fp4_mx_gb300 as fp4

    dev = torch.device("cuda", d.local_rank)
    torch.cuda.set_device(dev)
    d.init("nccl")
    fp4.load()
    ops = load_workload(args.workload)
    side = [] if args.no_side else side_workload(args.workload)
    for op in ops + side:
        op.to_device(torch, dev)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)

    step_elems = sum(op.elems for op in ops)
    step_bytes = sum(op.bytes for op in ops)

    def step(ev=None):
        for i, op in enumerate(ops):
            if ev is not None:
                ev[i][0].record(stream)
            op.launch(fp4, stream)
            if ev is not None:
                ev[i][1].record(stream)

    mk = lambda: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    sampler = ClockSampler(dev.index)
    sampler.start()
    events = [[mk() for _ in ops] for _ in range(args.steps)]
    start, end = mk()
    d.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    start.record(stream)
    for k in range(args.steps):
        step(events[k])
    end.record(stream)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    d.barrier()
    sampler.stop()
    elapsed_ms = d.max(start.elapsed_time(end), dev)
    k = args.steps
    value = step_elems * k * d.world / (elapsed_ms / 1e3)
    alg_gbs = step_bytes * k / (elapsed_ms / 1e3) / 1e9
    peak, peak_kind = measured_peak()
    tensor_peak, tensor_kind = measured_tensor_peak()

    # per workload: its launch inside the step, and the same launch run back to back
    op_ms = [sum(ev[i][0].elapsed_time(ev[i][1]) for ev in events) for i in range(len(ops))]
    configs = []
    for i, op in enumerate(ops):
        rec = {"workload": op_label(op), "kernel": op.kernel, "in_step": True,
               **per_launch_record(op, op_ms[i] / 1e3 / k, peak, tensor_peak)}
        # DRAM bytes of this launch from a committed ncu capture of the same kernel
        # source and workload, over this run's in-step time
        dram, dram_src = workload_traffic(op.kind, rec["workload"], op.elems)
        if dram is None and op.kind == "mx_unpack":
            dram, dram_src = ncu_traffic(op.kind, op.elems)
        if dram is not None:
            launch_s = op_ms[i] / 1e3 / k
            rec.update(dram_bytes_per_launch=dram, dram_gbs=dram / launch_s / 1e9,
                       dram_frac_of_peak=dram / launch_s / 1e9 / peak, dram_source=dram_src)
        configs.append(rec)
    for op in side:
        configs.append({"workload": op_label(op), "kernel": op.kernel, "in_step": False})
    if not args.no_alone:
        for rec, op in zip(configs, ops + side):
            launches = args.alone_launches if op.bytes > 64e6 else 10 * args.alone_launches
            alone = per_launch_record(op, time_alone(torch, fp4, op, stream, launches), peak,
                                      tensor_peak)
            if rec["in_step"]:
                rec["alone"] = {key: alone[key] for key in alone
                                if key not in ("elements", "algorithmic_bytes", "distinct_row_bytes")}
                rec["alone"]["launches"] = launches
            else:
                rec.update(alone, launches_timed=launches)

    # per kernel kind: summed bytes and durations of its launches inside the step
    kernels = {}
    for i, op in enumerate(ops):
        kk = kernels.setdefault(op.kind, {"kernel": op.kernel, "launches_per_step": 0, "ms": 0.0,
                                          "elements": 0, "bytes": 0, "min_bytes": 0, "flops": 0.0})
        kk["flops"] += getattr(op, "flops", 0.0)
        kk["launches_per_step"] += 1
        kk["ms"] += op_ms[i]
        kk["elements"] += op.elems
        kk["bytes"] += op.bytes
        kk["min_bytes"] += op.min_bytes
    for kk in kernels.values():
        n = kk["launches_per_step"]
        launch_s = kk.pop("ms") / 1e3 / (k * n)
        kk.update(avg_launch_us=launch_s * 1e6, elements_per_launch=kk["elements"] / n,
                  algorithmic_bytes_per_launch=kk["bytes"] / n,
                  gbs=kk["bytes"] / n / launch_s / 1e9,
                  frac_of_peak=kk["bytes"] / n / launch_s / 1e9 / peak)
        if kk["min_bytes"] != kk["bytes"]:
            kk["distinct_row_bytes_per_launch"] = kk["min_bytes"] / n
            kk["gbs_distinct_rows"] = kk["min_bytes"] / n / launch_s / 1e9
        if kk["flops"]:
            kk["tflops"] = kk["flops"] / n / launch_s / 1e12
            kk["frac_of_tensor_peak"] = kk["tflops"] / tensor_peak
        for key in ("elements", "bytes", "min_bytes", "flops"):
            kk.pop(key)
    dominant = max(kernels, key=lambda kind: kernels[kind]["avg_launch_us"]
                   * kernels[kind]["launches_per_step"])
    dk = kernels[dominant]
    traffic, capture = ncu_traffic(dominant, dk["elements_per_launch"])
    roofline = {"kernel": dk["kernel"], "bound": "hbm", "achieved": dk["gbs"], "peak": peak,
                "unit": "GB/s", "frac": dk["gbs"] / peak,
                "peak_source": "measured (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                else "fallback 6.8 TB/s",
                "traffic": traffic, "traffic_source": capture}
    hbm_bound = all(getattr(op, "hbm_bound", False) for op in ops if op.kind == dominant)
    if "tflops" in dk and hbm_bound:
        roofline.update(tflops=dk["tflops"], tensor_peak=tensor_peak,
                        tensor_frac=dk["tflops"] / tensor_peak,
                        note="weight streaming takes longer than the MMAs at the bf16 peak: "
                             "HBM roofline on the algorithmic bytes (codes, scales, "
                             "activations, output)")
    elif "tflops" in dk:
        roofline.update(bound="tensor", achieved=dk["tflops"], peak=tensor_peak, unit="TFLOP/s",
                        frac=dk["tflops"] / tensor_peak,
                        peak_source="measured dense bf16 burst (MEASURED_PEAKS.json bf16_tflops)"
                        if tensor_kind == "measured" else "fallback 1.9 PFLOP/s bf16",
                        hbm_gbs=dk["gbs"], hbm_frac=dk["gbs"] / peak)

    comparison = None
    if all(hasattr(op, "unfused") for op in ops):
        for _ in range(3):
            for op in ops:
                op.unfused(torch, fp4, stream)
        c0, c1 = mk()
        torch.cuda.synchronize()
        c0.record(stream)
        for _ in range(max(1, min(k, 50))):
            for op in ops:
                op.unfused(torch, fp4, stream)
        c1.record(stream)
        torch.cuda.synchronize()
        ms_unfused = c0.elapsed_time(c1) / max(1, min(k, 50))
        comparison = {"unfused_ms_per_step": ms_unfused,
                      "fused_ms_per_step": elapsed_ms / k,
                      "speedup": ms_unfused / (elapsed_ms / k),
                      "what": " + ".join(dict.fromkeys(op.unfused_what for op in ops))}
        for op in ops:
            op.launch(fp4, stream)  # leave the fused result in place
        torch.cuda.synchronize()

    e2e = None if args.no_e2e else run_e2e(args, d, dev, ops, step_elems)
    cpu = None
    if d.rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(ops, side, budget_s=args.cpu_budget)
        for rec in configs:
            oc = cpu["by_workload"].get(rec["workload"])
            if oc and "elements_per_s" in rec:
                rec["oracle"] = oc

    out_bytes = sum(getattr(op, "out_bytes", 2 * op.elems) for op in ops)  # bf16 outputs by default
    in_bytes = step_bytes - out_bytes
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": d.world, "steps": k,
        "warmup": args.warmup, "ms_per_step": elapsed_ms / k, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int16+fp32", "data": "synthetic",
        "config": {"workload": workload_label(args.workload),
                   "elements_per_step": step_elems,
                   "elements_per_step_by_kernel": {
                       kind: sum(op.elems for op in ops if op.kind == kind)
                       for kind in dict.fromkeys(op.kind for op in ops)},
                   "algorithmic_bytes_per_step": step_bytes,
                   "l2": ("no flush: inputs (%.0f MB) and outputs (%.0f MB) per step exceed the "
                          "129 MB L2" % (in_bytes / 1e6, out_bytes / 1e6))
                   if step_bytes > 129e6 else
                   ("no flush: the step's %.1f MB fit in the 129 MB L2 (a launch-bound parity "
                    "workload, L2-resident across steps)" % (step_bytes / 1e6)),
                   "parallelism": f"replicas x{d.world}"},
        "hbm_gbs_algorithmic": alg_gbs, "pct_of_peak_hbm": 100.0 * alg_gbs / peak,
        "roofline": roofline, "kernels": kernels, "configs": configs, "cpu_baseline": cpu,
        "e2e": e2e, **({"comparison": comparison} if comparison else {}),
        "gpu_launches": sum(getattr(op, "launches", 1) for op in ops) * k,
        "clocks": sampler.summary(t0, t1),
        "device": torch.cuda.get_device_name(dev),
    }
    if d.rank == 0:
        emit(line, args)
    d.close()


def _row_chunks(n: int, chunks: int):
    step = max(1, -(-n // max(1, chunks)))
    return [(r, min(n, r + step)) for r in range(0, n, step)]


def run_e2e(args, d, dev, ops, step_elems):
    """Same steps through the public API with pinned host buffers: every step
    copies its inputs host->device, decodes, and copies its outputs back. Each
    tensor is cut into row chunks issued round-robin on a few streams, so the
    host->device copies, the kernels and the device->host copies of different
    chunks overlap (the copy engines of both directions run at once)."""
    import torch

    import block_scaled_fp4_mx_gb300 as fp4

    main = torch.cuda.current_stream(dev)
    streams = [torch.cuda.Stream(dev) for _ in range(max(1, args.e2e_streams))]
    jobs, launches = [], 0
    for op in ops:
        op_jobs = op.e2e_jobs(torch, fp4, args.e2e_chunks)
        jobs += op_jobs
        launches += getattr(op, "launches", 1) * len(op_jobs)
    h2d = sum(j[0] for j in jobs)
    d2h = sum(j[1] for j in jobs)

    def step():
        start = torch.cuda.Event()
        start.record(main)
        for st in streams:
            st.wait_event(start)
        for n, (_, _, fn) in enumerate(jobs):
            st = streams[n % len(streams)]
            with torch.cuda.stream(st):
                fn(st)
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
            "ms_per_step": ms / steps, "gpu_launches_per_step": launches,
            "host_link_gbs": (h2d + d2h) / (ms / steps / 1e3) / 1e9,
            "note": f"each step's packed codes, scales and ids copied in and all bf16 outputs "
                    f"copied out, {len(jobs)} row chunks on {len(streams)} streams; an "
                    f"embedding table being gathered from stays resident (model weights)"}


# ---------------------------------------------------------------------------
# CPU oracle timings
# ---------------------------------------------------------------------------

def cpu_rates(ops, seconds: float, threads: int | None = None):
    """Oracle throughput (elements/s) per workload, on leading units (rows or ids)
    of that workload's input, sized to take about ``seconds`` each, on ``threads``
    host threads (default: all of them). Returns ({workload: (rate, units)},
    description, threads)."""
    import oracle

    o = oracle.get()
    threads = o.max_threads() if threads is None else threads
    rates, desc = {}, []
    for op in ops:
        label = op_label(op)
        n = max(1, min(op.units, getattr(op, "cpu_start_units", 16)))
        while True:
            t = time.perf_counter()
            op.oracle_units(o, n, threads)
            dt = time.perf_counter() - t
            if dt >= seconds / 4 or n == op.units:
                break
            n = min(op.units, int(n * max(2.0, seconds / 2 / max(dt, 1e-4))))
        reps, total = 0, 0.0
        while total < seconds and reps < 50:
            t = time.perf_counter()
            op.oracle_units(o, n, threads)
            total += time.perf_counter() - t
            reps += 1
        rates[label] = (n * op.elems_per_unit * reps / total, n)
        desc.append(f"{label}: first {n} {op.sample_name()} ({n * op.elems_per_unit} codes) x{reps}")
    return rates, "; ".join(desc), threads


def cpu_baseline(ops, side=(), budget_s: float = 12.0) -> dict:
    """The oracle on all host threads (the reported value) and, on a quarter of the
    budget, on one thread; per workload, the rate on a leading sample and the time
    the whole workload would take at that rate."""
    everything = list(ops) + list(side)
    total = sum(op.elems for op in ops)

    def combined(rates):
        return total / sum(op.elems / rates[op_label(op)][0] for op in ops)

    rates, desc, threads = cpu_rates(everything, budget_s / max(1, len(everything)))
    rates1, desc1, _ = cpu_rates(everything, budget_s / 4 / max(1, len(everything)), threads=1)
    by_workload = {}
    for op in everything:
        label = op_label(op)
        by_workload[label] = {
            "elements_per_s": rates[label][0], "elements_per_s_1_thread": rates1[label][0],
            "seconds_whole_workload": op.elems / rates[label][0],
            "seconds_whole_workload_1_thread": op.elems / rates1[label][0],
            "sample_units": rates[label][1], "whole": rates[label][1] == op.units}
    return {"value": combined(rates), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": desc + "; rates combined in the step's element mix",
            "by_workload": by_workload,
            "single_thread": {"value": combined(rates1), "cores": 1, "sample": desc1},
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
    ops = load_workload(args.workload)
    per_step = max(0.5, min(20.0, args.reference_budget / max(1, args.steps + args.warmup)))
    rates, desc, threads = cpu_rates(ops, per_step / len(ops))
    o = oracle.get()
    # each step: one leading slice of every workload, sized to about per_step / ops seconds
    plan = []
    for op in ops:
        rate = rates[op_label(op)][0]
        n = max(1, min(op.units, int(rate * per_step / len(ops) / op.elems_per_unit)))
        plan.append((op, n))
    sample_elems = sum(n * op.elems_per_unit for op, n in plan)
    times = []
    for i in range(args.warmup + args.steps):
        t = time.perf_counter()
        for op, n in plan:
            op.oracle_units(o, n, threads)
        dt = time.perf_counter() - t
        if i >= args.warmup:
            times.append(dt)
    sec = sum(times)
    value = sample_elems * len(times) / sec
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": d.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sec / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int16+fp32",
        "data": "synthetic",
        "config": {"workload": workload_label(args.workload),
                   "parallelism": "rank 0 only (CPU)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": "per step " + ", ".join(
                             f"{n} {op.sample_name()} ({n * op.elems_per_unit} codes)"
                             for op, n in plan), "cpu": _cpu_model()},
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
                    help="row chunks per tensor in the e2e leg (half as many for a gather)")
    ap.add_argument("--e2e-streams", type=int, default=3)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-side", action="store_true",
                    help="skip the small parity workloads timed outside the step")
    ap.add_argument("--no-alone", action="store_true",
                    help="skip timing each workload alone (launches back to back)")
    ap.add_argument("--alone-launches", type=int, default=20,
                    help="launches per large workload in the alone timing (10x for small ones)")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
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
