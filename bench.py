#!/usr/bin/env python3
"""Benchmark: fused attention forward TFLOPS on GB300 (one JSON line on stdout).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME]

A step is one fa_fwd launch over the whole workload (every (b, h) and every
query tile: Q tile load, K/V streaming, S = QK^T, mask, online softmax, P.V,
O = U / l and LSE).  The default workload is B=2, H=32, N=4096, d=128, bf16,
non-causal: the N=4096, d=128 point at which the throughput target is stated.
The metric is 4*B*H*N^2*d / t (halved for the causal mask), in TFLOPS, summed
over ranks.  Inputs are seeded synthetic tensors already resident in HBM; the
per-step working set (Q, K, V, O: 256 MiB) is larger than the 129 MB L2.

Multi-GPU: one process per GPU (torchrun); the (b, h) units are independent,
so each rank runs its own batch of heads with no data-path collective (weak
scaling); only the timing is reduced (max over ranks).

--impl reference times the oracle (the plain double-precision CPU
definition) on the host cores, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from online_softmax_tiling_gb300 import synth  # noqa: E402

DEFAULT_WORKLOAD = "T_b2h32n4096d128_bf16"
_CSRC = "online_softmax_tiling_gb300/csrc/"
# device code each timed path runs (the hash ties a committed ncu traffic
# figure to the kernel source it was measured on)
KERNEL_SOURCES = {
    "fused": [_CSRC + f for f in ("fa_fwd_kernel.cuh", "fa_fwd_qtile_kernel.cuh", "sm103_ptx.cuh")],
    "wide": [_CSRC + f for f in ("fa_fwd_kernel.cuh", "fa_fwd_wide_kernel.cuh", "sm103_ptx.cuh")],
    "naive": [_CSRC + f for f in ("fa_fwd_kernel.cuh", "naive_attention.cuh", "sm103_ptx.cuh")],
}
METRIC = "attn fwd TFLOPS (4*B*H*N^2*d/t, causal halved) @N=4096; % of GB300 dense TC peak"


# ----------------------------------------------------------------- helpers
def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_seed_base(w: synth.Workload, rank: int) -> int:
    """Each rank draws its own independent heads (weak scaling, disjoint units)."""
    return w.seed_base + 100 * rank


def max_over_ranks(value: float, world: int) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def kernel_hash(kind: str = "fused") -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, rel), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, khash: str):
    """DRAM bytes per launch recorded by an ncu capture of this exact kernel source."""
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    pat = re.compile(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)\s+kernel_hash:\s*([0-9a-f]+)"
                     r"\s+workload:\s*(\S+)")
    for name in sorted(os.listdir(pdir)):
        if not name.endswith((".md", ".txt")):
            continue
        with open(os.path.join(pdir, name), encoding="utf-8") as fh:
            for m in pat.finditer(fh.read()):
                if m.group(2) == khash and m.group(3) == workload:
                    return float(m.group(1))
    return None


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path, encoding="utf-8") as fh:
            return json.load(fh), "measured"
    return {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0}, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed
    region (the fallback where NVML cannot be loaded in-process)."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.lines = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        t0 = time.time()
        while not self.lines and time.time() - t0 < 10:
            time.sleep(0.02)
        self.lines.clear()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "source": "nvidia-smi"}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in list(self.lines):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons), "source": "nvidia-smi -lms 50"}


class NvmlClocks:
    """In-process clock record through NVML's read-only queries (ctypes on
    libnvidia-ml): the SM clock, its maximum, the power draw and the active
    clock-event (throttle) reasons, sampled by a thread about once per
    millisecond plus once at the start and the end of each timed region, so
    that even a region of a few milliseconds has samples.  The device is found
    by the PCI bus id of the CUDA device (NVML numbers every GPU of the
    machine, CUDA only the visible ones).  Nothing is ever set."""

    CLOCK_SM = 1
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch_device: int):
        import ctypes
        import torch
        self.ct = ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit_v2 failed")
        props = torch.cuda.get_device_properties(torch_device)
        self.handle = ctypes.c_void_p()
        ok = False
        if all(hasattr(props, a) for a in ("pci_domain_id", "pci_bus_id", "pci_device_id")):
            bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
            ok = lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(self.handle)) == 0
        if not ok:
            idx = torch_device
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            if vis and vis.split(",")[0].strip().isdigit():
                idx = int(vis.split(",")[torch_device].strip())
            if lib.nvmlDeviceGetHandleByIndex_v2(idx, ctypes.byref(self.handle)) != 0:
                raise OSError("no NVML handle for the CUDA device")
        self.lib = lib
        self._reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        mx = ctypes.c_uint()
        self.max_mhz = (float(mx.value) if lib.nvmlDeviceGetMaxClockInfo(
            self.handle, self.CLOCK_SM, ctypes.byref(mx)) == 0 else None)
        self.samples = []
        self._stop = threading.Event()
        self._thread = None

    def sample(self):
        ct = self.ct
        mhz, mw, rs = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.handle, self.CLOCK_SM, ct.byref(mhz)) != 0:
            return
        p = float(mw.value) / 1e3 if self.lib.nvmlDeviceGetPowerUsage(self.handle, ct.byref(mw)) == 0 \
            else None
        r = int(rs.value) if self._reasons_fn(self.handle, ct.byref(rs)) == 0 else 0
        self.samples.append((float(mhz.value), p, r))

    def _run(self):
        while not self._stop.is_set():
            self.sample()
            time.sleep(0.001)

    def start(self):
        self.samples = []
        self._stop.clear()
        self.sample()
        self._thread = threading.Thread(target=self._run, daemon=True)
        self._thread.start()

    def stop(self):
        self._stop.set()
        if self._thread is not None:
            self._thread.join(timeout=5)
        self.sample()
        sm = [s[0] for s in self.samples]
        pw = [s[1] for s in self.samples if s[1] is not None]
        reasons = set()
        for _, _, r in self.samples:
            reasons |= {nm for bit, nm in self.REASONS.items() if r & bit}
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz,
                "sm_mhz_min": min(sm) if sm else None,
                "power_w_max": max(pw) if pw else None, "samples": len(sm),
                "reasons": sorted(reasons), "source": "NVML in-process, ~1 kHz"}


def clock_sampler(torch_device: int):
    """NVML in-process where it loads, else nvidia-smi."""
    try:
        return NvmlClocks(torch_device)
    except (OSError, AttributeError, TypeError):
        return ClockSampler(torch_device)


def time_launches(step, stream, n: int, flush_buf=None):
    """CUDA-event times (ms) of n launches of `step` on `stream`: back to back
    (an event between consecutive launches), or with L2 flushed before each
    launch (a fill of flush_buf, outside the timed launch)."""
    import torch
    if flush_buf is None:
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
        evs[0].record(stream)
        for i in range(n):
            step()
            evs[i + 1].record(stream)
        torch.cuda.synchronize()
        return [evs[i].elapsed_time(evs[i + 1]) for i in range(n)]
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(n)]
    for a, b in pairs:
        flush_buf.fill_(1)
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in pairs]


L2_BYTES = 129 * 10 ** 6


def kernel_width(d: int) -> int:
    """Width of the kernel that serves head dimension d (64, 128, 192 or 256)."""
    return 64 if d <= 64 else 128 if d <= 128 else 192 if d <= 192 else 256


def ceiling_counts(w: synth.Workload) -> dict:
    """Per launch of the fused kernel: 2^x evaluations (one per visible query,
    key pair) and bytes read from L2 into the SMs (each CTA's Q tile and the K
    and V tiles it visits; tiles of 128 keys, with two 128-row query tiles per
    CTA for d <= 128 and one above)."""
    B, H, N, d = w.shape
    wide = kernel_width(d) > 128
    bm, bn = (128, 128) if wide else (256, 128)
    nkv = -(-N // bn)
    tiles = 0
    for qb in range(-(-N // bm)):
        if w.causal:
            last = min(qb * bm + bm - 1, N - 1)
            tiles += min(last // bn + 1, nkv)
        else:
            tiles += nkv
    exps = B * H * (N * (N + 1) // 2 if w.causal else N * N)
    l2 = B * H * (tiles * 2 * bn * d * 2 + N * d * 2)
    return {"exps": exps, "l2_bytes": l2}


def measure_ceilings(w, fa, torch, kernel_us: float, peaks: dict) -> dict:
    """Rates of the exp unit and of L2 -> SM reads (microbenchmarks in the
    library) turned into time floors for one launch of workload w."""
    cnt = ceiling_counts(w)
    buf = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
    ex2 = fa.fa_ceiling_ex2_rate(torch.cuda.current_stream())
    l2bw = fa.fa_ceiling_l2_read(buf.data_ptr(), buf.numel(), torch.cuda.current_stream())
    del buf
    return {
        "ex2_per_s": round(ex2, -6), "l2_read_GBps": round(l2bw / 1e9, 1),
        "per_launch": cnt,
        "floors_us": {
            "tensor": round(w.flops / (float(peaks.get("bf16_tflops", 1900.0)) * 1e12) * 1e6, 2),
            "exp": round(cnt["exps"] / ex2 * 1e6, 2),
            "l2_to_sm": round(cnt["l2_bytes"] / l2bw * 1e6, 2),
            "hbm": round(w.compulsory_bytes / (float(peaks.get("hbm_gbs", 6800.0)) * 1e9) * 1e6, 2)},
        "kernel_us": round(kernel_us, 2),
    }


def naive_model_bytes(w: synth.Workload) -> int:
    """HBM bytes of the step-by-step computation as "CUDA 算子工程" 14.2 counts
    them: Q, K, V read and O written once, S written once and read three
    times, P written once and read once (16-bit elements)."""
    B, H, N, d = w.shape
    return B * H * (4 * N * d * 2 + 6 * N * N * 2)


# -------------------------------------------------------------- our arm
def run_ours(args):
    import torch
    import online_softmax_tiling_gb300 as fa
    from online_softmax_tiling_gb300 import build

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    if rank == 0 or world > 1:
        build.build()
    barrier(world)

    w = synth.workload(args.workload)
    B, H, N, d = w.shape
    q_h, k_h, v_h = synth.make_inputs(w, seed_base=rank_seed_base(w, rank))
    tdt = torch.float16 if w.dtype == synth.FP16 else torch.bfloat16

    def host(bits):
        return torch.from_numpy(bits.view(np.int16)).view(tdt).pin_memory()

    qh, kh, vh = host(q_h), host(k_h), host(v_h)
    q, k, v = qh.cuda(), kh.cuda(), vh.cuda()
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    sptr = stream.cuda_stream
    naive = args.path == "naive"
    splits = 1 if naive else args.num_splits
    if splits == 0:
        splits = fa.fa_splitkv_num_splits(B, H, N, d, int(w.causal))
    if naive:
        ws_bytes = fa.fa_naive_workspace_size(B, H, N)
    else:
        ws_bytes = fa.fa_splitkv_workspace_size(B, H, N, d, splits) if splits > 1 else 0
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
    launches_per_step = 3 if naive else (2 if splits > 1 else 1)

    def step():
        if naive:
            st = fa.fa_naive_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                 lse.data_ptr(), B, H, N, d, w.scale, int(w.causal), w.dtype,
                                 ws.data_ptr(), ws_bytes, sptr)
        elif splits > 1:
            st = fa.fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), B, H, N, d, w.scale, int(w.causal), w.dtype,
                                   splits, ws.data_ptr(), ws_bytes, sptr)
        else:
            st = fa.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                           B, H, N, d, w.scale, int(w.causal), w.dtype, sptr)
        if st != fa.FA_OK:
            raise fa.FaError(st)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if fa.fa_check_device_status(sptr) != fa.FA_OK:
        raise RuntimeError("device status not OK after warm-up")

    # inputs larger than L2 stream from HBM anyway; smaller ones get L2
    # flushed (a 256 MiB fill, outside the timed launches) before every step
    flush = w.compulsory_bytes < 2 * L2_BYTES
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device="cuda") if flush else None
    clocks = clock_sampler(torch.cuda.current_device())
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    # every launch between two events on its stream: the sum is the timed
    # region (back to back), the median the typical launch
    per_launch = time_launches(step, stream, args.steps, flush_buf)
    wall_ms = (time.perf_counter() - t_wall) * 1e3
    barrier(world)
    clock_info = clocks.stop()
    dev_ms = sum(per_launch)
    median_ms = statistics.median(per_launch)
    del flush_buf
    # with L2 flushed before every step, also the warm figure: the same steps
    # back to back, inputs left in L2 by the previous step
    warm_ms = None
    if flush:
        warm_ms = statistics.median(time_launches(step, stream, args.steps))
    if fa.fa_check_device_status(sptr) != fa.FA_OK:
        raise RuntimeError("device status not OK after the timed region")
    ms_total = max_over_ranks(dev_ms, world)
    ms_per_step = ms_total / args.steps
    flops_rank = w.flops
    value = flops_rank * world / (ms_per_step * 1e-3) / 1e12

    # kernel roofline: one launch per step on `stream`, timed by the events above
    peaks, peak_src = measured_peaks()
    peak = float(peaks.get("bf16_tflops", 1900.0))
    achieved = flops_rank / (dev_ms / args.steps * 1e-3) / 1e12
    khash = kernel_hash("naive" if naive else ("wide" if kernel_width(d) > 128 else "fused"))
    traffic = profiled_traffic(w.name + ("_naive" if naive else ""), khash)
    if naive:
        # the step-by-step baseline is bound by memory traffic: report the
        # pages' byte count for it (S written, read three times, P written
        # and read, Q, K, V, O once) against the measured HBM copy rate
        hbm = float(peaks.get("hbm_gbs", 6800.0))
        model_bytes = naive_model_bytes(w)
        gbs = model_bytes / (dev_ms / args.steps * 1e-3) / 1e9
        roofline = {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                    "frac": round(gbs / hbm, 4), "traffic": traffic,
                    "algorithmic_bytes": model_bytes,
                    "peak_source": f"{peak_src} hbm_gbs", "kernel_hash": khash}
    else:
        roofline = {"bound": "tensor", "achieved": round(achieved, 3), "peak": peak,
                    "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                    "traffic": traffic, "peak_source": f"{peak_src} bf16_tflops (burst)",
                    "kernel_hash": khash}
        if "bf16_tflops_sustained" in peaks:
            # for context only: the same GEMM held for seconds under the power
            # cap, as long timed regions of this kernel are
            sus = float(peaks["bf16_tflops_sustained"])
            roofline["peak_sustained"] = sus
            roofline["frac_of_sustained"] = round(achieved / sus, 4)
    if traffic is not None:
        # measured DRAM bytes of one launch over this run's time per launch
        roofline["dram_gbps"] = round(traffic / (dev_ms / args.steps * 1e-3) / 1e9, 1)

    # end-to-end through the public API with host buffers: every step copies
    # its q, k, v from pinned host memory, calls the library and copies O and
    # LSE back.  Steps are pipelined two deep on three streams (H2D, compute,
    # D2H) with two device buffer sets, so that step i+1's inputs travel while
    # step i computes and step i-1's result returns.
    e2e_steps = max(4, min(args.steps, 20))
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    sets = []
    for bset in range(2):
        qb, kb, vb = (torch.empty_like(q) for _ in range(3))
        ob, lb = torch.empty_like(o), torch.empty_like(lse)
        oh = torch.empty(o.shape, dtype=tdt, pin_memory=True)
        lh = torch.empty(lse.shape, dtype=torch.float32, pin_memory=True)
        sets.append((qb, kb, vb, ob, lb, oh, lh))
    ev = {(name, bset): torch.cuda.Event() for name in ("in", "comp", "out") for bset in range(2)}

    def launch(qb, kb, vb, ob, lb, strm):
        if naive:
            st = fa.fa_naive_fwd(qb.data_ptr(), kb.data_ptr(), vb.data_ptr(), ob.data_ptr(),
                                 lb.data_ptr(), B, H, N, d, w.scale, int(w.causal), w.dtype,
                                 ws.data_ptr(), ws_bytes, strm.cuda_stream)
        elif splits > 1:
            st = fa.fa_fwd_splitkv(qb.data_ptr(), kb.data_ptr(), vb.data_ptr(), ob.data_ptr(),
                                   lb.data_ptr(), B, H, N, d, w.scale, int(w.causal), w.dtype,
                                   splits, ws.data_ptr(), ws_bytes, strm.cuda_stream)
        else:
            st = fa.fa_fwd(qb.data_ptr(), kb.data_ptr(), vb.data_ptr(), ob.data_ptr(),
                           lb.data_ptr(), B, H, N, d, w.scale, int(w.causal), w.dtype,
                           strm.cuda_stream)
        if st != fa.FA_OK:
            raise fa.FaError(st)

    def e2e_run(nsteps):
        for i in range(nsteps):
            bset = i & 1
            qb, kb, vb, ob, lb, oh, lh = sets[bset]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev[("comp", bset)])   # step i-2 has read this set
                qb.copy_(qh, non_blocking=True)
                kb.copy_(kh, non_blocking=True)
                vb.copy_(vh, non_blocking=True)
                ev[("in", bset)].record(s_in)
            stream.wait_event(ev[("in", bset)])
            if i >= 2:
                stream.wait_event(ev[("out", bset)])      # step i-2's result has left
            launch(qb, kb, vb, ob, lb, stream)
            ev[("comp", bset)].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev[("comp", bset)])
                oh.copy_(ob, non_blocking=True)
                lh.copy_(lb, non_blocking=True)
                ev[("out", bset)].record(s_out)

    e2e_run(2)
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    e2e_run(e2e_steps)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3, world) / e2e_steps
    h2d = 3 * q.numel() * q.element_size()
    d2h = o.numel() * o.element_size() + lse.numel() * 4
    del sets

    ceilings = None
    if rank == 0 and not args.no_ceilings and not naive:
        ceilings = measure_ceilings(w, fa, torch, dev_ms / args.steps * 1e3, peaks)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, q_h, k_h, v_h, budget_s=args.cpu_seconds)

    # every configured workload at its full size (rank 0; outside the timed
    # region above, which is the headline), with parity of sampled rows
    configs = None
    if rank == 0 and args.configs and not naive:
        del q, k, v, o, lse, ws
        torch.cuda.empty_cache()
        fbuf = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        configs = []
        for name in [c for c in args.configs.split(",") if c]:
            configs.append(sweep_config(name, fa, torch, peak, fbuf,
                                        with_parity=not args.no_cpu_baseline))
            torch.cuda.empty_cache()
        del fbuf

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": "TFLOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": synth.DTYPE_NAMES[w.dtype], "data": "synthetic (seeded N(0,1), SplitMix64 + Box-Muller)",
            "config": {**w.describe(), "parallelism": f"independent heads per rank x{world}",
                       "num_splits": splits, "path": args.path,
                       "l2": (f"L2 flushed before every step ({w.compulsory_bytes / 1e6:.1f} MB of "
                              f"Q, K, V, O, LSE per step vs 129 MB L2)") if flush else
                             (f"inputs larger than L2: {w.compulsory_bytes / 1e6:.1f} MB of Q, K, V, "
                              f"O, LSE per step vs 129 MB L2"),
                       "pct_of_peak": round(100 * value / world / peak, 2),
                       "warm_value": (round(flops_rank * world / (warm_ms * 1e-3) / 1e12, 3)
                                      if warm_ms else None)},
            "roofline": roofline,
            "e2e": {"value": round(flops_rank * world / (e2e_ms * 1e-3) / 1e12, 3),
                    "unit": "TFLOPS", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "steps": e2e_steps, "timing": "host wall clock around synchronised steps",
                    "pipelining": "2 buffer sets; H2D, compute, D2H on three streams"},
            "gpu_launches": args.steps * launches_per_step,
            "median_ms_per_launch": round(median_ms, 5),
            "kcycles_per_launch": (round(median_ms * clock_info["sm_mhz"], 1)
                                   if clock_info.get("sm_mhz") else None),
            "clocks": clock_info,
            "ceilings": ceilings,
            "wall_ms_timed_region": round(wall_ms, 3),
            "cpu_baseline": cpu,
            "configs": configs,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


SWEEP = ("C1", "C2", "C3", "C4", "C5", "C5r", "T_b2h32n4096d128_fp16", "T_b2h32n4096d128_bf16")


def sweep_config(name: str, fa, torch, peak: float, flush_buf, with_parity: bool,
                 seconds: float = 0.25) -> dict:
    """One workload at its full size, on the library's own split choice:
    the median per-launch time with L2 flushed before every launch and with
    launches back to back (warm), TFLOP/s and % of peak from the flushed
    median, the clock record of those launches, and (with_parity) the parity
    statistics of sampled rows against the oracle."""
    w = synth.workload(name)
    B, H, N, d = w.shape
    q_h, k_h, v_h = synth.make_inputs(w)
    tdt = torch.float16 if w.dtype == synth.FP16 else torch.bfloat16

    def dev(bits):
        return torch.from_numpy(bits.view(np.int16)).view(tdt).cuda()

    q, k, v = dev(q_h), dev(k_h), dev(v_h)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    sptr = stream.cuda_stream
    splits = fa.fa_splitkv_num_splits(B, H, N, d, int(w.causal))
    ws_bytes = fa.fa_splitkv_workspace_size(B, H, N, d, splits) if splits > 1 else 0
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")

    def step():
        if splits > 1:
            st = fa.fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), B, H, N, d, w.scale, int(w.causal), w.dtype,
                                   splits, ws.data_ptr(), ws_bytes, sptr)
        else:
            st = fa.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                           B, H, N, d, w.scale, int(w.causal), w.dtype, sptr)
        if st != fa.FA_OK:
            raise fa.FaError(st)

    for _ in range(3):
        step()
    one = statistics.median(time_launches(step, stream, 3))
    if fa.fa_check_device_status(sptr) != fa.FA_OK:
        raise RuntimeError(f"{name}: device status not OK after warm-up")
    n = int(min(300, max(20, seconds / (one * 1e-3))))
    clocks = clock_sampler(torch.cuda.current_device())
    clocks.start()
    flushed = time_launches(step, stream, n, flush_buf)
    warm = time_launches(step, stream, n)
    ci = clocks.stop()
    if fa.fa_check_device_status(sptr) != fa.FA_OK:
        raise RuntimeError(f"{name}: device status not OK after the timed launches")
    mf, mw = statistics.median(flushed), statistics.median(warm)
    tf = w.flops / (mf * 1e-3) / 1e12
    out = {"workload": w.name, "num_splits": splits, "launches": n,
           "launches_per_call": 2 if splits > 1 else 1,
           "median_ms_flushed": round(mf, 5), "median_ms_warm": round(mw, 5),
           "tflops": round(tf, 2), "tflops_warm": round(w.flops / (mw * 1e-3) / 1e12, 2),
           "pct_of_peak": round(100 * tf / peak, 2),
           "sm_mhz": ci.get("sm_mhz"), "clock_samples": ci.get("samples"),
           "clock_reasons": ci.get("reasons"),
           "kcycles_per_launch": (round(mf * ci["sm_mhz"], 1) if ci.get("sm_mhz") else None)}
    if with_parity:
        rows = synth.sample_rows(B * H, N, 256, w.seed_base + 9)
        if w.causal:   # the first rows see the fewest keys
            rows = np.unique(np.concatenate([rows, np.arange(min(N, 128), dtype=np.int64)]))
        rt = torch.from_numpy(rows).cuda()
        o_rows = o.view(-1, d).index_select(0, rt).view(torch.int16).cpu().numpy().view(np.uint16)
        lse_rows = lse.view(-1).index_select(0, rt).cpu().numpy()
        out["parity"] = cpu_leg_parity(w, q_h, k_h, v_h, rows, o_rows, lse_rows)
    del q, k, v, o, lse, ws
    return out


# --------------------------------------------------------- oracle timing
def _row_flops(w: synth.Workload, rows: np.ndarray) -> float:
    i = rows % w.N
    keys = np.minimum(i + 1, w.N) if w.causal else np.full(rows.shape, w.N)
    return float(4.0 * w.d * keys.sum())


def cpu_baseline(w, q_h, k_h, v_h, budget_s: float = 10.0):
    """Time the oracle (as it stands) on a bounded row sample of the workload."""
    import oracle
    cores = len(os.sched_getaffinity(0))
    BH = w.B * w.H
    # calibrate on a small sample, then size the sample to the time budget
    chunk = 16 * cores
    total_flops, total_t, nrows, s = 0.0, 0.0, 0, 0
    while total_t < budget_s and nrows < BH * w.N:
        rows = synth.sample_rows(BH, w.N, chunk, 777 + s, include_edges=False)
        t0 = time.perf_counter()
        oracle.attention_rows16(q_h, k_h, v_h, w.dtype, w.scale, w.causal, rows, nthreads=cores)
        total_t += time.perf_counter() - t0
        total_flops += _row_flops(w, rows)
        nrows += rows.size
        s += 1
    return {"value": round(total_flops / total_t / 1e12, 6), "unit": "TFLOPS", "cores": cores,
            "kind": "oracle",
            "sample": f"{nrows} seeded query rows (all their keys) of {w.name}, fp64, "
                      f"{total_t:.1f} s on {cores} host threads"}


def cpu_leg_parity(w, q_h, k_h, v_h, rows, o_rows, lse_rows) -> dict:
    """Part of the CPU-baseline leg: the oracle (as it stands) on sampled rows
    of one workload, timed on the host cores; its outputs are the parity
    reference for the same rows of the GPU run, gated as the tests gate them
    (error beyond half an output ulp: max <= 4e-3, mean <= 5e-4; LSE error
    <= 1e-4 relative to max(1, |LSE|); the ceilinged gate for the workload
    whose Q and K are drawn with std 2)."""
    import oracle
    from tests import parity
    cores = len(os.sched_getaffinity(0))
    t0 = time.perf_counter()
    o_ref, lse_ref, spread = oracle.attention_rows16(q_h, k_h, v_h, w.dtype, w.scale, w.causal,
                                                     rows, nthreads=cores, with_spread=True)
    t = time.perf_counter() - t0
    st = parity.compare(o_rows, lse_rows, o_ref, lse_ref, spread, w.dtype)
    gate = parity.gate_for(w)
    try:
        parity.assert_within(dict(st), w.name, gate)
        st["pass"] = True
    except AssertionError:
        st["pass"] = False
    st["gate"] = "plain" if gate is None else (
        f"widened: beyond both roundings <= {parity.MAX_EXCESS}, plain <= {gate.max_plain}, "
        f"at most {gate.max_frac} of elements over {parity.MAX_EXCESS}")
    st["rows"] = int(rows.size)
    st["oracle_s"] = round(t, 3)
    st["oracle_tflops"] = round(_row_flops(w, rows) / t / 1e12, 6)
    st["oracle_cores"] = cores
    return {k_: (float(f"{v_:.4g}") if isinstance(v_, float) else v_) for k_, v_ in st.items()}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    w = synth.workload(args.workload)
    q_h, k_h, v_h = synth.make_inputs(w)
    import oracle
    cores = len(os.sched_getaffinity(0))
    BH = w.B * w.H
    rows_per_step = args.ref_rows
    t_warm = 0.0
    for s in range(args.warmup):
        t0 = time.perf_counter()
        oracle.attention_rows16(q_h, k_h, v_h, w.dtype, w.scale, w.causal,
                                synth.sample_rows(BH, w.N, rows_per_step, 900 + s, False),
                                nthreads=cores)
        t_warm += time.perf_counter() - t0
    # each step a bounded sample: the timed steps together take at most about
    # --ref-seconds whatever --steps is (the rate, not the sample, is
    # reported).  The oracle hands its threads 16 rows at a time, so a step of
    # r rows lasts as long as one thread's share of 16-row chunks: the largest
    # r that fits is kept, and only the threads it keeps busy are started
    # (and reported).
    def chunks_per_thread(r):
        return -(-(-(-r // 16)) // cores)

    def step_rows(r):  # rows one thread works through in a step of r rows
        return r if r < 16 else 16 * chunks_per_thread(r)

    t_row = t_warm / args.warmup / step_rows(rows_per_step)  # one row on one thread
    while rows_per_step > 1 and args.steps * step_rows(rows_per_step) * t_row > args.ref_seconds:
        rows_per_step -= 16 if rows_per_step > 16 else 1
    threads = max(1, min(cores, -(-rows_per_step // 16)))
    flops, t = 0.0, 0.0
    for s in range(args.steps):
        rows = synth.sample_rows(BH, w.N, rows_per_step, 1900 + s, False)
        t0 = time.perf_counter()
        oracle.attention_rows16(q_h, k_h, v_h, w.dtype, w.scale, w.causal, rows, nthreads=threads)
        t += time.perf_counter() - t0
        flops += _row_flops(w, rows)
    value = flops / t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOPS",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(t / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1), SplitMix64 + Box-Muller)",
        "config": {**w.describe(), "parallelism": "host cores (oracle)"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOPS", "cores": threads,
                         "kind": "oracle",
                         "sample": f"{rows_per_step} seeded query rows per step of {w.name}"},
        "e2e": {"value": round(value, 6), "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--num-splits", type=int, default=1,
                    help="1 = one fused launch; 0 = library's split-KV choice; >= 2 = that many")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--path", choices=["fused", "naive"], default="fused",
                    help="naive: the step-by-step baseline with S and P in HBM")
    ap.add_argument("--no-ceilings", action="store_true",
                    help="skip the exp-rate and L2-bandwidth microbenchmarks")
    ap.add_argument("--configs", default=",".join(SWEEP),
                    help="workloads timed one by one after the headline (comma-separated; "
                         "empty = none), each with sampled-row parity against the oracle")
    ap.add_argument("--ref-rows", type=int, default=256,
                    help="--impl reference: at most this many query rows per step")
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="--impl reference: at most about this long for all timed steps together")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
