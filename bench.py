#!/usr/bin/env python
"""Benchmark of the fused attention library on one GB300 (or N replicas under torchrun).

Headline line: decode, B8 Hq=Hkv=32 Sq1 Skv4096 D128, BF16 in / BF16 O + FP32 LSE, split-KV.
`value` = algorithmic K/V bytes per step / device time per step (GB/s), inputs resident in HBM;
every step's K/V (512 MiB) is larger than L2, so no flush is needed between steps.
Also reported: the decode kernel's roofline fraction (timed alone through the library's timing
hook), an end-to-end figure through the C ABI with pinned host buffers, the CPU oracle baseline,
clock samples taken during the timed region, and the other specified workloads (single head,
prefill, wide-head decode, ragged GQA decode with NVFP4 output) under "workloads".

--impl reference times the CPU FP64 oracle on the same workload instead (bounded samples).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode KV GB/s and prefill TFLOP/s per GB300; fraction of HBM / tensor roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from one ncu capture of the
# named kernel, with the sha256 of its source file and the shared device headers at capture time;
# reported only while those sources are unchanged.
TRAFFIC = {
    # decode B8 H32 Sq1 Skv4096 D128 (decode_kernel<128, 0, 0>, 128 CTAs of two whole units): read
    # 537,030,656 + written 2,818,304 bytes (profiles/decode_kernel_decode-B8-H32-Skv4096-D128.md)
    "decode_kernel<128>": {"bytes": 539848960, "source_sha": "352c1ba17c15bf38"},
    # ragged GQA decode B64 Hq32 Hkv8 Skv<=32768 D128 (decode_kernel<128, 0, 1>): the quarter-size workload
    # (B16) read 1,005,865,216 + wrote 683,008 bytes for 1,001,226,240 algorithmic K/V bytes (1.005x); scaled
    # by the K/V bytes to the full workload's 4,106,002,432 (profiles/side-kernels_ragged-decode-wide-combine-nvfp4.md)
    "decode_kernel<128>/ragged": {"bytes": 4127827748, "source_sha": "352c1ba17c15bf38"},
    # speculative decode B8 Hq32 Hkv8 Sq4 Skv8192 D128, causal (decode_kernel<128, 1, 1>): read 268,839,424 +
    # written 2,847,232 bytes (profiles/decode_kernel_decode-B8-H32-Skv4096-D128.md)
    "decode_kernel<128>/speculative": {"bytes": 271686656, "source_sha": "352c1ba17c15bf38"},
    # wide-head B32 Hq128 Hkv1 Skv16384 D512, independent CTAs: read 1,081,726,464 + written 10,248,960
    # bytes (profiles/wide_kernel_wide-head-B32-Hq128-Hkv1-Skv16384-D512.md)
    "wide_kernel<independent>": {"bytes": 1091975424, "source_sha": "78a9a91c90649bc2"},
    # same workload, CTA-pair MMA: read 1,081,783,808 + written 10,341,632 bytes (same file)
    "wide_kernel<pair>": {"bytes": 1092125440, "source_sha": "78a9a91c90649bc2"},
}


# ------------------------------------------------------------------------------------------------
# clocks during the timed region (NVML through ctypes; read-only)
# ------------------------------------------------------------------------------------------------
class ClockSampler:
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown", 0x2: "applications_clocks"}

    def __init__(self, device_index: int = 0, period_s: float = 0.0002):
        self.ok = False
        self.samples = []
        self.period = period_s
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                return
            self.dev = ctypes.c_void_p()
            bus = None
            try:
                import torch
                pr = torch.cuda.get_device_properties(device_index)
                bus = f"{pr.pci_domain_id:08x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0".encode()
            except Exception:
                pass
            rc = self.nvml.nvmlDeviceGetHandleByPciBusId_v2(bus, ctypes.byref(self.dev)) if bus else 1
            if rc != 0 and self.nvml.nvmlDeviceGetHandleByIndex_v2(device_index, ctypes.byref(self.dev)) != 0:
                return
            mx = ctypes.c_uint()
            self.nvml.nvmlDeviceGetMaxClockInfo(self.dev, 1, ctypes.byref(mx))
            self.max_mhz = mx.value
            self.ok = True
        except OSError:
            pass

    def _sample(self):
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        self.nvml.nvmlDeviceGetClockInfo(self.dev, 1, ctypes.byref(clk))
        if self.nvml.nvmlDeviceGetCurrentClocksEventReasons(self.dev, ctypes.byref(rs)) != 0:
            self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons(self.dev, ctypes.byref(rs))
        self.samples.append((clk.value, rs.value))

    def _run(self):
        while not self._stop.is_set():
            self._sample()
            time.sleep(self.period)

    def start(self):
        if not self.ok:
            return
        self._stop = threading.Event()
        self._t = threading.Thread(target=self._run, daemon=True)
        self._t.start()

    def stop(self):
        if not self.ok:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvml unavailable"], "samples": 0}
        self._sample()          # one more at the end of the timed region
        self._stop.set()
        self._t.join()
        mhz = [s[0] for s in self.samples]
        bits = 0
        for s in self.samples:
            bits |= s[1]
        reasons = [n for b, n in self.REASONS.items() if bits & b]
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(mhz)}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


# headers every kernel file includes: a change there changes the kernels too
KERNEL_HEADERS = ("internal.h", "ptx.cuh", "nvfp4_dev.cuh")


def source_sha(name: str) -> str:
    """sha256 (first 16 hex digits) of a kernel file followed by the shared device headers."""
    h = hashlib.sha256()
    for f in (name,) + KERNEL_HEADERS:
        h.update(open(os.path.join(ROOT, "attention_tensor_cores_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def traffic_for(kernel: str, src: str, launches_per_step: int = 1):
    t = TRAFFIC.get(kernel)
    if not t or t.get("source_sha") != source_sha(src):
        return None
    return t["bytes"]


def causal_flops(w) -> int:
    """FLOPs of the two contractions under the bottom-right causal mask: query i of Sq sees
    min(n, max(0, i + n - Sq + 1)) of a sequence's n keys, 4 * D FLOPs per (query, key) pair."""
    import numpy as np
    sl = w.seqlens()
    ns = [w.Skv] * w.B if sl is None else [int(x) for x in sl]
    i = np.arange(w.Sq, dtype=np.int64)
    pairs = sum(int(np.clip(i + n - w.Sq + 1, 0, n).sum()) for n in ns)
    return 4 * w.D * w.Hq * pairs


def d128_prefill_workload():
    """The prefill workload at head dimension 128 (an extra line): B4 H16 Sq=Skv=8192 D128, N(0,1),
    non-causal, BF16 out (seed 1007)."""
    from attention_tensor_cores_gb300 import inputs
    return inputs.Workload("prefill B4 H16 Sq8192 Skv8192 D128 (non-causal, BF16 out)", 4, 16, 16, 8192, 8192,
                           128, 1.0, "bf16", 1007)


def chunked_prefill_workload():
    """Chunked prefill over a ragged KV cache: 1024 new causal query tokens per sequence, key
    lengths drawn from U{1..8192} (seed 1008), B8 Hq=Hkv=16 D128, BF16 out (an extra line)."""
    from attention_tensor_cores_gb300 import inputs
    return inputs.Workload("chunked prefill B8 H16 Sq1024 Skv<=8192 D128 (ragged, causal, BF16 out)",
                           8, 16, 16, 1024, 8192, 128, 1.0, "bf16", 1008, ragged=True)


def spec_decode_workload():
    """Decode with 4 new tokens per head under the causal mask (speculative or chunked decode):
    B8 Hq32 Hkv8 Sq4 Skv8192 D128, 16 query rows per key/value head, BF16 out (an extra line, not one
    of the five specified configurations)."""
    from attention_tensor_cores_gb300 import inputs
    return inputs.Workload("speculative decode B8 Hq32 Hkv8 Sq4 Skv8192 D128 (causal, BF16 out)",
                           8, 32, 8, 4, 8192, 128, 1.0, "bf16", 1006)


def ragged_nvfp4_small_workload():
    """A quarter of the ragged GQA NVFP4 workload (B16 instead of B64, same heads, key lengths from
    U{1..32768}, seed 1004): small enough for a multi-pass profiler capture (about 2 GiB of K/V)."""
    from attention_tensor_cores_gb300 import inputs
    return inputs.Workload("ragged GQA decode B16 Hq32 Hkv8 Sq1 Skv<=32768 D128 (NVFP4 out)", 16, 32, 8, 1, 32768,
                           128, 1.0, "nvfp4", 1004, ragged=True)


# ------------------------------------------------------------------------------------------------
# one workload on the GPU
# ------------------------------------------------------------------------------------------------
class Case:
    """Device inputs/outputs of one workload and the library call that processes them."""

    def __init__(self, F, w, num_splits=0, pad_fill=None, causal=False, wide_variant=0):
        import torch
        self.F, self.w = F, w
        self.causal = causal
        self.wv = wide_variant
        self.q, self.k, self.v, self.sl = w.make("cuda", pad_fill=pad_fill)
        B, Hq, Sq, D = self.q.shape
        self.n_out = B * Hq * Sq * D
        kind = {"bf16": F.FMHA_OUT_BF16, "f32": F.FMHA_OUT_F32, "nvfp4": F.FMHA_OUT_NVFP4}[w.out_kind]
        self.scales = self.ts = None
        if w.out_kind == "nvfp4":
            self.out = torch.empty(self.n_out // 2, dtype=torch.uint8, device="cuda")
            self.scales = torch.empty(self.n_out // 16, dtype=torch.uint8, device="cuda")
            self.ts = torch.empty(1, dtype=torch.float32, device="cuda")
        else:
            dt = torch.bfloat16 if w.out_kind == "bf16" else torch.float32
            self.out = torch.empty(B, Hq, Sq, D, dtype=dt, device="cuda")
        self.lse = torch.empty(B, Hq, Sq, dtype=torch.float32, device="cuda")
        opts = F.make_opts(kind, self.sl, num_splits, None, self.scales, self.ts, None, causal, wide_variant=self.wv)
        wsb = F.fmha_workspace_size(B, Hq, w.Hkv, Sq, w.Skv, D, opts)
        self.ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device="cuda") if wsb else None
        self.opts = F.make_opts(kind, self.sl, num_splits, self.ws, self.scales, self.ts, None, causal,
                                wide_variant=self.wv)
        self.kind, self.num_splits = kind, num_splits

    def use_given_scale(self, sg: float):
        """Single-pass NVFP4 from here on: the epilogues encode with this per-tensor scale."""
        import torch
        F, w = self.F, self.w
        B, Hq, Sq, D = self.q.shape
        self.sg_in = torch.tensor([sg], dtype=torch.float32, device="cuda")
        opts = F.make_opts(self.kind, self.sl, self.num_splits, None, self.scales, self.ts, None, self.causal, self.sg_in,
                           wide_variant=self.wv)
        wsb = F.fmha_workspace_size(B, Hq, w.Hkv, Sq, w.Skv, D, opts)
        self.ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device="cuda") if wsb else None
        self.opts = F.make_opts(self.kind, self.sl, self.num_splits, self.ws, self.scales, self.ts, None, self.causal,
                                self.sg_in, wide_variant=self.wv)

    def call(self, q=None, k=None, v=None):
        self.F.fmha_fwd_ex(self.q if q is None else q, self.k if k is None else k, self.v if v is None else v,
                           self.out, self.lse, self.w.scale, self.opts)

    def algorithmic_bytes(self) -> int:
        """K/V rows actually read, plus Q, O and LSE."""
        w = self.w
        o_bytes = {"bf16": 2, "f32": 4, "nvfp4": 0.5 + 1 / 16}[w.out_kind] * self.n_out
        return int(w.kv_bytes() + self.q.numel() * 2 + o_bytes + self.lse.numel() * 4)


# The dominant kernel is timed with CUDA events on one timed call in KERNEL_EVENT_EVERY (the first,
# then every KERNEL_EVENT_EVERY-th).  An event pair around a launch holds the stream between kernels
# (decode B8 H32: 90.1 us per call with a pair around every call, 86.7 with one call in four, 85.3
# with none), so timing every call would slow the step time that `value` is computed from.
KERNEL_EVENT_EVERY = 4


def time_case(F, case, steps, warmup, sampler=None, dist=None):
    import torch
    for _ in range(warmup):
        case.call()
    torch.cuda.synchronize()
    region = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    kev = {i: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for i in range(0, steps, KERNEL_EVENT_EVERY)}
    for a, b in kev.values():   # creates the event handles the library records
        a.record()
        b.record()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    l0 = F.fmha_launch_count()
    if sampler:
        sampler.start()
    # the region's own events bracket the K calls; inside it only the dominant kernel's events (the
    # library records them around that launch, on the sampled calls) are added, for the roofline's
    # kernel duration
    region[0].record()
    for i in range(steps):
        if i in kev:
            F.fmha_time_next_call(kev[i][0], kev[i][1])
        case.call()
    region[1].record()
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    if dist is not None:
        dist.barrier()
    launches = F.fmha_launch_count() - l0
    assert F.fmha_check_status() == 0, "device status word set during the benchmark"
    return {
        "region_ms": region[0].elapsed_time(region[1]),
        "kernel_ms": [a.elapsed_time(b) for a, b in kev.values()],
        "launches": launches,
        "clocks": clocks,
    }


def time_e2e(F, case, steps, warmup):
    """The same call from pinned host buffers through the C ABI's fmha_fwd_host: per step the
    host->device copies of Q, K and V, the attention and the device->host copies of O and the LSE
    (the library overlaps one batch chunk's copies with the previous chunk's attention)."""
    import torch
    qh = case.q.cpu().pin_memory()
    kh = case.k.cpu().pin_memory()
    vh = case.v.cpu().pin_memory()
    outh = torch.empty(case.out.shape, dtype=case.out.dtype, pin_memory=True)
    lseh = torch.empty(case.lse.shape, dtype=case.lse.dtype, pin_memory=True)
    B, Hq, Sq, D = case.q.shape
    opts = F.make_opts(case.kind, causal=case.causal)
    buf = torch.empty(F.fmha_host_buffer_size(B, Hq, case.w.Hkv, Sq, case.w.Skv, D, opts), dtype=torch.uint8,
                      device="cuda")

    def step():
        F.fmha_fwd_host(qh, kh, vh, outh, lseh, case.w.scale, buf, opts)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        step()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    h2d = (qh.numel() + kh.numel() + vh.numel()) * 2
    d2h = outh.numel() * outh.element_size() + lseh.numel() * 4
    del qh, kh, vh, buf
    return ms, h2d, d2h


# ------------------------------------------------------------------------------------------------
# CPU oracle baseline
# ------------------------------------------------------------------------------------------------
def oracle_sample(w, rows_per_step: int, step: int):
    """Inputs for a bounded sample of `w`: `rows_per_step` consecutive query rows (whole heads),
    regenerated on the CPU.  Returns (callable, algorithmic K/V bytes, FLOPs, description)."""
    import numpy as np
    import oracle
    total = w.B * w.Hq * w.Sq
    r0 = (step * rows_per_step) % total
    rows = np.arange(r0, min(total, r0 + rows_per_step), dtype=np.int64)
    sl = w.seqlens()
    g = w.Hq // w.Hkv
    groups = {}
    for r in rows:
        b = int(r // (w.Hq * w.Sq))
        hq = int((r // w.Sq) % w.Hq)
        groups.setdefault((b, hq // g), []).append(int(r))
    jobs = []
    kv_bytes = flops = 0
    for (b, kvh), rr in groups.items():
        n = w.Skv if sl is None else int(sl[b])
        kk, vv = w.kv_head_np(b, kvh, n)
        qq = w.q_rows_np(rr)
        jobs.append((qq.reshape(1, 1, len(rr), w.D), kk.reshape(1, 1, n, w.D), vv.reshape(1, 1, n, w.D)))
        kv_bytes += 2 * n * w.D * 2 * len(rr) / (g * w.Sq)   # each K/V head counted once per group
        flops += 4 * n * w.D * len(rr)

    def run():
        for qq, kk, vv in jobs:
            oracle.attention(qq, kk, vv, w.scale)

    return run, kv_bytes, flops, f"{len(rows)} query rows from row {r0}"


def cpu_baseline(w, metric_unit: str, budget_s: float = 6.0, rows_per_step: int = 64):
    """The oracle as it stands, timed on this host's cores on a bounded sample of workload `w`:
    `rows_per_step` consecutive query rows (the whole workload when it has fewer), repeated until
    `budget_s` of CPU time.  metric_unit: "GB/s" (K/V bytes of the sample's heads), "TFLOP/s"
    (its 4*D FLOPs per query-key pair) or "us" (time per pass over the whole workload)."""
    import oracle
    rows = min(rows_per_step, w.B * w.Hq * w.Sq)
    run, kvb, fl, desc = oracle_sample(w, rows, 0)
    run()   # builds/loads the library, touches memory
    t0 = time.perf_counter()
    reps = 0
    while True:
        run()
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= 200:
            break
    per = el / reps
    val = {"GB/s": lambda: kvb / per / 1e9, "TFLOP/s": lambda: fl / per / 1e12, "us": lambda: per * 1e6}[metric_unit]()
    return {"value": val, "unit": metric_unit, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{desc} of {w.name}, {reps} repetitions, {per * 1e3:.2f} ms each"}


# ------------------------------------------------------------------------------------------------
# arms
# ------------------------------------------------------------------------------------------------
def _max_over_ranks(x: float, dist, device="cuda"):
    """Largest value of x over all ranks (the timed region is the slowest rank's)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(units_per_rank_per_step: float, steps: int, world: int, region_ms_max: float) -> float:
    """Whole-job throughput: the units every rank processed over the slowest rank's timed region
    (replicas: each rank runs the same workload on its own GPU)."""
    return world * steps * units_per_rank_per_step / (region_ms_max / 1e3)


def read_only_peak_gbs(gib: float = 4.0, reps: int = 10) -> float:
    """A read-only stream rate for the KV-bound rows: torch.sum over `gib` GiB of FP32 (one pass,
    nothing written back but the scalar), best of `reps`, CUDA events.  The decode kernels mostly
    read, so they can exceed a copy benchmark (read + write) figure; this probe says by how much."""
    import torch
    n = int(gib * 2 ** 30) // 4
    x = torch.ones(n, dtype=torch.float32, device="cuda")
    best = float("inf")
    for _ in range(reps + 2):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        x.sum()
        b.record()
        torch.cuda.synchronize()
        best = min(best, a.elapsed_time(b))
    del x
    torch.cuda.empty_cache()
    return n * 4 / (best / 1e3) / 1e9


def hbm_roofline(achieved: float, peaks: dict, read_peak: float | None) -> dict:
    """HBM roofline entry against the measured copy bandwidth, with the read-only probe beside it;
    a fraction above 1 of the copy figure is flagged (read-mostly traffic, not a timing error, as
    long as the read-only fraction stays at or below 1)."""
    r = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
         "frac": achieved / peaks["hbm_gbs"]}
    if read_peak:
        r["read_only_peak"] = read_peak
        r["frac_of_read_only"] = achieved / read_peak
    if r["frac"] > 1.0:
        r["flag"] = "above the copy-bandwidth peak: the kernel reads far more than it writes"
    return r


def l2_note(in_bytes: int) -> str:
    """How the timed steps avoid measuring from a warm L2: inputs larger than L2, else say it fits."""
    import torch
    l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
    if in_bytes > l2:
        return f"inputs larger than L2 ({in_bytes / 2**20:.0f} MiB of Q/K/V per step, L2 {l2 / 2**20:.1f} MiB): no flush"
    return f"inputs fit in L2 ({in_bytes / 2**10:.0f} KiB, L2 {l2 / 2**20:.1f} MiB): latency figure, no roofline claim"


def _workload_entry(F, w, idx, steps, warmup, peaks, causal=False, given_scale=False, read_peak=None, cpu=False,
                    wide_variant=0):
    """Timing + roofline of one extra workload (rank 0 only).  given_scale: NVFP4 in one pass with the
    per-tensor scale of an earlier (two-pass) call on the same inputs, as a caller reusing the
    previous step's scale would.  cpu: also time the oracle on a bounded sample of it."""
    import torch
    case = Case(F, w, num_splits=0, causal=causal, wide_variant=wide_variant)
    if given_scale:
        case.call()
        torch.cuda.synchronize()
        case.use_given_scale(float(case.ts.cpu()[0]))
    r = time_case(F, case, steps, warmup)
    step_ms = r["region_ms"] / steps
    kern_ms = statistics.mean(r["kernel_ms"])
    e = {"workload": w.name, "ms_per_step": step_ms, "kernel_ms": kern_ms, "gpu_launches_per_step": r["launches"] / steps,
         "l2": l2_note(w.kv_bytes() + case.q.numel() * 2)}
    unit = "us"
    if idx == 2:   # prefill: tensor-bound
        flops = causal_flops(w) if causal else w.flops()
        tf = flops / (step_ms / 1e3) / 1e12
        ach = flops / (kern_ms / 1e3) / 1e12
        e["flops"] = flops
        e.update({"value": tf, "unit": "TFLOP/s",
                  "roofline": {"bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                               "frac": ach / peaks["bf16_tflops"], "traffic": None}})
        unit = "TFLOP/s"
    elif idx == 0:
        e.update({"value": step_ms * 1e3, "unit": "us", "note": "latency-bound, fits in L2: no roofline claim"})
    else:
        gbs = w.kv_bytes() / (step_ms / 1e3) / 1e9
        ach = case.algorithmic_bytes() / (kern_ms / 1e3) / 1e9
        if w.D == 512:
            traffic = traffic_for("wide_kernel<pair>" if wide_variant == 2 else "wide_kernel<independent>", "wide.cu")
        elif w.ragged and not causal and not given_scale:
            traffic = traffic_for("decode_kernel<128>/ragged", "decode.cu")
        elif causal and w.Sq == 4 and w.Skv == 8192 and w.B == 8:
            traffic = traffic_for("decode_kernel<128>/speculative", "decode.cu")
        else:
            traffic = None
        roof = hbm_roofline(ach, peaks, read_peak)
        roof["traffic"] = traffic
        e.update({"value": gbs, "unit": "GB/s", "kv_bytes": w.kv_bytes(), "flops": w.flops(),
                  "tflops": w.flops() / (step_ms / 1e3) / 1e12, "roofline": roof})
        unit = "GB/s"
    del case
    torch.cuda.empty_cache()
    if cpu:
        e["cpu_baseline"] = cpu_baseline(w, unit)
    return e


def _summary(head: dict, extra: dict) -> dict:
    """Compact per-configuration figures (step value, dominant kernel's roofline fraction, the
    oracle's rate on this host) printed last on the line, so that a reader of its tail sees all five."""
    def r4(x):
        return None if x is None else float(f"{x:.4g}")

    out = {"c2": {"value": r4(head["value"]), "unit": "GB/s", "ms": r4(head["ms_per_step"]),
                  "kernel_frac": r4(head["roofline"]["frac"]),
                  "cpu": r4(head["cpu"]["value"]) if head.get("cpu") else None}}
    for key in ("c1", "c3", "c4", "c5", "c4_pair", "c5_given_scale", "c2_spec_causal", "c3_d128", "c3_causal",
                "c3_chunked_varlen"):
        e = extra.get(key)
        if not e or "value" not in e:
            continue
        d = {"value": r4(e["value"]), "unit": e["unit"], "ms": r4(e["ms_per_step"])}
        if "roofline" in e:
            d["kernel_frac"] = r4(e["roofline"]["frac"])
        if "cpu_baseline" in e:
            d["cpu"] = r4(e["cpu_baseline"]["value"])
        out[key] = d
    return out


def run_ours(args, rank, world, local):
    import torch
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as td
        td.init_process_group("nccl", device_id=torch.device("cuda", local))
        dist = td
    import __graft_entry__ as ge
    if rank == 0:
        ge.build()
    if dist is not None:
        dist.barrier()
        if rank != 0:
            ge.build()
    import attention_tensor_cores_gb300 as F
    from attention_tensor_cores_gb300 import inputs
    F.load()
    peaks, peaks_src = load_peaks()
    read_peak = read_only_peak_gbs() if rank == 0 else None
    wl = inputs.workloads()
    w = wl[1]
    head = Case(F, w, num_splits=0)
    sampler = ClockSampler(local)
    r = time_case(F, head, args.steps, args.warmup, sampler, dist)
    region_ms = _max_over_ranks(r["region_ms"], dist)
    step_ms = region_ms / args.steps
    value = aggregate_rate(w.kv_bytes(), args.steps, world, region_ms) / 1e9
    kern_ms = statistics.mean(r["kernel_ms"])
    achieved = head.algorithmic_bytes() / (kern_ms / 1e3) / 1e9
    roof = hbm_roofline(achieved, peaks, read_peak)
    roof.update({"traffic": traffic_for("decode_kernel<128>", "decode.cu"),
                 "kernel": "decode_kernel<128>", "kernel_ms": kern_ms, "algorithmic_bytes": head.algorithmic_bytes(),
                 "kernel_events": f"CUDA events around {len(r['kernel_ms'])} of the {args.steps} timed calls "
                                  f"(one in {KERNEL_EVENT_EVERY})",
                 "peak_source": f"{peaks_src} HBM copy bandwidth (burst); read_only_peak: torch.sum over 4 GiB in this run"})
    e2e_ms, h2d, d2h = time_e2e(F, head, args.steps, min(args.warmup, 3))
    e2e_ms = _max_over_ranks(e2e_ms, dist)
    e2e = {"value": world * w.kv_bytes() / (e2e_ms / 1e3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}
    head_l2 = l2_note(w.kv_bytes() + head.q.numel() * 2)
    del head
    torch.cuda.empty_cache()
    extra = {}
    if rank == 0 and not args.only_headline:
        for idx in (0, 2, 3, 4):
            try:
                extra[f"c{idx + 1}"] = _workload_entry(F, wl[idx], idx, min(args.steps, 10), args.warmup, peaks,
                                                       read_peak=read_peak, cpu=(world == 1 and not args.no_cpu))
            except F.FmhaError as ex:
                extra[f"c{idx + 1}"] = {"workload": wl[idx].name, "unsupported": str(ex)}
        try:   # the ragged NVFP4 workload in one pass, with a given per-tensor scale
            extra["c5_given_scale"] = _workload_entry(F, wl[4], 4, min(args.steps, 10), args.warmup, peaks, given_scale=True, read_peak=read_peak)
            extra["c5_given_scale"]["workload"] = wl[4].name.replace("(NVFP4 out)", "(NVFP4 out, one pass with a given scale)")
        except F.FmhaError as ex:
            extra["c5_given_scale"] = {"workload": "ragged NVFP4, given scale", "unsupported": str(ex)}
        try:   # the wide-head workload on the CTA-pair MMA kernel (tcgen05 cta_group::2)
            extra["c4_pair"] = _workload_entry(F, wl[3], 3, min(args.steps, 10), args.warmup, peaks,
                                               read_peak=read_peak, wide_variant=F.FMHA_WIDE_PAIR)
            extra["c4_pair"]["workload"] = wl[3].name.replace("(BF16 out)", "(BF16 out, CTA-pair MMA)")
        except F.FmhaError as ex:
            extra["c4_pair"] = {"workload": "wide-head, CTA-pair MMA", "unsupported": str(ex)}
        try:   # decode with several new tokens per head (speculative or chunked decode), causal mask
            extra["c2_spec_causal"] = _workload_entry(F, spec_decode_workload(), 1, min(args.steps, 10), args.warmup, peaks, causal=True, read_peak=read_peak)
        except F.FmhaError as ex:
            extra["c2_spec_causal"] = {"workload": "speculative decode", "unsupported": str(ex)}
        try:   # the prefill workload at head dim 128
            extra["c3_d128"] = _workload_entry(F, d128_prefill_workload(), 2, min(args.steps, 10), args.warmup, peaks)
        except F.FmhaError as ex:
            extra["c3_d128"] = {"workload": "prefill D128", "unsupported": str(ex)}
        try:   # chunked prefill: ragged key lengths, causal, work items from the workspace counter
            extra["c3_chunked_varlen"] = _workload_entry(F, chunked_prefill_workload(), 2, min(args.steps, 10), args.warmup,
                                                         peaks, causal=True)
        except F.FmhaError as ex:
            extra["c3_chunked_varlen"] = {"workload": "chunked prefill", "unsupported": str(ex)}
        try:   # the prefill workload with the causal mask
            extra["c3_causal"] = _workload_entry(F, wl[2], 2, min(args.steps, 10), args.warmup, peaks, causal=True)
            extra["c3_causal"]["workload"] = wl[2].name.replace("non-causal", "causal")
        except F.FmhaError as ex:
            extra["c3_causal"] = {"workload": "causal prefill", "unsupported": str(ex)}
    cpu = cpu_baseline(w, "GB/s") if (rank == 0 and world == 1 and not args.no_cpu) else None
    if dist is not None:
        dist.barrier()
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name + ", + FP32 LSE", "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Sq": w.Sq,
                   "Skv": w.Skv, "D": w.D, "kv_bytes_per_step": w.kv_bytes(),
                   "l2": head_l2,
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": r["launches"],
        "clocks": r["clocks"], "workloads": extra,
    }
    line["summary"] = _summary({"value": value, "ms_per_step": step_ms, "roofline": roof, "cpu": cpu}, extra)
    print(json.dumps(line), flush=True)


def run_reference(args, rank, world):
    """The CPU FP64 oracle on the headline workload, bounded samples (whole heads) per step."""
    if rank != 0:
        return
    import oracle
    from attention_tensor_cores_gb300 import inputs
    oracle.build()
    w = inputs.workloads()[1]
    rows_per_step = 32
    cache = {}

    def sample(i):
        key = i % 8
        if key not in cache:
            cache[key] = oracle_sample(w, rows_per_step, key)
        return cache[key]

    for i in range(args.warmup):
        sample(i)[0]()
    times, kvb = [], 0.0
    for i in range(args.steps):
        run, b, _, _ = sample(args.warmup + i)
        t0 = time.perf_counter()
        run()
        times.append(time.perf_counter() - t0)
        kvb += b
    tot = sum(times)
    val = kvb / tot / 1e9
    desc = f"{rows_per_step} query rows (one batch entry, all heads) of {w.name} per step"
    line = {
        "metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": tot / args.steps * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": {"workload": w.name + ", + FP32 LSE", "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Sq": w.Sq, "Skv": w.Skv,
                   "D": w.D, "parallelism": "host cores (OpenMP)"},
        "cpu_baseline": {"value": val, "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle", "sample": desc},
        "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--only-headline", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle's CPU baselines")
    ap.add_argument("--profile", choices=["c1", "c2", "c3", "c4", "c5", "c3_causal", "c3_d128", "c5_given_scale", "c2_spec_causal",
                                          "c5_small", "c4_pair", "nvfp4"], default=None,
                    help="run one workload's call --repeat times, untimed (for a profiler)")
    ap.add_argument("--repeat", type=int, default=5)
    args = ap.parse_args()
    if args.profile:
        import torch
        import __graft_entry__ as ge
        ge.build()
        import attention_tensor_cores_gb300 as F
        from attention_tensor_cores_gb300 import inputs
        if args.profile == "nvfp4":   # the standalone two-pass quantiser on 64 Mi FP32 values (256 MiB)
            n = 1 << 26
            x = torch.randn(n, generator=torch.Generator().manual_seed(7)).cuda()
            qq = torch.empty(n // 2, dtype=torch.uint8, device="cuda")
            sc = torch.empty(F.nvfp4_scales_bytes(n), dtype=torch.uint8, device="cuda")
            for _ in range(args.repeat):
                F.nvfp4_quantize(x, qq, sc)
            torch.cuda.synchronize()
            assert F.fmha_check_status() == 0
            print(f"profile run of nvfp4_quantize on {n} values: {args.repeat} calls ok")
            return
        if args.profile == "c2_spec_causal":
            w = spec_decode_workload()
        elif args.profile == "c3_d128":
            w = d128_prefill_workload()
        elif args.profile == "c5_small":
            w = ragged_nvfp4_small_workload()
        else:
            w = inputs.workloads()[int(args.profile[1]) - 1]
        case = Case(F, w, num_splits=0, causal=args.profile in ("c3_causal", "c2_spec_causal"),
                    wide_variant=F.FMHA_WIDE_PAIR if args.profile == "c4_pair" else F.FMHA_WIDE_AUTO)
        if args.profile == "c5_given_scale":   # one two-pass call gives the scale the rest reuse
            case.call()
            torch.cuda.synchronize()
            case.use_given_scale(float(case.ts.cpu()[0]))
        for _ in range(args.repeat):
            case.call()
        torch.cuda.synchronize()
        assert F.fmha_check_status() == 0
        print(f"profile run of {case.w.name} ({args.profile}): {args.repeat} calls ok")
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
