"""Benchmark of the attention hot path on GB300.

Default step: one sdpa_forward over the long-context causal workload
(B1, L32768, H32, d128, bf16, causal, 4 outlier dims per head scaled x8 in
Q and K): rows a3-a7 of the path (QK^T, scale + mask, online softmax, P V,
epilogue) in one fused kernel launch.  `value` is that workload's SDPA
forward throughput in TFLOP/s (algorithmic flops: 4*d per unmasked
query/key pair, 2*B*H*d*L*(L+1) for causal), summed over all ranks.

Extra legs in the same JSON line:
  e2e          the same metric through the public call with host (pinned)
               buffers (sdpa_forward_host, which overlaps the copies with the
               attention chunk by chunk): H2D of Q/K/V and D2H of O inside the
               timed region
  roofline     the fused kernel against the measured bf16 tensor peak
  workloads    the other workloads, each with its own roofline: the
               key-padding encoder, decoder causal and cross-attention
               attention workloads (median of per-step CUDA events, L2
               flushed before each step unless the inputs exceed L2), and the
               base-shape fp32 layer in tokens/s with the oracle's layer on
               the host beside it (all threads and one thread)
  mha_layer    the whole layer (rows a1-a8: projections with head-split
               stores, attention with the concat store, output projection)
               in tokens/s, on the same shape (D = 4096, h = 32) and on the
               base fp32 shape (B1 L128 D512 h8)
  encoder_layer one post-norm encoder layer (attention with biases,
               residual + LayerNorm, ReLU FFN d_ff = 4D, residual +
               LayerNorm) in tokens/s, on the key-padding encoder shape
               (B32 L512 D512 h8, bf16) and the base fp32 shape (B1 L128)
  embed_pe     the first layer's input (embedding x sqrt(D) + positional
               encoding, one pass) in GB/s on the encoder shape with the
               pages' 37000-token vocabulary, and tokens/s of that pass plus
               one encoder layer
  decode       sdpa_decode (Lq new queries against a bf16 key/value cache,
               bottom-right causal) on the three decode workloads, in GB/s
               of cache streamed against the measured HBM peak
  backward     sdpa_backward (dQ, dK, dV) on the long-context and decoder
               causal shapes, in TFLOP/s (2.5x the forward's flops)
  cpu_baseline the fp64 oracle on this host's cores on a bounded row sample
               (the same sample every step of the reference arm times), with
               the full-output time extrapolated from it

Multi-GPU: the path has no exchange step, so N ranks run N replicas (one per
GPU, weak scaling); the time is the max over ranks after a barrier.

`--workload 1` makes the base-shape multi-head attention layer (B1 L128 D512
h8, fp32: rows a1-a8 through mha_forward) the step instead, in tokens/s; its
roofline is the fp32 FMA rate of the CUDA cores.

`--impl reference` times the CPU oracle (the reference arm of this build) on
the same workload, metric and unit.
"""
from __future__ import annotations

import argparse
import json
import math
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

METRIC = "SDPA fwd TFLOP/s and % of GB300 BF16 tensor peak; MHA layer tokens/s"
NOMINAL_BF16_TFLOPS = 2250.0
NOMINAL_HBM_GBS = 8000.0
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 1024 * 1024


# ------------------------------------------------------------ host helpers

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK}, "measured"
    except Exception:
        return dict(FALLBACK), "fallback"


def recorded_traffic(kernel_files, profile):
    """DRAM bytes per launch recorded in a committed profile summary, or None
    when the kernel sources changed since the capture (hash mismatch)."""
    import hashlib
    import re
    h = hashlib.sha256()
    try:
        for f in kernel_files:
            with open(os.path.join(ROOT, f), "rb") as fh:
                h.update(fh.read())
        with open(os.path.join(ROOT, profile)) as fh:
            text = fh.read()
    except OSError:
        return None
    m_hash = re.search(r"kernel_source_sha256:\s*([0-9a-f]{64})", text)
    m_bytes = re.search(r"dram_bytes_per_launch:\s*(\d+)", text)
    if not (m_hash and m_bytes) or m_hash.group(1) != h.hexdigest():
        return None
    return int(m_bytes.group(1))


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def whole_job_value(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Throughput of the whole job: the units all ranks processed over the
    slowest rank's time."""
    return units_per_rank * world / max_seconds


def max_over_ranks(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


class ClockSampler:
    """SM clock and clock-event reasons while active: every 2 ms through the
    driver's NVML library (read-only queries), so that timed regions of a
    few milliseconds are covered too; nvidia-smi's 20 ms loop when NVML
    cannot be loaded.  Only samples taken after entering count."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # NVML clock-event reason bits (nvml.h)
    NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                    0x40: "hw_thermal_slowdown"}

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self._t = None
        self._start = 0
        self._nvml = None
        self._stop = threading.Event()
        self.samples = []   # (sm_mhz, max_mhz, reasons bitmask) from NVML

    def _open_nvml(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            return None
        handle = ctypes.c_void_p()
        ok = False
        try:
            import torch
            uid = getattr(torch.cuda.get_device_properties(self.gpu), "uuid", None)
            if uid is not None:
                ok = lib.nvmlDeviceGetHandleByUUID(f"GPU-{uid}".encode(),
                                                   ctypes.byref(handle)) == 0
        except Exception:
            ok = False
        if not ok:
            return None
        reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        return lib, handle, reasons

    def _poll_nvml(self):
        import ctypes
        lib, handle, reasons = self._nvml
        clk, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            if (lib.nvmlDeviceGetClockInfo(handle, 1, ctypes.byref(clk)) == 0 and
                    lib.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx)) == 0 and
                    reasons(handle, ctypes.byref(rs)) == 0):
                self.samples.append((clk.value, mx.value, rs.value))
            time.sleep(0.002)

    def __enter__(self):
        try:
            self._nvml = self._open_nvml()
        except Exception:
            self._nvml = None
        if self._nvml is not None:
            self._t = threading.Thread(target=self._poll_nvml, daemon=True)
            self._t.start()
            t0 = time.perf_counter()
            while not self.samples and time.perf_counter() - t0 < 1.0:
                time.sleep(0.001)
            self._start = len(self.samples)
            return self
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            t0 = time.perf_counter()
            while not self.lines and time.perf_counter() - t0 < 3.0:
                time.sleep(0.005)
            self._start = len(self.lines)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self._nvml is not None:
            self._stop.set()
            if self._t is not None:
                self._t.join(timeout=2)
            return
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            if self._t is not None:
                self._t.join(timeout=2)

    def summary(self):
        if self._nvml is not None:
            got = self.samples[self._start:]
            if not got:
                return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                        "source": "nvml"}
            reasons = sorted({name for _, _, bits in got
                              for bit, name in self.NVML_REASONS.items() if bits & bit})
            return {"sm_mhz": statistics.median(c for c, _, _ in got),
                    "sm_max_mhz": max(m for _, m, _ in got), "reasons": reasons,
                    "samples": len(got), "source": "nvml, 2 ms"}
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines[self._start:]:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sms.append(float(parts[0]))
                maxes.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "source": "nvidia-smi"}
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes),
                "reasons": sorted(reasons), "samples": len(sms), "source": "nvidia-smi, 20 ms"}


# query rows per head of the oracle's sample, per attention workload: about
# 5 s of fp64 work on a 16-core host.  The CPU-baseline leg of the GPU arm
# and every step of the reference arm time this same sample.
ORACLE_ROWS_PER_HEAD = {2: 48, 3: 256, 4: 96, 5: 512}


def oracle_sample(w, per_head=None):
    """(rows, per_head): the seeded query-row sample the oracle is timed on."""
    from transformer_head_scaled_03_gb300.inputs import sample_rows
    n = min(per_head or ORACLE_ROWS_PER_HEAD.get(w.wid, 64), w.Lq)
    return sample_rows(w.B, w.H, w.Lq, n, seed=w.seed + 3000, must=()), n


def sample_description(w, rows, per_head):
    return (f"{rows.size} query rows ({per_head} per head, all {w.B * w.H} heads, seeded) "
            f"of the same workload, fp64")


def oracle_cpu_baseline(w, Q, K, V, lens, rows):
    """Time the fp64 oracle (as it stands) on a row sample; TFLOP/s."""
    import oracle
    orc = oracle.default()
    t0 = time.perf_counter()
    orc.sdpa_rows(Q, K, V, rows, mask_kind=w.mask, key_lengths=lens)
    dt = time.perf_counter() - t0
    i = rows % w.Lq
    if w.mask & 1:
        pairs = float(np.sum(i + 1))
    elif w.mask & 2:
        pairs = float(np.sum(lens[(rows // w.Lq) // w.H]))
    else:
        pairs = float(rows.size) * w.Lk
    flops = 4.0 * w.d * pairs
    return flops / dt / 1e12, dt, orc.num_threads()


def workload_from_args(args):
    """The chosen workload, optionally with a smaller sequence length or head
    count (same input recipe) for profiling captures."""
    import dataclasses
    from transformer_head_scaled_03_gb300.inputs import WORKLOADS
    w = WORKLOADS[args.workload]
    if w.kind == "decode":
        if args.batch is None:
            return w
        name = f"{w.name.split(' (')[0]} (B{args.batch} H{w.H} d{w.d}, cache {w.Lk}, reduced)"
        return dataclasses.replace(w, B=args.batch, name=name)
    if args.seq is None and args.heads is None:
        return w
    L = args.seq if args.seq is not None else w.Lq
    H = args.heads if args.heads is not None else w.H
    Lk = L if w.Lq == w.Lk else w.Lk
    name = f"{w.name.split(' (')[0]} (B{w.B} L{L} H{H} d{w.d} bf16, reduced)"
    return dataclasses.replace(w, Lq=L, Lk=Lk, H=H, name=name)


# ------------------------------------------------------------------ GPU arm

def attention_roofline(flops, alg_bytes, achieved_tflops, bf16_peak_tflops, hbm_peak_gbs,
                       peak_src):
    """The roofline object of an attention launch: the bound is whichever
    peak the workload's arithmetic intensity meets first -- tensor at or
    above the ridge (peak flop/s over peak B/s), HBM below it, where the same
    time is reported as algorithmic GB/s."""
    if flops / alg_bytes >= bf16_peak_tflops * 1e12 / (hbm_peak_gbs * 1e9):
        return {"bound": "tensor", "achieved": round(achieved_tflops, 2),
                "peak": bf16_peak_tflops, "unit": "TFLOP/s",
                "frac": round(achieved_tflops / bf16_peak_tflops, 4),
                "frac_nominal": round(achieved_tflops / NOMINAL_BF16_TFLOPS, 4),
                "peak_source": f"{peak_src} bf16 burst"}
    gbs = alg_bytes / (flops / (achieved_tflops * 1e12)) / 1e9
    return {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_peak_gbs, "unit": "GB/s",
            "frac": round(gbs / hbm_peak_gbs, 4),
            "frac_nominal": round(gbs / NOMINAL_HBM_GBS, 4),
            "peak_source": f"{peak_src} HBM copy"}


MASK_NAMES = {0: "none", 1: "causal", 2: "key_padding", 3: "causal+key_padding"}


def sdpa_l2_note(w) -> str:
    """How the timed steps treat L2 for workload w: its inputs and output
    (bf16) larger than two L2s stream from HBM anyway; smaller ones get a
    256 MB write between steps."""
    nbytes = 2 * w.H * w.d * (2 * w.B * w.Lq + 2 * w.B * w.Lk)
    return "inputs larger than L2" if nbytes >= 2 * L2_BYTES else "L2 flushed between steps"


def sdpa_config(w, lens, world, float_mask=False):
    """The `config` object of an attention workload's JSON line (both arms)."""
    return {"workload": w.name, "B": w.B, "H": w.H, "Lq": w.Lq, "Lk": w.Lk, "d": w.d,
            "mask": MASK_NAMES[w.mask] + (" (as additive float mask [Lq, Lk])" if float_mask
                                          else ""),
            "flops_per_step": w.flops(lens), "l2": sdpa_l2_note(w),
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def fwd_kernel_name(w):
    """The forward instantiation sdpa_forward picks for workload w:
    <head dim, query tiles per CTA, K/V stages, keys per tile>."""
    if w.d == 128:
        return f"sdpa_fwd_bf16_kernel<128,{2 if w.Lq > 128 else 1},2,128>"
    if w.Lq > 128:
        return "sdpa_fwd_bf16_kernel<64,2,3,64>"
    return f"sdpa_fwd_bf16_kernel<64,1,{2 if w.Lk <= 2048 else 3},128>"


def bench_sdpa(args, w, rank, world, local_rank):
    import torch
    import transformer_head_scaled_03_gb300 as mha
    from transformer_head_scaled_03_gb300.inputs import sample_rows, sdpa_inputs

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    Q, K, V, lens, dims = sdpa_inputs(w)
    to_bf16 = lambda a: torch.from_numpy(a).to(torch.bfloat16)
    Qh, Kh, Vh = (to_bf16(a).pin_memory() for a in (Q, K, V))
    lens_h = torch.from_numpy(lens).pin_memory() if lens is not None else None
    Qd, Kd, Vd = (t.to(dev) for t in (Qh, Kh, Vh))
    kl = lens_h.to(dev) if lens_h is not None else None
    Od = torch.empty_like(Qd)
    flops = w.flops(lens)
    in_bytes = sum(t.numel() * t.element_size() for t in (Qd, Kd, Vd))
    out_bytes = Od.numel() * Od.element_size()
    flush = None
    if sdpa_l2_note(w) != "inputs larger than L2":
        flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

    add_mask = None
    mask_kind = w.mask
    if args.float_mask:
        # the causal mask handed over as an opaque additive float mask [Lq, Lk]
        if w.mask != 1:
            raise SystemExit("--float-mask needs a causal workload")
        add_mask = torch.triu(torch.full((w.Lq, w.Lk), float("-inf"), device=dev), 1)
        mask_kind = 0

    def step():
        mha.sdpa_forward(Qd, Kd, Vd, mask_kind=mask_kind, key_lengths=kl, out=Od,
                         add_mask=add_mask)

    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert mha.mha_check() == mha.MHA_OK
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clocks:
        if flush is None:
            # one event between consecutive steps: the per-step spread comes
            # from the same timeline as the total
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
            evs[0].record(stream)
            for i in range(args.steps):
                step()
                evs[i + 1].record(stream)
            torch.cuda.synchronize()
            total_ms = evs[0].elapsed_time(evs[-1])
            step_ms = [evs[i].elapsed_time(evs[i + 1]) for i in range(args.steps)]
        else:
            total_ms = 0.0
            step_ms = []
            for _ in range(args.steps):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                step()
                e1.record(stream)
                torch.cuda.synchronize()
                step_ms.append(e0.elapsed_time(e1))
                total_ms += step_ms[-1]
    warm_ms = None
    if flush is not None:
        # the same steps back to back, inputs left in L2 (context for the
        # cold number above, which is the one reported)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        warm_ms = e0.elapsed_time(e1) / args.steps
    barrier()
    torch.cuda.synchronize()
    st = mha.mha_check()
    if st != mha.MHA_OK:
        raise RuntimeError(f"device error during timing: {mha.status_string(st)}")
    max_s = max_over_ranks(total_ms / 1e3, dev)
    per_step = max_s / args.steps
    value = whole_job_value(flops * args.steps, world, max_s) / 1e12
    kernel_tflops = flops / (total_ms / 1e3 / args.steps) / 1e12  # this rank's kernel

    # end to end through the public call from pinned host buffers
    bufs = {}
    for _ in range(2):
        mha.sdpa_forward_host(Qh, Kh, Vh, mask_kind=w.mask, lengths_h=lens_h, bufs=bufs)
    torch.cuda.synchronize()
    barrier()
    e2e_steps = max(3, min(args.steps, 10))
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        Oh = mha.sdpa_forward_host(Qh, Kh, Vh, mask_kind=w.mask, lengths_h=lens_h, bufs=bufs)
        torch.cuda.current_stream().synchronize()
        float(Oh[0, 0, 0, 0])  # read the result on the host
    e2e_s = max_over_ranks(time.perf_counter() - t0, dev)
    h2d = in_bytes + (lens_h.numel() * 4 if lens_h is not None else 0)
    e2e = {"value": round(whole_job_value(flops * e2e_steps, world, e2e_s) / 1e12, 2),
           "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": out_bytes,
           "ms_per_step": round(e2e_s / e2e_steps * 1e3, 3)}
    del bufs
    q = sorted(step_ms)
    pick = lambda f: q[min(len(q) - 1, int(round(f * (len(q) - 1))))]
    spread = {"median": round(statistics.median(q), 4), "p10": round(pick(0.1), 4),
              "p90": round(pick(0.9), 4), "unit": "ms"}
    if warm_ms is not None:
        spread["warm_l2_ms"] = round(warm_ms, 4)
    return dict(value=value, per_step=per_step, kernel_tflops=kernel_tflops, flops=flops,
                clocks=clocks.summary(), e2e=e2e, Q=Q, K=K, V=V, lens=lens, dims=dims,
                step_ms=spread,
                l2="inputs larger than L2" if flush is None else "L2 flushed between steps")


def _cold_steps(step, steps, flush):
    """Per-step device times (ms) of ``steps`` calls of ``step`` on the
    current stream: one event between consecutive steps when ``flush`` is
    None (inputs larger than L2), else a 256 MB write before each step and
    each step timed by its own event pair."""
    import torch
    stream = torch.cuda.current_stream()
    if flush is None:
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        evs[0].record(stream)
        for i in range(steps):
            step()
            evs[i + 1].record(stream)
        torch.cuda.synchronize()
        return [evs[i].elapsed_time(evs[i + 1]) for i in range(steps)]
    out = []
    for _ in range(steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        torch.cuda.synchronize()
        out.append(e0.elapsed_time(e1))
    return out


def bench_attention_workload(w, steps, warmup, local_rank, peaks, peak_src):
    """One attention workload (the inputs the parity tests use), cold L2:
    median step time, achieved TFLOP/s or GB/s against its roofline."""
    import torch
    import transformer_head_scaled_03_gb300 as mha
    from transformer_head_scaled_03_gb300.inputs import sdpa_inputs

    dev = torch.device("cuda", local_rank)
    Q, K, V, lens, _ = sdpa_inputs(w)
    mk = lambda a: torch.from_numpy(a).to(torch.bfloat16).to(dev)
    Qd, Kd, Vd = mk(Q), mk(K), mk(V)
    del Q, K, V
    kl = torch.from_numpy(lens).to(dev) if lens is not None else None
    Od = torch.empty_like(Qd)
    l2 = sdpa_l2_note(w)
    flush = (None if l2 == "inputs larger than L2"
             else torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev))

    def step():
        mha.sdpa_forward(Qd, Kd, Vd, mask_kind=w.mask, key_lengths=kl, out=Od)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    st = mha.mha_check()
    if st != mha.MHA_OK:
        raise RuntimeError(mha.status_string(st))
    ms = _cold_steps(step, steps, flush)
    st = mha.mha_check()
    if st != mha.MHA_OK:
        raise RuntimeError(mha.status_string(st))
    med = statistics.median(ms)
    flops, nbytes = w.flops(lens), w.sdpa_bytes(lens)
    tflops = flops / (med / 1e3) / 1e12
    roof = attention_roofline(flops, nbytes, tflops, peaks["bf16_tflops"], peaks["hbm_gbs"],
                              peak_src)
    roof.update({"algorithmic_bytes": int(nbytes), "kernel": fwd_kernel_name(w)})
    del Qd, Kd, Vd, Od, flush
    torch.cuda.empty_cache()
    return {"workload": w.name, "wid": w.wid, "mask": MASK_NAMES[w.mask],
            "us_per_step": round(med * 1e3, 2), "us_p10": round(sorted(ms)[len(ms) // 10] * 1e3, 2),
            "tflops": round(tflops, 2), "pct_bf16_peak_nominal": round(100 * tflops / NOMINAL_BF16_TFLOPS, 2),
            "flops_per_step": flops, "roofline": roof, "l2": l2, "steps": steps,
            "timing": "median of per-step CUDA events on the launching stream",
            "gpu_launches_per_step": 1}


def bench_base_layer_cold(steps, warmup, local_rank, peaks):
    """The base-shape layer (workload 1: B1 L128 D512 h8 fp32, mha_forward,
    three launches) with L2 flushed before every step: median tokens/s, and
    the oracle's layer on the host with all threads and with one."""
    import torch
    import transformer_head_scaled_03_gb300 as mha
    from transformer_head_scaled_03_gb300.inputs import WORKLOADS, mha_inputs

    w = WORKLOADS[1]
    dev = torch.device("cuda", local_rank)
    x_h, *Ws_h = mha_inputs(w)
    x = torch.from_numpy(x_h).to(dev)
    Ws = [torch.from_numpy(W).to(dev) for W in Ws_h]
    out = torch.empty_like(x)
    handle = mha.mha_create(w.D, torch.float32, w.B, w.Lq, w.Lk)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    try:
        step = lambda: mha.mha_forward(handle, x, x, *Ws, h=w.H, out=out)
        for _ in range(warmup):
            step()
        torch.cuda.synchronize()
        ms = _cold_steps(step, steps, flush)
        st = mha.mha_check(handle)
        if st != mha.MHA_OK:
            raise RuntimeError(mha.status_string(st))
    finally:
        handle.close()
    med = statistics.median(ms)
    flops = mha_layer_flops(w)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    fma_peak = sms * 128 * 2.0 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
    achieved = flops / (med / 1e3) / 1e12
    return {"workload": w.name, "wid": 1, "mask": "none",
            "us_per_step": round(med * 1e3, 2), "tokens_per_s": round(w.B * w.Lq / (med / 1e3), 1),
            "flops_per_step": flops,
            "roofline": {"bound": "alu", "achieved": round(achieved, 3), "peak": round(fma_peak, 2),
                         "unit": "TFLOP/s", "frac": round(achieved / fma_peak, 4),
                         "peak_source": "derived: SMs x 128 fp32 FMA lanes x 2 flops x max clock",
                         "kernel": "the layer's launches timed together"},
            "l2": "L2 flushed between steps", "steps": steps,
            "timing": "median of per-step CUDA events on the launching stream",
            "gpu_launches_per_step": 3}


def oracle_base_layer(min_seconds=1.0):
    """The oracle's base-shape layer on the host with all its threads:
    (tokens/s, seconds per layer, threads)."""
    from transformer_head_scaled_03_gb300.inputs import WORKLOADS, mha_inputs
    import oracle
    w = WORKLOADS[1]
    x, *Ws = mha_inputs(w)
    orc = oracle.default()
    orc.mha(x, x, *Ws, h=w.H)
    n, t0 = 0, time.perf_counter()
    while True:
        orc.mha(x, x, *Ws, h=w.H)
        n += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds:
            break
    return w.B * w.Lq * n / dt, dt / n, orc.num_threads()


def oracle_base_layer_one_thread(min_seconds=1.0):
    """The same on one thread, in a child process started with
    OMP_NUM_THREADS=1 (so this process's oracle keeps all its threads):
    (tokens/s, seconds per layer), or None if the child fails."""
    code = ("import json, sys, time; sys.path.insert(0, %r)\n"
            "import bench\n"
            "tps, sec, th = bench.oracle_base_layer(%r)\n"
            "print(json.dumps([tps, sec, th]))\n") % (ROOT, float(min_seconds))
    env = dict(os.environ, OMP_NUM_THREADS="1")
    try:
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True,
                           text=True, timeout=120, cwd=ROOT)
        tps, sec, th = json.loads(r.stdout.strip().splitlines()[-1])
    except Exception:
        return None
    return (tps, sec) if th == 1 else None


def bench_mha_layer(w_shape, dtype_name, steps, warmup, local_rank, seed_w=None):
    """Tokens/s of one mha_forward (all rows a1-a8) on the given shape."""
    import torch
    import transformer_head_scaled_03_gb300 as mha
    from transformer_head_scaled_03_gb300.inputs import Draws

    B, L, D, h = w_shape
    dev = torch.device("cuda", local_rank)
    dtype = torch.bfloat16 if dtype_name == "bf16" else torch.float32
    g = Draws(seed_w if seed_w is not None else 0x5EED0100 + D)
    mk = lambda a: torch.from_numpy(a).to(dtype).to(dev)
    x = mk(g.normal((B, L, D), dtype=dtype_name))
    Ws = [mk(g.normal((D, D), std=1.0 / math.sqrt(D), dtype=dtype_name)) for _ in range(4)]
    out = torch.empty_like(x)
    handle = mha.mha_create(D, dtype, B, L, L)
    try:
        # eager, and the same call captured once in a CUDA graph and replayed:
        # the library's device time without the per-call host overhead
        call = lambda: mha.mha_forward(handle, x, x, *Ws, h=h, out=out)
        eager_ms, graph_ms = _time_eager_and_graph(call, steps, warmup)
        layers_ms = (_time_graph_layers(call, GRAPH_LAYERS, max(steps, 60), warmup)
                     if graph_ms < 1.0 else None)
        st = mha.mha_check(handle)
        if st != mha.MHA_OK:
            raise RuntimeError(mha.status_string(st))
    finally:
        handle.close()
    d = D // h
    proj_flops = 4 * 2.0 * B * L * D * D
    attn_flops = 4.0 * B * h * L * L * d
    return {"shape": {"B": B, "L": L, "D": D, "h": h, "dtype": dtype_name, "mask": "none"},
            "tokens_per_s": round(B * L / (graph_ms / 1e3), 1),
            "ms_per_layer": round(graph_ms, 4),
            "tflops": round((proj_flops + attn_flops) / (graph_ms / 1e3) / 1e12, 2),
            "timing": "CUDA graph replay of one mha_forward call",
            "eager_tokens_per_s": round(B * L / (eager_ms / 1e3), 1),
            "eager_ms_per_layer": round(eager_ms, 4),
            **({} if layers_ms is None else {
                "graph6_tokens_per_s": round(B * L / (layers_ms / 1e3), 1),
                "graph6_ms_per_layer": round(layers_ms, 4),
                "graph6_timing": f"one CUDA graph of {GRAPH_LAYERS} back-to-back calls, per call"}),
            "gpu_launches_per_layer": 3}


def encoder_launches(dtype_name, D):
    """Launches of one encoder_forward: five when the residual add and
    LayerNorm run in the GEMM epilogues (bf16, d_model a multiple of 64 up
    to 512), seven otherwise."""
    return 5 if dtype_name == "bf16" and D <= 512 and D % 64 == 0 else 7


def bench_encoder_layer(shape, dtype_name, steps, warmup, local_rank, key_padding=None):
    """Tokens/s of one encoder_forward (post-norm encoder layer: MHA with
    biases, residual + LayerNorm, ReLU FFN, residual + LayerNorm)."""
    import torch
    import transformer_head_scaled_03_gb300 as mha
    from transformer_head_scaled_03_gb300.inputs import Draws

    B, L, D, h, F = shape
    dev = torch.device("cuda", local_rank)
    dtype = torch.bfloat16 if dtype_name == "bf16" else torch.float32
    g = Draws(0x5EED0200 + D + F)
    mk = lambda a: torch.from_numpy(a).to(dtype).to(dev)
    x = mk(g.normal((B, L, D), dtype=dtype_name))
    p = {}
    for n in ("Wq", "Wk", "Wv", "Wo"):
        p[n] = mk(g.normal((D, D), std=1.0 / math.sqrt(D), dtype=dtype_name))
    p["W1"] = mk(g.normal((D, F), std=1.0 / math.sqrt(D), dtype=dtype_name))
    p["W2"] = mk(g.normal((F, D), std=1.0 / math.sqrt(F), dtype=dtype_name))
    for n in ("bq", "bk", "bv", "bo", "b2", "ln1_beta", "ln2_beta"):
        p[n] = mk(g.normal((D,), std=0.1, dtype=dtype_name))
    p["b1"] = mk(g.normal((F,), std=0.1, dtype=dtype_name))
    for n in ("ln1_gamma", "ln2_gamma"):
        p[n] = mk(1.0 + g.normal((D,), std=0.1, dtype="f32"))
    lens = None
    mask = mha.MASK_NONE
    if key_padding is not None:
        lens = torch.from_numpy(g.integers(key_padding[0], key_padding[1], B)).to(dev)
        mask = mha.MASK_KEY_PADDING
    out = torch.empty_like(x)
    layer = mha.EncoderLayer(D, h, F, dtype, B, L)
    try:
        call = lambda: layer.forward(x, p, mask_kind=mask, key_lengths=lens, out=out)
        eager_ms, graph_ms = _time_eager_and_graph(call, steps, warmup)
        layers_ms = (_time_graph_layers(call, GRAPH_LAYERS, max(steps, 60), warmup)
                     if graph_ms < 1.0 else None)
        st = mha.mha_check()
        if st != mha.MHA_OK:
            raise RuntimeError(mha.status_string(st))
    finally:
        layer.close()
    # algorithmic flops: the six GEMMs, plus 4*d per unmasked query/key pair
    keys = B * L if lens is None else int(lens.sum().item())
    flops = 8.0 * B * L * D * D + 4.0 * B * L * D * F + 4.0 * L * keys * D
    return {"shape": {"B": B, "L": L, "D": D, "h": h, "d_ff": F, "dtype": dtype_name,
                      "mask": "none" if lens is None else
                      f"key_padding, lengths U[{key_padding[0]}, {key_padding[1]}]"},
            "tokens_per_s": round(B * L / (graph_ms / 1e3), 1),
            "ms_per_layer": round(graph_ms, 4),
            "tflops": round(flops / (graph_ms / 1e3) / 1e12, 2),
            "timing": "CUDA graph replay of one encoder_forward call",
            "eager_tokens_per_s": round(B * L / (eager_ms / 1e3), 1),
            "eager_ms_per_layer": round(eager_ms, 4),
            **({} if layers_ms is None else {
                "graph6_tokens_per_s": round(B * L / (layers_ms / 1e3), 1),
                "graph6_ms_per_layer": round(layers_ms, 4),
                "graph6_timing": f"one CUDA graph of {GRAPH_LAYERS} back-to-back calls, per call"}),
            "gpu_launches_per_layer": encoder_launches(dtype_name, D)}


def bench_decode(w, steps, warmup, local_rank, hbm_peak):
    """One sdpa_decode over a decode workload: bytes moved per second
    against the HBM peak (the pass is bound by streaming the cache)."""
    import torch
    import transformer_head_scaled_03_gb300 as mha
    from transformer_head_scaled_03_gb300.inputs import Draws

    dev = torch.device("cuda", local_rank)
    # the cache is drawn on the device (seeded) to keep the benchmark quick;
    # the parity tests draw the same shapes through the shared generator
    gen = torch.Generator(device=dev)
    gen.manual_seed(w.seed)
    mk = lambda *shape: torch.randn(*shape, generator=gen, device=dev,
                                    dtype=torch.float32).to(torch.bfloat16)
    Q = mk(w.B, w.H, w.Lq, w.d)
    K = mk(w.B, w.H, w.Lk, w.d)
    V = mk(w.B, w.H, w.Lk, w.d)
    lo, hi = w.len_range
    lens = Draws(w.seed).integers(lo, hi, w.B)
    kl = torch.from_numpy(lens).to(dev)
    out = torch.empty_like(Q)
    splits = mha.decode_splits(w.B, w.H, w.Lk, w.d)

    def step():
        mha.sdpa_decode(Q, K, V, kv_lengths=kl, causal=True, out=out)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    st = mha.mha_check()
    if st != mha.MHA_OK:
        raise RuntimeError(mha.status_string(st))
    nbytes = w.decode_bytes(lens)
    gbs = nbytes / (ms / 1e3) / 1e9
    del K, V
    return {"workload": w.name, "Lq": w.Lq, "splits": splits,
            "us_per_call": round(ms * 1e3, 2),
            "GB_per_s": round(gbs, 1), "hbm_frac": round(gbs / hbm_peak, 4),
            "hbm_frac_nominal": round(gbs / NOMINAL_HBM_GBS, 4),
            "bytes_per_call": int(nbytes),
            "tflops": round(w.flops(lens) / (ms / 1e3) / 1e12, 2),
            "tokens_per_s": round(w.B * w.Lq / (ms / 1e3), 1),
            "l2": "cache larger than L2", "gpu_launches_per_call": 1}


DECODE_METRIC = "decode attention GB/s of cache streamed (and % of GB300 HBM peak)"
DECODE_KERNEL_FILES = ["transformer_head_scaled_03_gb300/csrc/sdpa_decode.cu",
                       "transformer_head_scaled_03_gb300/csrc/ptx.cuh",
                       "transformer_head_scaled_03_gb300/csrc/ptx_cluster.cuh"]


def decode_device_inputs(w, dev):
    """Seeded device-side draws of one decode workload: Q, the K/V cache, the
    per-item lengths (host int32 and device)."""
    import torch
    from transformer_head_scaled_03_gb300.inputs import Draws
    gen = torch.Generator(device=dev)
    gen.manual_seed(w.seed)
    mk = lambda *shape: torch.randn(*shape, generator=gen, device=dev,
                                    dtype=torch.float32).to(torch.bfloat16)
    Q = mk(w.B, w.H, w.Lq, w.d)
    K = mk(w.B, w.H, w.Lk, w.d)
    V = mk(w.B, w.H, w.Lk, w.d)
    lens = Draws(w.seed).integers(w.len_range[0], w.len_range[1], w.B)
    return Q, K, V, lens, torch.from_numpy(lens).to(dev)


def decode_oracle_sample(w, Q, K, V, lens, n_heads, seed):
    """The oracle as it stands on every query row of ``n_heads`` seeded (b, h)
    pairs (host float32 copies of those heads); returns GB/s of the cache
    those rows read, seconds, threads, heads."""
    import oracle
    from transformer_head_scaled_03_gb300.inputs import Draws
    n = min(n_heads, w.B * w.H)
    bhs = Draws(seed).choice(w.B * w.H, n)
    host = lambda t, L: (t.reshape(w.B * w.H, L, w.d)[bhs].float().cpu().numpy()[:, None]
                         if hasattr(t, "cpu") else t.reshape(w.B * w.H, L, w.d)[bhs][:, None])
    q, k, v = host(Q, w.Lq), host(K, w.Lk), host(V, w.Lk)
    lb = np.asarray(lens)[bhs // w.H].astype(np.int32)
    orc = oracle.default()
    t0 = time.perf_counter()
    orc.sdpa(q, k, v, mask_kind=w.mask, key_lengths=lb)
    dt = time.perf_counter() - t0
    nbytes = 2.0 * w.d * (2.0 * float(np.sum(lb)) + 2.0 * n * w.Lq)
    return nbytes / dt / 1e9, dt, orc.num_threads(), n


def run_gpu_decode(args, w, rank, world, local_rank):
    """The decode workloads as the benchmark's main step: one sdpa_decode per
    step over a resident cache; value = whole-job GB/s of cache streamed."""
    import torch
    import torch.distributed as dist
    import transformer_head_scaled_03_gb300 as mha

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    peaks, peak_src = measured_peaks()
    Q, K, V, lens, kl = decode_device_inputs(w, dev)
    out = torch.empty_like(Q)
    nbytes = w.decode_bytes(lens)
    cache_bytes = 2 * K.numel() * K.element_size()
    flush = None
    if cache_bytes < 2 * L2_BYTES:
        flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

    def step():
        mha.sdpa_decode(Q, K, V, kv_lengths=kl, causal=True, out=out)

    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert mha.mha_check() == mha.MHA_OK
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clocks:
        total_ms = 0.0
        if flush is None:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(args.steps):
                step()
            e1.record(stream)
            torch.cuda.synchronize()
            total_ms = e0.elapsed_time(e1)
        else:
            for _ in range(args.steps):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                step()
                e1.record(stream)
                torch.cuda.synchronize()
                total_ms += e0.elapsed_time(e1)
    barrier()
    torch.cuda.synchronize()
    st = mha.mha_check()
    if st != mha.MHA_OK:
        raise RuntimeError(f"device error during timing: {mha.status_string(st)}")
    max_s = max_over_ranks(total_ms / 1e3, dev)
    value = whole_job_value(nbytes * args.steps, world, max_s) / 1e9
    kernel_gbs = nbytes / (total_ms / 1e3 / args.steps) / 1e9

    # end to end through the public call: the new queries copied in from
    # pinned host memory and the outputs read back every step (the cache is
    # the server's resident state)
    Qh = Q.cpu().pin_memory()
    Oh = torch.empty_like(Qh).pin_memory()
    Qd = torch.empty_like(Q)
    barrier()
    torch.cuda.synchronize()
    e2e_steps = max(2, min(args.steps, 20))
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        Qd.copy_(Qh, non_blocking=True)
        mha.sdpa_decode(Qd, K, V, kv_lengths=kl, causal=True, out=out)
        Oh.copy_(out, non_blocking=True)
        torch.cuda.current_stream().synchronize()
        float(Oh[0, 0, 0, 0])
    e2e_s = max_over_ranks(time.perf_counter() - t0, dev)
    e2e = {"value": round(whole_job_value(nbytes * e2e_steps, world, e2e_s) / 1e9, 1),
           "unit": "GB/s", "h2d_bytes_per_step": Qh.numel() * 2,
           "d2h_bytes_per_step": Oh.numel() * 2,
           "ms_per_step": round(e2e_s / e2e_steps * 1e3, 4)}

    cpu = None
    if rank == 0 and not args.skip_cpu:
        gbs, dt, cores, n = decode_oracle_sample(w, Q, K, V, lens, 64, w.seed + 3000)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
               "seconds": round(dt, 2),
               "sample": f"every query row of {n} seeded (b, h) pairs of the same workload, fp64"}
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    traffic = args.traffic
    if traffic is None and args.batch is None:
        traffic = recorded_traffic(DECODE_KERNEL_FILES,
                                   f"profiles/sdpa_decode_bf16_workload{args.workload}.md")
    peak = peaks["hbm_gbs"]
    line = {
        "metric": DECODE_METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(max_s / args.steps * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "Lq": w.Lq, "cache": w.Lk, "d": w.d,
                   "lengths": f"U[{w.len_range[0]}, {w.len_range[1]}]",
                   "mask": "bottom-right causal + per-item lengths",
                   "splits": mha.decode_splits(w.B, w.H, w.Lk, w.d),
                   "bytes_per_step": int(nbytes), "flops_per_step": w.flops(lens),
                   "l2": "cache larger than L2" if flush is None else "L2 flushed between steps",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": round(kernel_gbs, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(kernel_gbs / peak, 4),
                     "frac_nominal": round(kernel_gbs / NOMINAL_HBM_GBS, 4),
                     "peak_source": f"{peak_src} HBM copy", "traffic": traffic,
                     "kernel": f"sdpa_decode_bf16_kernel<{w.d}>"},
        "tflops": round(w.flops(lens) / (total_ms / 1e3 / args.steps) / 1e12, 2),
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clocks.summary(),
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def bench_embed_pe(shape, steps, warmup, local_rank, hbm_peak, layer_shape=None):
    """embed_pe_forward (embedding x sqrt(D) + PE, one pass) in GB/s against
    the HBM peak; with ``layer_shape`` (h, d_ff) also the embedding pass plus
    one encoder layer, tokens/s (CUDA graph replay of both calls)."""
    import torch
    import transformer_head_scaled_03_gb300 as mha
    from transformer_head_scaled_03_gb300.inputs import Draws

    B, L, D, vocab = shape
    dev = torch.device("cuda", local_rank)
    gen = torch.Generator(device=dev)
    gen.manual_seed(0x5EED0300 + D)
    table = (torch.randn(vocab, D, generator=gen, device=dev) / math.sqrt(D)).to(torch.bfloat16)
    ids = torch.from_numpy(Draws(0x5EED0300 + L).integers(0, vocab - 1, (B, L))).to(dev)
    pe = mha.sinusoidal_pe(L, D, device=dev)
    x = torch.empty((B, L, D), dtype=torch.bfloat16, device=dev)
    eager_ms, graph_ms = _time_eager_and_graph(lambda: mha.embed_pe(ids, table, pe, out=x),
                                               steps, warmup)
    rows = B * L
    nbytes = rows * (2 * D + 2 * D + 4) + L * D * 4
    out = {"shape": {"B": B, "L": L, "D": D, "vocab": vocab, "dtype": "bf16"},
           "us_per_call": round(graph_ms * 1e3, 2), "GB_per_s": round(nbytes / graph_ms / 1e6, 1),
           "hbm_frac": round(nbytes / graph_ms / 1e6 / hbm_peak, 4),
           "hbm_frac_nominal": round(nbytes / graph_ms / 1e6 / NOMINAL_HBM_GBS, 4),
           "bytes_per_call": nbytes, "tokens_per_s": round(rows / (graph_ms / 1e3), 1),
           "timing": "CUDA graph replay", "gpu_launches_per_call": 1}
    if layer_shape is not None:
        h, F = layer_shape
        g = Draws(0x5EED0400 + D)
        mk = lambda a: torch.from_numpy(a).to(torch.bfloat16).to(dev)
        p = {n: mk(g.normal((D, D), std=1.0 / math.sqrt(D), dtype="bf16"))
             for n in ("Wq", "Wk", "Wv", "Wo")}
        p["W1"] = mk(g.normal((D, F), std=1.0 / math.sqrt(D), dtype="bf16"))
        p["W2"] = mk(g.normal((F, D), std=1.0 / math.sqrt(F), dtype="bf16"))
        for n in ("bq", "bk", "bv", "bo", "b2", "ln1_beta", "ln2_beta"):
            p[n] = mk(g.normal((D,), std=0.1, dtype="bf16"))
        p["b1"] = mk(g.normal((F,), std=0.1, dtype="bf16"))
        for n in ("ln1_gamma", "ln2_gamma"):
            p[n] = mk(1.0 + g.normal((D,), std=0.1, dtype="f32"))
        y = torch.empty_like(x)
        layer = mha.EncoderLayer(D, h, F, torch.bfloat16, B, L)
        try:
            def both():
                mha.embed_pe(ids, table, pe, out=x)
                layer.forward(x, p, out=y)
            _, both_ms = _time_eager_and_graph(both, steps, warmup)
        finally:
            layer.close()
        out["with_encoder_layer"] = {"h": h, "d_ff": F, "ms": round(both_ms, 4),
                                     "tokens_per_s": round(rows / (both_ms / 1e3), 1),
                                     "gpu_launches": 1 + encoder_launches("bf16", D)}
    st = mha.mha_check()
    if st != mha.MHA_OK:
        raise RuntimeError(mha.status_string(st))
    return out


def bench_backward(w, steps, warmup, local_rank, peak):
    """sdpa_backward (dQ, dK, dV of a causal or unmasked SDPA) in TFLOP/s.

    Algorithmic flops are 2.5x the forward's: five products over the visible
    (query, key) pairs (S recomputed, dP, dV, dK, dQ), 2 d flops each.  Each
    call is the whole public call: the D = rowsum(dO * O) pass, the dQ zero
    fill and the fused kernel.  Inputs are N(0, 1) bf16 drawn on the device,
    larger than L2, and O and lse come from sdpa_forward_lse outside the
    timed region."""
    import torch
    import transformer_head_scaled_03_gb300 as mha

    dev = torch.device("cuda", local_rank)
    gen = torch.Generator(device=dev)
    gen.manual_seed(0x5EED0500 + w.wid)
    mk = lambda L: torch.randn(w.B, w.H, L, w.d, generator=gen, device=dev).to(torch.bfloat16)
    Q, K, V, dO = mk(w.Lq), mk(w.Lk), mk(w.Lk), mk(w.Lq)
    O, lse = mha.sdpa_forward_lse(Q, K, V, mask_kind=w.mask)
    ws = torch.empty(max(16, w.B * w.H * w.Lq * 4), dtype=torch.uint8, device=dev)
    grads = mha.sdpa_backward(Q, K, V, O, dO, lse, mask_kind=w.mask, workspace=ws)
    dQ, dK, dV = grads
    for _ in range(warmup):
        mha.sdpa_backward(Q, K, V, O, dO, lse, mask_kind=w.mask, workspace=ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        mha.sdpa_backward(Q, K, V, O, dO, lse, mask_kind=w.mask, workspace=ws)
    e1.record()
    torch.cuda.synchronize()
    st = mha.mha_check()
    if st != mha.MHA_OK:
        raise RuntimeError(mha.status_string(st))
    ms = e0.elapsed_time(e1) / steps
    flops = 2.5 * w.flops()
    tf = flops / (ms / 1e3) / 1e12
    del Q, K, V, dO, O, lse, dQ, dK, dV, grads, ws
    torch.cuda.empty_cache()
    return {"workload": w.name, "mask": {0: "none", 1: "causal"}[w.mask],
            "ms_per_call": round(ms, 4), "flops_per_call": flops, "tflops": round(tf, 2),
            "frac_of_peak": round(tf / peak, 4), "peak": peak, "grad_dtype": "bf16 dK dV, fp32 dQ",
            "gpu_launches_per_call": 2, "timing": "eager, CUDA events, inputs > L2"}


GRAPH_LAYERS = 6  # calls captured in one graph for the per-layer device time (the base model's depth)


def _time_graph_layers(step, n, steps, warmup):
    """ms per call of ``step`` inside one CUDA graph of ``n`` back-to-back
    calls: a single-call graph's replay also pays the graph launch, which for
    a layer of a few tens of microseconds is a visible share of it."""
    import torch

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(n):
            step()
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    reps = max(1, steps // n)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / (reps * n)


def _time_eager_and_graph(step, steps, warmup):
    """(eager ms, CUDA-graph-replay ms) per call of ``step``."""
    import torch

    def timed(fn, n):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    eager_ms = timed(step, steps)
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    with torch.cuda.graph(graph):
        step()
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    return eager_ms, timed(graph.replay, steps)


def run_gpu(args):
    import torch
    import torch.distributed as dist
    from transformer_head_scaled_03_gb300.inputs import WORKLOADS, sample_rows
    import __graft_entry__

    rank, world, local_rank = dist_env()
    if world > 1:
        torch.cuda.set_device(local_rank)
        dist.init_process_group(backend="nccl")
    __graft_entry__.build()
    w = workload_from_args(args)
    if w.kind == "decode":
        run_gpu_decode(args, w, rank, world, local_rank)
        return
    if w.kind == "mha":
        run_gpu_mha(args, w, rank, world, local_rank)
        return
    r = bench_sdpa(args, w, rank, world, local_rank)
    peaks, peak_src = measured_peaks()

    workloads = None
    if not args.skip_workloads:
        workloads = [bench_attention_workload(WORKLOADS[i], 20, 3, local_rank, peaks, peak_src)
                     for i in (2, 3, 4)]
        base = bench_base_layer_cold(50, 5, local_rank, peaks)
        if rank == 0 and not args.skip_cpu:
            tps, sec, cores = oracle_base_layer()
            one = oracle_base_layer_one_thread()
            base["cpu_baseline"] = {
                "value": round(tps, 1), "unit": "tokens/s", "cores": cores,
                "kind": "oracle", "seconds_per_layer": round(sec, 4),
                "one_thread": None if one is None else {
                    "value": round(one[0], 1), "unit": "tokens/s", "cores": 1,
                    "seconds_per_layer": round(one[1], 4)},
                "sample": "the whole layer (every token), fp64, repeated for ~1 s"}
        workloads.insert(0, base)

    mha_layer = None
    if not args.skip_mha:
        mha_layer = [bench_mha_layer((w.B, w.Lq, w.H * w.d, w.H), "bf16", 3, 3, local_rank),
                     bench_mha_layer((1, 128, 512, 8), "f32", 200, 5, local_rank,
                                     seed_w=WORKLOADS[1].seed)]
    encoder_layer = None
    embed = None
    if not args.skip_mha:
        w2 = WORKLOADS[2]
        encoder_layer = [
            bench_encoder_layer((w2.B, w2.Lq, w2.H * w2.d, w2.H, 4 * w2.H * w2.d), "bf16", 20, 3,
                                local_rank, key_padding=w2.len_range),
            bench_encoder_layer((1, 128, 512, 8, 2048), "f32", 100, 5, local_rank)]
        w2 = WORKLOADS[2]
        embed = bench_embed_pe((w2.B, w2.Lq, w2.H * w2.d, 37000), 20, 3, local_rank,
                               peaks["hbm_gbs"], layer_shape=(w2.H, 4 * w2.H * w2.d))

    decode = None
    if not args.skip_decode:
        decode = [bench_decode(WORKLOADS[i], 50, 5, local_rank, peaks["hbm_gbs"])
                  for i in (6, 7, 8)]

    backward = None
    if not args.skip_backward:
        # the selected shape (no mask or causal), then the decoder causal shape
        shapes = [w] if (w.mask in (0, 1) and w.wid != 3) else []
        backward = [bench_backward(x, 5 if x.Lq >= 16384 else 20, 3, local_rank,
                                   peaks["bf16_tflops"]) for x in shapes + [WORKLOADS[3]]]

    cpu = None
    if rank == 0 and not args.skip_cpu:
        # the sample the reference arm times at every step
        rows, per_head = oracle_sample(w, args.cpu_rows_per_head)
        tf, dt, cores = oracle_cpu_baseline(w, r["Q"], r["K"], r["V"], r["lens"], rows)
        cpu = {"value": round(tf, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "seconds": round(dt, 2), "sample": sample_description(w, rows, per_head)}
        if rows.size < w.B * w.H * w.Lq:
            # every output row at the sample's rate: the oracle's cost per row
            # is proportional to the keys the row sees, i.e. to its flops
            cpu["extrapolated_full_output_seconds"] = round(r["flops"] / (tf * 1e12), 1)
            cpu["extrapolation"] = ("extrapolated, not measured: the workload's algorithmic "
                                    "flops over the sample's measured oracle rate")

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    ach = r["kernel_tflops"]
    peak = peaks["bf16_tflops"]
    traffic = args.traffic
    if traffic is None and args.workload == 5 and args.seq is None and args.heads is None:
        traffic = recorded_traffic(["transformer_head_scaled_03_gb300/csrc/sdpa_bf16.cu",
                                    "transformer_head_scaled_03_gb300/csrc/ptx.cuh"],
                                   "profiles/sdpa_fwd_bf16_long_context.md")
    alg_bytes = w.sdpa_bytes(r["lens"])
    roofline = attention_roofline(r["flops"], alg_bytes, ach, peak, peaks["hbm_gbs"], peak_src)
    roofline.update({"traffic": traffic, "algorithmic_bytes": int(alg_bytes),
                     "kernel": fwd_kernel_name(w)})
    line = {
        "metric": METRIC,
        "value": round(r["value"], 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(r["per_step"] * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": sdpa_config(w, r["lens"], world, args.float_mask),
        "pct_bf16_peak_nominal": round(100.0 * ach / NOMINAL_BF16_TFLOPS, 2),
        "roofline": roofline,
        "e2e": r["e2e"],
        "step_ms": r["step_ms"],
        "gpu_launches": args.steps,
        "clocks": r["clocks"],
        "cpu_baseline": cpu,
        "workloads": workloads,
        "mha_layer": mha_layer,
        "encoder_layer": encoder_layer,
        "embed_pe": embed,
        "decode": decode,
        "backward": backward,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


MHA_METRIC = "MHA layer tokens/s"


def mha_layer_flops(w) -> float:
    """Algorithmic flops of one layer: four D x D projections of every token
    and the attention's two products over every (query, key) pair."""
    return 4 * 2.0 * w.B * w.Lq * w.D * w.D + 4.0 * w.B * w.H * w.Lq * w.Lk * w.d


def oracle_mha_baseline(w, x, Ws, min_seconds=2.0):
    """The fp64 oracle's layer (as it stands) on the whole input, repeated
    for about ``min_seconds``: (tokens/s, seconds per layer, threads)."""
    import oracle
    orc = oracle.default()
    n, t0 = 0, time.perf_counter()
    while True:
        orc.mha(x, x, *Ws, h=w.H)
        n += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds:
            break
    return w.B * w.Lq * n / dt, dt / n, orc.num_threads()


def run_gpu_mha(args, w, rank, world, local_rank):
    """The base-shape layer as the step: one mha_forward (three launches) per
    step on device-resident inputs, L2 flushed between steps."""
    import torch
    import torch.distributed as dist
    import transformer_head_scaled_03_gb300 as mha
    from transformer_head_scaled_03_gb300.inputs import mha_inputs

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    x_h, *Ws_h = mha_inputs(w)
    tf = lambda a: torch.from_numpy(a)
    x_pin = tf(x_h).pin_memory()
    x = x_pin.to(dev)
    Ws = [tf(W).to(dev) for W in Ws_h]
    out = torch.empty_like(x)
    handle = mha.mha_create(w.D, torch.float32, w.B, w.Lq, w.Lk)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        mha.mha_forward(handle, x, x, *Ws, h=w.H, out=out)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert mha.mha_check(handle) == mha.MHA_OK
    barrier()
    torch.cuda.synchronize()
    step_ms = []
    with ClockSampler(local_rank) as clocks:
        for _ in range(args.steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            step()
            e1.record(stream)
            torch.cuda.synchronize()
            step_ms.append(e0.elapsed_time(e1))
    barrier()
    torch.cuda.synchronize()
    st = mha.mha_check(handle)
    if st != mha.MHA_OK:
        raise RuntimeError(f"device error during timing: {mha.status_string(st)}")
    total_ms = sum(step_ms)
    max_s = max_over_ranks(total_ms / 1e3, dev)
    tokens = w.B * w.Lq
    value = whole_job_value(tokens * args.steps, world, max_s)
    per_step_ms = total_ms / args.steps
    # context: the same call back to back (inputs in L2) and as a graph replay
    eager_ms, graph_ms = _time_eager_and_graph(step, 200, 5)
    # end to end: x from pinned host memory, the layer, out back to the host
    out_h = torch.empty(x.shape, dtype=torch.float32).pin_memory()
    torch.cuda.synchronize()
    barrier()
    t0 = time.perf_counter()
    e2e_steps = 50
    for _ in range(e2e_steps):
        x.copy_(x_pin, non_blocking=True)
        step()
        out_h.copy_(out, non_blocking=True)
        torch.cuda.current_stream().synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, dev)
    handle.close()
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    flops = mha_layer_flops(w)
    # fp32 FMA rate of the CUDA cores: SMs x 128 lanes x 2 flops x max clock
    peaks, _ = measured_peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    fma_peak = sms * 128 * 2.0 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
    achieved = flops / (per_step_ms / 1e3) / 1e12
    cpu = None
    if not args.skip_cpu:
        tps, sec, cores = oracle_mha_baseline(w, x_h, Ws_h)
        cpu = {"value": round(tps, 2), "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "seconds_per_layer": round(sec, 4),
               "sample": "the whole workload (every token of the layer), fp64, repeated for ~2 s"}
    q = sorted(step_ms)
    pick = lambda f: q[min(len(q) - 1, int(round(f * (len(q) - 1))))]
    line = {
        "metric": MHA_METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(max_s / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "L": w.Lq, "D": w.D, "h": w.H, "mask": "none",
                   "flops_per_step": flops, "l2": "L2 flushed between steps",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "alu", "achieved": round(achieved, 3), "peak": round(fma_peak, 2),
                     "unit": "TFLOP/s", "frac": round(achieved / fma_peak, 4),
                     "peak_source": f"derived: {sms} SMs x 128 fp32 FMA lanes x 2 flops x "
                                    f"{peaks.get('sm_max_mhz', 2070.0):.0f} MHz",
                     "traffic": None,
                     "kernel": "the layer's three launches (Q/K/V projection, attention, "
                               "output projection) timed together"},
        "step_ms": {"median": round(statistics.median(q), 4), "p10": round(pick(0.1), 4),
                    "p90": round(pick(0.9), 4), "unit": "ms",
                    "warm_l2_ms": round(eager_ms, 4), "graph_replay_ms": round(graph_ms, 4)},
        "e2e": {"value": round(whole_job_value(tokens * e2e_steps, world, e2e_s), 1),
                "unit": "tokens/s", "h2d_bytes_per_step": x.numel() * 4,
                "d2h_bytes_per_step": out.numel() * 4,
                "ms_per_step": round(e2e_s / e2e_steps * 1e3, 4)},
        "gpu_launches": 3 * args.steps,
        "clocks": clocks.summary(),
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_reference_mha(args, w, world):
    """The oracle's layer on the whole base-shape input, as the reference arm."""
    from transformer_head_scaled_03_gb300.inputs import mha_inputs
    import oracle
    x, *Ws = mha_inputs(w)
    orc = oracle.default()
    for _ in range(args.warmup):
        orc.mha(x, x, *Ws, h=w.H)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        orc.mha(x, x, *Ws, h=w.H)
    total_s = time.perf_counter() - t0
    value = w.B * w.Lq * args.steps / total_s
    line = {
        "impl": "reference", "metric": MHA_METRIC, "value": round(value, 2), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_s / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "L": w.Lq, "D": w.D, "h": w.H, "mask": "none"},
        "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s",
                         "cores": orc.num_threads(), "kind": "oracle",
                         "sample": "the whole workload per step, fp64 oracle"},
        "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------ reference arm

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from transformer_head_scaled_03_gb300.inputs import WORKLOADS, sample_rows, sdpa_inputs

    w = workload_from_args(args)
    if w.kind == "decode":
        run_reference_decode(args, w, world)
        return
    if w.kind == "mha":
        run_reference_mha(args, w, world)
        return
    Q, K, V, lens, _ = sdpa_inputs(w)
    rows, per_head = oracle_sample(w, args.cpu_rows_per_head)
    for _ in range(args.warmup):
        oracle_cpu_baseline(w, Q, K, V, lens, rows[: max(1, rows.size // 8)])
    total_s, total_flops = 0.0, 0.0
    cores = 1
    for _ in range(args.steps):
        tf, dt, cores = oracle_cpu_baseline(w, Q, K, V, lens, rows)
        total_s += dt
        total_flops += tf * 1e12 * dt
    value = total_flops / total_s / 1e12
    sample = (f"per step, {sample_description(w, rows, per_head)} oracle (the CPU-baseline "
              f"leg's sample)")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_s / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": sdpa_config(w, lens, world, args.float_mask),
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_reference_decode(args, w, world):
    """The oracle on a seeded sample of (b, h) pairs of a decode workload,
    drawn on the host with the shared generator (only the sampled heads)."""
    from transformer_head_scaled_03_gb300.inputs import Draws
    n = min(16, w.B * w.H)
    g = Draws(w.seed + 5000)
    Q = g.normal((w.B * w.H, w.Lq, w.d))
    lens = Draws(w.seed).integers(w.len_range[0], w.len_range[1], w.B)
    # only the sampled heads' cache rows are drawn; the rest is never read
    bhs = Draws(w.seed + 4000).choice(w.B * w.H, n)
    Ks = g.normal((n, w.Lk, w.d))
    Vs = g.normal((n, w.Lk, w.d))
    lb = lens[bhs // w.H].astype(np.int32)
    import oracle
    orc = oracle.default()
    total_s, total_bytes = 0.0, 0.0
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        orc.sdpa(Q[bhs][:, None], Ks[:, None], Vs[:, None], mask_kind=w.mask, key_lengths=lb)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            total_s += dt
            total_bytes += 2.0 * w.d * (2.0 * float(np.sum(lb)) + 2.0 * n * w.Lq)
    value = total_bytes / total_s / 1e9
    sample = (f"every query row of {n} seeded (b, h) pairs per step, their cache rows "
              f"drawn on the host, fp64 oracle")
    line = {
        "impl": "reference", "metric": DECODE_METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_s / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "Lq": w.Lq, "cache": w.Lk, "d": w.d},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": orc.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", type=int, default=5, choices=[1, 2, 3, 4, 5, 6, 7, 8],
                    help="1: the fp32 base-shape layer; 2-5: attention workloads; "
                         "6-8: decode against a cache")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the batch size of a decode workload (profiling captures)")
    ap.add_argument("--seq", type=int, default=None,
                    help="override the sequence length (profiling captures)")
    ap.add_argument("--heads", type=int, default=None,
                    help="override the head count (profiling captures)")
    ap.add_argument("--float-mask", action="store_true",
                    help="pass the causal mask as an additive float mask [Lq, Lk]")
    ap.add_argument("--skip-mha", action="store_true")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--skip-decode", action="store_true")
    ap.add_argument("--skip-backward", action="store_true")
    ap.add_argument("--skip-workloads", action="store_true",
                    help="leave out the per-workload legs (workloads 1-4) of the default line")
    ap.add_argument("--cpu-rows-per-head", type=int, default=None,
                    help="query rows per head of the oracle's sample, for the CPU-baseline "
                         "leg and each reference-arm step (default: about 5 s of work)")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per launch of the fused kernel from an ncu capture")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)   # at least three untimed warm-up steps
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
