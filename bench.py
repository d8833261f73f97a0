#!/usr/bin/env python3
"""Benchmark of the DFlash draft block attention on GB300.

One step = one pass of the hot path over one batch of synthetic input: a
``dflash_attn_anchored`` call (validation, anchor-derived tile schedule,
TMA/tcgen05 attention with online softmax, epilogue) on the bf16 prefill
workload B=1 H=16 S=4096 nb=256 block_size=16 (Q=4096), d_nope=128, d_rope=64,
d_v=128, inputs N(0,1).  The metric is TFLOP/s over unmasked FLOPs
(2*(d_qk+d_v) per visible (query, key, head)).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--workload W] [--mode anchored|dense] [--pass forward|backward]
Under torchrun (N > 1) every rank runs the same workload on its own GPU
(independent replicas, weak scaling); timing is the max over ranks.

``--pass backward`` times the backward call instead (gradients of q, k_nope,
k_rope, v given the forward's out and lse), over 2*(3*d_qk + 2*d_v) FLOPs per
visible pair.

``--impl reference`` times the fp64 CPU oracle on the host cores on a bounded
sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from dflash_block_draft_gb300 import metrics, synth  # noqa: E402

WORKLOAD = "prefill_bf16"
METRIC = "DFlash block-attn TFLOP/s (unmasked FLOPs) & % of GB300 bf16 roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def workload_desc(d) -> str:
    return (f"{d['workload'].name}: B={d['B']} H={d['H']} S={d['S']} nb={d['nb']} block_size={d['block_size']} "
            f"Q={d['Q']} d_nope={d['d_nope']} d_rope={d['d_rope']} d_v={d['d_v']} anchored")


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------------------
# clocks during the timed region (NVML through ctypes; nvidia-smi as fallback)
# ---------------------------------------------------------------------------
_REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
            0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
            0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}


class ClockSampler:
    def __init__(self, torch_device_index: int = 0, period_s: float = 0.002):
        self.period = period_s
        self.samples = []  # (sm_mhz, reasons_mask)
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self._nvml = None
        self._h = None
        self._smi = None
        try:
            import torch
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            h = ctypes.c_void_p()
            uuid = "GPU-" + str(torch.cuda.get_device_properties(torch_device_index).uuid)
            if nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) != 0:
                raise OSError("no NVML handle")
            self._nvml, self._h = nv, h
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or nv.nvmlDeviceGetCurrentClocksThrottleReasons
            self._reasons_fn = fn
        except Exception:
            self._nvml = None

    def _sample_nvml(self):
        mhz, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        if self._nvml.nvmlDeviceGetClockInfo(self._h, 1, ctypes.byref(mhz)) != 0:
            return
        self._reasons_fn(self._h, ctypes.byref(rs))
        self.samples.append((mhz.value, rs.value))

    def _run(self):
        while not self._stop.is_set():
            self._sample_nvml()
            time.sleep(self.period)

    def start(self):
        if self._nvml is not None:
            self._sample_nvml()
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()
        else:
            try:
                self._smi = subprocess.Popen(
                    ["nvidia-smi", "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                     "--format=csv,noheader,nounits", "-lms", "100", "-i", "0"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except Exception:
                self._smi = None

    def stop(self):
        if self._thread is not None:
            self._stop.set()
            self._thread.join()
            self._sample_nvml()
        elif self._smi is not None:
            self._smi.terminate()
            out, _ = self._smi.communicate(timeout=5)
            for line in out.splitlines():
                try:
                    a, b, c = [x.strip() for x in line.split(",")]
                    self.samples.append((int(a), int(c, 16)))
                    self.max_mhz = int(b)
                except Exception:
                    pass

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "source": "unavailable"}
        mhz = [s[0] for s in self.samples]
        mask = 0
        for _, r in self.samples:
            mask |= r
        reasons = [name for bit, name in _REASONS.items() if mask & bit and bit != 0x1]
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(self.samples), "source": "nvml" if self._nvml is not None else "nvidia-smi"}


# ---------------------------------------------------------------------------
# distributed plumbing (replicas; the data path has no collective)
# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(units_per_rank: float, world: int, max_ms: float) -> float:
    """Whole-job throughput in units per second.  Every rank runs the same
    workload (replicas, weak scaling), so the job processes world x the units of
    one rank in the time of the slowest rank."""
    return world * units_per_rank / (max_ms / 1e3)


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------
# oracle timing (CPU baseline / reference arm)
# ---------------------------------------------------------------------------
def oracle_rows_flops(d, rows):
    counts = metrics.anchored_visible_counts(d["anchors"], d["S"], d["Q"], d["block_size"]).reshape(-1)
    return int(counts[rows].sum()) * d["H"] * metrics.flops_per_pair(d["d_nope"], d["d_rope"], d["d_v"])


def time_oracle(d, rows):
    import oracle
    t0 = time.perf_counter()
    oracle.anchored(d["q"], d["k_nope"], d["k_rope"], d["v"], d["anchors"], d["block_size"], rows=rows)
    dt = time.perf_counter() - t0
    return dt, oracle_rows_flops(d, rows), oracle.max_threads()


def cores_available() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    d = synth.make(WORKLOAD)
    # Each step: every 64th query row of the workload (all heads), ~1.3 GFLOP of oracle work.
    stride = 64
    rows = np.arange(0, d["B"] * d["Q"], stride, dtype=np.int64)
    for _ in range(args.warmup):
        time_oracle(d, rows)
    times, flops, threads = [], 0, 1
    for _ in range(args.steps):
        dt, fl, threads = time_oracle(d, rows)
        times.append(dt)
        flops = fl
    ms = 1e3 * sum(times) / len(times)
    value = flops / (ms / 1e3) / 1e12
    sample = (f"every {stride}th query row of {WORKLOAD} ({rows.size} rows x {d['H']} heads, "
              f"{flops / 1e9:.2f} GFLOP unmasked per step)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_desc(d), "l2": "n/a (host CPU)"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def to_dev(a, dtype, device):
    import torch
    a = np.ascontiguousarray(a)
    if dtype == "bf16":
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(a).to(device)


def run_ours(args):
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(device)
    import dflash_block_draft_gb300 as dfl
    dfl.load_library()

    workload, dense = args.workload, args.mode == "dense"
    backward = args.pass_ == "backward"
    d = synth.make(workload)
    B, Q, H, S, bs = d["B"], d["Q"], d["H"], d["S"], d["block_size"]
    dn, dr, dv = d["d_nope"], d["d_rope"], d["d_v"]
    work = metrics.anchored_work(d["anchors"], S, Q, H, bs, dn, dr, dv, esize=2)
    if dense:  # the mask is read once more; visibility is the same as the anchored rule's
        work["bytes"] += B * Q * (S + Q) * 2 - d["anchors"].size * 4
    host = {k: d[k] for k in ("q", "k_nope", "k_rope", "v")}
    dev = {k: to_dev(v, "bf16", device) for k, v in host.items()}
    anchors = torch.from_numpy(d["anchors"]).to(device)
    out = torch.empty((B, Q, H, dv), dtype=torch.bfloat16, device=device)
    mode_code = dfl.MODE_DENSE if dense else dfl.MODE_ANCHORED
    ws_bytes = dfl.dflash_attn_workspace_size(mode_code, B, H, S, Q, dn, dr, dv)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)  # 256 MiB > 129 MB L2
    mask = None
    if dense:  # the additive block mask, built on the device from the anchors (+ padding columns)
        mask = dfl.dflash_build_mask(anchors, bs, S, dtype=torch.bfloat16)
        if d.get("pad"):
            mask[:, :, :, S - d["pad"]:S] = float("-inf")

    def step():
        if dense:
            dfl.dflash_attn_dense(dev["q"], dev["k_nope"], dev["k_rope"], dev["v"], mask, out=out, workspace=ws,
                                  stream=stream)
        else:
            dfl.dflash_attn_anchored(dev["q"], dev["k_nope"], dev["k_rope"], dev["v"], anchors, bs, out=out,
                                     workspace=ws, stream=stream)

    if backward:
        # The backward step takes the forward's out and lse (computed here, once,
        # outside the timed region) and the output gradient dout.
        lse = torch.empty((B, H, Q), dtype=torch.float32, device=device)
        if dense:
            dfl.dflash_attn_dense(dev["q"], dev["k_nope"], dev["k_rope"], dev["v"], mask, out=out, lse=lse,
                                  workspace=ws, stream=stream)
        else:
            dfl.dflash_attn_anchored(dev["q"], dev["k_nope"], dev["k_rope"], dev["v"], anchors, bs, out=out,
                                     lse=lse, workspace=ws, stream=stream)
        dout = to_dev(synth.make_dout(d), "bf16", device)
        grads = tuple(torch.empty_like(dev[k]) for k in ("q", "k_nope", "k_rope", "v"))
        bmode = dfl.MODE_DENSE_BACKWARD if dense else dfl.MODE_ANCHORED_BACKWARD
        bws = torch.empty(dfl.dflash_attn_workspace_size(bmode, B, H, S, Q, dn, dr, dv), dtype=torch.uint8,
                          device=device)
        work = dict(work, flops=work["flops"] // metrics.flops_per_pair(dn, dr, dv)
                    * metrics.backward_flops_per_pair(dn, dr, dv))

        def step():  # noqa: F811
            if dense:
                dfl.dflash_attn_dense_backward(dev["q"], dev["k_nope"], dev["k_rope"], dev["v"], mask, out, lse,
                                               dout, grads=grads, workspace=bws, stream=stream)
            else:
                dfl.dflash_attn_anchored_backward(dev["q"], dev["k_nope"], dev["k_rope"], dev["v"], anchors, bs,
                                                  out, lse, dout, grads=grads, workspace=bws, stream=stream)

    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        step()
    torch.cuda.synchronize(device)
    if dfl.dflash_last_device_error() != 0:
        raise RuntimeError("device error during warm-up")

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = ClockSampler(device.index or 0)
    launches0 = dfl.dflash_kernel_launches()
    barrier(world)
    torch.cuda.synchronize(device)
    clocks.start()
    for k in range(args.steps):
        flush.zero_()  # L2 flushed between timed steps (outside the events)
        ev[k][0].record(stream)
        step()
        ev[k][1].record(stream)
    torch.cuda.synchronize(device)
    barrier(world)
    clocks.stop()
    launches = dfl.dflash_kernel_launches() - launches0
    times = [a.elapsed_time(b) for a, b in ev]
    ms = max_over_ranks(sum(times) / len(times), world, device)
    value = job_value(work["flops"], world, ms) / 1e12

    peaks, peak_src = load_peaks()
    # One kernel per step (anchored): the attention kernel is the whole step, so
    # its average launch duration is the per-step event time.  The dense entry
    # point adds the mask scan, whose time is included here.
    kernel_ms = sum(times) / len(times)
    achieved = work["flops"] / (kernel_ms / 1e3) / 1e12
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    traffic = load_traffic()

    # end to end through the public API from pinned host buffers
    headline = workload == WORKLOAD and not dense and not backward
    e2e = None
    if not args.no_e2e and headline:
        pinned = {k: torch.from_numpy(np.ascontiguousarray(v).view(np.int16)).view(torch.bfloat16).pin_memory()
                  for k, v in host.items()}
        an_h = torch.from_numpy(d["anchors"]).pin_memory()
        out_h = torch.empty((B, Q, H, dv), dtype=torch.bfloat16).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in pinned.values()) + an_h.numel() * 4
        d2h = out_h.numel() * out_h.element_size()

        # A serving loop overlaps transfers with compute: the inputs of step k+1
        # travel host->device and the output of step k-1 device->host while step k
        # computes (two device buffer sets; one stream per direction).  Every step
        # still copies all of its inputs in and its whole output out.
        bufs = []
        for _ in range(2):
            bset = {k: torch.empty_like(t) for k, t in dev.items()}
            bset["anchors"] = torch.empty_like(anchors)
            bset["out"] = torch.empty_like(out)
            bufs.append(bset)
        outs_h = [out_h, torch.empty_like(out_h).pin_memory()]
        h2d_stream, d2h_stream = torch.cuda.Stream(device), torch.cuda.Stream(device)
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_done = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]

        def e2e_steps(n):
            for k in range(n):
                bi = k % 2
                bset = bufs[bi]
                with torch.cuda.stream(h2d_stream):
                    if k >= 2:
                        h2d_stream.wait_event(ev_out[bi])  # step k-2 has computed and left
                    for name, t in pinned.items():
                        bset[name].copy_(t, non_blocking=True)
                    bset["anchors"].copy_(an_h, non_blocking=True)
                    ev_in[bi].record(h2d_stream)
                stream.wait_event(ev_in[bi])
                dfl.dflash_attn_anchored(bset["q"], bset["k_nope"], bset["k_rope"], bset["v"], bset["anchors"], bs,
                                         out=bset["out"], workspace=ws, stream=stream)
                ev_done[bi].record(stream)
                with torch.cuda.stream(d2h_stream):
                    d2h_stream.wait_event(ev_done[bi])
                    outs_h[bi].copy_(bset["out"], non_blocking=True)
                    ev_out[bi].record(d2h_stream)

        e2e_steps(4)
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(h2d_stream)
        e2e_steps(args.steps)
        h2d_stream.wait_stream(d2h_stream)
        h2d_stream.wait_stream(stream)
        e1.record(h2d_stream)
        torch.cuda.synchronize(device)
        e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, device)
        e2e = {"value": job_value(work["flops"], world, e_ms) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": e_ms,
               "overlap": "inputs of step k+1 in and output of step k-1 out while step k computes "
                          "(two device buffer sets, one stream per direction)"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and headline:
        # The whole workload (every query row, every head), repeated until about
        # 10 s of oracle time has accumulated.
        rows = np.arange(0, B * Q, dtype=np.int64)
        total_t, total_f, reps, threads = 0.0, 0, 0, 1
        while reps == 0 or total_t < 10.0:
            dt, fl, threads = time_oracle(d, rows)
            total_t += dt
            total_f += fl
            reps += 1
        cpu = {"value": total_f / total_t / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": f"the whole {WORKLOAD} workload ({rows.size} rows x {H} heads, {fl / 1e9:.1f} GFLOP "
                         f"unmasked) x {reps}, {total_t:.1f} s"}

    metric = METRIC
    if backward:
        metric = ("DFlash block-attn backward TFLOP/s (unmasked FLOPs, 2*(3*d_qk+2*d_v) per visible pair) "
                  "& % of GB300 bf16 roofline")
    line = {"metric": metric, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": workload_desc(d) + (" (dense mask entry point)" if dense else "")
                       + (" backward (dq, dk_nope, dk_rope, dv)" if backward else ""),
                       "l2": "flushed between timed steps (256 MiB write)",
                       "unmasked_flops_per_step": work["flops"], "algorithmic_bytes_per_step": work["bytes"],
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "traffic": traffic if headline else None,
                         "peak_source": f"bf16_tflops ({peak_src})",
                         "kernel": ("prep + dq + dk/dv + rope finish" + (" (+ mask scan)" if dense else ""))
                         if backward else ("mask scan + attention" if dense else "attention (one launch per step)")},
            "pct_bf16_roofline": 100.0 * achieved / peak,
            "e2e": e2e, "cpu_baseline": cpu, "gpu_launches": int(launches), "clocks": clocks.summary()}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_decode(args):
    """The ragged decode workload: 64 requests x 16 draft rows, contexts
    log-uniform in [1024, 32768], H=32.  HBM-bound: the roofline is bytes."""
    import torch
    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    import dflash_block_draft_gb300 as dfl
    dfl.load_library()
    d = synth.make("decode_bf16", **({"R": args.requests} if args.requests else {}))
    H, bs = d["H"], d["block_size"]
    work = metrics.ragged_work(d["q_offsets"], d["kv_offsets"], d["anchors"], H, bs, d["d_nope"], d["d_rope"],
                               d["d_v"])
    dev = {k: to_dev(d[k], "bf16", device) for k in ("q", "k_nope", "k_rope", "v")}
    qo, ko, an = (torch.from_numpy(d[k]).to(device) for k in ("q_offsets", "kv_offsets", "anchors"))
    out = torch.empty((d["total_q"], H, d["d_v"]), dtype=torch.bfloat16, device=device)
    nbytes = dfl.dflash_attn_workspace_size(dfl.MODE_RAGGED, H=H, d_nope=d["d_nope"], d_rope=d["d_rope"],
                                            d_v=d["d_v"], R=d["R"], total_q=d["total_q"], total_kv=d["total_kv"],
                                            max_q_len=16)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)

    def step():
        dfl.dflash_attn_ragged(dev["q"], dev["k_nope"], dev["k_rope"], dev["v"], qo, ko, an, bs, 16, out=out,
                               workspace=ws, stream=stream)

    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        step()
    torch.cuda.synchronize(device)
    if dfl.dflash_last_device_error() != 0:
        raise RuntimeError("device error during warm-up")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = ClockSampler(0)
    launches0 = dfl.dflash_kernel_launches()
    torch.cuda.synchronize(device)
    clocks.start()
    for k in range(args.steps):
        flush.zero_()
        ev[k][0].record(stream)
        step()
        ev[k][1].record(stream)
    torch.cuda.synchronize(device)
    clocks.stop()
    launches = dfl.dflash_kernel_launches() - launches0
    ms = sum(a.elapsed_time(b) for a, b in ev) / args.steps
    peaks, src = load_peaks()
    gbs = work["bytes"] / (ms / 1e3) / 1e9
    peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    line = {"metric": "DFlash block-attn ragged decode: algorithmic HBM GB/s (and unmasked TFLOP/s)",
            "value": gbs, "unit": "GB/s", "tflops": work["flops"] / (ms / 1e3) / 1e12, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"decode_bf16: R={d['R']} x 16 rows, H={H}, contexts log-uniform [1024,32768], "
                                   f"total_kv={d['total_kv']}", "l2": "flushed between timed steps (256 MiB write)",
                       "algorithmic_bytes_per_step": work["bytes"], "unmasked_flops_per_step": work["flops"]},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                         "traffic": load_traffic("decode_bf16", work["bytes"]), "peak_source": f"hbm_gbs ({src})",
                         "kernel": "plan + split attention + combine (one step; the attention kernel is 95 % of it)",
                         "traffic_note": "attn_decode_kernel DRAM bytes from a 16-request capture, scaled by "
                                         "algorithmic bytes"},
            "gpu_launches": int(launches), "clocks": clocks.summary()}
    print(json.dumps(line), flush=True)
    return 0


def load_traffic(key=None, alg_bytes=None):
    """DRAM bytes per launch of the attention kernel from the committed ncu
    summary, when it was taken on the kernel source as it is now; else None.
    A capture of a smaller case of the same recipe is scaled to this launch by
    its algorithmic bytes (traffic grows in proportion)."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        with open(p) as f:
            t = json.load(f).get(key or WORKLOAD)
        if not t:
            return None
        with open(os.path.join(ROOT, t["source"]), "rb") as f:
            if hashlib.md5(f.read()).hexdigest() != t["source_md5"]:
                return None  # kernel changed since the counters were taken
        if "algorithmic_bytes_of_capture" in t:
            if not alg_bytes:
                return None
            return int(round(t["bytes_per_launch"] * alg_bytes / t["algorithmic_bytes_of_capture"]))
        return int(t["bytes_per_launch"])
    except Exception:
        return None


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", choices=["prefill_bf16", "training_bf16", "long_bf16", "decode_bf16"],
                    default="prefill_bf16",
                    help="prefill_bf16 is the headline; the others are the remaining bf16 workloads "
                         "(decode_bf16 is HBM-bound and reported in GB/s)")
    ap.add_argument("--mode", choices=["anchored", "dense"], default="anchored",
                    help="entry point for the batched workloads")
    ap.add_argument("--pass", dest="pass_", choices=["forward", "backward"], default="forward",
                    help="batched workloads: time the forward call, or the backward call (gradients of "
                         "q, k_nope, k_rope, v) given the forward's out and lse")
    ap.add_argument("--requests", type=int, default=None,
                    help="decode_bf16 only: draw this many requests instead of 64 (same recipe; "
                         "for profiling captures that must stay small)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.workload == "decode_bf16":
        return run_decode(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
