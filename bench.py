#!/usr/bin/env python3
"""Benchmark of the DFlash draft block attention on GB300.

One step = one pass of the hot path over one batch of synthetic input.  The
headline is the largest single-GPU workload, bf16 long context: a
``dflash_attn_anchored`` call (validation, anchor-derived tile schedule,
TMA/tcgen05 attention with online softmax, epilogue) on B=2 H=16 S=32768
nb=2048 block_size=8 (Q=16384), d_nope=128, d_rope=64, d_v=128, inputs N(0,1),
the last 5 % of each row's context padding that no anchor reaches.  The metric
is TFLOP/s over unmasked FLOPs (2*(d_qk+d_v) per visible (query, key, head))
and its fraction of the measured bf16 dense tensor peak.

The same JSON line carries a ``per_config`` block: every other workload of the
suite measured the same way on the same GPU -- bf16 prefill and training
(anchored and dense-mask entry points), long context through the dense mask,
the ragged serving decode (algorithmic HBM GB/s against the measured HBM
peak), the same decode with keys and values as compressed MLA latents
(absorbed-form TFLOP/s) and the tiny fp32 case (its parity against the fp64
oracle, computed in the CPU-baseline leg).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--workload W] [--mode anchored|dense] [--pass forward|backward]
                       [--no-per-config] [--no-e2e] [--no-cpu-baseline]
Under torchrun (N > 1) every rank runs the same workload on its own GPU
(independent replicas, weak scaling); timing is the max over ranks, and the
per-config block is left out.

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

WORKLOAD = "long_bf16"  # the headline: the largest workload that fits one GPU
METRIC = "DFlash block-attn TFLOP/s (unmasked FLOPs) & % of GB300 bf16 roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# The rest of the suite, reported beside the headline: (workload, entry point).
PER_CONFIG = (("prefill_bf16", "anchored"), ("prefill_bf16", "dense"), ("training_bf16", "anchored"),
              ("training_bf16", "dense"), ("long_bf16", "dense"), ("decode_bf16", "ragged"),
              ("decode_latent_bf16", "latent"), ("prefill_bf16", "backward"), ("training_bf16", "backward"),
              ("long_bf16", "backward"), ("tiny_fp32", "anchored"))
# Targets: prefill-shaped workloads at >= 50 % of the bf16 tensor peak, the
# ragged decode at >= 60 % of HBM bandwidth.
TARGET_FRAC = {"tensor": 0.50, "hbm": 0.60}


def workload_desc(d, mode="anchored") -> str:
    w = d["workload"]
    if w.ragged:
        return (f"{w.name}: R={d['R']} requests x {w.nb * w.block_size} rows, "
                f"H={d['H']}, contexts log-uniform [{w.ctx_lo},{w.ctx_hi}], total_kv={d['total_kv']}")
    s = (f"{w.name}: B={d['B']} H={d['H']} S={d['S']} nb={d['nb']} block_size={d['block_size']} "
         f"Q={d['Q']} d_nope={d['d_nope']} d_rope={d['d_rope']} d_v={d['d_v']}")
    if d.get("pad"):
        s += f" pad={d['pad']}"
    return s + (" dense mask" if mode == "dense" else " anchored")


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
def block_stride(d, target_flops: float) -> int:
    """Stride over blocks so that every stride-th block of each batch row (plus
    the last) carries about target_flops of unmasked oracle work."""
    total = metrics.anchored_work(d["anchors"], d["S"], d["Q"], d["H"], d["block_size"], d["d_nope"],
                                  d["d_rope"], d["d_v"])["flops"]
    return max(1, int(total // max(target_flops, 1.0)))


def stratified_rows(d, stride: int):
    """Flat query rows (b*Q + i) of every stride-th block of each batch row,
    the first and the last block included; returns (rows, blocks per row)."""
    nb, bs, Q, B = d["nb"], d["block_size"], d["Q"], d["B"]
    blocks = np.unique(np.concatenate([np.arange(0, nb, stride), [nb - 1]]))
    per_b = (blocks[:, None] * bs + np.arange(bs)[None, :]).reshape(-1)
    rows = (np.arange(B)[:, None] * Q + per_b[None, :]).reshape(-1)
    return rows.astype(np.int64), int(blocks.size)


def oracle_rows_flops(d, rows):
    counts = metrics.anchored_visible_counts(d["anchors"], d["S"], d["Q"], d["block_size"]).reshape(-1)
    return int(counts[rows].sum()) * d["H"] * metrics.flops_per_pair(d["d_nope"], d["d_rope"], d["d_v"])


def time_oracle(d, rows):
    import oracle
    t0 = time.perf_counter()
    oracle.anchored(d["q"], d["k_nope"], d["k_rope"], d["v"], d["anchors"], d["block_size"], rows=rows)
    dt = time.perf_counter() - t0
    return dt, oracle_rows_flops(d, rows), oracle.max_threads()


def cpu_baseline_leg(d, tiny_gpu=None, min_seconds=8.0):
    """The CPU baseline: the fp64 oracle, as it stands, on the host cores, over a
    deterministic stratified sample of the headline workload (about 8 s of
    work, repeated until min_seconds have passed).  When tiny_gpu holds the GPU
    outputs of the tiny fp32 workload, the oracle also evaluates that workload
    and the leg reports the GPU's max abs error against it."""
    stride = block_stride(d, 150e9)
    rows, nblk = stratified_rows(d, stride)
    total_t, total_f, reps, threads = 0.0, 0, 0, 1
    while reps == 0 or total_t < min_seconds:
        dt, fl, threads = time_oracle(d, rows)
        total_t += dt
        total_f += fl
        reps += 1
    all_flops = metrics.anchored_work(d["anchors"], d["S"], d["Q"], d["H"], d["block_size"], d["d_nope"],
                                      d["d_rope"], d["d_v"])["flops"]
    cpu = {"value": total_f / total_t / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
           "sample": (f"{d['workload'].name}: every {stride}th block of each batch row, first and last included "
                      f"({nblk} of {d['nb']} blocks per row, {rows.size} query rows x {d['H']} heads, "
                      f"{fl / 1e9:.1f} GFLOP unmasked = {100.0 * fl / all_flops:.2f} % of the workload) "
                      f"x {reps}, {total_t:.1f} s")}
    parity = None
    if tiny_gpu is not None:
        import oracle
        t = tiny_gpu["inputs"]
        want_o, want_l = oracle.anchored(t["q"], t["k_nope"], t["k_rope"], t["v"], t["anchors"], t["block_size"])
        eo = float(np.abs(tiny_gpu["out"] - want_o).max())
        el = float(np.abs(tiny_gpu["lse"] - want_l).max())
        parity = {"max_abs_err_out": eo, "max_abs_err_lse": el, "tol": 1e-5, "ok": bool(max(eo, el) <= 1e-5)}
    return cpu, parity


def cores_available() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    if args.workload == "decode_bf16":
        return run_reference_decode(args, world)
    d = synth.make(args.workload)
    # Each step: a stratified sample of about 5 GFLOP of oracle work.
    stride = block_stride(d, 5e9)
    rows, nblk = stratified_rows(d, stride)
    for _ in range(args.warmup):
        time_oracle(d, rows)
    times, flops, threads = [], 0, 1
    for _ in range(args.steps):
        dt, fl, threads = time_oracle(d, rows)
        times.append(dt)
        flops = fl
    ms = 1e3 * sum(times) / len(times)
    value = flops / (ms / 1e3) / 1e12
    sample = (f"every {stride}th block of each batch row of {args.workload}, first and last included "
              f"({nblk} blocks per row, {rows.size} query rows x {d['H']} heads, {flops / 1e9:.2f} GFLOP "
              f"unmasked per step)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_desc(d, args.mode), "l2": "n/a (host CPU)"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_reference_decode(args, world):
    import oracle
    d = synth.make("decode_bf16")
    H = d["H"]
    qo, ko = d["q_offsets"], d["kv_offsets"]
    reqs = np.arange(0, d["R"], 16)  # every 16th request, all its rows
    rows = np.concatenate([np.arange(qo[r], qo[r + 1]) for r in reqs]).astype(np.int64)
    work = metrics.ragged_work(qo, ko, d["anchors"], H, d["block_size"], d["d_nope"], d["d_rope"], d["d_v"])
    frac = sum(int(ko[r + 1] - ko[r]) for r in reqs) / float(ko[-1])
    nbytes = work["bytes"] * frac

    def one():
        t0 = time.perf_counter()
        oracle.ragged(d["q"], d["k_nope"], d["k_rope"], d["v"], qo, ko, d["anchors"], d["block_size"], rows=rows)
        return time.perf_counter() - t0

    for _ in range(args.warmup):
        one()
    ms = 1e3 * sum(one() for _ in range(args.steps)) / args.steps
    value = nbytes / (ms / 1e3) / 1e9
    line = {"impl": "reference", "metric": "DFlash block-attn ragged decode: algorithmic HBM GB/s",
            "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": workload_desc(d), "l2": "n/a (host CPU)"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.max_threads(), "kind": "oracle",
                             "sample": f"every 16th request ({reqs.size} of {d['R']}), all rows and heads"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
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


def timed_loop(step, steps, warmup, device, stream, flush, world, dfl):
    """W untimed warm-up steps, then K steps each bracketed by CUDA events on the
    launching stream with an L2 flush (outside the events) before each.  Returns
    (per-step event times in ms, launches in the timed region, clock summary)."""
    import torch
    for _ in range(max(warmup, 3)):
        flush.zero_()
        step()
    torch.cuda.synchronize(device)
    if dfl.dflash_last_device_error() != 0:
        raise RuntimeError("device error during warm-up")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    clocks = ClockSampler(device.index or 0)
    launches0 = dfl.dflash_kernel_launches()
    barrier(world)
    torch.cuda.synchronize(device)
    clocks.start()
    for k in range(steps):
        flush.zero_()  # L2 flushed between timed steps (outside the events)
        ev[k][0].record(stream)
        step()
        ev[k][1].record(stream)
    torch.cuda.synchronize(device)
    barrier(world)
    clocks.stop()
    launches = dfl.dflash_kernel_launches() - launches0
    if dfl.dflash_last_device_error() != 0:
        raise RuntimeError("device error in the timed region")
    return [a.elapsed_time(b) for a, b in ev], int(launches), clocks.summary()


def measure_batched(dfl, d, mode, backward, steps, warmup, device, world, peaks, e2e=False, keep_out=False):
    """One workload of the batched entry points (anchored or dense mask), forward
    or backward.  Returns the measurement as a dict."""
    import torch
    dense = mode == "dense"
    dt = "bf16" if d["dtype"] == "bf16" else "fp32"
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    esize = 2 if dt == "bf16" else 4
    B, Q, H, S, bs = d["B"], d["Q"], d["H"], d["S"], d["block_size"]
    dn, dr, dv = d["d_nope"], d["d_rope"], d["d_v"]
    work = metrics.anchored_work(d["anchors"], S, Q, H, bs, dn, dr, dv, esize=esize)
    if dense:  # the mask is read once more; visibility is the same as the anchored rule's
        work["bytes"] += B * Q * (S + Q) * esize - d["anchors"].size * 4
    host = {k: d[k] for k in ("q", "k_nope", "k_rope", "v")}
    dev = {k: to_dev(v, dt, device) for k, v in host.items()}
    anchors = torch.from_numpy(d["anchors"]).to(device)
    out = torch.empty((B, Q, H, dv), dtype=tdt, device=device)
    lse = torch.empty((B, H, Q), dtype=torch.float32, device=device) if (keep_out or backward) else None
    mode_code = dfl.MODE_DENSE if dense else dfl.MODE_ANCHORED
    code = dfl.DFLASH_BF16 if dt == "bf16" else dfl.DFLASH_FP32
    ws = torch.empty(max(dfl.dflash_attn_workspace_size(mode_code, B, H, S, Q, dn, dr, dv, code), 1),
                     dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)  # 256 MiB > 129 MB L2
    mask = None
    if dense:  # the additive block mask, built on the device from the anchors (+ padding columns)
        mask = dfl.dflash_build_mask(anchors, bs, S, dtype=tdt)
        if d.get("pad"):
            mask[:, :, :, S - d["pad"]:S] = float("-inf")

    def fwd(o=out, l=lse):
        if dense:
            dfl.dflash_attn_dense(dev["q"], dev["k_nope"], dev["k_rope"], dev["v"], mask, out=o, lse=l,
                                  workspace=ws, stream=stream)
        else:
            dfl.dflash_attn_anchored(dev["q"], dev["k_nope"], dev["k_rope"], dev["v"], anchors, bs, out=o, lse=l,
                                     workspace=ws, stream=stream)

    step, kernel = fwd, ("mask scan + attention" if dense else "attention (one launch per step)")
    if backward:
        # The backward step takes the forward's out and lse (computed here, once,
        # outside the timed region) and the output gradient dout.
        fwd()
        dout = to_dev(synth.make_dout(d), dt, device)
        grads = tuple(torch.empty_like(dev[k]) for k in ("q", "k_nope", "k_rope", "v"))
        bmode = dfl.MODE_DENSE_BACKWARD if dense else dfl.MODE_ANCHORED_BACKWARD
        bws = torch.empty(dfl.dflash_attn_workspace_size(bmode, B, H, S, Q, dn, dr, dv, code), dtype=torch.uint8,
                          device=device)
        work = dict(work, flops=work["flops"] // metrics.flops_per_pair(dn, dr, dv)
                    * metrics.backward_flops_per_pair(dn, dr, dv))
        kernel = "prep + dq + dk/dv + rope finish" + (" (+ mask scan)" if dense else "")

        def step():
            if dense:
                dfl.dflash_attn_dense_backward(dev["q"], dev["k_nope"], dev["k_rope"], dev["v"], mask, out, lse,
                                               dout, grads=grads, workspace=bws, stream=stream)
            else:
                dfl.dflash_attn_anchored_backward(dev["q"], dev["k_nope"], dev["k_rope"], dev["v"], anchors, bs,
                                                  out, lse, dout, grads=grads, workspace=bws, stream=stream)

    times, launches, clocks = timed_loop(step, steps, warmup, device, stream, flush, world, dfl)
    kernel_ms = sum(times) / len(times)
    ms = max_over_ranks(kernel_ms, world, device)
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    sustained = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    achieved = work["flops"] / (kernel_ms / 1e3) / 1e12
    res = {"workload": workload_desc(d, mode) + (" backward (dq, dk_nope, dk_rope, dv)" if backward else ""),
           "value": job_value(work["flops"], world, ms) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms,
           "steps": steps, "unmasked_flops_per_step": work["flops"], "algorithmic_bytes_per_step": work["bytes"],
           "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                        "frac": achieved / peak, "frac_of_sustained": achieved / sustained, "kernel": kernel},
           "gpu_launches": launches, "clocks": clocks}
    if dt == "bf16" and not backward:
        res["target"] = {"frac": TARGET_FRAC["tensor"], "met": bool(achieved / peak >= TARGET_FRAC["tensor"])}
    if keep_out:
        fwd()
        torch.cuda.synchronize(device)
        res["_out"] = out.double().cpu().numpy()
        res["_lse"] = lse.double().cpu().numpy()
    if e2e and not dense and not backward:
        res["e2e"] = measure_e2e(dfl, d, dev, anchors, out, ws, stream, device, world, work, steps, dt)
    return res


def measure_e2e(dfl, d, dev, anchors, out, ws, stream, device, world, work, steps, dt):
    """The same metric end to end through the public API from pinned host
    buffers: every step copies its inputs host->device and its output back."""
    import torch
    bs = d["block_size"]
    host = {k: np.ascontiguousarray(d[k]) for k in ("q", "k_nope", "k_rope", "v")}
    if dt == "bf16":
        pinned = {k: torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).pin_memory() for k, v in host.items()}
    else:
        pinned = {k: torch.from_numpy(v).pin_memory() for k, v in host.items()}
    an_h = torch.from_numpy(d["anchors"]).pin_memory()
    out_h = torch.empty(tuple(out.shape), dtype=out.dtype).pin_memory()
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
    e2e_steps(steps)
    h2d_stream.wait_stream(d2h_stream)
    h2d_stream.wait_stream(stream)
    e1.record(h2d_stream)
    torch.cuda.synchronize(device)
    e_ms = max_over_ranks(e0.elapsed_time(e1) / steps, world, device)
    return {"value": job_value(work["flops"], world, e_ms) / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": e_ms,
            "overlap": "inputs of step k+1 in and output of step k-1 out while step k computes "
                       "(two device buffer sets, one stream per direction)"}


def measure_decode(dfl, steps, warmup, device, world, peaks, requests=None):
    """The ragged decode workload: 64 requests x 16 draft rows, contexts
    log-uniform in [1024, 32768], H=32.  HBM-bound: the roofline is bytes."""
    import torch
    d = synth.make("decode_bf16", **({"R": requests} if requests else {}))
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

    times, launches, clocks = timed_loop(step, steps, warmup, device, stream, flush, world, dfl)
    kernel_ms = sum(times) / len(times)
    ms = max_over_ranks(kernel_ms, world, device)
    peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    gbs = work["bytes"] / (kernel_ms / 1e3) / 1e9
    return {"workload": workload_desc(d), "value": job_value(work["bytes"], world, ms) / 1e9, "unit": "GB/s",
            "tflops": work["flops"] / (kernel_ms / 1e3) / 1e12, "ms_per_step": ms, "steps": steps,
            "algorithmic_bytes_per_step": work["bytes"], "unmasked_flops_per_step": work["flops"],
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                         "traffic": load_traffic("decode_bf16", work["bytes"]),
                         "kernel": "plan + split attention + combine (one step; the attention kernel is 95 % of it)",
                         "traffic_note": "attn_decode_kernel DRAM bytes from a 16-request capture, scaled by "
                                         "algorithmic bytes"},
            "target": {"frac": TARGET_FRAC["hbm"], "met": bool(gbs / peak >= TARGET_FRAC["hbm"])},
            "gpu_launches": launches, "clocks": clocks}


def measure_latent(dfl, steps, warmup, device, world, peaks, requests=None):
    """The decode workload with keys and values as compressed latents (kv_lora_rank
    512): query absorption, latent attention, split merge and output projection.
    Bound by the tensor cores: the roofline is the absorbed form's FLOPs."""
    import torch
    d = synth.make("decode_latent_bf16", **({"R": requests} if requests else {}))
    H, bs, rank = d["H"], d["block_size"], d["kv_rank"]
    work = metrics.latent_work(d["q_offsets"], d["kv_offsets"], d["anchors"], H, bs, d["d_nope"], d["d_rope"],
                               d["d_v"], rank)
    dev = {k: to_dev(d[k], "bf16", device) for k in ("q", "c_kv", "k_rope", "w_kv_b")}
    qo, ko, an = (torch.from_numpy(d[k]).to(device) for k in ("q_offsets", "kv_offsets", "anchors"))
    out = torch.empty((d["total_q"], H, d["d_v"]), dtype=torch.bfloat16, device=device)
    nbytes = dfl.dflash_attn_latent_workspace_size(d["R"], H, d["d_nope"], d["d_rope"], d["d_v"], rank,
                                                   dfl.DFLASH_BF16, d["total_q"], d["total_kv"], 16)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)

    def step():
        dfl.dflash_attn_latent_ragged(dev["q"], dev["c_kv"], dev["k_rope"], dev["w_kv_b"], qo, ko, an, bs, 16,
                                      out=out, workspace=ws, stream=stream)

    times, launches, clocks = timed_loop(step, steps, warmup, device, stream, flush, world, dfl)
    kernel_ms = sum(times) / len(times)
    ms = max_over_ranks(kernel_ms, world, device)
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    achieved = work["flops"] / (kernel_ms / 1e3) / 1e12
    return {"workload": workload_desc(d) + f", kv_rank={rank} (compressed latents)",
            "value": job_value(work["flops"], world, ms) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms,
            "steps": steps, "gbs": work["bytes"] / (kernel_ms / 1e3) / 1e9,
            "unmasked_flops_per_step": work["flops"], "algorithmic_bytes_per_step": work["bytes"],
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "traffic": load_traffic("decode_latent_bf16", work["bytes"]),
                         "kernel": "q absorption GEMM + split plan + latent attention + merge + output projection GEMM",
                         "flops_note": "2*(kv_rank+d_rope) + 2*kv_rank per visible (row, key, head), plus "
                                       "2*kv_rank*(d_nope+d_v) per (row, head)"},
            "gpu_launches": launches, "clocks": clocks}


def release_memory():
    import gc

    import torch
    gc.collect()
    torch.cuda.empty_cache()


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
    peaks, peak_src = load_peaks()
    backward = args.pass_ == "backward"

    if args.workload == "decode_bf16":
        head = measure_decode(dfl, args.steps, args.warmup, device, world, peaks, args.requests)
        metric = "DFlash block-attn ragged decode: algorithmic HBM GB/s (and unmasked TFLOP/s)"
        d_head = None
        head["roofline"]["peak_source"] = f"hbm_gbs ({peak_src})"
    elif args.workload == "decode_latent_bf16":
        head = measure_latent(dfl, args.steps, args.warmup, device, world, peaks, args.requests)
        metric = "DFlash block-attn compressed-latent decode: TFLOP/s (absorbed-form FLOPs)"
        d_head = None
        head["roofline"]["peak_source"] = f"bf16_tflops ({peak_src})"
    else:
        d_head = synth.make(args.workload, **({"H": args.heads} if args.heads else {}))
        head = measure_batched(dfl, d_head, args.mode, backward, args.steps, args.warmup, device, world, peaks,
                               e2e=not args.no_e2e)
        metric = METRIC
        if backward:
            metric = ("DFlash block-attn backward TFLOP/s (unmasked FLOPs, 2*(3*d_qk+2*d_v) per visible pair) "
                      "& % of GB300 bf16 roofline")
        head["roofline"]["peak_source"] = f"bf16_tflops ({peak_src}); frac_of_sustained against bf16_tflops_sustained"
        key = args.workload if args.mode == "anchored" else f"{args.workload}:dense"
        head["roofline"]["traffic"] = None if backward else load_traffic(key)
    release_memory()

    headline = args.workload == WORKLOAD and args.mode == "anchored" and not backward and not args.heads
    per_config, tiny = None, None
    if headline and world == 1 and not args.no_per_config:
        per_config = {}
        for w, mode in PER_CONFIG:
            if w == "decode_bf16":
                r = measure_decode(dfl, args.steps, args.warmup, device, 1, peaks)
            elif w == "decode_latent_bf16":
                r = measure_latent(dfl, args.steps, args.warmup, device, 1, peaks)
            elif mode == "backward":  # the anchored backward, given the forward's out and lse
                dw = synth.make(w)
                r = measure_batched(dfl, dw, "anchored", True, args.steps, args.warmup, device, 1, peaks)
                del dw
            else:
                dw = synth.make(w)
                r = measure_batched(dfl, dw, mode, False, args.steps, args.warmup, device, 1, peaks,
                                    keep_out=w == "tiny_fp32")
                if w == "tiny_fp32":
                    tiny = {"inputs": dw, "out": r.pop("_out"), "lse": r.pop("_lse")}
                    r["roofline"] = {"bound": "none (parity only)", "note": "fp32 exactness path (CUDA cores)"}
                    r.pop("target", None)
                else:
                    key = w if mode == "anchored" else f"{w}:dense"
                    r["roofline"]["traffic"] = load_traffic(key)
                del dw
            per_config[f"{w}:{mode}"] = r
            release_memory()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and headline:
        cpu, parity = cpu_baseline_leg(d_head, tiny)
        if parity is not None and per_config is not None:
            per_config["tiny_fp32:anchored"]["parity"] = parity

    line = {"metric": metric, "value": head["value"], "unit": head["unit"], "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": head["workload"], "l2": "flushed between timed steps (256 MiB write)",
                       "unmasked_flops_per_step": head["unmasked_flops_per_step"],
                       "algorithmic_bytes_per_step": head["algorithmic_bytes_per_step"],
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "roofline": head["roofline"],
            "e2e": head.get("e2e"), "cpu_baseline": cpu, "gpu_launches": head["gpu_launches"],
            "clocks": head["clocks"]}
    if head["roofline"]["unit"] == "TFLOP/s":
        line["pct_bf16_roofline"] = 100.0 * head["roofline"]["frac"]
    if "target" in head:
        line["target"] = head["target"]
    if per_config is not None:
        line["per_config"] = per_config
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
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
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="measure the headline workload only (no per_config block)")
    ap.add_argument("--workload", choices=["long_bf16", "prefill_bf16", "training_bf16", "decode_bf16",
                                           "decode_latent_bf16", "tiny_fp32"],
                    default=WORKLOAD,
                    help="long_bf16 (the largest workload) is the headline; the others are the rest of the suite "
                         "(decode_bf16 is HBM-bound and reported in GB/s)")
    ap.add_argument("--mode", choices=["anchored", "dense"], default="anchored",
                    help="entry point for the batched workloads")
    ap.add_argument("--pass", dest="pass_", choices=["forward", "backward"], default="forward",
                    help="batched workloads: time the forward call, or the backward call (gradients of "
                         "q, k_nope, k_rope, v) given the forward's out and lse")
    ap.add_argument("--heads", type=int, default=None,
                    help="batched workloads only: use this many heads instead of the workload's (same recipe "
                         "otherwise; for profiling captures that must stay small)")
    ap.add_argument("--requests", type=int, default=None,
                    help="decode workloads only: draw this many requests instead of 64 (same recipe; "
                         "for profiling captures that must stay small)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
