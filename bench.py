"""Benchmark of the HSTU attention forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl cuda|reference]

One step = one forward (scheduler + persistent tcgen05 kernel [+ combine]) over
the large jagged workload: B=64 sequences, nhead 4, bf16, UIH lengths
U_int[1024, 4096], targets U_int[1, 32], context 6, full causal, hdim 128
(repeated at hdim 256, 96 and 96/64 in the same run; with a relative
attention bias under "rab"; and the backward of the hdim 128 case under
"backward"), synthetic N(0,1) inputs, seed 7.
Prints one JSON line (rank 0).  Metric: useful TFLOP/s = 2 (hdim_qk + hdim_v)
x allowed (i, j) pairs / step time.

Multi-GPU (torchrun): every rank runs its own batch of the same shape (seed
7 + rank); no collective touches the data path ("scaling": "weak").  The time
is the max over ranks; value = all ranks' useful FLOPs / that time.

--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload on the host cores (rank 0 only).
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from recommender_attention_gb300 import workloads as W  # noqa: E402

METRIC = "HSTU fwd useful TFLOP/s (unmasked pairs) at 1 GB300 and % of bf16 dense peak"
UNIT = "TFLOP/s"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "hstu_fwd_large_jagged_d128_dram.txt")
KERNEL_SOURCES = ["hstu_fwd_kernel.cuh", "hstu_common.cuh", "ptx.cuh", "hstu_fwd_d128.cu"]


# ---------------------------------------------------------------- distributed plumbing
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def rank_workload(rank: int, hdim: int = 128) -> W.Workload:
    """Rank r's shard: the large jagged shape with its own seed (weak scaling)."""
    return W.large_jagged(hdim=hdim, seed=7 + rank)


def reduce_max(value: float, world: int, device=None) -> float:
    if world == 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(value: float, world: int, device=None) -> float:
    if world == 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- peaks, clocks, traffic
def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for r in csv.reader(f):
                if len(r) >= 9:
                    rows.append([x.strip() for x in r])
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        busy = [s for s in sm if smax and s > 0.3 * max(smax)] or sm
        return {"sm_mhz": statistics.median(busy) if busy else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows),
                "power_w_max": max((float(r[3]) for r in rows if _isnum(r[3])), default=None)}


def _isnum(x):
    try:
        float(x)
        return True
    except ValueError:
        return False


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "recommender_attention_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic():
    """DRAM bytes per launch of the forward kernel from the committed ncu summary,
    when it was taken on the current kernel sources; else None."""
    try:
        kv = {}
        with open(TRAFFIC_FILE) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("kernel_source_hash") != kernel_source_hash():
            return None
        return int(float(kv["dram_bytes_per_launch"]))
    except (OSError, KeyError, ValueError):
        return None


# ---------------------------------------------------------------- the workload's description
def workload_config(w, allowed_pairs: int, world: int) -> dict:
    """The `config` of both arms' lines: what the workload is, nothing about
    how an implementation runs it (split counts and tile counts go elsewhere)."""
    tok = w.total_q
    in_out = 2 * w.nhead * tok * (2 * w.hdim_qk + 2 * w.hdim_v)
    return {"workload": f"large jagged SiLU HSTU self-attention, hdim {w.hdim_qk}",
            "batch": w.batch, "nhead": w.nhead, "hdim_qk": w.hdim_qk, "hdim_v": w.hdim_v,
            "uih": "U_int[1024,4096]", "targets": "U_int[1,32]", "context_len": 6, "local_len": 0,
            "minfull_len": 0, "causal": 1, "total_tokens": tok, "allowed_pairs": int(allowed_pairs),
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": "inputs larger than L2 (q+k+v+o %.0f MB > 129 MB)" % (in_out / 1e6)}


# ---------------------------------------------------------------- CUDA arm
def device_call(w, q, k, v, device, cta_pairs: int = 0):
    from recommender_attention_gb300.hstu import HstuCall
    off_q = torch.from_numpy(w.seq_offsets_q()).to(device)
    tg = torch.from_numpy(w.num_targets()).to(device)
    dq, dk, dv = q.to(device), k.to(device), v.to(device)
    call = HstuCall(dq, dk, dv, off_q, None, tg, alpha=w.alpha, attn_scale=list(w.attn_scale),
                    causal=w.causal, local_len=list(w.local_len), context_len=list(w.context_len),
                    minfull_len=list(w.minfull_len), max_uih_len=list(w.max_uih_len),
                    num_groups=w.num_groups, softmax=w.softmax,
                    max_seqlen_q=int(w.lengths_q().max()), max_seqlen_kv=int(w.lengths_kv().max()),
                    cta_pairs=cta_pairs)
    return call, (dq, dk, dv, off_q, tg)


def time_device_steps(call, steps, warmup, world, stream):
    """K whole steps back to back (the metric), then K more with events around
    the forward kernel alone (the roofline's kernel time).  The per-kernel
    events sit between the scheduler and the forward launch, where they would
    stop the forward kernel's prologue from overlapping the scheduler, so the
    step pass records none."""
    for _ in range(warmup):
        call.launch(stream)
    call.check(stream)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(steps):
        call.launch(stream)
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    step_ms = start.elapsed_time(end) / steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for a, b in ev:   # materialise the event handles
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize()
    for i in range(steps):
        call.launch(stream, events=ev[i])
    torch.cuda.synchronize()
    fwd_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    call.check(stream)
    return step_ms, fwd_ms


def time_sustained(call, stream, step_ms: float, seconds: float, gpu_index: int, world: int):
    """The headline step back to back for about `seconds` (long enough for the
    power cap and clocks to settle), with its own clock samples.  Returns
    (ms per step, steps, clock summary)."""
    n = max(20, int(seconds / (step_ms * 1e-3)))
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier(world)
    with ClockSampler(gpu_index) as clk:
        start.record(stream)
        for _ in range(n):
            call.launch(stream)
        end.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    call.check(stream)
    return start.elapsed_time(end) / n, n, clk.summary()


def small_config_lines(device, stream, steps: int, warmup: int, hbm_peak: float, only=None):
    """The other workloads of the scope (tiny, jagged, batched, group cross
    split-KV in SiLU and softmax, an M-FALCON candidate microbatch over cached
    history keys): one whole call (scheduler + forward [+ combine]) timed with CUDA events on the launching stream, L2 flushed
    between calls (their inputs fit in L2).  Reported as useful TFLOP/s and
    algorithmic HBM GB/s (q, k, v read once, o and lse written once)."""
    from recommender_attention_gb300.hstu import HstuCall
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    cases = [("tiny", W.tiny_batched(), {}), ("jagged", W.jagged_readme(), {}),
             ("batched", W.batched_default(), {}),
             ("group_cross_splitkv_silu", W.group_cross_splitkv(softmax=False), {}),
             ("group_cross_splitkv_softmax", W.group_cross_splitkv(softmax=True), {}),
             ("mfalcon_microbatch", W.mfalcon(), {})]
    # the split-KV workload with the split count forced, beside the automatic choice
    for splits in (2, 4):
        for sm in (False, True):
            cases.append((f"group_cross_splitkv_{'softmax' if sm else 'silu'}_splits{splits}",
                          W.group_cross_splitkv(softmax=sm), {"num_splits": splits}))
    if only:
        unknown = set(only) - {c[0] for c in cases}
        if unknown:
            raise SystemExit(f"unknown scope workload(s): {sorted(unknown)}")
        cases = [c for c in cases if c[0] in only]
    out = {}
    for name, w, over in cases:
        q, k, v = w.tensors()
        off_q = torch.from_numpy(w.seq_offsets_q()).to(device)
        okv = w.seq_offsets_kv()
        off_kv = torch.from_numpy(okv).to(device) if okv is not None else None
        tg = w.num_targets()
        tg = torch.from_numpy(tg).to(device) if tg is not None else None
        dq, dk, dv = q.to(device), k.to(device), v.to(device)
        call = HstuCall(dq, dk, dv, off_q, off_kv, tg, alpha=w.alpha, attn_scale=list(w.attn_scale),
                        causal=w.causal, local_len=list(w.local_len), context_len=list(w.context_len),
                        minfull_len=list(w.minfull_len), max_uih_len=list(w.max_uih_len),
                        num_groups=w.num_groups, softmax=w.softmax,
                        max_seqlen_q=int(w.lengths_q().max()), max_seqlen_kv=int(w.lengths_kv().max()),
                        kv_targets=w.kv_targets, **over)
        st = call.stats(stream)
        for _ in range(warmup):
            call.launch(stream)
        call.check(stream)
        times = []
        for _ in range(steps):
            with torch.cuda.stream(stream):
                flush.fill_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call.launch(stream)
            b.record(stream)
            b.synchronize()
            times.append(a.elapsed_time(b))
        call.check(stream)
        ms = statistics.median(times)
        # the forward kernel alone (events between the scheduler and the forward
        # launch, which stop their overlap; the rest of the call is the
        # scheduler, the combine and the launch gaps)
        ktimes = []
        for _ in range(steps):
            with torch.cuda.stream(stream):
                flush.fill_(1)
            ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            ev[0].record(stream)
            ev[1].record(stream)
            call.launch(stream, events=ev)
            ev[1].synchronize()
            ktimes.append(ev[0].elapsed_time(ev[1]))
        call.check(stream)
        kms = statistics.median(ktimes)
        tq, tkv = dq.shape[0], dk.shape[0]
        nbytes = 2 * w.nhead * (tq * w.hdim_qk + tkv * (w.hdim_qk + w.hdim_v) + tq * w.hdim_v)
        if w.softmax:
            nbytes += 4 * w.nhead * tq
        flops = 2.0 * (w.hdim_qk + w.hdim_v) * st["allowed_pairs"]
        gbs = nbytes / (ms * 1e-3) / 1e9
        kgbs = nbytes / (kms * 1e-3) / 1e9
        out[name] = {"ms": ms, "tflops_useful": flops / (ms * 1e-3) / 1e12, "gbs_algorithmic": gbs,
                     "hbm_frac": gbs / hbm_peak, "algorithmic_bytes": nbytes,
                     "fwd_kernel_ms": kms, "fwd_kernel_hbm_frac": kgbs / hbm_peak,
                     "allowed_pairs": st["allowed_pairs"], "executed_tiles": st["executed_tiles"],
                     "num_splits": st["num_splits"], "timing": f"median of {steps}, L2 flushed between calls"}
        del call, dq, dk, dv
    del flush
    torch.cuda.empty_cache()
    return out


def rab_lines(rank, device, stream, steps: int, warmup: int, world: int, peak: float, cpu: bool):
    """The forward of the same large jagged workload (hdim 128) with a relative
    attention bias (per-token timestamps, an 11-bucket time table and a
    128-entry positional table per head; Workload.rab_inputs), SiLU and softmax.
    Useful FLOPs as the headline's (the bias adds no GEMM work)."""
    from recommender_attention_gb300.hstu import HstuCall
    out = {}
    for softmax in (False, True):
        w = rank_workload(rank, 128).with_(softmax=softmax, rab_pos_buckets=128)
        q, k, v = w.tensors()
        ts_q, _, rab_time, rab_pos = w.rab_inputs()
        dq, dk, dv = q.to(device), k.to(device), v.to(device)
        off_q = torch.from_numpy(w.seq_offsets_q()).to(device)
        tg = torch.from_numpy(w.num_targets()).to(device)
        call = HstuCall(dq, dk, dv, off_q, None, tg, alpha=w.alpha, attn_scale=list(w.attn_scale),
                        causal=w.causal, local_len=list(w.local_len), context_len=list(w.context_len),
                        minfull_len=list(w.minfull_len), max_uih_len=list(w.max_uih_len),
                        num_groups=w.num_groups, softmax=w.softmax,
                        max_seqlen_q=int(w.lengths_q().max()), max_seqlen_kv=int(w.lengths_kv().max()),
                        timestamps_q=torch.from_numpy(ts_q).to(device),
                        rab_time=torch.from_numpy(rab_time).to(device), rab_pos=torch.from_numpy(rab_pos).to(device))
        st = call.stats(stream)
        step_ms, fwd_ms = time_device_steps(call, steps, warmup, world, stream)
        step_ms = reduce_max(step_ms, world, device)
        flops = 2.0 * (w.hdim_qk + w.hdim_v) * st["allowed_pairs"]
        tot = reduce_sum(flops, world, device)
        kt = flops / (fwd_ms * 1e-3) / 1e12
        out["softmax" if softmax else "silu"] = {
            "value": tot / (step_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": step_ms,
            "fwd_kernel_ms": fwd_ms, "fwd_kernel_tflops": kt,
            "roofline": {"bound": "tensor", "achieved": kt, "peak": peak, "unit": "TFLOP/s", "frac": kt / peak,
                         "traffic": None, "kernel": "hstu_fwd_kernel<128,bf16,bias>"},
            "cpu_baseline": (cpu_baseline_rab(w, q, k, v, (ts_q, None, rab_time, rab_pos))
                             if cpu and rank == 0 else None)}
        del call, dq, dk, dv
        torch.cuda.empty_cache()
    return out


def backward_lines(rank, device, stream, steps: int, warmup: int, world: int, peak: float, cpu: bool):
    """The backward over the same large jagged workload (hdim 128; SiLU, and
    softmax fed the forward's own o and lse; SiLU with the relative attention
    bias, without and with the gradients of its tables): one step = one hstu_attn_bwd call
    (scheduler [+ row sums] + dQ kernel + dK/dV kernel), inputs and dO resident
    (larger than L2).  Useful FLOPs per allowed pair: 2 (3 hdim_qk + 2 hdim_v),
    the five products (S, dP, dV, dK, dQ) counted once; the two kernels
    recompute S and dP, so the executed count is 2 (5 hdim_qk + 4 hdim_v)."""
    from recommender_attention_gb300.hstu import HstuBwdCall
    out = {}
    for softmax, rab, rab_grads in ((False, False, False), (True, False, False), (False, True, False),
                                    (False, True, True)):
        w = rank_workload(rank, 128).with_(softmax=softmax, rab_pos_buckets=128 if rab else 0)
        q, k, v = w.tensors()
        call, (dq, dk, dv, off_q, tg) = device_call(w, q, k, v, device)
        bias = w.rab_inputs() if rab else None
        bias_kw = {} if not rab else dict(timestamps_q=torch.from_numpy(bias[0]).to(device),
                                          rab_time=torch.from_numpy(bias[2]).to(device),
                                          rab_pos=torch.from_numpy(bias[3]).to(device))
        st = call.stats(stream)
        call.launch(stream)
        call.check(stream)
        d_o = w.grad_output().to(device)
        bw = HstuBwdCall(dq, dk, dv, d_o, off_q, None, tg, o=call.o, lse=call.lse, alpha=w.alpha,
                         attn_scale=list(w.attn_scale), causal=w.causal, local_len=list(w.local_len),
                         context_len=list(w.context_len), minfull_len=list(w.minfull_len),
                         max_uih_len=list(w.max_uih_len), num_groups=w.num_groups, softmax=w.softmax,
                         max_seqlen_q=int(w.lengths_q().max()), max_seqlen_kv=int(w.lengths_kv().max()),
                         rab_grads=rab_grads, **bias_kw)
        for _ in range(warmup):
            bw.launch(stream)
        bw.check(stream)
        torch.cuda.synchronize()
        barrier(world)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            bw.launch(stream)
        b.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        bw.check(stream)
        ms = reduce_max(a.elapsed_time(b) / steps, world, device)
        # useful: S, dP, dV, dQ, dK once per allowed pair; executed: both
        # kernels form S and dP, the dQ kernel dQ, the dK/dV kernel dV and dK
        useful = 2.0 * (3 * w.hdim_qk + 2 * w.hdim_v) * st["allowed_pairs"]
        executed = 2.0 * 128 * 128 * (4 * w.hdim_qk + 3 * w.hdim_v) * st["executed_tiles"]
        tot = reduce_sum(useful, world, device)
        tf = tot / (ms * 1e-3) / 1e12
        per_gpu = useful / (ms * 1e-3) / 1e12
        out[("softmax" if softmax else "silu") + ("_rab" if rab else "") + ("_grads" if rab_grads else "")] = {
            "value": tf, "unit": "TFLOP/s", "ms_per_step": ms, "pct_of_bf16_peak": 100.0 * tf / world / peak,
            "executed_tflops": reduce_sum(executed, world, device) / (ms * 1e-3) / 1e12,
            "launches_per_step": 3 + (1 if softmax else 0),
            "roofline": {"bound": "tensor", "achieved": per_gpu, "peak": peak, "unit": "TFLOP/s",
                         "frac": per_gpu / peak, "traffic": None,
                         "kernel": "dQ + dK/dV kernels (whole backward step, useful FLOPs)"},
            "cpu_baseline": (cpu_baseline_backward(w, q, k, v, w.grad_output(), 4.0, bias)
                             if cpu and rank == 0 and not rab_grads else None)}
        del bw, call, dq, dk, dv, d_o, q, k, v
        torch.cuda.empty_cache()
    return out


def time_e2e_steps(w, host, device, steps, warmup, world, stream):
    """Public-API round trip per step from pinned host memory, pipelined over
    two buffer sets: step i's q/k/v/offsets/targets go host -> device on a copy
    stream, its forward (hstu_attn_fwd) runs on the compute stream once they
    have landed, and its o goes device -> pinned host on a third stream, so
    step i+1's copies overlap step i's forward.  Every step moves its own
    inputs and its own result; the events order each buffer's reuse."""
    hq, hk, hv, hoff, htg = host
    sets = []
    for _ in range(2):
        call, dev = device_call(w, hq, hk, hv, device)
        sets.append({"call": call, "dev": dev, "ho": torch.empty(call.o.shape, dtype=call.o.dtype, pin_memory=True),
                     "ev_in": torch.cuda.Event(), "ev_fwd": torch.cuda.Event(), "ev_out": torch.cuda.Event(),
                     "used": False})
    # (copies spread over three copy streams measured the same: the host link,
    # about 250 GB/s for both directions together, is the limit)
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)

    def one(i):
        b = sets[i % 2]
        dq, dk, dv, doff, dtg = b["dev"]
        with torch.cuda.stream(s_in):
            if b["used"]:
                s_in.wait_event(b["ev_fwd"])        # the last forward on this set has read its inputs
            for dst, src in ((dq, hq), (dk, hk), (dv, hv), (doff, hoff), (dtg, htg)):
                dst.copy_(src, non_blocking=True)
            b["ev_in"].record(s_in)
        stream.wait_event(b["ev_in"])
        if b["used"]:
            stream.wait_event(b["ev_out"])          # the last read-back of this set's o is done
        b["call"].launch(stream)
        b["ev_fwd"].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(b["ev_fwd"])
            b["ho"].copy_(b["call"].o, non_blocking=True)
            b["ev_out"].record(s_out)
        b["used"] = True

    for i in range(warmup):
        one(i)
    torch.cuda.synchronize()
    barrier(world)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    s_in.wait_event(start)
    for i in range(steps):
        one(warmup + i)
    stream.wait_stream(s_out)
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hoff, htg))
    d2h = sets[0]["ho"].numel() * sets[0]["ho"].element_size()
    for b in sets:
        b["call"].check(stream)
    return start.elapsed_time(end) / steps, h2d, d2h


def run_cuda(args):
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    from recommender_attention_gb300 import build as B
    from recommender_attention_gb300 import hstu
    if rank == 0 or not os.path.exists(B.LIB_PATH):
        B.build()
    barrier(world)
    hstu.load_library()
    stream = torch.cuda.Stream(device)
    if args.scope_only is not None:
        # only the other scope workloads (for profiling them); not the bench line
        if rank == 0:
            peaks0, _ = load_peaks()
            only = [x for x in args.scope_only.split(",") if x]
            lines = small_config_lines(device, stream, args.steps, args.warmup,
                                       float(peaks0.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])), only)
            print(json.dumps({"scope_only": True, "configs": lines}), flush=True)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    w = rank_workload(rank, args.hdim)
    q, k, v = w.tensors()
    call, dev = device_call(w, q, k, v, device, args.cta_pairs)
    st = call.stats(stream)
    if args.headline_only:
        # the headline call alone, warm-up then timed launches (for profiling
        # its kernels); not the bench line
        for _ in range(args.warmup + args.steps):
            call.launch(stream)
        call.check(stream)
        if rank == 0:
            print(json.dumps({"headline_only": True, "launches": args.warmup + args.steps,
                              "allowed_pairs": st["allowed_pairs"]}), flush=True)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    flops_step = 2.0 * (w.hdim_qk + w.hdim_v) * st["allowed_pairs"]
    exec_flops = 2.0 * 128 * 128 * (w.hdim_qk + w.hdim_v) * st["executed_tiles"]

    with ClockSampler(local) as clk:
        step_ms, fwd_ms = time_device_steps(call, args.steps, args.warmup, world, stream)
    clocks = clk.summary()
    sustained = None
    if args.sustained_seconds > 0:
        s_ms, s_n, s_clk = time_sustained(call, stream, step_ms, args.sustained_seconds, local, world)
        s_ms = reduce_max(s_ms, world, device)
        sustained = {"ms_per_step": s_ms, "steps": s_n, "seconds": s_ms * s_n * 1e-3, "clocks": s_clk,
                     "timing": "the headline step back to back on the same resident inputs (larger than L2)"}
    host = tuple(t.pin_memory() for t in (q, k, v, torch.from_numpy(w.seq_offsets_q()),
                                          torch.from_numpy(w.num_targets())))
    e2e_ms, h2d, d2h = time_e2e_steps(w, host, device, args.steps, args.warmup, world, stream)

    # the same workload at the other head dimensions (one forward kernel per
    # step, same timing rules): 256, 96 and the asymmetric 96/64
    extra = {}
    if args.hdim == 128 and not args.no_d256:
        del call, dev
        torch.cuda.empty_cache()
        for key, dqk, dv in (("hdim256", 256, 256), ("hdim96", 96, 96), ("hdim96_64", 96, 64)):
            w2 = W.large_jagged(hdim=dqk, hdim_v=dv, seed=7 + rank)
            q2, k2, v2 = w2.tensors()
            call2, dev2 = device_call(w2, q2, k2, v2, device)
            st2 = call2.stats(stream)
            f2 = 2.0 * (w2.hdim_qk + w2.hdim_v) * st2["allowed_pairs"]
            s2, fw2 = time_device_steps(call2, args.steps, args.warmup, world, stream)
            s2 = reduce_max(s2, world, device)
            tot2 = reduce_sum(f2, world, device)
            extra[key] = {"value": tot2 / (s2 * 1e-3) / 1e12, "ms_per_step": s2,
                          "fwd_kernel_ms": fw2, "fwd_kernel_tflops": f2 / (fw2 * 1e-3) / 1e12}
            del call2, dev2, q2, k2, v2
            torch.cuda.empty_cache()
        # the same hdim 128 workload on the CTA-pair kernel (hstu_fwd_args::cta_pairs)
        call2, dev2 = device_call(w, q, k, v, device, 1)
        s2, fw2 = time_device_steps(call2, args.steps, args.warmup, world, stream)
        s2 = reduce_max(s2, world, device)
        tot2 = reduce_sum(flops_step, world, device)
        extra["cta_pairs"] = {"value": tot2 / (s2 * 1e-3) / 1e12, "ms_per_step": s2, "fwd_kernel_ms": fw2,
                              "fwd_kernel_tflops": flops_step / (fw2 * 1e-3) / 1e12}
        del call2, dev2
        torch.cuda.empty_cache()

    if args.hdim == 128 and not args.no_rab:
        peaks_r, _ = load_peaks()
        extra["rab"] = rab_lines(rank, device, stream, args.steps, args.warmup, world,
                                 float(peaks_r.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])),
                                 not args.no_cpu_baseline)

    if args.hdim == 128 and not args.no_bwd:
        peaks_b, _ = load_peaks()
        extra["backward"] = backward_lines(rank, device, stream, args.steps, args.warmup, world,
                                           float(peaks_b.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])),
                                           not args.no_cpu_baseline)

    if rank == 0 and not args.no_configs:
        peaks0, _ = load_peaks()
        extra["configs"] = small_config_lines(device, stream, max(5, args.steps), args.warmup,
                                              float(peaks0.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])))

    step_ms_max = reduce_max(step_ms, world, device)
    e2e_ms_max = reduce_max(e2e_ms, world, device)
    total_flops = reduce_sum(flops_step, world, device)
    value = total_flops / (step_ms_max * 1e-3) / 1e12
    e2e_value = total_flops / (e2e_ms_max * 1e-3) / 1e12

    if rank == 0:
        peaks, src = load_peaks()
        peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
        achieved = flops_step / (fwd_ms * 1e-3) / 1e12
        traffic = recorded_traffic()
        cpu = None if args.no_cpu_baseline else cpu_baseline(w, q, k, v, budget_s=args.cpu_seconds)
        launches_per_step = 2 + (1 if st["num_splits"] > 1 else 0)   # scheduler, forward [, combine]
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms_max,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic N(0,1) bf16, seed 7 (+rank)",
            "config": workload_config(w, st["allowed_pairs"], world),
            "schedule": {"executed_tiles": st["executed_tiles"], "num_splits": st["num_splits"],
                         "work_units": st["work_units"]},
            "pct_of_bf16_peak": 100.0 * value / world / peak,
            "executed_tile_tflops": reduce_sum(exec_flops, 1) / (step_ms_max * 1e-3) / 1e12,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak,
                         "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                         "peak_source": f"{src} bf16 dense (burst)",
                         "kernel": "hstu_fwd_kernel<128,bf16,SiLU>", "kernel_ms": fwd_ms},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms_max,
                    "pipelining": "two buffer sets: step i+1's host-to-device copies and step i-1's "
                                  "read-back overlap step i's forward"},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
        }
        if sustained is not None:
            sp = float(peaks.get("bf16_tflops_sustained", peak))
            sv = total_flops / (sustained["ms_per_step"] * 1e-3) / 1e12
            sustained.update({"value": sv, "unit": UNIT, "peak": sp,
                              "peak_source": f"{src} bf16 dense (sustained)" if "bf16_tflops_sustained" in peaks
                              else f"{src} bf16 dense (burst; no sustained figure)",
                              "frac": sv / world / sp})
            line["sustained"] = sustained
        line.update(extra)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------- oracle arm
def _blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return os.cpu_count()


def cpu_baseline(w, q, k, v, budget_s: float = 12.0):
    """The fp64 oracle as it stands on a bounded sample: whole (sequence, head)
    problems of the workload, longest sequence first, until the budget is spent."""
    from oracle.hstu_oracle import HstuParams, SeqMaskParams, dense_mask, hstu_attention_forward_rows
    p = HstuParams(num_groups=w.num_groups, context_len=w.context_len, local_len=w.local_len,
                   minfull_len=w.minfull_len, max_uih_len=w.max_uih_len,
                   attn_scale=w.attn_scale, alpha=w.alpha, causal=w.causal, softmax=w.softmax)
    off = w.seq_offsets_q()
    tg = w.num_targets()
    f64 = lambda t: t.float().numpy().astype(np.float64)
    qd, kd, vd = f64(q), f64(k), f64(v)
    order = list(np.argsort(-w.lengths_q()))
    flops, done = 0.0, 0
    t0 = time.perf_counter()
    for b in order:
        L = int(off[b + 1] - off[b])
        rows = np.arange(L)
        for h in range(w.nhead):
            hstu_attention_forward_rows(qd, kd, vd, off, None, tg, p, int(b), h, rows)
            sp = SeqMaskParams(L_q=L, L_kv=L, context=int(w.context_len[0]), targets=int(tg[b]),
                               causal=w.causal, local=int(w.local_len[0]),
                               minfull=int(w.minfull_len[0]), cross=False)
            flops += 2.0 * (w.hdim_qk + w.hdim_v) * float(dense_mask(sp).sum())
            done += 1
            if time.perf_counter() - t0 >= budget_s:
                break
        if time.perf_counter() - t0 >= budget_s:
            break
    el = time.perf_counter() - t0
    return {"value": flops / el / 1e12, "unit": UNIT, "cores": _blas_threads(), "kind": "oracle",
            "sample": f"{done} whole (sequence, head) problems of the {w.batch}x{w.nhead}, "
                      f"longest first, fp64 numpy, {el:.1f} s"}


def cpu_baseline_backward(w, q, k, v, d_o, budget_s: float = 6.0, bias=None):
    """The oracle's backward as it stands on a bounded sample: whole sequences
    (all heads) of the workload, each with the attn_scale the full batch
    resolves to; longest first, or shortest first with a relative attention
    bias (whose dense per-pair arrays make the oracle much slower).  Value:
    useful backward TFLOP/s (the bench line's FLOP count)."""
    import dataclasses
    from oracle.hstu_oracle import (HstuParams, SeqMaskParams, dense_mask, hstu_attention_backward,
                                    resolved_attn_scales)
    p = HstuParams(num_groups=1, context_len=w.context_len, local_len=w.local_len, minfull_len=w.minfull_len,
                   max_uih_len=w.max_uih_len, attn_scale=w.attn_scale, alpha=w.alpha, causal=w.causal,
                   softmax=w.softmax)
    off = w.seq_offsets_q()
    tg = w.num_targets()
    sub = dataclasses.replace(p, attn_scale=[float(resolved_attn_scales(p, w.batch, off, tg)[0])])
    f64 = lambda t: t.float().numpy().astype(np.float64)
    flops, done = 0.0, 0
    t0 = time.perf_counter()
    order = np.argsort(w.lengths_q()) if bias is not None else np.argsort(-w.lengths_q())
    for b in list(order):
        s0, s1 = int(off[b]), int(off[b + 1])
        pb = sub if bias is None else dataclasses.replace(sub, timestamps_q=bias[0][s0:s1], rab_time=bias[2],
                                                          rab_pos=bias[3])
        hstu_attention_backward(f64(q[s0:s1]), f64(k[s0:s1]), f64(v[s0:s1]), f64(d_o[s0:s1]),
                                np.array([0, s1 - s0]), None, np.array([tg[b]]), pb)
        sp = SeqMaskParams(L_q=s1 - s0, L_kv=s1 - s0, context=int(w.context_len[0]), targets=int(tg[b]),
                           causal=w.causal, local=int(w.local_len[0]), minfull=int(w.minfull_len[0]), cross=False)
        flops += 2.0 * (3 * w.hdim_qk + 2 * w.hdim_v) * float(dense_mask(sp).sum()) * w.nhead
        done += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    el = time.perf_counter() - t0
    return {"value": flops / el / 1e12, "unit": UNIT, "cores": _blas_threads(), "kind": "oracle",
            "sample": f"{done} whole sequences (all {w.nhead} heads) of the {w.batch}, "
                      f"{'shortest first, with the bias' if bias is not None else 'longest first'}, "
                      f"fp64 numpy backward, {el:.1f} s"}


def cpu_baseline_rab(w, q, k, v, rab, budget_s: float = 6.0):
    """The oracle's forward with the relative attention bias on a bounded
    sample: whole (sequence, head) problems, longest first."""
    from oracle.hstu_oracle import HstuParams, SeqMaskParams, dense_mask, hstu_attention_forward_rows
    ts_q, _, rab_time, rab_pos = rab
    p = HstuParams(num_groups=1, context_len=w.context_len, local_len=w.local_len, minfull_len=w.minfull_len,
                   max_uih_len=w.max_uih_len, attn_scale=w.attn_scale, alpha=w.alpha, causal=w.causal,
                   softmax=w.softmax, timestamps_q=ts_q, rab_time=rab_time, rab_pos=rab_pos)
    off = w.seq_offsets_q()
    tg = w.num_targets()
    f64 = lambda t: t.float().numpy().astype(np.float64)
    qd, kd, vd = f64(q), f64(k), f64(v)
    flops, done = 0.0, 0
    t0 = time.perf_counter()
    for b in list(np.argsort(-w.lengths_q())):
        L = int(off[b + 1] - off[b])
        for h in range(w.nhead):
            hstu_attention_forward_rows(qd, kd, vd, off, None, tg, p, int(b), h, np.arange(L))
            sp = SeqMaskParams(L_q=L, L_kv=L, context=int(w.context_len[0]), targets=int(tg[b]),
                               causal=w.causal, local=int(w.local_len[0]), minfull=int(w.minfull_len[0]),
                               cross=False)
            flops += 2.0 * (w.hdim_qk + w.hdim_v) * float(dense_mask(sp).sum())
            done += 1
            if time.perf_counter() - t0 >= budget_s:
                break
        if time.perf_counter() - t0 >= budget_s:
            break
    el = time.perf_counter() - t0
    return {"value": flops / el / 1e12, "unit": UNIT, "cores": _blas_threads(), "kind": "oracle",
            "sample": f"{done} whole (sequence, head) problems with the bias, longest first, fp64 numpy, {el:.1f} s"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    w = rank_workload(0, args.hdim)
    q, k, v = w.tensors()
    from oracle.hstu_oracle import HstuParams, allowed_pair_count
    p = HstuParams(num_groups=w.num_groups, context_len=w.context_len, local_len=w.local_len,
                   minfull_len=w.minfull_len, max_uih_len=w.max_uih_len, attn_scale=w.attn_scale,
                   alpha=w.alpha, causal=w.causal, softmax=w.softmax)
    pairs = allowed_pair_count(w.seq_offsets_q(), None, w.num_targets(), p, w.nhead)
    # Each step is one bounded sample of the workload through the oracle (whole
    # (sequence, head) problems, longest first, for a fixed time budget); the
    # step's time is that sample's measured time and its rate the sample's.
    per_step = max(1.0, min(20.0, args.ref_seconds / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        cpu_baseline(w, q, k, v, budget_s=per_step)
    vals, secs = [], []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        vals.append(cpu_baseline(w, q, k, v, budget_s=per_step))
        secs.append(time.perf_counter() - t0)
    value = statistics.mean(x["value"] for x in vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(secs),
        "ms_per_step_basis": f"measured wall time of one step; a step is a bounded sample of about "
                             f"{per_step:.1f} s of the workload (whole (sequence, head) problems, longest "
                             f"first), not the whole workload",
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic N(0,1) bf16, seed 7 (+rank)",
        "config": workload_config(w, pairs, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "kind": "oracle",
                         "cores": vals[0]["cores"], "sample": vals[0]["sample"]},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["cuda", "reference"], default="cuda")
    ap.add_argument("--hdim", type=int, default=128, choices=[64, 128, 256])
    ap.add_argument("--no-d256", action="store_true",
                    help="skip the hdim 256, 96 and 96/64 repeats and the CTA-pair repeat")
    ap.add_argument("--cta-pairs", type=int, default=0, choices=[-1, 0, 1],
                    help="forward kernel of the headline call (hstu_fwd_args::cta_pairs; for profiling)")
    ap.add_argument("--no-bwd", action="store_true", help="skip the backward lines")
    ap.add_argument("--no-rab", action="store_true", help="skip the relative attention bias lines")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the other scope workloads")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-seconds", type=float, default=60.0)
    ap.add_argument("--scope-only", default=None, metavar="NAMES",
                    help="run only these scope workloads (comma-separated names of the 'configs' lines; "
                         "empty: all) and print their lines alone; for profiling")
    ap.add_argument("--headline-only", action="store_true",
                    help="launch only the headline call (warm-up + steps times) and print a short line; for profiling")
    ap.add_argument("--sustained-seconds", type=float, default=2.0,
                    help="seconds of back-to-back headline steps for the 'sustained' figure (0: skip)")
    args = ap.parse_args(argv)
    if args.impl == "cuda":
        args.warmup = max(3, args.warmup)   # timing rule: at least 3 untimed warm-up steps
    if args.impl == "reference":
        run_reference(args)
    else:
        run_cuda(args)


if __name__ == "__main__":
    main()
