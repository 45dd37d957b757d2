"""Throughput of exact attention (forward + recompute backward) on GB300, one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

A step is one pass of the whole path over one batch: fa_forward then fa_backward on the
workload's synthetic inputs (seeded N(0,1), see workloads/).  The default workload is the
long-context shape B1 H16 N16384 d128, non-causal, the shape the bf16 tensor-peak target is
quoted on.  Its inputs (Q, K, V, O, dO: 5 x 64 MiB) are larger than the 129 MB L2, so no flush
is needed between steps.

FLOP convention: forward F = 4*B*H*N^2*d (halved when causal; kept 128x128 tiles only when
block-sparse).  The headline value counts 2.5*F per forward+backward step; the algorithmic
count (2 products forward, 5 backward: 3.5*F) is reported beside it.

Under torchrun (N > 1) every rank runs the same workload on its own GPU (independent replicas,
weak scaling); the ranks only meet at the barriers around the timed region and for the max of
the elapsed times.  --impl reference times the fp64 CPU oracle on a bounded sample of the same
workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd & fwd+bwd TFLOPS, % of GB300 BF16 tensor peak, N=512–16K"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = ["exact_io_aware_23_gb300/csrc"]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# host-only translation units (argument checks, descriptor encoding): not part of the kernels
HOST_ONLY_SOURCES = {"fa_api.cu", "fa_noalloc.cu", "fa_tmap.cu"}


def kernel_source_hash():
    """Hash of the device-code sources (a traffic record stays valid while they are unchanged)."""
    h = hashlib.sha256()
    for d in KERNEL_SOURCES:
        base = os.path.join(ROOT, d)
        for fn in sorted(os.listdir(base)):
            if fn.endswith((".cu", ".cuh")) and fn not in HOST_ONLY_SOURCES:
                with open(os.path.join(base, fn), "rb") as f:
                    h.update(fn.encode() + f.read())
    return h.hexdigest()[:16]


def forward_flops(w, B, H, N, block_mask=None):
    full = 4.0 * B * H * N * N * w.d
    if block_mask is not None:
        T = block_mask.shape[0]
        return full * float(block_mask.sum()) / float(T * T)
    return full / 2 if w.causal else full


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons every 100 ms while running.

    The sampler is started before the timed region and waits (up to 3 s) for its first sample,
    so that it is running when the region starts; `mark_start` / `mark_end` bracket the region,
    and the summary uses the samples that arrived inside it (all of them if none did).
    """
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.rows, self.proc = index, [], None
        self.t_start, self.t_end = None, None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            t0 = time.monotonic()
            while not self.rows and time.monotonic() - t0 < 3.0 and self.proc.poll() is None:
                time.sleep(0.01)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.monotonic(), [x.strip() for x in line.split(",")]))

    def mark_start(self):
        self.t_start = time.monotonic()

    def mark_end(self):
        self.t_end = time.monotonic()

    def __exit__(self, *exc):
        if self.t_end is None:
            self.mark_end()
        if self.proc is not None:
            time.sleep(0.15)                 # the sample that covers the region's last moments
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = [r for t, r in self.rows
                if self.t_start is not None and self.t_start <= t <= (self.t_end or t) + 0.15]
        inside = bool(rows)
        if not inside:
            rows = [r for _, r in self.rows]
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[4:8]) if v == "Active"})
        pw = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        out = {"sm_mhz": statistics.median(sm) if sm else None,
               "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
               "power_w_max": max(pw) if pw else None, "samples": len(rows)}
        if not inside:
            out["note"] = "no sample arrived inside the timed region; all samples summarised"
        return out


def cpu_oracle_sample(x, w, rows_per_head, heads=(0,)):
    """Time the fp64 oracle, forward + backward, on a sample of query rows of some heads."""
    import numpy as np
    import torch

    import oracle
    f64 = lambda t: t[:, list(heads)].to(torch.float64).numpy()
    qq, kk, vv, dd = (f64(x[n]) for n in ("q", "k", "v", "do"))
    kv = None if x["kv_lens"] is None else x["kv_lens"].numpy()
    bm = None if x["block_mask"] is None else x["block_mask"].numpy()
    rows = np.arange(rows_per_head)
    t0 = time.perf_counter()
    oracle.forward(qq, kk, vv, x["scale"], causal=x["causal"], kv_lens=kv, block_mask=bm, rows=rows)
    oracle.backward(qq, kk, vv, dd, x["scale"], causal=x["causal"], kv_lens=kv, block_mask=bm,
                    rows=rows)
    return time.perf_counter() - t0


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def run_reference(args, w):
    """The oracle as the reference arm: each step = fwd+bwd on a bounded row sample of one head."""
    from workloads import make_inputs
    if int(os.environ.get("RANK", "0")) != 0:
        return
    x = make_inputs(w, seed=0, heads=1, B=1)
    F1 = forward_flops(w, 1, 1, w.N, x["block_mask"])       # one head
    rows = args.ref_rows
    f_sample = 2.5 * F1 * rows / w.N
    for _ in range(args.warmup):
        cpu_oracle_sample(x, w, rows)
    t = sum(cpu_oracle_sample(x, w, rows) for _ in range(args.steps))
    value = f_sample * args.steps / t / 1e12
    sample = f"fp64 oracle fwd+bwd on query rows [0,{rows}) of head 0 of {w.name} per step"
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": workload_config(w),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def max_over_ranks(values, device, world):
    """Element-wise maximum of per-rank timings (the slowest rank sets the job's time)."""
    if world <= 1:
        return list(values)
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def needs_l2_flush(w):
    """True when the forward's compulsory bytes are under twice the L2: timed back to back, such
    inputs would stay warm in L2 from one step to the next."""
    elt = 4 if w.dtype == "fp32" else 2
    fwd, _ = compulsory_bytes(w.B, w.H, w.Hkv or w.H, w.N, w.d, elt)
    return fwd < 2 * L2_BYTES


def workload_config(w):
    return {"workload": w.name, "B": w.B, "H": w.H, "Hkv": w.Hkv or w.H, "N": w.N, "d": w.d,
            "causal": w.causal,
            "key_padding": w.pad_lengths is not None, "block_sparse": w.block_sparse,
            "dtype": w.dtype, "parallelism": "replicas",
            "l2": (f"L2 flushed between timed steps ({FLUSH_BYTES >> 20} MiB write, untimed)"
                   if needs_l2_flush(w) else "inputs larger than L2 (no flush)")}


L2_BYTES = 129_000_000             # GB300 L2, nominal
FLUSH_BYTES = 256 * 2 ** 20         # written between timed steps when the inputs fit in L2


def compulsory_bytes(B, H, Hkv, N, d, elt):
    """Algorithmic HBM bytes of one forward and one backward (the compulsory traffic): the
    forward reads Q, K, V and writes O and LSE; the backward reads Q, K, V, O, dO and LSE and
    writes dQ, dK, dV."""
    q_side = B * H * N * d * elt
    kv_side = B * Hkv * N * d * elt
    lse = B * H * N * 4
    fwd = q_side + 2 * kv_side + q_side + lse
    bwd = 3 * q_side + 2 * kv_side + lse + q_side + 2 * kv_side
    return fwd, bwd


def effective_forward_flops(w, x, B, H, N):
    """Forward FLOPs over the allowed (query, key) pairs only: with key padding a row attends to
    kv_len keys (the nominal count includes the padded ones the kernel skips)."""
    if x["kv_lens"] is None:
        return forward_flops(w, B, H, N, x["block_mask"])
    lens = [int(v) for v in x["kv_lens"]]
    if w.causal:
        return sum(4.0 * H * w.d * sum(min(i + 1, L) for i in range(N)) for L in lens)
    return sum(4.0 * H * w.d * N * L for L in lens)


def peak_memory(fa, torch, q, k, v, do, kw, bkw):
    """Device memory of one forward + backward through the public API: the inputs plus the
    largest amount allocated during the calls (outputs, LSE, workspace), from the allocator's
    own peak counter."""
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    base = torch.cuda.memory_allocated()
    o, lse = fa.forward(q, k, v, **kw)
    grads = fa.backward(q, k, v, o, lse, do, **bkw)
    torch.cuda.synchronize()
    peak = torch.cuda.max_memory_allocated() - base
    del o, lse, grads
    inputs = sum(t.numel() * t.element_size() for t in (q, k, v, do))
    return inputs + peak, inputs, peak


def run_ours(args, w):
    import torch
    import torch.distributed as dist

    import exact_io_aware_23_gb300 as fa
    from workloads import make_inputs

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            dist.barrier()

    x = make_inputs(w, seed=rank)
    B, H, N, d = x["q"].shape
    Hkv = x["k"].shape[1]
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    bm = None if x["block_mask"] is None else x["block_mask"].to(dev)
    kl = None if x["kv_lens"] is None else x["kv_lens"].to(dev)
    o, lse = torch.empty_like(q), torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_bytes = (fa.backward_fused_workspace_size(B, H, N, d) if args.fused_backward
                else fa.backward_workspace_size(B, H, N, d))
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    kw = dict(causal=w.causal, scale=w.scale, block_mask=bm, kv_lens=kl)
    if args.dropout > 0.0:
        kw.update(dropout_p=args.dropout, seed=1234, offset=0)
    bkw = dict(kw, deterministic=args.deterministic, fused=args.fused_backward)
    fwd_bytes, bwd_bytes = compulsory_bytes(B, H, Hkv, N, d, q.element_size())
    # Inputs that fit in L2 would be timed warm: then L2 is flushed between timed steps (a
    # 256 MB write outside the timed events) and every step is timed on its own.
    flush = needs_l2_flush(w)

    def step():
        fa.forward(q, k, v, o=o, lse=lse, **kw)
        fa.backward(q, k, v, o, lse, do, dq=dq, dk=dk, dv=dv, workspace=ws, **bkw)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if fa.check_device_status() != 0:
        raise RuntimeError("device error during warm-up")

    stream = torch.cuda.current_stream()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    scrub = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev) if flush else None
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        clocks.mark_start()
        if flush:
            # hold the stream while every step is queued, so no step waits for the host
            torch.cuda._sleep(int(2e8))
        start.record(stream)
        for i in range(args.steps):
            if flush:
                scrub.zero_()
            ev[i][0].record(stream)
            fa.forward(q, k, v, o=o, lse=lse, **kw)
            ev[i][1].record(stream)
            fa.backward(q, k, v, o, lse, do, dq=dq, dk=dk, dv=dv, workspace=ws, **bkw)
            ev[i][2].record(stream)
        end.record(stream)
        torch.cuda.synchronize()
        clocks.mark_end()
    barrier()
    fwd_ms = [e[0].elapsed_time(e[1]) for e in ev]
    bwd_ms = [e[1].elapsed_time(e[2]) for e in ev]
    # with flushes, the timed work is the sum of the steps' own intervals (the flushes between
    # them are not the method's work); without, the whole region between the two events
    total_ms = sum(f + b for f, b in zip(fwd_ms, bwd_ms)) if flush else start.elapsed_time(end)
    t_fwd = sum(fwd_ms) / args.steps
    t_bwd = sum(bwd_ms) / args.steps
    med_fwd, med_bwd = statistics.median(fwd_ms), statistics.median(bwd_ms)
    if fa.check_device_status() != 0:
        raise RuntimeError("device error during the timed region")

    # End to end: every step copies its inputs from pinned host memory, runs forward + backward
    # through the public API and copies all results back to pinned host memory.  The three legs
    # run on their own streams and the device buffers are double-buffered, so step k's compute
    # overlaps step k+1's input copies and step k-1's result copies; every copy of every step is
    # inside the timed region.
    hin = [t.pin_memory() for t in (x["q"], x["k"], x["v"], x["do"])]
    h2d = sum(t.numel() * t.element_size() for t in hin)
    bufs = []
    for _ in range(2):
        din_b = [torch.empty_like(t) for t in (q, k, v, do)]
        dout_b = [torch.empty_like(t) for t in (o, lse, dq, dk, dv)]
        hout_b = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in dout_b]
        ws_b = torch.empty_like(ws)
        bufs.append((din_b, dout_b, hout_b, ws_b))
    d2h = sum(t.numel() * t.element_size() for t in bufs[0][2])
    s_in, s_run, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_run = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    for e in ev_run + ev_out:                          # start "completed"
        e.record(stream)

    def e2e_step(kstep):
        b_ = kstep & 1
        (qi, ki, vi, doi), (ob, lb, dqb, dkb, dvb), hout_b, ws_b = bufs[b_]
        s_in.wait_event(ev_run[b_])                    # the inputs' last reader is done
        with torch.cuda.stream(s_in):
            for dst, src in zip((qi, ki, vi, doi), hin):
                dst.copy_(src, non_blocking=True)
            ev_in[b_].record(s_in)
        s_run.wait_event(ev_in[b_])
        s_run.wait_event(ev_out[b_])                   # the outputs' last copy-out is done
        fa.forward(qi, ki, vi, o=ob, lse=lb, stream=s_run, **kw)
        fa.backward(qi, ki, vi, ob, lb, doi, dq=dqb, dk=dkb, dv=dvb, workspace=ws_b, stream=s_run, **bkw)
        ev_run[b_].record(s_run)
        s_out.wait_event(ev_run[b_])
        with torch.cuda.stream(s_out):
            for dst, src in zip(hout_b, (ob, lb, dqb, dkb, dvb)):
                dst.copy_(src, non_blocking=True)
            ev_out[b_].record(s_out)

    for kstep in range(max(1, args.warmup)):
        e2e_step(kstep)
    s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    s2.record(s_in)
    for kstep in range(args.steps):
        e2e_step(kstep)
    s_in.wait_stream(s_out)
    s_in.wait_stream(s_run)
    e2.record(s_in)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = s2.elapsed_time(e2)
    del bufs

    mem_total, mem_inputs, mem_calls = peak_memory(fa, torch, q, k, v, do, kw, bkw)

    total_ms, e2e_ms, t_fwd, t_bwd, med_fwd, med_bwd = max_over_ranks(
        [total_ms, e2e_ms, t_fwd, t_bwd, med_fwd, med_bwd], dev, world)

    F = forward_flops(w, B, H, N, x["block_mask"])
    F_eff = effective_forward_flops(w, x, B, H, N)
    ms_step = total_ms / args.steps
    value = world * 2.5 * F / (ms_step * 1e-3) / 1e12
    e2e_value = world * 2.5 * F / (e2e_ms / args.steps * 1e-3) / 1e12
    peaks, peak_src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    hbm = float(peaks["hbm_gbs"])
    fwd_tf = F / (t_fwd * 1e-3) / 1e12
    bwd_tf = 2.5 * F / (t_bwd * 1e-3) / 1e12
    dominant = "backward" if t_bwd >= t_fwd else "forward"
    # roofline of the dominant call: max(F / F_peak, bytes / B_HBM) decides the bound; the
    # achieved rate is reported in that bound's unit (effective FLOPs when keys are padded)
    flops_dom = (2.5 if dominant == "backward" else 1.0) * F_eff
    bytes_dom = bwd_bytes if dominant == "backward" else fwd_bytes
    t_dom = (t_bwd if dominant == "backward" else t_fwd) * 1e-3
    t_tensor, t_hbm = flops_dom / (peak * 1e12), bytes_dom / (hbm * 1e9)
    if t_hbm > t_tensor:
        roof = {"bound": "hbm", "achieved": bytes_dom / t_dom / 1e9, "peak": hbm, "unit": "GB/s",
                "frac": bytes_dom / t_dom / 1e9 / hbm, "peak_source": f"hbm_gbs of {peak_src}"}
    else:
        roof = {"bound": "tensor", "achieved": flops_dom / t_dom / 1e12, "peak": peak,
                "unit": "TFLOP/s", "frac": flops_dom / t_dom / 1e12 / peak,
                "peak_source": f"bf16_tflops of {peak_src}"}
    traffic = None
    tp = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tp):
        with open(tp) as f:
            rec = json.load(f)
        # records are per kernel variant: the dropout and fused-backward instantiations have their own
        key = w.name + ("_dropout" if args.dropout > 0.0 else "") + ("_fused" if args.fused_backward else "")
        ent = rec.get(key, {}).get(dominant)
        if ent and ent.get("source_hash") == kernel_source_hash():
            traffic = ent.get("bytes_per_launch")
    roof.update(kernel=f"fa_{dominant} (all launches of the call)", traffic=traffic)

    def roofline_time_fraction(flops, nbytes, t_ms):
        return max(flops / (peak * 1e12), nbytes / (hbm * 1e9)) / (t_ms * 1e-3)

    config = dict(workload_config(w),
                  backward="fused_atomic_dq" if args.fused_backward else "two_pass",
                  **({"dropout": args.dropout} if args.dropout > 0.0 else {}))
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": config,
        "fwd_tflops": fwd_tf, "bwd_tflops": bwd_tf,
        "fwd_bwd_tflops_algorithmic": world * 3.5 * F / (ms_step * 1e-3) / 1e12,
        "pct_of_bf16_peak": {"forward": fwd_tf / peak, "fwd_bwd": value / world / peak,
                             "peak_tflops": peak, "peak_source": peak_src},
        "ms_fwd": t_fwd, "ms_bwd": t_bwd, "ms_fwd_median": med_fwd, "ms_bwd_median": med_bwd,
        "roofline_time_fraction": {
            "forward": roofline_time_fraction(F_eff, fwd_bytes, med_fwd),
            "backward": roofline_time_fraction(2.5 * F_eff, bwd_bytes, med_bwd),
            "compulsory_bytes": {"forward": fwd_bytes, "backward": bwd_bytes},
            "timing": "median of the per-step event times"},
        "roofline": roof,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "pipelined": "copies in, compute and copies out on three streams, double-buffered",
                "d2h_bytes_per_step": d2h},
        "peak_mem_bytes": mem_total,
        "peak_mem": {"inputs_bytes": mem_inputs, "allocated_by_the_calls_bytes": mem_calls,
                     "workspace_bytes": ws_bytes,
                     "bytes_per_q_row_element": mem_total / float(B * H * N * d),
                     "one_fp32_score_matrix_bytes": 4 * B * H * N * N},
        "gpu_launches": launches_per_step(args, x) * args.steps,
        "clocks": clocks.summary(),
    }
    if F_eff != F:
        line["effective_flops"] = {"forward_flops": F_eff, "nominal_forward_flops": F,
                                   "fwd_tflops": F_eff / (t_fwd * 1e-3) / 1e12,
                                   "bwd_tflops": 2.5 * F_eff / (t_bwd * 1e-3) / 1e12,
                                   "note": "allowed (query, key) pairs only"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rows = min(N, args.cpu_rows)
        t_cpu = cpu_oracle_sample(x, w, rows)
        f_cpu = 2.5 * forward_flops(w, 1, 1, N, x["block_mask"]) * rows / N
        line["cpu_baseline"] = {"value": f_cpu / t_cpu / 1e12, "unit": UNIT, "cores": cpu_cores(),
                                "kind": "oracle",
                                "sample": f"fp64 oracle fwd+bwd, head 0, query rows [0,{rows}), "
                                          f"{t_cpu:.1f} s"}
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


# kernels of ours launched per step: forward 1; backward 2 (preprocess, two-pass kernel) or, with
# --fused-backward, 3 (preprocess, fused kernel, dQ convert)
LAUNCHES_PER_STEP = {"two_pass": 3, "fused": 4}


def launches_per_step(args, x):
    """Our kernel launches in one forward + backward step: with a tile mask the balanced forward
    adds its two plan kernels and the two-pass backward its two unit-order kernels."""
    n = LAUNCHES_PER_STEP["fused" if args.fused_backward else "two_pass"]
    if x["block_mask"] is not None and args.dropout == 0.0:
        n += 2 + (0 if args.fused_backward else 2)
    elif x["block_mask"] is not None and not args.fused_backward:
        n += 2
    return n


def run_decode(args, w):
    """Decode-shaped workloads: one step = one split-KV forward (fa_forward_splitkv); the bound is
    HBM (the key/value cache is read once), so the roofline is reported in GB/s."""
    import torch

    import exact_io_aware_23_gb300 as fa
    from workloads import make_inputs

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    x = make_inputs(w, seed=0)
    B, H, Nq, d = x["q"].shape
    Nk, Hkv = x["k"].shape[2], x["k"].shape[1]
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=dev)
    # grouped heads: a group's G * Nq queries run as one block against its key/value head
    splits = (args.splits if args.splits > 0
              else int(fa.lib.fa_forward_splitkv_auto_splits(B, Hkv, (H // Hkv) * Nq, Nk)))
    ws = torch.empty(int(fa.lib.fa_forward_splitkv_workspace_size(B, H, Nq, d, splits)), dtype=torch.uint8, device=dev)
    step = lambda: fa.forward_splitkv(q, k, v, scale=w.scale, n_splits=splits, o=o, lse=lse, workspace=ws)
    for _ in range(args.warmup):
        step()
    stream = torch.cuda.current_stream()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with ClockSampler(0) as clocks:
        clocks.mark_start()
        s0.record(stream)
        for _ in range(args.steps):
            step()
        s1.record(stream)
        torch.cuda.synchronize()
        clocks.mark_end()
    ms = s0.elapsed_time(s1) / args.steps
    if fa.check_device_status() != 0:
        raise RuntimeError("device error during the timed region")
    hin = [t.pin_memory() for t in (x["q"], x["k"], x["v"])]
    hout = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (o, lse)]

    def e2e_step():
        for dst, src in zip((q, k, v), hin):
            dst.copy_(src, non_blocking=True)
        step()
        for dst, src in zip(hout, (o, lse)):
            dst.copy_(src, non_blocking=True)

    e2e_step()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    F = 4.0 * B * H * Nq * Nk * d
    elt = q.element_size()
    algo_bytes = elt * (2 * B * Hkv * Nk * d + 2 * B * H * Nq * d) + 4 * B * H * Nq
    peaks, src = load_peaks()
    gbs = algo_bytes / (ms * 1e-3) / 1e9
    line = {"metric": METRIC, "value": F / (ms * 1e-3) / 1e12, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": dict(workload_config(w), Nk=Nk, n_splits=splits, forward_only=True),
            "roofline": {"bound": "hbm", "kernel": "fa_forward_splitkv (split kernel + merge)",
                         "achieved": gbs, "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
                         "frac": gbs / float(peaks["hbm_gbs"]), "traffic": None,
                         "peak_source": f"hbm_gbs of {src}"},
            "e2e": {"value": F / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
                    "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in hin),
                    "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in hout)},
            "gpu_launches": 2 * args.steps, "clocks": clocks.summary()}
    print(json.dumps(line), flush=True)


def run_varlen(args, w):
    """Packed-sequence workloads: one step = fa_forward_varlen + fa_backward_varlen over all the
    packed sequences; FLOPs summed per sequence (4*H*L^2*d, halved when causal)."""
    import torch

    import exact_io_aware_23_gb300 as fa
    from workloads import make_packed_inputs

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    x = make_packed_inputs(w, seed=0)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    cu, maxl = x["cu_seqlens"].to(dev), x["max_seqlen"]
    H, T, d = q.shape
    kw = dict(causal=w.causal, scale=w.scale)

    def fwd():
        return fa.forward_varlen(q, k, v, cu, maxl, **kw)

    o, lse = fwd()
    for _ in range(args.warmup):
        o, lse = fwd()
        fa.backward_varlen(q, k, v, o, lse, do, cu, maxl, **kw)
    stream = torch.cuda.current_stream()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    torch.cuda.synchronize()
    with ClockSampler(0) as clocks:
        clocks.mark_start()
        for i in range(args.steps):
            ev[i][0].record(stream)
            o, lse = fwd()
            ev[i][1].record(stream)
            fa.backward_varlen(q, k, v, o, lse, do, cu, maxl, **kw)
            ev[i][2].record(stream)
        torch.cuda.synchronize()
        clocks.mark_end()
    if fa.check_device_status() != 0:
        raise RuntimeError("device error during the timed region")
    # End to end, the legs in sequence: each step copies q, k, v, dO from pinned host memory,
    # runs forward + backward through the public API and copies O, LSE, dQ, dK, dV back.
    hin = [x[n].pin_memory() for n in ("q", "k", "v", "do")]
    grads = fa.backward_varlen(q, k, v, o, lse, do, cu, maxl, **kw)
    hout = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (o, lse) + tuple(grads)]

    def e2e_step():
        for dst, src in zip((q, k, v, do), hin):
            dst.copy_(src, non_blocking=True)
        o_, lse_ = fwd()
        g_ = fa.backward_varlen(q, k, v, o_, lse_, do, cu, maxl, **kw)
        for dst, src in zip(hout, (o_, lse_) + tuple(g_)):
            dst.copy_(src, non_blocking=True)

    e2e_step()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    t_fwd = sum(e[0].elapsed_time(e[1]) for e in ev) / args.steps
    t_bwd = sum(e[1].elapsed_time(e[2]) for e in ev) / args.steps
    F = sum(4.0 * H * n * n * d for n in w.seq_lens) * (0.5 if w.causal else 1.0)
    ms = t_fwd + t_bwd
    peaks, src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    bwd_tf = 2.5 * F / (t_bwd * 1e-3) / 1e12
    line = {"metric": METRIC, "value": 2.5 * F / (ms * 1e-3) / 1e12, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": dict(workload_config(w), n_seqs=len(w.seq_lens), max_seqlen=maxl, total=T),
            "fwd_tflops": F / (t_fwd * 1e-3) / 1e12, "bwd_tflops": bwd_tf,
            "ms_fwd": t_fwd, "ms_bwd": t_bwd,
            "roofline": {"bound": "tensor", "kernel": "fa_backward_varlen (all launches of the call)",
                         "achieved": bwd_tf, "peak": peak, "unit": "TFLOP/s", "frac": bwd_tf / peak,
                         "traffic": None, "peak_source": f"bf16_tflops of {src}"},
            "e2e": {"value": 2.5 * F / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
                    "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in hin),
                    "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in hout),
                    "pipelined": "no: copies in, compute and copies out in sequence on one stream"},
            "gpu_launches": 3 * args.steps, "clocks": clocks.summary()}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="long_n16k_d128")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--deterministic", action="store_true",
                    help="call fa_backward_deterministic (the default two-pass backward, by name)")
    ap.add_argument("--fused-backward", action="store_true",
                    help="time the fused atomic-dQ backward variant (fa_backward_fused)")
    ap.add_argument("--dropout", type=float, default=0.0,
                    help="dropout probability on P for the timed forward and backward")
    ap.add_argument("--splits", type=int, default=0,
                    help="key ranges of the split-KV decode workloads (0: the library's choice)")
    ap.add_argument("--cpu-rows", type=int, default=16384)
    ap.add_argument("--ref-rows", type=int, default=1024)
    args = ap.parse_args()
    from workloads import WORKLOADS
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    elif w.Nk is not None:
        run_decode(args, w)
    elif w.seq_lens is not None:
        run_varlen(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
