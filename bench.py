#!/usr/bin/env python3
"""Benchmark of the causal LSSAR attention forward on GB300.

One step = one call of the whole hot path (normalisation prologue + the
tcgen05 attention kernel) on one batch of seeded synthetic input resident in
HBM.  Default workload: B=1 H=12 L=8192 d=64, LSSAR p=15, causal (the 8K
extrapolation shape).  L2 is flushed (256 MiB write) before every timed step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--mode lssar|lssa|softmax] [--p P]

Prints one JSON line on rank 0.  `--impl reference` times the float64 CPU
oracle instead, on bounded samples of the same workload.
"""

import argparse
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

from lssar_attn_fwd_gb300.inputs import (  # noqa: E402
    MODE_LSSA, MODE_LSSAR, MODE_SIGMOID_RW, MODE_SOFTMAX, MODE_SOFTMAX_RW, WORKLOADS,
    bf16_bits_to_f64, make_qkv)

METRIC = "LSSAR causal fwd TFLOP/s (3 GEMMs) + % BF16 tensor peak, 1×GB300, L=1K–16K"
MODE_NAMES = {"lssar": MODE_LSSAR, "lssa": MODE_LSSA, "softmax": MODE_SOFTMAX,
              "softmax_rw": MODE_SOFTMAX_RW, "sigmoid_rw": MODE_SIGMOID_RW}
REWEIGHT_MODES = (MODE_LSSAR, MODE_SOFTMAX_RW, MODE_SIGMOID_RW)
FLUSH_BYTES = 256 << 20
L2_BYTES = 129 << 20   # GB300 L2
FALLBACK_BF16_TFLOPS = 1900.0
SPEC_DENSE_BF16_TFLOPS = 2250.0   # GB300 nominal dense bf16 tensor peak (context beside the measured one)
MIN_LOAD_S = 1.5                  # seconds of the same step under load for the clock record (nvidia-smi
                                  # averages utilisation over up to a second)


def gemm_count(mode):
    """GEMMs the method performs: re-weighting modes need the full first-stage
    row sum before any weight, hence a second Q.K^T (3 GEMMs); LSSA and
    softmax are counted with their 2 GEMMs."""
    return 3 if mode in REWEIGHT_MODES else 2


def flops(B, H, L, d, mode):
    """Algorithmic flops: 2 flops per multiply-add, causal half of each GEMM."""
    return gemm_count(mode) * 2.0 * B * H * d * L * (L + 1) / 2.0


def causal_flops_rows(rows, d, mode):
    return gemm_count(mode) * 2.0 * d * float(np.sum(rows))


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def kernel_source_sha():
    """Hash of the attention kernel's device sources (the kernel template, the
    headers it includes and its launch dispatch), to tell whether recorded
    counters still apply."""
    import hashlib
    h = hashlib.sha256()
    for name in ("tc_kernel.cuh", "fast_weights.cuh", "softplus_poly.cuh", "tc_ptx.cuh", "lssar_internal.cuh",
                 "tc_dispatch.cuh"):
        with open(os.path.join(ROOT, "lssar_attn_fwd_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def kernel_traffic(workload, mode, p):
    """dram read+write bytes per launch of the attention kernel from the
    committed ncu summary, if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        h = kernel_source_sha()
        key = f"{workload}:{mode}:{p}"
        ent = rec.get(key)
        if ent and ent.get("kernel_src_sha") == h:
            return float(ent["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


def hold_load(step, seconds):
    """Untimed repeats of one step (synchronised every 20 calls) until the GPU
    has run it for `seconds`, so that the clock record holds samples taken
    under load also when the timed region is short."""
    import torch
    t = time.time()
    while time.time() - t < seconds:
        for _ in range(20):
            step()
        torch.cuda.synchronize()


class ClockSampler:
    """nvidia-smi samples of SM clock, utilisation and throttle reasons: a
    background poll 50 ms apart, plus synchronous single queries (taken at
    both ends of the timed region, so that even a region shorter than the
    poll interval has clock evidence)."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
              "utilization.gpu")

    def __init__(self, index):
        self.samples = []
        self.proc = None
        self.index = index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        threading.Thread(target=self._reader, daemon=True).start()

    def _reader(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def query_once(self):
        """One synchronous sample, stamped with the time the query returned."""
        try:
            r = subprocess.run(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=10)
            line = r.stdout.strip().splitlines()[0]
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))
        except Exception:
            pass

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1, timed=None):
        """Clock record over the load window [t0, t1] (the same step running
        back to back: warm-up, timed region, untimed repeats); `timed` =
        (w0, w1) also reports the samples inside the timed region itself (the
        synchronous queries at its two ends fall on its edges)."""
        win = [(t, s) for (t, s) in self.samples if t0 <= t <= t1 and len(s) >= 8]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "samples_under_load": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        loaded = [s for _, s in win if len(s) < 9 or (num(s[8]) is not None and num(s[8]) >= 50.0)]
        use = loaded or [s for _, s in win]
        reasons = sorted({names[i] for s in use for i in range(4) if s[4 + i].lower().startswith("active")})
        sm = [num(s[0]) for s in use if num(s[0]) is not None]
        mx = [num(s[1]) for _, s in win if num(s[1]) is not None]
        pw = [num(s[2]) for s in use if num(s[2]) is not None]
        out = {"sm_mhz": statistics.median(sm) if sm else None,
               "sm_max_mhz": max(mx) if mx else None,
               "power_w_max": max(pw) if pw else None,
               "reasons": reasons, "samples": len(win), "samples_under_load": len(loaded),
               "window_s": round(t1 - t0, 3)}
        if timed is not None:
            w0, w1 = timed
            tw = [s for (t, s) in win if w0 - 0.05 <= t <= w1 + 0.05]
            tsm = [num(s[0]) for s in tw if num(s[0]) is not None]
            out["samples_timed"] = len(tw)
            out["sm_mhz_timed"] = statistics.median(tsm) if tsm else None
        return out


def reduce_max_over_ranks(values, device):
    """Element-wise max over all ranks of a list of floats (no-op on one rank).

    Used for the step and kernel times: the job is as slow as its slowest rank.
    """
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(x) for x in values]
    t = torch.tensor([float(x) for x in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_tflops(world_size, flops_per_rank_step, ms_per_step):
    """Units processed by all ranks divided by the (slowest rank's) step time."""
    return world_size * flops_per_rank_step / (ms_per_step * 1e-3) / 1e12


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def oracle_sample_rate(q, k, v, mode, p, seconds, max_blocks=None, block=64):
    """Times the oracle on row blocks taken from the end of successive heads
    (the longest rows) until `seconds` elapse.  Returns (flop/s, rows, blocks)."""
    from oracle import attention_forward
    B, H, L, d = q.shape
    done_flops = 0.0
    t0 = time.perf_counter()
    nblk = 0
    nrows = 0
    while True:
        h = nblk % (B * H)
        b, hh = divmod(h, H)
        hi = L - (nblk // (B * H)) * block % L
        lo = max(1, hi - block + 1)
        rows = np.arange(lo, hi + 1)
        qf, kf, vf = (bf16_bits_to_f64(t[b, hh, :hi]) for t in (q, k, v))
        attention_forward(qf, kf, vf, mode, p, rows=rows)
        done_flops += causal_flops_rows(rows, d, mode)
        nrows += rows.size
        nblk += 1
        el = time.perf_counter() - t0
        if el >= seconds or (max_blocks and nblk >= max_blocks):
            return done_flops / el, nrows, nblk, el


def run_reference(args, wl, mode, p):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    q, k, v = make_qkv(*wl.shape, seed=0, structure=wl.structure)
    from oracle import attention_forward
    B, H, L, d = wl.shape
    rows_per_step = 32

    def step(s):
        b, hh = divmod(s % (B * H), H)
        hi = L - ((s // (B * H)) * rows_per_step) % L
        lo = max(1, hi - rows_per_step + 1)
        rows = np.arange(lo, hi + 1)
        qf, kf, vf = (bf16_bits_to_f64(t[b, hh, :hi]) for t in (q, k, v))
        attention_forward(qf, kf, vf, mode, p, rows=rows)
        return causal_flops_rows(rows, d, mode)

    for s in range(args.warmup):
        step(s)
    t0 = time.perf_counter()
    total = 0.0
    for s in range(args.steps):
        total += step(s)
    el = time.perf_counter() - t0
    val = total / el / 1e12
    sample = (f"{args.steps} steps x {rows_per_step} query rows (the last rows of successive heads) "
              f"of the {wl.name} workload, float64 NumPy oracle")
    line = {
        "metric": METRIC, "value": val, "unit": "TFLOP/s", "impl": "reference",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(wl, mode, p),
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": os.cpu_count(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_dict(wl, mode, p):
    mname = {v: k for k, v in MODE_NAMES.items()}[mode]
    return {"workload": f"{wl.name}: B={wl.B} H={wl.H} L={wl.L} d={wl.d} {mname}"
                        + (f" p={p}" if mode in REWEIGHT_MODES else "") + f" causal, {wl.structure} bf16 inputs",
            "B": wl.B, "H": wl.H, "L": wl.L, "d": wl.d, "mode": mname, "p": p if mode in REWEIGHT_MODES else None,
            "gemms_counted": gemm_count(mode),
            "l2": "flushed before every timed step (256 MiB write); inputs 37.7 MiB < L2",
            "operands": "fp16 normalised q,k and bf16 P,V on tcgen05, fp32 accumulate, bf16 out"}


def run_ours(args, wl, mode, p):
    import torch
    ws, rank, local = dist_env()
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)   # each rank's GPU before any CUDA work or communicator
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    from lssar_attn_fwd_gb300 import api
    from lssar_attn_fwd_gb300.build import build
    if rank == 0:
        build()
    if ws > 1:
        dist.barrier()
    api.load_library()

    qb, kb, vb = make_qkv(*wl.shape, seed=rank, structure=wl.structure)
    to_t = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16)  # noqa: E731
    q_h, k_h, v_h = (to_t(b).pin_memory() for b in (qb, kb, vb))
    q, k, v = (t.to(dev) for t in (q_h, k_h, v_h))
    out = torch.empty_like(q)
    out_h = torch.empty(out.shape, dtype=torch.bfloat16).pin_memory()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    F = flops(wl.B, wl.H, wl.L, wl.d, mode)
    launches_per_step = 1 if mode == MODE_SOFTMAX else 2

    K, W = args.steps, args.warmup
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    for trio in ev:
        for e in trio:
            e.record(stream)
    sampler = ClockSampler(dev.index if dev.index is not None else 0) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.2)
    load0 = time.time()
    for _ in range(W):
        flush.zero_()
        api.lssar_attn_fwd(q, k, v, p=p, mode=mode, out=out)
    torch.cuda.synchronize(dev)

    if sampler:
        sampler.query_once()
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    w0 = time.time()
    # events only around the whole call: an event between the prologue and
    # the attention kernel would hold the kernel's launch until the prologue
    # has finished (it is a programmatic dependent of the prologue), which a
    # user's call does not do
    for i in range(K):
        flush.zero_()
        api.lssar_attn_fwd_profiled(q, k, v, p, mode, out, stream, ev[i][0], None, ev[i][2])
    torch.cuda.synchronize(dev)
    if ws > 1:
        dist.barrier()
    w1 = time.time()
    if sampler:
        sampler.query_once()
    step_ms = [ev[i][0].elapsed_time(ev[i][2]) for i in range(K)]
    assert api.device_error_word() == 0, "device error word set during the timed region"

    # the attention kernel's own time (the roofline's denominator), from the
    # same flushed steps with an event also between the prologue and the kernel
    KK = min(K, 2000)
    for i in range(KK):
        flush.zero_()
        api.lssar_attn_fwd_profiled(q, k, v, p, mode, out, stream, ev[i][0], ev[i][1], ev[i][2])
    torch.cuda.synchronize(dev)
    kern_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(KK)]
    tot, kern_mean = reduce_max_over_ranks([sum(step_ms), sum(kern_ms) / KK], dev)
    kern_median = statistics.median(kern_ms)
    assert api.device_error_word() == 0, "device error word set while timing the kernel"

    # for reference, outside the timed region: the same steps without the L2
    # flush between them (the step's inputs then stay in L2)
    KW = min(K, 200)
    for i in range(KW):
        api.lssar_attn_fwd_profiled(q, k, v, p, mode, out, stream, ev[i][0], ev[i][1], ev[i][2])
    torch.cuda.synchronize(dev)
    warm_ms = sum(ev[i][0].elapsed_time(ev[i][2]) for i in range(KW)) / KW
    warm_kern_ms = sum(ev[i][1].elapsed_time(ev[i][2]) for i in range(KW)) / KW

    # end to end through the public API: every step copies its inputs from
    # pinned host memory, runs lssar_attn_fwd and copies its output back.  As a
    # user's input pipeline would, the copies run on their own streams over two
    # buffer sets, so that the copy-in of step i+1 and the copy-out of step i-1
    # overlap the kernel of step i; every copy of every step is inside [e0, e1].
    KE = max(3, min(K, 100))
    h2d, d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    bufs = [(q, k, v, out)] + [tuple(torch.empty_like(t) for t in (q, k, v, out))]
    ev_in = [torch.cuda.Event() for _ in range(2)]      # inputs of buffer b landed
    ev_run = [torch.cuda.Event() for _ in range(2)]     # kernel on buffer b done
    ev_out = [torch.cuda.Event() for _ in range(2)]     # output of buffer b copied out
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for it in range(2):
        torch.cuda.synchronize(dev)
        e0.record(stream)
        h2d.wait_event(e0)
        d2h.wait_event(e0)
        steps = KE if it else 2
        for i in range(steps):
            b = i % 2
            qb_, kb_, vb_, ob_ = bufs[b]
            with torch.cuda.stream(h2d):
                if i >= 2:
                    h2d.wait_event(ev_run[b])            # buffer b's previous kernel read its inputs
                qb_.copy_(q_h, non_blocking=True)
                kb_.copy_(k_h, non_blocking=True)
                vb_.copy_(v_h, non_blocking=True)
                ev_in[b].record(h2d)
            stream.wait_event(ev_in[b])
            if i >= 2:
                stream.wait_event(ev_out[b])             # buffer b's previous output is out
            api.lssar_attn_fwd(qb_, kb_, vb_, p=p, mode=mode, out=ob_, stream=stream)
            ev_run[b].record(stream)
            with torch.cuda.stream(d2h):
                d2h.wait_event(ev_run[b])
                out_h.copy_(ob_, non_blocking=True)
                ev_out[b].record(d2h)
        for b in range(2):
            stream.wait_event(ev_out[b])
        e1.record(stream)
        torch.cuda.synchronize(dev)
    e2e_ms = reduce_max_over_ranks([e0.elapsed_time(e1) / KE], dev)[0]
    # the same steps with copies and kernel back to back on one stream (no
    # overlap), reported beside the pipelined figure to show the copy cost
    for it in range(2):
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(KE if it else 2):
            with torch.cuda.stream(stream):
                q.copy_(q_h, non_blocking=True)
                k.copy_(k_h, non_blocking=True)
                v.copy_(v_h, non_blocking=True)
            api.lssar_attn_fwd(q, k, v, p=p, mode=mode, out=out, stream=stream)
            with torch.cuda.stream(stream):
                out_h.copy_(out, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize(dev)
    serial_ms = reduce_max_over_ranks([e0.elapsed_time(e1) / KE], dev)[0]
    # untimed repeats of the timed step (same flush, same call) until the GPU
    # has run this load for MIN_LOAD_S, so that the clock record has samples
    # under load even when the timed region is shorter than the poll interval
    while time.time() - load0 < MIN_LOAD_S:
        for _ in range(20):
            flush.zero_()
            api.lssar_attn_fwd(q, k, v, p=p, mode=mode, out=out)
        torch.cuda.synchronize(dev)
    load1 = time.time()
    if sampler:
        sampler.query_once()
        time.sleep(0.1)
        sampler.stop()

    if rank == 0:
        ms = tot / K
        value = whole_job_tflops(ws, F, ms)
        peak, peak_kind = peaks()
        achieved = F / (kern_mean * 1e-3) / 1e12
        cpu = None
        if ws == 1 and not args.no_cpu_baseline:
            rate, nrows, nblk, el = oracle_sample_rate(qb, kb, vb, mode, p, seconds=args.cpu_seconds)
            cpu = {"value": rate / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                   "sample": f"{nrows} query rows ({nblk} blocks of 64, the last rows of successive heads) "
                             f"of this workload, float64 NumPy oracle, {el:.1f} s; cores = host threads "
                             "available to its BLAS"}
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": K, "warmup": W,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic", "config": config_dict(wl, mode, p),
            "pct_bf16_peak": 100.0 * value / ws / peak,
            "pct_bf16_spec_peak": 100.0 * value / ws / SPEC_DENSE_BF16_TFLOPS,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "peak_source": f"{peak_kind} bf16_tflops (burst)",
                         "frac_of_spec_dense_bf16": achieved / SPEC_DENSE_BF16_TFLOPS,
                         "kernel": "lssar_tc_kernel", "kernel_ms": kern_mean,
                         "kernel_ms_median": kern_median,
                         "kernel_steps": KK,
                         "kernel_timing": "separate flushed steps with an event also between the prologue "
                                          "and the kernel (value's steps record none there)",
                         "traffic": kernel_traffic(wl.name, mode, p)},
            "warm": {"value": F / (warm_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": warm_ms,
                     "kernel_ms": warm_kern_ms, "kernel_tflops": F / (warm_kern_ms * 1e-3) / 1e12,
                     "steps": KW, "note": "not timed for value: no L2 flush between steps, rank 0"},
            "e2e": {"value": whole_job_tflops(ws, F, e2e_ms), "unit": "TFLOP/s",
                    "ms_per_step": e2e_ms,
                    "pipeline": "copy-in of step i+1 and copy-out of step i-1 on their own streams "
                                "overlap the kernel of step i (two device buffer sets)",
                    "serial": {"value": whole_job_tflops(ws, F, serial_ms), "ms_per_step": serial_ms,
                               "note": "copies and kernel back to back on one stream"},
                    "l2": "no flush between steps: every step's inputs are written by that step's "
                          "host-to-device copy, and the kernel reads them where the copy left them "
                          "(in L2 when they fit, as in a user's input pipeline); the device-resident "
                          "value flushes L2 before every step instead",
                    "h2d_bytes_per_step": 3 * q.numel() * 2, "d2h_bytes_per_step": out.numel() * 2},
            "gpu_launches": K * launches_per_step,
            "clocks": sampler.summary(load0, load1, timed=(w0, w1)) if sampler else None,
            "wall_s_timed": w1 - w0,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def run_decode(args, mode, p):
    """Decode step: one query per head (position L) against a K/V cache,
    B=8 H=12 L=16384 d=64 unless overridden.  Bound by HBM: the metric is the
    K/V cache bytes read per second against the measured copy bandwidth."""
    import torch
    from lssar_attn_fwd_gb300 import api
    from lssar_attn_fwd_gb300.build import build
    build()
    api.load_library()
    B, H, L, d = args.decode_shape
    qb, kb, vb = make_qkv(B, H, L, d, seed=0)
    to_t = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()  # noqa: E731
    q, k, v = to_t(qb[:, :, -1]), to_t(kb), to_t(vb)
    out = torch.empty_like(q)
    cache_bytes = 2 * B * H * L * d * 2
    # A cache of at least twice the L2 size leaves nothing of the previous
    # step's keys in L2 by the time they are read again: no flush (a write
    # flush would also leave dirty lines whose write-back competes with the
    # step).  Smaller caches are flushed by a 256 MiB write before each step.
    flush_each = cache_bytes < 2 * L2_BYTES
    flush = torch.empty(FLUSH_BYTES if flush_each else 1, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream()
    for _ in range(args.warmup):
        api.lssar_attn_decode(q, k, v, p=p, mode=mode, out=out)
    plan = api.decode_plan(B, H, L, d)   # path, launches per step, chunking
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    torch.cuda.synchronize()
    sampler.query_once()
    t0 = time.time()
    for a, b in ev:
        if flush_each:
            flush.zero_()
        a.record(s)
        api.lssar_attn_decode(q, k, v, p=p, mode=mode, out=out)
        b.record(s)
    torch.cuda.synchronize()
    t1 = time.time()
    sampler.query_once()

    def step():
        if flush_each:
            flush.zero_()
        api.lssar_attn_decode(q, k, v, p=p, mode=mode, out=out)
    hold_load(step, MIN_LOAD_S)
    t2 = time.time()
    sampler.query_once()
    sampler.stop()
    ms = sum(a.elapsed_time(b) for a, b in ev) / len(ev)
    gbs = cache_bytes / (ms * 1e-3) / 1e9
    try:
        peak = float(json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["hbm_gbs"])
        kind = "measured"
    except Exception:
        peak, kind = 6800.0, "fallback"
    print(json.dumps({
        "metric": "LSSAR decode step: K/V cache bytes read per second", "value": gbs, "unit": "GB/s",
        "ms_per_step": ms, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
        "config": {"workload": f"decode: B={B} H={H} L={L} d={d} mode={mode} p={p}, one query per head",
                   "l2": ("flushed before every step (256 MiB write)" if flush_each else
                          f"not flushed: the {cache_bytes / 2**20:.0f} MiB cache is over twice the L2 size")},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                     "peak_source": f"{kind} hbm_gbs"},
        "plan": plan,
        "clocks": sampler.summary(t0, t2, timed=(t0, t1)),
        "gpu_launches": plan["launches"] * args.steps}), flush=True)


def run_backward(args, wl, mode, p):
    """Backward step: lssar_attn_bwd (row pass, column pass, normalisation
    gradient) on the workload's q, k, v and a seeded upstream gradient, with
    the row statistics of one lssar_attn_fwd_train call made before timing.
    FLOPs: the five causal products of an attention backward (S recomputed,
    dP = dO V^T, dV = P^T dO, dQ = dS K, dK = dS^T Q), 10 d per causal score
    element; the kernels execute nine (the row pass streams the keys twice)."""
    import torch
    from lssar_attn_fwd_gb300 import api
    from lssar_attn_fwd_gb300.build import build
    from lssar_attn_fwd_gb300.inputs import make_dout
    build()
    api.load_library()
    B, H, L, d = wl.B, wl.H, wl.L, wl.d
    qb, kb, vb = make_qkv(*wl.shape, seed=0, structure=wl.structure)
    db = make_dout(B, H, L, d, seed=0)
    to_t = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()  # noqa: E731
    q, k, v, dout = (to_t(x) for x in (qb, kb, vb, db))
    _, stats = api.lssar_attn_fwd_train(q, k, v, p=p, mode=mode)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream()
    for _ in range(args.warmup):
        api.lssar_attn_bwd(q, k, v, dout, stats, p=p, mode=mode)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    torch.cuda.synchronize()
    sampler.query_once()
    t0 = time.time()
    for a, b in ev:
        flush.zero_()
        a.record(s)
        api.lssar_attn_bwd(q, k, v, dout, stats, p=p, mode=mode)
        b.record(s)
    torch.cuda.synchronize()
    t1 = time.time()
    sampler.query_once()

    def step():
        flush.zero_()
        api.lssar_attn_bwd(q, k, v, dout, stats, p=p, mode=mode)
    hold_load(step, MIN_LOAD_S)
    t2 = time.time()
    sampler.query_once()
    sampler.stop()
    assert api.device_error_word() == 0
    ms = sum(a.elapsed_time(b) for a, b in ev) / len(ev)
    elems = B * H * L * (L + 1) / 2
    tflops = 10 * d * elems / (ms * 1e-3) / 1e12
    peak, kind = peaks()
    mname = {v: k for k, v in MODE_NAMES.items()}[mode]
    print(json.dumps({
        "metric": "LSSAR causal bwd TFLOP/s (5 GEMMs: S, dP, dV, dQ, dK)", "value": tflops,
        "unit": "TFLOP/s", "ms_per_step": ms, "steps": args.steps, "warmup": args.warmup,
        "higher_is_better": True, "dtype": "fp16/bf16 operands, fp32 accumulate",
        "config": {"workload": f"backward: {wl.name} B={B} H={H} L={L} d={d} mode={mname} p={p}",
                   "l2": "flushed before every step (256 MiB write)"},
        "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                     "frac": tflops / peak, "peak_source": f"{kind} bf16_tflops (burst)"},
        "clocks": sampler.summary(t0, t2, timed=(t0, t1)),
        "gpu_launches": (3 if uses_normalised(mode) else 2) * args.steps}), flush=True)   # prologue, row, column pass


def uses_normalised(mode):
    return mode in (MODE_LSSA, MODE_LSSAR, MODE_SIGMOID_RW)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="extrap", choices=sorted(WORKLOADS))
    ap.add_argument("--mode", default=None, choices=sorted(MODE_NAMES))
    ap.add_argument("--p", type=int, default=None)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode", action="store_true", help="benchmark the decode step instead")
    ap.add_argument("--backward", action="store_true", help="benchmark the backward pass instead")
    ap.add_argument("--decode-shape", type=int, nargs=4, default=[8, 12, 16384, 64],
                    metavar=("B", "H", "L", "D"))
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    wl = WORKLOADS[args.workload]
    mode, p = wl.runs[0]
    if args.mode is not None:
        mode = MODE_NAMES[args.mode]
    if args.p is not None:
        p = args.p
    if args.decode:
        run_decode(args, mode, p)
    elif args.backward:
        run_backward(args, wl, mode, p)
    elif args.impl == "reference":
        run_reference(args, wl, mode, p)
    else:
        run_ours(args, wl, mode, p)


if __name__ == "__main__":
    main()
