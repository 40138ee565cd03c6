"""Benchmark: fused multi-head scaled dot-product attention forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one forward pass of the whole hot path (one ``attn_fwd`` call: QK^T,
mask, online softmax, PV, epilogue) over one batch of the workload.  The
default workload is the base encoder self-attention (B=64, h=8, n_q=n_k=512,
d_k=d_v=64, bf16, no mask).  Prints ONE JSON line (rank 0).

Backward workloads (names ending in ``_bwd``): one step = one ``attn_bwd``
call (its three kernels) on the same problems, O and LSE computed once by the
forward beforehand; FLOPs count the five n_q x n_k x d products of the
backward (2.5 times the forward's).  Decoding workloads: one ``attn_decode``
call, reported against HBM bandwidth.

Timing: W untimed warm-up steps, then K timed steps.  Before every timed step
the L2 is flushed by writing a 256 MiB buffer and then reading another one, so
that the timed step finds a cold L2 holding only clean lines (outside the timed interval);
each step is bracketed by CUDA events on the launching stream, and the whole
timed loop by a barrier and a device synchronisation on both sides.  SM clocks
are sampled with nvidia-smi during the timed loop.

``--impl reference`` times the float64 CPU oracle (the only reference this
method has) on a bounded sample of the same workload, on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from transformer_head_scaled_gb300 import inputs, shard  # noqa: E402

L2_FLUSH_BYTES = 256 << 20
METRIC = "fused attention fwd TFLOP/s (bf16) and % of GB300 dense BF16 tensor peak"
METRIC_BWD = "fused attention bwd TFLOP/s (bf16) and % of GB300 dense BF16 tensor peak"


def metric_name(w: inputs.Workload) -> str:
    """The forward's metric; backward workloads report the same quantity for the backward."""
    return METRIC_BWD if w.kind == "bwd" else METRIC


# The sources of each pass's main kernel, and the committed ncu DRAM bytes per
# launch measured for that exact source (matched by hash).
_CSRC = "transformer_head_scaled_gb300/csrc/"
KERNEL_SOURCES = {
    "fwd": (_CSRC + "attn_fwd_tc.cu", _CSRC + "ptx.cuh"),
    "bwd": (_CSRC + "attn_bwd.cu", _CSRC + "ptx.cuh"),
    "decode": (_CSRC + "attn_decode.cu", _CSRC + "ptx.cuh"),
}
TRAFFIC_FILES = {
    "fwd": os.path.join(ROOT, "profiles", "attn_fwd_tc_traffic.json"),
    "bwd": os.path.join(ROOT, "profiles", "attn_bwd_tc_traffic.json"),
    "decode": os.path.join(ROOT, "profiles", "attn_decode_traffic.json"),
}


def kernel_hash(kind: str = "fwd") -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        d["_source"] = "measured"
        return d
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0,
            "_source": "fallback"}


def dram_traffic(w: inputs.Workload):
    """ncu DRAM bytes per launch of this pass's main kernel for its current
    source and this workload, or None."""
    path = TRAFFIC_FILES[w.kind]
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(w.name)
    if not e or e.get("kernel_hash") != kernel_hash(w.kind):
        return None
    return e.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi SM-clock / throttle-reason samples while running."""

    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.out = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t_start: float, t_end: float) -> dict:
        if self.proc is None or self.out is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.out.seek(0)
        rows = [r.split(", ") for r in self.out.read().strip().splitlines() if r.count(",") >= 9]
        load, allr = [], []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        max_mhz = None
        for r in rows:
            try:
                ts = time.mktime(time.strptime(r[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                sm, mx = float(r[2]), float(r[3])
            except ValueError:
                continue
            max_mhz = mx
            allr.append(sm)
            if t_start - 1.0 <= ts <= t_end + 1.0:
                load.append(sm)
                for name, val in zip(names, r[6:10]):
                    if val.strip() == "Active":
                        reasons.add(name)
        vals = load or allr
        return {"sm_mhz": statistics.median(vals) if vals else None, "sm_max_mhz": max_mhz,
                "reasons": sorted(reasons), "samples": len(load)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def workload_desc(w: inputs.Workload) -> str:
    mask = {0: "no mask", 1: "causal", 2: f"key padding L~U[{w.lens_lo},n_k]",
            3: f"window i-{w.win_left}..i+{w.win_right}"}[w.mask]
    if inputs.decode_window(w) is not None:
        mask += f", keys L-1-{inputs.decode_window(w)}..L-1"
    return f"{w.name}: B={w.B} h={w.h} n_q={w.n_q} n_k={w.n_k} d_k=d_v={w.d} {w.dtype} {mask}"


# ---------------------------------------------------------------------- oracle (CPU)

def _row_flops(w: inputs.Workload, rows, lens) -> float:
    if w.mask == inputs.MASK_NONE:
        keys = np.full(rows.size, w.n_k)
    elif w.mask == inputs.MASK_CAUSAL:
        keys = np.minimum(rows % w.n_q + 1, w.n_k)
    elif w.mask == inputs.MASK_BAND:
        i = rows % w.n_q
        keys = np.maximum(np.minimum(w.n_k - 1, i + w.win_right) - np.maximum(0, i - w.win_left) + 1, 0)
    else:
        keys = inputs.seen_keys(w, lens[(rows // w.n_q) // w.h])
    return float(4.0 * w.d * keys.sum())


def _oracle_rows(oracle, w, q, k, v, rows, kl, threads):
    if w.mask == inputs.MASK_BAND:
        return oracle.attn_band(q, k, v, w.scale, w.win_left, w.win_right, rows=rows,
                                threads=threads)
    win = inputs.decode_window(w)
    if win is not None:
        # restricted decoding step: batch entry b's rows against its window's
        # slice of the cache
        lens = np.asarray(kl.cpu())
        per_b = w.h * w.n_q
        for b in np.unique(rows // per_b):
            L = int(min(max(lens[b], 0), w.n_k))
            lo = max(0, L - 1 - win)
            sub = rows[rows // per_b == b] - b * per_b
            if L > lo:
                oracle.attn_rows(q[b:b + 1], k[b:b + 1, :, lo:L], v[b:b + 1, :, lo:L], sub,
                                 w.scale, inputs.MASK_NONE, threads=threads)
        return None
    return oracle.attn_rows(q, k, v, rows, w.scale, w.mask, kl, threads=threads)


def oracle_sample(w: inputs.Workload, q, k, v, kl, target_s: float, threads: int = 0,
                  rows_hint: int | None = None):
    """Time the float64 oracle on a sample of the workload's query rows, about
    target_s seconds of work (whole passes over the workload when it is
    shorter).  Returns (tflops, seconds, rows_done, flops)."""
    import oracle
    oracle.build()
    total_rows = w.B * w.h * w.n_q
    lens = None if kl is None else np.asarray(kl.cpu())
    rng = np.random.default_rng(123)
    if rows_hint is None:
        n = min(total_rows, 1024)
        rows = np.sort(rng.choice(total_rows, size=n, replace=False))
        t0 = time.perf_counter()
        _oracle_rows(oracle, w, q, k, v, rows, kl, threads)
        per_row = (time.perf_counter() - t0) / n
        rows_hint = max(1, int(target_s / max(per_row, 1e-9)))
    done, flops, dt = 0, 0.0, 0.0
    while done < rows_hint:
        n = min(total_rows, rows_hint - done)
        rows = (np.arange(total_rows, dtype=np.int64) if n == total_rows
                else np.sort(rng.choice(total_rows, size=n, replace=False)))
        t0 = time.perf_counter()
        _oracle_rows(oracle, w, q, k, v, rows, kl, threads)
        dt += time.perf_counter() - t0
        flops += _row_flops(w, rows, lens)
        done += n
    return flops / dt / 1e12, dt, done, flops


def oracle_bwd_sample(w: inputs.Workload, q, k, v, g, kl, target_s: float, threads: int = 0,
                      heads_hint: int | None = None):
    """Time the float64 oracle's backward on whole sampled heads (a head's
    gradients depend only on its own data), about target_s seconds of work.
    Returns (tflops, seconds, heads_done, flops)."""
    import oracle
    oracle.build()
    BH = w.B * w.h
    lens = None if kl is None else np.asarray(kl.cpu()).astype(np.int32)
    rng = np.random.default_rng(321)

    def run(sel):
        b_idx, h_idx = sel // w.h, sel % w.h
        sub = lambda t: np.ascontiguousarray(t[b_idx, h_idx][:, None])  # noqa: E731
        sl = None if lens is None else lens[b_idx]
        t0 = time.perf_counter()
        if w.mask == inputs.MASK_BAND:
            oracle.attn_bwd_band(sub(q), sub(k), sub(v), sub(g), w.scale, w.win_left,
                                 w.win_right, threads=threads)
        else:
            oracle.attn_bwd(sub(q), sub(k), sub(v), sub(g), w.scale, w.mask, sl, threads=threads)
        dt = time.perf_counter() - t0
        rows = np.concatenate([np.arange(w.n_q) + int(bh) * w.n_q for bh in sel])
        return dt, _row_flops(w, rows, lens) * inputs.products(w) / 2.0

    if heads_hint is None:
        n = min(BH, max(1, oracle.max_threads()))
        dt, _ = run(np.sort(rng.choice(BH, size=n, replace=False)))
        heads_hint = max(1, int(n * target_s / max(dt, 1e-9)))
    done, flops, dt = 0, 0.0, 0.0
    while done < heads_hint:
        n = min(BH, heads_hint - done)
        sel = np.sort(rng.choice(BH, size=n, replace=False))
        d, f = run(sel)
        dt += d
        flops += f
        done += n
    return flops / dt / 1e12, dt, done, flops


def cpu_cores_used() -> int:
    import oracle
    return oracle.max_threads()


# ---------------------------------------------------------------------- reference arm

def run_reference(args, w):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    q, k, v, kl = inputs.make_inputs(w)
    qf, kf, vf = q.float().numpy(), k.float().numpy(), v.float().numpy()
    bwd = w.kind == "bwd"
    gf = inputs.make_dout(w).float().numpy() if bwd else None
    # the whole run (warm-up included) is sized to about two minutes of CPU time
    per_step = min(20.0, 120.0 / max(1, args.steps + args.warmup))
    if bwd:
        sample = lambda target, hint: oracle_bwd_sample(  # noqa: E731
            w, qf, kf, vf, gf, kl, target, heads_hint=hint)
    else:
        sample = lambda target, hint: oracle_sample(  # noqa: E731
            w, qf, kf, vf, kl, target, rows_hint=hint)
    _, dt, n, _ = sample(min(per_step, 1.0), None)
    per_step_units = max(1, int(n * per_step / max(dt, 1e-9)))
    for _ in range(args.warmup):
        sample(0.0, per_step_units)
    vals, secs, fls = [], [], []
    for _ in range(args.steps):
        tf, dt, _, fl = sample(0.0, per_step_units)
        vals.append(tf)
        secs.append(dt)
        fls.append(fl)
    value = statistics.median(vals)
    cores = cpu_cores_used()
    if bwd:
        total = w.B * w.h
        desc = (f"{per_step_units} whole heads per step ({per_step_units / total:.2f} passes over "
                f"the {total} heads of the workload; dQ, dK, dV of each), float64")
    else:
        total = w.B * w.h * w.n_q
        desc = (f"{per_step_units} query rows per step ({per_step_units / total:.2f} passes over "
                f"the {total} rows of the workload, each against all its visible keys), float64")
    line = {
        "impl": "reference", "metric": metric_name(w), "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.median(secs), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_desc(w), "global_batch": w.B,
                   "parallelism": "host cores of rank 0 (the float64 oracle; no GPU)",
                   "l2": "n/a (CPU)", "flops_per_step": inputs.flops(w),
                   "sample_flops_per_step": statistics.median(fls)},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------- our arm

def run_ours(args, w):
    from transformer_head_scaled_gb300 import binding
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    binding.load()

    # weak scaling: every rank owns a slice of B batch entries of a global
    # batch of world * B (independent (batch, head) problems, no exchange)
    q, k, v, kl = inputs.make_inputs(w, device=dev, seeds=shard.rank_seeds(rank))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.h, w.n_q), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    clean = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2():
        # write a buffer larger than L2, then read another one: the timed
        # step starts with a cold L2 that holds only clean, unrelated lines
        # (no write-backs of the flush's dirty lines inside the timed region)
        flush.zero_()
        clean.sum()
    stream = torch.cuda.current_stream(dev)
    sptr = int(stream.cuda_stream)
    f32 = w.dtype == "f32"
    ptrs = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr())
    klp = None if kl is None else kl.data_ptr()
    decode = w.kind == "decode"
    bwd = w.kind == "bwd"
    if decode:
        ws_bytes = binding.decode_workspace_bytes(w.B, w.h, w.n_q, w.n_k, w.d,
                                                  inputs.decode_window(w))
    elif bwd:
        ws_bytes = binding.bwd_workspace_bytes(w.B, w.h, w.n_q, w.d)
    else:
        ws_bytes = 0
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    g = None
    if bwd:
        # O and LSE of the same inputs come from the forward, outside the timing
        g = inputs.make_dout(w, device=dev, seed=inputs.SEED_DOUT + 8 * rank)
        if w.mask == inputs.MASK_BAND:
            binding.attn_fwd_window(q, k, v, w.win_left, w.win_right, scale=w.scale, out=o,
                                    lse=lse)
        else:
            binding.attn_fwd(q, k, v, scale=w.scale, mask=w.mask, key_lens=kl, out=o, lse=lse)
        grads = [torch.empty_like(t) for t in (q, k, v)]
        bptrs = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), g.data_ptr(),
                 lse.data_ptr(), *(t.data_ptr() for t in grads))

    def step():
        if decode and inputs.decode_window(w) is not None:
            rc = binding.attn_decode_window_raw(*ptrs, w.B, w.h, w.n_q, w.n_k, w.d, w.scale, klp,
                                                inputs.decode_window(w), ws.data_ptr(), ws_bytes,
                                                sptr)
        elif decode:
            rc = binding.attn_decode_raw(*ptrs, w.B, w.h, w.n_q, w.n_k, w.d, w.scale, klp,
                                         ws.data_ptr(), ws_bytes, sptr)
        elif bwd and w.mask == inputs.MASK_BAND:
            rc = binding.attn_bwd_window_raw(*bptrs, w.B, w.h, w.n_q, w.n_k, w.d, w.scale,
                                             w.win_left, w.win_right, ws.data_ptr(), ws_bytes,
                                             sptr)
        elif bwd:
            rc = binding.attn_bwd_raw(*bptrs, w.B, w.h, w.n_q, w.n_k, w.d, w.scale, w.mask, klp,
                                      ws.data_ptr(), ws_bytes, sptr)
        elif w.mask == inputs.MASK_BAND:
            rc = binding.attn_fwd_window_raw(*ptrs, w.B, w.h, w.n_q, w.n_k, w.d, w.scale,
                                             w.win_left, w.win_right, sptr)
        else:
            rc = binding.attn_fwd_raw(*ptrs, w.B, w.h, w.n_q, w.n_k, w.d, w.scale, w.mask, klp,
                                      sptr, f32=f32)
        if rc != 0:
            raise binding.AttnError(rc, w.kind)

    for _ in range(max(3, args.warmup)):
        flush_l2()
        step()
    binding.check(stream)

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    launches0 = binding.launch_count()
    with ClockSampler(local) as clocks:
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)
        t_start = time.time()
        wall0 = time.perf_counter()
        for i in range(args.steps):
            flush_l2()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()
        wall = time.perf_counter() - wall0
        t_end = time.time()
    launches = binding.launch_count() - launches0
    binding.check(stream)
    times = [s.elapsed_time(e) for s, e in zip(starts, ends)]  # ms
    ms = sum(times) / len(times)
    ms = shard.max_over_ranks(ms, device=dev)
    ms_median = shard.max_over_ranks(statistics.median(times), device=dev)
    ms_best = shard.max_over_ranks(min(times), device=dev)

    fl = inputs.flops(w)
    fl_alg = inputs.algorithmic_flops(w, kl)
    value = world * fl / (ms * 1e-3) / 1e12
    peaks = measured_peaks()
    achieved = fl_alg / (ms * 1e-3) / 1e12
    hbm = inputs.hbm_bytes(w, kl)

    # end to end through the public API: pinned host inputs -> device -> call -> host
    e2e = (run_e2e_bwd(args, w, q, k, v, o, lse, g, kl, dev, stream) if bwd else
           run_e2e(args, w, q, k, v, kl, dev, stream, f32))

    clk = clocks.summary(t_start, t_end)
    line = {
        "metric": metric_name(w), "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "ms_median": ms_median, "ms_best": ms_best,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32" if f32 else "bf16", "data": "synthetic",
        "config": {"workload": workload_desc(w), "global_batch": world * w.B,
                   "parallelism": f"dp{world}: batch entries split across ranks, no collective on the data path",
                   "l2": "flushed before every timed step (256 MiB write, then 256 MiB read so that no dirty line is written back inside the timed step; outside the events)",
                   "flops_per_step": fl, "algorithmic_flops_per_step": fl_alg,
                   "hbm_bytes_per_step": hbm, "timed_loop_wall_s": wall},
        "pct_of_peak": 100.0 * (value / world) / peaks["bf16_tflops"],
        "roofline": ({"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                      "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                      "traffic": dram_traffic(w),
                      "peak_source": f"{peaks['_source']} bf16_tflops (burst; kernel timed alone)",
                      "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
                      "hbm_gbs": hbm / (ms * 1e-3) / 1e9,
                      "kernel": ("attn_bwd_tc_kernel, timed together with its preprocess and "
                                 "dQ-convert launches (one C call)") if bwd else
                                ("attn_fwd_tc_kernel" if not f32 else "attn_fwd_f32_kernel")}
                     if not decode else
                     {"bound": "hbm", "achieved": hbm / (ms * 1e-3) / 1e9, "peak": peaks["hbm_gbs"],
                      "unit": "GB/s", "frac": hbm / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                      "traffic": dram_traffic(w), "algorithmic_bytes": hbm,
                      "peak_source": f"{peaks['_source']} hbm_gbs (copy bandwidth)",
                      "kernel": ("attn_decode_split_kernel" if w.d == 64 else "attn_decode_rows_kernel")
                                + (" + combine" if ws_bytes else "")}),
        "e2e": e2e,
        "gpu_launches": int(launches),
        "clocks": {k2: clk[k2] for k2 in ("sm_mhz", "sm_max_mhz", "reasons")},
    }
    if rank == 0 and not args.no_cpu_baseline:
        qf, kf, vf = (t.float().cpu().numpy() for t in (q, k, v))
        if bwd:
            gf = g.float().cpu().numpy()
            tf, dt, nh, _ = oracle_bwd_sample(w, qf, kf, vf, gf, kl, target_s=args.cpu_seconds)
            desc = (f"{nh} whole heads of the {w.B * w.h} of the same workload (dQ, dK, dV of "
                    f"each), float64, {dt:.1f} s")
        else:
            tf, dt, nrows, _ = oracle_sample(w, qf, kf, vf, kl, target_s=args.cpu_seconds)
            desc = (f"{nrows} query rows ({nrows / (w.B * w.h * w.n_q):.2f} passes over the "
                    f"{w.B * w.h * w.n_q} rows of the same workload), float64, {dt:.1f} s")
        line["cpu_baseline"] = {"value": tf, "unit": "TFLOP/s", "cores": cpu_cores_used(),
                                "kind": "oracle", "sample": desc}
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_e2e(args, w, q, k, v, kl, dev, stream, f32):
    from transformer_head_scaled_gb300 import binding
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
    hkl = None if kl is None else kl.cpu().pin_memory()
    ho = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    hl = torch.empty((w.B, w.h, w.n_q), dtype=torch.float32).pin_memory()
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dkl = None if kl is None else torch.empty_like(kl)
    do = torch.empty_like(q)
    dl = torch.empty((w.B, w.h, w.n_q), dtype=torch.float32, device=dev)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv)) + (
        0 if hkl is None else hkl.numel() * 4)
    d2h = ho.numel() * ho.element_size() + hl.numel() * 4
    sptr = int(stream.cuda_stream)
    ws_bytes = (binding.decode_workspace_bytes(w.B, w.h, w.n_q, w.n_k, w.d,
                                               inputs.decode_window(w))
                if w.kind == "decode" else 0)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    # the bf16 forward goes through attn_fwd_host: host buffers in and out, the
    # copies pipelined with the kernels over batch slices inside the call
    host_api = w.kind == "fwd" and not f32
    if host_api:
        band = w.mask == inputs.MASK_BAND
        stage = torch.empty(binding.host_buffer_bytes(w.B, w.h, w.n_q, w.n_k, w.d),
                            dtype=torch.uint8, device=dev)

    def step():
        if host_api:
            rc = binding.attn_fwd_host_raw(
                hq.data_ptr(), hk.data_ptr(), hv.data_ptr(), ho.data_ptr(), hl.data_ptr(), w.B,
                w.h, w.n_q, w.n_k, w.d, w.scale, inputs.MASK_BAND if band else w.mask,
                None if hkl is None else hkl.data_ptr(), w.win_left if band else 0,
                w.win_right if band else 0, stage.data_ptr(), stage.numel(), sptr)
            if rc != 0:
                raise binding.AttnError(rc, "attn_fwd_host")
            return
        dq.copy_(hq, non_blocking=True)
        dk.copy_(hk, non_blocking=True)
        dv.copy_(hv, non_blocking=True)
        if dkl is not None:
            dkl.copy_(hkl, non_blocking=True)
        if w.kind == "decode" and inputs.decode_window(w) is not None:
            rc = binding.attn_decode_window_raw(dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                                do.data_ptr(), dl.data_ptr(), w.B, w.h, w.n_q,
                                                w.n_k, w.d, w.scale,
                                                None if dkl is None else dkl.data_ptr(),
                                                inputs.decode_window(w), ws.data_ptr(), ws_bytes,
                                                sptr)
        elif w.kind == "decode":
            rc = binding.attn_decode_raw(dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                         do.data_ptr(), dl.data_ptr(), w.B, w.h, w.n_q, w.n_k,
                                         w.d, w.scale, None if dkl is None else dkl.data_ptr(),
                                         ws.data_ptr(), ws_bytes, sptr)
        elif w.mask == inputs.MASK_BAND:
            rc = binding.attn_fwd_window_raw(dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                             do.data_ptr(), dl.data_ptr(), w.B, w.h, w.n_q, w.n_k,
                                             w.d, w.scale, w.win_left, w.win_right, sptr)
        else:
            rc = binding.attn_fwd_raw(dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), do.data_ptr(),
                                      dl.data_ptr(), w.B, w.h, w.n_q, w.n_k, w.d, w.scale,
                                      w.mask, None if dkl is None else dkl.data_ptr(), sptr,
                                      f32=f32)
        if rc != 0:
            raise binding.AttnError(rc, "attention")
        ho.copy_(do, non_blocking=True)
        hl.copy_(dl, non_blocking=True)

    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    n = max(3, min(args.steps, 50))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    binding.check(stream)
    ms = e0.elapsed_time(e1) / n
    world = dist_env()[0]
    return {"value": world * inputs.flops(w) / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": ms,
            "steps": n, "call": ("attn_fwd_host (host buffers; copies pipelined over batch "
                                 "slices)" if host_api else
                                 "host-to-device copies, the device call, device-to-host copies")}


def run_e2e_bwd(args, w, q, k, v, o, lse, g, kl, dev, stream):
    """The backward end to end: Q, K, V, O, LSE, dO (and key lengths) copied in
    from pinned host memory, dQ, dK, dV copied back, every step."""
    from transformer_head_scaled_gb300 import binding
    host_in = [t.cpu().pin_memory() for t in (q, k, v, o, lse, g)]
    hkl = None if kl is None else kl.cpu().pin_memory()
    dev_in = [torch.empty_like(t) for t in (q, k, v, o, lse, g)]
    dkl = None if kl is None else torch.empty_like(kl)
    dev_out = [torch.empty_like(t) for t in (q, k, v)]
    host_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in dev_out]
    ws_bytes = binding.bwd_workspace_bytes(w.B, w.h, w.n_q, w.d)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    h2d = sum(t.numel() * t.element_size() for t in host_in) + (0 if hkl is None else hkl.numel() * 4)
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    sptr = int(stream.cuda_stream)

    def step():
        for d, h in zip(dev_in, host_in):
            d.copy_(h, non_blocking=True)
        if dkl is not None:
            dkl.copy_(hkl, non_blocking=True)
        qd, kd, vd, od, ld, gd = dev_in
        if w.mask == inputs.MASK_BAND:
            rc = binding.attn_bwd_window_raw(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(),
                                             od.data_ptr(), gd.data_ptr(), ld.data_ptr(),
                                             *(t.data_ptr() for t in dev_out), w.B, w.h, w.n_q,
                                             w.n_k, w.d, w.scale, w.win_left, w.win_right,
                                             ws.data_ptr(), ws_bytes, sptr)
        else:
            rc = binding.attn_bwd_raw(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), od.data_ptr(),
                                      gd.data_ptr(), ld.data_ptr(),
                                      *(t.data_ptr() for t in dev_out), w.B, w.h, w.n_q, w.n_k,
                                      w.d, w.scale, w.mask,
                                      None if dkl is None else dkl.data_ptr(), ws.data_ptr(),
                                      ws_bytes, sptr)
        if rc != 0:
            raise binding.AttnError(rc, "attn_bwd")
        for h, d in zip(host_out, dev_out):
            h.copy_(d, non_blocking=True)

    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    n = max(3, min(args.steps, 50))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    binding.check(stream)
    ms = e0.elapsed_time(e1) / n
    world = dist_env()[0]
    return {"value": world * inputs.flops(w) / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": ms,
            "steps": n}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="base_enc", choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    w = inputs.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
