"""Benchmark: fused multi-head scaled dot-product attention forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one forward pass of the whole hot path (one ``attn_fwd`` call: QK^T,
mask, online softmax, PV, epilogue) over one batch of the workload.  The
default workload is the base encoder self-attention (B=64, h=8, n_q=n_k=512,
d_k=d_v=64, bf16, no mask).  Prints ONE JSON line (rank 0).

Timing: W untimed warm-up steps, then K timed steps.  Before every timed step
the L2 is flushed by writing a 256 MiB buffer (outside the timed interval);
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
KERNEL_SOURCES = ("transformer_head_scaled_gb300/csrc/attn_fwd_tc.cu",
                  "transformer_head_scaled_gb300/csrc/ptx.cuh")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "attn_fwd_tc_traffic.json")


def kernel_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
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


def dram_traffic(workload: str):
    """ncu DRAM bytes per launch for this kernel source and workload, or None."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("kernel_hash") != kernel_hash():
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
    mask = {0: "no mask", 1: "causal", 2: "key padding L~U[64,n_k]"}[w.mask]
    return f"{w.name}: B={w.B} h={w.h} n_q={w.n_q} n_k={w.n_k} d_k=d_v={w.d} {w.dtype} {mask}"


# ---------------------------------------------------------------------- oracle (CPU)

def _row_flops(w: inputs.Workload, rows, lens) -> float:
    if w.mask == inputs.MASK_NONE:
        keys = np.full(rows.size, w.n_k)
    elif w.mask == inputs.MASK_CAUSAL:
        keys = np.minimum(rows % w.n_q + 1, w.n_k)
    else:
        keys = np.minimum(lens[(rows // w.n_q) // w.h], w.n_k)
    return float(4.0 * w.d * keys.sum())


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
        oracle.attn_rows(q, k, v, rows, w.scale, w.mask, kl, threads=threads)
        per_row = (time.perf_counter() - t0) / n
        rows_hint = max(1, int(target_s / max(per_row, 1e-9)))
    done, flops, dt = 0, 0.0, 0.0
    while done < rows_hint:
        n = min(total_rows, rows_hint - done)
        rows = (np.arange(total_rows, dtype=np.int64) if n == total_rows
                else np.sort(rng.choice(total_rows, size=n, replace=False)))
        t0 = time.perf_counter()
        oracle.attn_rows(q, k, v, rows, w.scale, w.mask, kl, threads=threads)
        dt += time.perf_counter() - t0
        flops += _row_flops(w, rows, lens)
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
    # the whole run (warm-up included) is sized to about two minutes of CPU time
    per_step = min(20.0, 120.0 / max(1, args.steps + args.warmup))
    _, dt, n, _ = oracle_sample(w, qf, kf, vf, kl, target_s=min(per_step, 1.0))
    rows_per_step = max(1, int(n * per_step / max(dt, 1e-9)))
    for _ in range(args.warmup):
        oracle_sample(w, qf, kf, vf, kl, 0.0, rows_hint=rows_per_step)
    vals, secs = [], []
    for _ in range(args.steps):
        tf, dt, _, _ = oracle_sample(w, qf, kf, vf, kl, 0.0, rows_hint=rows_per_step)
        vals.append(tf)
        secs.append(dt)
    rows_used = rows_per_step
    value = statistics.median(vals)
    cores = cpu_cores_used()
    sample = (f"{rows_used} query rows per step, drawn from the {w.B * w.h * w.n_q} rows of the "
              f"workload (each against all its visible keys), float64")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.median(secs), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_desc(w), "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
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
    stream = torch.cuda.current_stream(dev)
    sptr = int(stream.cuda_stream)
    f32 = w.dtype == "f32"
    ptrs = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr())
    klp = None if kl is None else kl.data_ptr()
    decode = w.kind == "decode"
    ws_bytes = binding.decode_workspace_bytes(w.B, w.h, w.n_q, w.n_k, w.d) if decode else 0
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)

    def step():
        if decode:
            rc = binding.attn_decode_raw(*ptrs, w.B, w.h, w.n_q, w.n_k, w.d, w.scale, klp,
                                         ws.data_ptr(), ws_bytes, sptr)
        else:
            rc = binding.attn_fwd_raw(*ptrs, w.B, w.h, w.n_q, w.n_k, w.d, w.scale, w.mask, klp,
                                      sptr, f32=f32)
        if rc != 0:
            raise binding.AttnError(rc, "attn_decode" if decode else "attn_fwd")

    for _ in range(max(3, args.warmup)):
        flush.zero_()
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
            flush.zero_()
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

    fl = inputs.flops(w)
    fl_alg = inputs.algorithmic_flops(w, kl)
    value = world * fl / (ms * 1e-3) / 1e12
    peaks = measured_peaks()
    achieved = fl_alg / (ms * 1e-3) / 1e12
    hbm = inputs.hbm_bytes(w, kl)

    # end to end through the public API: pinned host inputs -> device -> attn_fwd -> host
    e2e = run_e2e(args, w, q, k, v, kl, dev, stream, f32)

    clk = clocks.summary(t_start, t_end)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32" if f32 else "bf16", "data": "synthetic",
        "config": {"workload": workload_desc(w), "global_batch": world * w.B,
                   "parallelism": f"dp{world}: batch entries split across ranks, no collective on the data path",
                   "l2": "flushed before every timed step (256 MiB write, outside the events)",
                   "flops_per_step": fl, "algorithmic_flops_per_step": fl_alg,
                   "hbm_bytes_per_step": hbm, "timed_loop_wall_s": wall},
        "pct_of_peak": 100.0 * (value / world) / peaks["bf16_tflops"],
        "roofline": ({"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                      "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                      "traffic": dram_traffic(w.name),
                      "peak_source": f"{peaks['_source']} bf16_tflops (burst; kernel timed alone)",
                      "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
                      "hbm_gbs": hbm / (ms * 1e-3) / 1e9,
                      "kernel": "attn_fwd_tc_kernel" if not f32 else "attn_fwd_f32_kernel"}
                     if not decode else
                     {"bound": "hbm", "achieved": hbm / (ms * 1e-3) / 1e9, "peak": peaks["hbm_gbs"],
                      "unit": "GB/s", "frac": hbm / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                      "traffic": dram_traffic(w.name), "algorithmic_bytes": hbm,
                      "peak_source": f"{peaks['_source']} hbm_gbs (copy bandwidth)",
                      "kernel": "attn_decode_split_kernel" + (" + combine" if ws_bytes else "")}),
        "e2e": e2e,
        "gpu_launches": int(launches),
        "clocks": {k2: clk[k2] for k2 in ("sm_mhz", "sm_max_mhz", "reasons")},
    }
    if rank == 0 and not args.no_cpu_baseline:
        qf, kf, vf = (t.float().cpu().numpy() for t in (q, k, v))
        tf, dt, nrows, _ = oracle_sample(w, qf, kf, vf, kl, target_s=args.cpu_seconds)
        line["cpu_baseline"] = {
            "value": tf, "unit": "TFLOP/s", "cores": cpu_cores_used(), "kind": "oracle",
            "sample": f"{nrows} query rows ({nrows / (w.B * w.h * w.n_q):.2f} passes over the "
                      f"{w.B * w.h * w.n_q} rows of the same workload), float64, {dt:.1f} s"}
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
    ws_bytes = (binding.decode_workspace_bytes(w.B, w.h, w.n_q, w.n_k, w.d)
                if w.kind == "decode" else 0)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)

    def step():
        dq.copy_(hq, non_blocking=True)
        dk.copy_(hk, non_blocking=True)
        dv.copy_(hv, non_blocking=True)
        if dkl is not None:
            dkl.copy_(hkl, non_blocking=True)
        if w.kind == "decode":
            rc = binding.attn_decode_raw(dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                         do.data_ptr(), dl.data_ptr(), w.B, w.h, w.n_q, w.n_k,
                                         w.d, w.scale, None if dkl is None else dkl.data_ptr(),
                                         ws.data_ptr(), ws_bytes, sptr)
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
