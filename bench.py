#!/usr/bin/env python
"""Benchmark of the folded, KV-balanced FP8 MLA decode on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...        # the CPU oracle, timed on the host

A step is one pass of the whole decode path over one synthetic batch with the
inputs resident in HBM: the device planner, the split-KV decode and the LSE
reduction (the fold itself is a free view). L2 is flushed before every step by
writing a buffer of twice its size; the flush is outside the timed region.
Every step is timed with CUDA events on the launching stream. Under torchrun
each rank decodes its own batch of the same shape (requests are independent:
weak scaling, no collective on the data path) and the slowest rank's time sets
the value. Prints one JSON line on rank 0.
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
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import D_QK, WORKLOADS, make_batch  # noqa: E402

METRIC = "decode rows/s and KV HBM GB/s (fraction of 8 TB/s) vs unfolded, 1 GB300"
UNIT = "rows/s"
DEFAULT_WORKLOAD = "R32_k4_H8_len1k-8k"
FALLBACK_HBM_GBS = 6800.0
DECODE_SOURCES = ("decode_tc.cu", "internal.h", "ptx.cuh", "tc.cuh")


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(WORKLOADS))
    p.add_argument("--variant-steps", type=int, default=300)
    p.add_argument("--e2e-steps", type=int, default=30)
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--no-variants", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    return p.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


# ---------------------------------------------------------------- oracle timing
def oracle_rows_per_s(batch, seconds: float):
    """Time the CPU oracle, as it stands, on whole requests of the batch until
    ``seconds`` of CPU work have passed. Returns (rows/s, requests, elapsed)."""
    import oracle.attention as att
    lens = batch.seq_lens.numpy()
    order = list(range(batch.R))
    done, t0 = 0, time.perf_counter()
    while done < len(order):
        r = order[done]
        att.mla_decode(batch.q.numpy(), batch.kv.numpy(), batch.block_table.numpy(), lens,
                       batch.k, batch.sm_scale, batch.q_scale, batch.kv_scale, requests=[r])
        done += 1
        if time.perf_counter() - t0 >= seconds:
            break
    el = time.perf_counter() - t0
    return done * batch.k / el, done, el


def cpu_threads() -> int:
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[4:]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = set()
        for _, _, flags in rows:
            for n, f in zip(names[1:], flags[1:]):
                if f.lower() == "active":
                    reasons.add(n)
        sm = [r[0] for r in rows]
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(r[1] for r in rows),
                "samples": len(rows), "reasons": sorted(reasons)}


# ---------------------------------------------------------------- measurement
def algorithmic_bytes(lens, M: int) -> int:
    """KV rows read once, queries read, BF16 out + FP32 LSE written, block table."""
    lens = np.asarray(lens, dtype=np.int64)
    pages = (lens + 63) // 64
    return int(D_QK * lens.sum() + len(lens) * M * (D_QK + 512 * 2 + 4) + 4 * pages.sum())


def source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mla_decode_attention_folded_gb300", "csrc")
    for name in DECODE_SOURCES:
        path = os.path.join(csrc, name)
        if os.path.exists(path):
            h.update(open(path, "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on the current decode source."""
    path = os.path.join(ROOT, "profiles", f"decode_{workload}.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path):
        if ":" in line:
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip()
    if vals.get("decode_source_sha256_16") != source_hash():
        return None
    try:
        return int(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        v = float(json.load(open(path))["hbm_gbs"])
        return v, "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


class Runner:
    """One decode configuration with its buffers, timed step by step."""

    def __init__(self, batch, dev, policy, folded=True):
        import mla_decode_attention_folded_gb300 as mla
        self.mla = mla
        self.b = batch
        if folded:
            R, k, H = batch.R, batch.k, batch.H
            bt, lens = batch.block_table, batch.seq_lens
        else:
            rep = torch.arange(batch.R).repeat_interleave(batch.k)
            R, k, H = batch.R * batch.k, 1, batch.H
            bt, lens = batch.block_table[rep].contiguous(), batch.seq_lens[rep].contiguous()
        self.q = batch.q.to(dev)
        self.kv = batch.kv.to(dev)
        self.bt = bt.to(dev)
        self.lens = lens.to(dev)
        self.eng = mla.FoldedMla(R, k, H, self.bt.shape[1], self.kv.shape[0], dev, policy=policy)
        self.out = torch.empty((R, k * H, 512), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((R, k * H), dtype=torch.float32, device=dev)
        self.bmm1 = float(np.float32(batch.sm_scale) * np.float32(batch.q_scale)
                          * np.float32(batch.kv_scale))
        self.bmm2 = float(batch.kv_scale)
        self.launches = 3 if self.mla.workspace_bytes(self.eng.shape) > 0 else 2

    def step(self, ev=None):
        e = self.eng
        e.plan(self.lens)
        if ev is not None:
            ev[0].record()
        self.mla.folded_decode(e.shape, self.q, self.kv, self.bt, self.lens, self.bmm1,
                               self.bmm2, e.counts, e.work, e.workspace, self.out, self.lse,
                               e.status)
        if ev is not None:
            ev[1].record()
        self.mla.split_combine(e.shape, e.counts, e.work, e.workspace, self.bmm2, self.out,
                               self.lse)

    def timed(self, steps, warmup, flush, barrier=None):
        for _ in range(warmup):
            flush.zero_()
            self.step()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
        torch.cuda.synchronize()
        if barrier:
            barrier()
        torch.cuda.synchronize()
        for i in range(steps):
            flush.zero_()
            ev[i][0].record()
            self.step(ev=(ev[i][1], ev[i][2]))
            ev[i][3].record()
        torch.cuda.synchronize()
        if barrier:
            barrier()
        step_ms = [e[0].elapsed_time(e[3]) for e in ev]
        dec_ms = [e[1].elapsed_time(e[2]) for e in ev]
        return statistics.mean(step_ms), statistics.mean(dec_ms)


def e2e_rows_per_s(batch, dev, steps):
    """The same metric through the public API with HOST buffers: every step
    copies the inputs from pinned host memory, decodes, and reads the outputs
    back into pinned host memory."""
    import mla_decode_attention_folded_gb300 as mla
    hq, hkv = batch.q.pin_memory(), batch.kv.pin_memory()
    hbt, hlens = batch.block_table.pin_memory(), batch.seq_lens.pin_memory()
    R, M = batch.R, batch.M
    hout = torch.empty((R, M, 512), dtype=torch.bfloat16).pin_memory()
    hlse = torch.empty((R, M), dtype=torch.float32).pin_memory()
    q = torch.empty_like(hq, device=dev)
    kv = torch.empty_like(hkv, device=dev)
    bt = torch.empty_like(hbt, device=dev)
    lens = torch.empty_like(hlens, device=dev)
    out = torch.empty((R, M, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((R, M), dtype=torch.float32, device=dev)
    eng = mla.FoldedMla(R, batch.k, batch.H, hbt.shape[1], hkv.shape[0], dev)
    bmm1 = float(np.float32(batch.sm_scale) * np.float32(batch.q_scale) * np.float32(batch.kv_scale))
    bmm2 = float(batch.kv_scale)

    def one():
        q.copy_(hq, non_blocking=True)
        kv.copy_(hkv, non_blocking=True)
        bt.copy_(hbt, non_blocking=True)
        lens.copy_(hlens, non_blocking=True)
        eng.plan(lens)
        eng.decode(q, kv, bt, lens, bmm1, bmm2, out=out, lse=lse)
        hout.copy_(out, non_blocking=True)
        hlse.copy_(lse, non_blocking=True)

    for _ in range(3):
        one()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(steps):
        one()
    t1.record()
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps
    h2d = sum(t.numel() * t.element_size() for t in (hq, hkv, hbt, hlens))
    d2h = hout.numel() * hout.element_size() + hlse.numel() * hlse.element_size()
    return R * batch.k / (ms / 1e3), h2d, d2h


def run_ours(args):
    rank, world, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    barrier = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

        def barrier():
            dist.barrier()

    w = WORKLOADS[args.workload]
    batch = make_batch(args.workload)
    props = torch.cuda.get_device_properties(dev)
    flush = torch.empty(2 * max(props.L2_cache_size, 64 << 20), dtype=torch.uint8, device=dev)

    main = Runner(batch, dev, policy=0, folded=True)
    clocks = ClockSampler(local)
    clocks.start()
    step_ms, dec_ms = main.timed(args.steps, max(args.warmup, 3), flush, barrier)
    clk = clocks.stop()
    status = int(main.eng.status.item())
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([step_ms, dec_ms], device=dev, dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        step_ms, dec_ms = float(t[0]), float(t[1])

    lens = batch.seq_lens.numpy()
    rows = batch.R * batch.k
    kv_b = D_QK * int(lens.sum())
    value = world * rows / (step_ms / 1e3)
    algo = algorithmic_bytes(lens, batch.M)
    peak, peak_src = measured_hbm_peak()
    achieved = algo / (dec_ms / 1e3) / 1e9

    variants = {}
    if rank == 0 and not args.no_variants:
        for name, policy, folded in (("folded_uniform", 1, True), ("unfolded_balanced", 0, False),
                                     ("unfolded_uniform", 1, False)):
            r = Runner(batch, dev, policy=policy, folded=folded)
            ms, dms = r.timed(args.variant_steps, 5, flush)
            variants[name] = {"rows_per_s": rows / (ms / 1e3), "ms_per_step": ms,
                              "decode_ms": dms, "kv_gbs": kv_b / (ms / 1e3) / 1e9}
            del r

    e2e_v, h2d, d2h = e2e_rows_per_s(batch, dev, args.e2e_steps)
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([e2e_v], device=dev, dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MIN)
        e2e_v = float(t[0]) * world

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rps, nreq, el = oracle_rows_per_s(batch, args.cpu_seconds)
        cpu = {"value": rps, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
               "sample": f"{nreq} of {batch.R} requests of {args.workload} "
                         f"({el:.1f} s, float64 numpy)"}

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f8e4m3",
        "data": "synthetic",
        "config": {"workload": args.workload, "R": batch.R, "k": batch.k, "H": batch.H,
                   "M": batch.M, "policy": "balanced", "num_ctas": main.eng.shape.num_ctas,
                   "kv_tokens": int(lens.sum()), "accumulate": "f32",
                   "l2": "flushed before every step (2x L2 write, untimed)",
                   "parallelism": f"replicas{world}"},
        "kv_gbs": kv_b / (step_ms / 1e3) / 1e9,
        "kv_frac_of_8tbs": kv_b / (step_ms / 1e3) / 8e12,
        "head_rows_per_s": world * batch.R * batch.M / (step_ms / 1e3),
        "decode_ms": dec_ms,
        "variants": variants,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": peak_src,
                     "traffic": profiled_traffic(args.workload),
                     "kernel": "mla_folded_decode", "algorithmic_bytes_per_launch": algo},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_v, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps * main.launches,
        "clocks": clk,
        "status": status,
    }
    print(json.dumps(line), flush=True)


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    batch = make_batch(args.workload)
    per_step = max(1.0, min(args.cpu_seconds, 240.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_rows_per_s(batch, per_step)
    vals, reqs = [], []
    for _ in range(args.steps):
        v, n, _ = oracle_rows_per_s(batch, per_step)
        vals.append(v)
        reqs.append(n)
    value = statistics.mean(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": args.workload, "R": batch.R, "k": batch.k, "H": batch.H,
                   "M": batch.M},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
                         "sample": f"each step: whole requests of {args.workload} for "
                                   f"{per_step:.1f} s ({min(reqs)}-{max(reqs)} requests)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
