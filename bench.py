#!/usr/bin/env python
"""Benchmark of the folded, KV-balanced FP8 MLA decode on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...        # the CPU oracle, timed on the host

A step is one pass of the whole decode path over one synthetic batch with the
inputs resident in HBM: the device planner, the split-KV decode and the LSE
reduction (the fold itself is a free view). The headline line is measured on
the largest single-GPU workload (R128_k7_H64_skewed128k: 128 requests x 7
draft tokens x 64 heads, skewed lengths); the four other workloads are
measured the same way and reported beside it under "per_workload". L2 is flushed before every step by
writing a buffer of twice its size; the flush is outside the timed region.
Every step is timed with CUDA events on the launching stream. Under torchrun
each rank decodes its own batch of the same shape (requests are independent:
weak scaling, no collective on the data path) and the slowest rank's time sets
the value. Prints one JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import hashlib
import re
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
DEFAULT_WORKLOAD = "R128_k7_H64_skewed128k"
# Oracle timed single-threaded on these workloads as well (the small ones).
ONE_THREAD_WORKLOADS = ("R2_k4_H8_len100+37", "R32_k4_H8_len1k-8k", "R64_k7_H8_lognormal2k")
REFERENCE_BUDGET_S = 120.0
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
DECODE_SOURCES = ("decode_tc.cu", "decode_common.cuh", "internal.h", "ptx.cuh", "tc.cuh")


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
    p.add_argument("--per-workload-steps", type=int, default=200)
    p.add_argument("--one-thread-seconds", type=float, default=3.0)
    p.add_argument("--no-variants", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-per-workload", action="store_true")
    return p.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


# ---------------------------------------------------------------- oracle timing
class OracleSampler:
    """Times the CPU oracle, as it stands, on consecutive 256-key chunks of the
    batch's requests (request by request, cycling). A chunk of c keys of a
    request of L keys is c / L of that request's k query-token rows, so the
    rate is in the headline unit whatever the sample size; the merge of the
    chunks (negligible work) is not run."""
    CHUNK = 256

    def __init__(self, batch):
        import oracle.attention as att
        self.att = att
        self.b = batch
        self.q, self.kv = batch.q.numpy(), batch.kv.numpy()
        self.bt, self.lens = batch.block_table.numpy(), batch.seq_lens.numpy()
        self.ranges = np.zeros((batch.R, 2), dtype=np.int64)
        self.r, self.j = 0, 0
        if int(self.lens.max(initial=0)) <= 0:
            raise ValueError("every request is empty")

    def run(self, seconds: float):
        """At least one chunk, then chunks until `seconds` have passed.
        Returns (rows/s, rows, elapsed s, chunks)."""
        b, rows, chunks = self.b, 0.0, 0
        t0 = time.perf_counter()
        while True:
            L = int(self.lens[self.r])
            if L > 0:
                j1 = min(L, self.j + self.CHUNK)
                self.ranges[self.r] = (self.j, j1)
                self.att.mla_decode(self.q, self.kv, self.bt, self.lens, b.k, b.sm_scale,
                                    b.q_scale, b.kv_scale, key_range=self.ranges,
                                    requests=[self.r])
                rows += (j1 - self.j) / L * b.k
                chunks += 1
                self.j = j1
            if L <= 0 or self.j >= L:
                self.r, self.j = (self.r + 1) % b.R, 0
            el = time.perf_counter() - t0
            if chunks > 0 and el >= seconds:
                return rows / el, rows, el, chunks


def cpu_threads() -> int:
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def one_thread_oracle(workload: str, seconds: float):
    """The oracle's rate on one host thread: a fresh interpreter with the BLAS
    thread count pinned to 1 before numpy loads runs the same sampler."""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = ("import json, sys; sys.path.insert(0, %r); import bench; "
            "from workloads import make_batch; "
            "r = bench.OracleSampler(make_batch(%r)).run(%r); "
            "print(json.dumps(r))") % (ROOT, workload, float(seconds))
    try:
        p = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                           timeout=120 + 4 * seconds)
        rps, rows, el, chunks = json.loads(p.stdout.strip().splitlines()[-1])
    except (subprocess.SubprocessError, ValueError, IndexError, OSError) as e:
        return {"workload": workload, "error": str(e)[:200]}
    return {"workload": workload, "value": rps, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{chunks} consecutive {OracleSampler.CHUNK}-key chunks = {rows:.2f} "
                      f"query-token rows in {el:.1f} s"}


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


_COMMENT = re.compile(r"//[^\n]*|/\*.*?\*/", re.S)


def strip_comments(text: str) -> str:
    """C/C++ source without its comments and trailing blanks (the decode
    sources hold no string literal containing a comment marker)."""
    text = _COMMENT.sub("", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def source_hash() -> str:
    """Hash of the decode kernels' code, comments excluded: an ncu capture
    stays valid for the source it was taken on whatever its comments say."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mla_decode_attention_folded_gb300", "csrc")
    for name in DECODE_SOURCES:
        path = os.path.join(csrc, name)
        if os.path.exists(path):
            h.update(strip_comments(open(path).read()).encode())
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


def max_over_ranks(values, device):
    """Element-wise max of per-rank values over the process group (identity
    without one): the slowest rank's time sets a multi-rank result."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        v = float(json.load(open(path))["hbm_gbs"])
        return v, "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def fp8_tensor_peak():
    """Dense FP8 TFLOP/s: the measured burst bf16 GEMM rate times the nominal
    FP8 / bf16 ratio (4.5 / 2.25 PFLOP/s dense)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        v = float(json.load(open(path))["bf16_tflops"])
        return 2.0 * v, "measured bf16 x nominal fp8/bf16 ratio 2"
    except (OSError, KeyError, ValueError):
        return 2.0 * FALLBACK_BF16_TFLOPS, "fallback bf16 x nominal fp8/bf16 ratio 2"


def algorithmic_flops(lens, M: int) -> int:
    """S = Q.K^T over 576 dims and O = P.V over 512 dims: 2 * M * len * 1088."""
    return int(2 * M * (D_QK + 512) * np.asarray(lens, dtype=np.int64).sum())


def roofline(algo_bytes: int, flops: int, kernel_s: float):
    """The bound that binds at this arithmetic intensity (HBM below the ridge
    of the two measured peaks, the FP8 tensor pipe above it), with both
    fractions."""
    hbm, hbm_src = measured_hbm_peak()
    fp8, fp8_src = fp8_tensor_peak()
    gbs = algo_bytes / kernel_s / 1e9
    tfs = flops / kernel_s / 1e12
    ridge = fp8 * 1e12 / (hbm * 1e9)
    intensity = flops / algo_bytes
    r = {"hbm_frac": gbs / hbm, "tensor_frac": tfs / fp8,
         "intensity_flop_per_byte": intensity, "ridge_flop_per_byte": ridge}
    if intensity < ridge:
        r.update(bound="hbm", achieved=gbs, peak=hbm, unit="GB/s", frac=gbs / hbm,
                 peak_source=hbm_src)
    else:
        r.update(bound="tensor", achieved=tfs, peak=fp8, unit="TFLOP/s", frac=tfs / fp8,
                 peak_source=fp8_src)
    return r


class Runner:
    """One decode configuration with its buffers, timed step by step."""

    def __init__(self, batch, dev, policy, folded=True):
        import mla_decode_attention_folded_gb300 as mla
        self.mla = mla
        self.b = batch
        # Unfolded = the stock layout: k single-token row groups per request,
        # each reading the request's KV on its own.
        R, k, H = batch.R, batch.k, batch.H
        groups = 1 if folded else batch.k
        bt, lens = batch.block_table, batch.seq_lens
        self.q = batch.q.to(dev)
        self.kv = batch.kv.to(dev)
        self.bt = bt.to(dev)
        self.lens = lens.to(dev)
        self.eng = mla.FoldedMla(R, k, H, self.bt.shape[1], self.kv.shape[0], dev, policy=policy,
                                 groups=groups)
        self.out = torch.empty((R, k * H, 512), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((R, k * H), dtype=torch.float32, device=dev)
        self.bmm1 = float(np.float32(batch.sm_scale) * np.float32(batch.q_scale)
                          * np.float32(batch.kv_scale))
        self.bmm2 = float(batch.kv_scale)
        self.launches = 3 if self.mla.workspace_bytes(self.eng.shape) > 0 else 2

    def plan(self):
        self.eng.plan(self.lens)

    def decode(self):
        e = self.eng
        self.mla.folded_decode(e.shape, self.q, self.kv, self.bt, self.lens, self.bmm1,
                               self.bmm2, e.counts, e.work, e.workspace, self.out, self.lse,
                               e.status)

    def combine(self):
        e = self.eng
        self.mla.split_combine(e.shape, e.counts, e.work, e.workspace, self.bmm2, self.out,
                               self.lse)

    def step(self):
        self.plan()
        self.decode()
        self.combine()

    # The W_UV leg: the decode without an LSE, then the split reduction fused
    # with the up-projection (synthetic BF16 weights).
    def uv_setup(self, dev):
        from workloads import make_w_uv
        b = self.b
        self.w_uv = make_w_uv(b.H, seed=2024).transpose(1, 2).contiguous().to(dev)
        self.y = torch.empty((b.R * b.k, b.H, 128), dtype=torch.bfloat16, device=dev)

    def decode_nolse(self):
        e = self.eng
        self.mla.folded_decode(e.shape, self.q, self.kv, self.bt, self.lens, self.bmm1,
                               self.bmm2, e.counts, e.work, e.workspace, self.out, None,
                               e.status)

    def uv(self):
        e = self.eng
        self.mla.uv_combine(e.shape, e.counts, e.work, e.workspace, self.bmm2, self.out,
                            self.w_uv, self.y, e.status)

    def uv_times(self, steps, flush):
        """(plan -> decode -> fused W_UV reduction) per step, and the fused
        reduction alone after an untimed plan + decode."""
        chain = self.graph(lambda: (self.plan(), self.decode_nolse(), self.uv()))
        gpd = self.graph(lambda: (self.plan(), self.decode_nolse()))
        guv = self.graph(self.uv)
        return self._time(chain, steps, flush), self._time(guv, steps, flush, before=gpd)

    def graph(self, fn):
        """fn's launches captured once into a CUDA graph (replayed per step, so
        host launch overhead stays out of the timed region)."""
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            fn()                                  # warm: lazy set-up happens outside capture
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="thread_local"):
            fn()
        torch.cuda.synchronize()
        return g

    def _time(self, g, steps, flush, before=None):
        """Mean event time of replaying graph g over `steps` replays, L2
        flushed (and `before` replayed) untimed ahead of each."""
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        for i in range(steps):
            flush()
            if before is not None:
                before.replay()
            ev[i][0].record()
            g.replay()
            ev[i][1].record()
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in ev)

    def timed(self, steps, warmup, flush, barrier=None):
        """Whole steps (plan + decode + combine, chained as a caller runs them)
        timed one by one; returns the mean step time in ms."""
        g = self.graph(self.step)
        for _ in range(warmup):
            flush()
            g.replay()
        torch.cuda.synchronize()
        if barrier:
            barrier()
        torch.cuda.synchronize()
        ms = self._time(g, steps, flush)
        if barrier:
            barrier()
        return ms

    def kernel_times(self, steps, flush):
        """Each kernel alone (its inputs prepared untimed): plan, decode, combine."""
        gp, gd, gc = self.graph(self.plan), self.graph(self.decode), self.graph(self.combine)
        gpd = self.graph(lambda: (self.plan(), self.decode()))
        plan = self._time(gp, steps, flush)
        dec = self._time(gd, steps, flush, before=gp)
        comb = self._time(gc, steps, flush, before=gpd)
        return plan, dec, comb

    def marginal_times(self, steps, flush):
        """Chained step time without the plan, and without the combine: how
        much each adds to the chain (PDL overlap included)."""
        g_no_comb = self.graph(lambda: (self.plan(), self.decode()))
        g_no_plan = self.graph(lambda: (self.decode(), self.combine()))
        gp = self.graph(self.plan)
        return (self._time(g_no_plan, steps, flush, before=gp),
                self._time(g_no_comb, steps, flush))


class TieredRunner(Runner):
    """The pages' tiered launch (unsplit launch + split tiers on prioritised
    streams, built from the same kernels), timed like a Runner step."""

    def __init__(self, batch, dev):
        import mla_decode_attention_folded_gb300 as mla
        self.mla = mla
        self.b = batch
        self.q = batch.q.to(dev)
        self.kv = batch.kv.to(dev)
        self.bt = batch.block_table.to(dev)
        self.lens = batch.seq_lens.to(dev)
        self.tiered = mla.TieredMla(batch.R, batch.k, batch.H, self.bt.shape[1],
                                    self.kv.shape[0], dev)
        self.out = torch.empty((batch.R, batch.M, 512), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((batch.R, batch.M), dtype=torch.float32, device=dev)
        self.bmm1 = float(np.float32(batch.sm_scale) * np.float32(batch.q_scale)
                          * np.float32(batch.kv_scale))
        self.bmm2 = float(batch.kv_scale)

    def step(self):
        self.tiered.decode(self.q, self.kv, self.bt, self.lens, self.bmm1, self.bmm2,
                           out=self.out, lse=self.lse)


def has_tiers(batch, dev) -> bool:
    import mla_decode_attention_folded_gb300 as mla
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    return len(mla.balanced_tiers(batch.R, sms)) > 0


class L2Flush:
    """Evicts L2 before a timed step: write a buffer of twice the L2 size, then
    read another one, so L2 holds neither the inputs nor dirty lines whose
    write-back would land inside the timed region."""

    def __init__(self, dev):
        n = 2 * max(torch.cuda.get_device_properties(dev).L2_cache_size, 64 << 20)
        self.w = torch.empty(n, dtype=torch.uint8, device=dev)
        self.r = torch.ones(n // 4, dtype=torch.float32, device=dev)
        self.sink = torch.empty(1, dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.zero_()
        torch.sum(self.r, dim=0, keepdim=True, out=self.sink)


def e2e_rows_per_s(batch, dev, steps):
    """The same metric through the public API with HOST buffers: every step
    copies its inputs from pinned host memory, plans, decodes and reads out
    and lse back into pinned host memory; every byte crosses the host link
    inside the timed region.

    Returns (pipelined rows/s, serial rows/s, H2D bytes, D2H bytes). Serial:
    one stream, copy -> plan -> decode -> read-back, step after step.
    Pipelined: two sets of device buffers, the copies on their own streams,
    so that step i+1's inputs stream in while step i computes and step i-1's
    outputs stream back, as a serving loop overlaps them; the host-to-device
    link then sets the pace."""
    import mla_decode_attention_folded_gb300 as mla
    hq, hkv = batch.q.pin_memory(), batch.kv.pin_memory()
    hbt, hlens = batch.block_table.pin_memory(), batch.seq_lens.pin_memory()
    R, M = batch.R, batch.M
    host_in = (hq, hkv, hbt, hlens)

    def device_set():
        return ([torch.empty_like(t, device=dev) for t in host_in],
                torch.empty((R, M, 512), dtype=torch.bfloat16, device=dev),
                torch.empty((R, M), dtype=torch.float32, device=dev),
                torch.empty((R, M, 512), dtype=torch.bfloat16).pin_memory(),
                torch.empty((R, M), dtype=torch.float32).pin_memory())

    sets = [device_set(), device_set()]
    eng = mla.FoldedMla(R, batch.k, batch.H, hbt.shape[1], hkv.shape[0], dev)
    bmm1 = float(np.float32(batch.sm_scale) * np.float32(batch.q_scale) * np.float32(batch.kv_scale))
    bmm2 = float(batch.kv_scale)

    def compute(ins, out, lse):
        q, kv, bt, lens = ins
        eng.plan(lens)
        eng.decode(q, kv, bt, lens, bmm1, bmm2, out=out, lse=lse)

    def serial(i):
        ins, out, lse, hout, hlse = sets[0]
        for d, h in zip(ins, host_in):
            d.copy_(h, non_blocking=True)
        compute(ins, out, lse)
        hout.copy_(out, non_blocking=True)
        hlse.copy_(lse, non_blocking=True)

    s_in, s_comp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev = [{k: torch.cuda.Event() for k in ("in", "comp", "out")} for _ in range(2)]
    used = [False, False]

    def pipelined(i):
        b = i % 2
        ins, out, lse, hout, hlse = sets[b]
        e = ev[b]
        if used[b]:
            s_in.wait_event(e["comp"])      # step i-2 has read these inputs
            s_comp.wait_event(e["out"])     # and its outputs are back on the host
        with torch.cuda.stream(s_in):
            for d, h in zip(ins, host_in):
                d.copy_(h, non_blocking=True)
            e["in"].record(s_in)
        s_comp.wait_event(e["in"])
        with torch.cuda.stream(s_comp):
            compute(ins, out, lse)
            e["comp"].record(s_comp)
        s_out.wait_event(e["comp"])
        with torch.cuda.stream(s_out):
            hout.copy_(out, non_blocking=True)
            hlse.copy_(lse, non_blocking=True)
            e["out"].record(s_out)
        used[b] = True

    def timed(step, streams, reps=3):
        """Median over `reps` timed runs of `steps` steps each (a host hiccup
        in one run, which starves the pipelined loop, does not set the figure)."""
        cur = torch.cuda.current_stream(dev)
        for i in range(3):
            step(i)
        torch.cuda.synchronize(dev)
        rates, i = [], 3
        for _ in range(reps):
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            t0.record(cur)
            for st in streams:
                st.wait_event(t0)
            for _ in range(steps):
                step(i)
                i += 1
            for st in streams:
                cur.wait_stream(st)
            t1.record(cur)
            torch.cuda.synchronize(dev)
            rates.append(R * batch.k / (t0.elapsed_time(t1) / steps / 1e3))
        return float(np.median(rates))

    serial_v = timed(serial, [])
    piped_v = timed(pipelined, [s_in, s_comp, s_out])
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = R * M * 512 * 2 + R * M * 4
    return piped_v, serial_v, h2d, d2h


VARIANTS = (("folded_uniform", 1, True), ("unfolded_balanced", 0, False),
            ("unfolded_uniform", 1, False))


def workload_summary(name, batch, step_ms, dec_ms, variants):
    """Step time, decode time, the binding roofline and the variants of one
    workload, with the fold and balance gains derived from them."""
    lens = batch.seq_lens.numpy()
    rows = batch.R * batch.k
    kv_b = D_QK * int(lens.sum())
    roof = roofline(algorithmic_bytes(lens, batch.M), algorithmic_flops(lens, batch.M),
                    dec_ms / 1e3)
    r = {"step_us": step_ms * 1e3, "decode_us": dec_ms * 1e3,
         "rows_per_s": rows / (step_ms / 1e3),
         "head_rows_per_s": batch.R * batch.M / (step_ms / 1e3),
         "kv_gbs_step": kv_b / (step_ms / 1e3) / 1e9,
         "bound": roof["bound"], "frac": roof["frac"], "hbm_frac": roof["hbm_frac"],
         "tensor_frac": roof["tensor_frac"], "traffic": profiled_traffic(name),
         "variants_step_us": {"folded_balanced": step_ms * 1e3}}
    for v, ms in variants.items():
        r["variants_step_us"][v] = ms * 1e3
    if "folded_uniform" in variants:
        r["balanced_over_uniform"] = variants["folded_uniform"] / step_ms
    if "unfolded_balanced" in variants:
        r["folded_over_unfolded"] = variants["unfolded_balanced"] / step_ms
    if "tiered" in variants:
        r["persistent_over_tiered"] = variants["tiered"] / step_ms
    return r


def measure_variants(batch, dev, flush, steps):
    out = {}
    for name, policy, folded in VARIANTS:
        r = Runner(batch, dev, policy=policy, folded=folded)
        out[name] = r.timed(steps, 5, flush)
        del r
    if has_tiers(batch, dev):
        r = TieredRunner(batch, dev)
        out["tiered"] = r.timed(steps, 5, flush)
        del r
    return out


def measure_side_workload(name, dev, flush, steps, with_variants):
    """One of the other workloads: the chained step and the decode alone, plus
    the three variants."""
    batch = make_batch(name)
    r = Runner(batch, dev, policy=0, folded=True)
    step_ms = r.timed(steps, 5, flush)
    _, dec_ms, _ = r.kernel_times(steps, flush)
    status = int(r.eng.status.item())
    del r
    variants = measure_variants(batch, dev, flush, steps) if with_variants else {}
    out = workload_summary(name, batch, step_ms, dec_ms, variants)
    out["status"] = status
    return out


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

    batch = make_batch(args.workload)
    flush = L2Flush(dev)

    main = Runner(batch, dev, policy=0, folded=True)
    clocks = ClockSampler(local)
    clocks.start()
    step_ms = main.timed(args.steps, max(args.warmup, 3), flush, barrier)
    clk = clocks.stop()
    aux_steps = min(args.steps, 1000)
    plan_ms, dec_ms, comb_ms = main.kernel_times(aux_steps, flush)
    main.uv_setup(dev)
    uv_step_ms, uv_ms = main.uv_times(aux_steps, flush)
    no_plan_ms, no_comb_ms = main.marginal_times(aux_steps, flush)
    status = int(main.eng.status.item())
    step_ms, dec_ms = max_over_ranks([step_ms, dec_ms], dev)

    lens = batch.seq_lens.numpy()
    rows = batch.R * batch.k
    kv_b = D_QK * int(lens.sum())
    value = world * rows / (step_ms / 1e3)
    algo = algorithmic_bytes(lens, batch.M)
    flops = algorithmic_flops(lens, batch.M)
    roof = roofline(algo, flops, dec_ms / 1e3)
    # The decode as it runs in the chain: (plan -> decode) minus the plan alone.
    # Its launch overlaps the plan there (PDL), so no launch latency is counted.
    dec_chain_ms = no_comb_ms - plan_ms
    in_chain = None
    if dec_chain_ms > 0:
        rc = roofline(algo, flops, dec_chain_ms / 1e3)
        in_chain = {"decode_ms": dec_chain_ms, "achieved": rc["achieved"], "frac": rc["frac"],
                    "unit": rc["unit"]}

    variants_ms = {}
    if rank == 0 and not args.no_variants:
        variants_ms = measure_variants(batch, dev, flush, args.variant_steps)
    variants = {name: {"rows_per_s": rows / (ms / 1e3), "ms_per_step": ms,
                       "kv_gbs": kv_b / (ms / 1e3) / 1e9} for name, ms in variants_ms.items()}

    per_workload = {}
    if rank == 0 and not args.no_per_workload:
        per_workload[args.workload] = workload_summary(args.workload, batch, step_ms, dec_ms,
                                                       variants_ms)
        for name in WORKLOADS:
            if name != args.workload:
                per_workload[name] = measure_side_workload(
                    name, dev, flush, args.per_workload_steps, not args.no_variants)

    e2e_v, e2e_serial, h2d, d2h = e2e_rows_per_s(batch, dev, args.e2e_steps)
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([e2e_v, e2e_serial], device=dev, dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MIN)
        e2e_v, e2e_serial = float(t[0]) * world, float(t[1]) * world

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rps, cpu_rows, el, chunks = OracleSampler(batch).run(args.cpu_seconds)
        cpu = {"value": rps, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
               "sample": f"{chunks} consecutive {OracleSampler.CHUNK}-key chunks of the "
                         f"requests of {args.workload} = {cpu_rows:.1f} query-token rows (the batch "
                         f"has {batch.R * batch.k}; {el:.1f} s, float64 numpy)",
               "one_thread": [one_thread_oracle(w, args.one_thread_seconds)
                              for w in ONE_THREAD_WORKLOADS]}

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
                   "l2": "flushed before every step (2x L2 write + 2x L2 read, untimed)",
                   "timing": "CUDA graph per step, events around each replay",
                   "parallelism": f"replicas{world}"},
        "kv_gbs": kv_b / (step_ms / 1e3) / 1e9,
        "kv_frac_of_8tbs": kv_b / (step_ms / 1e3) / 8e12,
        "head_rows_per_s": world * batch.R * batch.M / (step_ms / 1e3),
        "kernel_ms": {"plan": plan_ms, "decode": dec_ms, "combine": comb_ms},
        "chain_ms": {"step": step_ms, "without_plan": no_plan_ms, "without_combine": no_comb_ms},
        "variants": variants,
        "per_workload": per_workload,
        "w_uv": {"step_ms": uv_step_ms, "rows_per_s": world * rows / (uv_step_ms / 1e3),
                 "uv_kernel_ms": uv_ms,
                 "what": "plan -> decode (no LSE) -> split reduction fused with the W_UV "
                         "up-projection to [R*k, H, 128] BF16 (synthetic BF16 W_UV)",
                 "gemm_flops": 2 * batch.R * batch.k * batch.H * 512 * 128},
        "roofline": dict(roof, traffic=profiled_traffic(args.workload),
                         kernel="mla_folded_decode", algorithmic_bytes_per_launch=algo,
                         algorithmic_flops_per_launch=flops,
                         timing="decode launched alone (graph replay, launch latency included)",
                         in_chain=in_chain),
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_v, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "serial_value": e2e_serial,
                "mode": "pipelined: step i+1's host-to-device copies overlap step i's plan "
                        "and decode and step i-1's read-back (two device buffer sets); "
                        "serial_value runs copy, compute and read-back in order on one "
                        "stream; each the median of three timed runs of e2e_steps steps"},
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
    sampler = OracleSampler(batch)
    # The whole run (warm-up included) targets about REFERENCE_BUDGET_S of CPU
    # work; each step runs at least one chunk.
    per_step = REFERENCE_BUDGET_S / max(1, args.steps + args.warmup)
    for _ in range(args.warmup):
        sampler.run(per_step)
    rows_t, el_t, chunks_t = 0.0, 0.0, 0
    for _ in range(args.steps):
        _, rows, el, chunks = sampler.run(per_step)
        rows_t, el_t, chunks_t = rows_t + rows, el_t + el, chunks_t + chunks
    value = rows_t / el_t
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el_t / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": args.workload, "R": batch.R, "k": batch.k, "H": batch.H,
                   "M": batch.M},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
                         "sample": f"each step: consecutive {OracleSampler.CHUNK}-key chunks of "
                                   f"the requests of {args.workload} for about "
                                   f"{per_step * 1e3:.0f} ms (at least one chunk); "
                                   f"{chunks_t} chunks = {rows_t:.1f} query-token rows "
                                   f"over the timed steps"},
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
