#!/usr/bin/env python3
"""Benchmark: paged decode attention over a chunked-slab KV pool on GB300.

One step = one decode pass over every layer of the workload (one
pkv_paged_decode_attention launch per layer) with K/V, block tables and q already
resident in HBM.  Default workload: Qwen3-0.6B-shaped decode (28 layers, Hq 16 / Hkv 8
/ D 128, bf16, 8 sequences x 4096 tokens, fragmented slab-crossing block tables).

Prints one JSON line (rank 0).  `value` is achieved HBM bandwidth in GB/s of
algorithmic bytes (K/V payload + metadata + q/out + block-table entries used +
context lengths) summed over ranks; `kv_tokens_per_s` is the other half of the metric.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl pkv|reference]
                  [--workload NAME]

`--impl reference` times the oracle (plain FP64 C on the host cores) on a bounded
sample of the same workload.  Multi-GPU runs (torchrun) are independent replicas:
every rank processes its own batch, with no collective on the data path.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from paged_kv_cache_split_gb300 import workloads as wl  # noqa: E402

METRIC = "paged decode attention: achieved HBM GB/s (% of peak), KV tokens read/s"
LAUNCHES_PER_CALL = 2  # attention kernel + split-K combine kernel
FMT_ROW_BYTES = {wl.FMT_BF16: (2.0, 2.0, 0), wl.FMT_K4V4: (0.5, 0.5, 1), wl.FMT_K8V4: (1.0, 0.5, 1),
                 wl.FMT_K8V8: (1.0, 1.0, 1)}


def token_head_bytes(fmt: int, D: int, group: int = 32) -> int:
    kb, vb, packed = FMT_ROW_BYTES[fmt]
    return int(kb * D + vb * D + packed * 2 * (D // group) * 8)


def algorithmic_bytes(fmt, D, Hkv, Hq, lens, group: int = 32) -> int:
    """K/V payload + metadata of tokens < L, q and out, block-table entries used, ctx."""
    B = len(lens)
    kv = sum(lens) * Hkv * token_head_bytes(fmt, D, group)
    qo = 2 * B * Hq * D * 2
    bt = sum(wl.nblocks(L) for L in lens) * 4
    return kv + qo + bt + 4 * B


MIXED = "d256-mixed"
STEPS_PER_REP = 8  # mixed workload: steps per repetition, each repetition from a fresh setup


def workload_for(name: str):
    if name == MIXED:
        return wl.MixedWorkload()
    if name == "qwen3-0.6b":
        return wl.qwen3_0_6b()
    if name == "tiny":
        return wl.tiny()
    if name == "qwen3-1.7b-k4v4":
        return wl.qwen3_1_7b_k4v4()
    if name == "qwen3-1.7b-k4v4-g64":
        return wl.qwen3_1_7b_k4v4_g64()
    if name == "llama-3.2-1b-k8v4":
        return wl.llama_1b(wl.FMT_K8V4)
    if name == "llama-3.2-1b-k8v8":
        return wl.llama_1b(wl.FMT_K8V8)
    raise SystemExit(f"unknown workload {name}")


def describe(w) -> str:
    L = sorted(set(w.lens))
    lens = f"{w.B} x {L[0]}" if len(L) == 1 else f"{w.B} x [{min(w.lens)}..{max(w.lens)}]"
    return (f"{w.name}-shaped decode: {w.n_layers} layer(s), Hq {w.Hq} / Hkv {w.Hkv} / D {w.D}, "
            f"{wl.FMT_NAMES[w.fmt]}{'' if w.fmt == wl.FMT_BF16 else f' (groups of {w.group})'}, {lens} tokens, "
            f"32-token blocks, 32-block slabs")


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ---------------------------------------------------------------------------

def dist_init(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def dist_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def timed_steps(run, steps: int, stream):
    """Run `steps` steps on `stream` with a CUDA event after each.  Returns the total
    time (first event to last) and the per-step times, in ms."""
    import torch
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ev[0].record(stream)
    for i in range(steps):
        run()
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    return ev[0].elapsed_time(ev[steps]), [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]


def step_stats(per_ms):
    """Distribution of per-step times (ms): median, 10th and 90th percentiles."""
    a = np.asarray(per_ms, np.float64)
    if a.size == 0:
        return None
    return {"median": round(float(np.median(a)), 5), "p10": round(float(np.percentile(a, 10)), 5),
            "p90": round(float(np.percentile(a, 90)), 5), "n": int(a.size)}


# ---------------------------------------------------------------------------
# clocks (nvidia-smi sampled in the background during the timed region)
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.samples = []
        self.proc = None
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            ident = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        except Exception:
            ident = str(device_index)
        self.cmd = ["nvidia-smi", "-i", ident, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                    "-lms", "50"]

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.samples.append(parts)

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.12)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self):
        if not self.samples:
            return None
        sm = [float(s[0]) for s in self.samples if s[0].replace(".", "").isdigit()]
        mx = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in self.samples for i in range(4) if s[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.samples)}


# ---------------------------------------------------------------------------
# measured peaks, ncu traffic record
# ---------------------------------------------------------------------------

def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured copy bandwidth (MEASURED_PEAKS.json)"
    except Exception:
        return 6800.0, "fallback 6.8 TB/s (no MEASURED_PEAKS.json)"


def _code_only(text: str) -> str:
    """C++ source without comments and blank-line or trailing-space differences."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln)


def kernel_source_hash() -> str:
    """Hash of the decode kernels' code (comments ignored): ncu figures taken on one
    kernel source stay attached to it."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_split_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.startswith("decode") or f in ("pkv_internal.cuh", "plan.cu"):
            with open(os.path.join(csrc, f), encoding="utf-8") as fh:
                h.update(f.encode() + _code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    current kernel source (else null)."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        e = rec.get(workload)
        if e and e.get("kernel_hash") == kernel_source_hash():
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


# ---------------------------------------------------------------------------
# CPU baseline (the oracle)
# ---------------------------------------------------------------------------

class OracleRun:
    """The oracle on one layer of the workload (sequences 0..n-1), using every core of
    this process's affinity (or `threads` of them)."""

    def __init__(self, w, max_seqs=None, threads=None):
        import oracle
        self.cores = threads or len(os.sched_getaffinity(0))
        self.seqs = list(range(w.B if max_seqs is None else min(max_seqs, w.B)))
        o = oracle.OraclePool(1, w.Hkv, w.D, w.fmt, seed=w.hadamard_seed, group_size=w.group)
        o.reserve_rows(w.rows_used)
        for b in self.seqs:
            k, v = w.kv(0, b)
            r, s = w.token_placement(b)
            o.write_block(0, r, s, k, v)
        self.o, self.w = o, w
        self.q = w.q(0)[self.seqs]
        self.bt = w.block_table()[self.seqs]
        self.ctx = w.ctx()[self.seqs]
        self.lens = [w.lens[b] for b in self.seqs]
        self.nbytes = algorithmic_bytes(w.fmt, w.D, w.Hkv, w.Hq, self.lens, w.group)

    def run(self) -> float:
        t0 = time.perf_counter()
        self.o.decode_attention(0, self.q, self.bt, self.ctx, self.w.scale, n_threads=self.cores)
        return time.perf_counter() - t0

    def sample_text(self, runs: int) -> str:
        w = self.w
        return (f"1 of {w.n_layers} layer(s), {len(self.seqs)} of {w.B} sequences ({sum(self.lens)} tokens), "
                f"all {w.Hq} query heads; median of {runs} runs")


def oracle_sample(w, budget_s: float = 10.0, max_seqs=None, threads=None):
    """Time the oracle until `budget_s` of CPU work (at least one run)."""
    r = OracleRun(w, max_seqs, threads)
    times = []
    t_end = time.perf_counter() + budget_s
    while True:
        times.append(r.run())
        if time.perf_counter() > t_end or len(times) >= 50:
            break
    t = statistics.median(times)
    return {"value": r.nbytes / t / 1e9, "unit": "GB/s", "cores": r.cores, "kind": "oracle",
            "sample": r.sample_text(len(times)), "seconds_per_sample": t, "kv_tokens_per_s": sum(r.lens) / t}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def run_gpu(args, rank, world, local):
    import torch
    import paged_kv_cache_split_gb300 as pkv

    torch.cuda.set_device(local)
    w = workload_for(args.workload)
    if args.layers:
        w = wl.scaled(w, w.name, n_layers=args.layers)
    dev = torch.device("cuda", local)
    pool = pkv.Pool(w.n_layers, w.Hkv, w.D, pkv.FORMAT_NAMES[w.fmt], hadamard_seed=w.hadamard_seed,
                    max_slabs=(w.rows_used + 31) // 32 + 8, group_size=w.group)
    pool.reserve_rows(w.rows_used)
    gen = torch.Generator(device=dev)
    gen.manual_seed(1000 + w.seed * 100 + rank)
    rows = np.concatenate([w.token_placement(b)[0] for b in range(w.B)])
    slots = np.concatenate([w.token_placement(b)[1] for b in range(w.B)])
    rows_d = torch.from_numpy(rows).to(dev)
    slots_d = torch.from_numpy(slots).to(dev)
    ntok = rows.size
    for layer in range(w.n_layers):
        k = torch.randn((ntok, w.Hkv, w.D), generator=gen, device=dev).to(torch.bfloat16)
        v = torch.randn((ntok, w.Hkv, w.D), generator=gen, device=dev).to(torch.bfloat16)
        pool.write_block(layer, rows_d, slots_d, k, v)
        del k, v
    q = torch.randn((w.n_layers, w.B, w.Hq, w.D), generator=gen, device=dev).to(torch.bfloat16)
    bt = torch.from_numpy(w.block_table()).to(dev)
    ctx = torch.from_numpy(w.ctx()).to(dev)
    out = torch.empty_like(q)
    ws = pool.workspace(w.B, w.Hq, dev)
    max_ctx = max(w.lens)

    def step():
        for layer in range(w.n_layers):
            pool.paged_decode_attention(layer, q[layer], bt, ctx, w.scale, max_ctx=max_ctx, out=out[layer],
                                        workspace=ws)

    # Eager pass: per-launch CUDA events on the launching stream.
    stream = torch.cuda.current_stream()
    step()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * w.n_layers)]
    for layer in range(w.n_layers):
        ev[2 * layer].record(stream)
        pool.paged_decode_attention(layer, q[layer], bt, ctx, w.scale, max_ctx=max_ctx, out=out[layer], workspace=ws)
        ev[2 * layer + 1].record(stream)
    torch.cuda.synchronize()
    eager_launch_us = statistics.median(ev[2 * i].elapsed_time(ev[2 * i + 1]) * 1e3 for i in range(w.n_layers))
    if pool.check_errors():
        raise SystemExit("device error word set during setup")

    # CUDA graph of one step (all layers) for the timed region.
    graph = None
    if not args.no_graph:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            step()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        torch.cuda.synchronize()
    run = graph.replay if graph is not None else step

    # End-to-end arm: the step's inputs (q, block table, context lengths) packed in one
    # pinned host buffer and copied in with one copy, the result copied out, every step.
    # Two device input buffers and two output buffers let step i+1's copy in and step
    # i-1's copy out (one copy stream each way) run under step i's kernels.
    def seg(nbytes):
        return (nbytes + 255) // 256 * 256

    qb, btb, cb = q.numel() * 2, bt.numel() * 4, ctx.numel() * 4
    off_bt = seg(qb)
    off_ctx = off_bt + seg(btb)
    in_h = torch.zeros(off_ctx + seg(cb), dtype=torch.uint8, pin_memory=True)
    in_h[:qb].copy_(q.cpu().reshape(-1).view(torch.uint8))
    in_h[off_bt:off_bt + btb].copy_(bt.cpu().reshape(-1).view(torch.uint8))
    in_h[off_ctx:off_ctx + cb].copy_(ctx.cpu().reshape(-1).view(torch.uint8))
    in_e = [torch.empty(in_h.shape, dtype=torch.uint8, device=dev) for _ in range(2)]
    views = [(x[:qb].view(torch.bfloat16).view(q.shape), x[off_bt:off_bt + btb].view(torch.int32).view(bt.shape),
              x[off_ctx:off_ctx + cb].view(torch.int32).view(ctx.shape)) for x in in_e]
    out_h = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
    out_e = [torch.empty_like(out) for _ in range(2)]
    h2d_s, d2h_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    h2d_done, comp_done, d2h_done = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))

    def e2e_steps(n):
        """Enqueue n end-to-end steps on the current stream; it then waits for the last copy out."""
        cur = torch.cuda.current_stream()
        for i in range(n):
            j = i & 1
            with torch.cuda.stream(h2d_s):
                if i == 0:
                    h2d_s.wait_stream(cur)
                elif i >= 2:
                    h2d_s.wait_event(comp_done[j])  # step i-2 has read in_e[j]
                in_e[j].copy_(in_h, non_blocking=True)
                h2d_done[j].record(h2d_s)
            cur.wait_event(h2d_done[j])
            if i >= 2:
                cur.wait_event(d2h_done[j])  # step i-2's result has left out_e[j]
            qv, btv, cv = views[j]
            for layer in range(w.n_layers):
                pool.paged_decode_attention(layer, qv[layer], btv, cv, w.scale, max_ctx=max_ctx,
                                            out=out_e[j][layer], workspace=ws)
            comp_done[j].record(cur)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(comp_done[j])
                out_h[j].copy_(out_e[j], non_blocking=True)
                d2h_done[j].record(d2h_s)
        cur.wait_stream(d2h_s)

    sampler = ClockSampler(local)
    with sampler:
        for _ in range(args.warmup):
            run()
        torch.cuda.synchronize()
        dist_barrier(world)
        torch.cuda.synchronize()
        total, per_step = timed_steps(run, args.steps, stream)
        dist_barrier(world)
        ms_step = total / args.steps
        # end-to-end, through the public API with host buffers
        e2e_steps(max(2, args.warmup))
        torch.cuda.synchronize()
        dist_barrier(world)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        e2e_steps(args.steps)
        e1.record(stream)
        torch.cuda.synchronize()
        dist_barrier(world)
        ms_e2e = e0.elapsed_time(e1) / args.steps
    if pool.check_errors():
        raise SystemExit("device error word set during the timed region")
    if not all(torch.equal(x, out) for x in out_e) or not all(torch.equal(x, out.cpu()) for x in out_h):
        raise SystemExit("end-to-end result differs from the device-resident result")

    ms_step = dist_max(ms_step, world)
    ms_e2e = dist_max(ms_e2e, world)
    bytes_layer = algorithmic_bytes(w.fmt, w.D, w.Hkv, w.Hq, w.lens, w.group)
    bytes_step = bytes_layer * w.n_layers
    tokens_step = sum(w.lens) * w.n_layers
    value = bytes_step * world / (ms_step * 1e-3) / 1e9
    launch_us = ms_step * 1e3 / w.n_layers
    achieved = bytes_layer / (launch_us * 1e-6) / 1e9
    peak, peak_src = measured_peak()
    h2d = in_h.numel()
    d2h = out.numel() * 2
    res = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "step_ms": step_stats(per_step),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded N(0,1) bf16 K/V and q; no model weights)",
        "config": {"workload": describe(w), "global_batch": w.B * world, "seq_len": max(w.lens),
                   "layers": w.n_layers, "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": f"inputs larger than L2 ({bytes_step / 1e9:.2f} GB read per step vs 129 MB L2)",
                   "cuda_graph": graph is not None},
        "kv_tokens_per_s": round(tokens_step * world / (ms_step * 1e-3), 1),
        "pct_of_nominal_8tbs": round(100 * value / world / 8000.0, 2),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": ncu_traffic(args.workload),
                     "per_launch_bytes": bytes_layer, "avg_launch_us": round(launch_us, 3),
                     "eager_launch_us": round(eager_launch_us, 3), "peak_source": peak_src,
                     "kernel": "decode attention kernel + split-K combine kernel (per-launch time is their sum)"},
        "e2e": {"value": round(bytes_step * world / (ms_e2e * 1e-3) / 1e9, 1), "unit": "GB/s",
                "ms_per_step": round(ms_e2e, 5), "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": LAUNCHES_PER_CALL * w.n_layers * args.steps,
        "clocks": sampler.summary(),
    }
    return res, w


def mixed_row_bytes(fmt: int, Hkv: int, D: int) -> int:
    """Bytes of one 32-token block (row) of one layer, all stored tensors."""
    return 32 * Hkv * token_head_bytes(fmt, D)


class MixedRun:
    """D256 mixed workload on the GPU: two pools (bf16, K4/V4) of one layer.  A
    repetition is a fresh setup (untimed: initial K/V written, the host plans of its
    steps and their inputs made resident) followed by STEPS_PER_REP timed steps; a
    step is, per pool, copy_on_write_block of the step's pairs, write_block of one
    token per sequence and paged_decode_attention of every sequence."""

    def __init__(self, dev, rank: int):
        import torch
        import paged_kv_cache_split_gb300 as pkv
        self.torch, self.pkv, self.dev, self.rank = torch, pkv, dev, rank
        m = wl.MixedWorkload()
        self.m0 = m
        self.Hq, self.Hkv, self.D, self.scale = m.Hq, m.Hkv, m.D, m.scale
        self.max_ctx = m.Lmax + 64
        # rows needed after the last step of a repetition bound the pools' capacity
        probe = wl.MixedWorkload()
        for _ in range(STEPS_PER_REP):
            probe.plan_step()
        self.pools = []
        for P, Pp in zip(m.pools, probe.pools):
            rows = Pp.next_row
            pool = pkv.Pool(1, m.Hkv, m.D, "bf16" if P.fmt == wl.FMT_BF16 else "k4v4",
                            hadamard_seed=m.hadamard_seed, max_slabs=(rows + 31) // 32 + 8)
            pool.reserve_rows(rows)
            self.pools.append(pool)
        self.outs = [torch.empty((len(P.seqs), m.Hq, m.D), dtype=torch.bfloat16, device=dev) for P in m.pools]
        self.ws = [pool.workspace(len(P.seqs), m.Hq, dev) for pool, P in zip(self.pools, m.pools)]

    def setup_rep(self):
        """Fresh workload state: write every sequence's initial K/V (prefix blocks once
        per group) and prepare the inputs of the repetition's steps on the device and
        in pinned host memory."""
        torch = self.torch
        m = wl.MixedWorkload()
        gen = torch.Generator(device=self.dev)
        for pi, (P, pool) in enumerate(zip(m.pools, self.pools)):
            rr, ss = [], []
            for i in range(len(P.seqs)):
                t = np.arange(P.lens[i])
                own = np.ones(P.lens[i], bool)
                if P.group_of[i] * m.group_size != i:
                    own[: m.prefix] = False
                rr.append(np.asarray(P.rows[i], np.int32)[t // 32][own])
                ss.append((t % 32).astype(np.int32)[own])
            rows = torch.from_numpy(np.concatenate(rr)).to(self.dev)
            slots = torch.from_numpy(np.concatenate(ss)).to(self.dev)
            gen.manual_seed(4000 + 10 * pi + self.rank)
            n = rows.numel()
            for a in range(0, n, 1 << 18):  # chunks keep the temporaries small
                b = min(n, a + (1 << 18))
                k = torch.randn((b - a, m.Hkv, m.D), generator=gen, device=self.dev).to(torch.bfloat16)
                v = torch.randn((b - a, m.Hkv, m.D), generator=gen, device=self.dev).to(torch.bfloat16)
                pool.write_block(0, rows[a:b], slots[a:b], k, v)
        steps = []
        for step in range(STEPS_PER_REP):
            plan = m.plan_step()
            per_pool = []
            for pi, P in enumerate(m.pools):
                st = plan[pi]
                k, v = m.step_kv(step, pi)
                host = {
                    "cow_src": st["cow_src"], "cow_dst": st["cow_dst"],
                    "rows": st["write_rows"], "slots": st["write_slots"],
                    "k": self._bf16(k), "v": self._bf16(v), "q": self._bf16(m.step_q(step, pi)),
                    "bt": m.block_table(pi, wl.nblocks(self.max_ctx)), "ctx": m.ctx(pi),
                }
                per_pool.append(host)
            steps.append(per_pool)
        self.steps_host = steps
        self.steps_dev = [[{k: self._dev(v) for k, v in h.items()} for h in sp] for sp in steps]
        # end-to-end arm: each step's inputs of both pools packed in one pinned host buffer
        # (256-byte aligned segments), copied in with one copy, used through device views
        self.step_in_h, self.step_in_e, self.steps_e2e = [], [], []
        for sp in steps:
            hosts = [self._host(v) for h in sp for v in h.values()]
            offs, total = [], 0
            for t in hosts:
                offs.append(total)
                total += (t.numel() * t.element_size() + 255) // 256 * 256
            buf_h = torch.zeros(max(total, 256), dtype=torch.uint8, pin_memory=True)
            buf_e = torch.empty(buf_h.shape, dtype=torch.uint8, device=self.dev)
            views, j = [], 0
            for h in sp:
                vh = {}
                for key in h:
                    t, off = hosts[j], offs[j]
                    n = t.numel() * t.element_size()
                    if n:
                        buf_h[off:off + n].copy_(t.reshape(-1).view(torch.uint8))
                    vh[key] = buf_e[off:off + n].view(t.dtype).view(t.shape)
                    j += 1
                views.append(vh)
            self.step_in_h.append(buf_h)
            self.step_in_e.append(buf_e)
            self.steps_e2e.append(views)
        self.out_h = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in self.outs]
        torch.cuda.synchronize()
        self.m = m

    def _bf16(self, bits):
        return self.torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(self.torch.bfloat16)

    def _dev(self, x):
        t = x if isinstance(x, self.torch.Tensor) else self.torch.from_numpy(np.ascontiguousarray(x))
        return t.to(self.dev)

    def _host(self, x):
        return (x if isinstance(x, self.torch.Tensor) else self.torch.from_numpy(np.ascontiguousarray(x))).contiguous()

    def run_step(self, i: int, e2e: bool = False):
        if e2e:
            self.step_in_e[i].copy_(self.step_in_h[i], non_blocking=True)
        for pi, pool in enumerate(self.pools):
            d = self.steps_e2e[i][pi] if e2e else self.steps_dev[i][pi]
            if d["cow_src"].numel():
                pool.copy_on_write_block(d["cow_src"], d["cow_dst"])
            pool.write_block(0, d["rows"], d["slots"], d["k"], d["v"])
            pool.paged_decode_attention(0, d["q"], d["bt"], d["ctx"], self.scale, max_ctx=self.max_ctx,
                                        out=self.outs[pi], workspace=self.ws[pi])
            if e2e:
                self.out_h[pi].copy_(self.outs[pi], non_blocking=True)

    def step_bytes(self, i: int) -> int:
        """Decode algorithmic bytes of both pools at the step's lengths, plus the
        write (bf16 K/V in, stored rows out) and copy-on-write (block read + write)."""
        total = 0
        for pi, P in enumerate(self.m.pools):
            h = self.steps_host[i][pi]
            lens = [int(x) for x in h["ctx"]]
            total += algorithmic_bytes(P.fmt, self.D, self.Hkv, self.Hq, lens)
            n = len(h["rows"])
            total += n * self.Hkv * (2 * self.D * 2 + token_head_bytes(P.fmt, self.D))
            total += 2 * len(h["cow_src"]) * mixed_row_bytes(P.fmt, self.Hkv, self.D)
        return total

    def launches(self, i: int) -> int:
        return sum((1 if len(self.steps_host[i][pi]["cow_src"]) else 0) + 1 + LAUNCHES_PER_CALL
                   for pi in range(len(self.pools)))

    def h2d_d2h(self, i: int):
        h2d = int(self.step_in_h[i].numel())
        d2h = sum(int(o.numel() * o.element_size()) for o in self.outs)
        return h2d, d2h


def run_gpu_mixed(args, rank, world, local):
    import torch

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    mr = MixedRun(dev, rank)
    stream = torch.cuda.current_stream()
    reps = max(1, math.ceil(args.steps / STEPS_PER_REP))
    wreps = max(1, math.ceil(args.warmup / STEPS_PER_REP))
    sampler = ClockSampler(local)
    t_dev, t_e2e, nbytes, launches, h2d, d2h = 0.0, 0.0, 0, 0, 0, 0
    per_step = []
    with sampler:
        for r in range(wreps + reps):
            timed = r >= wreps
            for e2e in (False, True):
                mr.setup_rep()
                dist_barrier(world)
                torch.cuda.synchronize()
                it = iter(range(STEPS_PER_REP))
                ms, per = timed_steps(lambda: mr.run_step(next(it), e2e=e2e), STEPS_PER_REP, stream)
                dist_barrier(world)
                if timed:
                    if e2e:
                        t_e2e += ms
                    else:
                        t_dev += ms
                        per_step += per
                        nbytes += sum(mr.step_bytes(i) for i in range(STEPS_PER_REP))
                        launches += sum(mr.launches(i) for i in range(STEPS_PER_REP))
                        io = [mr.h2d_d2h(i) for i in range(STEPS_PER_REP)]
                        h2d += sum(x for x, _ in io)
                        d2h += sum(y for _, y in io)
    for pool in mr.pools:
        if pool.check_errors():
            raise SystemExit("device error word set during the timed region")
    nsteps = reps * STEPS_PER_REP
    ms_step = dist_max(t_dev / nsteps, world)
    ms_e2e = dist_max(t_e2e / nsteps, world)
    bytes_step = nbytes / nsteps
    value = bytes_step * world / (ms_step * 1e-3) / 1e9
    peak, peak_src = measured_peak()
    m = mr.m0
    tokens_step = sum(int(x) for sp in mr.steps_host for h in sp for x in h["ctx"]) / STEPS_PER_REP
    res = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": nsteps,
        "warmup": wreps * STEPS_PER_REP,
        "ms_per_step": round(ms_step, 5),
        "step_ms": step_stats(per_step),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded N(0,1) bf16 K/V and q; no model weights)",
        "config": {"workload": (f"D256 long-context mixed: 1 layer, Hq {m.Hq} / Hkv {m.Hkv} / D {m.D}, "
                                f"{m.B} sequences (16 bf16 + 16 K4/V4 pools), lengths 1024 + U[1..{m.Lmax - 1024}], "
                                f"8 prefix groups sharing 1024 tokens; per step: 1 token written per sequence, "
                                f"copy-on-write of {m.n_cow} shared blocks, decode of both pools"),
                   "global_batch": m.B * world, "seq_len": m.Lmax, "layers": 1,
                   "steps_per_repetition": STEPS_PER_REP,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": f"inputs larger than L2 ({bytes_step / 1e9:.2f} GB read per step vs 129 MB L2)",
                   "cuda_graph": False},
        "kv_tokens_per_s": round(tokens_step * world / (ms_step * 1e-3), 1),
        "pct_of_nominal_8tbs": round(100 * value / world / 8000.0, 2),
        "roofline": {"bound": "hbm", "achieved": round(bytes_step / (ms_step * 1e-3) / 1e9, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(bytes_step / (ms_step * 1e-3) / 1e9 / peak, 4),
                     "traffic": ncu_traffic(MIXED), "per_launch_bytes": int(bytes_step),
                     "avg_launch_us": round(ms_step * 1e3, 3), "peak_source": peak_src,
                     "kernel": "whole step: copy-on-write, write_block and decode (attention + combine) of both pools"},
        "e2e": {"value": round(bytes_step * world / (ms_e2e * 1e-3) / 1e9, 1), "unit": "GB/s",
                "ms_per_step": round(ms_e2e, 5), "h2d_bytes_per_step": int(h2d / nsteps),
                "d2h_bytes_per_step": int(d2h / nsteps)},
        "gpu_launches": int(launches),
        "clocks": sampler.summary(),
    }
    return res, mr


def mixed_oracle_sample(budget_s: float = 10.0):
    """The oracle on one sequence of each pool of the mixed workload (initial state),
    timed until `budget_s` of CPU work."""
    import oracle
    m = wl.MixedWorkload()
    cores = len(os.sched_getaffinity(0))
    runs = []
    for pi, P in enumerate(m.pools):
        o = oracle.OraclePool(1, m.Hkv, m.D, P.fmt, seed=m.hadamard_seed)
        o.reserve_rows(P.next_row)
        k, v = m.initial_kv(pi, 0)
        t = np.arange(P.lens[0])
        o.write_block(0, np.asarray(P.rows[0], np.int32)[t // 32], (t % 32).astype(np.int32), k, v)
        q = m.step_q(0, pi)[:1]
        bt = m.block_table(pi)[:1]
        ctx = m.ctx(pi)[:1]
        runs.append((o, q, bt, ctx, P.fmt, int(ctx[0])))
    times = []
    t_end = time.perf_counter() + budget_s
    while True:
        t0 = time.perf_counter()
        for o, q, bt, ctx, _, _ in runs:
            o.decode_attention(0, q, bt, ctx, m.scale, n_threads=cores)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() > t_end or len(times) >= 50:
            break
    t = statistics.median(times)
    nbytes = sum(algorithmic_bytes(f, m.D, m.Hkv, m.Hq, [L]) for _, _, _, _, f, L in runs)
    return {"value": nbytes / t / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": (f"decode of sequence 0 of each pool (bf16 {runs[0][5]} and K4/V4 {runs[1][5]} tokens, "
                       f"all {m.Hq} query heads, 1 layer); median of {len(times)} runs"),
            "seconds_per_sample": t, "kv_tokens_per_s": sum(r[5] for r in runs) / t}


BLOCKS = "blocks-export"


def blocks_oracle_sample(budget_s: float = 10.0, n_blocks: int = 64):
    """The oracle's export of n_blocks blocks of a 28-layer Qwen3-0.6B-shaped bf16 image."""
    import oracle
    oracle.build()
    w = wl.qwen3_0_6b()
    o = oracle.OraclePool(w.n_layers, w.Hkv, w.D, w.fmt, seed=w.hadamard_seed)
    o.reserve_rows(n_blocks)
    rng = wl.rng_for(77)
    rows = np.repeat(np.arange(n_blocks, dtype=np.int32), 32)
    slots = np.tile(np.arange(32, dtype=np.int32), n_blocks)
    for layer in range(w.n_layers):
        o.write_block(layer, rows, slots, wl.bf16_normal(rng, (rows.size, w.Hkv, w.D)),
                      wl.bf16_normal(rng, (rows.size, w.Hkv, w.D)))
    blk = np.arange(n_blocks, dtype=np.int32)
    times, t_end = [], time.perf_counter() + budget_s
    while time.perf_counter() < t_end or len(times) < 3:
        t0 = time.perf_counter()
        o.export_blocks(blk)
        times.append(time.perf_counter() - t0)
    t = statistics.median(times)
    nbytes = 2 * n_blocks * o.record_bytes
    return {"value": nbytes / t / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"export of {n_blocks} of 1024 blocks (28 layers, bf16), read + write bytes; median of {len(times)} runs",
            "seconds_per_sample": t}


def run_gpu_blocks(args, rank, world, local):
    """Block records: export every block of the Qwen3-0.6B-shaped pool (28 layers, 8 x 4096
    tokens) to a device buffer; a step moves each record's bytes once in and once out."""
    import torch
    import paged_kv_cache_split_gb300 as pkv

    torch.cuda.set_device(local)
    w = wl.qwen3_0_6b(n_layers=args.layers) if args.layers else wl.qwen3_0_6b()
    dev = torch.device("cuda", local)
    pool = pkv.Pool(w.n_layers, w.Hkv, w.D, pkv.FORMAT_NAMES[w.fmt], hadamard_seed=w.hadamard_seed,
                    max_slabs=(w.rows_used + 31) // 32 + 8)
    pool.reserve_rows(w.rows_used)
    gen = torch.Generator(device=dev)
    gen.manual_seed(2000 + rank)
    rows = np.concatenate([w.token_placement(b)[0] for b in range(w.B)])
    slots = np.concatenate([w.token_placement(b)[1] for b in range(w.B)])
    rows_d, slots_d = torch.from_numpy(rows).to(dev), torch.from_numpy(slots).to(dev)
    for layer in range(w.n_layers):
        k = torch.randn((rows.size, w.Hkv, w.D), generator=gen, device=dev).to(torch.bfloat16)
        v = torch.randn((rows.size, w.Hkv, w.D), generator=gen, device=dev).to(torch.bfloat16)
        pool.write_block(layer, rows_d, slots_d, k, v)
        del k, v
    bt = w.block_table()
    blocks = np.concatenate([bt[b][: wl.nblocks(w.lens[b])] for b in range(w.B)]).astype(np.int32)
    blocks_d = torch.from_numpy(blocks).to(dev)
    rec = pool.export_blocks(blocks_d)
    stream = torch.cuda.current_stream()
    rec_h = torch.empty(rec.shape, dtype=torch.uint8, pin_memory=True)
    blocks_h = torch.from_numpy(blocks).pin_memory()
    blocks_e = torch.empty_like(blocks_d)

    def step():
        pool.export_blocks(blocks_d, out=rec)

    def e2e_step():
        blocks_e.copy_(blocks_h, non_blocking=True)
        pool.export_blocks(blocks_e, out=rec)
        rec_h.copy_(rec, non_blocking=True)

    sampler = ClockSampler(local)
    with sampler:
        for _ in range(max(3, args.warmup)):
            step()
        torch.cuda.synchronize()
        dist_barrier(world)
        total, per_step = timed_steps(step, args.steps, stream)
        dist_barrier(world)
        ms_step = total / args.steps
        for _ in range(max(1, args.warmup)):
            e2e_step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        dist_barrier(world)
        ms_e2e = e0.elapsed_time(e1) / args.steps
    if pool.check_errors():
        raise SystemExit("device error word set during the timed region")
    ms_step, ms_e2e = dist_max(ms_step, world), dist_max(ms_e2e, world)
    moved = 2 * rec.numel()  # each record byte read from the slabs and written to the buffer
    value = moved * world / (ms_step * 1e-3) / 1e9
    peak, peak_src = measured_peak()
    res = {"metric": "block export: achieved HBM GB/s (read + write bytes)", "value": round(value, 1), "unit": "GB/s",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
           "step_ms": step_stats(per_step),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
           "data": "synthetic (seeded N(0,1) bf16 K/V; no model weights)",
           "config": {"workload": f"block export: {blocks.size} blocks x {pool.block_record_bytes()} B records "
                                  f"(Qwen3-0.6B-shaped pool, {w.n_layers} layers, bf16)",
                      "global_batch": w.B * world, "seq_len": max(w.lens), "layers": w.n_layers,
                      "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                      "l2": f"inputs larger than L2 ({rec.numel() / 1e9:.2f} GB per step vs 129 MB L2)"},
           "roofline": {"bound": "hbm", "achieved": round(value / world, 1), "peak": peak, "unit": "GB/s",
                        "frac": round(value / world / peak, 4), "traffic": None, "per_launch_bytes": int(moved),
                        "avg_launch_us": round(ms_step * 1e3, 3), "peak_source": peak_src, "kernel": "serde_blocks_kernel"},
           "e2e": {"value": round(moved * world / (ms_e2e * 1e-3) / 1e9, 1), "unit": "GB/s", "ms_per_step": round(ms_e2e, 5),
                   "h2d_bytes_per_step": int(blocks.nbytes), "d2h_bytes_per_step": int(rec.numel())},
           "gpu_launches": args.steps, "clocks": sampler.summary()}
    return res


PREFILL = "prefill-qwen3-0.6b"
PREFILL_PACKED = "prefill-qwen3-1.7b-k4v4"
PREFILL_NQ = 8  # new tokens per sequence in the chunk


def prefill_launches_per_call(fmt: int, D: int, G: int, n_q: int) -> int:
    """Kernels one prefill call launches: attention and combine, plus the expansion of
    the block table unless the chunk's queries fit one tile (the library's choice of
    queries per tile, restated: up to 16 (query, head) rows at head_dim <= 128, 8 at
    256; bf16 takes the largest power of two dividing the chunk, the packed formats
    the count filling 16 rows, else 8)."""
    rows = 16 if D <= 128 else 8
    nq = 1
    if fmt == wl.FMT_BF16:
        for c in (16, 8, 4, 2):
            if c * G <= rows and n_q % c == 0:
                nq = c
                break
    else:
        for r in (rows, 8) if rows == 16 else (8,):
            c = r // G
            if c > 1 and n_q % c == 0:
                nq = c
                break
    return 2 if (nq == n_q and nq > 1) else 3


def prefill_oracle_sample(budget_s: float = 10.0, n_seqs: int = 2):
    """The oracle's chunked prefill on one layer of the Qwen3-0.6B-shaped workload,
    sequences 0..n_seqs-1, all host cores it may use."""
    import oracle
    oracle.build()
    w = wl.qwen3_0_6b(n_layers=1)
    o = oracle.OraclePool(1, w.Hkv, w.D, w.fmt, seed=w.hadamard_seed)
    o.reserve_rows(w.rows_used)
    for b in range(n_seqs):
        k, v = w.kv(0, b)
        r, sl = w.token_placement(b)
        o.write_block(0, r, sl, k, v)
    q = wl.bf16_normal(wl.rng_for(91), (n_seqs, PREFILL_NQ, w.Hq, w.D))
    bt = w.block_table()[:n_seqs]
    ctx = w.ctx()[:n_seqs]
    times, t_end = [], time.perf_counter() + budget_s
    while time.perf_counter() < t_end or len(times) < 2:
        t0 = time.perf_counter()
        o.prefill_attention(0, q, bt, ctx, w.scale)
        times.append(time.perf_counter() - t0)
    t = statistics.median(times)
    nbytes = int(ctx.sum()) * w.Hkv * token_head_bytes(w.fmt, w.D) + 2 * n_seqs * PREFILL_NQ * w.Hq * w.D * 2
    return {"value": nbytes / t / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"1 of 28 layers, {n_seqs} of 8 sequences, chunk of {PREFILL_NQ} queries; median of {len(times)} runs",
            "seconds_per_sample": t}


def run_gpu_prefill(args, rank, world, local):
    """Chunked prefill: the Qwen3-0.6B-shaped pool (28 layers, 8 x 4096 tokens), the last
    PREFILL_NQ tokens of every sequence being the chunk; a step is one causal prefill
    attention call per layer.  Bytes are the decode's (K/V of every visible token once,
    q and out of every query, block-table entries, context lengths)."""
    import torch
    import paged_kv_cache_split_gb300 as pkv

    torch.cuda.set_device(local)
    if args.workload == PREFILL_PACKED:
        w = wl.qwen3_1_7b_k4v4()
    else:
        w = wl.qwen3_0_6b(n_layers=args.layers) if args.layers else wl.qwen3_0_6b()
    n_q = PREFILL_NQ
    dev = torch.device("cuda", local)
    pool = pkv.Pool(w.n_layers, w.Hkv, w.D, pkv.FORMAT_NAMES[w.fmt], hadamard_seed=w.hadamard_seed,
                    max_slabs=(w.rows_used + 31) // 32 + 8)
    pool.reserve_rows(w.rows_used)
    gen = torch.Generator(device=dev)
    gen.manual_seed(3000 + rank)
    rows = np.concatenate([w.token_placement(b)[0] for b in range(w.B)])
    slots = np.concatenate([w.token_placement(b)[1] for b in range(w.B)])
    rows_d, slots_d = torch.from_numpy(rows).to(dev), torch.from_numpy(slots).to(dev)
    for layer in range(w.n_layers):
        k = torch.randn((rows.size, w.Hkv, w.D), generator=gen, device=dev).to(torch.bfloat16)
        v = torch.randn((rows.size, w.Hkv, w.D), generator=gen, device=dev).to(torch.bfloat16)
        pool.write_block(layer, rows_d, slots_d, k, v)
        del k, v
    q = torch.randn((w.n_layers, w.B, n_q, w.Hq, w.D), generator=gen, device=dev).to(torch.bfloat16)
    bt = torch.from_numpy(w.block_table()).to(dev)
    ctx = torch.from_numpy(w.ctx()).to(dev)
    out = torch.empty_like(q)
    ws = torch.zeros(pool.prefill_workspace_bytes(w.B, n_q, w.Hq, int(bt.shape[1])), dtype=torch.uint8, device=dev)
    max_ctx = max(w.lens)

    def step():
        for layer in range(w.n_layers):
            pool.paged_prefill_attention(layer, q[layer], bt, ctx, w.scale, max_ctx=max_ctx, out=out[layer], workspace=ws)

    step()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    q_h, out_h = q.cpu().pin_memory(), torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    q_e = torch.empty_like(q)

    def e2e_step():
        q_e.copy_(q_h, non_blocking=True)
        for layer in range(w.n_layers):
            pool.paged_prefill_attention(layer, q_e[layer], bt, ctx, w.scale, max_ctx=max_ctx, out=out[layer], workspace=ws)
        out_h.copy_(out, non_blocking=True)

    sampler = ClockSampler(local)
    with sampler:
        for _ in range(max(3, args.warmup)):
            graph.replay()
        torch.cuda.synchronize()
        dist_barrier(world)
        total, per_step = timed_steps(graph.replay, args.steps, stream)
        dist_barrier(world)
        ms_step = total / args.steps
        for _ in range(max(1, args.warmup)):
            e2e_step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        dist_barrier(world)
        ms_e2e = e0.elapsed_time(e1) / args.steps
    if pool.check_errors():
        raise SystemExit("device error word set during the timed region")
    ms_step, ms_e2e = dist_max(ms_step, world), dist_max(ms_e2e, world)
    kv = sum(w.lens) * w.Hkv * token_head_bytes(w.fmt, w.D)
    qo = 2 * w.B * n_q * w.Hq * w.D * 2
    bytes_layer = kv + qo + sum(wl.nblocks(L) for L in w.lens) * 4 + 4 * w.B
    bytes_step = bytes_layer * w.n_layers
    value = bytes_step * world / (ms_step * 1e-3) / 1e9
    peak, peak_src = measured_peak()
    launch_us = ms_step * 1e3 / w.n_layers
    per_call = prefill_launches_per_call(w.fmt, w.D, w.Hq // w.Hkv, n_q)
    res = {"metric": "chunked prefill attention: achieved HBM GB/s (K/V of the visible context once), query tokens/s",
           "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(ms_step, 5), "step_ms": step_stats(per_step), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None,
           "dtype": "f32", "data": "synthetic (seeded N(0,1) bf16 K/V and q; no model weights)",
           "config": {"workload": f"chunked prefill: {describe(w)}; the last {n_q} tokens of each sequence are the chunk",
                      "global_batch": w.B * world, "seq_len": max(w.lens), "layers": w.n_layers,
                      "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                      "l2": f"inputs larger than L2 ({bytes_step / 1e9:.2f} GB per step vs 129 MB L2)", "cuda_graph": True},
           "query_tokens_per_s": round(w.B * n_q * w.n_layers * world / (ms_step * 1e-3), 1),
           "roofline": {"bound": "hbm", "achieved": round(bytes_layer / (launch_us * 1e-6) / 1e9, 1), "peak": peak,
                        "unit": "GB/s", "frac": round(bytes_layer / (launch_us * 1e-6) / 1e9 / peak, 4), "traffic": ncu_traffic(args.workload),
                        "per_launch_bytes": bytes_layer, "avg_launch_us": round(launch_us, 3), "peak_source": peak_src,
                        "kernel": ("attention + combine kernels per layer" if per_call == 2 else
                                   "expansion + attention + combine kernels per layer")},
           "e2e": {"value": round(bytes_step * world / (ms_e2e * 1e-3) / 1e9, 1), "unit": "GB/s",
                   "ms_per_step": round(ms_e2e, 5), "h2d_bytes_per_step": int(q.numel() * 2),
                   "d2h_bytes_per_step": int(out.numel() * 2)},
           "gpu_launches": per_call * w.n_layers * args.steps, "clocks": sampler.summary()}
    return res


DEFAULT_WORKLOAD = "qwen3-0.6b"
# Sub-records of the default line: every other configuration measured in the same
# process (same box, same clock sampler conventions), each with its own steps.
EXTRA_WORKLOADS = ["qwen3-1.7b-k4v4", "qwen3-1.7b-k4v4-g64", "llama-3.2-1b-k8v4", "llama-3.2-1b-k8v8",
                   "d256-mixed", "prefill-qwen3-0.6b", "prefill-qwen3-1.7b-k4v4"]
EXTRA_KEYS = ("metric", "value", "unit", "ms_per_step", "step_ms", "steps", "warmup", "pct_of_nominal_8tbs",
              "kv_tokens_per_s", "query_tokens_per_s", "roofline", "e2e", "gpu_launches", "clocks")


def run_extras(args, rank, world, local):
    """Measure EXTRA_WORKLOADS one after another (pools freed in between) with the
    default line's warm-up and at most 100 timed steps each (32 for the mixed
    workload, whose repetitions start from a fresh setup)."""
    import gc
    import torch
    out = []
    for name in EXTRA_WORKLOADS:
        a = argparse.Namespace(**vars(args))
        a.workload = name
        a.layers = 0
        a.steps = min(args.steps, 32 if name == MIXED else 100)
        if name == MIXED:
            r, _ = run_gpu_mixed(a, rank, world, local)
        elif name in (PREFILL, PREFILL_PACKED):
            r = run_gpu_prefill(a, rank, world, local)
        else:
            r, _ = run_gpu(a, rank, world, local)
        rec = {"workload": name, "config": r["config"]["workload"]}
        rec.update({k: r[k] for k in EXTRA_KEYS if k in r})
        out.append(rec)
        del r
        gc.collect()
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="pkv", choices=["pkv", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-extra", action="store_true",
                    help="with the default workload, skip the other workloads' sub-records")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0,
                    help="override the workload's layer count: fewer for profiling captures, or a whole "
                         "model's count for the one-layer packed workloads (16 for the Llama-3.2-1B "
                         "shapes, 28 for Qwen3-1.7B); never fewer than the default for a reported number")
    args = ap.parse_args()
    rank, world, local = dist_init(args.gpus)

    if args.impl == "reference" and args.workload == MIXED:
        if rank != 0:
            return
        import oracle
        oracle.build()
        cb = mixed_oracle_sample(budget_s=max(2.0, 0.05 * (args.warmup + args.steps)))
        m = wl.MixedWorkload()
        t = cb["seconds_per_sample"]
        res = {"impl": "reference", "metric": METRIC, "value": round(cb["value"], 4), "unit": "GB/s", "n_gpus": 1,
               "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t * 1e3, 3),
               "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
               "data": "synthetic (seeded N(0,1) bf16 K/V and q; no model weights)",
               "config": {"workload": "D256 long-context mixed (decode of one sequence per pool)",
                          "global_batch": m.B, "seq_len": m.Lmax, "layers": 1, "parallelism": "host cores"},
               "kv_tokens_per_s": round(cb["kv_tokens_per_s"], 1),
               "cpu_baseline": {"value": round(cb["value"], 4), "unit": "GB/s", "cores": cb["cores"],
                                "kind": "oracle", "sample": cb["sample"]},
               "e2e": {"value": round(cb["value"], 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                       "d2h_bytes_per_step": 0}}
        print(json.dumps(res), flush=True)
        return

    if args.workload in (PREFILL, PREFILL_PACKED):
        if args.impl == "reference":
            if rank == 0:
                cb = prefill_oracle_sample(budget_s=max(2.0, 0.05 * (args.warmup + args.steps)))
                print(json.dumps({"impl": "reference", "metric": "chunked prefill attention: achieved HBM GB/s "
                                  "(K/V of the visible context once), query tokens/s", "value": round(cb["value"], 4),
                                  "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
                                  "ms_per_step": round(cb["seconds_per_sample"] * 1e3, 3), "higher_is_better": True,
                                  "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                                  "data": "synthetic (seeded N(0,1) bf16 K/V and q; no model weights)",
                                  "config": {"workload": "chunked prefill (oracle sample)", "parallelism": "host cores"},
                                  "cpu_baseline": {**{k: cb[k] for k in ("unit", "cores", "kind", "sample")},
                                                   "value": round(cb["value"], 4)},
                                  "e2e": {"value": round(cb["value"], 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                                          "d2h_bytes_per_step": 0}}), flush=True)
            return
        res = run_gpu_prefill(args, rank, world, local)
        if rank == 0:
            if not args.no_cpu_baseline:
                cb = prefill_oracle_sample(budget_s=10.0)
                res["cpu_baseline"] = {k: (round(v, 5) if isinstance(v, float) else v) for k, v in cb.items()}
            print(json.dumps(res), flush=True)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    if args.workload == BLOCKS:
        if rank != 0 and args.impl == "reference":
            return
        if args.impl == "reference":
            cb = blocks_oracle_sample(budget_s=max(2.0, 0.05 * (args.warmup + args.steps)))
            res = {"impl": "reference", "metric": "block export: achieved HBM GB/s (read + write bytes)",
                   "value": round(cb["value"], 4), "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
                   "warmup": args.warmup, "ms_per_step": round(cb["seconds_per_sample"] * 1e3, 3),
                   "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
                   "data": "synthetic (seeded N(0,1) bf16 K/V; no model weights)",
                   "config": {"workload": "block export (oracle sample)", "parallelism": "host cores"},
                   "cpu_baseline": {**{k: cb[k] for k in ("unit", "cores", "kind", "sample")},
                                    "value": round(cb["value"], 4)},
                   "e2e": {"value": round(cb["value"], 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}}
            print(json.dumps(res), flush=True)
            return
        res = run_gpu_blocks(args, rank, world, local)
        if rank == 0:
            if not args.no_cpu_baseline:
                cb = blocks_oracle_sample(budget_s=10.0)
                res["cpu_baseline"] = {k: (round(v, 5) if isinstance(v, float) else v) for k, v in cb.items()}
            print(json.dumps(res), flush=True)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    if args.impl == "reference":
        if rank != 0:
            return
        w = workload_for(args.workload)
        import oracle
        oracle.build()
        cores = len(os.sched_getaffinity(0))
        r = OracleRun(w, max_seqs=2)
        times = []
        for i in range(args.warmup + args.steps):
            dt = r.run()
            if i >= args.warmup:
                times.append(dt)
        t = statistics.median(times) if times else r.run()
        lens = r.lens
        nbytes = r.nbytes
        v = nbytes / t / 1e9
        cores = r.cores
        base = {"sample": r.sample_text(len(times))}
        res = {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": 1,
               "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t * 1e3, 3),
               "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
               "data": "synthetic (seeded N(0,1) bf16 K/V and q; no model weights)",
               "config": {"workload": describe(w), "global_batch": w.B, "seq_len": max(w.lens),
                          "layers": w.n_layers, "parallelism": "host cores"},
               "kv_tokens_per_s": round(sum(lens) / t, 1),
               "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                                "sample": base["sample"]},
               "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(res), flush=True)
        return

    if args.workload == MIXED:
        res, _ = run_gpu_mixed(args, rank, world, local)
        if rank == 0:
            if not args.no_cpu_baseline:
                cb = mixed_oracle_sample(budget_s=10.0)
                res["cpu_baseline"] = {k: (round(v, 5) if isinstance(v, float) else v) for k, v in cb.items()}
            print(json.dumps(res), flush=True)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    res, w = run_gpu(args, rank, world, local)
    if args.workload == DEFAULT_WORKLOAD and not args.no_extra:
        res["extra"] = run_extras(args, rank, world, local)
    if rank == 0:
        if not args.no_cpu_baseline:
            cb = oracle_sample(w, budget_s=10.0, max_seqs=w.B)
            res["cpu_baseline"] = {k: (round(v, 5) if isinstance(v, float) else v) for k, v in cb.items()}
            one = oracle_sample(w, budget_s=6.0, max_seqs=w.B, threads=1)
            res["cpu_baseline"]["single_thread"] = {
                "value": round(one["value"], 5), "unit": one["unit"], "cores": 1,
                "kv_tokens_per_s": round(one["kv_tokens_per_s"], 1), "sample": one["sample"]}
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
