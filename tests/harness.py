"""Helpers shared by the GPU parity tests: fill a GPU pool and an oracle pool with the
same seeded data, then compare.  The GPU side goes through the C ABI (via the Python
binding); the oracle side never sees a value produced by the GPU."""
from __future__ import annotations

import numpy as np

import oracle
import paged_kv_cache_split_gb300 as pkv
from paged_kv_cache_split_gb300 import workloads as wl

FMT = {wl.FMT_BF16: "bf16", wl.FMT_K4V4: "k4v4", wl.FMT_K8V4: "k8v4", wl.FMT_K8V8: "k8v8"}

ATOL, RTOL, REL_L2 = 2e-2, 1e-2, 1e-2


def to_dev_bf16(bits: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def to_dev_i32(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()


def bf16_dev_to_f64(t) -> np.ndarray:
    import torch
    return t.float().cpu().numpy().astype(np.float64)


def make_pools(w: wl.Workload, layers=None, oracle_layers=None, max_slabs=None):
    """GPU pool (all w.n_layers) and oracle pool (only `oracle_layers`, mapped 0..)."""
    rows = max(w.rows_used, 1)
    ms = max_slabs or (rows + 31) // 32 + 4
    g = pkv.Pool(w.n_layers, w.Hkv, w.D, FMT[w.fmt], hadamard_seed=w.hadamard_seed, max_slabs=ms, group_size=w.group)
    g.reserve_rows(rows)
    ol = list(range(w.n_layers)) if oracle_layers is None else list(oracle_layers)
    o = oracle.OraclePool(len(ol), w.Hkv, w.D, w.fmt, seed=w.hadamard_seed, group_size=w.group) if ol else None
    if o is not None:
        o.reserve_rows(rows)
    return g, o, ol


def fill(w: wl.Workload, g, o, oracle_layers, layers=None, seqs=None):
    """Write every sequence's K/V of `layers` into the GPU pool and (for oracle_layers)
    into the oracle pool, one write_block call per layer on each side."""
    layers = range(w.n_layers) if layers is None else layers
    seqs = range(w.B) if seqs is None else seqs
    for layer in layers:
        ks, vs, rs, ss = [], [], [], []
        for b in seqs:
            k, v = w.kv(layer, b)
            r, s = w.token_placement(b)
            ks.append(k); vs.append(v); rs.append(r); ss.append(s)
        k = np.concatenate(ks); v = np.concatenate(vs)
        r = np.concatenate(rs); s = np.concatenate(ss)
        g.write_block(layer, to_dev_i32(r), to_dev_i32(s), to_dev_bf16(k), to_dev_bf16(v))
        if o is not None and layer in oracle_layers:
            o.write_block(oracle_layers.index(layer), r, s, k, v)


def compare(got: np.ndarray, ref: np.ndarray, what: str = ""):
    """|got-ref| <= ATOL + RTOL*|ref| elementwise, and relative L2 <= REL_L2."""
    diff = np.abs(got - ref)
    bad = diff > ATOL + RTOL * np.abs(ref)
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert not bad.any(), f"{what}: {bad.sum()} elements out of tolerance, max abs {diff.max():.3e}"
    assert rel <= REL_L2, f"{what}: relative L2 error {rel:.3e}"
    return float(diff.max()), float(rel)
