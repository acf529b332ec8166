"""Seeded synthetic inputs for paged decode attention.

This module is the one piece shared by the GPU path's tests/benchmark and the oracle:
it draws random bf16 data and plans which pool rows each sequence's blocks live in.
It holds none of the method's arithmetic (no slab mapping, quantisation, rotation or
attention) and imports neither the library nor the oracle.

Shapes follow the attention geometry of the models the source pages measure on
(qwen3-0.6b in mlxcel #235 "Problem"; Qwen3-1.7B and Llama-3.2-1B in mlxcel #2171
"Acceptance Criteria").  No weights or datasets exist here: every tensor is drawn
from a seeded generator with the stated distribution.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np

BLOCK = 32          # tokens per block
SLAB_BLOCKS = 32    # blocks per slab (POOL_SLAB_BLOCKS)

FMT_BF16, FMT_K4V4, FMT_K8V4, FMT_K8V8 = 0, 1, 2, 3
FMT_NAMES = {FMT_BF16: "bf16", FMT_K4V4: "k4v4", FMT_K8V4: "k8v4", FMT_K8V8: "k8v8"}

TINY_MAGNITUDE = 2.0 ** -16   # |x| below this is drawn as 0 (see bf16_normal)


def rng_for(*key: int) -> np.random.Generator:
    """Independent, platform-stable stream for a tuple of non-negative ints."""
    return np.random.default_rng(np.random.SeedSequence([int(k) & 0xFFFFFFFF for k in key]))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32)
    u = u + (((u >> 16) & 1) + 0x7FFF)
    return (u >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_normal(rng: np.random.Generator, shape, outlier_frac: float = 0.0,
                outlier_scale: float = 8.0) -> np.ndarray:
    """bf16 bit patterns of N(0,1) draws; a seeded Bernoulli(outlier_frac) subset is
    multiplied by outlier_scale.  Values with |x| < 2^-16 are drawn as exactly 0, so
    every row keeps a binary-exponent spread well under 37 (the packed formats'
    K rotation is then exact in FP64; the change to the distribution is ~1e-5)."""
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if outlier_frac > 0:
        x = np.where(rng.random(size=shape, dtype=np.float32) < outlier_frac, x * outlier_scale, x)
    x[np.abs(x) < TINY_MAGNITUDE] = 0.0
    return f32_to_bf16_bits(x)


def scale_pow2(bits: np.ndarray, e) -> np.ndarray:
    """bf16 bits times 2^e (e broadcast against bits): exact while the results stay
    normal bf16 numbers, which the magnitude plans here keep to."""
    x = bf16_bits_to_f32(bits).astype(np.float64) * np.exp2(np.asarray(e, np.float64))
    return f32_to_bf16_bits(x.astype(np.float32)).reshape(np.shape(bits))


# ---------------------------------------------------------------------------
# Row planning (which pool row holds each logical block of each sequence)
# ---------------------------------------------------------------------------

def nblocks(L: int) -> int:
    return (L + BLOCK - 1) // BLOCK


def fragmented_rows(nblk: Sequence[int], rng: np.random.Generator, n_decoys: int = 2):
    """Interleaved allocation with freed-row reuse.

    1. Blocks are handed out one per sequence per round (round robin) over the real
       sequences plus `n_decoys` decoy sequences, from fresh ascending rows, until each
       real sequence has half of its blocks (decoys take the mean half-length).
    2. The decoys finish: their rows are freed, shuffled (seeded) and pushed on a LIFO
       free list.
    3. Round robin continues over the real sequences, popping the free list first and
       then taking fresh rows.
    Returns (rows per sequence, rows used)."""
    B = len(nblk)
    half = [(n + 1) // 2 for n in nblk]
    dec = max(1, int(np.mean(nblk)) // 2) if B else 1
    seqs: List[List[int]] = [[] for _ in range(B + n_decoys)]
    want = half + [dec] * n_decoys
    nxt = 0
    while any(len(seqs[i]) < want[i] for i in range(B + n_decoys)):
        for i in range(B + n_decoys):
            if len(seqs[i]) < want[i]:
                seqs[i].append(nxt)
                nxt += 1
    free = [r for i in range(B, B + n_decoys) for r in seqs[i]]
    free = [free[i] for i in rng.permutation(len(free))]
    while any(len(seqs[i]) < nblk[i] for i in range(B)):
        for i in range(B):
            if len(seqs[i]) < nblk[i]:
                if free:
                    seqs[i].append(free.pop())
                else:
                    seqs[i].append(nxt)
                    nxt += 1
    return seqs[:B], nxt


def interleaved_monotone_rows(nblk: Sequence[int], rng: np.random.Generator, chunk: int = 16):
    """Each sequence takes fresh rows in chunks of `chunk` blocks; the order in which
    sequences take their chunks is a seeded shuffle.  Rows of one sequence therefore
    increase monotonically but are interleaved with other sequences."""
    req = [b for b in range(len(nblk)) for _ in range((nblk[b] + chunk - 1) // chunk)]
    order = [req[i] for i in rng.permutation(len(req))]
    seqs: List[List[int]] = [[] for _ in nblk]
    nxt = 0
    for b in order:
        take = min(chunk, nblk[b] - len(seqs[b]))
        seqs[b].extend(range(nxt, nxt + take))
        nxt += take
    return seqs, nxt


def block_table(rows: Sequence[Sequence[int]], max_blocks: Optional[int] = None,
                pad: int = -1) -> np.ndarray:
    mb = max_blocks if max_blocks is not None else max([len(r) for r in rows] + [1])
    bt = np.full((len(rows), mb), pad, np.int32)
    for b, r in enumerate(rows):
        bt[b, : len(r)] = r
    return bt


# ---------------------------------------------------------------------------
# Workload definitions
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class Workload:
    name: str
    n_layers: int
    Hq: int
    Hkv: int
    D: int
    fmt: int
    lens: List[int]
    rows: List[List[int]]
    rows_used: int
    scale: float
    hadamard_seed: int
    seed: int
    outlier_frac: float = 0.0
    group: int = 32  # values per affine group of the packed formats (64: the five-bit K4/V4 layout)
    # Magnitude plan (powers of two, so every value stays an exact bf16 and a row's
    # exponent spread is unchanged): q, K and V are multiplied by 2^q_exp, 2^k_exp and
    # 2^v_exp; a seeded 1/boost_every of each sequence's tokens has K multiplied by
    # 2^k_boost and V by 2^v_boost; the second half of each sequence's tokens has V
    # multiplied by 2^v_ramp.
    q_exp: int = 0
    k_exp: int = 0
    v_exp: int = 0
    boost_every: int = 64
    k_boost: int = 0
    v_boost: int = 0
    v_ramp: int = 0

    @property
    def B(self) -> int:
        return len(self.lens)

    @property
    def max_blocks(self) -> int:
        return max([len(r) for r in self.rows] + [1])

    def block_table(self) -> np.ndarray:
        return block_table(self.rows, self.max_blocks)

    def ctx(self) -> np.ndarray:
        return np.asarray(self.lens, np.int32)

    def kv(self, layer: int, b: int):
        """K and V of sequence b at `layer`: two [L_b, Hkv, D] bf16 bit arrays."""
        r = rng_for(self.seed, 1, layer, b)
        L = self.lens[b]
        shape = (L, self.Hkv, self.D)
        k = bf16_normal(r, shape, self.outlier_frac)
        v = bf16_normal(r, shape, self.outlier_frac)
        if self.k_exp or self.v_exp or self.k_boost or self.v_boost or self.v_ramp:
            ke = np.full(L, self.k_exp, np.int32)
            ve = np.full(L, self.v_exp, np.int32)
            if self.k_boost or self.v_boost:
                hit = rng_for(self.seed, 3, layer, b).integers(0, self.boost_every, size=L) == 0
                ke[hit] += self.k_boost
                ve[hit] += self.v_boost
            ve[L // 2:] += self.v_ramp
            k, v = scale_pow2(k, ke[:, None, None]), scale_pow2(v, ve[:, None, None])
        return k, v

    def q(self, layer: int) -> np.ndarray:
        """[B, Hq, D] bf16 bits."""
        q = bf16_normal(rng_for(self.seed, 2, layer), (self.B, self.Hq, self.D))
        return scale_pow2(q, self.q_exp) if self.q_exp else q

    def token_placement(self, b: int):
        """(rows, slots) of the tokens of sequence b in logical order."""
        t = np.arange(self.lens[b])
        r = np.asarray(self.rows[b], np.int32)
        return r[t // BLOCK].astype(np.int32), (t % BLOCK).astype(np.int32)


def tiny(seed: int = 0) -> Workload:
    """1 layer, one 256-token sequence (8 blocks in one slab) whose block table is a
    seeded permutation of rows 0..7; Hq 16 / Hkv 8 / D 128, native bf16."""
    perm = [int(x) for x in rng_for(seed, 10).permutation(8)]
    return Workload("tiny", 1, 16, 8, 128, FMT_BF16, [256], [perm], 8, 1 / math.sqrt(128), 0, seed)


def qwen3_0_6b(seed: int = 1, n_layers: int = 28, B: int = 8, L: int = 4096) -> Workload:
    """Qwen3-0.6B attention shape: 28 layers, Hq 16 / Hkv 8 / D 128, bf16, B x L with
    interleaved allocation and freed-row reuse (fragmented, slab-crossing)."""
    nblk = [nblocks(L)] * B
    rows, used = fragmented_rows(nblk, rng_for(seed, 11))
    return Workload("qwen3-0.6b", n_layers, 16, 8, 128, FMT_BF16, [L] * B, rows, used,
                    1 / math.sqrt(128), 0, seed)


def qwen3_1_7b_k4v4(seed: int = 2, B: int = 16, L: int = 16384) -> Workload:
    """Qwen3-1.7B attention shape in K4/V4: Hq 16 / Hkv 8 / D 128, B x L, Hadamard
    seed 0x5EED, K/V ~ N(0,1) with 1% of values x8; monotone rows, seeded interleave."""
    nblk = [nblocks(L)] * B
    rows, used = interleaved_monotone_rows(nblk, rng_for(seed, 12))
    return Workload("qwen3-1.7b-k4v4", 1, 16, 8, 128, FMT_K4V4, [L] * B, rows, used,
                    1 / math.sqrt(128), 0x5EED, seed, outlier_frac=0.01)


def qwen3_1_7b_k4v4_g64(seed: int = 2, B: int = 16, L: int = 16384) -> Workload:
    """The Qwen3-1.7B K4/V4 workload stored with groups of 64 values (one FP32 scale/offset
    pair per 64: five bits per value, the packed-formats PR's 3.2x)."""
    return dataclasses.replace(qwen3_1_7b_k4v4(seed, B, L), name="qwen3-1.7b-k4v4-g64", group=64)


def llama_1b(fmt: int = FMT_K8V4, seed: int = 3, B: int = 64, lo: int = 512, hi: int = 8192) -> Workload:
    """Llama-3.2-1B attention shape: Hq 32 / Hkv 8 / D 64, scale 1/8, B sequences with
    lengths uniform on [lo, hi] (not block aligned), fragmented block tables."""
    lens = [int(x) for x in rng_for(seed, 13).integers(lo, hi + 1, size=B)]
    rows, used = fragmented_rows([nblocks(L) for L in lens], rng_for(seed, 14))
    return Workload(f"llama-3.2-1b-{FMT_NAMES[fmt]}", 1, 32, 8, 64, fmt, lens, rows, used, 1 / 8,
                    0x1A11A, seed)


def scaled(w: Workload, name: str, **kw) -> Workload:
    return dataclasses.replace(w, name=name, **kw)


# ---------------------------------------------------------------------------
# D256 long-context mixed workload (two pools, per-step writes and copy-on-write)
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class MixedPoolPlan:
    """Host-side row plan of one pool of the mixed workload."""
    fmt: int
    seqs: List[int]                 # global sequence ids served by this pool
    rows: List[List[int]]           # per local sequence
    lens: List[int]
    refcount: dict                  # row -> number of sequences referencing it
    free: List[int]                 # LIFO free list
    next_row: int
    shared: List[tuple]             # (group, block) pairs still shared
    group_of: List[int]             # local sequence -> group id (local)
    prefix_rows: List[List[int]]    # per local group

    def take_row(self) -> int:
        if self.free:
            return self.free.pop()
        r = self.next_row
        self.next_row += 1
        return r


class MixedWorkload:
    """D256 long-context mixed workload: B=32, Hq 16 / Hkv 4 / D 256; sequences 0-15
    live in a bf16 pool and 16-31 in a K4/V4 pool.  Eight prefix groups of four
    sequences (same format) share a 1024-token prefix (32 refcounted blocks); each
    length is 1024 + U{1..Lmax-1024}.  Every step writes one token per sequence
    (taking a new row when its last block is full) and gives one sequence a private
    copy of ceil(10% of 256) = 26 still-shared (group, block) pairs, chosen by a seeded
    draw; then both pools are decoded."""

    def __init__(self, seed: int = 4, B: int = 32, Lmax: int = 32768, prefix: int = 1024,
                 group_size: int = 4, cow_frac: float = 0.10, hadamard_seed: int = 0xD256):
        self.seed, self.B, self.Lmax, self.prefix = seed, B, Lmax, prefix
        self.Hq, self.Hkv, self.D = 16, 4, 256
        self.scale = 1 / math.sqrt(256)
        self.hadamard_seed = hadamard_seed
        self.group_size = group_size
        n_groups = B // group_size
        self.n_cow = math.ceil(cow_frac * n_groups * (prefix // BLOCK))
        r = rng_for(seed, 20)
        lens = [prefix + int(x) for x in r.integers(1, Lmax - prefix + 1, size=B)]
        half = B // 2
        self.pools = []
        for p, fmt in enumerate((FMT_BF16, FMT_K4V4)):
            seqs = list(range(p * half, (p + 1) * half))
            ng = half // group_size
            pb = prefix // BLOCK
            nxt = 0
            prefix_rows = []
            for g in range(ng):
                prefix_rows.append(list(range(nxt, nxt + pb)))
                nxt += pb
            suffix = [nblocks(lens[s]) - pb for s in seqs]
            srows, used = interleaved_monotone_rows(suffix, rng_for(seed, 21, p))
            rows = []
            refc = {}
            for i, s in enumerate(seqs):
                g = i // group_size
                rws = list(prefix_rows[g]) + [nxt + x for x in srows[i]]
                rows.append(rws)
                for x in rws:
                    refc[x] = refc.get(x, 0) + 1
            nxt += used
            shared = [(g, j) for g in range(ng) for j in range(pb)]
            self.pools.append(MixedPoolPlan(fmt, seqs, rows, [lens[s] for s in seqs], refc, [], nxt,
                                            shared, [i // group_size for i in range(len(seqs))],
                                            prefix_rows))
        self.step_index = 0

    # Data ------------------------------------------------------------------
    def initial_kv(self, pool: int, i: int):
        """Initial K, V ([L, Hkv, D] bf16 bits) of local sequence i of `pool`.  The
        prefix tokens come from the group's stream so that the sharers agree."""
        P = self.pools[pool]
        g = P.group_of[i]
        rp = rng_for(self.seed, 22, pool, g)
        kp = bf16_normal(rp, (self.prefix, self.Hkv, self.D))
        vp = bf16_normal(rp, (self.prefix, self.Hkv, self.D))
        rs = rng_for(self.seed, 23, pool, i)
        n = P.lens[i] - self.prefix
        ks = bf16_normal(rs, (n, self.Hkv, self.D))
        vs = bf16_normal(rs, (n, self.Hkv, self.D))
        return np.concatenate([kp, ks]), np.concatenate([vp, vs])

    def step_kv(self, step: int, pool: int):
        """K, V of the one new token of every sequence of `pool` at `step`."""
        r = rng_for(self.seed, 24, step, pool)
        n = len(self.pools[pool].seqs)
        return (bf16_normal(r, (n, self.Hkv, self.D)), bf16_normal(r, (n, self.Hkv, self.D)))

    def step_q(self, step: int, pool: int):
        n = len(self.pools[pool].seqs)
        return bf16_normal(rng_for(self.seed, 25, step, pool), (n, self.Hq, self.D))

    # Plan ------------------------------------------------------------------
    def plan_step(self):
        """Advance the host plan by one step.  Returns, per pool, a dict with
        write_rows/write_slots (one token per sequence), cow_src/cow_dst and
        new_rows (rows that must exist in the pool before the writes)."""
        step = self.step_index
        self.step_index += 1
        out = []
        rdraw = rng_for(self.seed, 26, step)
        # choose the copy-on-write pairs over both pools' still-shared pairs
        cands = [(p, g, j) for p, P in enumerate(self.pools) for (g, j) in P.shared]
        pick = [cands[i] for i in sorted(rdraw.choice(len(cands), size=min(self.n_cow, len(cands)),
                                                      replace=False))]
        for p, P in enumerate(self.pools):
            wr, ws = [], []
            for i in range(len(P.seqs)):
                t = P.lens[i]
                if t % BLOCK == 0:
                    r = P.take_row()
                    P.rows[i].append(r)
                    P.refcount[r] = 1
                wr.append(P.rows[i][t // BLOCK])
                ws.append(t % BLOCK)
                P.lens[i] = t + 1
            cs, cd = [], []
            for (pp, g, j) in pick:
                if pp != p:
                    continue
                src = P.prefix_rows[g][j]
                sharers = [i for i in range(len(P.seqs)) if P.group_of[i] == g and P.rows[i][j] == src]
                i = sharers[int(rdraw.integers(len(sharers)))]
                dst = P.take_row()
                P.rows[i][j] = dst
                P.refcount[dst] = 1
                P.refcount[src] -= 1
                cs.append(src)
                cd.append(dst)
                if P.refcount[src] < 2:
                    P.shared.remove((g, j))
            out.append(dict(write_rows=np.asarray(wr, np.int32), write_slots=np.asarray(ws, np.int32),
                            cow_src=np.asarray(cs, np.int32), cow_dst=np.asarray(cd, np.int32),
                            rows_needed=P.next_row))
        return out

    def block_table(self, pool: int, max_blocks: Optional[int] = None) -> np.ndarray:
        P = self.pools[pool]
        mb = max_blocks if max_blocks is not None else nblocks(self.Lmax + 64)
        return block_table(P.rows, mb)

    def ctx(self, pool: int) -> np.ndarray:
        return np.asarray(self.pools[pool].lens, np.int32)
