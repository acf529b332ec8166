"""The seeded input generators (CPU only): each named workload has the shapes, sizes
and value distributions of the configuration it stands for; row plans are valid
(every block a distinct row, fragmented or monotone as stated, slab-crossing); bf16
rounding is nearest-even by its definition; streams are deterministic per key."""
import math

import numpy as np
import pytest

from paged_kv_cache_split_gb300 import workloads as wl


def _valid_plan(rows, used, nblk):
    flat = [r for seq in rows for r in seq]
    assert [len(seq) for seq in rows] == list(nblk)
    assert len(set(flat)) == len(flat), "a row is given to two blocks"
    assert all(0 <= r < used for r in flat)


@pytest.mark.parametrize("seed", [0, 1, 7])
def test_fragmented_rows_reuse_freed_rows_and_cross_slabs(seed):
    nblk = [128] * 8
    rows, used = wl.fragmented_rows(nblk, wl.rng_for(seed))
    _valid_plan(rows, used, nblk)
    # decoys' rows are reused: fewer fresh rows than real blocks plus the decoys' share
    assert used < sum(nblk) + 2 * 64
    assert any(any(b < a for a, b in zip(seq, seq[1:])) for seq in rows), "no freed-row reuse"
    assert all(len({r // 32 for r in seq}) > 4 for seq in rows), "rows should interleave over slabs"


def test_interleaved_monotone_rows():
    nblk = [512] * 16
    rows, used = wl.interleaved_monotone_rows(nblk, wl.rng_for(5))
    _valid_plan(rows, used, nblk)
    assert used == sum(nblk)
    assert all(all(b > a for a, b in zip(seq, seq[1:])) for seq in rows)
    assert any(seq[16] != seq[15] + 1 for seq in rows), "sequences should interleave by chunks"


def test_block_table_pads_with_minus_one():
    bt = wl.block_table([[3, 4], [9]], 3)
    assert bt.dtype == np.int32 and bt.tolist() == [[3, 4, -1], [9, -1, -1]]


def test_bf16_rounding_is_nearest_even():
    rng = np.random.default_rng(11)
    x = rng.standard_normal(20000).astype(np.float32) * np.float32(3.0)
    # exact halfway values (upper halves below 0x7F00: finite, both signs via the negation below)
    ties = (rng.integers(0, 0x7F00, 64).astype(np.uint32) << 16) | np.uint32(0x8000)
    ties = np.concatenate([ties.view(np.float32), -ties.view(np.float32)])
    x = np.concatenate([x, ties, np.float32([0.0, -0.0, 1.0, -2.5])])
    got = wl.bf16_bits_to_f32(wl.f32_to_bf16_bits(x)).astype(np.float64)
    u = x.view(np.uint32)
    lo = (u & np.uint32(0xFFFF0000)).view(np.float32).astype(np.float64)
    hi = ((u & np.uint32(0xFFFF0000)) + np.uint32(0x10000)).view(np.float32).astype(np.float64)
    xd = x.astype(np.float64)
    dlo, dhi = np.abs(xd - lo), np.abs(hi - xd)
    even_lo = ((u >> 16) & 1) == 0
    want = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(even_lo, lo, hi)))
    assert np.array_equal(got, want)


def test_streams_are_deterministic_per_key():
    a = wl.bf16_normal(wl.rng_for(1, 2, 3), (64, 8))
    assert np.array_equal(a, wl.bf16_normal(wl.rng_for(1, 2, 3), (64, 8)))
    assert not np.array_equal(a, wl.bf16_normal(wl.rng_for(1, 2, 4), (64, 8)))


def test_bf16_normal_distribution_and_outliers():
    x = wl.bf16_bits_to_f32(wl.bf16_normal(wl.rng_for(9), (400000,))).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01
    y = wl.bf16_bits_to_f32(wl.bf16_normal(wl.rng_for(9), (400000,), outlier_frac=0.01)).astype(np.float64)
    frac_big = np.mean(np.abs(y) > 6.0)  # |N(0,1)| > 6 is ~2e-9; outliers x8 exceed it ~55% of the time
    assert 0.004 < frac_big < 0.007


def test_named_workloads_have_their_configured_shapes():
    t = wl.tiny()
    assert (t.n_layers, t.Hq, t.Hkv, t.D, t.fmt, t.lens) == (1, 16, 8, 128, wl.FMT_BF16, [256])
    assert sorted(t.rows[0]) == list(range(8)) and t.scale == 1 / math.sqrt(128)
    q = wl.qwen3_0_6b()
    assert (q.n_layers, q.Hq, q.Hkv, q.D, q.fmt, q.lens) == (28, 16, 8, 128, wl.FMT_BF16, [4096] * 8)
    k = wl.qwen3_1_7b_k4v4()
    assert (k.Hq, k.Hkv, k.D, k.fmt, k.lens, k.outlier_frac, k.group) == \
        (16, 8, 128, wl.FMT_K4V4, [16384] * 16, 0.01, 32)
    assert wl.qwen3_1_7b_k4v4_g64().group == 64
    for fmt in (wl.FMT_K8V4, wl.FMT_K8V8):
        m = wl.llama_1b(fmt)
        assert (m.Hq, m.Hkv, m.D, m.fmt, m.B, m.scale) == (32, 8, 64, fmt, 64, 1 / 8)
        assert all(512 <= L <= 8192 for L in m.lens) and len(set(m.lens)) > 32
        assert any(L % 32 for L in m.lens), "lengths should not all be block aligned"
    for w in (q, k, wl.llama_1b()):
        _valid_plan(w.rows, w.rows_used, [wl.nblocks(L) for L in w.lens])


def test_mixed_workload_plan():
    m = wl.MixedWorkload()
    assert (m.B, m.Hq, m.Hkv, m.D, m.Lmax) == (32, 16, 4, 256, 32768)
    assert [P.fmt for P in m.pools] == [wl.FMT_BF16, wl.FMT_K4V4]
    assert m.n_cow == math.ceil(0.10 * 8 * 32)
    for P in m.pools:
        assert len(P.seqs) == 16 and all(1024 < L <= 32768 for L in P.lens)
        for i, seq in enumerate(P.rows):
            assert len(seq) == wl.nblocks(P.lens[i])
            assert seq[:32] == P.prefix_rows[P.group_of[i]]  # the group's shared 1024-token prefix
        for r, c in P.refcount.items():
            assert c == (4 if r < 4 * 32 else 1)
