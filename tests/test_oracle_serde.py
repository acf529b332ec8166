"""Pins of the oracle's block records (export / import), CPU only.

The record layout is fixed by the serde touch point of the chunked-slab issue
(a block's content is read and written within the slab that holds its row) and
the packed-formats PR's Summary (a full checkpoint keeps the packed bytes as they
are): a record is every stored byte of one block,
layer-major, then K, V, K meta, V meta.  The pins tie the oracle's export to its
already-pinned per-block reads and gathers, and check the size by closed form.
"""
import numpy as np
import pytest

from oracle import FMT_BF16, FMT_K4V4, FMT_K8V4, FMT_K8V8, OraclePool
from paged_kv_cache_split_gb300 import workloads as wl

BITS = {FMT_BF16: (16, 16), FMT_K4V4: (4, 4), FMT_K8V4: (8, 4), FMT_K8V8: (8, 8)}


def _filled(fmt, n_layers, hkv, D, rows, seed):
    p = OraclePool(n_layers, hkv, D, fmt, seed=0x5EED)
    p.reserve_rows(int(max(rows)) + 1)
    rng = wl.rng_for(seed)
    toks_rows = np.repeat(np.asarray(rows, np.int32), 32)
    toks_slots = np.tile(np.arange(32, dtype=np.int32), len(rows))
    for layer in range(n_layers):
        n = toks_rows.size
        p.write_block(layer, toks_rows, toks_slots, wl.bf16_normal(rng, (n, hkv, D)), wl.bf16_normal(rng, (n, hkv, D)))
    return p


@pytest.mark.parametrize("fmt", [FMT_BF16, FMT_K4V4, FMT_K8V4, FMT_K8V8])
@pytest.mark.parametrize("D", [64, 256])
def test_record_size_closed_form(fmt, D):
    kb, vb = BITS[fmt]
    per_token_head = D * kb // 8 + D * vb // 8 + (0 if fmt == FMT_BF16 else 2 * (D // 32) * 8)
    p = OraclePool(3, 4, D, fmt, seed=1)
    assert p.record_bytes == 3 * 32 * 4 * per_token_head


@pytest.mark.parametrize("fmt", [FMT_BF16, FMT_K4V4, FMT_K8V4, FMT_K8V8])
def test_record_is_blocks_in_layer_then_kind_order(fmt):
    rows = [37, 2, 64, 5]  # slab-crossing, not sorted
    p = _filled(fmt, 2, 2, 64, rows, seed=21)
    rec = p.export_blocks(rows)
    kinds = 2 if fmt == FMT_BF16 else 4
    for i, r in enumerate(rows):
        parts = [p.read_block(layer, k, r) for layer in range(2) for k in range(kinds)]
        assert np.array_equal(rec[i], np.concatenate(parts))


@pytest.mark.parametrize("fmt", [FMT_BF16, FMT_K4V4, FMT_K8V4, FMT_K8V8])
def test_restore_into_other_rows_gives_same_context(fmt):
    src_rows = [3, 40, 9, 70]
    a = _filled(fmt, 2, 2, 64, src_rows, seed=22)
    rec = a.export_blocks(src_rows)
    # a second pool with unrelated contents; the records go to other rows
    dst_rows = [100, 7, 55, 31]
    b = _filled(fmt, 2, 2, 64, [7, 8, 31, 55, 100], seed=23)
    untouched = b.read_block(1, 0, 8).copy()
    b.import_blocks(dst_rows, rec)
    assert np.array_equal(b.export_blocks(dst_rows), rec)
    assert np.array_equal(b.read_block(1, 0, 8), untouched)
    L = 4 * 32 - 5  # ragged tail
    for layer in range(2):
        ga = a.gather_visible(layer, src_rows, L)
        gb = b.gather_visible(layer, dst_rows, L)
        for x, y in zip(ga, gb):
            assert np.array_equal(x, y)
    rng = wl.rng_for(24)
    q = wl.bf16_normal(rng, (1, 4, 64))
    oa = a.decode_attention(1, q, np.asarray([src_rows], np.int32), [L], 0.125)
    ob = b.decode_attention(1, q, np.asarray([dst_rows], np.int32), [L], 0.125)
    assert np.array_equal(oa, ob)


def test_export_rejects_rows_outside_the_pool():
    p = _filled(FMT_K8V4, 1, 2, 64, [0, 1], seed=25)
    with pytest.raises(Exception):
        p.export_blocks([0, 10_000])
