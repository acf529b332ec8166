"""Causal chunked-prefill attention of the CUDA path (through the C ABI) against the
oracle: every format, chunk sizes 1 to 16 with ragged contexts that start chunks
mid-block and on block boundaries, and the device error for a sequence shorter than
its chunk.  Tolerance as for decode: |gpu - ref| <= 2e-2 + 1e-2 |ref| elementwise and
relative L2 <= 1e-2 against the FP64 oracle."""
import math

import numpy as np
import pytest

import paged_kv_cache_split_gb300 as pkv
from paged_kv_cache_split_gb300 import workloads as wl
from tests.harness import bf16_dev_to_f64, compare, fill, make_pools, to_dev_bf16, to_dev_i32

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(autouse=True)
def _needs_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _case(fmt, D, Hkv, G, lens, seed, group=32):
    rows, used = wl.fragmented_rows([wl.nblocks(L) for L in lens], wl.rng_for(seed, D, G))
    return wl.Workload(f"prefill-{fmt}-{D}-{G}", 1, Hkv * G, Hkv, D, fmt, lens, rows, used, 1 / math.sqrt(D),
                       0xF1, seed, group=group)


@pytest.mark.parametrize("fmt,D,group", [(wl.FMT_BF16, 128, 32), (wl.FMT_K4V4, 128, 32), (wl.FMT_K8V4, 64, 32),
                                         (wl.FMT_K8V8, 256, 32), (wl.FMT_K4V4, 256, 64)])
@pytest.mark.parametrize("n_q", [1, 5, 16])
def test_prefill_matches_oracle(fmt, D, group, n_q):
    lens = [16, 31, 64, 300, 1025]
    w = _case(fmt, D, 4, 2, lens, 61 + n_q, group)
    g, o, ol = make_pools(w)
    fill(w, g, o, ol)
    q = wl.bf16_normal(wl.rng_for(62, n_q), (w.B, n_q, w.Hq, D))
    bt = w.block_table()
    out = g.paged_prefill_attention(0, to_dev_bf16(q), to_dev_i32(bt), to_dev_i32(w.ctx()), w.scale, max_ctx=max(lens))
    ref = o.prefill_attention(0, q, bt, w.ctx(), w.scale)
    got = bf16_dev_to_f64(out)
    compare(got.reshape(-1, D), ref.reshape(-1, D), f"prefill {w.name} n_q={n_q}")
    assert g.check_errors() == 0


def test_prefill_rows_of_a_too_short_sequence_are_zero_and_flagged():
    lens = [40, 3]
    w = _case(wl.FMT_BF16, 64, 2, 2, lens, 71)
    g, o, ol = make_pools(w)
    fill(w, g, o, ol)
    q = wl.bf16_normal(wl.rng_for(72), (2, 4, w.Hq, 64))
    out = g.paged_prefill_attention(0, to_dev_bf16(q), to_dev_i32(w.block_table()), to_dev_i32(w.ctx()), w.scale)
    got = bf16_dev_to_f64(out)
    assert not got[1].any()
    assert g.check_errors() & pkv.ERR_CTX
    ref = o.prefill_attention(0, q[:1], w.block_table()[:1], w.ctx()[:1], w.scale)
    compare(got[:1].reshape(-1, 64), ref.reshape(-1, 64), "prefill, valid sequence beside a short one")


def test_prefill_rejects_too_many_queries():
    w = _case(wl.FMT_BF16, 64, 2, 1, [64], 81)
    g, _, _ = make_pools(w, oracle_layers=[])
    with pytest.raises(pkv.PkvError) as e:
        g.prefill_workspace_bytes(1, 4097, 2, 2)
    assert e.value.status == pkv.PKV_ERR_INVALID


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("G,n_q", [(1, 8), (2, 4), (4, 2), (2, 8), (1, 16), (4, 4), (8, 2)])
def test_prefill_several_queries_per_tile_bf16(D, G, n_q):
    """bf16 chunks served several queries per tile (up to 16 rows of (query, head)
    pairs at head dims 64/128, 8 at 256; several tiles per chunk when n_q is larger),
    with CTA counts that start split-K segments inside the chunk, so some rows see no
    token of their segment."""
    lens = [n_q, n_q + 1, 33, 47, 64, 500, 1031]
    w = _case(wl.FMT_BF16, D, 2, G, lens, 91 + G + n_q)
    g, o, ol = make_pools(w)
    fill(w, g, o, ol)
    q = wl.bf16_normal(wl.rng_for(92, n_q), (w.B, n_q, w.Hq, D))
    bt = w.block_table()
    ref = o.prefill_attention(0, q, bt, w.ctx(), w.scale)
    for ctas in [5, 97, 0]:
        g.decode_set_ctas(ctas)
        out = g.paged_prefill_attention(0, to_dev_bf16(q), to_dev_i32(bt), to_dev_i32(w.ctx()), w.scale)
        got = bf16_dev_to_f64(out)
        assert np.isfinite(got).all()
        compare(got.reshape(-1, D), ref.reshape(-1, D), f"prefill {w.name} n_q={n_q} ctas={ctas}")
    assert g.check_errors() == 0


@pytest.mark.parametrize("fmt,D,group", [(wl.FMT_K4V4, 128, 32), (wl.FMT_K8V4, 64, 32), (wl.FMT_K8V8, 128, 32),
                                         (wl.FMT_K4V4, 256, 64), (wl.FMT_K4V4, 128, 64)])
@pytest.mark.parametrize("hkv", [2, 4])
@pytest.mark.parametrize("G,n_q", [(1, 8), (2, 8), (4, 2), (1, 16), (4, 4), (8, 2)])
def test_prefill_several_queries_per_tile_packed(fmt, D, group, hkv, G, n_q):
    """Packed chunks served several queries per tile: 16 rows of (query, head) pairs
    when 16 / G queries divide the chunk (head dims up to 128; rows 8..15 with their
    own softmax state), else 8 rows; with CTA counts that start split-K segments
    inside the chunk.  Four kv heads give 128-byte rows at head_dim 128 (the
    register-split variant); two give narrower boxes at 64 (the plain variant)."""
    lens = [n_q, n_q + 1, 33, 64, 500, 1031]
    w = _case(fmt, D, hkv, G, lens, 101 + G + n_q + hkv, group)
    g, o, ol = make_pools(w)
    fill(w, g, o, ol)
    q = wl.bf16_normal(wl.rng_for(102, n_q, hkv), (w.B, n_q, w.Hq, D))
    bt = w.block_table()
    ref = o.prefill_attention(0, q, bt, w.ctx(), w.scale)
    for ctas in [5, 97, 0]:
        g.decode_set_ctas(ctas)
        out = g.paged_prefill_attention(0, to_dev_bf16(q), to_dev_i32(bt), to_dev_i32(w.ctx()), w.scale)
        got = bf16_dev_to_f64(out)
        assert np.isfinite(got).all()
        compare(got.reshape(-1, D), ref.reshape(-1, D), f"prefill {w.name} hkv={hkv} n_q={n_q} ctas={ctas}")
    assert g.check_errors() == 0
