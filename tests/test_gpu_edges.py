"""Degenerate and extreme cases of the CUDA path, through the C ABI: an empty batch, a
batch of empty sequences, one-token contexts (softmax over one token returns that
token's V: bit-exact in bf16), and one 64k-token sequence whose split-K parts span
every CTA.  Tolerance as in the parity tests."""
import math

import numpy as np
import pytest

import paged_kv_cache_split_gb300 as pkv
from paged_kv_cache_split_gb300 import workloads as wl
from tests.harness import FMT, bf16_dev_to_f64, compare, fill, make_pools, to_dev_bf16, to_dev_i32

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

FORMATS = [wl.FMT_BF16, wl.FMT_K4V4, wl.FMT_K8V4, wl.FMT_K8V8]


@pytest.fixture(autouse=True)
def _needs_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _case(fmt, D, Hkv, G, lens, seed):
    rows, used = wl.fragmented_rows([wl.nblocks(L) for L in lens], wl.rng_for(seed, D, G))
    return wl.Workload(f"edge-{fmt}-{D}-{G}", 1, Hkv * G, Hkv, D, fmt, lens, rows, used, 1 / math.sqrt(D),
                       0xE06E, seed)


@pytest.mark.parametrize("fmt", FORMATS)
def test_empty_batch_is_a_no_op(fmt):
    p = pkv.Pool(1, 2, 128, FMT[fmt], hadamard_seed=1, max_slabs=4)
    p.append_slab(1)
    q = torch.empty((0, 8, 128), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((0, 1), dtype=torch.int32, device="cuda")
    ctx = torch.zeros((0,), dtype=torch.int32, device="cuda")
    assert p.paged_decode_attention(0, q, bt, ctx, 0.1).shape == (0, 8, 128)
    assert p.paged_prefill_attention(0, q.view(0, 1, 8, 128), bt, ctx, 0.1).shape == (0, 1, 8, 128)
    torch.cuda.synchronize()
    assert p.check_errors() == 0


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("D,G", [(64, 1), (128, 8), (256, 2)])
def test_batch_of_empty_sequences_writes_zeros(fmt, D, G):
    p = pkv.Pool(1, 4, D, FMT[fmt], hadamard_seed=2, max_slabs=4)
    p.append_slab(1)
    q = to_dev_bf16(wl.bf16_normal(wl.rng_for(3, D), (5, 4 * G, D)))
    bt = torch.zeros((5, 1), dtype=torch.int32, device="cuda")
    ctx = torch.zeros((5,), dtype=torch.int32, device="cuda")
    for ctas in [1, 0]:
        p.decode_set_ctas(ctas)
        out = torch.full((5, 4 * G, D), 7.0, dtype=torch.bfloat16, device="cuda")
        p.paged_decode_attention(0, q, bt, ctx, 0.1, out=out)
        assert not out.float().cpu().numpy().any()
    assert p.check_errors() == 0


@pytest.mark.parametrize("fmt", FORMATS)
def test_one_token_contexts_return_that_token(fmt):
    lens = [1, 1, 1, 33]
    w = _case(fmt, 128, 2, 4, lens, 5)
    g, o, ol = make_pools(w)
    fill(w, g, o, ol)
    out = g.paged_decode_attention(0, to_dev_bf16(w.q(0)), to_dev_i32(w.block_table()), to_dev_i32(w.ctx()),
                                   w.scale)
    got = bf16_dev_to_f64(out)
    ref = o.decode_attention(0, w.q(0), w.block_table(), w.ctx(), w.scale)
    compare(got, ref, f"{w.name} one-token contexts")
    if fmt == wl.FMT_BF16:
        bits = out.view(torch.int16).cpu().numpy().view(np.uint16)
        for b in range(3):
            v = w.kv(0, b)[1]  # [1, Hkv, D] bf16 bits
            for h in range(w.Hq):
                assert np.array_equal(bits[b, h], v[0, h // 4]), f"seq {b} head {h}"
    assert g.check_errors() == 0


@pytest.mark.parametrize("fmt", [wl.FMT_BF16, wl.FMT_K4V4])
def test_one_long_sequence_spans_every_cta(fmt):
    lens = [65536 + 17]
    w = _case(fmt, 128, 2, 4, lens, 9)
    g, o, ol = make_pools(w)
    fill(w, g, o, ol)
    ref = o.decode_attention(0, w.q(0), w.block_table(), w.ctx(), w.scale)
    for ctas in [0, 7]:
        g.decode_set_ctas(ctas)
        got = bf16_dev_to_f64(g.paged_decode_attention(0, to_dev_bf16(w.q(0)), to_dev_i32(w.block_table()),
                                                       to_dev_i32(w.ctx()), w.scale, max_ctx=lens[0]))
        compare(got, ref, f"{w.name} L={lens[0]} ctas={ctas}")
    assert g.check_errors() == 0


@pytest.mark.parametrize("fmt,D,G", [(wl.FMT_BF16, 128, 2), (wl.FMT_K4V4, 128, 2), (wl.FMT_K8V4, 64, 4),
                                     (wl.FMT_K8V8, 256, 2)])
def test_many_short_and_empty_sequences_over_the_cost_split(fmt, D, G):
    """Eighty sequences of 0 to 70 tokens (a quarter empty, many of one unit or less):
    the CTA split weighs every sequence start, so a CTA holds many segments, several
    CTAs hold none, and with few units the positions per CTA are clamped to one unit's
    step.  Parity with the oracle and bit-identical repeats at 1, 5, 37 CTAs, the
    default grid and 400 CTAs."""
    rng = np.random.default_rng(4242)
    lens = [int(x) if rng.random() > 0.25 else 0 for x in rng.integers(1, 71, size=80)]
    w = _case(fmt, D, 4, G, lens, 97 + D + G)
    g, o, ol = make_pools(w)
    fill(w, g, o, ol)
    ref = o.decode_attention(0, w.q(0), w.block_table(), w.ctx(), w.scale)
    q, bt, ctx = to_dev_bf16(w.q(0)), to_dev_i32(w.block_table()), to_dev_i32(w.ctx())
    for ctas in [1, 5, 37, 0, 400]:
        g.decode_set_ctas(ctas)
        a = bf16_dev_to_f64(g.paged_decode_attention(0, q, bt, ctx, w.scale, max_ctx=max(lens)))
        b = bf16_dev_to_f64(g.paged_decode_attention(0, q, bt, ctx, w.scale, max_ctx=max(lens)))
        assert np.array_equal(a, b), f"run-to-run difference with {ctas} CTAs"
        assert not a[np.asarray(lens) == 0].any(), "empty sequences must give zero rows"
        compare(a, ref, f"ctas={ctas}")
    assert g.check_errors() == 0
