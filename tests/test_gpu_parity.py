"""Parity of the CUDA path (through the C ABI) with the oracle.

Bit-exact: gather bytes (slab mapping, runs), packed codes and FP32 scale/offset
bit patterns, copy-on-write bytes.  Attention: |gpu - ref| <= 2e-2 + 1e-2 |ref|
elementwise and relative L2 <= 1e-2 against the FP64 oracle (for packed formats the
oracle attends over the same dequantised values: its codes are asserted bit-exact
first).  Sizes span several units, slabs and a ragged tail; the full-size cases use
the launch configuration the benchmark times and compare sampled sequences."""
import math

import numpy as np
import pytest

import oracle
import paged_kv_cache_split_gb300 as pkv
from paged_kv_cache_split_gb300 import workloads as wl
from tests.harness import bf16_dev_to_f64, compare, fill, make_pools, to_dev_bf16, to_dev_i32

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(autouse=True)
def _needs_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _gather_equal(w, g, o, glayer, olayer, seqs):
    bt = w.block_table()
    for b in seqs:
        L = w.lens[b]
        got = [t.cpu().numpy() for t in g.gather_visible(glayer, to_dev_i32(bt[b][: wl.nblocks(L)]), L)]
        want = o.gather_visible(olayer, bt[b][: wl.nblocks(L)], L)
        for kind, (x, y) in enumerate(zip(got, want)):
            assert np.array_equal(x, y), f"gather mismatch: seq {b} kind {kind}"


def _decode(w, g, layer, q_bits=None):
    q = to_dev_bf16(w.q(layer) if q_bits is None else q_bits)
    bt = to_dev_i32(w.block_table())
    ctx = to_dev_i32(w.ctx())
    out = g.paged_decode_attention(layer, q, bt, ctx, w.scale, max_ctx=max(w.lens))
    return bf16_dev_to_f64(out)


def _check(w, g, o, ol, layers=None, seqs=None):
    layers = ol if layers is None else layers
    seqs = list(range(w.B)) if seqs is None else seqs
    for layer in layers:
        _gather_equal(w, g, o, layer, ol.index(layer), seqs)
        got = _decode(w, g, layer)
        ref = o.decode_attention(ol.index(layer), w.q(layer), w.block_table(), w.ctx(), w.scale)
        compare(got[seqs], ref[seqs], f"{w.name} layer {layer}")
    assert g.check_errors() == 0
    assert o.inexact_rotations == 0


# ---------------------------------------------------------------------------
# Oracle-sized cases (all outputs compared)
# ---------------------------------------------------------------------------

def test_tiny():
    w = wl.tiny()
    g, o, ol = make_pools(w)
    fill(w, g, o, ol)
    _check(w, g, o, ol)


def test_qwen3_0_6b_shape_small():
    w = wl.qwen3_0_6b(n_layers=3, B=3, L=1000)
    g, o, ol = make_pools(w)
    fill(w, g, o, ol)
    _check(w, g, o, ol)


def test_qwen3_1_7b_k4v4_small():
    w = wl.qwen3_1_7b_k4v4(B=3, L=2000)
    g, o, ol = make_pools(w)
    fill(w, g, o, ol)
    _check(w, g, o, ol)


def test_qwen3_1_7b_k4v4_groups_of_64_small():
    """The five-bit K4/V4 layout (one FP32 scale/offset pair per 64 values)."""
    w = wl.qwen3_1_7b_k4v4_g64(B=3, L=2000)
    g, o, ol = make_pools(w)
    fill(w, g, o, ol)
    assert g.row_bytes == [64, 64, 16, 16]
    _check(w, g, o, ol)


@pytest.mark.parametrize("D,Hkv,G", [(128, 4, 1), (128, 8, 2), (128, 2, 8), (256, 4, 2), (256, 2, 4), (256, 8, 1)])
def test_groups_of_64_geometry_sweep(D, Hkv, G):
    """Groups of 64 at both head dims: 64- and 128-byte metadata rows, the two-warp
    split at D = 256 with 4 kv heads, ragged lengths incl. 0 and 1, several CTA counts."""
    lens = [0, 1, 33, 95, 400, 1500]
    rows, used = wl.fragmented_rows([wl.nblocks(L) for L in lens], wl.rng_for(9, D, G))
    w = wl.Workload(f"g64-{D}-{Hkv}-{G}", 1, Hkv * G, Hkv, D, wl.FMT_K4V4, lens, rows, used, 1 / math.sqrt(D),
                    0x64, 23 + D + G, group=64)
    g, o, ol = make_pools(w)
    fill(w, g, o, ol)
    _check(w, g, o, ol)
    ref = o.decode_attention(0, w.q(0), w.block_table(), w.ctx(), w.scale)
    for ctas in [3, 41, 0]:
        g.decode_set_ctas(ctas)
        a = _decode(w, g, 0)
        compare(a, ref, f"{w.name} ctas={ctas}")
        assert not a[0].any()
    assert g.check_errors() == 0


def test_groups_of_64_only_for_k4v4_at_head_dim_128_and_256():
    for fmt, D in [("k8v4", 128), ("k8v8", 256), ("k4v4", 64)]:
        with pytest.raises(pkv.PkvError) as e:
            pkv.Pool(1, 4, D, fmt, hadamard_seed=1, group_size=64)
        assert e.value.status == pkv.PKV_ERR_INVALID


@pytest.mark.parametrize("fmt", [wl.FMT_K8V4, wl.FMT_K8V8])
def test_llama_1b_small(fmt):
    w = wl.llama_1b(fmt, B=6, lo=20, hi=700)
    g, o, ol = make_pools(w)
    fill(w, g, o, ol)
    _check(w, g, o, ol)


@pytest.mark.parametrize("fmt", [wl.FMT_BF16, wl.FMT_K4V4, wl.FMT_K8V4, wl.FMT_K8V8])
@pytest.mark.parametrize("D,G", [(64, 1), (128, 8), (256, 2)])
def test_geometry_sweep(fmt, D, G):
    """Every head_dim with a spread of GQA group sizes, ragged lengths incl. 0 and 1."""
    lens = [0, 1, 33, 95, 400]
    rows, used = wl.fragmented_rows([wl.nblocks(L) for L in lens], wl.rng_for(7, D, G))
    w = wl.Workload(f"sweep-{fmt}-{D}-{G}", 1, 4 * G, 4, D, fmt, lens, rows, used, 1 / math.sqrt(D),
                    0xBEEF, 17 + D + G)
    g, o, ol = make_pools(w)
    fill(w, g, o, ol)
    _check(w, g, o, ol)
    got = _decode(w, g, 0)
    assert not got[0].any()  # empty sequence -> zeros


@pytest.mark.parametrize("fmt", [wl.FMT_K4V4, wl.FMT_K8V4, wl.FMT_K8V8])
@pytest.mark.parametrize("Hkv,G", [(2, 4), (4, 1), (4, 4)])
def test_head_dim_256_two_warps_per_kv_head(fmt, Hkv, G):
    """Packed D = 256 with 2 or 4 kv heads: each kv head's groups are split over two
    warps that exchange partial logits every 16 tokens.  Lengths with full and ragged
    units, sequences spread over many CTAs (partial records) or few (direct writes),
    and the same bits on a second run."""
    lens = [0, 1, 17, 32, 500, 2100]
    rows, used = wl.fragmented_rows([wl.nblocks(L) for L in lens], wl.rng_for(11, Hkv, G))
    w = wl.Workload(f"d256-{fmt}-{Hkv}-{G}", 1, Hkv * G, Hkv, 256, fmt, lens, rows, used, 1 / 16.0,
                    0xD256, 5 + Hkv + G)
    g, o, ol = make_pools(w)
    fill(w, g, o, ol)
    ref = o.decode_attention(0, w.q(0), w.block_table(), w.ctx(), w.scale)
    for ctas in [2, 37, 0]:
        g.decode_set_ctas(ctas)
        a = _decode(w, g, 0)
        assert np.array_equal(a, _decode(w, g, 0)), f"run-to-run difference with {ctas} CTAs"
        compare(a, ref, f"{w.name} ctas={ctas}")
        assert not a[0].any()
    assert g.check_errors() == 0
    assert o.inexact_rotations == 0


def test_split_count_invariance_and_determinism():
    w = wl.llama_1b(wl.FMT_K8V4, B=5, lo=100, hi=3000)
    g, o, ol = make_pools(w)
    fill(w, g, o, ol)
    ref = o.decode_attention(0, w.q(0), w.block_table(), w.ctx(), w.scale)
    outs = []
    for ctas in [1, 3, 7, 64, 0, 400]:
        g.decode_set_ctas(ctas)
        a = _decode(w, g, 0)
        b = _decode(w, g, 0)
        assert np.array_equal(a, b), f"run-to-run difference with {ctas} CTAs"
        compare(a, ref, f"ctas={ctas}")
        outs.append(a)
    assert g.check_errors() == 0


def test_negative_controls_fail():
    """The comparison must reject a zero output, a wrong GQA mapping and an oracle
    that reads a block one slab off (mistakes planted on the oracle side)."""
    w = wl.qwen3_0_6b(n_layers=1, B=2, L=3000)
    g, o, ol = make_pools(w)
    fill(w, g, o, ol)
    got = _decode(w, g, 0)
    ref = o.decode_attention(0, w.q(0), w.block_table(), w.ctx(), w.scale)
    compare(got, ref, "baseline")
    with pytest.raises(AssertionError):
        compare(np.zeros_like(got), ref, "zero output")
    G = w.Hq // w.Hkv
    perm = (np.arange(w.Hq) + G) % w.Hq  # query head h compared with kv head h/G + 1
    with pytest.raises(AssertionError):
        compare(got, ref[:, perm], "wrong GQA mapping")
    bt = w.block_table().copy()
    bt[0, 5] = (bt[0, 5] + 32) % w.rows_used  # one block one slab off
    bad = o.decode_attention(0, w.q(0), bt, w.ctx(), w.scale)
    with pytest.raises(AssertionError):
        compare(got, bad, "off-by-one slab")


def test_copy_on_write_bit_exact():
    w = wl.qwen3_1_7b_k4v4(B=2, L=700)
    g, o, ol = make_pools(w)
    g.reserve_rows(w.rows_used + 8)
    o.reserve_rows(w.rows_used + 8)
    fill(w, g, o, ol)
    src = np.array([w.rows[0][3], w.rows[1][0], w.rows[0][20]], np.int32)
    dst = np.array([w.rows_used, w.rows_used + 5, w.rows_used + 7], np.int32)
    g.copy_on_write_block(to_dev_i32(src), to_dev_i32(dst))
    o.copy_block(src, dst)
    for i in range(3):
        for r in (src[i], dst[i]):
            got = [t.cpu().numpy() for t in g.gather_visible(0, to_dev_i32([r]), 32)]
            want = o.gather_visible(0, np.array([r], np.int32), 32)
            assert all(np.array_equal(x, y) for x, y in zip(got, want))
    assert g.check_errors() == 0


def test_mixed_d256_steps_small():
    """Two pools (bf16, K4/V4), per-step writes with new rows/slabs and copy-on-write."""
    m = wl.MixedWorkload(B=16, Lmax=2048)
    gp, op = [], []
    for pi, P in enumerate(m.pools):
        g = pkv.Pool(1, m.Hkv, m.D, "bf16" if P.fmt == wl.FMT_BF16 else "k4v4", hadamard_seed=m.hadamard_seed,
                     max_slabs=64)
        o = oracle.OraclePool(1, m.Hkv, m.D, P.fmt, seed=m.hadamard_seed)
        g.reserve_rows(P.next_row)
        o.reserve_rows(P.next_row)
        for i in range(len(P.seqs)):
            k, v = m.initial_kv(pi, i)
            t = np.arange(P.lens[i])
            r = np.asarray(P.rows[i], np.int32)[t // 32]
            s = (t % 32).astype(np.int32)
            # prefix blocks are shared: write them once (from the first sharer)
            own = np.ones(P.lens[i], bool)
            if P.group_of[i] * m.group_size != i:
                own[: m.prefix] = False
            g.write_block(0, to_dev_i32(r[own]), to_dev_i32(s[own]), to_dev_bf16(k[own]), to_dev_bf16(v[own]))
            o.write_block(0, r[own], s[own], k[own], v[own])
        gp.append(g)
        op.append(o)
    for step in range(3):
        plan = m.plan_step()
        for pi, P in enumerate(m.pools):
            g, o, st = gp[pi], op[pi], plan[pi]
            g.reserve_rows(st["rows_needed"])
            o.reserve_rows(st["rows_needed"])
            if st["cow_src"].size:
                g.copy_on_write_block(to_dev_i32(st["cow_src"]), to_dev_i32(st["cow_dst"]))
                o.copy_block(st["cow_src"], st["cow_dst"])
            k, v = m.step_kv(step, pi)
            g.write_block(0, to_dev_i32(st["write_rows"]), to_dev_i32(st["write_slots"]), to_dev_bf16(k),
                          to_dev_bf16(v))
            o.write_block(0, st["write_rows"], st["write_slots"], k, v)
            q = m.step_q(step, pi)
            bt = m.block_table(pi)
            ctx = m.ctx(pi)
            out = g.paged_decode_attention(0, to_dev_bf16(q), to_dev_i32(bt), to_dev_i32(ctx), m.scale,
                                           max_ctx=m.Lmax + 64)
            ref = o.decode_attention(0, q, bt, ctx, m.scale)
            compare(bf16_dev_to_f64(out), ref, f"mixed step {step} pool {pi}")
            assert g.check_errors() == 0
