"""Parity at the benchmark's full sizes, in the launch configuration it times.

Each case builds the full pool (every sequence, every layer, the full context
lengths, the same block tables) and decodes every sequence with the same calls the
benchmark makes; the oracle then recomputes a sample of sequences (and layers) one
by one.  In the compared layers every sequence holds its seeded data (so every CTA
of the launch streams real packed groups, not zeros); the oracle is given only the
sample.  Layers that are not compared hold device-generated N(0,1) data.  The sample
spreads over the CTA range (first, last, shortest, longest and sequences between,
whose segments start and end inside CTAs).  Bit-exact checks (gather bytes, codes,
scale/offset bit patterns) run on the sample too."""
import numpy as np
import pytest

import oracle
import paged_kv_cache_split_gb300 as pkv
from paged_kv_cache_split_gb300 import workloads as wl
from tests.harness import FMT, bf16_dev_to_f64, compare, to_dev_bf16, to_dev_i32

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
torch = pytest.importorskip("torch")


@pytest.fixture(autouse=True)
def _needs_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _write_seqs(w, g, o, layer, olayer, seqs):
    ks, vs, rs, ss = [], [], [], []
    for b in seqs:
        k, v = w.kv(layer, b)
        r, s = w.token_placement(b)
        ks.append(k); vs.append(v); rs.append(r); ss.append(s)
    k, v = np.concatenate(ks), np.concatenate(vs)
    r, s = np.concatenate(rs), np.concatenate(ss)
    g.write_block(layer, to_dev_i32(r), to_dev_i32(s), to_dev_bf16(k), to_dev_bf16(v))
    if o is not None:
        o.write_block(olayer, r, s, k, v)


def _gather_equal(w, g, o, layer, olayer, seqs):
    bt = w.block_table()
    for b in seqs:
        L = w.lens[b]
        nb = wl.nblocks(L)
        got = [t.cpu().numpy() for t in g.gather_visible(layer, to_dev_i32(bt[b][:nb]), L)]
        want = o.gather_visible(olayer, bt[b][:nb], L)
        for kind, (x, y) in enumerate(zip(got, want)):
            assert np.array_equal(x, y), f"{w.name}: gather mismatch, seq {b} kind {kind}"


def _device_fill(w, g, layer):
    """Device-generated N(0,1) bf16 K/V for every sequence of `layer`."""
    gen = torch.Generator(device="cuda")
    gen.manual_seed(7000 + layer)
    r = np.concatenate([w.token_placement(b)[0] for b in range(w.B)])
    s = np.concatenate([w.token_placement(b)[1] for b in range(w.B)])
    k = torch.randn((r.size, w.Hkv, w.D), generator=gen, device="cuda").to(torch.bfloat16)
    v = torch.randn((r.size, w.Hkv, w.D), generator=gen, device="cuda").to(torch.bfloat16)
    g.write_block(layer, to_dev_i32(r), to_dev_i32(s), k, v)


def _full_case(w, sample, layers):
    """Full pool of `w`: seeded host data for every sequence of `layers` (the oracle
    gets `sample`), device data elsewhere; all layers decoded with one shared
    workspace in layer order (the benchmark's step); sample compared."""
    g = pkv.Pool(w.n_layers, w.Hkv, w.D, FMT[w.fmt], hadamard_seed=w.hadamard_seed,
                 max_slabs=(w.rows_used + 31) // 32 + 8, group_size=w.group)
    g.reserve_rows(w.rows_used)
    o = oracle.OraclePool(len(layers), w.Hkv, w.D, w.fmt, seed=w.hadamard_seed, group_size=w.group)
    o.reserve_rows(w.rows_used)
    rest = [b for b in range(w.B) if b not in sample]
    for layer in range(w.n_layers):
        if layer in layers:
            i = layers.index(layer)
            _write_seqs(w, g, o, layer, i, sample)
            for c in range(0, len(rest), 4):
                _write_seqs(w, g, None, layer, i, rest[c:c + 4])
        else:
            _device_fill(w, g, layer)
    torch.cuda.synchronize()
    dev = torch.device("cuda")
    bt = to_dev_i32(w.block_table())
    ctx = to_dev_i32(w.ctx())
    q = torch.stack([to_dev_bf16(w.q(layer)) for layer in range(w.n_layers)])
    out = torch.empty_like(q)
    ws = g.workspace(w.B, w.Hq, dev)
    for layer in range(w.n_layers):
        g.paged_decode_attention(layer, q[layer], bt, ctx, w.scale, max_ctx=max(w.lens), out=out[layer],
                                 workspace=ws)
    torch.cuda.synchronize()
    assert g.check_errors() == 0
    sel = np.asarray(sample)
    for i, layer in enumerate(layers):
        _gather_equal(w, g, o, layer, i, sample)
        ref = o.decode_attention(i, w.q(layer)[sel], w.block_table()[sel], w.ctx()[sel], w.scale)
        got = bf16_dev_to_f64(out[layer])[sel]
        compare(got, ref, f"{w.name} layer {layer} sample {sample}")
    assert o.inexact_rotations == 0


def test_qwen3_0_6b_full_size():
    """28 layers, 8 x 4096, fragmented slab-crossing rows: every sequence of the first
    and last layers compared."""
    w = wl.qwen3_0_6b()
    _full_case(w, sample=list(range(w.B)), layers=[0, w.n_layers - 1])


def test_qwen3_1_7b_k4v4_full_size_sampled():
    """16 x 16384 K4/V4 with outliers, every sequence holding data: eight sequences
    spread over the launch compared (each spans about nine CTAs)."""
    w = wl.qwen3_1_7b_k4v4()
    _full_case(w, sample=[0, 2, 5, 7, 9, 11, 13, w.B - 1], layers=[0])


def test_qwen3_1_7b_k4v4_groups_of_64_full_size_sampled():
    """16 x 16384 in the five-bit K4/V4 layout: eight sequences compared."""
    w = wl.qwen3_1_7b_k4v4_g64()
    _full_case(w, sample=[0, 3, 4, 6, 8, 10, 12, w.B - 1], layers=[0])


def _spread_sample(lens, n=8):
    """First, last, shortest and longest sequence, plus others evenly spaced."""
    lens = np.asarray(lens)
    pick = {0, len(lens) - 1, int(lens.argmin()), int(lens.argmax())}
    for x in np.linspace(0, len(lens) - 1, n + 2)[1:-1]:
        if len(pick) >= n:
            break
        pick.add(int(round(x)))
    return sorted(pick)


@pytest.mark.parametrize("fmt", [wl.FMT_K8V4, wl.FMT_K8V8])
def test_llama_1b_full_size_sampled(fmt):
    """64 ragged sequences in [512, 8192], every one holding data: the shortest, the
    longest, the first, the last and four between compared."""
    w = wl.llama_1b(fmt)
    sample = _spread_sample(w.lens)
    assert len(sample) >= 8
    _full_case(w, sample=sample, layers=[0])


def test_mixed_d256_full_size_sampled():
    """B=32 up to 32768 tokens, two pools, every sequence holding data; three steps of
    per-sequence writes and copy-on-write; per pool a group leader and a sharer
    compared after each step."""
    m = wl.MixedWorkload()
    gp, op, samples = [], [], []
    for pi, P in enumerate(m.pools):
        # capacity for the three steps' new rows
        g = pkv.Pool(1, m.Hkv, m.D, "bf16" if P.fmt == wl.FMT_BF16 else "k4v4", hadamard_seed=m.hadamard_seed,
                     max_slabs=(P.next_row + 3 * 64 + 31) // 32 + 8)
        o = oracle.OraclePool(1, m.Hkv, m.D, P.fmt, seed=m.hadamard_seed)
        g.reserve_rows(P.next_row)
        o.reserve_rows(P.next_row)
        sample = [0, 3 * m.group_size + 1]
        # Every sequence's tokens go to the GPU pool: each group's leader writes the
        # shared prefix and its own suffix, the other members their suffixes.  The
        # oracle gets every group's prefix and the sample's suffixes.
        for i in range(len(P.seqs)):
            lead = i % m.group_size == 0
            k, v = m.initial_kv(pi, i)
            t = np.arange(0 if lead else m.prefix, P.lens[i])
            r = np.asarray(P.rows[i], np.int32)[t // 32]
            s = (t % 32).astype(np.int32)
            kk, vv = k[t], v[t]
            g.write_block(0, to_dev_i32(r), to_dev_i32(s), to_dev_bf16(kk), to_dev_bf16(vv))
            if i in sample:
                o.write_block(0, r, s, kk, vv)
            elif lead:
                n = m.prefix
                o.write_block(0, r[:n], s[:n], kk[:n], vv[:n])
        gp.append(g)
        op.append(o)
        samples.append(sample)
    dev = torch.device("cuda")
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
            ws = g.workspace(len(P.seqs), m.Hq, dev)
            out = g.paged_decode_attention(0, to_dev_bf16(q), to_dev_i32(bt), to_dev_i32(ctx), m.scale,
                                           max_ctx=m.Lmax + 64, workspace=ws)
            sel = np.asarray(samples[pi])
            ref = o.decode_attention(0, q[sel], bt[sel], ctx[sel], m.scale)
            compare(bf16_dev_to_f64(out)[sel], ref, f"mixed full step {step} pool {pi}")
            for b in sel:
                L = int(ctx[b])
                nb = wl.nblocks(L)
                got = [t.cpu().numpy() for t in g.gather_visible(0, to_dev_i32(bt[b][:nb]), L)]
                want = o.gather_visible(0, bt[b][:nb], L)
                assert all(np.array_equal(x, y) for x, y in zip(got, want)), f"mixed gather pool {pi} seq {b}"
            assert g.check_errors() == 0
    assert all(o.inexact_rotations == 0 for o in op)
