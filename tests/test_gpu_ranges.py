"""Dynamic range of the decode kernels, and stale bytes past the context.

Range: q, K and V are multiplied (each on its own) by powers of two from 2^-20 to
2^16, by token-level boosts (a seeded 1/64 of the tokens with K or V times 2^8 or
2^12 beside ordinary ones) and by a ramp (V of a sequence's second half 2^16 times
its first half, and the reverse).  The packed formats carry FP32 scales and offsets
(mlx-swift-lm PR #142, Summary), so nothing in the stored data limits the range; the
comparison is the one every parity test uses (|gpu - ref| <= 2e-2 + 1e-2 |ref| and
relative L2 <= 1e-2 against the FP64 oracle over the same dequantised values).

What the scaling must not change is the conditioning of the softmax, or a tie
between two logits that the FP64 oracle resolves one way could flip: a case that
multiplies q or K by 2^e passes the attention scale times 2^-e, so the logits are
those of the unscaled case while the kernel sees the scaled operands.  A case that
multiplies V by 2^e compares out * 2^-e with ref * 2^-e (attention is linear in V,
and bf16 rounding commutes with powers of two), so the tolerance keeps its meaning.

Stale slots: the slots of a sequence's last block past its context length hold
whatever an earlier owner of the row, or an imported record, left there; they are not
part of the sequence, so nothing in them may reach an output.  The tests fill them
with NaN or infinity bit patterns (through import_blocks, which writes raw bytes)
and expect the same output as with clean slots."""
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


EXPS = [-20, -14, -8, 6, 10, 16]

# (format, head_dim, kv heads, group size): every packed format at every head dim
# (4 kv heads: two warps per kv head at head_dim 256), the five-bit K4/V4 layout, one
# 8-kv-head case at head_dim 256 (one warp per kv head), and native bf16.
GEOMS = [(f, D, 4, 32) for f in (wl.FMT_K4V4, wl.FMT_K8V4, wl.FMT_K8V8, wl.FMT_BF16) for D in (64, 128, 256)]
GEOMS += [(wl.FMT_K4V4, 128, 4, 64), (wl.FMT_K4V4, 256, 4, 64), (wl.FMT_K8V8, 256, 8, 32), (wl.FMT_K4V4, 256, 8, 32)]


def _geom_id(gm):
    f, D, hkv, gs = gm
    return f"{wl.FMT_NAMES[f]}-D{D}-hkv{hkv}" + ("-g64" if gs == 64 else "")


def _base(fmt, D, hkv, gs, lens, seed):
    G = 2
    rows, used = wl.fragmented_rows([wl.nblocks(L) for L in lens], wl.rng_for(31, D, hkv, gs))
    return wl.Workload(f"range-{wl.FMT_NAMES[fmt]}-{D}", 1, hkv * G, hkv, D, fmt, lens, rows, used,
                       1 / math.sqrt(D), 0x3A9E, seed, group=gs)


def _cases():
    """(label, workload changes, attention-scale factor, output factor)."""
    out = []
    for e in EXPS:
        out.append((f"q*2^{e}", dict(q_exp=e), 2.0 ** -e, 1.0))
        out.append((f"K*2^{e}", dict(k_exp=e), 2.0 ** -e, 1.0))
        out.append((f"V*2^{e}", dict(v_exp=e), 1.0, 2.0 ** -e))
    out.append(("1/64 of K *2^8", dict(k_boost=8), 2.0 ** -8, 1.0))
    # V outliers: the output's own unit is set by the boosted tokens, so it is compared
    # at a scale that puts them at 2^4 (with large V terms that nearly cancel, bf16
    # probabilities alone give errors of 2^-9 of those terms)
    out.append(("1/64 of V *2^8", dict(v_boost=8), 1.0, 2.0 ** -4))
    out.append(("1/64 of V *2^12", dict(v_boost=12), 1.0, 2.0 ** -8))
    out.append(("V 2^-10 then 2^6", dict(v_exp=-10, v_ramp=16), 1.0, 2.0 ** -6))
    out.append(("V 2^6 then 2^-10", dict(v_exp=6, v_ramp=-16), 1.0, 2.0 ** -6))
    out.append(("q*2^-14, K*2^10, V*2^-14", dict(q_exp=-14, k_exp=10, v_exp=-14), 2.0 ** 4, 2.0 ** 14))
    return out


@pytest.mark.parametrize("geom", GEOMS, ids=_geom_id)
def test_operand_ranges(geom):
    """Every case of _cases() at one geometry, over the default grid and over 3 CTAs
    (long segments), all failures reported together."""
    fmt, D, hkv, gs = geom
    lens = [1, 33, 95, 700, 2100]
    fails = []
    for ci, (label, chg, sfac, ofac) in enumerate(_cases()):
        import dataclasses
        w = dataclasses.replace(_base(fmt, D, hkv, gs, lens, 40 + ci), **chg)
        g, o, ol = make_pools(w)
        fill(w, g, o, ol)
        scale = w.scale * sfac
        ref = o.decode_attention(0, w.q(0), w.block_table(), w.ctx(), scale) * ofac
        for ctas in (0, 3):
            g.decode_set_ctas(ctas)
            out = g.paged_decode_attention(0, to_dev_bf16(w.q(0)), to_dev_i32(w.block_table()),
                                           to_dev_i32(w.ctx()), scale, max_ctx=max(lens))
            got = bf16_dev_to_f64(out) * ofac
            try:
                compare(got, ref, f"{label} ctas={ctas}")
            except AssertionError as ex:
                fails.append(str(ex))
        assert g.check_errors() == 0
        assert o.inexact_rotations == 0
        g.close()
    assert not fails, "\n".join(fails)


# ---------------------------------------------------------------------------
# Stale slots past the context
# ---------------------------------------------------------------------------

def _poison_tails(w, g, pattern):
    """Overwrite slots >= L % 32 of each sequence's last block, in every layer and
    stored tensor, with a non-finite pattern (export, patch on the host, import)."""
    rec = g.block_record_bytes()
    hkv = w.Hkv
    rbs = g.row_bytes
    per_layer = sum(32 * hkv * rb for rb in rbs)
    assert per_layer * w.n_layers == rec
    for b, L in enumerate(w.lens):
        if L == 0 or L % 32 == 0:
            continue
        row = int(w.rows[b][wl.nblocks(L) - 1])
        r = to_dev_i32([row])
        buf = g.export_blocks(r).cpu().numpy().copy()
        for layer in range(w.n_layers):
            off = layer * per_layer
            for kind, rb in enumerate(rbs):
                piece = buf[0, off: off + 32 * hkv * rb].reshape(32, hkv * rb)
                tail = piece[L % 32:]
                if pattern == "nan":
                    tail[:] = 0xFF  # bf16 0xFFFF, f32 0xFFFFFFFF: NaN; codes: the largest code
                elif kind in (0, 1) and w.fmt == wl.FMT_BF16:
                    tail.view(np.uint16)[:] = 0x7F80  # bf16 +inf
                elif kind in (2, 3):
                    tail.view(np.uint32)[:] = 0x7F800000  # f32 +inf scale and offset
                else:
                    tail[:] = 0xFF
                off += 32 * hkv * rb
        g.import_blocks(g.config(), r, torch.from_numpy(buf).cuda())
    torch.cuda.synchronize()


@pytest.mark.parametrize("pattern", ["nan", "inf"])
@pytest.mark.parametrize("fmt,D,gs", [(wl.FMT_BF16, 64, 32), (wl.FMT_BF16, 128, 32), (wl.FMT_K4V4, 128, 32),
                                      (wl.FMT_K8V4, 64, 32), (wl.FMT_K8V8, 64, 32), (wl.FMT_K4V4, 256, 32),
                                      (wl.FMT_K8V8, 256, 32), (wl.FMT_K4V4, 128, 64)],
                         ids=lambda v: str(v))
def test_stale_tail_slots_are_ignored(fmt, D, gs, pattern):
    lens = [1, 17, 40, 95, 401, 1000, 2047]
    rows, used = wl.fragmented_rows([wl.nblocks(L) for L in lens], wl.rng_for(33, D, gs))
    w = wl.Workload(f"stale-{wl.FMT_NAMES[fmt]}-{D}", 2, 8, 4, D, fmt, lens, rows, used, 1 / math.sqrt(D),
                    0x57A1, 71 + D + gs, group=gs)
    g, o, ol = make_pools(w)
    fill(w, g, o, ol)
    _poison_tails(w, g, pattern)
    for layer in range(w.n_layers):
        ref = o.decode_attention(layer, w.q(layer), w.block_table(), w.ctx(), w.scale)
        for ctas in (0, 2):
            g.decode_set_ctas(ctas)
            out = g.paged_decode_attention(layer, to_dev_bf16(w.q(layer)), to_dev_i32(w.block_table()),
                                           to_dev_i32(w.ctx()), w.scale, max_ctx=max(lens))
            got = bf16_dev_to_f64(out)
            assert np.isfinite(got).all(), f"layer {layer} ctas {ctas}: non-finite output"
            compare(got, ref, f"layer {layer} ctas {ctas}")
    assert g.check_errors() == 0


@pytest.mark.parametrize("n_q", [5, 8])
@pytest.mark.parametrize("fmt", [wl.FMT_BF16, wl.FMT_K4V4, wl.FMT_K8V8])
def test_stale_tail_slots_are_ignored_by_prefill(fmt, n_q):
    """n_q = 5: one query per tile; 8: the chunk in one 16-row tile."""
    lens = [40, 95, 401, 1000]
    D = 128
    rows, used = wl.fragmented_rows([wl.nblocks(L) for L in lens], wl.rng_for(35, fmt))
    w = wl.Workload(f"stale-prefill-{wl.FMT_NAMES[fmt]}", 1, 8, 4, D, fmt, lens, rows, used, 1 / math.sqrt(D),
                    0x57A2, 91 + fmt + n_q)
    g, o, ol = make_pools(w)
    fill(w, g, o, ol)
    _poison_tails(w, g, "nan")
    q = wl.bf16_normal(wl.rng_for(36, fmt, n_q), (w.B, n_q, w.Hq, D))
    ref = o.prefill_attention(0, q, w.block_table(), w.ctx(), w.scale)
    out = g.paged_prefill_attention(0, to_dev_bf16(q), to_dev_i32(w.block_table()), to_dev_i32(w.ctx()), w.scale,
                                    max_ctx=max(lens))
    got = bf16_dev_to_f64(out)
    assert np.isfinite(got).all()
    compare(got, ref, "prefill")
    assert g.check_errors() == 0


# ---------------------------------------------------------------------------
# Prefill tiles: every row of a 16-row tile picks its own q~ exponent
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("fmt", [wl.FMT_K4V4, wl.FMT_K8V4, wl.FMT_K8V8])
def test_prefill_operand_ranges(fmt):
    """Chunks of 8 queries at 2 heads per kv head (one 16-row tile at head_dim 128;
    queries 4..7 in rows 8..15) with q scaled per query by powers of two from 2^-20
    to 2^16, so the rows of one tile need exponents 36 apart.  The attention scale
    carries 2^-16: the 2^16 queries see the logits of unscaled ones, the others a
    flatter softmax (well conditioned), and a row that took another row's exponent
    would see its logits off by up to 2^36.  K or V is also scaled as in the decode
    cases."""
    D, hkv, G, n_q = 128, 4, 2, 8
    lens = [9, 40, 700, 2100]
    qexp = np.array([-20, -8, 16, 0, 6, 16, -14, 10])[None, :, None, None]
    base = 2.0 ** -16
    cases = [("q per query", {}, base, 1.0), ("K*2^-14", dict(k_exp=-14), base * 2.0 ** 14, 1.0),
             ("K*2^16", dict(k_exp=16), base * 2.0 ** -16, 1.0), ("V*2^-20", dict(v_exp=-20), base, 2.0 ** 20),
             ("V*2^16", dict(v_exp=16), base, 2.0 ** -16), ("1/64 of V *2^12", dict(v_boost=12), base, 2.0 ** -8)]
    fails = []
    import dataclasses
    for ci, (label, chg, sfac, ofac) in enumerate(cases):
        rows, used = wl.fragmented_rows([wl.nblocks(L) for L in lens], wl.rng_for(37, fmt, ci))
        w = wl.Workload(f"range-prefill-{wl.FMT_NAMES[fmt]}", 1, hkv * G, hkv, D, fmt, lens, rows, used,
                        1 / math.sqrt(D), 0x3A9F, 120 + ci)
        w = dataclasses.replace(w, **chg)
        g, o, ol = make_pools(w)
        fill(w, g, o, ol)
        q = wl.scale_pow2(wl.bf16_normal(wl.rng_for(38, fmt, ci), (w.B, n_q, w.Hq, D)), qexp)
        ref = o.prefill_attention(0, q, w.block_table(), w.ctx(), w.scale * sfac) * ofac
        for ctas in (0, 3):
            g.decode_set_ctas(ctas)
            out = g.paged_prefill_attention(0, to_dev_bf16(q), to_dev_i32(w.block_table()), to_dev_i32(w.ctx()),
                                            w.scale * sfac, max_ctx=max(lens))
            got = bf16_dev_to_f64(out) * ofac
            try:
                assert np.isfinite(got).all(), f"{label} ctas={ctas}: non-finite output"
                compare(got.reshape(-1, D), ref.reshape(-1, D), f"{label} ctas={ctas}")
            except AssertionError as ex:
                fails.append(str(ex))
        assert g.check_errors() == 0
        g.close()
    assert not fails, "\n".join(fails)
