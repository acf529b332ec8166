"""Pins for the oracle: each check ties the oracle to something other than itself —
values the pages print, published test vectors, closed forms, exact arithmetic,
invariants, or brute force on tiny inputs.  CPU only."""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import FMT_BF16, FMT_K4V4, FMT_K8V4, FMT_K8V8, OraclePool
from paged_kv_cache_split_gb300 import workloads as wl


def _golden_rows(path):
    with open(path) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


# ---------------------------------------------------------------------------
# Hadamard basis
# ---------------------------------------------------------------------------

def test_splitmix64_published_vectors(golden_dir):
    gamma = 0x9E3779B97F4A7C15
    for idx, hexval in _golden_rows(os.path.join(golden_dir, "splitmix64_seed0.txt")):
        state = (int(idx) * gamma) % 2**64
        assert oracle.splitmix64(state) == int(hexval, 16)


def _sylvester(D):
    """Sylvester construction by Kronecker products (independent of popcount indexing)."""
    H = np.array([[1.0]])
    while H.shape[0] < D:
        H = np.kron(np.array([[1.0, 1.0], [1.0, -1.0]]), H)
    return H / math.sqrt(D)


@pytest.mark.parametrize("D", [2, 4, 8, 16, 32, 64, 128, 256])
def test_hadamard_orthonormal_and_sylvester(D):
    H = oracle.hadamard_matrix(D)
    assert np.abs(H @ H.T - np.eye(D)).max() < 1e-15 * D
    assert np.array_equal(H, _sylvester(D))


def test_hadamard_d2_closed_form():
    r = 1 / math.sqrt(2)
    assert np.array_equal(oracle.hadamard_matrix(2), np.array([[r, r], [r, -r]]))


def test_signs_are_plus_minus_one_and_seeded():
    s = oracle.hadamard_signs(0x5EED, 128)
    assert set(np.unique(s)) <= {-1.0, 1.0}
    assert 32 < (s < 0).sum() < 96
    gamma = 0x9E3779B97F4A7C15
    # seed 0: sign i comes from the top bit of the i-th published output... only
    # index 0 of the stream is the published value at state 0; pin that one:
    assert (oracle.hadamard_signs(0, 1)[0] < 0) == bool(0xE220A8397B1DCDAF >> 63)
    assert (oracle.hadamard_signs(gamma, 1)[0] < 0) == bool(0x6E789E6AA1B965F4 >> 63)
    assert not np.array_equal(oracle.hadamard_signs(1, 128), s)


@pytest.mark.parametrize("D", [64, 128, 256])
def test_rotate_q_matches_kronecker_and_preserves_dot(D):
    rng = np.random.default_rng(D)
    s = oracle.hadamard_signs(77, D)
    q, k = rng.standard_normal(D), rng.standard_normal(D)
    qr, kr = oracle.rotate_q(q, s), oracle.rotate_q(k, s)
    R = _sylvester(D) @ np.diag(s)
    np.testing.assert_allclose(qr, R @ q, rtol=0, atol=1e-13)
    assert abs(qr @ kr - q @ k) <= 1e-12 * max(1.0, abs(q @ k)) + 1e-12 * D
    assert abs(np.linalg.norm(qr) - np.linalg.norm(q)) < 1e-12 * D


@pytest.mark.parametrize("D", [64, 128, 256])
def test_rotate_k_bit_exact_against_exact_arithmetic(D):
    """Rotated K = fl32(fl64(exact_sum * fl64(1/sqrt(D)))) computed with Fractions."""
    rng = wl.rng_for(5, D)
    k = wl.bf16_normal(rng, (3, D), outlier_frac=0.05)
    s = oracle.hadamard_signs(0xABC, D)
    Hs = np.rint(_sylvester(D) * math.sqrt(D)).astype(int)
    inv = Fraction(1.0 / math.sqrt(D))
    for row in k:
        vals = [Fraction(float(v)) for v in wl.bf16_bits_to_f32(row)]
        got, exact = oracle.rotate_k(row, s)
        assert exact
        want = []
        for i in range(D):
            tot = sum((Hs[i, j] * int(s[j])) * vals[j] for j in range(D))
            want.append(np.float32(float(float(tot) * inv)))
        assert np.array_equal(got.view(np.uint32), np.array(want, np.float32).view(np.uint32))


def test_rotate_k_flags_inexact_sums():
    D = 128
    x = np.zeros(D, np.float32)
    x[0], x[1] = 2.0 ** 20, 2.0 ** -30   # exponent spread 50 > 45 - 7
    got, exact = oracle.rotate_k(wl.f32_to_bf16_bits(x), oracle.hadamard_signs(1, D))
    assert not exact


# ---------------------------------------------------------------------------
# Affine quantiser
# ---------------------------------------------------------------------------

def test_quant_worked_example(golden_dir):
    rows = {r[0]: r[1:] for r in _golden_rows(os.path.join(golden_dir, "quant_nibble_order.txt"))}
    x = np.array([float(v) for v in rows["values"]], np.float32)
    codes, meta = oracle.quantize(x, 4)
    assert codes.tobytes().hex() == "".join(rows["packed_hex"])
    assert meta[0, 0] == float(rows["scale"][0]) and meta[0, 1] == float(rows["offset"][0])


@pytest.mark.parametrize("group", [32, 64])
@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("D", [64, 128, 256])
def test_quant_error_bound(bits, D, group):
    rng = np.random.default_rng(bits * 1000 + D + group)
    for trial in range(20):
        x = (rng.standard_normal(D) * rng.choice([1e-3, 1.0, 40.0])).astype(np.float32)
        codes, meta = oracle.quantize(x, bits, group)
        assert meta.shape == (D // group, 2)
        xh = oracle.dequantize(codes, meta, D, bits, group)
        for g in range(D // group):
            xs = x[group * g: group * g + group].astype(np.float64)
            sc = float(meta[g, 0])
            # half a step plus the float32 rounding of the scale, offset and difference
            slack = 4 * np.spacing(np.float32(np.abs(xs).max()))
            assert np.abs(xs - xh[group * g: group * g + group]).max() <= sc / 2 + slack
            assert meta[g, 1] == np.float32(xs.min())
            assert sc == np.float32(np.float32(xs.max()) - np.float32(xs.min())) / np.float32(2 ** bits - 1)


@pytest.mark.parametrize("bits", [4, 8])
def test_quant_constant_group_exact(bits):
    x = np.full(64, 3.25, np.float32)
    codes, meta = oracle.quantize(x, bits)
    assert not codes.any()
    assert np.all(meta[:, 0] == 0) and np.all(meta[:, 1] == np.float32(3.25))
    assert np.array_equal(oracle.dequantize(codes, meta, 64, bits), x.astype(np.float64))


@pytest.mark.parametrize("bits", [4, 8])
def test_quant_integer_grid_exact(bits):
    top = 2 ** bits - 1
    rng = np.random.default_rng(bits)
    c = 0.375  # exact binary fraction
    ints = np.concatenate([[0, top], rng.integers(0, top + 1, 30)])
    rng.shuffle(ints)
    x = (ints * c - 2.0).astype(np.float32)
    codes, meta = oracle.quantize(x, bits)
    unpacked = codes if bits == 8 else np.stack([codes & 15, codes >> 4], 1).reshape(-1)
    assert np.array_equal(unpacked, ints)
    assert meta[0, 0] == np.float32(c) and meta[0, 1] == np.float32(-2.0)
    assert np.array_equal(oracle.dequantize(codes, meta, 32, bits), x.astype(np.float64))


def test_quant_round_half_to_even():
    # scale 1 (min 0, max 15); (x - min)/scale = 0.5, 1.5, 2.5, 3.5 -> 0, 2, 2, 4
    x = np.array([0, 15, 0.5, 1.5, 2.5, 3.5] + [0] * 26, np.float32)
    codes, _ = oracle.quantize(x, 4)
    c = np.stack([codes & 15, codes >> 4], 1).reshape(-1)
    assert list(c[:6]) == [0, 15, 0, 2, 2, 4]


def test_payload_ratio(golden_dir):
    rows = {r[0]: (float(r[1]), float(r[2])) for r in _golden_rows(os.path.join(golden_dir, "payload_ratio.txt"))}
    assert rows["page_k4v4_5bit"][1] == 16 / rows["page_k4v4_5bit"][0]
    for fmt, key in [(FMT_K4V4, "k4v4_g32_f32pair"), (FMT_K8V4, "k8v4_g32_f32pair"), (FMT_K8V8, "k8v8_g32_f32pair")]:
        p = OraclePool(1, 8, 128, fmt)
        bits = 8 * sum(p.row_bytes) / (2 * 128)
        assert bits == rows[key][0]
        assert abs(16 / bits - rows[key][1]) < 1e-12
    # groups of 64 with one FP32 pair reach the page's five bits
    p = OraclePool(1, 8, 128, FMT_K4V4, group_size=64)
    bits = 8 * sum(p.row_bytes) / (2 * 128)
    assert bits == rows["k4v4_g64_f32pair"][0] == rows["page_k4v4_5bit"][0]
    assert 16 / bits == rows["k4v4_g64_f32pair"][1]


# ---------------------------------------------------------------------------
# Slab mapping, runs, gather, copy-on-write
# ---------------------------------------------------------------------------

def test_slab_mapping_places_rows(golden_dir):
    H, D = 2, 64
    p = OraclePool(1, H, D, FMT_BF16)
    p.reserve_rows(34 * 32)
    rng = wl.rng_for(9)
    for row, slab, r in [tuple(map(int, x)) for x in _golden_rows(os.path.join(golden_dir, "slab_mapping.txt"))]:
        k = wl.bf16_normal(rng, (1, H, D))
        v = wl.bf16_normal(rng, (1, H, D))
        slot = (row * 7) % 32
        p.write_block(0, [row], [slot], k, v)
        raw = p.read_slab(0, 0, slab).view(np.uint16)
        off = ((r * 32 + slot) * H) * D
        assert np.array_equal(raw[off: off + H * D], k.reshape(-1))


def test_slab_runs_golden(golden_dir):
    for first, n, nruns, starts in _golden_rows(os.path.join(golden_dir, "slab_runs_4k.txt")):
        rows = np.arange(int(first), int(first) + int(n))
        got = oracle.slab_runs(rows)
        assert len(got) == int(nruns)
        assert list(got) == [int(s) for s in starts.split(",")]


def test_slab_runs_brute_force():
    rng = np.random.default_rng(3)
    for trial in range(200):
        n = int(rng.integers(1, 60))
        rows = rng.integers(0, 200, n)
        got = list(oracle.slab_runs(rows))
        # brute force: i starts a run iff it is the first index or its slab differs
        # from the previous one; every run is a maximal constant-slab interval
        slabs = [int(r) // 32 for r in rows]
        want = [i for i in range(n) if i == 0 or slabs[i] != slabs[i - 1]]
        assert got == want
        bounds = want + [n]
        for a, b in zip(bounds[:-1], bounds[1:]):
            assert len(set(slabs[a:b])) == 1
            if b < n:
                assert slabs[b] != slabs[b - 1]


def _fill(pool, layer, rows_per_seq, lens, data):
    for b, L in enumerate(lens):
        t = np.arange(L)
        r = np.asarray(rows_per_seq[b], np.int32)[t // 32]
        pool.write_block(layer, r, (t % 32).astype(np.int32), data[b][0], data[b][1])


@pytest.mark.parametrize("fmt", [FMT_BF16, FMT_K4V4, FMT_K8V4, FMT_K8V8])
def test_fragmented_equals_contiguous(fmt):
    """Acceptance criteria of mlxcel #235: a gather through a fragmented block table
    (freed rows reused, sequences interleaved) gives the same bytes as the contiguous
    layout, for spans crossing slabs."""
    H, D = 2, 64
    lens = [700, 1500, 33]
    rng = wl.rng_for(11, fmt)
    data = [(wl.bf16_normal(rng, (L, H, D)), wl.bf16_normal(rng, (L, H, D))) for L in lens]
    nblk = [wl.nblocks(L) for L in lens]
    frag, used_f = wl.fragmented_rows(nblk, wl.rng_for(12))
    cont, used_c = [], 0
    for n in nblk:
        cont.append(list(range(used_c, used_c + n)))
        used_c += n
    a = OraclePool(1, H, D, fmt, seed=3)
    b = OraclePool(1, H, D, fmt, seed=3)
    a.reserve_rows(used_f)
    b.reserve_rows(used_c)
    _fill(a, 0, frag, lens, data)
    _fill(b, 0, cont, lens, data)
    for i, L in enumerate(lens):
        assert len(oracle.slab_runs(frag[i])) > 1
        ga = a.gather_visible(0, frag[i], L)
        gb = b.gather_visible(0, cont[i], L)
        for x, y in zip(ga, gb):
            assert np.array_equal(x, y)
        if fmt == FMT_BF16:
            k = ga[0].view(np.uint16).reshape(H, L, D)
            assert np.array_equal(k, data[i][0].transpose(1, 0, 2))


def test_copy_block_copies_every_layer_and_tensor():
    p = OraclePool(3, 2, 64, FMT_K4V4, seed=5)
    p.reserve_rows(64)
    rng = wl.rng_for(13)
    for layer in range(3):
        p.write_block(layer, np.arange(40, dtype=np.int32) // 4, np.arange(40, dtype=np.int32) % 32,
                      wl.bf16_normal(rng, (40, 2, 64)), wl.bf16_normal(rng, (40, 2, 64)))
    before = {(l, k, r): p.read_block(l, k, r) for l in range(3) for k in range(4) for r in range(12)}
    p.copy_block([3, 7], [40, 41])
    for l in range(3):
        for k in range(4):
            assert np.array_equal(p.read_block(l, k, 40), before[(l, k, 3)])
            assert np.array_equal(p.read_block(l, k, 41), before[(l, k, 7)])
            for r in range(12):
                assert np.array_equal(p.read_block(l, k, r), before[(l, k, r)])


def test_reserve_appends_without_touching_existing_slabs():
    p = OraclePool(1, 2, 64)
    p.reserve_rows(32)
    p.write_block(0, [5], [3], np.full((1, 2, 64), 0x3F80, np.uint16), np.full((1, 2, 64), 0x4000, np.uint16))
    s0 = p.read_slab(0, 0, 0)
    p.reserve_rows(32 * 5)
    assert p.rows == 160
    assert np.array_equal(p.read_slab(0, 0, 0), s0)
    assert not p.read_slab(0, 0, 4).any()


# ---------------------------------------------------------------------------
# Attention
# ---------------------------------------------------------------------------

def _decode_gathered(p, g, L):
    """FP64 K, V [Hkv, L, D] from gathered bytes (bf16 or codes + meta)."""
    H, D = p.n_kv_heads, p.head_dim
    if p.fmt == FMT_BF16:
        k = wl.bf16_bits_to_f32(g[0].view(np.uint16)).reshape(H, L, D).astype(np.float64)
        v = wl.bf16_bits_to_f32(g[1].view(np.uint16)).reshape(H, L, D).astype(np.float64)
        return k, v
    kb, vb = oracle.FORMAT_BITS[p.fmt]
    out = []
    gs = p.group_size
    for codes, meta, bits in [(g[0], g[2], kb), (g[1], g[3], vb)]:
        m = meta.view(np.float32).reshape(H, L, D // gs, 2)
        if bits == 8:
            c = codes.reshape(H, L, D).astype(np.float64)
        else:
            c = np.stack([codes & 15, codes >> 4], -1).reshape(H, L, D).astype(np.float64)
        sc = np.repeat(m[..., 0].astype(np.float64), gs, axis=-1)
        of = np.repeat(m[..., 1].astype(np.float64), gs, axis=-1)
        out.append(c * sc + of)
    return out[0], out[1]


def _brute(p, q_bits, bt, lens, scale):
    """Dense softmax(q K^T scale) V in FP64 on the gathered K/V (numpy)."""
    B, Hq, D = q_bits.shape
    G = Hq // p.n_kv_heads
    out = np.zeros((B, Hq, D))
    for b in range(B):
        L = int(lens[b])
        if L == 0:
            continue
        k, v = _decode_gathered(p, p.gather_visible(0, bt[b], L), L)
        q = wl.bf16_bits_to_f32(q_bits[b]).astype(np.float64)
        if p.fmt != FMT_BF16:
            q = q @ (_sylvester(D) @ np.diag(oracle.hadamard_signs(p.seed, D))).T
        for h in range(Hq):
            z = k[h // G] @ q[h] * scale
            w = np.exp(z - z.max())
            out[b, h] = w @ v[h // G] / w.sum()
    return out


@pytest.mark.parametrize("fmt,group,D", [(FMT_BF16, 32, 64), (FMT_K4V4, 32, 64), (FMT_K8V4, 32, 64),
                                         (FMT_K8V8, 32, 64), (FMT_K4V4, 64, 128)])
def test_attention_brute_force(fmt, group, D):
    H, G = 2, 3
    lens = [1, 31, 33, 97, 0]
    rng = wl.rng_for(21, fmt)
    nblk = [max(1, wl.nblocks(L)) for L in lens]
    rows, used = wl.fragmented_rows(nblk, wl.rng_for(22))
    p = OraclePool(1, H, D, fmt, seed=0x77, group_size=group)
    p.reserve_rows(used)
    _fill(p, 0, rows, lens, [(wl.bf16_normal(rng, (L, H, D)), wl.bf16_normal(rng, (L, H, D))) for L in lens])
    q = wl.bf16_normal(rng, (len(lens), H * G, D))
    bt = wl.block_table(rows)
    got = p.decode_attention(0, q, bt, lens, 0.125)
    want = _brute(p, q, bt, lens, 0.125)
    np.testing.assert_allclose(got, want, rtol=1e-11, atol=1e-12)
    assert not got[4].any()


def test_attention_special_cases():
    H, D = 1, 64
    p = OraclePool(1, H, D)
    p.reserve_rows(64)
    rng = wl.rng_for(31)
    q = wl.bf16_normal(rng, (1, 2, D))
    # L = 1: output is v_0 exactly
    k1, v1 = wl.bf16_normal(rng, (1, H, D)), wl.bf16_normal(rng, (1, H, D))
    p.write_block(0, [9], [0], k1, v1)
    out = p.decode_attention(0, q, np.array([[9]], np.int32), [1], 0.3)
    assert np.array_equal(out[0, 0], wl.bf16_bits_to_f32(v1[0, 0]).astype(np.float64))
    # all keys equal: output is the mean of V
    L = 45
    kk = np.repeat(wl.bf16_normal(rng, (1, H, D)), L, 0)
    vv = wl.bf16_normal(rng, (L, H, D))
    t = np.arange(L)
    rows = np.array([20, 3], np.int32)
    p.write_block(0, rows[t // 32], (t % 32).astype(np.int32), kk, vv)
    out = p.decode_attention(0, q, rows[None], [L], 0.3)
    np.testing.assert_allclose(out[0, 1], wl.bf16_bits_to_f32(vv[:, 0]).astype(np.float64).mean(0), atol=1e-13)
    # one dominant logit: output is that token's V
    kd = np.zeros((L, H, D), np.uint16)
    kd[17] = wl.f32_to_bf16_bits(np.sign(wl.bf16_bits_to_f32(q[0, 0])) * 64.0)
    p.write_block(0, rows[t // 32], (t % 32).astype(np.int32), kd, vv)
    out = p.decode_attention(0, q, rows[None], [L], 1.0)
    np.testing.assert_allclose(out[0, 0], wl.bf16_bits_to_f32(vv[17, 0]).astype(np.float64), atol=1e-12)


def test_attention_permutation_invariance():
    H, D = 2, 64
    L = 150
    rng = wl.rng_for(41)
    k, v = wl.bf16_normal(rng, (L, H, D)), wl.bf16_normal(rng, (L, H, D))
    q = wl.bf16_normal(rng, (1, 4, D))
    perm = wl.rng_for(42).permutation(L)
    p = OraclePool(1, H, D, FMT_K8V8, seed=2)
    p.reserve_rows(16)
    t = np.arange(L)
    rows_a = np.array([0, 1, 2, 3, 4], np.int32)
    rows_b = np.array([8, 9, 10, 11, 12], np.int32)
    p.write_block(0, rows_a[t // 32], (t % 32).astype(np.int32), k, v)
    p.write_block(0, rows_b[t // 32], (t % 32).astype(np.int32), k[perm], v[perm])
    a = p.decode_attention(0, q, rows_a[None], [L], 0.125)
    b = p.decode_attention(0, q, rows_b[None], [L], 0.125)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14)


def test_gqa_mapping_uses_floor_division():
    """Query head h reads kv head h // G: give each kv head constant V = its index."""
    H, G, D = 4, 2, 64
    p = OraclePool(1, H, D)
    p.reserve_rows(32)
    rng = wl.rng_for(51)
    k = wl.bf16_normal(rng, (40, H, D))
    v = np.zeros((40, H, D), np.uint16)
    for h in range(H):
        v[:, h] = wl.f32_to_bf16_bits(np.full(D, float(h), np.float32))
    t = np.arange(40)
    rows = np.array([0, 1], np.int32)
    p.write_block(0, rows[t // 32], (t % 32).astype(np.int32), k, v)
    out = p.decode_attention(0, wl.bf16_normal(rng, (1, H * G, D)), rows[None], [40], 0.125)
    assert np.allclose(out[0, :, 0], np.arange(H * G) // G)


@pytest.mark.parametrize("fmt,kb,vb,group", [(FMT_K4V4, 4, 4, 32), (FMT_K8V4, 8, 4, 32), (FMT_K8V8, 8, 8, 32),
                                            (FMT_K4V4, 4, 4, 64)])
def test_pool_write_equals_rotate_then_quantize(fmt, kb, vb, group):
    """The pool image's packed write path equals the pinned primitives composed."""
    H, D = 2, 128
    p = OraclePool(1, H, D, fmt, seed=0x5EED, group_size=group)
    p.reserve_rows(32)
    rng = wl.rng_for(61)
    k, v = wl.bf16_normal(rng, (5, H, D), 0.01), wl.bf16_normal(rng, (5, H, D), 0.01)
    p.write_block(0, np.full(5, 3, np.int32), np.arange(5, dtype=np.int32), k, v)
    kc, vc, km, vm = p.gather_visible(0, np.array([3], np.int32), 5)
    s = oracle.hadamard_signs(0x5EED, D)
    for t in range(5):
        for h in range(H):
            rk, exact = oracle.rotate_k(k[t, h], s)
            assert exact
            c, m = oracle.quantize(rk, kb, group)
            assert np.array_equal(kc[h, t], c) and np.array_equal(km[h, t].view(np.float32), m.reshape(-1))
            c, m = oracle.quantize(wl.bf16_bits_to_f32(v[t, h]), vb, group)
            assert np.array_equal(vc[h, t], c) and np.array_equal(vm[h, t].view(np.float32), m.reshape(-1))
    assert p.inexact_rotations == 0
