"""Pins of the oracle's causal chunked-prefill attention, CPU only.

Query i of a chunk of n new tokens (positions L - n .. L - 1 of a sequence holding L
tokens) attends to tokens [0, L - n + i].  Pinned by a dense FP64 softmax with an
explicit causal mask over the gathered K/V (numpy, not the oracle's attention
routine), and by the reductions to decode: n = 1 is decode, the chunk's last query
is decode over all L tokens, its first query is decode over the first L - n + 1.
"""
import numpy as np
import pytest

import oracle
from oracle import FMT_BF16, FMT_K4V4, FMT_K8V4, FMT_K8V8, OraclePool
from paged_kv_cache_split_gb300 import workloads as wl
from tests.test_oracle_pins import _decode_gathered, _sylvester


def _pool(fmt, H, D, lens, seed, group=32):
    rows, used = wl.fragmented_rows([max(1, wl.nblocks(L)) for L in lens], wl.rng_for(seed, 1))
    p = OraclePool(1, H, D, fmt, seed=0x99, group_size=group)
    p.reserve_rows(used)
    rng = wl.rng_for(seed, 2)
    for b, L in enumerate(lens):
        t = np.arange(L)
        r = np.asarray(rows[b], np.int32)[t // 32]
        p.write_block(0, r, (t % 32).astype(np.int32), wl.bf16_normal(rng, (L, H, D)), wl.bf16_normal(rng, (L, H, D)))
    return p, wl.block_table(rows)


@pytest.mark.parametrize("fmt,group,D", [(FMT_BF16, 32, 64), (FMT_K4V4, 32, 64), (FMT_K8V4, 32, 128),
                                         (FMT_K8V8, 32, 64), (FMT_K4V4, 64, 128)])
def test_prefill_brute_force_causal_mask(fmt, group, D):
    H, G, n = 2, 2, 5
    lens = [5, 37, 70]
    p, bt = _pool(fmt, H, D, lens, 31, group)
    rng = wl.rng_for(32)
    q = wl.bf16_normal(rng, (len(lens), n, H * G, D))
    got = p.prefill_attention(0, q, bt, lens, 0.2)
    for b, L in enumerate(lens):
        k, v = _decode_gathered(p, p.gather_visible(0, bt[b], L), L)
        qf = wl.bf16_bits_to_f32(q[b]).astype(np.float64)  # [n, Hq, D]
        if fmt != FMT_BF16:
            qf = qf @ (_sylvester(D) @ np.diag(oracle.hadamard_signs(0x99, D))).T
        for h in range(H * G):
            z = (qf[:, h, :] @ k[h // G].T) * 0.2  # [n, L]
            mask = np.arange(L)[None, :] > (L - n + np.arange(n))[:, None]
            z[mask] = -np.inf
            w = np.exp(z - z.max(axis=1, keepdims=True))
            want = (w @ v[h // G]) / w.sum(axis=1, keepdims=True)
            np.testing.assert_allclose(got[b, :, h], want, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("fmt", [FMT_BF16, FMT_K8V4])
def test_prefill_reduces_to_decode(fmt):
    H, G, D, n = 2, 4, 64, 6
    lens = [6, 33, 200]
    p, bt = _pool(fmt, H, D, lens, 41)
    rng = wl.rng_for(42)
    q = wl.bf16_normal(rng, (len(lens), n, H * G, D))
    got = p.prefill_attention(0, q, bt, lens, 0.125)
    last = p.decode_attention(0, np.ascontiguousarray(q[:, -1]), bt, lens, 0.125)
    assert np.array_equal(got[:, -1], last)
    first = p.decode_attention(0, np.ascontiguousarray(q[:, 0]), bt, [L - n + 1 for L in lens], 0.125)
    assert np.array_equal(got[:, 0], first)
    one = p.prefill_attention(0, q[:, -1:], bt, lens, 0.125)
    assert np.array_equal(one[:, 0], last)


def test_prefill_rejects_sequences_shorter_than_the_chunk():
    p, bt = _pool(FMT_BF16, 1, 64, [3], 51)
    with pytest.raises(Exception):
        p.prefill_attention(0, np.zeros((1, 4, 1, 64), np.uint16), bt, [3], 0.1)
