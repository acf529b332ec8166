"""The benchmark's algorithmic byte counts, pinned to closed forms (CPU only).

Bytes per (token, kv head): bf16 4D; K4/V4 D/2 + D/2 codes plus two FP32 (scale,
offset) pairs per group for K and V; K8/V4 D + D/2 plus metadata; K8/V8 2D plus
metadata.  A call adds q and out (2 B H_q D bf16 each way), the block-table entries
used and the context lengths."""
import math

import pytest

import bench
from paged_kv_cache_split_gb300 import workloads as wl


@pytest.mark.parametrize("D", [64, 128, 256])
def test_bytes_per_token_head(D):
    meta32 = 2 * (D // 32) * 8
    assert bench.token_head_bytes(wl.FMT_BF16, D) == 4 * D
    assert bench.token_head_bytes(wl.FMT_K4V4, D) == D // 2 + D // 2 + meta32
    assert bench.token_head_bytes(wl.FMT_K8V4, D) == D + D // 2 + meta32
    assert bench.token_head_bytes(wl.FMT_K8V8, D) == 2 * D + meta32
    # groups of 32 with FP32 pairs: 6 bits per value for K4/V4
    assert 8 * bench.token_head_bytes(wl.FMT_K4V4, D) / (2 * D) == 6


@pytest.mark.parametrize("D", [128, 256])
def test_five_bit_layout(D):
    # groups of 64 with one FP32 pair: 4 + 64 / 64 = 5 bits per value, 3.2x against bf16
    b = bench.token_head_bytes(wl.FMT_K4V4, D, 64)
    assert 8 * b / (2 * D) == 5
    assert bench.token_head_bytes(wl.FMT_BF16, D) / b == 3.2


def test_qwen3_0_6b_step_bytes():
    w = wl.qwen3_0_6b()
    per_layer = bench.algorithmic_bytes(w.fmt, w.D, w.Hkv, w.Hq, w.lens)
    kv = 8 * 4096 * 8 * 4 * 128
    qo = 2 * 8 * 16 * 128 * 2
    bt = 8 * (4096 // 32) * 4
    assert per_layer == kv + qo + bt + 4 * 8 == 134_287_392
    assert per_layer * 28 == 3_760_046_976


def test_partial_last_block_not_rounded_up():
    lens = [33, 1, 64]
    got = bench.algorithmic_bytes(wl.FMT_K8V8, 64, 8, 32, lens)
    kv = sum(lens) * 8 * (2 * 64 + 2 * 2 * 8)
    qo = 2 * 3 * 32 * 64 * 2
    bt = sum(math.ceil(L / 32) for L in lens) * 4
    assert got == kv + qo + bt + 4 * 3


def test_mixed_row_bytes_is_one_block_of_every_stored_tensor():
    # one 32-token block of one layer: bf16 K and V, or codes plus (scale, offset) pairs
    assert bench.mixed_row_bytes(wl.FMT_BF16, 4, 256) == 32 * 4 * 2 * 256 * 2
    assert bench.mixed_row_bytes(wl.FMT_K4V4, 4, 256) == 32 * 4 * (128 + 128 + 2 * 8 * 8)


@pytest.mark.parametrize("fmt,D,G,n_q,launches", [
    (wl.FMT_BF16, 128, 2, 8, 2),    # 16 rows: the chunk is one tile, no expansion kernel
    (wl.FMT_BF16, 128, 2, 5, 3),    # one query per tile: expansion + attention + combine
    (wl.FMT_BF16, 256, 2, 8, 3),    # 8 rows at head_dim 256: two tiles of 4 queries
    (wl.FMT_K4V4, 128, 2, 8, 2),    # packed, 16 rows
    (wl.FMT_K4V4, 128, 2, 4, 2),    # packed, 8 rows hold the chunk
    (wl.FMT_K8V4, 64, 4, 16, 3),    # packed, 16 rows = 4 queries: four tiles
    (wl.FMT_K4V4, 128, 1, 1, 3),    # a single query keeps the expansion (short sequences flagged)
])
def test_prefill_launches_per_call(fmt, D, G, n_q, launches):
    """The launches the prefill bench line counts per call follow the library's choice
    of queries per tile (documented with pkv_paged_prefill_attention)."""
    assert bench.prefill_launches_per_call(fmt, D, G, n_q) == launches


def test_kernel_hash_ignores_comments():
    a = "int f(int x) {  // twice\n  return 2 * x; /* doubled */\n}\n"
    b = "/* header */\nint f(int x) {\n\n  return 2 * x;   \n}\n"
    c = "int f(int x) {\n  return 3 * x;\n}\n"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)
