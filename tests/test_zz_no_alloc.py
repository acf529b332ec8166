"""The allocation-free decode entry point.

Some callers cannot allocate device memory for the decode workspace (a serving loop
that reserved all of its memory at start-up, a plugin whose host framework owns the
allocator).  pkv_paged_decode_attention_noalloc serves them from a fixed scratch
array inside the library.  This file checks, through the C ABI, that two calls in a
row give the same results as the regular entry point with a caller workspace, and
that oversize requests are refused.  Both entry points run the same kernel over the
same split-K partition, and decode is deterministic, so the outputs must agree bit
for bit (a stale counter or partial left over from the first call would show up as
a difference).  It is named so that pytest collects it last."""
import ctypes

import numpy as np
import pytest

import paged_kv_cache_split_gb300 as pkv
from paged_kv_cache_split_gb300 import workloads as wl
from tests.harness import fill, make_pools, to_dev_bf16, to_dev_i32

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(autouse=True)
def _needs_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _noalloc(g, layer, q, bt, ctx, scale, max_ctx):
    B, Hq, D = q.shape
    out = torch.empty_like(q)
    st = g._lib.pkv_paged_decode_attention_noalloc(
        g.handle, layer, B, Hq, q.data_ptr(), bt.data_ptr(), int(bt.shape[1]), ctx.data_ptr(), max_ctx,
        ctypes.c_float(scale), out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == pkv.PKV_OK, pkv.lib().pkv_last_error()
    return out


@pytest.mark.parametrize("make", [lambda: wl.qwen3_0_6b(n_layers=2, B=3, L=1500),
                                  lambda: wl.llama_1b(wl.FMT_K8V4, B=6, lo=30, hi=900),
                                  lambda: wl.qwen3_1_7b_k4v4(B=2, L=700)])
def test_noalloc_matches_workspace_entry_point(make):
    w = make()
    g, o, ol = make_pools(w, oracle_layers=[])
    fill(w, g, None, [])
    bt = to_dev_i32(w.block_table())
    ctx = to_dev_i32(w.ctx())
    for layer in range(w.n_layers):
        q = to_dev_bf16(w.q(layer))
        ref = g.paged_decode_attention(layer, q, bt, ctx, w.scale, max_ctx=max(w.lens))
        first = _noalloc(g, layer, q, bt, ctx, w.scale, max(w.lens))
        second = _noalloc(g, layer, q, bt, ctx, w.scale, max(w.lens))
        torch.cuda.synchronize()
        assert torch.equal(first.view(torch.int16), ref.view(torch.int16)), f"{w.name} layer {layer}, first call"
        assert torch.equal(second.view(torch.int16), ref.view(torch.int16)), f"{w.name} layer {layer}, second call"
    assert g.check_errors() == 0


def test_noalloc_rejects_requests_beyond_the_fixed_array():
    g = pkv.Pool(1, 8, 256, "bf16", max_slabs=4)
    g.reserve_rows(32)
    B, Hq = 2048, 64   # partials for this batch exceed the fixed array
    q = torch.zeros((B, Hq, 256), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((B, 1), dtype=torch.int32, device="cuda")
    ctx = torch.ones((B,), dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    assert g.decode_workspace_bytes(B, Hq) > 8 * 1024 * 1024
    st = g._lib.pkv_paged_decode_attention_noalloc(g.handle, 0, B, Hq, q.data_ptr(), bt.data_ptr(), 1, ctx.data_ptr(),
                                                   1, ctypes.c_float(0.1), out.data_ptr(),
                                                   torch.cuda.current_stream().cuda_stream)
    assert st == pkv.PKV_ERR_RANGE
    assert b"fixed array" in pkv.lib().pkv_last_error()
