"""Pool runtime on the GPU: slab append without copy (counter-pinned), pointer
stability, reserved bytes, row allocator (LIFO reuse, refcounts), allocator-failure
atomicity, storage identity, and the device error word.  Calls go through the C ABI."""
import ctypes

import numpy as np
import pytest

import paged_kv_cache_split_gb300 as pkv
from paged_kv_cache_split_gb300 import workloads as wl
from tests.harness import to_dev_bf16, to_dev_i32

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(autouse=True)
def _needs_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_append_counter_pointer_stability_and_bytes():
    p = pkv.Pool(3, 8, 128, "k4v4", hadamard_seed=1, max_slabs=16)
    p.append_slab(1)
    first = {(l, k): p.slab_address(l, k, 0) for l in range(3) for k in range(4)}
    assert all(first.values())
    p.append_slab(3)
    p.append_slab(2)
    s = p.stats()
    assert s["n_slabs"] == 6 and s["slab_append_events"] == 6
    assert s["rows_capacity"] == 6 * 32
    per_slab = sum(32 * 32 * 8 * rb for rb in s["row_bytes"][:4]) * 3
    assert s["bytes_reserved"] == 6 * per_slab
    assert {(l, k): p.slab_address(l, k, 0) for l in range(3) for k in range(4)} == first
    addrs = {p.slab_address(l, k, sl) for l in range(3) for k in range(4) for sl in range(6)}
    assert len(addrs) == 3 * 4 * 6
    with pytest.raises(pkv.PkvError):
        p.slab_address(0, 0, 6)
    p.close()


def test_fresh_slabs_read_as_zero_and_old_data_survives_growth():
    p = pkv.Pool(1, 2, 64, "bf16", max_slabs=8)
    p.append_slab(1)
    rng = wl.rng_for(1)
    k, v = wl.bf16_normal(rng, (32, 2, 64)), wl.bf16_normal(rng, (32, 2, 64))
    p.write_block(0, to_dev_i32(np.full(32, 5)), to_dev_i32(np.arange(32)), to_dev_bf16(k), to_dev_bf16(v))
    before = [t.cpu().numpy() for t in p.gather_visible(0, to_dev_i32([5]), 32)]
    p.append_slab(2)
    after = [t.cpu().numpy() for t in p.gather_visible(0, to_dev_i32([5]), 32)]
    assert all(np.array_equal(a, b) for a, b in zip(before, after))
    zero = [t.cpu().numpy() for t in p.gather_visible(0, to_dev_i32([40, 95]), 64)]
    assert not any(z.any() for z in zero)
    assert p.check_errors() == 0


def test_row_allocator_lifo_and_refcounts():
    p = pkv.Pool(1, 1, 64, "bf16", max_slabs=8)
    rows = p.alloc_rows(40)
    assert list(rows) == list(range(40))
    assert p.stats()["slab_append_events"] == 2
    assert p.stats()["rows_in_use"] == 40
    p.release_row(5)
    p.release_row(7)
    assert p.stats()["rows_in_use"] == 38
    assert list(p.alloc_rows(3)) == [7, 5, 40]
    assert p.stats()["rows_in_use"] == 41
    p.retain_row(9)
    p.release_row(9)
    assert p.stats()["rows_in_use"] == 41
    p.release_row(9)
    assert p.stats()["rows_in_use"] == 40
    with pytest.raises(pkv.PkvError):
        p.release_row(9)
    with pytest.raises(pkv.PkvError):
        p.retain_row(1000)


class _TorchAllocator:
    """Stream-ordered allocator backed by torch's caching allocator; fails at call n."""

    def __init__(self, fail_at=None):
        self.live, self.calls, self.fail_at = {}, 0, fail_at

        def alloc(ctx, nbytes, stream):
            self.calls += 1
            if self.fail_at is not None and self.calls == self.fail_at:
                return None
            t = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
            self.live[t.data_ptr()] = t
            return t.data_ptr()

        def release(ctx, ptr, stream):
            self.live.pop(ptr, None)

        self.struct = pkv.Allocator(pkv.ALLOC_FN(alloc), pkv.RELEASE_FN(release), None)


def test_allocator_failure_leaves_pool_unchanged():
    a = _TorchAllocator(fail_at=4)
    p = pkv.Pool(2, 4, 64, "k8v4", hadamard_seed=3, max_slabs=16, allocator=a.struct)
    p.append_slab(2)
    s0 = p.stats()
    addr0 = [p.slab_address(l, k, s) for l in range(2) for k in range(4) for s in range(2)]
    live0 = len(a.live)
    with pytest.raises(pkv.PkvError) as e:
        p.append_slab(3)  # calls 3, 4(fails), -> rolls back call 3
    assert e.value.status == pkv.PKV_ERR_OOM
    assert p.stats() == s0
    assert [p.slab_address(l, k, s) for l in range(2) for k in range(4) for s in range(2)] == addr0
    assert len(a.live) == live0
    p.append_slab(1)  # later calls succeed
    assert p.stats()["n_slabs"] == 3
    p.close()
    assert not a.live


def test_storage_identity_check():
    p = pkv.Pool(1, 8, 128, "k4v4", hadamard_seed=0x5EED)
    assert p.check_identity(pkv.make_config(4, 8, 128, "k4v4", hadamard_seed=0x5EED))
    assert not p.check_identity(pkv.make_config(1, 8, 128, "k4v4", hadamard_seed=0x5EEE))
    assert not p.check_identity(pkv.make_config(1, 8, 128, "k8v4", hadamard_seed=0x5EED))
    assert not p.check_identity(pkv.make_config(1, 4, 128, "k4v4", hadamard_seed=0x5EED))


def test_gather_meta_arguments_must_match_format():
    p = pkv.Pool(1, 2, 64, "k4v4", max_slabs=4)
    p.append_slab(1)
    bt = to_dev_i32([0])
    k = torch.empty((2, 32, 32), dtype=torch.uint8, device="cuda")
    st = p._lib.pkv_gather_visible(p.handle, 0, bt.data_ptr(), 32, k.data_ptr(), k.data_ptr(), None, None,
                                   torch.cuda.current_stream().cuda_stream)
    assert st == pkv.PKV_ERR_FORMAT


def test_device_error_word_reports_and_skips():
    p = pkv.Pool(1, 2, 64, "bf16", max_slabs=4)
    p.append_slab(1)
    rng = wl.rng_for(2)
    k, v = wl.bf16_normal(rng, (2, 2, 64)), wl.bf16_normal(rng, (2, 2, 64))
    # row 32 is beyond the 32 rows of one slab; slot 40 is beyond a block
    p.write_block(0, to_dev_i32([32, 1]), to_dev_i32([0, 0]), to_dev_bf16(k), to_dev_bf16(v))
    assert p.check_errors() & pkv.ERR_ROW
    p.write_block(0, to_dev_i32([1]), to_dev_i32([40]), to_dev_bf16(k[:1]), to_dev_bf16(v[:1]))
    assert p.check_errors() & pkv.ERR_SLOT
    assert p.check_errors() == 0  # cleared
    q = to_dev_bf16(wl.bf16_normal(rng, (1, 4, 64)))
    out = p.paged_decode_attention(0, q, to_dev_i32([[1, 99]]), to_dev_i32([40]), 0.125)
    assert p.check_errors() & pkv.ERR_ROW
    out = p.paged_decode_attention(0, q, to_dev_i32([[1, 2]]), to_dev_i32([65]), 0.125)
    assert p.check_errors() & pkv.ERR_CTX
    torch.cuda.synchronize()


@pytest.mark.parametrize("fmt,D,hkv,gs", [("bf16", 128, 8, 32), ("k4v4", 128, 8, 32), ("k8v4", 64, 8, 32),
                                          ("k8v8", 256, 4, 32), ("k4v4", 256, 4, 64)])
def test_price_request_closed_forms_and_growth(fmt, D, hkv, gs):
    """The admission price (mlx-swift-lm PR #142, Summary: storage growth, page and
    fixed costs and the step's guaranteed workspace priced apart): each figure
    against its closed form, and the predicted growth against what alloc_rows then
    asks of the allocator."""
    requested = []

    def alloc(ctx, n, stream):
        t = torch.empty(n, dtype=torch.uint8, device="cuda")
        requested.append(n)
        keep[t.data_ptr()] = t
        return t.data_ptr()

    def release(ctx, ptr, stream):
        keep.pop(ptr, None)

    keep = {}
    a = pkv.Allocator(pkv.ALLOC_FN(alloc), pkv.RELEASE_FN(release), None)
    L, Hq = 3, 2 * hkv
    g = pkv.Pool(L, hkv, D, fmt, hadamard_seed=1, max_slabs=6, allocator=a, group_size=gs)
    rb = g.row_bytes
    block = sum(32 * hkv * r for r in rb)          # one block of one layer, every tensor
    slab_data = 32 * block * L                     # 32 blocks per slab, every layer
    group = -(-slab_data // 128) * 128 + L * len(rb) * 128  # + one 128-byte tensor map per (layer, tensor)
    pr = g.price_request(40, B=4, Hq=Hq, n_q=1, max_blocks=64)
    assert pr["slabs_to_append"] == 2 and pr["free_rows"] == 0
    assert pr["storage_bytes"] == 2 * group
    assert pr["page_bytes"] == 40 * block * L == 40 * g.block_record_bytes()
    assert pr["fixed_bytes"] == 64 * 4 + 4 + 2 * Hq * D * 2
    assert pr["workspace_bytes"] == g.decode_workspace_bytes(4, Hq)
    before = g.stats()
    g.alloc_rows(40)
    after = g.stats()
    assert after["n_slabs"] - before["n_slabs"] == 2
    assert sum(requested) == pr["storage_bytes"]
    assert after["bytes_reserved"] - before["bytes_reserved"] == 2 * slab_data
    # 24 rows left on the free list
    p20 = g.price_request(20, B=4, Hq=Hq)
    assert p20["slabs_to_append"] == 0 and p20["storage_bytes"] == 0 and p20["free_rows"] == 24
    p30 = g.price_request(30, B=4, Hq=Hq)
    assert p30["slabs_to_append"] == 1 and p30["storage_bytes"] == group
    # a chunked-prefill step prices the prefill workspace
    pp = g.price_request(10, B=2, Hq=Hq, n_q=8, max_blocks=16)
    assert pp["workspace_bytes"] == g.prefill_workspace_bytes(2, 8, Hq, 16)
    assert pp["fixed_bytes"] == 16 * 4 + 4 + 2 * 8 * Hq * D * 2
    # more slabs than the table holds: the pool can never take the request
    with pytest.raises(pkv.PkvError) as e:
        g.price_request(24 + 4 * 32 + 1, B=1, Hq=Hq)
    assert e.value.status == pkv.PKV_ERR_RANGE
    g.price_request(24 + 4 * 32, B=1, Hq=Hq)
    for bad in (dict(new_blocks=-1, B=1, Hq=Hq), dict(new_blocks=1, B=0, Hq=Hq),
                dict(new_blocks=1, B=1, Hq=Hq + 1), dict(new_blocks=1, B=1024, Hq=Hq, n_q=8)):
        with pytest.raises(pkv.PkvError) as e:
            g.price_request(**bad)
        assert e.value.status == pkv.PKV_ERR_INVALID
    assert g.stats()["n_slabs"] == 2  # pricing changes nothing
    g.close()
