"""Memory footprint of slab growth on the GPU (Qwen3-0.6B shape: 28 layers, 8 kv heads,
head_dim 128, bf16): eight sequential pool-extending spans of about 4.2k distinct tokens.

The slab pool's allocator high-water equals its live capacity (growth appends a slab and
never holds an old and a new copy at once) and stays within 1.15x of the dense K/V bytes of
the same tokens (the page's footprint gate for eight ~4k prompts), while a pool grown by
reallocate-and-copy under the same caching allocator retains every outgrown size (the
"ladder" that made the paged backend's peak exceed the dense one).  The reallocating pool
here is a counter-example written in torch for this test only: it grows once per span, the
presized form of the old scheme.  Figures are printed (run with -s to see them)."""
import os

import pytest

import paged_kv_cache_split_gb300 as pkv

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

N_LAYERS, HKV, D, BLOCK = 28, 8, 128, 32
SPANS = [4200 + 29 * s for s in range(8)]
TOKEN_BYTES = N_LAYERS * 2 * HKV * D * 2  # K and V, bf16, every layer


@pytest.fixture(autouse=True)
def _needs_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


class _CountingAllocator:
    """Stream-ordered allocator on torch's caching allocator that tracks outstanding bytes."""

    def __init__(self):
        self.live, self.outstanding, self.high_water, self.calls = {}, 0, 0, 0

        def alloc(ctx, nbytes, stream):
            self.calls += 1
            t = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
            self.live[t.data_ptr()] = t
            self.outstanding += nbytes
            self.high_water = max(self.high_water, self.outstanding)
            return t.data_ptr()

        def release(ctx, ptr, stream):
            t = self.live.pop(ptr, None)
            if t is not None:
                self.outstanding -= t.numel()

        self.struct = pkv.Allocator(pkv.ALLOC_FN(alloc), pkv.RELEASE_FN(release), None)


def _span_kv(L, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    k = torch.randn((L, HKV, D), generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn((L, HKV, D), generator=g, device="cuda").to(torch.bfloat16)
    return k, v


def _reserved_growth(fn):
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    base = torch.cuda.memory_reserved()
    torch.cuda.reset_peak_memory_stats()
    out = fn()
    torch.cuda.synchronize()
    return out, torch.cuda.max_memory_reserved() - base


def test_slab_growth_high_water_is_live_capacity():
    dense = sum(SPANS) * TOKEN_BYTES
    a = _CountingAllocator()

    def run():
        p = pkv.Pool(N_LAYERS, HKV, D, "bf16", max_slabs=64, allocator=a.struct)
        last = None
        for s, L in enumerate(SPANS):
            k, v = _span_kv(L, 100 + s)
            rows = torch.from_numpy(p.alloc_rows(-(-L // BLOCK))).cuda()
            t = torch.arange(L, device="cuda", dtype=torch.int32)
            for layer in range(N_LAYERS):
                p.write_block(layer, rows[(t // BLOCK).long()], t % BLOCK, k, v)
            last = (rows, k, v, L)
        return p, last

    (p, (rows, k, v, L)), reserved = _reserved_growth(run)
    st = p.stats()
    slab_bytes = BLOCK * BLOCK * TOKEN_BYTES
    maps_bytes = N_LAYERS * 2 * 128  # one 128-byte tensor map per layer and kind, at the slab's tail
    assert st["bytes_reserved"] == st["n_slabs"] * slab_bytes
    assert a.calls == st["n_slabs"] == st["slab_append_events"]
    assert a.high_water == a.outstanding == st["n_slabs"] * (slab_bytes + maps_bytes)
    assert a.high_water <= 1.15 * dense
    assert reserved <= 1.15 * dense + (64 << 20)
    # the last span's K/V, written after 30-odd slab appends, reads back unchanged
    gk, gv = p.gather_visible(N_LAYERS - 1, rows, L)
    assert torch.equal(gk, k.view(torch.uint8).view(L, HKV, 2 * D).transpose(0, 1))
    assert torch.equal(gv, v.view(torch.uint8).view(L, HKV, 2 * D).transpose(0, 1))
    assert p.check_errors() == 0
    print(f"\nslab pool: {st['n_slabs']} slabs, high-water {a.high_water / 2**20:.0f} MiB, torch reserved "
          f"+{reserved / 2**20:.0f} MiB, dense {dense / 2**20:.0f} MiB, ratio {a.high_water / dense:.3f}")
    p.close()
    assert a.outstanding == 0 and not a.live


def test_reallocating_growth_retains_outgrown_sizes():
    if "expandable_segments:True" in os.environ.get("PYTORCH_CUDA_ALLOC_CONF", ""):
        pytest.skip("expandable segments reuse outgrown memory")
    dense = sum(SPANS) * TOKEN_BYTES

    def run():
        pool = [[torch.empty((0, HKV, D), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
                for _ in range(N_LAYERS)]
        for s, L in enumerate(SPANS):
            k, v = _span_kv(L, 100 + s)
            for layer in range(N_LAYERS):
                for i, x in enumerate((k, v)):
                    old = pool[layer][i]
                    new = torch.empty((old.shape[0] + L, HKV, D), dtype=torch.bfloat16, device="cuda")
                    new[:old.shape[0]].copy_(old)
                    new[old.shape[0]:].copy_(x)
                    pool[layer][i] = new
        return pool

    pool, reserved = _reserved_growth(run)
    live = sum(x.numel() * 2 for pair in pool for x in pair)
    assert live == dense
    assert reserved > 2 * dense
    print(f"\nreallocating pool: torch reserved +{reserved / 2**20:.0f} MiB, dense {dense / 2**20:.0f} MiB, "
          f"ratio {reserved / dense:.3f}")
    del pool
    torch.cuda.empty_cache()
