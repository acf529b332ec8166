"""Block records (export / import) of the CUDA path, through the C ABI, against the
oracle.

Bit-exact: the exported records equal the oracle's records of the same blocks;
records imported into other rows of a second pool give byte-identical gathers, and
decode attention over the restored blocks matches the oracle within the parity
tolerance.  An incompatible storage identity is rejected before any device work;
a buffer too small is rejected on the host; a row outside the pool sets the
device error word."""
import numpy as np
import pytest

import paged_kv_cache_split_gb300 as pkv
from paged_kv_cache_split_gb300 import workloads as wl
from tests.harness import FMT, bf16_dev_to_f64, compare, fill, make_pools, to_dev_bf16, to_dev_i32

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(autouse=True)
def _needs_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _workload(fmt):
    if fmt == wl.FMT_BF16:
        return wl.qwen3_0_6b(n_layers=2, B=3, L=700)
    if fmt == wl.FMT_K4V4:
        return wl.qwen3_1_7b_k4v4(B=2, L=900)
    return wl.llama_1b(fmt, B=4, lo=40, hi=600)


@pytest.mark.parametrize("fmt", [wl.FMT_BF16, wl.FMT_K4V4, wl.FMT_K8V4, wl.FMT_K8V8])
def test_export_import_roundtrip(fmt):
    w = _workload(fmt)
    g, o, ol = make_pools(w)
    fill(w, g, o, ol)
    bt = w.block_table()
    rows = np.concatenate([bt[b][: wl.nblocks(w.lens[b])] for b in range(w.B)]).astype(np.int32)
    rec = g.export_blocks(to_dev_i32(rows))
    want = o.export_blocks(rows)
    assert rec.shape == want.shape and g.block_record_bytes() == o.record_bytes
    assert np.array_equal(rec.cpu().numpy(), want)

    # restore into a second pool, at rows of its own (a reversed permutation)
    g2 = pkv.Pool(w.n_layers, w.Hkv, w.D, FMT[w.fmt], hadamard_seed=w.hadamard_seed,
                  max_slabs=(rows.size + 31) // 32 + 4)
    g2.reserve_rows(rows.size)
    new_rows = rows.size - 1 - np.arange(rows.size, dtype=np.int32)
    g2.import_blocks(g.config(), to_dev_i32(new_rows), rec)
    assert np.array_equal(g2.export_blocks(to_dev_i32(new_rows)).cpu().numpy(), want)

    # the same contexts through the remapped block tables
    remap = dict(zip(rows.tolist(), new_rows.tolist()))
    bt2 = np.full_like(bt, -1)
    for b in range(w.B):
        n = wl.nblocks(w.lens[b])
        bt2[b][:n] = [remap[int(r)] for r in bt[b][:n]]
    for layer in range(w.n_layers):
        for b in range(w.B):
            L, n = w.lens[b], wl.nblocks(w.lens[b])
            a = [t.cpu().numpy() for t in g.gather_visible(layer, to_dev_i32(bt[b][:n]), L)]
            c = [t.cpu().numpy() for t in g2.gather_visible(layer, to_dev_i32(bt2[b][:n]), L)]
            for x, y in zip(a, c):
                assert np.array_equal(x, y)
        out = g2.paged_decode_attention(layer, to_dev_bf16(w.q(layer)), to_dev_i32(bt2), to_dev_i32(w.ctx()),
                                        w.scale, max_ctx=max(w.lens))
        ref = o.decode_attention(ol.index(layer), w.q(layer), bt, w.ctx(), w.scale)
        compare(bf16_dev_to_f64(out), ref, f"restored {w.name} layer {layer}")
    assert g.check_errors() == 0 and g2.check_errors() == 0


def test_import_rejects_other_identities_before_any_write():
    w = wl.llama_1b(wl.FMT_K8V4, B=2, lo=40, hi=100)
    g, o, ol = make_pools(w)
    fill(w, g, o, ol)
    rows = to_dev_i32([0, 1])
    rec = g.export_blocks(rows)
    before = g.export_blocks(rows).cpu().numpy()
    for change in [dict(format=wl.FMT_K8V8), dict(hadamard_seed=w.hadamard_seed + 1), dict(n_layers=w.n_layers + 1),
                   dict(head_dim=128), dict(n_kv_heads=4)]:
        ident = g.config()
        for k, v in change.items():
            setattr(ident, k, v)
        with pytest.raises(pkv.PkvError) as e:
            g.import_blocks(ident, rows, torch.zeros_like(rec))
        assert e.value.status == pkv.PKV_ERR_FORMAT
    assert np.array_equal(g.export_blocks(rows).cpu().numpy(), before)
    small = torch.empty((1, g.block_record_bytes()), dtype=torch.uint8, device="cuda")
    with pytest.raises(pkv.PkvError) as e:
        g.export_blocks(rows, out=small)
    assert e.value.status == pkv.PKV_ERR_RANGE
    g.export_blocks(to_dev_i32([0, 1 << 20]))
    assert g.check_errors() & 1
