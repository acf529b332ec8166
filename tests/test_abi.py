"""The C-ABI library loads and exports every symbol include/pkv.h declares; host-only
entry points work without a GPU.  CPU only (no compute call touches a device)."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import paged_kv_cache_split_gb300 as pkv
from paged_kv_cache_split_gb300 import build as pkv_build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pkv.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    pkv_build.build()
    return pkv.lib()


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ["pkv_pool_create", "pkv_append_slab", "pkv_write_block", "pkv_copy_on_write_block",
                     "pkv_gather_visible", "pkv_paged_decode_attention"]:
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    assert set(names) == set(pkv.SIGNATURES), "binding signatures must cover the header exactly"


def test_slab_runs_host_entry_point(lib):
    rng = np.random.default_rng(0)
    for _ in range(100):
        rows = rng.integers(0, 300, int(rng.integers(1, 80))).astype(np.int32)
        sb = int(rng.choice([1, 8, 32, 64]))
        assert np.array_equal(pkv.slab_runs(rows, sb), oracle.slab_runs(rows, sb))
    assert pkv.slab_runs(np.zeros(0, np.int32)).size == 0


def test_status_strings(lib):
    for st in range(-6, 1):
        assert lib.pkv_status_string(st)


def test_invalid_config_rejected_before_device_use(lib):
    cfg = pkv.make_config(1, 8, 96)  # head_dim 96 is unsupported
    h = ctypes.c_void_p()
    assert lib.pkv_pool_create(ctypes.byref(cfg), None, None, ctypes.byref(h)) == pkv.PKV_ERR_INVALID
    assert not h.value


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(pkv, "_lib_handle", None)
    monkeypatch.setattr(pkv, "LIB_PATH", str(tmp_path / "libpkv.so"))
    with pytest.raises(RuntimeError, match="is missing"):
        pkv.lib()
    with pytest.raises(RuntimeError, match="is missing"):
        pkv.Pool(1, 1, 64, "bf16")


def test_no_cpu_path_without_a_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    with pytest.raises(RuntimeError):  # PkvError is a RuntimeError too
        pkv.Pool(1, 1, 64, "bf16")
