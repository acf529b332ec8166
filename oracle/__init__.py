"""The oracle: a plain, slow CPU (FP64) statement of paged decode attention over a
chunked-slab KV pool, in native bf16 and in the packed K4/V4, K8/V4, K8/V8 formats.

TEST INFRASTRUCTURE ONLY.  ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` are its only users; the
GPU library never imports, links or calls it, and the two share no code.  The
arithmetic lives in ``pkv_oracle.c`` (compiled without FMA contraction); this module
only marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

FMT_BF16, FMT_K4V4, FMT_K8V4, FMT_K8V8 = 0, 1, 2, 3
FORMAT_BITS = {FMT_BF16: (16, 16), FMT_K4V4: (4, 4), FMT_K8V4: (8, 4), FMT_K8V8: (8, 8)}


def build(force: bool = False) -> str:
    """Compile pkv_oracle.c into liboracle.so (gcc, no FMA contraction)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, u64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_uint64, ctypes.c_double
        lib.oracle_splitmix64.argtypes = [u64]
        lib.oracle_splitmix64.restype = u64
        lib.oracle_hadamard_signs.argtypes = [u64, i32, P]
        lib.oracle_hadamard_entry.argtypes = [i32, i32, i32]
        lib.oracle_hadamard_entry.restype = dbl
        lib.oracle_rotate_k.argtypes = [P, i32, P, P]
        lib.oracle_rotate_k.restype = i32
        lib.oracle_rotate_q.argtypes = [P, i32, P, P]
        lib.oracle_quantize.argtypes = [P, i32, i32, i32, P, P]
        lib.oracle_quantize.restype = i32
        lib.oracle_dequantize.argtypes = [P, P, i32, i32, i32, P]
        lib.oracle_dequantize.restype = i32
        lib.oracle_pool_new.argtypes = [i32, i32, i32, i32, u64, i32, i32, i32]
        lib.oracle_pool_new.restype = P
        lib.oracle_pool_free.argtypes = [P]
        lib.oracle_pool_reserve_rows.argtypes = [P, i64]
        lib.oracle_pool_reserve_rows.restype = i32
        lib.oracle_pool_rows.argtypes = [P]
        lib.oracle_pool_rows.restype = i64
        lib.oracle_pool_inexact_rotations.argtypes = [P]
        lib.oracle_pool_inexact_rotations.restype = ctypes.c_long
        lib.oracle_write_block.argtypes = [P, i32, i32, P, P, P, P]
        lib.oracle_write_block.restype = i32
        lib.oracle_copy_block.argtypes = [P, i32, P, P]
        lib.oracle_copy_block.restype = i32
        lib.oracle_slab_runs.argtypes = [P, i32, i32, P]
        lib.oracle_slab_runs.restype = i32
        lib.oracle_gather_visible.argtypes = [P, i32, P, i32, P, P, P, P]
        lib.oracle_gather_visible.restype = i32
        lib.oracle_decode_attention.argtypes = [P, i32, i32, i32, P, P, i32, P, dbl, P, i32]
        lib.oracle_decode_attention.restype = i32
        lib.oracle_read_block.argtypes = [P, i32, i32, i32, P]
        lib.oracle_read_block.restype = i32
        lib.oracle_read_slab.argtypes = [P, i32, i32, i32, P]
        lib.oracle_read_slab.restype = i32
        lib.oracle_prefill_attention.argtypes = [P, i32, i32, i32, i32, P, P, i32, P, dbl, P]
        lib.oracle_prefill_attention.restype = i32
        lib.oracle_record_bytes.argtypes = [P]
        lib.oracle_record_bytes.restype = ctypes.c_size_t
        lib.oracle_export_blocks.argtypes = [P, i32, P, P]
        lib.oracle_export_blocks.restype = i32
        lib.oracle_import_blocks.argtypes = [P, i32, P, P]
        lib.oracle_import_blocks.restype = i32
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


class OracleError(RuntimeError):
    pass


def _check(rc: int, what: str):
    if rc != 0:
        raise OracleError(f"{what} failed with status {rc}")


# ---- scalar primitives ------------------------------------------------------

def splitmix64(x: int) -> int:
    return int(_load().oracle_splitmix64(x & (2**64 - 1)))


def hadamard_signs(seed: int, D: int) -> np.ndarray:
    s = np.empty(D, np.float64)
    _load().oracle_hadamard_signs(seed & (2**64 - 1), D, _ptr(s))
    return s


def hadamard_matrix(D: int) -> np.ndarray:
    lib = _load()
    return np.array([[lib.oracle_hadamard_entry(i, j, D) for j in range(D)] for i in range(D)])


def rotate_k(k_bf16: np.ndarray, signs: np.ndarray):
    """Rotated K row (float32) and whether its FP64 sum was exact."""
    k = np.ascontiguousarray(k_bf16, np.uint16)
    out = np.empty(k.shape[-1], np.float32)
    ok = _load().oracle_rotate_k(_ptr(k), k.shape[-1], _ptr(np.ascontiguousarray(signs, np.float64)), _ptr(out))
    return out, bool(ok)


def rotate_q(q: np.ndarray, signs: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q, np.float64)
    out = np.empty_like(q)
    _load().oracle_rotate_q(_ptr(q), q.shape[-1], _ptr(np.ascontiguousarray(signs, np.float64)), _ptr(out))
    return out


def quantize(x: np.ndarray, bits: int, group: int = 32):
    """(packed codes uint8, meta float32 [D/group, 2]) of one row."""
    x = np.ascontiguousarray(x, np.float32)
    D = x.shape[-1]
    codes = np.empty(D * bits // 8, np.uint8)
    meta = np.empty((D // group, 2), np.float32)
    _check(_load().oracle_quantize(_ptr(x), D, bits, group, _ptr(codes), _ptr(meta)), "quantize")
    return codes, meta


def dequantize(codes: np.ndarray, meta: np.ndarray, D: int, bits: int, group: int = 32) -> np.ndarray:
    out = np.empty(D, np.float64)
    _check(_load().oracle_dequantize(_ptr(np.ascontiguousarray(codes, np.uint8)),
                                     _ptr(np.ascontiguousarray(meta, np.float32)), D, bits, group, _ptr(out)),
           "dequantize")
    return out


def slab_runs(rows: np.ndarray, slab_blocks: int = 32) -> np.ndarray:
    rows = np.ascontiguousarray(rows, np.int32)
    starts = np.empty(max(1, rows.size), np.int32)
    n = _load().oracle_slab_runs(_ptr(rows), rows.size, slab_blocks, _ptr(starts))
    return starts[:n].copy()


# ---- pool image --------------------------------------------------------------

class OraclePool:
    """Host image of a chunked-slab pool (every layer, K/V and, when packed, meta)."""

    def __init__(self, n_layers: int, n_kv_heads: int, head_dim: int, fmt: int = FMT_BF16,
                 seed: int = 0, block_size: int = 32, slab_blocks: int = 32, group_size: int = 32):
        self._lib = _load()
        self.n_layers, self.n_kv_heads, self.head_dim = n_layers, n_kv_heads, head_dim
        self.fmt, self.seed = fmt, seed
        self.block_size, self.slab_blocks, self.group_size = block_size, slab_blocks, group_size
        self._h = self._lib.oracle_pool_new(n_layers, n_kv_heads, head_dim, fmt, seed & (2**64 - 1),
                                            block_size, slab_blocks, group_size)
        if not self._h:
            raise OracleError("oracle_pool_new rejected the configuration")
        kb, vb = FORMAT_BITS[fmt]
        self.row_bytes = [head_dim * kb // 8, head_dim * vb // 8]
        if fmt != FMT_BF16:
            self.row_bytes += [head_dim // group_size * 8] * 2

    def close(self):
        if self._h:
            self._lib.oracle_pool_free(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def rows(self) -> int:
        return int(self._lib.oracle_pool_rows(self._h))

    @property
    def inexact_rotations(self) -> int:
        return int(self._lib.oracle_pool_inexact_rotations(self._h))

    def reserve_rows(self, rows: int):
        _check(self._lib.oracle_pool_reserve_rows(self._h, rows), "reserve_rows")

    def write_block(self, layer: int, rows, slots, k_bf16: np.ndarray, v_bf16: np.ndarray):
        rows = np.ascontiguousarray(rows, np.int32)
        slots = np.ascontiguousarray(slots, np.int32)
        k = np.ascontiguousarray(k_bf16, np.uint16)
        v = np.ascontiguousarray(v_bf16, np.uint16)
        n = rows.size
        assert k.shape == (n, self.n_kv_heads, self.head_dim) and v.shape == k.shape
        _check(self._lib.oracle_write_block(self._h, layer, n, _ptr(rows), _ptr(slots), _ptr(k), _ptr(v)),
               "write_block")

    def copy_block(self, src, dst):
        src = np.ascontiguousarray(src, np.int32)
        dst = np.ascontiguousarray(dst, np.int32)
        _check(self._lib.oracle_copy_block(self._h, src.size, _ptr(src), _ptr(dst)), "copy_block")

    def gather_visible(self, layer: int, bt_row, ctx: int):
        """Dense [Hkv, ctx, row_bytes] uint8 arrays for K, V (and K/V meta if packed)."""
        bt_row = np.ascontiguousarray(bt_row, np.int32)
        outs = [np.zeros((self.n_kv_heads, ctx, rb), np.uint8) for rb in self.row_bytes]
        while len(outs) < 4:
            outs.append(np.zeros(1, np.uint8))
        _check(self._lib.oracle_gather_visible(self._h, layer, _ptr(bt_row), ctx, *[_ptr(o) for o in outs]),
               "gather_visible")
        return outs[: len(self.row_bytes)]

    def read_block(self, layer: int, kind: int, row: int) -> np.ndarray:
        out = np.zeros(self.block_size * self.n_kv_heads * self.row_bytes[kind], np.uint8)
        _check(self._lib.oracle_read_block(self._h, layer, kind, row, _ptr(out)), "read_block")
        return out

    def prefill_attention(self, layer: int, q_bf16: np.ndarray, bt: np.ndarray, ctx, scale: float) -> np.ndarray:
        """[B, n_q, Hq, D] float64 causal attention of the last n_q tokens of each sequence."""
        q = np.ascontiguousarray(q_bf16, np.uint16)
        B, n_q, Hq, D = q.shape
        bt = np.ascontiguousarray(bt, np.int32)
        ctx = np.ascontiguousarray(ctx, np.int32)
        out = np.zeros((B, n_q, Hq, D), np.float64)
        _check(self._lib.oracle_prefill_attention(self._h, layer, B, n_q, Hq, _ptr(q), _ptr(bt), bt.shape[1],
                                                  _ptr(ctx), float(scale), _ptr(out)), "prefill_attention")
        return out

    @property
    def record_bytes(self) -> int:
        return int(self._lib.oracle_record_bytes(self._h))

    def export_blocks(self, rows) -> np.ndarray:
        """[n, record_bytes] uint8 records of blocks `rows` (layer-major, then K, V, K meta, V meta)."""
        rows = np.ascontiguousarray(rows, np.int32)
        out = np.zeros((rows.size, self.record_bytes), np.uint8)
        _check(self._lib.oracle_export_blocks(self._h, rows.size, _ptr(rows), _ptr(out)), "export_blocks")
        return out

    def import_blocks(self, rows, records: np.ndarray):
        rows = np.ascontiguousarray(rows, np.int32)
        rec = np.ascontiguousarray(records, np.uint8)
        assert rec.size == rows.size * self.record_bytes
        _check(self._lib.oracle_import_blocks(self._h, rows.size, _ptr(rows), _ptr(rec)), "import_blocks")

    def read_slab(self, layer: int, kind: int, slab: int) -> np.ndarray:
        n = self.slab_blocks * self.block_size * self.n_kv_heads * self.row_bytes[kind]
        out = np.zeros(n, np.uint8)
        _check(self._lib.oracle_read_slab(self._h, layer, kind, slab, _ptr(out)), "read_slab")
        return out

    def decode_attention(self, layer: int, q_bf16: np.ndarray, bt: np.ndarray, ctx, scale: float,
                         n_threads: int = 0) -> np.ndarray:
        """[B, Hq, D] float64 attention output."""
        q = np.ascontiguousarray(q_bf16, np.uint16)
        bt = np.ascontiguousarray(bt, np.int32)
        ctx = np.ascontiguousarray(ctx, np.int32)
        B, Hq, D = q.shape
        out = np.zeros((B, Hq, D), np.float64)
        _check(self._lib.oracle_decode_attention(self._h, layer, B, Hq, _ptr(q), _ptr(bt), bt.shape[1],
                                                 _ptr(ctx), float(scale), _ptr(out), n_threads),
               "decode_attention")
        return out
