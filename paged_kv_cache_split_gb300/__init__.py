"""Python binding of libpkv.so: paged decode attention over a chunked-slab KV pool on
GB300 (sm_103a).

Argument marshalling only: every step runs in the library's CUDA kernels.  PyTorch
supplies device memory and streams (tensors are passed by ``data_ptr()`` and the
current stream's handle).  There is no CPU fallback: without the compiled library
every call raises.  Names follow the C ABI in ``include/pkv.h`` without the ``pkv_``
prefix.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpkv.so")

FORMATS = {"bf16": 0, "k4v4": 1, "k8v4": 2, "k8v8": 3}
FORMAT_NAMES = {v: k for k, v in FORMATS.items()}
KIND_K, KIND_V, KIND_KMETA, KIND_VMETA = 0, 1, 2, 3

STATUS = {0: "ok", -1: "invalid argument", -2: "allocation failed", -3: "CUDA error",
          -4: "format mismatch", -5: "out of range", -6: "device error word set"}
PKV_OK, PKV_ERR_INVALID, PKV_ERR_OOM, PKV_ERR_CUDA, PKV_ERR_FORMAT, PKV_ERR_RANGE, PKV_ERR_DEVICE = \
    0, -1, -2, -3, -4, -5, -6
ERR_ROW, ERR_CTX, ERR_SLOT, ERR_TIMEOUT = 1, 2, 4, 8


class PkvError(RuntimeError):
    def __init__(self, status: int, what: str, detail: str = ""):
        self.status = status
        msg = f"{what}: {STATUS.get(status, status)}"
        if detail:
            msg += f" ({detail})"
        super().__init__(msg)


class PoolConfig(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("slab_blocks", ctypes.c_int32), ("group_size", ctypes.c_int32),
                ("format", ctypes.c_int32), ("max_slabs", ctypes.c_int32), ("hadamard_seed", ctypes.c_uint64)]


class Stats(ctypes.Structure):
    _fields_ = [("n_slabs", ctypes.c_int32), ("n_kinds", ctypes.c_int32),
                ("slab_append_events", ctypes.c_int64), ("rows_capacity", ctypes.c_int64),
                ("rows_in_use", ctypes.c_int64), ("bytes_reserved", ctypes.c_int64),
                ("row_bytes", ctypes.c_int64 * 4)]

    def as_dict(self):
        return {"n_slabs": self.n_slabs, "n_kinds": self.n_kinds, "slab_append_events": self.slab_append_events,
                "rows_capacity": self.rows_capacity, "rows_in_use": self.rows_in_use,
                "bytes_reserved": self.bytes_reserved, "row_bytes": list(self.row_bytes)}


ALLOC_FN = ctypes.CFUNCTYPE(ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p)
RELEASE_FN = ctypes.CFUNCTYPE(None, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p)


class Request(ctypes.Structure):
    _fields_ = [("new_blocks", ctypes.c_int32), ("B", ctypes.c_int32), ("Hq", ctypes.c_int32),
                ("n_q", ctypes.c_int32), ("max_blocks", ctypes.c_int32)]


class Price(ctypes.Structure):
    _fields_ = [("slabs_to_append", ctypes.c_int32), ("free_rows", ctypes.c_int64),
                ("storage_bytes", ctypes.c_uint64), ("page_bytes", ctypes.c_uint64),
                ("fixed_bytes", ctypes.c_uint64), ("workspace_bytes", ctypes.c_uint64)]

    def as_dict(self):
        return {k: int(getattr(self, k)) for k, _ in self._fields_}


class Allocator(ctypes.Structure):
    _fields_ = [("alloc", ALLOC_FN), ("release", RELEASE_FN), ("ctx", ctypes.c_void_p)]


# Every symbol of include/pkv.h with its ctypes signature.
_P, _I, _I64, _SZ, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
SIGNATURES = {
    "pkv_pool_create": ([ctypes.POINTER(PoolConfig), ctypes.POINTER(Allocator), _P, ctypes.POINTER(_P)], _I),
    "pkv_pool_destroy": ([_P], None),
    "pkv_append_slab": ([_P, _I, _P], _I),
    "pkv_alloc_rows": ([_P, _I, _P, _P], _I),
    "pkv_retain_row": ([_P, ctypes.c_int32], _I),
    "pkv_release_row": ([_P, ctypes.c_int32], _I),
    "pkv_slab_runs": ([_P, _I, _I, _P], _I),
    "pkv_write_block": ([_P, _I, _I, _P, _P, _P, _P, _P], _I),
    "pkv_copy_on_write_block": ([_P, _I, _P, _P, _P], _I),
    "pkv_gather_visible": ([_P, _I, _P, _I, _P, _P, _P, _P, _P], _I),
    "pkv_decode_workspace_bytes": ([_P, _I, _I, _I, ctypes.POINTER(_SZ)], _I),
    "pkv_paged_decode_attention": ([_P, _I, _I, _I, _P, _P, _I, _P, _I, _F, _P, _P, _SZ, _P], _I),
    "pkv_paged_decode_attention_noalloc": ([_P, _I, _I, _I, _P, _P, _I, _P, _I, _F, _P, _P], _I),
    "pkv_decode_set_ctas": ([_P, _I], _I),
    "pkv_pool_stats": ([_P, ctypes.POINTER(Stats)], _I),
    "pkv_slab_address": ([_P, _I, _I, _I, ctypes.POINTER(_P)], _I),
    "pkv_pool_check_identity": ([_P, ctypes.POINTER(PoolConfig)], _I),
    "pkv_price_request": ([_P, ctypes.POINTER(Request), ctypes.POINTER(Price)], _I),
    "pkv_pool_check_errors": ([_P, _P, ctypes.POINTER(ctypes.c_int32)], _I),
    "pkv_pool_get_config": ([_P, ctypes.POINTER(PoolConfig)], _I),
    "pkv_prefill_workspace_bytes": ([_P, _I, _I, _I, _I, ctypes.POINTER(_SZ)], _I),
    "pkv_paged_prefill_attention": ([_P, _I, _I, _I, _I, _P, _P, _I, _P, _I, _F, _P, _P, _SZ, _P], _I),
    "pkv_block_record_bytes": ([_P, ctypes.POINTER(_SZ)], _I),
    "pkv_export_blocks": ([_P, _I, _P, _P, _SZ, _P], _I),
    "pkv_import_blocks": ([_P, ctypes.POINTER(PoolConfig), _I, _P, _P, _SZ, _P], _I),
    "pkv_status_string": ([_I], ctypes.c_char_p),
    "pkv_last_error": ([], ctypes.c_char_p),
}

_lock = threading.Lock()
_lib_handle = None


def lib():
    """The loaded libpkv.so (raises if it has not been built)."""
    global _lib_handle
    with _lock:
        if _lib_handle is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                   "`python -m paged_kv_cache_split_gb300.build` (nvcc, sm_103a)")
            h = ctypes.CDLL(LIB_PATH)
            for name, (args, res) in SIGNATURES.items():
                fn = getattr(h, name)
                fn.argtypes = args
                fn.restype = res
            _lib_handle = h
        return _lib_handle


def _check(status: int, what: str):
    if status != PKV_OK:
        detail = ""
        if status == PKV_ERR_CUDA:
            detail = lib().pkv_last_error().decode(errors="replace")
        raise PkvError(status, what, detail)


def _torch():
    import torch
    return torch


def _stream(stream=None) -> int:
    torch = _torch()
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dev(t, dtype, name: str, shape=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t.data_ptr()


def slab_runs(rows, slab_blocks: int = 32) -> np.ndarray:
    """Start index of each maximal same-slab run of a block-table row list (host)."""
    r = np.ascontiguousarray(rows, np.int32)
    out = np.zeros(max(1, r.size), np.int32)
    n = lib().pkv_slab_runs(r.ctypes.data_as(_P), r.size, slab_blocks, out.ctypes.data_as(_P))
    if n < 0:
        raise PkvError(PKV_ERR_INVALID, "slab_runs")
    return out[:n].copy()


def make_config(n_layers: int, n_kv_heads: int, head_dim: int, format="bf16", hadamard_seed: int = 0,
                slab_blocks: int = 32, max_slabs: int = 1024, block_size: int = 32, group_size: int = 32):
    fmt = FORMATS[format] if isinstance(format, str) else int(format)
    return PoolConfig(n_layers, n_kv_heads, head_dim, block_size, slab_blocks, group_size, fmt, max_slabs,
                      hadamard_seed & (2**64 - 1))


class Pool:
    """A chunked-slab KV pool on the current CUDA device (see pkv_pool_create)."""

    def __init__(self, n_layers: int, n_kv_heads: int, head_dim: int, format="bf16", hadamard_seed: int = 0,
                 slab_blocks: int = 32, max_slabs: int = 1024, allocator: Optional[Allocator] = None,
                 stream=None, group_size: int = 32):
        self._lib = lib()
        self.cfg = make_config(n_layers, n_kv_heads, head_dim, format, hadamard_seed, slab_blocks, max_slabs,
                               group_size=group_size)
        self.n_layers, self.n_kv_heads, self.head_dim = n_layers, n_kv_heads, head_dim
        self.format = FORMAT_NAMES[self.cfg.format]
        self.slab_blocks = slab_blocks
        self._allocator = allocator  # keep callbacks alive
        h = _P()
        st = self._lib.pkv_pool_create(ctypes.byref(self.cfg), ctypes.byref(allocator) if allocator else None,
                                       _stream(stream), ctypes.byref(h))
        _check(st, "pool_create")
        self._h = h
        self._ws = {}
        s = self.stats()
        self.row_bytes = s["row_bytes"][: s["n_kinds"]]

    # -- lifetime ------------------------------------------------------------
    def close(self):
        if getattr(self, "_h", None):
            self._lib.pkv_pool_destroy(self._h)
            self._h = None
            self._ws = {}

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        return self._h

    # -- growth and rows -----------------------------------------------------
    def append_slab(self, n_slabs: int = 1, stream=None):
        _check(self._lib.pkv_append_slab(self._h, n_slabs, _stream(stream)), "append_slab")

    def reserve_rows(self, rows: int, stream=None):
        """Append slabs until the pool has at least `rows` rows."""
        have = self.stats()["rows_capacity"]
        if rows > have:
            self.append_slab(-(-(rows - have) // self.slab_blocks), stream)

    def alloc_rows(self, n: int, stream=None) -> np.ndarray:
        out = np.zeros(max(1, n), np.int32)
        _check(self._lib.pkv_alloc_rows(self._h, n, out.ctypes.data_as(_P), _stream(stream)), "alloc_rows")
        return out[:n].copy()

    def retain_row(self, row: int):
        _check(self._lib.pkv_retain_row(self._h, int(row)), "retain_row")

    def release_row(self, row: int):
        _check(self._lib.pkv_release_row(self._h, int(row)), "release_row")

    # -- data movement -------------------------------------------------------
    def write_block(self, layer: int, rows, slots, k, v, stream=None):
        torch = _torch()
        n = int(rows.numel())
        shape = (n, self.n_kv_heads, self.head_dim)
        _check(self._lib.pkv_write_block(self._h, layer, n, _dev(rows, torch.int32, "rows"),
                                         _dev(slots, torch.int32, "slots"), _dev(k, torch.bfloat16, "k", shape),
                                         _dev(v, torch.bfloat16, "v", shape), _stream(stream)), "write_block")

    def copy_on_write_block(self, src_rows, dst_rows, stream=None):
        torch = _torch()
        n = int(src_rows.numel())
        if int(dst_rows.numel()) != n:
            raise ValueError("src_rows and dst_rows differ in length")
        _check(self._lib.pkv_copy_on_write_block(self._h, n, _dev(src_rows, torch.int32, "src_rows"),
                                                 _dev(dst_rows, torch.int32, "dst_rows"), _stream(stream)),
               "copy_on_write_block")

    def gather_visible(self, layer: int, bt_row, ctx_len: int, stream=None):
        """Dense [Hkv, ctx, row_bytes] uint8 tensors (K, V[, K meta, V meta])."""
        torch = _torch()
        outs = [torch.empty((self.n_kv_heads, ctx_len, rb), dtype=torch.uint8, device=bt_row.device)
                for rb in self.row_bytes]
        ptrs = [o.data_ptr() for o in outs] + [None] * (4 - len(outs))
        _check(self._lib.pkv_gather_visible(self._h, layer, _dev(bt_row, torch.int32, "bt_row"), ctx_len,
                                            *ptrs, _stream(stream)), "gather_visible")
        return outs

    # -- block records (export / import) ---------------------------------------
    def config(self) -> PoolConfig:
        """The pool's configuration (storage identity, layer count, table size)."""
        c = PoolConfig()
        _check(self._lib.pkv_pool_get_config(self._h, ctypes.byref(c)), "pool_get_config")
        return c

    def block_record_bytes(self) -> int:
        n = _SZ()
        _check(self._lib.pkv_block_record_bytes(self._h, ctypes.byref(n)), "block_record_bytes")
        return int(n.value)

    def export_blocks(self, rows, out=None, stream=None):
        """[n, record_bytes] uint8 device tensor with the records of blocks `rows`."""
        torch = _torch()
        n, rec = int(rows.numel()), self.block_record_bytes()
        if out is None:
            out = torch.empty((n, rec), dtype=torch.uint8, device=rows.device)
        _check(self._lib.pkv_export_blocks(self._h, n, _dev(rows, torch.int32, "rows"),
                                           _dev(out, torch.uint8, "out"), out.numel(), _stream(stream)),
               "export_blocks")
        return out

    def import_blocks(self, identity: PoolConfig, rows, records, stream=None):
        """Write records (layout of export_blocks) into blocks `rows`; raises PkvError
        (status PKV_ERR_FORMAT) before any device work if `identity` differs."""
        torch = _torch()
        _check(self._lib.pkv_import_blocks(self._h, ctypes.byref(identity), int(rows.numel()),
                                           _dev(rows, torch.int32, "rows"), _dev(records, torch.uint8, "records"),
                                           records.numel(), _stream(stream)), "import_blocks")

    # -- attention -----------------------------------------------------------
    def decode_workspace_bytes(self, B: int, Hq: int, max_ctx: int = 0) -> int:
        n = _SZ()
        _check(self._lib.pkv_decode_workspace_bytes(self._h, B, Hq, max_ctx, ctypes.byref(n)),
               "decode_workspace_bytes")
        return int(n.value)

    def workspace(self, B: int, Hq: int, device=None):
        """A zero-filled workspace tensor for (B, Hq), cached on the pool."""
        torch = _torch()
        nbytes = self.decode_workspace_bytes(B, Hq)
        key = (B, Hq)
        ws = self._ws.get(key)
        if ws is None or ws.numel() < nbytes:
            ws = torch.zeros(nbytes, dtype=torch.uint8, device=device or "cuda")
            self._ws[key] = ws
        return ws

    def decode_set_ctas(self, n_ctas: int):
        _check(self._lib.pkv_decode_set_ctas(self._h, n_ctas), "decode_set_ctas")
        self._ws = {}

    def paged_decode_attention(self, layer: int, q, block_table, ctx_lens, scale: float, max_ctx: int = 0,
                               out=None, workspace=None, stream=None):
        torch = _torch()
        B, Hq, D = q.shape
        if D != self.head_dim:
            raise ValueError(f"q head_dim {D} != pool head_dim {self.head_dim}")
        if block_table.dim() != 2 or block_table.shape[0] != B:
            raise ValueError("block_table must be [B, max_blocks]")
        if out is None:
            out = torch.empty_like(q)
        if workspace is None:
            workspace = self.workspace(B, Hq, q.device)
        _check(self._lib.pkv_paged_decode_attention(
            self._h, layer, B, Hq, _dev(q, torch.bfloat16, "q"), _dev(block_table, torch.int32, "block_table"),
            int(block_table.shape[1]), _dev(ctx_lens, torch.int32, "ctx_lens", (B,)), int(max_ctx), float(scale),
            _dev(out, torch.bfloat16, "out", (B, Hq, D)), workspace.data_ptr(), int(workspace.numel()),
            _stream(stream)), "paged_decode_attention")
        return out

    def prefill_workspace_bytes(self, B: int, n_q: int, Hq: int, max_blocks: int) -> int:
        n = _SZ()
        _check(self._lib.pkv_prefill_workspace_bytes(self._h, B, n_q, Hq, max_blocks, ctypes.byref(n)),
               "prefill_workspace_bytes")
        return int(n.value)

    def paged_prefill_attention(self, layer: int, q, block_table, ctx_lens, scale: float, max_ctx: int = 0,
                                out=None, workspace=None, stream=None):
        """Causal attention of the last n_q tokens of each sequence: q [B, n_q, Hq, D] bf16."""
        torch = _torch()
        B, n_q, Hq, D = q.shape
        if D != self.head_dim:
            raise ValueError(f"q head_dim {D} != pool head_dim {self.head_dim}")
        if block_table.dim() != 2 or block_table.shape[0] != B:
            raise ValueError("block_table must be [B, max_blocks]")
        if out is None:
            out = torch.empty_like(q)
        mb = int(block_table.shape[1])
        if workspace is None:
            n = self.prefill_workspace_bytes(B, n_q, Hq, mb)
            workspace = torch.zeros(n, dtype=torch.uint8, device=q.device)
        _check(self._lib.pkv_paged_prefill_attention(
            self._h, layer, B, n_q, Hq, _dev(q, torch.bfloat16, "q"), _dev(block_table, torch.int32, "block_table"), mb,
            _dev(ctx_lens, torch.int32, "ctx_lens", (B,)), int(max_ctx), float(scale),
            _dev(out, torch.bfloat16, "out", (B, n_q, Hq, D)), workspace.data_ptr(), int(workspace.numel()),
            _stream(stream)), "paged_prefill_attention")
        return out

    def paged_decode_attention_noalloc(self, layer: int, q, block_table, ctx_lens, scale: float,
                                       max_ctx: int = 0, out=None, stream=None):
        """Decode attention with no workspace argument: the library's fixed device
        scratch array is used instead (see pkv_paged_decode_attention_noalloc)."""
        torch = _torch()
        B, Hq, D = q.shape
        if out is None:
            out = torch.empty_like(q)
        _check(self._lib.pkv_paged_decode_attention_noalloc(
            self._h, layer, B, Hq, _dev(q, torch.bfloat16, "q"), _dev(block_table, torch.int32, "block_table"),
            int(block_table.shape[1]), _dev(ctx_lens, torch.int32, "ctx_lens", (B,)), int(max_ctx), float(scale),
            _dev(out, torch.bfloat16, "out", (B, Hq, D)), _stream(stream)), "paged_decode_attention_noalloc")
        return out

    # -- introspection -------------------------------------------------------
    def stats(self) -> dict:
        s = Stats()
        _check(self._lib.pkv_pool_stats(self._h, ctypes.byref(s)), "pool_stats")
        return s.as_dict()

    def slab_address(self, layer: int, kind: int, slab: int) -> int:
        a = _P()
        _check(self._lib.pkv_slab_address(self._h, layer, kind, slab, ctypes.byref(a)), "slab_address")
        return int(a.value or 0)

    def price_request(self, new_blocks: int, B: int, Hq: int, n_q: int = 1, max_blocks: int = 0) -> dict:
        """Admission price of a request (see pkv_price_request): slabs to append, free
        rows, and the storage, page, fixed and workspace bytes."""
        req = Request(int(new_blocks), int(B), int(Hq), int(n_q), int(max_blocks))
        out = Price()
        _check(self._lib.pkv_price_request(self._h, ctypes.byref(req), ctypes.byref(out)), "price_request")
        return out.as_dict()

    def check_identity(self, cfg: PoolConfig) -> bool:
        st = self._lib.pkv_pool_check_identity(self._h, ctypes.byref(cfg))
        if st == PKV_ERR_FORMAT:
            return False
        _check(st, "pool_check_identity")
        return True

    def check_errors(self, stream=None) -> int:
        """Synchronise, then return and clear the device error word (0 if clean)."""
        w = ctypes.c_int32(0)
        st = self._lib.pkv_pool_check_errors(self._h, _stream(stream), ctypes.byref(w))
        if st not in (PKV_OK, PKV_ERR_DEVICE):
            _check(st, "pool_check_errors")
        return int(w.value)


def pool_create(*args, **kw) -> Pool:
    return Pool(*args, **kw)
