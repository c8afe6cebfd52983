"""Python binding of libpagedattn (paged GQA attention for GB300).

Argument marshalling only: torch tensors become device pointers and sizes for the
C ABI in include/pagedattn.h; every step of the computation runs in the CUDA
kernels of libpagedattn.so.  There is no CPU or PyTorch fallback -- if the
library is not built, loading it raises.

Names follow the C ABI: pa_kv_append, pa_decode, pa_decode_splitkv,
pa_combine, pa_prefill_chunked, pa_device_status.  Tensors must be CUDA,
contiguous, and of the dtypes the header states (bf16 data, int32 tables,
int64 slot mapping, fp32 split-KV workspace).  Calls are asynchronous on the
given stream (default: torch's current stream).
"""
from __future__ import annotations

import ctypes
import math
from pathlib import Path
from typing import Optional, Tuple

import torch

__all__ = ["PaPool", "pa_kv_append", "pa_kv_copy", "pa_decode", "pa_append_decode", "pa_decode_splitkv",
           "pa_combine", "pa_prefill_chunked",
           "pa_device_status", "pa_selftest_wait_timeout", "pa_splitkv_workspace_bytes", "pa_decode_num_splits", "pa_splitkv_num_partitions",
           "pa_decode_splitkv_noalloc", "pa_noalloc_scratch_bytes", "PagedAttnError",
           "BlockManager", "pa_kv_block_bytes", "pa_kv_budget_blocks",
           "library", "library_path", "BLOCK_SIZE", "EXPORTED_SYMBOLS"]

BLOCK_SIZE = 16
PKG = Path(__file__).resolve().parent
_LIB_PATH = PKG / "libpagedattn.so"
EXPORTED_SYMBOLS = ("pa_kv_append", "pa_kv_copy", "pa_decode", "pa_append_decode", "pa_splitkv_workspace_bytes",
                    "pa_decode_splitkv", "pa_combine",
                    "pa_prefill_chunked", "pa_device_status", "pa_decode_num_splits", "pa_splitkv_num_partitions",
                    "pa_status_str", "pa_version", "pa_decode_splitkv_noalloc", "pa_noalloc_scratch_bytes",
                    "pa_selftest_wait_timeout",
                    "pa_kv_block_bytes", "pa_kv_budget_blocks", "pa_bm_create", "pa_bm_destroy", "pa_bm_admit", "pa_bm_admit_cow",
                    "pa_bm_commit", "pa_bm_release", "pa_bm_slots", "pa_bm_stats")

PA_OK = 0
PA_ERR_INVALID_ARG = -1
PA_ERR_REJECTED = -7
PA_ERR_UNSUPPORTED = -2
PA_ERR_CUDA = -3
PA_ERR_OUT_OF_RANGE = -4
PA_ERR_TIMEOUT = -5
PA_ERR_TOO_LARGE = -6
PA_DEV_OUT_OF_RANGE = 1
PA_DEV_TIMEOUT = 2


class PagedAttnError(RuntimeError):
    def __init__(self, what: str, code: int):
        super().__init__(f"{what} failed: {_status_str(code)} ({code})")
        self.code = code


class _PaPoolC(ctypes.Structure):
    _fields_ = [("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p), ("num_blocks", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32)]


_lib: Optional[ctypes.CDLL] = None


def library_path() -> Path:
    return _LIB_PATH


def library() -> ctypes.CDLL:
    """Load libpagedattn.so (built by paged_kv_gqa_slot_gb300.build); raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not _LIB_PATH.exists():
        raise RuntimeError(f"{_LIB_PATH} is not built; run `python -m paged_kv_gqa_slot_gb300.build` "
                           "(or __graft_entry__.build()) first -- there is no fallback path")
    lib = ctypes.CDLL(str(_LIB_PATH))
    P, I32, F32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
    pool = ctypes.POINTER(_PaPoolC)
    sig = {
        "pa_kv_append": (ctypes.c_int, [pool, P, P, P, I32, P]),
        "pa_kv_copy": (ctypes.c_int, [pool, P, P, I32, P]),
        "pa_decode": (ctypes.c_int, [pool, P, P, I32, P, I32, I32, F32, P, P]),
        "pa_append_decode": (ctypes.c_int, [pool, P, P, P, P, P, I32, P, I32, I32, F32, P, P]),
        "pa_splitkv_workspace_bytes": (SZ, [I32, I32, I32, I32]),
        "pa_decode_splitkv": (ctypes.c_int, [pool, P, P, I32, P, I32, I32, F32, I32, P, P, P]),
        "pa_combine": (ctypes.c_int, [P, P, I32, I32, I32, I32, P, P]),
        "pa_prefill_chunked": (ctypes.c_int, [pool, P, P, P, I32, P, I32, I32, I32, F32, P, P]),
        "pa_device_status": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32), I32, P]),
        "pa_selftest_wait_timeout": (ctypes.c_int, [ctypes.c_uint64, P]),
        "pa_decode_num_splits": (ctypes.c_int, [I32, I32, I32]),
        "pa_splitkv_num_partitions": (ctypes.c_int, [I32, I32, I32]),
        "pa_decode_splitkv_noalloc": (ctypes.c_int, [pool, P, P, I32, P, I32, I32, F32, I32, P, P]),
        "pa_noalloc_scratch_bytes": (SZ, []),
        "pa_status_str": (ctypes.c_char_p, [ctypes.c_int]),
        "pa_kv_block_bytes": (ctypes.c_int64, [I32, I32, I32, I32, I32]),
        "pa_kv_budget_blocks": (I32, [ctypes.c_int64, I32, I32, I32, I32, I32]),
        "pa_bm_create": (P, [I32, I32, I32]),
        "pa_bm_destroy": (None, [P]),
        "pa_bm_admit": (ctypes.c_int, [P, ctypes.c_int64, P, I32, I32, P, I32, P, P]),
        "pa_bm_admit_cow": (ctypes.c_int, [P, ctypes.c_int64, P, I32, I32, P, I32, P, P, P, P, P]),
        "pa_bm_commit": (ctypes.c_int, [P, ctypes.c_int64, P, I32, I32]),
        "pa_bm_release": (ctypes.c_int, [P, ctypes.c_int64]),
        "pa_bm_slots": (ctypes.c_int, [P, ctypes.c_int64, I32, I32, P]),
        "pa_bm_stats": (ctypes.c_int, [P, P, P, P]),
        "pa_version": (ctypes.c_int, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _status_str(code: int) -> str:
    try:
        return library().pa_status_str(code).decode()
    except Exception:  # pragma: no cover - used while raising
        return str(code)


def _check(code: int, what: str) -> None:
    if code != PA_OK:
        raise PagedAttnError(what, code)


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev(t: torch.Tensor, dtype, name: str) -> int:
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name}: need a contiguous CUDA {dtype} tensor, got {t.dtype} on {t.device}")
    return t.data_ptr()


def _tables(block_tables: torch.Tensor, seq_lens: torch.Tensor, batch: int) -> None:
    """The kernels read block_tables[b] and seq_lens[b] for every b < batch."""
    if block_tables.dim() != 2 or block_tables.shape[0] != batch or seq_lens.numel() != batch:
        raise ValueError(f"block_tables [batch, max_blocks] and seq_lens [batch] must match batch {batch}, got "
                         f"{tuple(block_tables.shape)} and {tuple(seq_lens.shape)}")


def _rows(k_new: torch.Tensor, v_new: torch.Tensor, pool: "PaPool", n: int) -> None:
    """The append kernels read n rows of [num_kv_heads, head_dim] from k_new and v_new."""
    shape = (n, pool.num_kv_heads, pool.head_dim)
    if tuple(k_new.shape) != shape or tuple(v_new.shape) != shape:
        raise ValueError(f"k_new / v_new: need shape {shape}, got {tuple(k_new.shape)} / {tuple(v_new.shape)}")


def _out(out: Optional[torch.Tensor], shape, like: torch.Tensor) -> torch.Tensor:
    """The caller's output tensor, checked to be exactly `shape` (the kernels write all of it),
    or a new one."""
    if out is None:
        return torch.empty(tuple(shape), dtype=torch.bfloat16, device=like.device)
    if tuple(out.shape) != tuple(shape):
        raise ValueError(f"out: need shape {tuple(shape)}, got {tuple(out.shape)}")
    return out


class PaPool:
    """The paged KV pool: k_cache, v_cache = [num_blocks, num_kv_heads, 16, head_dim] bf16 on the GPU."""

    def __init__(self, k_cache: torch.Tensor, v_cache: torch.Tensor):
        if k_cache.shape != v_cache.shape or k_cache.dim() != 4:
            raise ValueError("k_cache and v_cache must both be [num_blocks, num_kv_heads, block_size, head_dim]")
        self.k_cache, self.v_cache = k_cache, v_cache
        nb, hkv, bs, d = k_cache.shape
        self.c = _PaPoolC(_dev(k_cache, torch.bfloat16, "k_cache"), _dev(v_cache, torch.bfloat16, "v_cache"),
                          nb, bs, hkv, d)
        self.ref = ctypes.byref(self.c)

    @property
    def num_kv_heads(self) -> int:
        return self.c.num_kv_heads

    @property
    def head_dim(self) -> int:
        return self.c.head_dim


def pa_kv_append(pool: PaPool, k_new: torch.Tensor, v_new: torch.Tensor, slot_mapping: torch.Tensor,
                 stream=None) -> None:
    T = int(slot_mapping.numel())
    _rows(k_new, v_new, pool, T)
    rc = library().pa_kv_append(pool.ref, _dev(k_new, torch.bfloat16, "k_new") if T else None,
                                _dev(v_new, torch.bfloat16, "v_new") if T else None,
                                _dev(slot_mapping, torch.int64, "slot_mapping") if T else None, T, _stream(stream))
    _check(rc, "pa_kv_append")


def pa_kv_copy(pool: PaPool, src_slots: torch.Tensor, dst_slots: torch.Tensor, stream=None) -> None:
    """Copy pool rows src_slots[t] -> dst_slots[t] (K and V, every kv head)."""
    n = int(src_slots.numel())
    if dst_slots.numel() != n:
        raise ValueError(f"src_slots / dst_slots: need equal lengths, got {n} / {dst_slots.numel()}")
    rc = library().pa_kv_copy(pool.ref, _dev(src_slots, torch.int64, "src_slots") if n else None,
                              _dev(dst_slots, torch.int64, "dst_slots") if n else None, n, _stream(stream))
    _check(rc, "pa_kv_copy")


def pa_decode(pool: PaPool, q: torch.Tensor, block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float,
              out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    B, Hq, _ = q.shape
    _tables(block_tables, seq_lens, B)
    out = _out(out, q.shape, q)
    rc = library().pa_decode(pool.ref, _dev(q, torch.bfloat16, "q"), _dev(block_tables, torch.int32, "block_tables"),
                             block_tables.shape[1], _dev(seq_lens, torch.int32, "seq_lens"), B, Hq, float(scale),
                             _dev(out, torch.bfloat16, "out"), _stream(stream))
    _check(rc, "pa_decode")
    return out


def pa_append_decode(pool: PaPool, k_new: torch.Tensor, v_new: torch.Tensor, slot_mapping: torch.Tensor,
                     q: torch.Tensor, block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                     out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """pa_kv_append of one new row per sequence followed by pa_decode, in one launch."""
    B, Hq, _ = q.shape
    _tables(block_tables, seq_lens, B)
    _rows(k_new, v_new, pool, B)
    if slot_mapping.numel() != B:
        raise ValueError(f"slot_mapping: need {B} entries, got {slot_mapping.numel()}")
    out = _out(out, q.shape, q)
    rc = library().pa_append_decode(pool.ref, _dev(k_new, torch.bfloat16, "k_new"), _dev(v_new, torch.bfloat16, "v_new"),
                                    _dev(slot_mapping, torch.int64, "slot_mapping"), _dev(q, torch.bfloat16, "q"),
                                    _dev(block_tables, torch.int32, "block_tables"), block_tables.shape[1],
                                    _dev(seq_lens, torch.int32, "seq_lens"), B, Hq, float(scale),
                                    _dev(out, torch.bfloat16, "out"), _stream(stream))
    _check(rc, "pa_append_decode")
    return out


def pa_splitkv_workspace_bytes(batch: int, num_heads: int, head_dim: int, num_partitions: int) -> int:
    return int(library().pa_splitkv_workspace_bytes(batch, num_heads, head_dim, num_partitions))


def pa_decode_splitkv(pool: PaPool, q: torch.Tensor, block_tables: torch.Tensor, seq_lens: torch.Tensor,
                      scale: float, num_partitions: int, ws_o: Optional[torch.Tensor] = None,
                      ws_lse: Optional[torch.Tensor] = None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    B, Hq, D = q.shape
    _tables(block_tables, seq_lens, B)
    P = int(num_partitions)
    if ws_o is None:
        ws_o = torch.empty((B, Hq, P, D), dtype=torch.float32, device=q.device)
    if ws_lse is None:
        ws_lse = torch.empty((B, Hq, P), dtype=torch.float32, device=q.device)
    if tuple(ws_o.shape) != (B, Hq, P, D) or tuple(ws_lse.shape) != (B, Hq, P):
        raise ValueError(f"ws_o / ws_lse: need shapes {(B, Hq, P, D)} / {(B, Hq, P)}, "
                         f"got {tuple(ws_o.shape)} / {tuple(ws_lse.shape)}")
    rc = library().pa_decode_splitkv(pool.ref, _dev(q, torch.bfloat16, "q"),
                                     _dev(block_tables, torch.int32, "block_tables"), block_tables.shape[1],
                                     _dev(seq_lens, torch.int32, "seq_lens"), B, Hq, float(scale), P,
                                     _dev(ws_o, torch.float32, "ws_o"), _dev(ws_lse, torch.float32, "ws_lse"),
                                     _stream(stream))
    _check(rc, "pa_decode_splitkv")
    return ws_o, ws_lse


def pa_decode_splitkv_noalloc(pool: PaPool, q: torch.Tensor, block_tables: torch.Tensor, seq_lens: torch.Tensor,
                              scale: float, num_partitions: int, out: Optional[torch.Tensor] = None,
                              stream=None) -> torch.Tensor:
    """Split-KV decode + merge with no workspace argument: for callers that cannot allocate
    device memory (see include/pagedattn.h).  Pass a preallocated `out` to allocate nothing
    at all; its partition results live in a static array inside the library."""
    B, Hq, _ = q.shape
    _tables(block_tables, seq_lens, B)
    out = _out(out, q.shape, q)
    rc = library().pa_decode_splitkv_noalloc(pool.ref, _dev(q, torch.bfloat16, "q"),
                                             _dev(block_tables, torch.int32, "block_tables"), block_tables.shape[1],
                                             _dev(seq_lens, torch.int32, "seq_lens"), B, Hq, float(scale),
                                             int(num_partitions), _dev(out, torch.bfloat16, "out"), _stream(stream))
    _check(rc, "pa_decode_splitkv_noalloc")
    return out


def pa_noalloc_scratch_bytes() -> int:
    return int(library().pa_noalloc_scratch_bytes())


def pa_combine(ws_o: torch.Tensor, ws_lse: torch.Tensor, out: Optional[torch.Tensor] = None,
               stream=None) -> torch.Tensor:
    B, Hq, P, D = ws_o.shape
    if tuple(ws_lse.shape) != (B, Hq, P):
        raise ValueError(f"ws_lse: need shape {(B, Hq, P)}, got {tuple(ws_lse.shape)}")
    out = _out(out, (B, Hq, D), ws_o)
    rc = library().pa_combine(_dev(ws_o, torch.float32, "ws_o"), _dev(ws_lse, torch.float32, "ws_lse"), B, Hq, D, P,
                              _dev(out, torch.bfloat16, "out"), _stream(stream))
    _check(rc, "pa_combine")
    return out


def pa_prefill_chunked(pool: PaPool, q: torch.Tensor, cu_q_lens: torch.Tensor, block_tables: torch.Tensor,
                       seq_lens: torch.Tensor, scale: float, max_chunk: int, out: Optional[torch.Tensor] = None,
                       stream=None) -> torch.Tensor:
    _, Hq, _ = q.shape
    B = int(seq_lens.numel())
    _tables(block_tables, seq_lens, B)
    if cu_q_lens.numel() != B + 1:
        raise ValueError(f"cu_q_lens: need {B + 1} entries, got {cu_q_lens.numel()}")
    out = _out(out, q.shape, q)
    rc = library().pa_prefill_chunked(pool.ref, _dev(q, torch.bfloat16, "q"), _dev(cu_q_lens, torch.int32, "cu_q_lens"),
                                      _dev(block_tables, torch.int32, "block_tables"), block_tables.shape[1],
                                      _dev(seq_lens, torch.int32, "seq_lens"), B, Hq, int(max_chunk), float(scale),
                                      _dev(out, torch.bfloat16, "out"), _stream(stream))
    _check(rc, "pa_prefill_chunked")
    return out


def pa_device_status(clear: bool = True, stream=None) -> int:
    """Synchronise the stream and return the device status bits (0 = clean)."""
    flags = ctypes.c_uint32(0)
    rc = library().pa_device_status(ctypes.byref(flags), 1 if clear else 0, _stream(stream))
    if rc == PA_ERR_CUDA:
        raise PagedAttnError("pa_device_status", rc)
    return int(flags.value)


def pa_selftest_wait_timeout(limit_cycles: int = 2_000_000, stream=None) -> None:
    """Make one bounded device wait run out (an mbarrier nothing arrives on); afterwards the
    device status has PA_DEV_TIMEOUT set.  Asynchronous on `stream`."""
    _check(library().pa_selftest_wait_timeout(int(limit_cycles), _stream(stream)), "pa_selftest_wait_timeout")


def pa_decode_num_splits(batch: int, num_kv_heads: int, max_blocks: int) -> int:
    return int(library().pa_decode_num_splits(batch, num_kv_heads, max_blocks))


def pa_splitkv_num_partitions(batch: int, num_kv_heads: int, max_blocks: int) -> int:
    return int(library().pa_splitkv_num_partitions(batch, num_kv_heads, max_blocks))


def default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)


# ----------------------------------------------------------------------------- host block manager
def pa_kv_block_bytes(num_layers: int, num_kv_heads: int, head_dim: int, block_size: int = BLOCK_SIZE,
                      dtype_bytes: int = 2) -> int:
    return int(library().pa_kv_block_bytes(num_layers, num_kv_heads, head_dim, block_size, dtype_bytes))


def pa_kv_budget_blocks(budget_bytes: int, num_layers: int, num_kv_heads: int, head_dim: int,
                        block_size: int = BLOCK_SIZE, dtype_bytes: int = 2) -> int:
    return int(library().pa_kv_budget_blocks(int(budget_bytes), num_layers, num_kv_heads, head_dim, block_size,
                                             dtype_bytes))


class BlockManager:
    """The library's host-side KV block manager (pa_bm_*): refcounted blocks, a prefix cache
    of full blocks, full-lifetime admission.  Block tables and slot mappings come back as
    int32 / int64 numpy arrays, ready for the attention calls."""

    def __init__(self, num_blocks: int, block_size: int = BLOCK_SIZE, prefix_cache: bool = True):
        import numpy as np
        self._np = np
        self.block_size = block_size
        self._h = library().pa_bm_create(num_blocks, block_size, 1 if prefix_cache else 0)
        if not self._h:
            raise PagedAttnError("pa_bm_create failed")

    def close(self):
        if self._h:
            library().pa_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def admit(self, request_id: int, tokens, max_new_tokens: int):
        """(block_table, n_cached_tokens), or None when the request is rejected."""
        np = self._np
        toks = np.ascontiguousarray(tokens, dtype=np.int32)
        cap = (len(toks) + max_new_tokens + self.block_size - 1) // self.block_size
        table = np.empty(max(cap, 1), dtype=np.int32)
        nb, nc = ctypes.c_int32(0), ctypes.c_int32(0)
        rc = library().pa_bm_admit(self._h, request_id, toks.ctypes.data, len(toks), max_new_tokens,
                                   table.ctypes.data, len(table), ctypes.byref(nb), ctypes.byref(nc))
        if rc == PA_ERR_REJECTED:
            return None
        _check(rc, "pa_bm_admit")
        return table[:nb.value].copy(), nc.value

    def admit_cow(self, request_id: int, tokens, max_new_tokens: int):
        """(block_table, n_cached_tokens, copy_src, copy_dst), or None when rejected: a prefix
        hit may end inside a block, whose leading rows copy_src -> copy_dst (slot arrays for
        pa_kv_copy) must be copied before the request's own tokens are appended."""
        np = self._np
        toks = np.ascontiguousarray(tokens, dtype=np.int32)
        cap = (len(toks) + max_new_tokens + self.block_size - 1) // self.block_size
        table = np.empty(max(cap, 1), dtype=np.int32)
        src = np.empty(self.block_size, dtype=np.int64)
        dst = np.empty(self.block_size, dtype=np.int64)
        nb, nc, ncp = ctypes.c_int32(0), ctypes.c_int32(0), ctypes.c_int32(0)
        rc = library().pa_bm_admit_cow(self._h, request_id, toks.ctypes.data, len(toks), max_new_tokens,
                                       table.ctypes.data, len(table), ctypes.byref(nb), ctypes.byref(nc),
                                       src.ctypes.data, dst.ctypes.data, ctypes.byref(ncp))
        if rc == PA_ERR_REJECTED:
            return None
        _check(rc, "pa_bm_admit_cow")
        return table[:nb.value].copy(), nc.value, src[:ncp.value].copy(), dst[:ncp.value].copy()

    def commit(self, request_id: int, new_tokens, computed: int):
        np = self._np
        toks = np.ascontiguousarray(new_tokens if new_tokens is not None else [], dtype=np.int32)
        _check(library().pa_bm_commit(self._h, request_id, toks.ctypes.data if len(toks) else None, len(toks),
                                      computed), "pa_bm_commit")

    def release(self, request_id: int):
        _check(library().pa_bm_release(self._h, request_id), "pa_bm_release")

    def slots(self, request_id: int, start: int, n: int):
        np = self._np
        out = np.empty(max(n, 1), dtype=np.int64)
        _check(library().pa_bm_slots(self._h, request_id, start, n, out.ctypes.data), "pa_bm_slots")
        return out[:n].copy()

    def stats(self):
        """(free, cached_idle, used) block counts."""
        f, c, u = ctypes.c_int32(0), ctypes.c_int32(0), ctypes.c_int32(0)
        _check(library().pa_bm_stats(self._h, ctypes.byref(f), ctypes.byref(c), ctypes.byref(u)), "pa_bm_stats")
        return f.value, c.value, u.value

