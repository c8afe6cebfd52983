"""fp64 CPU oracle for paged grouped-query attention -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package.  The product path (``paged_kv_gqa_slot_gb300``) never
does: it has no CPU fallback.  The C source (``pa_oracle.c``) is compiled with
gcc into ``oracle/_build/libpa_oracle.so`` on first use (or by ``build()``),
with floating-point contraction off so that x86 and Arm give the same bits.

The functions here only marshal numpy arrays into the C calls; every step of
the arithmetic is in ``pa_oracle.c``.  bf16 tensors travel as their uint16 bits.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path
from typing import Optional

import numpy as np

HERE = Path(__file__).resolve().parent
SOURCE = HERE / "pa_oracle.c"
BUILD_DIR = HERE / "_build"
LIB_PATH = BUILD_DIR / "libpa_oracle.so"

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(source: Path = SOURCE, out: Path = LIB_PATH, force: bool = False) -> Path:
    """Compile the oracle (plain C, gcc) if the shared object is missing or stale: with
    OpenMP where gcc has it (the row loops may then run on several threads), else without."""
    source, out = Path(source), Path(out)
    if not force and out.exists() and out.stat().st_mtime >= source.stat().st_mtime:
        return out
    out.parent.mkdir(parents=True, exist_ok=True)
    tmp = out.with_suffix(f".{os.getpid()}.tmp.so")
    r = subprocess.run(["gcc", *CFLAGS, "-fopenmp", str(source), "-o", str(tmp), "-lm"], capture_output=True)
    if r.returncode != 0:
        subprocess.run(["gcc", *CFLAGS, str(source), "-o", str(tmp), "-lm"], check=True)
    os.replace(tmp, out)
    return out


_i32 = ctypes.c_int32
_dbl = ctypes.c_double
_p = ctypes.c_void_p


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _arr(a, dtype) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(a), dtype=dtype)
    return a


class OracleError(RuntimeError):
    pass


class Oracle:
    """ctypes front of one compiled oracle library (the real one or a planted-mistake copy)."""

    def __init__(self, path: Path):
        self.path = Path(path)
        self.lib = ctypes.CDLL(str(self.path))
        L = self.lib
        L.pa_oracle_kv_append.argtypes = [_p, _p, _i32, _i32, _i32, _i32, _p, _p, _p, _i32]
        L.pa_oracle_decode.argtypes = [_p, _p, _i32, _i32, _i32, _i32, _p, _p, _i32, _p, _i32, _i32, _dbl, _p]
        L.pa_oracle_decode_partitions.argtypes = [_p, _p, _i32, _i32, _i32, _i32, _p, _p, _i32, _p, _i32, _i32,
                                                  _dbl, _i32, _p, _p]
        L.pa_oracle_combine.argtypes = [_p, _p, _i32, _i32, _i32, _i32, _p]
        L.pa_oracle_prefill.argtypes = [_p, _p, _i32, _i32, _i32, _i32, _p, _p, _p, _i32, _p, _i32, _i32, _dbl, _p]
        L.pa_oracle_prefill_rows.argtypes = [_p, _p, _i32, _i32, _i32, _i32, _p, _p, _p, _i32, _p, _i32, _i32,
                                             _dbl, _p, _p, _i32, _p]
        for f in ("pa_oracle_kv_append", "pa_oracle_decode", "pa_oracle_decode_partitions", "pa_oracle_combine",
                  "pa_oracle_prefill", "pa_oracle_prefill_rows"):
            getattr(L, f).restype = ctypes.c_int
        L.pa_oracle_set_threads.argtypes = [_i32]
        L.pa_oracle_set_threads.restype = ctypes.c_int
        self.threads = self.set_threads(int(os.environ.get("PA_ORACLE_THREADS", os.cpu_count() or 1)))

    def set_threads(self, n: int) -> int:
        """Threads the per-row loops may use (1 if built without OpenMP); returns the count in
        effect.  The results are the same bits for any count: each row is one thread's work."""
        self.threads = int(self.lib.pa_oracle_set_threads(int(n)))
        return self.threads

    @staticmethod
    def _check(rc: int, what: str):
        if rc != 0:
            raise OracleError(f"{what} returned {rc}")

    @staticmethod
    def _pool(k_cache: np.ndarray, v_cache: np.ndarray):
        assert k_cache.dtype == np.uint16 and v_cache.dtype == np.uint16 and k_cache.shape == v_cache.shape
        nblk, hkv, bs, d = k_cache.shape
        return np.ascontiguousarray(k_cache), np.ascontiguousarray(v_cache), nblk, bs, hkv, d

    def kv_append(self, k_cache: np.ndarray, v_cache: np.ndarray, k_new, v_new, slot_mapping) -> None:
        """In-place scatter into the (uint16) pool arrays."""
        assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
        nblk, hkv, bs, d = k_cache.shape
        k_new = _arr(k_new, np.uint16)
        v_new = _arr(v_new, np.uint16)
        slots = _arr(slot_mapping, np.int64)
        rc = self.lib.pa_oracle_kv_append(_ptr(k_cache), _ptr(v_cache), nblk, bs, hkv, d, _ptr(k_new),
                                          _ptr(v_new), _ptr(slots), int(slots.size))
        self._check(rc, "kv_append")

    def decode(self, k_cache, v_cache, q, block_tables, seq_lens, scale: float) -> np.ndarray:
        k, v, nblk, bs, hkv, d = self._pool(k_cache, v_cache)
        q = _arr(q, np.uint16)
        bt = _arr(block_tables, np.int32)
        sl = _arr(seq_lens, np.int32)
        B, Hq = q.shape[0], q.shape[1]
        out = np.zeros((B, Hq, d), dtype=np.float64)
        rc = self.lib.pa_oracle_decode(_ptr(k), _ptr(v), nblk, bs, hkv, d, _ptr(q), _ptr(bt), bt.shape[1],
                                       _ptr(sl), B, Hq, float(scale), _ptr(out))
        self._check(rc, "decode")
        return out

    def decode_partitions(self, k_cache, v_cache, q, block_tables, seq_lens, scale: float, num_partitions: int):
        k, v, nblk, bs, hkv, d = self._pool(k_cache, v_cache)
        q = _arr(q, np.uint16)
        bt = _arr(block_tables, np.int32)
        sl = _arr(seq_lens, np.int32)
        B, Hq = q.shape[0], q.shape[1]
        P = int(num_partitions)
        o = np.zeros((B, Hq, P, d), dtype=np.float64)
        lse = np.zeros((B, Hq, P), dtype=np.float64)
        rc = self.lib.pa_oracle_decode_partitions(_ptr(k), _ptr(v), nblk, bs, hkv, d, _ptr(q), _ptr(bt),
                                                  bt.shape[1], _ptr(sl), B, Hq, float(scale), P, _ptr(o),
                                                  _ptr(lse))
        self._check(rc, "decode_partitions")
        return o, lse

    def combine(self, o_part, lse_part) -> np.ndarray:
        o = _arr(o_part, np.float64)
        lse = _arr(lse_part, np.float64)
        B, Hq, P, d = o.shape
        out = np.zeros((B, Hq, d), dtype=np.float64)
        rc = self.lib.pa_oracle_combine(_ptr(o), _ptr(lse), B, Hq, d, P, _ptr(out))
        self._check(rc, "combine")
        return out

    def prefill(self, k_cache, v_cache, q, cu_q_lens, block_tables, seq_lens, scale: float) -> np.ndarray:
        k, v, nblk, bs, hkv, d = self._pool(k_cache, v_cache)
        q = _arr(q, np.uint16)
        cu = _arr(cu_q_lens, np.int32)
        bt = _arr(block_tables, np.int32)
        sl = _arr(seq_lens, np.int32)
        T, Hq = q.shape[0], q.shape[1]
        out = np.zeros((T, Hq, d), dtype=np.float64)
        rc = self.lib.pa_oracle_prefill(_ptr(k), _ptr(v), nblk, bs, hkv, d, _ptr(q), _ptr(cu), _ptr(bt),
                                        bt.shape[1], _ptr(sl), sl.size, Hq, float(scale), _ptr(out))
        self._check(rc, "prefill")
        return out

    def prefill_rows(self, k_cache, v_cache, q, cu_q_lens, block_tables, seq_lens, scale: float,
                     row_tokens, row_heads) -> np.ndarray:
        k, v, nblk, bs, hkv, d = self._pool(k_cache, v_cache)
        q = _arr(q, np.uint16)
        cu = _arr(cu_q_lens, np.int32)
        bt = _arr(block_tables, np.int32)
        sl = _arr(seq_lens, np.int32)
        rt = _arr(row_tokens, np.int32)
        rh = _arr(row_heads, np.int32)
        out = np.zeros((rt.size, d), dtype=np.float64)
        rc = self.lib.pa_oracle_prefill_rows(_ptr(k), _ptr(v), nblk, bs, hkv, d, _ptr(q), _ptr(cu), _ptr(bt),
                                             bt.shape[1], _ptr(sl), sl.size, q.shape[1], float(scale), _ptr(rt),
                                             _ptr(rh), int(rt.size), _ptr(out))
        self._check(rc, "prefill_rows")
        return out


_default: Optional[Oracle] = None


def load() -> Oracle:
    """The oracle compiled from ``pa_oracle.c`` (built on first use)."""
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default
