"""Run a workloads.PagedCase through the CUDA library and through the oracle, and compare.

Tolerance (bf16 inputs, fp32 accumulation, bf16 output):
  * absolute: every element within max(1e-2, ulp_bf16(oracle) / 2) of the oracle.  The 1e-2
    is the stated bound; the half ulp only takes over where the final rounding of the result
    to bf16, which no bf16 output can avoid, alone exceeds it (|o| >= 4);
  * relative: per (token, head) row, max|gpu - oracle| / max|oracle| <= 2e-2.
Rows whose oracle output is exactly zero (a sequence of length 0) must be exactly zero.

Every comparison is recorded in REPORT (raw max-abs, row max-rel and their headroom), which
the test session prints at its end.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import paged_kv_gqa_slot_gb300 as pa
from workloads import u16

ATOL = 1e-2
RTOL_ROW = 2e-2

# (what, elements, raw max |gpu - oracle|, max row-relative error) of every comparison made
REPORT = []


def half_ulp_bf16(x: np.ndarray) -> np.ndarray:
    """Half the spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, np.exp2(e - 8), 0.0)


def compare(gpu: torch.Tensor, ref: np.ndarray, what: str, atol: float = ATOL, rtol_row: float = RTOL_ROW):
    """Assert the tolerance above; returns (raw max-abs error, max row-relative error)."""
    g = gpu.detach().to("cpu", torch.float64).numpy().reshape(ref.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output (read outside a sequence?)"
    diff = np.abs(g - ref)
    max_abs = float(diff.max()) if diff.size else 0.0
    bound = np.maximum(atol, half_ulp_bf16(ref))
    over = diff > bound
    rows_d = diff.reshape(-1, ref.shape[-1]).max(axis=1) if diff.size else np.zeros(0)
    rows_r = np.abs(ref).reshape(-1, ref.shape[-1]).max(axis=1) if diff.size else np.zeros(0)
    zero = rows_r == 0
    rel = float((rows_d[~zero] / rows_r[~zero]).max()) if np.any(~zero) else 0.0
    REPORT.append((what, int(diff.size), max_abs, rel))
    assert np.all(rows_d[zero] == 0), f"{what}: rows with an all-zero reference are not zero"
    if np.any(over):
        i = np.unravel_index(int(np.argmax(diff - bound)), diff.shape)
        raise AssertionError(f"{what}: {int(over.sum())} elements beyond max({atol}, half ulp); worst at {i}: "
                             f"gpu {g[i]!r} oracle {ref[i]!r} (max abs err {max_abs:.3e})")
    assert rel <= rtol_row, f"{what}: max row-rel err {rel:.3e} > {rtol_row}"
    return max_abs, rel


class GpuCase:
    """Device copies of one case, with the append already run on the GPU."""

    def __init__(self, case, device="cuda", append=True):
        self.case = case
        self.k = case.k_cache.to(device)
        self.v = case.v_cache.to(device)
        self.pool = pa.PaPool(self.k, self.v)
        self.q = case.q.to(device)
        self.bt = case.block_tables.to(device)
        self.sl = case.seq_lens.to(device)
        self.cu = case.cu_q_lens.to(device)
        self.k_new = case.k_new.to(device)
        self.v_new = case.v_new.to(device)
        self.slots = case.slot_mapping.to(device)
        if append:
            pa.pa_kv_append(self.pool, self.k_new, self.v_new, self.slots)

    def decode(self):
        return pa.pa_decode(self.pool, self.q, self.bt, self.sl, self.case.scale)

    def splitkv(self, P):
        return pa.pa_decode_splitkv(self.pool, self.q, self.bt, self.sl, self.case.scale, P)

    def prefill(self):
        return pa.pa_prefill_chunked(self.pool, self.q, self.cu, self.bt, self.sl, self.case.scale,
                                     max(self.case.q_lens))


def oracle_pool(case):
    """The pool after the oracle's own append (uint16 bits)."""
    orc = oracle.load()
    k = u16(case.k_cache).copy()
    v = u16(case.v_cache).copy()
    orc.kv_append(k, v, u16(case.k_new), u16(case.v_new), case.slot_mapping.numpy())
    return k, v


def oracle_decode(case, pool=None):
    k, v = pool if pool is not None else oracle_pool(case)
    return oracle.load().decode(k, v, u16(case.q), case.block_tables.numpy(), case.seq_lens.numpy(), case.scale)


def oracle_prefill(case, pool=None):
    k, v = pool if pool is not None else oracle_pool(case)
    return oracle.load().prefill(k, v, u16(case.q), case.cu_q_lens.numpy(), case.block_tables.numpy(),
                                 case.seq_lens.numpy(), case.scale)


def check_status_clean(what: str):
    flags = pa.pa_device_status(clear=True)
    assert flags == 0, f"{what}: device status {flags:#x}"
