"""The C-ABI library on the CPU: it loads, exports every symbol the header declares, and its
host-side validation rejects bad arguments before any CUDA call (no GPU needed)."""
import ctypes
import re
from pathlib import Path

import pytest

import paged_kv_gqa_slot_gb300 as pa
from paged_kv_gqa_slot_gb300 import build as pbuild

HEADER = Path(__file__).resolve().parent.parent / "include" / "pagedattn.h"


@pytest.fixture(scope="module")
def lib():
    pbuild.build()
    return pa.library()


def declared_functions():
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_functions()
    for n in ("pa_kv_append", "pa_decode", "pa_decode_splitkv", "pa_combine", "pa_prefill_chunked",
              "pa_splitkv_workspace_bytes", "pa_device_status", "pa_status_str"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in pagedattn.h but not exported"
    assert set(declared_functions()) <= set(pa.EXPORTED_SYMBOLS)


def test_status_strings_and_version(lib):
    assert lib.pa_status_str(0) == b"PA_OK"
    assert lib.pa_status_str(-1) == b"PA_ERR_INVALID_ARG"
    assert lib.pa_status_str(-4) == b"PA_ERR_OUT_OF_RANGE"
    assert lib.pa_status_str(-99) == b"PA_ERR_UNKNOWN"
    assert lib.pa_version() >= 100


def test_workspace_bytes(lib):
    B, H, D, P = 4, 64, 128, 16
    o = B * H * P * D * 4
    assert pa.pa_splitkv_workspace_bytes(B, H, D, P) == ((o + 15) // 16) * 16 + B * H * P * 4
    assert pa.pa_splitkv_workspace_bytes(-1, H, D, P) == 0


def _pool(nb=16, bs=16, hkv=2, d=128, k=0x10000, v=0x20000):
    return pa._PaPoolC(k, v, nb, bs, hkv, d)


FAKE = 0x40000  # a 16-byte-aligned address that validation never dereferences


def test_validation_rejects_before_launch(lib):
    P = ctypes.byref
    ok_pool = _pool()
    # null pool, null tensors
    assert lib.pa_decode(None, FAKE, FAKE, 4, FAKE, 1, 4, 0.1, FAKE, None) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_decode(P(_pool(k=0)), FAKE, FAKE, 4, FAKE, 1, 4, 0.1, FAKE, None) == pa.PA_ERR_INVALID_ARG
    # block size and head dim outside the compiled set
    assert lib.pa_decode(P(_pool(bs=8)), FAKE, FAKE, 4, FAKE, 1, 4, 0.1, FAKE, None) == pa.PA_ERR_UNSUPPORTED
    assert lib.pa_decode(P(_pool(d=96)), FAKE, FAKE, 4, FAKE, 1, 4, 0.1, FAKE, None) == pa.PA_ERR_UNSUPPORTED
    # heads not a multiple of kv heads; group too large for decode
    assert lib.pa_decode(P(ok_pool), FAKE, FAKE, 4, FAKE, 1, 5, 0.1, FAKE, None) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_decode(P(ok_pool), FAKE, FAKE, 4, FAKE, 1, 64, 0.1, FAKE, None) == pa.PA_ERR_UNSUPPORTED
    # misaligned q, null out, bad max_blocks, negative batch, non-finite scale
    assert lib.pa_decode(P(ok_pool), FAKE + 2, FAKE, 4, FAKE, 1, 4, 0.1, FAKE, None) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_decode(P(ok_pool), FAKE, FAKE, 4, FAKE, 1, 4, 0.1, None, None) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_decode(P(ok_pool), FAKE, FAKE, 0, FAKE, 1, 4, 0.1, FAKE, None) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_decode(P(ok_pool), FAKE, FAKE, 4, FAKE, -1, 4, 0.1, FAKE, None) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_decode(P(ok_pool), FAKE, FAKE, 4, FAKE, 1, 4, float("nan"), FAKE, None) == pa.PA_ERR_INVALID_ARG
    # empty batch is a no-op that needs no GPU
    assert lib.pa_decode(P(ok_pool), FAKE, FAKE, 4, FAKE, 0, 4, 0.1, FAKE, None) == pa.PA_OK
    # split-KV: partitions out of range, missing lse workspace
    assert lib.pa_decode_splitkv(P(ok_pool), FAKE, FAKE, 4, FAKE, 1, 4, 0.1, 0, FAKE, FAKE, None) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_decode_splitkv(P(ok_pool), FAKE, FAKE, 4, FAKE, 1, 4, 0.1, 5000, FAKE, FAKE, None) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_decode_splitkv(P(ok_pool), FAKE, FAKE, 4, FAKE, 1, 4, 0.1, 8, FAKE, None, None) == pa.PA_ERR_INVALID_ARG
    # combine
    assert lib.pa_combine(FAKE, FAKE, 1, 4, 96, 8, FAKE, None) == pa.PA_ERR_UNSUPPORTED
    assert lib.pa_combine(FAKE, FAKE, 1, 4, 128, 0, FAKE, None) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_combine(None, FAKE, 1, 4, 128, 8, FAKE, None) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_combine(FAKE, FAKE, 0, 4, 128, 8, FAKE, None) == pa.PA_OK
    # prefill
    assert lib.pa_prefill_chunked(P(ok_pool), FAKE, None, FAKE, 4, FAKE, 1, 4, 16, 0.1, FAKE, None) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_prefill_chunked(P(ok_pool), FAKE, FAKE, FAKE, 4, FAKE, 1, 4, -1, 0.1, FAKE, None) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_prefill_chunked(P(ok_pool), FAKE, FAKE, FAKE, 4, FAKE, 1, 4, 0, 0.1, FAKE, None) == pa.PA_OK
    # append
    assert lib.pa_kv_append(P(ok_pool), FAKE, FAKE, None, 3, None) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_kv_append(P(ok_pool), FAKE, FAKE, FAKE, -1, None) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_kv_append(P(ok_pool), FAKE, FAKE, FAKE, 0, None) == pa.PA_OK
    # the workspace-free split-KV call refuses what does not fit its static scratch, before any launch
    assert lib.pa_noalloc_scratch_bytes() == 8 << 20
    assert lib.pa_decode_splitkv_noalloc(P(ok_pool), FAKE, FAKE, 4, FAKE, 1, 64, 0.1, 4096, FAKE, None) == \
        pa.PA_ERR_TOO_LARGE
    assert lib.pa_decode_splitkv_noalloc(P(_pool(d=96)), FAKE, FAKE, 4, FAKE, 1, 4, 0.1, 8, FAKE, None) == \
        pa.PA_ERR_UNSUPPORTED
    assert lib.pa_decode_splitkv_noalloc(P(ok_pool), FAKE, FAKE, 4, FAKE, 0, 4, 0.1, 8, FAKE, None) == pa.PA_OK
    # fused append + decode: missing rows, batch 0, head dim outside the compiled set
    assert lib.pa_append_decode(P(ok_pool), None, FAKE, FAKE, FAKE, FAKE, 4, FAKE, 1, 4, 0.1, FAKE, None) == \
        pa.PA_ERR_INVALID_ARG
    assert lib.pa_append_decode(P(ok_pool), FAKE, FAKE, FAKE, FAKE, FAKE, 4, FAKE, 0, 4, 0.1, FAKE, None) == pa.PA_OK
    assert lib.pa_append_decode(P(_pool(d=96)), FAKE, FAKE, FAKE, FAKE, FAKE, 4, FAKE, 1, 4, 0.1, FAKE, None) == \
        pa.PA_ERR_UNSUPPORTED
    # status needs a flags pointer
    assert lib.pa_device_status(None, 1, None) == pa.PA_ERR_INVALID_ARG


def test_selftest_wait_timeout_rejects_limits_outside_its_range(lib):
    # checked before any CUDA call, so it runs without a GPU
    assert lib.pa_selftest_wait_timeout(0, None) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_selftest_wait_timeout((1 << 40) + 1, None) == pa.PA_ERR_INVALID_ARG
