"""The workspace-free split-KV decode (pa_decode_splitkv_noalloc) against the oracle and
against the workspace path.

The no-allocation entry point is for callers that cannot allocate device memory -- a fixed
arena owned by someone else, a plugin without an allocator, a hot loop that must not call
cudaMalloc.  It keeps the partition results in a static array inside the library, shared by
every call, so these tests check that two calls in a row (with a different problem in
between) each meet the tolerance against the fp64 oracle and reproduce the workspace path,
and that an oversized request is refused before any launch.  This file is collected last so
that a failure here stops a run only after every other test has run.
"""
import pytest
import torch

import paged_kv_gqa_slot_gb300 as pa
import workloads as W
from parity import GpuCase, compare, oracle_decode

pytestmark = pytest.mark.gpu


def _reference(g, P):
    ws_o, ws_lse = g.splitkv(P)
    return pa.pa_combine(ws_o, ws_lse).to(torch.float64).cpu().numpy()


def test_noalloc_matches_workspace_path_on_consecutive_calls():
    a = GpuCase(W.splitkv_decode(1004, 4, 8192))
    b = GpuCase(W.random_case(4200, batch=6, num_heads=16, num_kv_heads=2, head_dim=128, min_len=1, max_len=300))
    ref_a, ref_b = _reference(a, 16), _reference(b, 8)
    orc_a, orc_b = oracle_decode(a.case), oracle_decode(b.case)
    out = torch.empty_like(a.q)
    for call in range(2):
        pa.pa_decode_splitkv_noalloc(a.pool, a.q, a.bt, a.sl, a.case.scale, 16, out)
        compare(out, orc_a, f"no-alloc 4x8192 P=16 vs oracle, call {call}")
        compare(out, ref_a, f"no-alloc 4x8192 P=16 vs workspace path, call {call}")
        # a different, smaller problem in between reuses the same static scratch
        out_b = pa.pa_decode_splitkv_noalloc(b.pool, b.q, b.bt, b.sl, b.case.scale, 8)
        compare(out_b, orc_b, f"no-alloc ragged P=8 vs oracle, call {call}")
        compare(out_b, ref_b, f"no-alloc ragged P=8 vs workspace path, call {call}")
    assert pa.pa_device_status(clear=True) == 0


def test_noalloc_refuses_requests_beyond_its_scratch():
    a = GpuCase(W.splitkv_decode(1004, 1, 32768))
    limit = pa.pa_noalloc_scratch_bytes()
    P = 4096  # 1 x 64 heads x 4096 partitions x 128 x 4 B = 128 MiB > the 8 MiB scratch
    assert pa.pa_splitkv_workspace_bytes(1, a.case.num_heads, 128, P) > limit
    with pytest.raises(pa.PagedAttnError) as e:
        pa.pa_decode_splitkv_noalloc(a.pool, a.q, a.bt, a.sl, a.case.scale, P)
    assert e.value.code == pa.PA_ERR_TOO_LARGE
