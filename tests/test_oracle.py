"""The CPU oracle against its pins (no GPU)."""
import math

import numpy as np
import pytest
import torch

import oracle
import oracle_pins as pins
import golden_cases as G
import workloads as W
from workloads import u16


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


@pytest.mark.parametrize("spec", G.load_cases(), ids=lambda c: c["name"])
def test_golden_closed_form(orc, spec):
    case = G.build(spec)
    got = pins.oracle_attention(orc, case)
    want = G.expected(spec)
    assert got.shape == want.shape
    if spec["name"] == "single_key":
        assert np.array_equal(got, want)
    else:
        assert np.max(np.abs(got - want)) <= 1e-14
    for P in map(int, spec.get("partitions", {})):
        o, lse = orc.decode_partitions(u16(case.k_cache), u16(case.v_cache), u16(case.q),
                                       case.block_tables.numpy(), case.seq_lens.numpy(), case.scale, P)
        wo, wl = G.expected_partitions(spec, P)
        assert np.max(np.abs(o[0, 0] - wo)) <= 1e-14
        fin = np.isfinite(wl)
        assert np.all(np.isneginf(lse[0, 0][~fin]))
        assert np.max(np.abs(lse[0, 0][fin] - wl[fin])) <= 1e-14


def test_empty_sequence_gives_zero(orc):
    case = W.paged_case(name="empty", seed=3, seq_lens=[0, 20], q_lens=[1, 1], new_lens=[0, 0], num_heads=4,
                        num_kv_heads=2, head_dim=64, num_blocks=4)
    out = pins.oracle_attention(orc, case)
    assert not np.any(out[0])
    assert np.all(np.isfinite(out[1]))
    o, lse = orc.decode_partitions(u16(case.k_cache), u16(case.v_cache), u16(case.q), case.block_tables.numpy(),
                                   case.seq_lens.numpy(), case.scale, 4)
    assert np.all(np.isneginf(lse[0])) and not np.any(o[0])
    merged = orc.combine(o, lse)
    assert not np.any(merged[0])


def test_out_of_range_block_is_an_error(orc):
    case = W.tiny_decode()
    bt = case.block_tables.clone()
    bt[0, 1] = case.num_blocks            # one past the pool
    with pytest.raises(oracle.OracleError):
        orc.decode(u16(case.k_cache), u16(case.v_cache), u16(case.q), bt.numpy(), case.seq_lens.numpy(),
                   case.scale)
    k = u16(case.k_cache).copy()
    v = u16(case.v_cache).copy()
    with pytest.raises(oracle.OracleError):
        orc.kv_append(k, v, u16(case.k_seq[0][:1]), u16(case.v_seq[0][:1]),
                      np.array([case.num_blocks * 16], dtype=np.int64))


def test_leak_sentinels_are_not_read(orc):
    """Unused pool slots and the tail of each last block hold NaN; the output stays finite."""
    for seed in range(5):
        case = W.random_case(8100 + seed, batch=4, num_heads=8, num_kv_heads=2, head_dim=64, max_len=50)
        out = pins.oracle_attention(orc, case)
        assert np.all(np.isfinite(out))


def test_prefill_rows_match_full(orc):
    case = W.random_case(8200, batch=3, num_heads=8, num_kv_heads=2, head_dim=64, min_len=20, max_len=70,
                         q_len=12, prefill=True)
    full = pins.oracle_attention(orc, case)
    k, v = pins.post_append_pool(orc, case)
    T = case.q.shape[0]
    rt = np.array([0, T - 1, T // 2, 1], dtype=np.int32)
    rh = np.array([0, 7, 3, 5], dtype=np.int32)
    rows = orc.prefill_rows(k, v, u16(case.q), case.cu_q_lens.numpy(), case.block_tables.numpy(),
                            case.seq_lens.numpy(), case.scale, rt, rh)
    assert np.array_equal(rows, full[rt, rh])


def test_workload_shapes():
    c = W.tiny_decode()
    assert (c.batch, c.num_heads, c.num_kv_heads, c.head_dim, c.num_blocks) == (1, 4, 1, 64, 16)
    assert int(c.seq_lens[0]) == 37 and (c.block_tables[0] >= 0).sum() == 3 and c.scale == 0.125
    c = W.chunked_prefill()
    assert c.q.shape == (2048, 32, 128) and c.slot_mapping.numel() == 2048
    # all eight sequences share the same 48 prefix blocks, and own distinct chunk blocks
    assert torch.all(c.block_tables[:, :48] == c.block_tables[0, :48])
    own = c.block_tables[:, 48:64].flatten()
    assert own.unique().numel() == 128 and not set(own.tolist()) & set(c.block_tables[0, :48].tolist())
