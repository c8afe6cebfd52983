"""CUDA path against the fp64 oracle, through the C ABI, on the same seeded inputs.

Covers every call: the append (bit-exact), decode (single CTA and thread-block-cluster
splits), split-KV partitions and their combine, chunked prefill; the five workloads at
full size, every output element compared, plus ragged
sweeps over sequence length, group size, head dim and partition count, the degenerate
cases (empty sequences, one key, more partitions than blocks), NaN leak sentinels, and
the device status word for out-of-pool ids.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_slot_gb300 as pa
import workloads as W
import golden_cases as G
from parity import GpuCase, compare, oracle_pool, oracle_decode, oracle_prefill, check_status_clean
from workloads import u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pa.library()
    pa.pa_device_status(clear=True)
    yield


# ------------------------------------------------------------------ append
@pytest.mark.parametrize("make", [W.batched_decode, W.chunked_prefill,
                                  lambda: W.random_case(11, batch=5, num_heads=8, num_kv_heads=2, head_dim=64,
                                                        prefill=True, q_len=30)],
                         ids=["batched_decode", "chunked_prefill", "random_d64"])
def test_kv_append_bit_exact(make):
    case = make()
    g = GpuCase(case)
    k_ref, v_ref = oracle_pool(case)
    torch.cuda.synchronize()
    assert np.array_equal(u16(g.k.cpu()), k_ref)
    assert np.array_equal(u16(g.v.cpu()), v_ref)
    check_status_clean("append")


def test_kv_append_skips_negative_and_flags_out_of_pool():
    case = W.random_case(12, batch=3, num_heads=4, num_kv_heads=2, head_dim=128, prefill=True, q_len=10)
    g = GpuCase(case, append=False)
    slots = case.slot_mapping.clone()
    slots[0] = -1
    bad = slots.clone()
    bad[1] = case.num_blocks * 16 + 3
    pa.pa_kv_append(g.pool, g.k_new, g.v_new, bad.cuda())
    assert pa.pa_device_status(clear=True) == pa.PA_DEV_OUT_OF_RANGE
    # reference: the same scatter with rows 0 and 1 skipped
    k = u16(case.k_cache).copy()
    v = u16(case.v_cache).copy()
    sm = bad.numpy().copy()
    sm[1] = -1
    oracle.load().kv_append(k, v, u16(case.k_new), u16(case.v_new), sm)
    assert np.array_equal(u16(g.k.cpu()), k) and np.array_equal(u16(g.v.cpu()), v)


# ------------------------------------------------------------------ decode
@pytest.mark.parametrize("make", [W.tiny_decode, W.qwen3_4b_decode, W.batched_decode],
                         ids=["tiny_decode", "qwen3_4b_decode", "batched_decode"])
def test_decode_workloads(make):
    case = make()
    g = GpuCase(case)
    out = g.decode()
    compare(out, oracle_decode(case), case.name)
    check_status_clean(case.name)


SWEEP = [(hq, hkv, d) for d in (64, 128) for (hq, hkv) in ((4, 4), (8, 4), (8, 2), (16, 2), (32, 8), (32, 2))]


@pytest.mark.parametrize("hq,hkv,d", SWEEP)
def test_decode_ragged_sweep(hq, hkv, d):
    for j, (lo, hi) in enumerate(((1, 17), (15, 70), (100, 400))):
        case = W.random_case(2000 + 31 * hq + hkv + d + j, batch=7, num_heads=hq, num_kv_heads=hkv, head_dim=d,
                             min_len=lo, max_len=hi)
        g = GpuCase(case)
        compare(g.decode(), oracle_decode(case), f"decode {hq}/{hkv}/{d} len {lo}-{hi}")
    check_status_clean("decode sweep")


@pytest.mark.parametrize("L", [1, 15, 16, 17, 33, 64, 255, 256, 257, 1000])
def test_decode_lengths_single_sequence(L):
    """One sequence: few CTAs, so the cluster-split path with ragged per-split ranges."""
    case = W.paged_case(name=f"len{L}", seed=3000 + L, seq_lens=[L], q_lens=[1], new_lens=[1], num_heads=32,
                        num_kv_heads=8, head_dim=128, num_blocks=max(8, 2 * (L // 16 + 1)))
    g = GpuCase(case)
    compare(g.decode(), oracle_decode(case), case.name)
    check_status_clean(case.name)


def test_decode_empty_sequences_give_zero():
    case = W.paged_case(name="empty", seed=5, seq_lens=[0, 40, 0, 3], q_lens=[1] * 4, new_lens=[0] * 4, num_heads=8,
                        num_kv_heads=2, head_dim=128, num_blocks=16)
    g = GpuCase(case)
    out = g.decode()
    ref = oracle_decode(case)
    compare(out, ref, "empty")
    assert torch.all(out[0] == 0) and torch.all(out[2] == 0)


@pytest.mark.parametrize("spec", [c for c in G.load_cases() if c["kind"] == "decode"], ids=lambda c: c["name"])
def test_decode_golden_closed_forms(spec):
    case = G.build(spec)
    g = GpuCase(case, append=False)
    compare(g.decode(), G.expected(spec), spec["name"])


def test_decode_flags_out_of_pool_block():
    case = W.random_case(13, batch=2, num_heads=8, num_kv_heads=2, head_dim=128, min_len=40, max_len=60)
    g = GpuCase(case)
    bt = case.block_tables.clone()
    bt[1, 1] = case.num_blocks + 7
    pa.pa_decode(g.pool, g.q, bt.cuda(), g.sl, case.scale)
    assert pa.pa_device_status(clear=True) == pa.PA_DEV_OUT_OF_RANGE
    # the other sequence is untouched by the bad id
    out = pa.pa_decode(g.pool, g.q, bt.cuda(), g.sl, case.scale)
    pa.pa_device_status(clear=True)
    ref = oracle_decode(case)
    compare(out[:1], ref[:1], "good sequence next to a bad block id")


# ------------------------------------------------------------------ split-KV + combine
def _check_split(case, P, pool=None):
    g = GpuCase(case)
    ws_o, ws_lse = g.splitkv(P)
    k, v = pool if pool is not None else oracle_pool(case)
    orc = oracle.load()
    o_ref, lse_ref = orc.decode_partitions(k, v, u16(case.q), case.block_tables.numpy(), case.seq_lens.numpy(),
                                           case.scale, P)
    lse = ws_lse.cpu().double().numpy()
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse), fin), "empty partitions must have lse = -inf"
    assert np.all(np.isneginf(lse[~fin]))
    if fin.any():
        assert np.max(np.abs(lse[fin] - lse_ref[fin])) <= 1e-2
    compare(ws_o[torch.from_numpy(fin).to(ws_o.device)], o_ref[fin], f"{case.name} P={P} partial O")
    out = pa.pa_combine(ws_o, ws_lse)
    compare(out, orc.decode(k, v, u16(case.q), case.block_tables.numpy(), case.seq_lens.numpy(), case.scale),
            f"{case.name} P={P} combined")
    check_status_clean(f"split P={P}")
    return out


@pytest.mark.parametrize("P", [8, 15, 16, 19, 32])
def test_splitkv_4x8192(P):
    """P = 15 is the count the library suggests for 4 sequences x 8 kv heads on 152 SMs, the
    one the benchmark runs (partitions of 34 and 35 blocks); 19 fills one wave of four CTAs
    per SM exactly."""
    case = W.splitkv_decode(1004, 4, 8192)
    _check_split(case, P)


@pytest.mark.parametrize("P", [8, 16, 32])
def test_splitkv_1x32768(P):
    """P = 16 is the count the library suggests for 1 sequence x 8 kv heads (each partition
    on a 4-CTA cluster), the one the benchmark runs."""
    case = W.splitkv_decode(1004, 1, 32768)
    _check_split(case, P)


@pytest.mark.parametrize("P", [1, 2, 3, 8, 64])
def test_splitkv_ragged_and_empty_partitions(P):
    case = W.random_case(4000 + P, batch=6, num_heads=16, num_kv_heads=2, head_dim=128, min_len=1, max_len=300)
    _check_split(case, P)


def test_splitkv_one_partition_equals_decode():
    case = W.random_case(4100, batch=4, num_heads=32, num_kv_heads=8, head_dim=128, min_len=50, max_len=200)
    g = GpuCase(case)
    dec = g.decode()
    ws_o, ws_lse = g.splitkv(1)
    merged = pa.pa_combine(ws_o, ws_lse)
    assert (merged.float() - dec.float()).abs().max().item() <= 2 ** -7


def test_splitkv_golden_partitions():
    spec = [c for c in G.load_cases() if c["name"] == "three_blocks"][0]
    case = G.build(spec)
    g = GpuCase(case, append=False)
    for P in (2, 3, 4):
        ws_o, ws_lse = g.splitkv(P)
        wo, wl = G.expected_partitions(spec, P)
        fin = np.isfinite(wl)
        lse = ws_lse[0, 0].cpu().double().numpy()
        assert np.all(np.isneginf(lse[~fin]))
        assert np.max(np.abs(lse[fin] - wl[fin])) <= 1e-3
        assert np.max(np.abs(ws_o[0, 0].cpu().double().numpy() - wo)) <= 1e-3
        compare(pa.pa_combine(ws_o, ws_lse), G.expected(spec), f"golden P={P}")


# ------------------------------------------------------------------ chunked prefill
def test_prefill_chunked_full_size_whole():
    """The full workload (8 x 256-token chunks over a shared 768-token prefix), the launch the
    benchmark times, every one of its 2048 x 32 x 128 output elements against the oracle."""
    case = W.chunked_prefill()
    g = GpuCase(case)
    out = g.prefill()
    check_status_clean("chunked_prefill")
    compare(out, oracle_prefill(case), "chunked_prefill 8x256 over 768 (whole)")


def test_prefill_chunked_reduced_whole():
    case = W.chunked_prefill(seed=1105, batch=3, prefix_blocks=5, chunk=100)
    g = GpuCase(case)
    compare(g.prefill(), oracle_prefill(case), "chunked_prefill reduced")
    check_status_clean("prefill reduced")


@pytest.mark.parametrize("hq,hkv,d", [(4, 4, 64), (8, 2, 64), (32, 8, 128), (16, 2, 128), (12, 4, 128), (64, 8, 128)])
def test_prefill_ragged_sweep(hq, hkv, d):
    for j, shared in enumerate((0, 32)):
        case = W.random_case(5000 + hq * 7 + hkv + d + j, batch=4, num_heads=hq, num_kv_heads=hkv, head_dim=d,
                             min_len=1 + shared, max_len=200, q_len=70, prefill=True, shared_prefix_tokens=shared)
        g = GpuCase(case)
        compare(g.prefill(), oracle_prefill(case), f"prefill {hq}/{hkv}/{d} shared {shared}")
    check_status_clean("prefill sweep")


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 8), (32, 8), (64, 8), (64, 4), (64, 2)],
                         ids=["g1", "g2", "g4", "g8", "g16", "g32"])
def test_prefill_group_sweep(hq, hkv):
    """Every group size the tensor-core prefill takes from 1 to 32 (128 to 4 queries a tile),
    chunks of up to 300 queries over sequences of up to 700 tokens -- several query tiles, odd
    tile counts (a pair with one tile), ragged last tiles and sequence ends inside a stage --
    without and with a 48-token shared prefix."""
    for j, shared in enumerate((0, 48)):
        case = W.random_case(5400 + hq + 3 * hkv + j, batch=4, num_heads=hq, num_kv_heads=hkv, head_dim=128,
                             min_len=1 + shared, max_len=700, q_len=300, prefill=True, shared_prefix_tokens=shared)
        g = GpuCase(case)
        compare(g.prefill(), oracle_prefill(case), f"prefill group {hq // hkv} shared {shared}")
    check_status_clean("prefill group sweep")


def test_prefill_late_dominant_keys_rebase():
    """Keys far into the cached prefix whose scores exceed everything before them by far more
    than the lazy re-basing threshold (2^8): rows re-base in stages wholly below the diagonal,
    which rescales O and the stage's stored P.  Planted by overwriting, in the pool and in the
    unpaged copy alike, the K rows of tokens 700 and 1500 of every sequence with 4x a query of
    the chunk (its own score is then about 4|q|^2 scale = 45, against about 1 elsewhere)."""
    case = W.random_case(5710, batch=3, num_heads=32, num_kv_heads=8, head_dim=128, min_len=1700, max_len=1900,
                         q_len=256, prefill=True)
    g_ = case.group
    for s_, tok in ((0, 700), (1, 1500), (2, 700), (2, 1500)):
        L = int(case.seq_lens[s_])
        blk, off = int(case.block_tables[s_, tok // 16]), tok % 16
        q0 = int(case.cu_q_lens[s_]) + 5
        for kvh in range(case.num_kv_heads):
            row = (case.q[q0, kvh * g_].float() * 4).to(torch.bfloat16)
            case.k_cache[blk, kvh, off] = row
            case.k_seq[s_][tok, kvh] = row
    g = GpuCase(case)
    compare(g.prefill(), oracle_prefill(case), "prefill, late dominant keys (re-base below the diagonal)")
    check_status_clean("late dominant keys")


def test_prefill_large_scale_peaked_rows():
    """Scores spread far wider than 1/sqrt(d) would make them (scale 0.25 at d = 128): a few
    weights dominate each row, and the bf16 rounding of P alone took single elements at |o| ~ 2
    past the 1e-2 bound (1.004e-2 and 1.079e-2, found by a random sweep of prefill shapes); the
    prefill then carries P as bf16 high and low halves."""
    for seed, kw in ((113006, dict(batch=4, num_heads=128, num_kv_heads=8, max_len=200, q_len=5)),
                     (121020, dict(batch=6, num_heads=8, num_kv_heads=2, max_len=1300, q_len=400))):
        case = W.random_case(seed, head_dim=128, min_len=1, prefill=True, scale=0.25, **kw)
        g = GpuCase(case)
        compare(g.prefill(), oracle_prefill(case), f"prefill scale 0.25, seed {seed}")
    check_status_clean("large scale")


def test_decode_few_keys():
    """Sequences of 2 to 4 tokens: a row's softmax then rests on a few weights, whose bf16
    rounding (up to 2^-9 of each) is not averaged away.  With P as one bf16 value these seeds
    put single elements past the 1e-2 bound, at the usual scale and at 0.25 (found with a numpy
    model of that arithmetic; seed 97003 of the random sweep was 1.008e-2 off on the GPU).
    Decode carries P as high and low bf16 parts."""
    for seed, scale in ((7109, None), (7096, None), (7118, None), (7017, 0.25), (7068, 0.25)):
        case = W.random_case(seed, batch=16, num_heads=32, num_kv_heads=8, head_dim=128, min_len=2, max_len=4,
                             scale=scale)
        compare(GpuCase(case).decode(), oracle_decode(case), f"decode few keys, seed {seed}")
    check_status_clean("decode few keys")


def test_prefill_first_queries_of_a_sequence():
    """Whole prompts as one chunk: a sequence's first queries see 1, 2, 3 ... keys, the same
    few-weight rows as a short decode, and with P as one bf16 value these seeds put single
    elements past the bound (the numpy model again).  The tiles that hold a query seeing at
    most 128 keys carry P as two halves; the last case mixes such tiles with long ones in one
    launch.  Head dim 64 and groups that do not divide 128 (3, 6) run on the warp-MMA kernel,
    which carries two parts throughout."""
    for seed, H, hkv, d, L in ((8036, 32, 8, 128, 40), (8120, 64, 8, 128, 24), (8102, 32, 8, 128, 24),
                               (8111, 32, 8, 128, 24), (8339, 16, 4, 64, 24), (8301, 24, 8, 128, 24),
                               (8300, 48, 8, 64, 24)):
        case = W.paged_case(name="fresh", seed=seed, seq_lens=[L] * 8, q_lens=[L] * 8, new_lens=[L] * 8,
                            num_heads=H, num_kv_heads=hkv, head_dim=d, num_blocks=64)
        compare(GpuCase(case).prefill(), oracle_prefill(case), f"whole prompts, seed {seed}")
    mixed = W.paged_case(name="mixed", seed=8200, seq_lens=[24, 900, 200, 1500, 130], q_lens=[24, 200, 200, 64, 9],
                         new_lens=[24, 200, 200, 64, 9], num_heads=32, num_kv_heads=8, head_dim=128, num_blocks=256)
    compare(GpuCase(mixed).prefill(), oracle_prefill(mixed), "fresh and cached prompts in one launch")
    check_status_clean("first queries")


def test_prefill_one_row_chunk_equals_decode():
    case = W.random_case(5100, batch=5, num_heads=32, num_kv_heads=8, head_dim=128, min_len=20, max_len=300)
    g = GpuCase(case)
    dec = g.decode()
    cu = torch.arange(case.batch + 1, dtype=torch.int32, device="cuda")
    pre = pa.pa_prefill_chunked(g.pool, g.q, cu, g.bt, g.sl, case.scale, 1)
    # same arithmetic order is not required; both must be within tolerance of the oracle
    ref = oracle_decode(case)
    compare(dec, ref, "decode")
    compare(pre, ref, "one-row prefill")


def test_prefill_golden_causal_chunk():
    spec = [c for c in G.load_cases() if c["kind"] == "prefill"][0]
    case = G.build(spec)
    g = GpuCase(case, append=False)
    compare(g.prefill(), G.expected(spec), spec["name"])


@pytest.mark.parametrize("scale", [-0.09, 0.0, 0.3])
@pytest.mark.parametrize("d", [64, 128])
def test_scale_sign_and_zero(scale, d):
    """A negative, zero or large softmax scale: zero gives the mean of the visible values,
    a negative scale weights the least similar keys most."""
    case = W.random_case(5200 + d, batch=3, num_heads=16, num_kv_heads=4, head_dim=d, min_len=1, max_len=180,
                         q_len=40, prefill=True, shared_prefix_tokens=16, scale=scale)
    g = GpuCase(case)
    compare(g.prefill(), oracle_prefill(case), f"prefill scale {scale} d {d}")
    dec = W.random_case(5300 + d, batch=3, num_heads=16, num_kv_heads=4, head_dim=d, min_len=1, max_len=400,
                        scale=scale)
    gd = GpuCase(dec)
    compare(gd.decode(), oracle_decode(dec), f"decode scale {scale} d {d}")
    ws_o, ws_lse = gd.splitkv(4)
    compare(pa.pa_combine(ws_o, ws_lse), oracle_decode(dec), f"split-KV scale {scale} d {d}")
    check_status_clean("scale sweep")


FUSED_CASES = {
    # one CTA per (sequence, kv head)
    "batched_decode": lambda: W.batched_decode(),
    # one sequence: split over a 16-CTA cluster, the last member owns the new token's block
    "one_seq_cluster": lambda: W.random_case(5400, batch=1, num_heads=32, num_kv_heads=8, head_dim=128,
                                             min_len=1100, max_len=1200),
    # d = 64, single kv head, tokens landing at every offset of a block
    "tiny_d64": lambda: W.random_case(5401, batch=6, num_heads=4, num_kv_heads=1, head_dim=64, min_len=1, max_len=40),
    # group 8, ragged lengths
    "g8_ragged": lambda: W.random_case(5402, batch=5, num_heads=64, num_kv_heads=8, head_dim=128, min_len=1,
                                       max_len=700),
}


@pytest.mark.parametrize("name", sorted(FUSED_CASES))
def test_append_decode_fused(name):
    """pa_append_decode equals pa_kv_append then pa_decode: the pool afterwards is
    bit-identical to the oracle's append, the output matches the oracle's decode."""
    case = FUSED_CASES[name]()
    assert list(case.q_lens) == [1] * case.batch and case.k_new.shape[0] == case.batch
    g = GpuCase(case, append=False)  # the new rows' slots still hold NaN
    out = pa.pa_append_decode(g.pool, g.k_new, g.v_new, g.slots, g.q, g.bt, g.sl, case.scale)
    check_status_clean(f"fused {name}")
    k_ref, v_ref = oracle_pool(case)
    assert np.array_equal(u16(g.k.cpu()), k_ref) and np.array_equal(u16(g.v.cpu()), v_ref), "pool after fused append"
    compare(out, oracle_decode(case), f"fused append+decode {name}")


def test_append_decode_slot_checks():
    """A skipped slot (< 0) is not written; a slot that is not token seq_len-1 of its sequence
    is reported (PA_DEV_OUT_OF_RANGE) and not written; the other sequences are unaffected."""
    case = W.random_case(5403, batch=4, num_heads=32, num_kv_heads=8, head_dim=128, min_len=20, max_len=300)
    g = GpuCase(case, append=False)
    slots = g.slots.clone()
    good0, good1 = int(slots[0]), int(slots[1])
    slots[0] = -1                        # skip
    slots[1] = good1 + 1 if good1 % 16 != 15 else good1 - 1  # a neighbouring slot: wrong token
    k_before = u16(g.k.cpu()).copy()
    out = pa.pa_append_decode(g.pool, g.k_new, g.v_new, slots, g.q, g.bt, g.sl, case.scale)
    flags = pa.pa_device_status(clear=True)
    assert flags == pa.PA_DEV_OUT_OF_RANGE, f"status {flags:#x}"
    k_after = u16(g.k.cpu())
    def rows(slot):
        blk, off = divmod(slot, 16)
        return k_after[blk, :, off, :], k_before[blk, :, off, :]
    for s in (good0, good1, int(slots[1])):
        after, before = rows(s)
        assert np.array_equal(after, before), f"slot {s} written"
    # sequences 2 and 3 were appended and decoded normally
    k_ref, v_ref = oracle_pool(case)
    ref = oracle_decode(case, (k_ref, v_ref))
    compare(out[2:], ref[2:], "fused, untouched sequences")


@pytest.mark.parametrize("hq,hkv,d,q_len,shared", [(32, 8, 128, 4, 0), (32, 8, 128, 3, 32), (64, 8, 128, 2, 0),
                                                   (16, 4, 64, 4, 16), (4, 4, 64, 16, 0), (8, 8, 128, 16, 0)])
def test_multi_query_decode(hq, hkv, d, q_len, shared):
    """Chunks of a few queries (the shape of a speculative-decoding verify) with
    chunk x group <= 16 run on the decode kernel, their (query, head) rows on the MMA N
    dimension with a causal mask per column; ragged chunk lengths, chunks that start
    anywhere inside a block, a shared prefix."""
    case = W.random_case(5500 + hq + hkv + d + q_len + shared, batch=6, num_heads=hq, num_kv_heads=hkv,
                         head_dim=d, min_len=1 + shared, max_len=300, q_len=q_len, prefill=True,
                         shared_prefix_tokens=shared)
    assert max(case.q_lens) * (hq // hkv) <= 16
    g = GpuCase(case)
    compare(g.prefill(), oracle_prefill(case), f"multi-query {hq}/{hkv}/{d} C<={q_len}")
    check_status_clean("multi-query decode")


def test_multi_query_decode_cluster_and_empty_chunk():
    """One long sequence (split over a CTA cluster) with a 4-query chunk, and a batch in
    which one sequence has an empty chunk and another is all chunk (C == seq_len)."""
    c1 = W.paged_case(name="mq_cluster", seed=5510, seq_lens=[1131], q_lens=[4], new_lens=[4], num_heads=32,
                      num_kv_heads=8, head_dim=128, num_blocks=4096)
    g1 = GpuCase(c1)
    compare(g1.prefill(), oracle_prefill(c1), "multi-query over a cluster")
    c2 = W.paged_case(name="mq_empty", seed=5511, seq_lens=[40, 3, 18, 77], q_lens=[0, 3, 2, 4],
                      new_lens=[0, 3, 2, 4], num_heads=16, num_kv_heads=4, head_dim=128, num_blocks=64)
    g2 = GpuCase(c2)
    compare(g2.prefill(), oracle_prefill(c2), "multi-query with an empty chunk")
    check_status_clean("multi-query cluster / empty chunk")


def test_prefix_cache_warm_hit_end_to_end():
    """The block manager and the kernels together: a cold request's 800 prompt tokens go
    into the pool through its slots; after it is released, a warm request with the same
    first 768 tokens is admitted with those 48 blocks shared, appends only its own 256
    tokens and runs the chunked prefill over the cached prefix.  The output matches the
    oracle's prefill over the warm request's whole sequence."""
    Hq, Hkv, D, nblk = 32, 8, 128, 160
    gen = torch.Generator().manual_seed(6001)
    bf = lambda *s: torch.randn(*s, generator=gen).to(torch.bfloat16)
    bm = pa.BlockManager(nblk)
    toks_a = torch.randint(0, 5000, (800,), generator=gen).tolist()
    table_a, cached_a = bm.admit(1, toks_a, 0)
    assert cached_a == 0
    k_pool = torch.full((nblk, Hkv, 16, D), float("nan"), dtype=torch.bfloat16)
    v_pool = k_pool.clone()
    k_np, v_np = u16(k_pool).copy(), u16(v_pool).copy()      # the oracle's own pool
    kd, vd = k_pool.cuda(), v_pool.cuda()
    pool = pa.PaPool(kd, vd)
    orc = oracle.load()
    k_a, v_a = bf(800, Hkv, D), bf(800, Hkv, D)
    slots_a = bm.slots(1, 0, 800)
    pa.pa_kv_append(pool, k_a.cuda(), v_a.cuda(), torch.from_numpy(slots_a).cuda())
    orc.kv_append(k_np, v_np, u16(k_a), u16(v_a), slots_a)
    bm.commit(1, [], 800)
    bm.release(1)

    toks_b = toks_a[:768] + torch.randint(0, 5000, (256,), generator=gen).tolist()
    table_b, cached_b = bm.admit(2, toks_b, 0)
    assert cached_b == 768 and list(table_b[:48]) == list(table_a[:48])
    k_b, v_b = bf(256, Hkv, D), bf(256, Hkv, D)
    slots_b = bm.slots(2, 768, 256)
    pa.pa_kv_append(pool, k_b.cuda(), v_b.cuda(), torch.from_numpy(slots_b).cuda())
    orc.kv_append(k_np, v_np, u16(k_b), u16(v_b), slots_b)
    q = bf(256, Hq, D)
    bt = torch.from_numpy(table_b.astype(np.int32)).view(1, -1)
    sl = torch.tensor([1024], dtype=torch.int32)
    cu = torch.tensor([0, 256], dtype=torch.int32)
    scale = 1.0 / math.sqrt(D)
    out = pa.pa_prefill_chunked(pool, q.cuda(), cu.cuda(), bt.cuda(), sl.cuda(), scale, 256)
    check_status_clean("warm prefix hit")
    assert np.array_equal(u16(kd.cpu()), k_np) and np.array_equal(u16(vd.cpu()), v_np)
    ref = orc.prefill(k_np, v_np, u16(q), cu.numpy(), bt.numpy(), sl.numpy(), scale)
    compare(out, ref, "warm prefix hit through the block manager")


def test_kv_copy_bit_exact():
    """pa_kv_copy moves whole pool rows (every kv head, K and V): against the same copies done
    on the host; skipped pairs (negative slot) and an out-of-pool slot (flagged) copy nothing."""
    case = W.random_case(6100, batch=4, num_heads=16, num_kv_heads=4, head_dim=128, min_len=100, max_len=300)
    g = GpuCase(case)
    k_ref, v_ref = oracle_pool(case)
    torch.cuda.synchronize()
    rng = np.random.default_rng(6100)
    nslots = case.num_blocks * 16
    perm = rng.permutation(nslots)
    src, dst = perm[:300].astype(np.int64), perm[300:600].astype(np.int64)  # disjoint
    src[5] = -1
    dst[7] = nslots + 2
    pa.pa_kv_copy(g.pool, torch.from_numpy(src).cuda(), torch.from_numpy(dst).cuda())
    assert pa.pa_device_status(clear=True) == pa.PA_DEV_OUT_OF_RANGE
    kf = k_ref.reshape(case.num_blocks, case.num_kv_heads, 16, -1)
    vf = v_ref.reshape(kf.shape)
    for s_, d_ in zip(src, dst):
        if s_ < 0 or d_ >= nslots:
            continue
        kf[d_ // 16, :, d_ % 16] = kf[s_ // 16, :, s_ % 16]
        vf[d_ // 16, :, d_ % 16] = vf[s_ // 16, :, s_ % 16]
    assert np.array_equal(u16(g.k.cpu()), kf) and np.array_equal(u16(g.v.cpu()), vf)


def test_prefix_cache_partial_block_hit_end_to_end():
    """A warm prefix that ends inside a block: a cold request's 800 tokens are appended and
    released; a warm request whose first 770 tokens match is admitted with 48 shared blocks and
    the first 2 rows of the 49th copied into its own block (pa_kv_copy, copy on write), appends
    only its own 254 tokens and runs the chunked prefill of those 254 queries over the 770
    cached ones.  The pool matches the oracle's pool (the cold append, then the warm request's
    rows 768-769 and 770-1023 appended by the oracle), and the output the oracle's prefill."""
    Hq, Hkv, D, nblk = 32, 8, 128, 160
    gen = torch.Generator().manual_seed(6002)
    bf = lambda *s: torch.randn(*s, generator=gen).to(torch.bfloat16)
    bm = pa.BlockManager(nblk)
    toks_a = torch.randint(0, 5000, (800,), generator=gen).tolist()
    table_a, cached_a, src, _ = bm.admit_cow(1, toks_a, 0)
    assert cached_a == 0 and len(src) == 0
    k_pool = torch.full((nblk, Hkv, 16, D), float("nan"), dtype=torch.bfloat16)
    v_pool = k_pool.clone()
    k_np, v_np = u16(k_pool).copy(), u16(v_pool).copy()      # the oracle's own pool
    kd, vd = k_pool.cuda(), v_pool.cuda()
    pool = pa.PaPool(kd, vd)
    orc = oracle.load()
    k_a, v_a = bf(800, Hkv, D), bf(800, Hkv, D)
    slots_a = bm.slots(1, 0, 800)
    pa.pa_kv_append(pool, k_a.cuda(), v_a.cuda(), torch.from_numpy(slots_a).cuda())
    orc.kv_append(k_np, v_np, u16(k_a), u16(v_a), slots_a)
    bm.commit(1, [], 800)
    bm.release(1)

    toks_b = toks_a[:770] + torch.randint(5000, 9000, (254,), generator=gen).tolist()
    table_b, cached_b, src, dst = bm.admit_cow(2, toks_b, 0)
    assert cached_b == 770 and list(table_b[:48]) == list(table_a[:48]) and table_b[48] not in table_a
    assert len(src) == 2
    pa.pa_kv_copy(pool, torch.from_numpy(src).cuda(), torch.from_numpy(dst).cuda())
    # the oracle's pool: the warm request's rows 768-769 are the cold request's (same tokens)
    orc.kv_append(k_np, v_np, u16(k_a[768:770]), u16(v_a[768:770]), bm.slots(2, 768, 2))
    k_b, v_b = bf(254, Hkv, D), bf(254, Hkv, D)
    slots_b = bm.slots(2, 770, 254)
    pa.pa_kv_append(pool, k_b.cuda(), v_b.cuda(), torch.from_numpy(slots_b).cuda())
    orc.kv_append(k_np, v_np, u16(k_b), u16(v_b), slots_b)
    q = bf(254, Hq, D)
    bt = torch.from_numpy(table_b.astype(np.int32)).view(1, -1)
    sl = torch.tensor([1024], dtype=torch.int32)
    cu = torch.tensor([0, 254], dtype=torch.int32)
    scale = 1.0 / math.sqrt(D)
    out = pa.pa_prefill_chunked(pool, q.cuda(), cu.cuda(), bt.cuda(), sl.cuda(), scale, 254)
    check_status_clean("partial-block prefix hit")
    assert np.array_equal(u16(kd.cpu()), k_np) and np.array_equal(u16(vd.cpu()), v_np)
    ref = orc.prefill(k_np, v_np, u16(q), cu.numpy(), bt.numpy(), sl.numpy(), scale)
    compare(out, ref, "warm prefix ending inside a block (copy on write)")


def test_decode_large_batch_and_pool():
    """2048 sequences (a grid dimension far past the SM count) over a 65536-block pool whose
    block ids run to the end of the pool; decode and the split-KV path."""
    case = W.random_case(5600, batch=2048, num_heads=8, num_kv_heads=1, head_dim=128, min_len=1, max_len=48,
                         num_blocks=65536)
    assert int(case.block_tables.max()) > 60000
    g = GpuCase(case)
    ref = oracle_decode(case)
    compare(g.decode(), ref, "decode, 2048 sequences")
    ws_o, ws_lse = g.splitkv(3)
    compare(pa.pa_combine(ws_o, ws_lse), ref, "split-KV, 2048 sequences")
    check_status_clean("large batch / pool")


def test_prefill_whole_sequence_chunks():
    """Chunks that are the whole sequence (no cached prefix): 1000 queries (32 query tiles, one
    CTA each), an odd tile count (517 queries) and a single token, in one launch whose shorter
    chunks leave most of the grid's tile ranks empty."""
    case = W.paged_case(name="whole_seq", seed=5601, seq_lens=[1000, 517, 1], q_lens=[1000, 517, 1],
                        new_lens=[1000, 517, 1], num_heads=32, num_kv_heads=8, head_dim=128, num_blocks=256)
    g = GpuCase(case)
    compare(g.prefill(), oracle_prefill(case), "whole-sequence chunks")
    check_status_clean("whole-sequence chunks")


@pytest.mark.parametrize("hq", [32, 64])
def test_prefill_row_limits_at_stage_ends(hq):
    """Rows whose causal limit falls exactly on the last key of a 64-key stage, or one past
    it, inside a warp whose other rows see fewer keys (group 4: 8 queries to a warp, group 8:
    4).  Every such warp must take the masked path together: a lane whose own limit alone
    reads "the whole stage" may not branch away from its warp's collective tensor-memory
    accesses.  Chunk lengths 33-40 over sequence ends 141-148 put rows on every stage end."""
    lens = [141, 142, 144, 147, 148, 129, 192, 193]
    qls = [33, 34, 36, 39, 40, 33, 64, 65]
    case = W.paged_case(name="stage_ends", seed=5604, seq_lens=lens, q_lens=qls, new_lens=qls, num_heads=hq,
                        num_kv_heads=8, head_dim=128, num_blocks=160)
    g = GpuCase(case)
    compare(g.prefill(), oracle_prefill(case), f"rows at stage ends, {hq} heads")
    check_status_clean("rows at stage ends")


def test_prefill_group16_and_oversized_max_chunk():
    """Group 16 on the tensor-core prefill (8 queries per 128-row tile), and a max_chunk far
    above the longest chunk (the grid is sized for it; the extra tiles have no rows)."""
    case = W.random_case(5602, batch=3, num_heads=64, num_kv_heads=4, head_dim=128, min_len=40, max_len=400,
                         q_len=150, prefill=True, shared_prefix_tokens=16)
    g = GpuCase(case)
    ref = oracle_prefill(case)
    compare(g.prefill(), ref, "prefill group 16")
    out = pa.pa_prefill_chunked(g.pool, g.q, g.cu, g.bt, g.sl, case.scale, 2000)
    compare(out, ref, "prefill with max_chunk 2000")
    check_status_clean("group 16 / oversized max_chunk")


def test_decode_seq_len_past_table_is_flagged():
    """seq_len beyond max_blocks * 16 is clamped to the table and reported; the other
    sequences are unaffected."""
    case = W.random_case(5603, batch=3, num_heads=8, num_kv_heads=2, head_dim=128, min_len=20, max_len=60)
    g = GpuCase(case)
    sl = g.sl.clone()
    sl[1] = case.block_tables.shape[1] * 16 + 5
    out = pa.pa_decode(g.pool, g.q, g.bt, sl, case.scale)
    assert pa.pa_device_status(clear=True) == pa.PA_DEV_OUT_OF_RANGE
    ref = oracle_decode(case)
    compare(out[[0, 2]], ref[[0, 2]], "decode beside a clamped sequence")


def test_prefill_max_chunk_below_a_chunk_is_flagged():
    """max_chunk smaller than a sequence's chunk: that chunk's tiles past the grid cannot be
    computed, and the device status says so; a chunk the grid covers comes out right."""
    case = W.paged_case(name="short_max_chunk", seed=5605, seq_lens=[400, 300], q_lens=[100, 40], new_lens=[100, 40],
                        num_heads=32, num_kv_heads=8, head_dim=128, num_blocks=64)
    g = GpuCase(case)
    pa.pa_device_status(clear=True)
    out = pa.pa_prefill_chunked(g.pool, g.q, g.cu, g.bt, g.sl, case.scale, 50)
    assert pa.pa_device_status(clear=True) == pa.PA_DEV_OUT_OF_RANGE
    ref = oracle_prefill(case)
    compare(out[100:], ref[100:], "the chunk the grid covers, beside one it does not")
    # the same on the multi-query decode route (max_chunk x g <= 16): a 10-query chunk against
    # max_chunk 4 is reported and skipped, the 3-query chunk beside it is right
    case = W.paged_case(name="short_max_chunk_mq", seed=5607, seq_lens=[300, 200], q_lens=[10, 3], new_lens=[10, 3],
                        num_heads=32, num_kv_heads=8, head_dim=128, num_blocks=48)
    g = GpuCase(case)
    pa.pa_device_status(clear=True)
    out = pa.pa_prefill_chunked(g.pool, g.q, g.cu, g.bt, g.sl, case.scale, 4)
    assert pa.pa_device_status(clear=True) == pa.PA_DEV_OUT_OF_RANGE
    compare(out[10:], oracle_prefill(case)[10:], "a short chunk on the multi-query route beside an over-long one")


def test_prefill_flags_out_of_pool_block():
    """A block id past the pool in one sequence's table is reported, read as a valid block
    instead (never out of bounds), and leaves the other sequences' results right."""
    case = W.random_case(5606, batch=3, num_heads=32, num_kv_heads=8, head_dim=128, min_len=150, max_len=300,
                         q_len=80, prefill=True)
    g = GpuCase(case)
    bt = case.block_tables.clone()
    bt[1, 2] = case.num_blocks + 5
    pa.pa_device_status(clear=True)
    out = pa.pa_prefill_chunked(g.pool, g.q, g.cu, bt.cuda(), g.sl, case.scale, max(case.q_lens))
    assert pa.pa_device_status(clear=True) == pa.PA_DEV_OUT_OF_RANGE
    ref = oracle_prefill(case)
    cu = case.cu_q_lens.tolist()
    keep = np.r_[cu[0]:cu[1], cu[2]:cu[3]]
    compare(out[torch.from_numpy(keep).to(out.device)], ref[keep], "prefill beside a sequence with a bad block id")


def test_bounded_wait_reports_timeout_and_context_stays_usable():
    """A device wait that runs out (an mbarrier nothing arrives on, waited for through the
    kernels' own bounded helper with a short limit) sets PA_DEV_TIMEOUT and returns; nothing
    faults, and the next calls on the same context are right and report clean."""
    import time
    pa.pa_device_status(clear=True)
    t0 = time.time()
    pa.pa_selftest_wait_timeout(2_000_000)  # about a millisecond of SM cycles
    assert pa.pa_device_status(clear=True) == pa.PA_DEV_TIMEOUT
    assert time.time() - t0 < 5.0
    case = W.random_case(5608, batch=4, num_heads=32, num_kv_heads=8, head_dim=128, min_len=50, max_len=400)
    compare(GpuCase(case).decode(), oracle_decode(case), "decode right after a wait that ran out")
    check_status_clean("after the timeout self-test")


def test_prefill_invalid_sequence_is_skipped():
    """A sequence whose chunk is longer than its length is skipped and flagged: its rows are
    not written, and the sequences around it come out right."""
    case = W.random_case(5701, batch=4, num_heads=32, num_kv_heads=8, head_dim=128, min_len=200, max_len=400,
                         q_len=200, prefill=True)
    g = GpuCase(case)
    sl = g.sl.clone()
    sl[1] = case.q_lens[1] - 1  # L < C
    out = torch.zeros_like(g.q)
    pa.pa_prefill_chunked(g.pool, g.q, g.cu, g.bt, sl, case.scale, max(case.q_lens), out=out)
    assert pa.pa_device_status(clear=True) == pa.PA_DEV_OUT_OF_RANGE
    ref = oracle_prefill(case)
    cu = case.cu_q_lens.tolist()
    keep = [i for b in (0, 2, 3) for i in range(cu[b], cu[b + 1])]
    compare(out[keep], ref[keep], "prefill beside a skipped sequence")
    assert not torch.any(out[cu[1]:cu[2]].float() != 0), "the skipped sequence's rows were written"


_CONCURRENT_FIRST_CALLS = r'''
import sys, threading
import numpy as np, torch
sys.path[:0] = [sys.argv[1], sys.argv[1] + "/tests"]
import paged_kv_gqa_slot_gb300 as pa
import workloads as W
from parity import GpuCase, compare, oracle_decode, oracle_prefill, oracle_pool
import oracle
cases = {
    "decode": W.random_case(5801, batch=6, num_heads=32, num_kv_heads=8, head_dim=128, min_len=30, max_len=500),
    "decode64": W.random_case(5802, batch=3, num_heads=8, num_kv_heads=2, head_dim=64, min_len=30, max_len=300),
    "split": W.random_case(5803, batch=2, num_heads=64, num_kv_heads=8, head_dim=128, min_len=300, max_len=900),
    "prefill": W.random_case(5804, batch=3, num_heads=32, num_kv_heads=8, head_dim=128, min_len=100, max_len=400,
                             q_len=150, prefill=True),
}
gpu = {k: GpuCase(c) for k, c in cases.items()}
torch.cuda.synchronize()
outs, errors = {}, []
barrier = threading.Barrier(len(cases))
def work(name):
    try:
        g, c = gpu[name], cases[name]
        st = torch.cuda.Stream()
        barrier.wait()
        with torch.cuda.stream(st):
            if name == "split":
                outs[name] = pa.pa_combine(*g.splitkv(5))
            elif name == "prefill":
                outs[name] = g.prefill()
            else:
                outs[name] = g.decode()
        st.synchronize()
    except Exception as e:  # reported by the main thread
        errors.append(f"{name}: {e!r}")
ts = [threading.Thread(target=work, args=(n,)) for n in cases]
for t in ts: t.start()
for t in ts: t.join()
assert not errors, errors
assert pa.pa_device_status(clear=True) == 0
for name, c in cases.items():
    ref = oracle_prefill(c) if name == "prefill" else oracle_decode(c)
    compare(outs[name], ref, f"concurrent first call: {name}")
print("ok")
'''


def test_concurrent_first_calls_from_threads(tmp_path):
    """The library's first calls in a process, from four host threads at once on their own
    streams (decode d128 and d64, split-KV with its merge, the tensor-core prefill): every
    kernel's one-time set-up runs under contention, and every result must still match the
    oracle."""
    import subprocess
    import sys
    from pathlib import Path
    script = tmp_path / "pa_threaded_first_calls.py"
    script.write_text(_CONCURRENT_FIRST_CALLS)
    root = str(Path(__file__).resolve().parents[1])
    r = subprocess.run([sys.executable, str(script), root], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-4000:]


_ALTERNATE_PREFILL = r'''
import sys
import torch
sys.path[:0] = [sys.argv[1], sys.argv[1] + "/tests"]
import workloads as W
from parity import GpuCase, compare, oracle_prefill, check_status_clean
cases = [
    W.chunked_prefill(seed=1105, batch=3, prefix_blocks=5, chunk=100),
    W.random_case(5901, batch=4, num_heads=32, num_kv_heads=8, head_dim=128, min_len=1, max_len=200, q_len=70,
                  prefill=True, shared_prefix_tokens=32),
    W.paged_case(name="stage_ends", seed=5604, seq_lens=[141, 142, 144, 147, 148, 129, 192, 193],
                 q_lens=[33, 34, 36, 39, 40, 33, 64, 65], new_lens=[33, 34, 36, 39, 40, 33, 64, 65],
                 num_heads=32, num_kv_heads=8, head_dim=128, num_blocks=160),
    W.random_case(5902, batch=3, num_heads=16, num_kv_heads=4, head_dim=128, min_len=1, max_len=180, q_len=40,
                  prefill=True, shared_prefix_tokens=16, scale=-0.09),
    W.random_case(5903, batch=3, num_heads=64, num_kv_heads=4, head_dim=128, min_len=40, max_len=400, q_len=150,
                  prefill=True, shared_prefix_tokens=16),
]
for i, c in enumerate(cases):
    compare(GpuCase(c).prefill(), oracle_prefill(c), f"{sys.argv[2]} prefill case {i}")
    check_status_clean(f"{sys.argv[2]} prefill case {i}")
# max_chunk below a chunk's length is reported; the chunk the grid covers is right
import paged_kv_gqa_slot_gb300 as pa
c = W.paged_case(name="short_max_chunk", seed=5605, seq_lens=[400, 300], q_lens=[100, 40], new_lens=[100, 40],
                 num_heads=32, num_kv_heads=8, head_dim=128, num_blocks=64)
g = GpuCase(c)
pa.pa_device_status(clear=True)
out = pa.pa_prefill_chunked(g.pool, g.q, g.cu, g.bt, g.sl, c.scale, 50)
assert pa.pa_device_status(clear=True) == pa.PA_DEV_OUT_OF_RANGE, "short max_chunk not reported"
compare(out[100:], oracle_prefill(c)[100:], f"{sys.argv[2]} chunk the grid covers")
# a block id past the pool is reported; the other sequences are right
import numpy as np
c = W.random_case(5606, batch=3, num_heads=32, num_kv_heads=8, head_dim=128, min_len=150, max_len=300, q_len=80,
                  prefill=True)
g = GpuCase(c)
bt = c.block_tables.clone()
bt[1, 2] = c.num_blocks + 5
pa.pa_device_status(clear=True)
out = pa.pa_prefill_chunked(g.pool, g.q, g.cu, bt.cuda(), g.sl, c.scale, max(c.q_lens))
assert pa.pa_device_status(clear=True) == pa.PA_DEV_OUT_OF_RANGE, "bad block id not reported"
cu = c.cu_q_lens.tolist()
keep = np.r_[cu[0]:cu[1], cu[2]:cu[3]]
compare(out[torch.from_numpy(keep).to(out.device)], oracle_prefill(c)[keep], f"{sys.argv[2]} beside a bad block id")
print("ok")
'''


@pytest.mark.parametrize("impl", ["t", "m"])
def test_alternate_prefill_kernels(impl, tmp_path):
    """The prefill kernels the default path does not pick for these shapes, forced by
    PA_PREFILL_IMPL in a child process (the choice is read once per process): t, the
    tensor-core kernel with Q in tensor memory and P in shared memory; m, the warp-MMA
    kernel.  Ragged chunks, rows on stage ends, a negative scale and group 16, against the
    oracle."""
    import os
    import subprocess
    import sys
    from pathlib import Path
    script = tmp_path / "pa_alternate_prefill.py"
    script.write_text(_ALTERNATE_PREFILL)
    root = str(Path(__file__).resolve().parents[1])
    env = dict(os.environ, PA_PREFILL_IMPL=impl)
    r = subprocess.run([sys.executable, str(script), root, impl], capture_output=True, text=True, timeout=600,
                       env=env)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-4000:]


def test_random_shape_sweep():
    """Seeded random shapes across the paths: chunked prefills (group 1 to 32, shared prefixes,
    short and long chunks, the usual, a negative and a large scale), split-KV partitions with
    their merge (P from 1 to 32, d 64 and 128) and chunks of two to four queries --
    each against the oracle.  The sweep that found the large-scale P rounding limit, kept small."""
    import random
    rng = random.Random(20261203)
    for it in range(36):
        hkv = rng.choice([1, 2, 4, 8])
        g = rng.choice([1, 2, 4, 8, 16, 32])
        if g * hkv > 128:
            g = 128 // hkv
        shared = rng.choice([0, 16, 48])
        scale = rng.choice([None, None, -0.07, 0.25])
        case = W.random_case(97000 + it, batch=rng.randint(1, 5), num_heads=g * hkv, num_kv_heads=hkv,
                             head_dim=128, min_len=1 + shared, max_len=rng.choice([60, 300, 900]) + shared,
                             q_len=rng.choice([5, 40, 200]), prefill=True, shared_prefix_tokens=shared, scale=scale)
        compare(GpuCase(case).prefill(), oracle_prefill(case), f"random prefill {it}")
        check_status_clean(f"random prefill {it}")
    for it in range(24):
        hkv = rng.choice([1, 2, 4, 8])
        g = rng.choice([1, 2, 4, 8, 16])
        d = rng.choice([64, 128])
        scale = rng.choice([None, 0.25, -0.2])
        case = W.random_case(98000 + it, batch=rng.randint(1, 6), num_heads=g * hkv, num_kv_heads=hkv, head_dim=d,
                             min_len=1, max_len=rng.choice([40, 700, 3000]), scale=scale)
        ws_o, ws_lse = GpuCase(case).splitkv(rng.choice([1, 2, 5, 8, 16, 32]))
        compare(pa.pa_combine(ws_o, ws_lse), oracle_decode(case), f"random split-KV {it}")
        pc = W.random_case(99000 + it, batch=rng.randint(1, 6), num_heads=g * hkv, num_kv_heads=hkv, head_dim=d,
                           min_len=2, max_len=rng.choice([40, 700]), q_len=rng.choice([2, 3, 4]), prefill=True,
                           scale=scale)
        compare(GpuCase(pc).prefill(), oracle_prefill(pc), f"random short chunks {it}")
        check_status_clean(f"random split-KV {it}")
