"""Checks that pin the CPU oracle to something other than itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError when
the oracle disagrees with what the definition of grouped-query attention over a
paged cache fixes ("Qwen3-4B / 8B / 32B", section "Architecture Notes": GQA with
32 query heads over 8 KV heads, Qwen3-32B group 8, paged KV cache):

* brute force: torch's fp64 scaled_dot_product_attention on the UNPAGED per-
  sequence K/V (kv heads repeated g times), for decode and causal chunks;
* invariance of the output under a relabelling of physical block ids;
* closed forms: identical keys give the mean of V, one key gives V_0;
* causal equivalence: decode at length L == a one-row chunk at position L-1;
* MHA expansion: repeating every kv head g times (group 1) changes nothing;
* split-KV: the partition log-sum-exp equals scipy's logsumexp of that
  partition's scores, the merge of the partitions equals the unsplit output,
  and P = 1 equals decode;
* the append equals numpy's indexed scatter of the same rows.

The planted-mistake tests run the same pins against mutated copies of the
oracle's C source and require each copy to fail at least one of them.
"""
from __future__ import annotations

import math

import numpy as np
import torch
from scipy.special import logsumexp

import workloads as W
from workloads import u16

ATOL_EXACT = 1e-12


def bf16_to_f64(t: torch.Tensor) -> torch.Tensor:
    return t.to(torch.float64)


def post_append_pool(orc, case):
    k = u16(case.k_cache).copy()
    v = u16(case.v_cache).copy()
    orc.kv_append(k, v, u16(case.k_new), u16(case.v_new), case.slot_mapping.numpy())
    return k, v


def oracle_attention(orc, case):
    """Oracle output for a case: decode -> [B, Hq, D], prefill -> [sum C, Hq, D]."""
    k, v = post_append_pool(orc, case)
    if case.is_decode:
        return orc.decode(k, v, u16(case.q), case.block_tables.numpy(), case.seq_lens.numpy(), case.scale)
    return orc.prefill(k, v, u16(case.q), case.cu_q_lens.numpy(), case.block_tables.numpy(),
                       case.seq_lens.numpy(), case.scale)


def sdpa_reference(case) -> np.ndarray:
    """Unpaged brute force: torch fp64 SDPA per sequence with an explicit causal mask."""
    g = case.group
    out = np.zeros((case.q.shape[0], case.num_heads, case.head_dim), dtype=np.float64)
    cu = case.cu_q_lens.tolist()
    for s in range(case.batch):
        L = int(case.seq_lens[s])
        C = cu[s + 1] - cu[s]
        if L == 0 or C == 0:
            continue
        q = bf16_to_f64(case.q[cu[s]:cu[s + 1]]).permute(1, 0, 2).unsqueeze(0)           # [1, Hq, C, D]
        k = bf16_to_f64(case.k_seq[s]).permute(1, 0, 2).repeat_interleave(g, dim=0)[None]  # [1, Hq, L, D]
        v = bf16_to_f64(case.v_seq[s]).permute(1, 0, 2).repeat_interleave(g, dim=0)[None]
        pos = torch.arange(L - C, L).unsqueeze(1)
        mask = torch.arange(L).unsqueeze(0) <= pos                                          # [C, L]
        o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=case.scale)
        out[cu[s]:cu[s + 1]] = o[0].permute(1, 0, 2).numpy()
    return out


def _small_cases():
    cases = [W.tiny_decode()]
    i = 0
    for hq, hkv, d in ((4, 1, 64), (8, 2, 128), (8, 8, 64), (16, 2, 128), (4, 4, 128)):
        for prefill in (False, True):
            cases.append(W.random_case(7000 + i, batch=3, num_heads=hq, num_kv_heads=hkv, head_dim=d,
                                       min_len=1, max_len=70, q_len=20, prefill=prefill,
                                       name=f"r{i}"))
            i += 1
    cases.append(W.random_case(7100, batch=2, num_heads=8, num_kv_heads=2, head_dim=64, min_len=40, max_len=60,
                               q_len=9, prefill=True, shared_prefix_tokens=32, name="shared"))
    return cases


def pin_bruteforce(orc):
    for case in _small_cases():
        got = oracle_attention(orc, case)
        ref = sdpa_reference(case)
        err = float(np.max(np.abs(got - ref)))
        assert err <= ATOL_EXACT, f"{case.name}: oracle vs unpaged SDPA max |diff| = {err}"


def _relabel_blocks(case, seed):
    """Same problem with physical block ids relabelled by a random permutation."""
    gen = W.generator(seed)
    perm = torch.randperm(case.num_blocks, generator=gen)           # new id of old block b is perm[b]
    k = torch.empty_like(case.k_cache)
    v = torch.empty_like(case.v_cache)
    k[perm] = case.k_cache
    v[perm] = case.v_cache
    bt = case.block_tables.clone()
    used = bt >= 0
    bt[used] = perm[bt[used].long()].to(torch.int32)
    sm = case.slot_mapping.clone()
    ok = sm >= 0
    sm[ok] = perm[(sm[ok] // case.block_size)].long() * case.block_size + sm[ok] % case.block_size
    return k, v, bt, sm


def pin_permutation(orc):
    for j, case in enumerate(_small_cases()[:6]):
        a = oracle_attention(orc, case)
        k, v, bt, sm = _relabel_blocks(case, 9000 + j)
        case2 = W.PagedCase(**{**case.__dict__, "k_cache": k, "v_cache": v, "block_tables": bt,
                               "slot_mapping": sm})
        b = oracle_attention(orc, case2)
        assert np.array_equal(a, b), f"{case.name}: output changed under block relabelling"


def _uniform_key_case(seed, L, d=64, hq=4, hkv=2):
    case = W.paged_case(name="same_keys", seed=seed, seq_lens=[L], q_lens=[1], new_lens=[0], num_heads=hq,
                        num_kv_heads=hkv, head_dim=d, num_blocks=8 + L // 16)
    # every key row of the sequence equals its first row
    k = case.k_cache.clone()
    bs = case.block_size
    for t in range(L):
        blk = int(case.block_tables[0, t // bs])
        k[blk, :, t % bs, :] = case.k_seq[0][0]
    return W.PagedCase(**{**case.__dict__, "k_cache": k})


def pin_closed_forms(orc):
    for L in (1, 5, 16, 17, 40):
        case = _uniform_key_case(500 + L, L)
        got = oracle_attention(orc, case)
        g = case.group
        vmean = bf16_to_f64(case.v_seq[0]).mean(dim=0).numpy()            # [Hkv, D]
        for h in range(case.num_heads):
            want = vmean[h // g]
            if L == 1:
                assert np.array_equal(got[0, h], want), "single key must return V_0 exactly"
            else:
                err = float(np.max(np.abs(got[0, h] - want)))
                assert err <= ATOL_EXACT, f"identical keys: |o - mean V| = {err} (L={L}, h={h})"


def pin_causal_equivalence(orc):
    for j, case in enumerate(_small_cases()):
        if not case.is_decode:
            continue
        # the same problem read as prefill: a one-row chunk at position L-1
        dec = oracle_attention(orc, case)
        k, v = post_append_pool(orc, case)
        sl = case.seq_lens.numpy()
        cu = np.arange(case.batch + 1, dtype=np.int32)
        pre = orc.prefill(k, v, u16(case.q), cu, case.block_tables.numpy(), sl, case.scale)
        assert np.array_equal(dec, pre), f"{case.name}: decode != one-row prefill"


def pin_mha_expansion(orc):
    for case in _small_cases():
        g = case.group
        if g == 1:
            continue
        a = oracle_attention(orc, case)
        # kv head j of the expanded problem holds the copy of original kv head j // g
        k = case.k_cache.repeat_interleave(g, dim=1)
        v = case.v_cache.repeat_interleave(g, dim=1)
        kn = case.k_new.repeat_interleave(g, dim=1)
        vn = case.v_new.repeat_interleave(g, dim=1)
        case2 = W.PagedCase(**{**case.__dict__, "k_cache": k, "v_cache": v, "k_new": kn, "v_new": vn,
                               "num_kv_heads": case.num_heads})
        b = oracle_attention(orc, case2)
        assert np.array_equal(a, b), f"{case.name}: GQA output != MHA-expanded output"


def pin_split(orc):
    cases = [c for c in _small_cases() if c.is_decode]
    cases.append(W.random_case(7300, batch=2, num_heads=8, num_kv_heads=1, head_dim=64, min_len=100,
                               max_len=300, name="longer"))
    for case in cases:
        k, v = post_append_pool(orc, case)
        q, bt, sl = u16(case.q), case.block_tables.numpy(), case.seq_lens.numpy()
        full = orc.decode(k, v, q, bt, sl, case.scale)
        for P in (1, 2, 3, 8, 64):
            o, lse = orc.decode_partitions(k, v, q, bt, sl, case.scale, P)
            merged = orc.combine(o, lse)
            err = float(np.max(np.abs(merged - full)))
            assert err <= ATOL_EXACT, f"{case.name} P={P}: merge of partitions != unsplit, {err}"
            if P == 1:
                assert np.array_equal(o[:, :, 0, :], full), "P = 1 must equal decode"
            # each partition's lse against scipy on the unpaged scores
            bs = case.block_size
            for b in range(case.batch):
                L = int(sl[b])
                nb = -(-L // bs)
                per = -(-nb // P)
                kk = bf16_to_f64(case.k_seq[b])
                for h in range(case.num_heads):
                    qh = bf16_to_f64(case.q[b, h])
                    scores = (kk[:, h // case.group, :] @ qh).numpy() * case.scale
                    for j in range(P):
                        t0, t1 = j * per * bs, min((j + 1) * per * bs, L)
                        if t1 <= t0:
                            assert lse[b, h, j] == -math.inf and not np.any(o[b, h, j]), "empty partition"
                        else:
                            want = logsumexp(scores[t0:t1])
                            assert abs(lse[b, h, j] - want) <= 1e-12 * max(1.0, abs(want)), \
                                f"{case.name} P={P}: lse mismatch {lse[b, h, j]} vs {want}"


def pin_append(orc):
    for case in _small_cases() + [W.batched_decode(batch=4)]:
        k = u16(case.k_cache).copy()
        v = u16(case.v_cache).copy()
        orc.kv_append(k, v, u16(case.k_new), u16(case.v_new), case.slot_mapping.numpy())
        # numpy's indexed scatter of the same rows into the same layout
        kk = u16(case.k_cache).copy()
        vv = u16(case.v_cache).copy()
        sm = case.slot_mapping.numpy()
        keep = sm >= 0
        blk, off = sm[keep] // case.block_size, sm[keep] % case.block_size
        kk[blk, :, off, :] = u16(case.k_new)[keep]
        vv[blk, :, off, :] = u16(case.v_new)[keep]
        assert np.array_equal(k, kk) and np.array_equal(v, vv), f"{case.name}: append differs from scatter"


ALL_PINS = [pin_bruteforce, pin_permutation, pin_closed_forms, pin_causal_equivalence, pin_mha_expansion,
            pin_split, pin_append]
