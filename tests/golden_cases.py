"""Build paged inputs from the hand-derived worked examples in golden/closed_forms.json.

Input construction only (no attention arithmetic): vectors are filled as the
fixture states and laid into the pool at the fixture's physical block ids.
Expected values are the fixture's closed-form expressions, evaluated with math.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "closed_forms.json")
_NAMES = {"e": math.e, "exp": math.exp, "log": math.log, "tanh": math.tanh, "inf": math.inf}


def _vec(spec, d):
    if isinstance(spec, (int, float)):
        return torch.full((d,), float(spec), dtype=torch.float32)
    v = torch.zeros(d, dtype=torch.float32)
    v[int(spec["onehot"])] = float(spec["value"])
    return v


def _expect(spec, d):
    rest = eval(spec.get("rest", "0"), {"__builtins__": {}}, _NAMES)
    out = np.full(d, float(rest))
    for key, expr in spec.items():
        if key != "rest":
            out[int(key)] = float(eval(expr, {"__builtins__": {}}, _NAMES))
    return out


def load_cases():
    with open(GOLDEN) as f:
        data = json.load(f)
    return data["cases"]


def build(case: dict) -> W.PagedCase:
    d, hq, hkv, bs = case["head_dim"], case["num_heads"], case["num_kv_heads"], W.BLOCK_SIZE
    if "k_blocks" in case:
        L = case["seq_len"]
        k_rows = [case["k_blocks"][t // bs] for t in range(L)]
        v_rows = [case["v_blocks"][t // bs] for t in range(L)]
    else:
        k_rows, v_rows = case["k"], case["v"]
        L = len(k_rows)
    k_seq = torch.stack([torch.stack([_vec(k_rows[t][h], d) for h in range(hkv)]) for t in range(L)])
    v_seq = torch.stack([torch.stack([_vec(v_rows[t][h], d) for h in range(hkv)]) for t in range(L)])
    k_seq, v_seq = k_seq.to(torch.bfloat16), v_seq.to(torch.bfloat16)
    nq = len(case["q"])
    q = torch.stack([torch.stack([_vec(case["q"][i][h], d) for h in range(hq)]) for i in range(nq)])
    q = q.to(torch.bfloat16)
    bt_row = case["block_table"]
    nblk = case["num_blocks"]
    k_cache = W.bf16_filled((nblk, hkv, bs, d), W.BF16_NAN_BITS)
    v_cache = W.bf16_filled((nblk, hkv, bs, d), W.BF16_NAN_BITS)
    for t in range(L):
        k_cache[bt_row[t // bs], :, t % bs, :] = k_seq[t]
        v_cache[bt_row[t // bs], :, t % bs, :] = v_seq[t]
    decode = case["kind"] == "decode"
    q_lens = [1] if decode else [nq]
    return W.PagedCase(
        name=case["name"], seed=0, num_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs, num_blocks=nblk,
        scale=float(case["scale"]), k_cache=k_cache, v_cache=v_cache,
        block_tables=torch.tensor([bt_row], dtype=torch.int32), seq_lens=torch.tensor([L], dtype=torch.int32),
        q=q, q_lens=q_lens, cu_q_lens=torch.tensor([0, q_lens[0]], dtype=torch.int32),
        k_new=torch.zeros((0, hkv, d), dtype=torch.bfloat16), v_new=torch.zeros((0, hkv, d), dtype=torch.bfloat16),
        slot_mapping=torch.zeros(0, dtype=torch.int64), k_seq=[k_seq], v_seq=[v_seq])


def expected(case: dict) -> np.ndarray:
    """[rows, Hq, D] closed-form outputs."""
    d = case["head_dim"]
    return np.stack([np.stack([_expect(h, d) for h in row]) for row in case["expected"]])


def expected_partitions(case: dict, P: int):
    spec = case["partitions"][str(P)]
    d = case["head_dim"]
    lse = np.array([float(eval(x, {"__builtins__": {}}, _NAMES)) for x in spec["lse"]])
    o = np.stack([_expect(x, d) for x in spec["o"]])
    return o, lse
