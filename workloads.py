"""Seeded synthetic inputs for paged grouped-query attention.

This module draws tensors and lays them out in a block-paged KV pool; it holds
none of the attention arithmetic.  Both sides of every parity check read their
inputs from here: the CPU oracle (through numpy views of the same bf16 bits)
and the CUDA library (through device copies of the same tensors).

Layout of the pool (a design choice; the pages fix only the 16-token block,
"Qwen3-4B / 8B / 32B", section "Qwen3-32B Serving Load", 21.4 GB = 5360 blocks):

  k_cache, v_cache : [num_blocks, num_kv_heads, block_size, head_dim] bf16
  slot             : block_id * block_size + offset_in_block
  block_tables     : [batch, max_blocks] int32, entry j = physical block of the
                     sequence's logical block j, -1 past the last used block
  seq_lens         : [batch] int32, tokens in the sequence INCLUDING any tokens
                     delivered by the append that precedes the attention call

Every value is drawn as fp32 N(0, 1) from a seeded CPU torch.Generator and
rounded to bf16 (round-to-nearest-even, torch's cast).  Pool slots that no
sequence owns, and the slots the append will write, hold bf16 NaN, so any read
outside a sequence shows up as NaN in the output.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np
import torch

BLOCK_SIZE = 16
BF16_NAN_BITS = 0x7FC0


def generator(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def bf16_randn(gen: torch.Generator, *shape: int) -> torch.Tensor:
    return torch.randn(*shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def bf16_filled(shape, bits: int) -> torch.Tensor:
    t = torch.empty(shape, dtype=torch.int16)
    t.fill_(bits if bits < 0x8000 else bits - 0x10000)
    return t.view(torch.bfloat16)


def u16(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 array of the same bits (no copy if contiguous)."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


@dataclass
class PagedCase:
    """One synthetic paged-attention problem (all tensors on the CPU)."""
    name: str
    seed: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    scale: float
    k_cache: torch.Tensor            # pool BEFORE the append
    v_cache: torch.Tensor
    block_tables: torch.Tensor       # [B, max_blocks] int32
    seq_lens: torch.Tensor           # [B] int32, after the append
    q: torch.Tensor                  # [sum(q_lens), Hq, D] bf16 (decode: [B, Hq, D])
    q_lens: List[int]
    cu_q_lens: torch.Tensor          # [B+1] int32
    k_new: torch.Tensor              # [T, Hkv, D] bf16, rows the append writes
    v_new: torch.Tensor
    slot_mapping: torch.Tensor       # [T] int64
    k_seq: List[torch.Tensor] = field(default_factory=list)   # per seq [L, Hkv, D], unpaged
    v_seq: List[torch.Tensor] = field(default_factory=list)
    notes: str = ""

    @property
    def batch(self) -> int:
        return int(self.seq_lens.numel())

    @property
    def group(self) -> int:
        return self.num_heads // self.num_kv_heads

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def is_decode(self) -> bool:
        return all(c == 1 for c in self.q_lens)

    def kv_bytes(self) -> int:
        """Bytes of K and V that the attention must read, counted once per kv head."""
        esz = 2
        return int(sum(int(L) for L in self.seq_lens.tolist())) * self.num_kv_heads * self.head_dim * esz * 2


def paged_case(*, name: str, seed: int, seq_lens: Sequence[int], q_lens: Sequence[int],
               num_heads: int, num_kv_heads: int, head_dim: int, num_blocks: int,
               new_lens: Optional[Sequence[int]] = None, shared_prefix_tokens: int = 0,
               block_size: int = BLOCK_SIZE, scale: Optional[float] = None,
               max_blocks: Optional[int] = None, gen: Optional[torch.Generator] = None,
               nan_fill: bool = True, notes: str = "") -> PagedCase:
    """Draw a paged problem.

    Sequence s holds seq_lens[s] tokens; its last q_lens[s] positions are the
    queries, its last new_lens[s] positions are delivered by the append (they are
    NaN in the returned pool).  With shared_prefix_tokens > 0 (a multiple of the
    block size) every sequence maps its first blocks to the same physical blocks,
    which hold one shared K/V content (a prefix-cache hit).
    """
    B = len(seq_lens)
    assert len(q_lens) == B
    new_lens = list(q_lens) if new_lens is None else list(new_lens)
    assert num_heads % num_kv_heads == 0
    assert shared_prefix_tokens % block_size == 0
    gen = generator(seed) if gen is None else gen
    Hkv, D, bs = num_kv_heads, head_dim, block_size
    for L, c, n in zip(seq_lens, q_lens, new_lens):
        assert 0 <= c <= max(L, 1) and 0 <= n <= L - shared_prefix_tokens
        assert L >= shared_prefix_tokens
    n_shared = shared_prefix_tokens // bs
    own_blocks = [math.ceil((L - shared_prefix_tokens) / bs) for L in seq_lens]
    need = n_shared + sum(own_blocks)
    assert need <= num_blocks, f"pool too small: {need} > {num_blocks}"
    nb_max = max([n_shared + o for o in own_blocks] + [1])
    max_blocks = nb_max if max_blocks is None else max_blocks
    assert max_blocks >= nb_max

    perm = torch.randperm(num_blocks, generator=gen)
    shared_ids = perm[:n_shared]
    cursor = n_shared
    block_tables = torch.full((B, max_blocks), -1, dtype=torch.int32)
    for s in range(B):
        ids = perm[cursor:cursor + own_blocks[s]]
        cursor += own_blocks[s]
        row = torch.cat([shared_ids, ids]).to(torch.int32)
        block_tables[s, :row.numel()] = row

    if nan_fill:
        k_cache = bf16_filled((num_blocks, Hkv, bs, D), BF16_NAN_BITS)
        v_cache = bf16_filled((num_blocks, Hkv, bs, D), BF16_NAN_BITS)
    else:
        k_cache = torch.zeros((num_blocks, Hkv, bs, D), dtype=torch.bfloat16)
        v_cache = torch.zeros((num_blocks, Hkv, bs, D), dtype=torch.bfloat16)

    k_shared = bf16_randn(gen, shared_prefix_tokens, Hkv, D)
    v_shared = bf16_randn(gen, shared_prefix_tokens, Hkv, D)
    k_seq, v_seq = [], []
    for s in range(B):
        own = seq_lens[s] - shared_prefix_tokens
        k_seq.append(torch.cat([k_shared, bf16_randn(gen, own, Hkv, D)]))
        v_seq.append(torch.cat([v_shared, bf16_randn(gen, own, Hkv, D)]))
    q = bf16_randn(gen, int(sum(q_lens)), num_heads, D)

    # lay the resident part of each sequence into the pool
    k_rows, v_rows, slots = [], [], []
    for s in range(B):
        L = seq_lens[s]
        resident = L - new_lens[s]
        start = shared_prefix_tokens if s > 0 else 0
        t = torch.arange(start, resident)
        if t.numel():
            blk = block_tables[s, (t // bs)].long()
            off = t % bs
            k_cache[blk, :, off, :] = k_seq[s][start:resident]
            v_cache[blk, :, off, :] = v_seq[s][start:resident]
        t_new = torch.arange(resident, L)
        if t_new.numel():
            slots.append(block_tables[s, (t_new // bs)].long() * bs + t_new % bs)
            k_rows.append(k_seq[s][resident:L])
            v_rows.append(v_seq[s][resident:L])
    if slots:
        slot_mapping = torch.cat(slots).to(torch.int64)
        k_new = torch.cat(k_rows).contiguous()
        v_new = torch.cat(v_rows).contiguous()
    else:
        slot_mapping = torch.zeros(0, dtype=torch.int64)
        k_new = torch.zeros((0, Hkv, D), dtype=torch.bfloat16)
        v_new = torch.zeros((0, Hkv, D), dtype=torch.bfloat16)

    cu = torch.zeros(B + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(list(q_lens), dtype=torch.int64), 0).to(torch.int32)
    return PagedCase(name=name, seed=seed, num_heads=num_heads, num_kv_heads=num_kv_heads,
                     head_dim=head_dim, block_size=bs, num_blocks=num_blocks,
                     scale=(1.0 / math.sqrt(head_dim)) if scale is None else float(scale),
                     k_cache=k_cache, v_cache=v_cache, block_tables=block_tables,
                     seq_lens=torch.tensor(list(seq_lens), dtype=torch.int32), q=q,
                     q_lens=list(q_lens), cu_q_lens=cu, k_new=k_new, v_new=v_new,
                     slot_mapping=slot_mapping, k_seq=k_seq, v_seq=v_seq, notes=notes)


# --------------------------------------------------------------------------------------
# The five workloads.  Seeds are 1000 + workload number.
# --------------------------------------------------------------------------------------

def tiny_decode(seed: int = 1001) -> PagedCase:
    """1 sequence, 4 q heads / 1 kv head, d=64, 37 tokens in 3 blocks of a 16-block pool, scale 1/8."""
    return paged_case(name="tiny_decode", seed=seed, seq_lens=[37], q_lens=[1], new_lens=[0],
                      num_heads=4, num_kv_heads=1, head_dim=64, num_blocks=16, scale=1.0 / 8)


def qwen3_4b_decode(seed: int = 1002) -> PagedCase:
    """Qwen3-4B-shaped single-layer decode: 32/8/128, batch 1, context 1152, 4096-block pool."""
    return paged_case(name="qwen3_4b_decode", seed=seed, seq_lens=[1152], q_lens=[1], new_lens=[0],
                      num_heads=32, num_kv_heads=8, head_dim=128, num_blocks=4096)


def batched_decode(seed: int = 1003, batch: int = 64) -> PagedCase:
    """64 sequences, context ~U[1024, 1152], 32/8/128, 16384-block pool; the newest token of
    every sequence arrives through one append of 64 rows."""
    gen = generator(seed)
    lens = torch.randint(1024, 1153, (batch,), generator=gen).tolist()
    return paged_case(name="batched_decode", seed=seed, seq_lens=lens, q_lens=[1] * batch,
                      new_lens=[1] * batch, num_heads=32, num_kv_heads=8, head_dim=128,
                      num_blocks=16384, gen=gen)


def spec_verify(seed: int = 1006, batch: int = 64, drafts: int = 4) -> PagedCase:
    """The batched-decode shape with `drafts` query tokens per sequence instead of one (a
    speculative-decoding verify: the last `drafts` tokens of each sequence are appended and
    attend causally), 32/8/128, context ~U[1024, 1152], 16384-block pool."""
    gen = generator(seed)
    lens = torch.randint(1024, 1153, (batch,), generator=gen).tolist()
    return paged_case(name="spec_verify", seed=seed, seq_lens=lens, q_lens=[drafts] * batch,
                      new_lens=[drafts] * batch, num_heads=32, num_kv_heads=8, head_dim=128,
                      num_blocks=16384, gen=gen)


def splitkv_decode(seed: int = 1004, batch: int = 4, context: int = 8192) -> PagedCase:
    """Qwen3-32B-shaped long-context decode, 64/8/128 (group 8), 4096-block pool."""
    return paged_case(name=f"splitkv_{batch}x{context}", seed=seed, seq_lens=[context] * batch,
                      q_lens=[1] * batch, new_lens=[0] * batch, num_heads=64, num_kv_heads=8,
                      head_dim=128, num_blocks=4096)


def chunked_prefill(seed: int = 1005, batch: int = 8, prefix_blocks: int = 48, chunk: int = 256) -> PagedCase:
    """8 sequences share 48 cached prefix blocks (768 tokens); each appends its own 256-token
    causal chunk through the slot mapping and attends over prefix + chunk.  32/8/128."""
    pre = prefix_blocks * BLOCK_SIZE
    return paged_case(name="chunked_prefill", seed=seed, seq_lens=[pre + chunk] * batch,
                      q_lens=[chunk] * batch, new_lens=[chunk] * batch, num_heads=32,
                      num_kv_heads=8, head_dim=128, num_blocks=4096, shared_prefix_tokens=pre)


WORKLOADS = {
    "tiny_decode": tiny_decode,
    "qwen3_4b_decode": qwen3_4b_decode,
    "batched_decode": batched_decode,
    "splitkv_4x8192": lambda seed=1004: splitkv_decode(seed, 4, 8192),
    "splitkv_1x32768": lambda seed=1004: splitkv_decode(seed, 1, 32768),
    "chunked_prefill": chunked_prefill,
}


def random_case(seed: int, *, batch: int, num_heads: int, num_kv_heads: int, head_dim: int,
                min_len: int = 1, max_len: int = 80, q_len: int = 1, num_blocks: Optional[int] = None,
                prefill: bool = False, shared_prefix_tokens: int = 0, append: bool = True,
                scale: Optional[float] = None, name: str = "random") -> PagedCase:
    """Small ragged problem for sweeps: lengths ~U[min_len, max_len]; prefill chunks ~U[1, q_len]."""
    gen = generator(seed)
    lens = torch.randint(min_len, max_len + 1, (batch,), generator=gen).tolist()
    lens = [max(L, shared_prefix_tokens + (1 if prefill else 0)) for L in lens]
    if prefill:
        qls = [int(torch.randint(1, min(q_len, L - shared_prefix_tokens) + 1, (1,), generator=gen))
               for L in lens]
    else:
        qls = [1] * batch
    news = [min(c, L - shared_prefix_tokens) for c, L in zip(qls, lens)] if append else [0] * batch
    need = shared_prefix_tokens // BLOCK_SIZE + sum(math.ceil((L - shared_prefix_tokens) / BLOCK_SIZE)
                                                     for L in lens)
    nblk = num_blocks if num_blocks is not None else max(need + 7, 2 * need)
    return paged_case(name=name, seed=seed, seq_lens=lens, q_lens=qls, new_lens=news,
                      num_heads=num_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                      num_blocks=nblk, shared_prefix_tokens=shared_prefix_tokens, scale=scale,
                      gen=gen)
