"""The host-side KV block manager (pa_bm_*): budget arithmetic, full-lifetime admission,
refcounted sharing through the prefix cache, eviction order, slot mapping, and a random
workload checked against a plain Python model of the same rules (no GPU needed)."""
import random

import numpy as np
import pytest

import paged_kv_gqa_slot_gb300 as pa
from paged_kv_gqa_slot_gb300 import build as pbuild


@pytest.fixture(scope="module", autouse=True)
def lib():
    pbuild.build()
    return pa.library()


def test_budget_arithmetic_qwen3_32b():
    # 64 layers x (K, V) x 8 kv heads x 16 tokens x 128 x 2 B = 4 MiB per block
    assert pa.pa_kv_block_bytes(64, 8, 128) == 4 * 2 ** 20
    # 5360 blocks (the "Qwen3-32B Serving Load" figure) are 22.48 GB = 20.94 GiB
    assert pa.pa_kv_budget_blocks(5360 * 4 * 2 ** 20, 64, 8, 128) == 5360
    assert pa.pa_kv_budget_blocks(5360 * 4 * 2 ** 20 - 1, 64, 8, 128) == 5359
    # the quoted "21.4 GB" brackets it under either unit reading (the residual is not on the pages)
    assert pa.pa_kv_budget_blocks(int(21.4e9), 64, 8, 128) == 5102
    assert pa.pa_kv_budget_blocks(int(21.4 * 2 ** 30), 64, 8, 128) == 5478
    assert pa.pa_kv_block_bytes(0, 8, 128) == 0 and pa.pa_kv_budget_blocks(10 ** 9, 64, 0, 128) == 0


def test_budget_hybrid_stack():
    """The hybrid line pages only its full-attention layers, one in four ("Qwen3.5 Dense",
    Notes: the 8 full-attention layers of a 32-layer stack keep a paged KV cache; the other
    24 carry a fixed-size state), so a 16-token block spans a quarter of the layers and a
    budget holds four times as many blocks.  The attention layers' head counts are not on the
    pages; 8 kv heads of 128 (the Qwen3 line's) stand in, and the ratio does not depend on
    them."""
    full, hybrid = pa.pa_kv_block_bytes(32, 8, 128), pa.pa_kv_block_bytes(8, 8, 128)
    assert full == 4 * hybrid == 2 * 2 ** 20
    budget = 1000 * full
    assert pa.pa_kv_budget_blocks(budget, 32, 8, 128) == 1000
    assert pa.pa_kv_budget_blocks(budget, 8, 8, 128) == 4000
    # The recurrent state is reserved ahead of the KV pool (two ~147 MB states for each of
    # the default 64 decode slots at 27B: the 18.8 GB the pages quote); the pool is sized
    # from what is left.
    reserve = 64 * 2 * 147 * 10 ** 6
    assert round(reserve / 1e8) == 188
    assert pa.pa_kv_budget_blocks(budget + reserve, 8, 8, 128) - pa.pa_kv_budget_blocks(budget, 8, 8, 128) == \
        reserve // hybrid


def test_full_lifetime_admission():
    bm = pa.BlockManager(10, prefix_cache=False)
    t1, c1 = bm.admit(1, range(50), 30)          # 80 tokens -> 5 blocks
    assert len(t1) == 5 and c1 == 0 and sorted(t1) == list(range(5))
    t2, _ = bm.admit(2, range(60), 20)           # 5 more: the pool is full
    assert bm.stats() == (0, 0, 10)
    assert bm.admit(3, range(1), 0) is None      # even one token is rejected, nothing changes
    assert bm.stats() == (0, 0, 10)
    bm.release(1)
    assert bm.stats() == (5, 0, 5)
    assert bm.admit(4, range(70), 11) is None    # 81 tokens -> 6 blocks > 5 free
    t4, _ = bm.admit(4, range(70), 10)           # 80 tokens -> 5 blocks
    assert set(t4) == set(t1) and not set(t4) & set(t2)
    assert bm.admit(5, range(10 * 16 + 1), 0) is None   # larger than the whole pool


def test_prefix_sharing_and_refcounts():
    bm = pa.BlockManager(16)
    prompt = list(range(100, 150))               # 50 tokens: 3 full blocks
    ta, ca = bm.admit(1, prompt, 14)             # 64 tokens -> 4 blocks
    assert ca == 0
    bm.commit(1, [], 50)                          # prefill done: blocks 0..2 enter the cache
    # a second live request with the same prompt prefix shares the 3 full blocks
    tb, cb = bm.admit(2, prompt[:48] + [7, 8, 9], 5)
    assert cb == 48 and list(tb[:3]) == list(ta[:3]) and tb[3] not in ta
    free, idle, used = bm.stats()
    assert used == 5 and idle == 0 and free == 11
    bm.release(1)                                 # the shared blocks still have a user
    assert bm.stats() == (12, 0, 4)
    bm.release(2)                                 # now cached and idle
    assert bm.stats() == (13, 3, 0)
    # the whole prompt cached: the last token is still left to compute
    bm2 = pa.BlockManager(8)
    bm2.admit(1, list(range(32)), 0)
    bm2.commit(1, [], 32)
    bm2.release(1)
    _, c = bm2.admit(2, list(range(32)), 0)
    assert c == 16


def test_chained_hash_needs_the_same_prefix():
    bm = pa.BlockManager(16)
    a = [1] * 16 + list(range(16))
    bm.admit(1, a + [0], 0)
    bm.commit(1, [], 33)
    bm.release(1)
    b = [2] * 16 + list(range(16))               # same second block, different first block
    _, c = bm.admit(2, b + [0], 0)
    assert c == 0
    _, c = bm.admit(3, a + [5], 0)                # the original prefix hits both blocks
    assert c == 32


def test_generated_tokens_are_cached_and_eviction_order():
    bm = pa.BlockManager(6)
    t, _ = bm.admit(1, list(range(10)), 30)       # 40 tokens -> 3 blocks
    gen = list(range(1000, 1022))
    bm.commit(1, [], 10)
    bm.commit(1, gen, 32)                         # 32 tokens have K/V: blocks 0, 1 full
    bm.release(1)
    assert bm.stats() == (4, 2, 0)
    seq = list(range(10)) + gen[:22] + [5]
    _, c = bm.admit(2, seq, 0)                    # a follow-up turn hits both blocks
    assert c == 32
    bm.release(2)
    # uncached allocations take free blocks first, then the block released longest ago: the
    # prefix's later block goes before its first one
    bm.admit(3, list(range(500, 500 + 64)), 0)    # 4 free blocks
    assert bm.stats() == (0, 2, 4)
    bm.admit(4, [9], 0)                           # evicts one cached block
    bm.release(3)
    _, c = bm.admit(5, seq, 0)
    assert c == 16                                # block 0 survived, block 1 was evicted


def test_partial_block_hit_copy_on_write():
    """A cached prefix that ends inside a block ("Warm Prefix-Cache TTFT": a warm request
    computes only what its cached prefix does not cover): the leading rows of the cached block
    that follows the same prefix are copied into the request's own block, never written in
    place, and the source block is held until the request is released."""
    rng = np.random.default_rng(7)
    a = rng.integers(0, 5000, 800).tolist()
    bm = pa.BlockManager(100)
    ta, ca, sa, da = bm.admit_cow(1, a, 0)
    assert ca == 0 and len(sa) == 0 and len(ta) == 50
    bm.commit(1, [], 800)                         # 50 full blocks enter the cache
    bm.release(1)
    assert bm.stats() == (50, 50, 0)
    b = a[:770] + rng.integers(5000, 9000, 254).tolist()
    tb, cb, src, dst = bm.admit_cow(2, b, 0)
    assert cb == 770 and list(tb[:48]) == list(ta[:48]) and tb[48] not in ta
    assert list(src) == [ta[48] * 16, ta[48] * 16 + 1] and list(dst) == [tb[48] * 16, tb[48] * 16 + 1]
    # 48 shared + the pinned source (held, idle no more) + 16 own blocks
    assert bm.stats() == (50 - 16, 50 - 49, 48 + 1 + 16)
    # the plain admission of the same prompt shares whole blocks only
    tc, cc = bm.admit(3, b, 0)
    assert cc == 768 and list(tc[:48]) == list(ta[:48])
    bm.release(3)
    bm.release(2)                                 # the pinned source goes back to the idle cache
    free, idle, used = bm.stats()
    assert used == 0 and idle >= 50
    # a divergence at the first token of the block: no partial hit
    c = a[:768] + [9999] + a[769:790]
    _, cc, src, _ = bm.admit_cow(4, c, 0)
    assert cc == 768 and len(src) == 0
    bm.release(4)
    # the prompt's last token is always left to compute: 790 tokens match 49 full blocks
    # (784 tokens) and at most 5 more rows
    _, cc, src, _ = bm.admit_cow(5, a[:790], 0)
    assert cc == 789 and len(src) == 5
    bm.release(5)
    # the longest matching child wins among several blocks after the same prefix
    d = a[:784] + a[784:787] + [4242] * 13
    bm.admit(6, d, 0)
    bm.commit(6, [], 800)
    bm.release(6)
    _, cc, src, _ = bm.admit_cow(7, a[:784] + a[784:794] + [1], 0)
    assert cc == 794 and list(src) == [int(ta[49]) * 16 + k for k in range(10)]


def test_partial_block_hit_admission_counts_the_pinned_block():
    """Full-lifetime admission counts the held source block: a request that would fit only by
    evicting that very block is rejected and nothing changes."""
    a = list(range(1000, 1040))                   # 40 tokens, 3 blocks: blocks 0 and 1 full and cached
    bm = pa.BlockManager(4)
    bm.admit_cow(1, a, 0)
    bm.commit(1, [], 40)
    bm.release(1)
    assert bm.stats() == (2, 2, 0)
    # 20 matching tokens + 40 more: block 0 shared, 4 rows of block 1 copied (it is held), 3 new
    # blocks needed but only 2 left without evicting the held block: rejected, nothing changes
    assert bm.admit_cow(2, a[:20] + list(range(5000, 5040)), 0) is None
    assert bm.stats() == (2, 2, 0)
    t, cc, src, dst = bm.admit_cow(3, a[:20] + list(range(5000, 5020)), 0)   # 40 tokens: 3 blocks
    assert cc == 20 and len(src) == 4 and list(t[:1]) == [0]
    assert bm.stats() == (0, 0, 4)
    bm.release(3)
    assert bm.stats()[2] == 0


def test_slots_and_errors():
    bm = pa.BlockManager(8)
    t, _ = bm.admit(7, list(range(20)), 12)       # 32 tokens -> 2 blocks
    s = bm.slots(7, 0, 32)
    assert list(s) == [int(t[p // 16]) * 16 + p % 16 for p in range(32)]
    with pytest.raises(pa.PagedAttnError):
        bm.slots(7, 20, 13)                       # beyond the reservation
    with pytest.raises(pa.PagedAttnError):
        bm.admit(7, [1], 0)                       # id already admitted
    with pytest.raises(pa.PagedAttnError):
        bm.commit(8, [], 0)                       # unknown id
    with pytest.raises(pa.PagedAttnError):
        bm.commit(7, list(range(13)), 20)         # more tokens than reserved
    with pytest.raises(pa.PagedAttnError):
        bm.commit(7, [], 21)                      # more computed than known tokens
    with pytest.raises(pa.PagedAttnError):
        bm.release(9)
    assert pa.library().pa_bm_create(0, 16, 1) is None


class Model:
    """The manager's rules restated plainly: blocks, refcounts, a cache of full blocks keyed
    by their whole token prefix, evictable blocks in release order."""

    def __init__(self, n, bs=16):
        self.bs, self.n = bs, n
        self.refs = [0] * n
        self.key = {}                  # block id -> prefix tuple (cached blocks)
        self.by_key = {}               # prefix tuple -> block id
        self.free = list(range(n - 1, -1, -1))
        self.idle = []                 # evictable, oldest first
        self.req = {}

    def admit(self, rid, toks, max_new):
        bs = self.bs
        total = -(-(len(toks) + max_new) // bs)
        hits = []
        i = 0
        while (i + 1) * bs <= len(toks) - 1:
            k = tuple(toks[:(i + 1) * bs])
            if k not in self.by_key:
                break
            hits.append(self.by_key[k])
            i += 1
        idle_hits = sum(1 for b in hits if self.refs[b] == 0)
        if total > self.n or total - len(hits) > len(self.free) + len(self.idle) - idle_hits:
            return None
        table = []
        for b in hits:
            if self.refs[b] == 0:
                self.idle.remove(b)
            self.refs[b] += 1
            table.append(b)
        for _ in range(total - len(hits)):
            if self.free:
                b = self.free.pop()
            else:
                b = self.idle.pop(0)
                del self.by_key[self.key.pop(b)]
            self.refs[b] = 1
            table.append(b)
        self.req[rid] = {"toks": list(toks), "table": table, "reg": len(hits)}
        return table, len(hits) * bs

    def commit(self, rid, new, computed):
        r = self.req[rid]
        r["toks"] += list(new)
        full = min(computed, len(r["toks"])) // self.bs
        for i in range(r["reg"], full):
            b = r["table"][i]
            k = tuple(r["toks"][:(i + 1) * self.bs])
            if b not in self.key and k not in self.by_key:
                self.key[b] = k
                self.by_key[k] = b
            r["reg"] = i + 1

    def release(self, rid):
        for b in reversed(self.req.pop(rid)["table"]):
            self.refs[b] -= 1
            if self.refs[b] == 0:
                (self.idle if b in self.key else self.free).append(b)

    def stats(self):
        return len(self.free), len(self.idle), self.n - len(self.free) - len(self.idle)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_random_workload_matches_model(seed):
    rng = random.Random(seed)
    n = 48
    bm, model = pa.BlockManager(n), Model(n)
    prompts = [[rng.randrange(4) for _ in range(rng.randrange(1, 90))] for _ in range(6)]
    live, rid = {}, 0
    for step in range(600):
        op = rng.random()
        if op < 0.45 or not live:
            base = rng.choice(prompts)
            toks = base[:rng.randrange(1, len(base) + 1)] + [rng.randrange(4) for _ in range(rng.randrange(0, 20))]
            max_new = rng.randrange(0, 40)
            got, want = bm.admit(rid, toks, max_new), model.admit(rid, toks, max_new)
            assert (got is None) == (want is None), f"step {step}: admission differs"
            if got is not None:
                assert list(got[0]) == want[0] and got[1] == want[1], f"step {step}"
                live[rid] = (len(toks), max_new)
            rid += 1
        elif op < 0.75:
            r = rng.choice(list(live))
            n_tok, max_new = live[r]
            gen = [rng.randrange(4) for _ in range(rng.randrange(0, max_new + 1))]
            live[r] = (n_tok + len(gen), max_new - len(gen))
            computed = rng.randrange(0, n_tok + len(gen) + 1)
            bm.commit(r, gen, computed)
            model.commit(r, gen, computed)
        else:
            r = rng.choice(list(live))
            del live[r]
            bm.release(r)
            model.release(r)
        assert bm.stats() == model.stats(), f"step {step}"
        # no block is held by two live requests unless it is a shared cached block
        owners = {}
        for r in live:
            for b in model.req[r]["table"]:
                owners.setdefault(b, []).append(r)
        for b, rs in owners.items():
            assert len(rs) == 1 or b in model.key
