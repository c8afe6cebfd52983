// pa_blockmgr.cpp -- host-side manager of the paged KV pool: a refcounted block allocator,
// a prefix cache of full blocks, and full-lifetime admission against the pool's budget.
//
// Method: "Qwen3-4B / 8B / 32B", sections "Architecture Notes" (a paged KV cache with
// full-lifetime admission: a request that cannot fit is rejected instead of hanging under
// memory pressure; prefix cache on by default), "Qwen3-32B Serving Load" (a profiled KV
// budget of 21.4 GB = 5360 blocks next to the weights) and "Warm Prefix-Cache TTFT" (a warm
// request reuses the cached K/V of its prompt prefix and computes only the rest).
//
// Blocks hold 16 tokens of every layer's K and V.  A full block is identified by a chained
// hash of its tokens and of every token before it (FNV-1a over the parent block's hash and
// the block's token ids), so equal token runs after different prefixes never match; a match
// also compares the stored token ids, so a hash collision cannot return wrong K/V.  A block
// whose last user has released it stays cached (reusable by a later request with the same
// prefix) in least-recently-released order until the allocator needs it back.
//
// A prompt whose cached prefix ends inside a block (pa_bm_admit_cow) also reuses the leading
// tokens of that block: among the cached blocks that follow the same prefix (same parent
// hash), the one whose first tokens match the prompt longest gives its first k rows, which
// are copied into the request's own block (copy on write: a cached block is never written),
// so only the tokens after them are computed.  The source block is pinned (one reference) for
// the request's lifetime, so no other request can take it and overwrite it before the copy.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <iterator>
#include <list>
#include <mutex>
#include <new>
#include <unordered_map>
#include <vector>

#include "pagedattn.h"

namespace {

constexpr uint64_t kFnvOffset = 14695981039346656037ull;
constexpr uint64_t kFnvPrime = 1099511628211ull;

uint64_t fnv_bytes(uint64_t h, const void* p, size_t n) {
    const unsigned char* b = static_cast<const unsigned char*>(p);
    for (size_t i = 0; i < n; ++i) {
        h ^= b[i];
        h *= kFnvPrime;
    }
    return h;
}

struct Block {
    int32_t refs = 0;
    bool cached = false;                 // registered in the prefix cache
    uint64_t hash = 0;
    uint64_t parent = 0;                 // hash of the block before it (0 for a first block), when cached
    std::vector<int32_t> tokens;         // the block's token ids, when cached
    std::list<int32_t>::iterator lru;    // position in the evictable list (refs == 0 && cached)
};

struct Request {
    std::vector<int32_t> tokens;         // prompt, then generated tokens
    std::vector<int32_t> blocks;         // block table: the whole lifetime, reserved at admission
    int32_t registered = 0;              // leading blocks already in the prefix cache (or matched)
    int32_t capacity = 0;                // tokens the reservation covers
    int32_t pinned = -1;                 // copy-on-write source block held for the request, or -1
};

}  // namespace

struct pa_blockmgr {
    int32_t block_size;
    bool prefix_cache;
    std::vector<Block> blocks;
    std::vector<int32_t> free_list;      // never used or released uncached; popped from the back
    std::list<int32_t> evictable;        // cached with no user; front = released longest ago
    std::unordered_multimap<uint64_t, int32_t> by_hash;
    std::unordered_multimap<uint64_t, int32_t> by_parent;  // cached blocks by their parent's hash
    std::unordered_map<int64_t, Request> requests;
    std::mutex mu;

    uint64_t chain(uint64_t parent, const int32_t* toks) const {
        uint64_t h = fnv_bytes(kFnvOffset, &parent, sizeof parent);
        return fnv_bytes(h, toks, sizeof(int32_t) * block_size);
    }

    int32_t lookup(uint64_t h, const int32_t* toks) const {
        auto range = by_hash.equal_range(h);
        for (auto it = range.first; it != range.second; ++it) {
            const Block& b = blocks[it->second];
            if (std::memcmp(b.tokens.data(), toks, sizeof(int32_t) * block_size) == 0) return it->second;
        }
        return -1;
    }

    // The cached block after `parent` whose leading tokens match toks[0, n) longest: (id, k),
    // or (-1, 0) when none matches even its first token.
    std::pair<int32_t, int32_t> longest_child(uint64_t parent, const int32_t* toks, int32_t n) const {
        std::pair<int32_t, int32_t> best(-1, 0);
        auto range = by_parent.equal_range(parent);
        for (auto it = range.first; it != range.second; ++it) {
            const Block& b = blocks[it->second];
            int32_t k = 0;
            while (k < n && k < block_size && b.tokens[k] == toks[k]) ++k;
            if (k > best.second || (k == best.second && k > 0 && it->second < best.first)) best = {it->second, k};
        }
        return best;
    }

    static void erase_pair(std::unordered_multimap<uint64_t, int32_t>& m, uint64_t key, int32_t id) {
        auto range = m.equal_range(key);
        for (auto it = range.first; it != range.second; ++it)
            if (it->second == id) {
                m.erase(it);
                return;
            }
    }

    void uncache(int32_t id) {
        Block& b = blocks[id];
        erase_pair(by_hash, b.hash, id);
        erase_pair(by_parent, b.parent, id);
        b.cached = false;
        b.tokens.clear();
    }

    // one block for a new owner: a never-used or uncached block first, else the cached block
    // released longest ago (its prefix-cache entry goes)
    int32_t take() {
        if (!free_list.empty()) {
            const int32_t id = free_list.back();
            free_list.pop_back();
            return id;
        }
        const int32_t id = evictable.front();
        evictable.pop_front();
        uncache(id);
        return id;
    }

    void drop_ref(int32_t id) {
        Block& b = blocks[id];
        if (--b.refs > 0) return;
        if (b.cached) {
            evictable.push_back(id);
            b.lru = std::prev(evictable.end());
        } else {
            free_list.push_back(id);
        }
    }

    void register_full_blocks(Request& r, int32_t computed) {
        if (!prefix_cache) return;
        const int32_t full = std::min<int32_t>(computed, (int32_t)r.tokens.size()) / block_size;
        for (int32_t i = r.registered; i < full; ++i) {
            const int32_t id = r.blocks[i];
            const uint64_t parent = i == 0 ? 0 : blocks[r.blocks[i - 1]].hash;
            const int32_t* toks = r.tokens.data() + (size_t)i * block_size;
            const uint64_t h = chain(parent, toks);
            Block& b = blocks[id];
            if (!b.cached) {
                if (lookup(h, toks) < 0) {  // another request may already hold this content
                    b.cached = true;
                    b.hash = h;
                    b.parent = parent;
                    b.tokens.assign(toks, toks + block_size);
                    by_hash.emplace(h, id);
                    by_parent.emplace(parent, id);
                } else {
                    b.hash = h;  // the chain continues through an uncached duplicate
                }
            }
            r.registered = i + 1;
        }
    }
};

extern "C" {

int64_t pa_kv_block_bytes(int32_t num_layers, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                          int32_t dtype_bytes) {
    if (num_layers <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || dtype_bytes <= 0) return 0;
    return (int64_t)num_layers * 2 * num_kv_heads * block_size * head_dim * dtype_bytes;
}

int32_t pa_kv_budget_blocks(int64_t budget_bytes, int32_t num_layers, int32_t num_kv_heads, int32_t head_dim,
                            int32_t block_size, int32_t dtype_bytes) {
    const int64_t per = pa_kv_block_bytes(num_layers, num_kv_heads, head_dim, block_size, dtype_bytes);
    if (per <= 0 || budget_bytes < 0) return 0;
    const int64_t n = budget_bytes / per;
    return n > INT32_MAX ? INT32_MAX : (int32_t)n;
}

pa_blockmgr* pa_bm_create(int32_t num_blocks, int32_t block_size, int32_t enable_prefix_cache) {
    if (num_blocks <= 0 || block_size <= 0) return nullptr;
    pa_blockmgr* m = new (std::nothrow) pa_blockmgr();
    if (!m) return nullptr;
    m->block_size = block_size;
    m->prefix_cache = enable_prefix_cache != 0;
    m->blocks.resize(num_blocks);
    m->free_list.reserve(num_blocks);
    for (int32_t i = num_blocks - 1; i >= 0; --i) m->free_list.push_back(i);  // hand out 0, 1, 2, ... first
    return m;
}

void pa_bm_destroy(pa_blockmgr* m) { delete m; }

}  // extern "C"

namespace {

// Admission shared by pa_bm_admit and pa_bm_admit_cow (cow: also reuse the leading rows of a
// partly matching cached block; copy_src / copy_dst receive the slot pairs to copy).
int admit(pa_blockmgr* m, int64_t request_id, const int32_t* tokens, int32_t n_tokens, int32_t max_new_tokens,
          int32_t* block_table, int32_t table_cap, int32_t* n_blocks, int32_t* n_cached_tokens, bool cow,
          int64_t* copy_src, int64_t* copy_dst, int32_t* n_copy) {
    if (!m || n_tokens <= 0 || max_new_tokens < 0 || !tokens || !n_blocks || !n_cached_tokens) return PA_ERR_INVALID_ARG;
    if (cow && (!copy_src || !copy_dst || !n_copy)) return PA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(m->mu);
    if (m->requests.count(request_id)) return PA_ERR_INVALID_ARG;
    const int32_t bs = m->block_size;
    const int64_t lifetime = (int64_t)n_tokens + max_new_tokens;
    const int64_t need_total = (lifetime + bs - 1) / bs;
    if (need_total > (int64_t)m->blocks.size()) return PA_ERR_REJECTED;
    if (need_total > table_cap || (need_total > 0 && !block_table)) return PA_ERR_INVALID_ARG;
    // prefix hits: full blocks of the prompt, leaving at least its last token to compute
    std::vector<int32_t> hits;
    uint64_t parent = 0;
    if (m->prefix_cache) {
        for (int32_t i = 0; (int64_t)(i + 1) * bs <= n_tokens - 1; ++i) {
            const int32_t* toks = tokens + (size_t)i * bs;
            const uint64_t h = m->chain(parent, toks);
            const int32_t id = m->lookup(h, toks);
            if (id < 0) break;
            hits.push_back(id);
            parent = h;
        }
    }
    // a partial hit: the leading rows of a cached block that follows the same prefix
    int32_t src = -1, rows = 0;
    if (cow && m->prefix_cache) {
        const int32_t start = (int32_t)hits.size() * bs;
        const int32_t room = std::min(bs - 1, n_tokens - 1 - start);  // the last prompt token is computed
        if (room > 0) {
            const auto best = m->longest_child(parent, tokens + start, room);
            src = best.first;
            rows = best.second;
            if (rows == 0) src = -1;
        }
    }
    // full-lifetime admission: every block the request can ever need, or nothing
    int64_t reusable_idle = 0;  // matched (or pinned) blocks that sit in the evictable list
    for (int32_t id : hits)
        if (m->blocks[id].refs == 0) ++reusable_idle;
    if (src >= 0 && m->blocks[src].refs == 0) ++reusable_idle;
    const int64_t need_new = need_total - (int64_t)hits.size();
    const int64_t available = (int64_t)m->free_list.size() + (int64_t)m->evictable.size() - reusable_idle;
    if (need_new > available) return PA_ERR_REJECTED;
    Request r;
    r.tokens.assign(tokens, tokens + n_tokens);
    r.capacity = (int32_t)lifetime;
    auto hold = [&](int32_t id) {
        Block& b = m->blocks[id];
        if (b.refs++ == 0) m->evictable.erase(b.lru);
    };
    for (int32_t id : hits) {
        hold(id);
        r.blocks.push_back(id);
    }
    r.registered = (int32_t)hits.size();
    if (src >= 0) {
        hold(src);  // pinned until release: nobody else can take it before the copy has run
        r.pinned = src;
    }
    for (int64_t i = 0; i < need_new; ++i) {
        const int32_t id = m->take();
        m->blocks[id].refs = 1;
        r.blocks.push_back(id);
    }
    for (size_t i = 0; i < r.blocks.size(); ++i) block_table[i] = r.blocks[i];
    *n_blocks = (int32_t)r.blocks.size();
    *n_cached_tokens = (int32_t)hits.size() * bs + rows;
    if (cow) {
        const int32_t dst = src >= 0 ? r.blocks[hits.size()] : -1;
        for (int32_t k = 0; k < rows; ++k) {
            copy_src[k] = (int64_t)src * bs + k;
            copy_dst[k] = (int64_t)dst * bs + k;
        }
        *n_copy = rows;
    }
    m->requests.emplace(request_id, std::move(r));
    return PA_OK;
}

}  // namespace

extern "C" {

int pa_bm_admit(pa_blockmgr* m, int64_t request_id, const int32_t* tokens, int32_t n_tokens, int32_t max_new_tokens,
                int32_t* block_table, int32_t table_cap, int32_t* n_blocks, int32_t* n_cached_tokens) {
    return admit(m, request_id, tokens, n_tokens, max_new_tokens, block_table, table_cap, n_blocks, n_cached_tokens,
                 false, nullptr, nullptr, nullptr);
}

int pa_bm_admit_cow(pa_blockmgr* m, int64_t request_id, const int32_t* tokens, int32_t n_tokens,
                    int32_t max_new_tokens, int32_t* block_table, int32_t table_cap, int32_t* n_blocks,
                    int32_t* n_cached_tokens, int64_t* copy_src, int64_t* copy_dst, int32_t* n_copy) {
    return admit(m, request_id, tokens, n_tokens, max_new_tokens, block_table, table_cap, n_blocks, n_cached_tokens,
                 true, copy_src, copy_dst, n_copy);
}

int pa_bm_commit(pa_blockmgr* m, int64_t request_id, const int32_t* new_tokens, int32_t n_new, int32_t computed) {
    if (!m || n_new < 0 || (n_new > 0 && !new_tokens)) return PA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(m->mu);
    auto it = m->requests.find(request_id);
    if (it == m->requests.end()) return PA_ERR_INVALID_ARG;
    Request& r = it->second;
    const int64_t len = (int64_t)r.tokens.size() + n_new;
    if (len > r.capacity || computed < 0 || computed > len) return PA_ERR_INVALID_ARG;
    r.tokens.insert(r.tokens.end(), new_tokens, new_tokens + n_new);
    m->register_full_blocks(r, computed);
    return PA_OK;
}

int pa_bm_release(pa_blockmgr* m, int64_t request_id) {
    if (!m) return PA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(m->mu);
    auto it = m->requests.find(request_id);
    if (it == m->requests.end()) return PA_ERR_INVALID_ARG;
    // later blocks first, so a long cached prefix is evicted from its end
    const std::vector<int32_t>& bl = it->second.blocks;
    for (auto b = bl.rbegin(); b != bl.rend(); ++b) m->drop_ref(*b);
    if (it->second.pinned >= 0) m->drop_ref(it->second.pinned);
    m->requests.erase(it);
    return PA_OK;
}

int pa_bm_slots(pa_blockmgr* m, int64_t request_id, int32_t start, int32_t n, int64_t* slots) {
    if (!m || start < 0 || n < 0 || (n > 0 && !slots)) return PA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(m->mu);
    auto it = m->requests.find(request_id);
    if (it == m->requests.end()) return PA_ERR_INVALID_ARG;
    const Request& r = it->second;
    if ((int64_t)start + n > r.capacity) return PA_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n; ++i) {
        const int32_t pos = start + i;
        slots[i] = (int64_t)r.blocks[pos / m->block_size] * m->block_size + pos % m->block_size;
    }
    return PA_OK;
}

int pa_bm_stats(pa_blockmgr* m, int32_t* free_blocks, int32_t* cached_idle_blocks, int32_t* used_blocks) {
    if (!m) return PA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(m->mu);
    if (free_blocks) *free_blocks = (int32_t)m->free_list.size();
    if (cached_idle_blocks) *cached_idle_blocks = (int32_t)m->evictable.size();
    if (used_blocks) *used_blocks = (int32_t)(m->blocks.size() - m->free_list.size() - m->evictable.size());
    return PA_OK;
}

}  // extern "C"
