/*
 * pagedattn.h -- C ABI of libpagedattn: grouped-query attention over a block-paged
 * KV cache, hand-written CUDA for GB300 (sm_103a).
 *
 * The operation.  The pages "Qwen3-4B / 8B / 32B" (section "Architecture Notes")
 * describe full attention with grouped-query attention -- Qwen3-4B: 32 query heads
 * over 8 KV heads, head dim 128; Qwen3-32B: 64 query heads, group 8 -- served from a
 * paged KV cache with prefix caching; section "Qwen3-32B Serving Load" gives a KV
 * budget of 21.4 GB = 5360 blocks for Qwen3-32B, which fixes 16-token blocks; section
 * "Warm Prefix-Cache TTFT" is the chunked prefill over a warm prefix.  For query head
 * h of a sequence, with g = num_heads / num_kv_heads and kv head h / g:
 *
 *     o = sum_{t in keys} softmax_t(scale * <q, K_t>) V_t
 *
 * K_t, V_t read at pool[block_tables[s][t / 16], h / g, t % 16, :].  Softmax in fp32
 * (online, base 2), bf16 inputs, bf16 output rounded to nearest even.  The probabilities
 * enter the P V product on the tensor cores as bf16 -- as two bf16 parts (about 16 bits)
 * wherever a few weights can dominate a row: always in pa_decode, pa_decode_splitkv and
 * pa_append_decode; in pa_prefill_chunked always at head_dim 64 or a group size that does
 * not divide 128, else in the query tiles holding a query that sees at most 128 keys, and
 * everywhere at |scale| sqrt(head_dim) > 2 -- with the softmax sum taken over exactly those
 * values; accumulation is fp32.
 *
 * Memory.  Every pointer argument is a DEVICE pointer of the current CUDA device
 * unless stated otherwise; the caller allocates and owns every buffer (the library
 * allocates no device memory).  Every call is asynchronous on `stream` (NULL = the
 * legacy default stream) and returns after the launch: the return code reports host
 * validation and launch errors only.  Problems the device finds (a block id or slot
 * outside the pool, a pipeline wait that timed out) set bits of a device status word
 * that pa_device_status() reads.  Calls are thread-safe.
 *
 * Layouts (all row-major, contiguous):
 *   pool K, V      [num_blocks, num_kv_heads, 16, head_dim]   bf16, 16-byte aligned
 *   slot           block_id * 16 + offset_in_block
 *   block_tables   [batch, max_blocks] int32; entries past ceil(seq_len / 16) never affect
 *                  a result (a decode may load up to 32 entries of a row, all within the row,
 *                  before it knows seq_len, and ignores those it does not need)
 *   seq_lens       [batch] int32, tokens in the sequence including any appended this step
 *   q, out         decode [batch, num_heads, head_dim]; prefill [sum of chunk lengths,
 *                  num_heads, head_dim]; bf16, 16-byte aligned
 *
 * Supported: block_size 16; head_dim 64 or 128; any group size for prefill, group
 * size <= 16 for decode; batch <= 65535.
 */
#ifndef PAGEDATTN_H
#define PAGEDATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same handle as cudaStream_t. */
typedef struct CUstream_st *pa_stream_t;

enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = -1,  /* host validation failed; nothing was launched */
    PA_ERR_UNSUPPORTED = -2,  /* block size, head dim or group size outside the compiled set */
    PA_ERR_CUDA = -3,         /* a CUDA runtime call or launch failed */
    PA_ERR_OUT_OF_RANGE = -4, /* pa_device_status: a block id / slot / length outside the pool was skipped */
    PA_ERR_TIMEOUT = -5,      /* pa_device_status: a pipeline wait ran out (a bug, never expected) */
    PA_ERR_TOO_LARGE = -6,    /* pa_decode_splitkv_noalloc: the request does not fit its static scratch */
    PA_ERR_REJECTED = -7      /* pa_bm_admit: the request's whole lifetime does not fit the pool */
};

/* Device status bits reported by pa_device_status. */
#define PA_DEV_OUT_OF_RANGE 1u
#define PA_DEV_TIMEOUT 2u

/* The paged KV pool: two device tensors [num_blocks, num_kv_heads, block_size, head_dim] bf16. */
typedef struct {
    void *k_cache;
    void *v_cache;
    int32_t num_blocks;
    int32_t block_size;   /* must be 16 */
    int32_t num_kv_heads;
    int32_t head_dim;     /* 64 or 128 */
} pa_pool;

/*
 * pa_kv_append -- write new K/V rows into their pool slots.
 * Defines: for t in [0, num_tokens) with slot_mapping[t] >= 0,
 *   k_cache[slot / 16, h, slot % 16, :] = k_new[t, h, :]  (and v likewise), every kv head h.
 * This is how a decode token or a prefill chunk enters the paged cache ("Qwen3-4B / 8B /
 * 32B", "Architecture Notes": paged KV cache; "Warm Prefix-Cache TTFT": only new tokens
 * are written on a prefix hit).  It must precede, on the same stream, the attention call
 * that reads those tokens.
 *   k_new, v_new   [num_tokens, num_kv_heads, head_dim] bf16, 16-byte aligned
 *   slot_mapping   [num_tokens] int64; < 0 skips the row; >= num_blocks*16 is skipped and
 *                  sets PA_DEV_OUT_OF_RANGE.  Duplicate slots are a caller error.
 * Bit-exact copy.  num_tokens == 0 is a no-op; a call that would move 2^31 or more
 * 16-byte chunks (num_tokens * 2 * num_kv_heads * head_dim / 8) is PA_ERR_INVALID_ARG.
 */
int pa_kv_append(const pa_pool *pool, const void *k_new, const void *v_new, const int64_t *slot_mapping,
                 int32_t num_tokens, pa_stream_t stream);

/*
 * pa_kv_copy -- copy whole pool rows (every kv head, K and V): for t in [0, n),
 *   k_cache[dst / 16, h, dst % 16, :] = k_cache[src / 16, h, src % 16, :]  (and v likewise)
 * with src = src_slots[t], dst = dst_slots[t].  This is the copy on write of a prefix-cache
 * hit that ends inside a cached block ("Qwen3-4B / 8B / 32B", "Warm Prefix-Cache TTFT": a
 * warm request reuses the cached K/V of its prompt prefix): pa_bm_admit_cow returns the slot
 * pairs, and the copy must precede, on the same stream, the append of the request's own
 * tokens and any attention call that reads them.
 *   src_slots, dst_slots  [n] int64 device arrays; a pair with a negative slot is skipped, one
 *                         past the pool is skipped and sets PA_DEV_OUT_OF_RANGE.  A dst slot
 *                         that is also some pair's src slot is a caller error.
 * Bit-exact copy.
 */
int pa_kv_copy(const pa_pool *pool, const int64_t *src_slots, const int64_t *dst_slots, int32_t n,
               pa_stream_t stream);

/*
 * pa_decode -- one query token per sequence attends to keys [0, seq_lens[b]).
 * ("Qwen3-4B / 8B / 32B", "Architecture Notes": GQA over a paged KV cache; the query is
 * the newest token, already appended.)
 *   q, out         [batch, num_heads, head_dim] bf16
 *   scale          softmax scale, normally 1/sqrt(head_dim)
 * seq_lens[b] == 0 gives a zero row.  seq_lens[b] outside [0, max_blocks*16] is clamped
 * and sets PA_DEV_OUT_OF_RANGE.  When batch * num_kv_heads is small the library splits
 * each sequence over a thread-block cluster and merges in on-chip memory (no workspace).
 */
int pa_decode(const pa_pool *pool, const void *q, const int32_t *block_tables, int32_t max_blocks,
              const int32_t *seq_lens, int32_t batch, int32_t num_heads, float scale, void *out,
              pa_stream_t stream);

/*
 * pa_append_decode -- pa_kv_append of one new row per sequence followed by pa_decode, in
 * one launch (a decode step's append and attention fused; the pages' engines write a
 * token's K/V and then attend over it in every full-attention layer).  Equivalent to
 *   pa_kv_append(pool, k_new, v_new, slot_mapping, batch); pa_decode(pool, q, ...);
 * on the same stream, given that slot_mapping[b] is the slot of token seq_lens[b] - 1 of
 * sequence b (block_tables[b][(seq_lens[b]-1)/16] * 16 + (seq_lens[b]-1) % 16), as an
 * append for that token must be.
 *   k_new, v_new   [batch, num_kv_heads, head_dim] bf16, 16-byte aligned: the new rows
 *   slot_mapping   [batch] int64; < 0 skips the write (the decode then reads whatever the
 *                  slot holds).  Any other slot than the one above is not written and sets
 *                  PA_DEV_OUT_OF_RANGE.
 * Other arguments, errors and results as pa_decode.
 */
int pa_append_decode(const pa_pool *pool, const void *k_new, const void *v_new, const int64_t *slot_mapping,
                     const void *q, const int32_t *block_tables, int32_t max_blocks, const int32_t *seq_lens,
                     int32_t batch, int32_t num_heads, float scale, void *out, pa_stream_t stream);

/*
 * Workspace of pa_decode_splitkv, in bytes: ws_o [batch, num_heads, P, head_dim] fp32
 * followed by ws_lse [batch, num_heads, P] fp32 (ws_lse may live anywhere 16-byte aligned;
 * this is their sum).  Host-only, no CUDA call.
 */
size_t pa_splitkv_workspace_bytes(int32_t batch, int32_t num_heads, int32_t head_dim, int32_t num_partitions);

/*
 * pa_decode_splitkv -- flash-decoding partitions of the decode above.  Partition p of P
 * covers logical blocks [p*ceil(nb/P), (p+1)*ceil(nb/P)) of the nb = ceil(seq_len/16)
 * blocks and writes its own normalised output O_p and natural-log log-sum-exp
 * lse_p = m_p + ln(l_p) of its scaled scores; an empty partition writes O_p = 0,
 * lse_p = -inf.  (Long-context decode: the pages' long prompts are 4097-16384 tokens,
 * "Warm Prefix-Cache TTFT" and the 4097/8192-token golden prompts.)
 *   num_partitions P in [1, 4096]
 *   ws_o           [batch, num_heads, P, head_dim] fp32, 16-byte aligned (scratch owned by caller)
 *   ws_lse         [batch, num_heads, P] fp32
 */
int pa_decode_splitkv(const pa_pool *pool, const void *q, const int32_t *block_tables, int32_t max_blocks,
                      const int32_t *seq_lens, int32_t batch, int32_t num_heads, float scale,
                      int32_t num_partitions, float *ws_o, float *ws_lse, pa_stream_t stream);

/*
 * pa_combine -- log-sum-exp merge of split-KV partitions:
 *   M = max_p lse_p;  w_p = exp(lse_p - M);  out = sum_p w_p O_p / sum_p w_p
 * (partitions with lse_p = -inf weigh 0; all empty gives a zero row).
 *   ws_o, ws_lse   as written by pa_decode_splitkv;  out [batch, num_heads, head_dim] bf16
 */
int pa_combine(const float *ws_o, const float *ws_lse, int32_t batch, int32_t num_heads, int32_t head_dim,
               int32_t num_partitions, void *out, pa_stream_t stream);

/*
 * pa_prefill_chunked -- a causal query chunk over a cached paged prefix plus itself.
 * Sequence b's chunk is q rows [cu_q_lens[b], cu_q_lens[b+1]) (C_b tokens); seq_lens[b]
 * counts the prefix AND the chunk (whose K/V pa_kv_append already wrote).  Chunk query i
 * sits at position seq_lens[b] - C_b + i and attends to keys 0 .. that position.
 * ("Qwen3-4B / 8B / 32B", "Warm Prefix-Cache TTFT": warm prefix hit, only the new chunk
 * is computed.)
 *   q, out         [cu_q_lens[batch], num_heads, head_dim] bf16
 *   cu_q_lens      [batch + 1] int32, non-decreasing, cu_q_lens[0] = 0
 *   max_chunk      an upper bound of max_b C_b (sizes the grid; rows beyond C_b are idle).  A
 *                  chunk longer than the grid covers is reported (PA_DEV_OUT_OF_RANGE in the
 *                  device status) and its rows past the grid are not written; the other
 *                  sequences' results are unaffected
 * A sequence with C_b > seq_lens[b] or seq_lens[b] > max_blocks*16 is skipped and sets
 * PA_DEV_OUT_OF_RANGE.
 */
int pa_prefill_chunked(const pa_pool *pool, const void *q, const int32_t *cu_q_lens, const int32_t *block_tables,
                       int32_t max_blocks, const int32_t *seq_lens, int32_t batch, int32_t num_heads,
                       int32_t max_chunk, float scale, void *out, pa_stream_t stream);

/*
 * pa_device_status -- synchronise `stream`, then read the device status word of the
 * current device into *flags (PA_DEV_* bits, 0 = clean), clearing it when `clear` != 0.
 * Returns PA_OK, PA_ERR_OUT_OF_RANGE or PA_ERR_TIMEOUT according to the bits (timeout
 * first), PA_ERR_INVALID_ARG for a NULL flags pointer, PA_ERR_CUDA on a CUDA error.
 */
int pa_device_status(uint32_t *flags, int32_t clear, pa_stream_t stream);

/*
 * pa_selftest_wait_timeout -- a check of the error path the device status describes: one
 * thread waits, through the same bounded-wait helper the kernels use, on an mbarrier that
 * nothing ever arrives on, gives up after `limit_cycles` SM cycles (1 .. 2^40) and sets
 * PA_DEV_TIMEOUT, so that pa_device_status afterwards returns PA_ERR_TIMEOUT.  Nothing faults
 * and the context stays usable.  Asynchronous on `stream`.  Returns PA_OK,
 * PA_ERR_INVALID_ARG for a limit outside the range, or PA_ERR_CUDA.
 */
int pa_selftest_wait_timeout(uint64_t limit_cycles, pa_stream_t stream);

/*
 * pa_decode_splitkv_noalloc -- split-KV decode and its log-sum-exp merge in one call that
 * allocates nothing and takes no workspace: out = pa_combine(pa_decode_splitkv(...)).
 * The pages have no counterpart of this call; it exists for callers that cannot allocate
 * device memory -- an engine whose memory is a fixed arena owned by someone else, a plugin
 * in a host framework that exposes no allocator, or a serving loop that must never call
 * cudaMalloc on its hot path (an allocation there can synchronise the whole device).
 *   Arguments as pa_decode_splitkv plus out [batch, num_heads, head_dim] bf16.
 *   The partition results live in one static device array of pa_noalloc_scratch_bytes()
 *   bytes (8 MiB) inside the library, held by every GPU that loads the library until the
 *   process exits.  A request whose workspace (pa_splitkv_workspace_bytes) exceeds it
 *   returns PA_ERR_TOO_LARGE before any launch.
 *   The first call on a device looks up the array's device address (one-time set-up on that
 *   device); make that first call before capturing any stream into a CUDA graph.  The address
 *   is kept for the life of the process: after cudaDeviceReset on a device, do not call this
 *   entry point on that device again (the library's module, and the array, may have moved).
 *   Every call uses the same array, so calls that may run at the same time on the GPU
 *   (different streams, or different host threads) race and must be serialised by the
 *   caller.  Nothing needs clearing between calls: each call overwrites every slot it reads.
 */
int pa_decode_splitkv_noalloc(const pa_pool *pool, const void *q, const int32_t *block_tables, int32_t max_blocks,
                              const int32_t *seq_lens, int32_t batch, int32_t num_heads, float scale,
                              int32_t num_partitions, void *out, pa_stream_t stream);

/* Size in bytes of the static scratch array of pa_decode_splitkv_noalloc. */
size_t pa_noalloc_scratch_bytes(void);

/* Number of cluster splits pa_decode uses for this shape on the current device. */
int pa_decode_num_splits(int32_t batch, int32_t num_kv_heads, int32_t max_blocks);

/*
 * Partition count suggested for pa_decode_splitkv on the current device (1..16): the
 * largest count, at most 16, whose CTAs (batch x num_kv_heads x count) fill no more than
 * four fifths of one wave of four per SM, keeping >= 8 blocks per partition (the library
 * runs each partition on a thread-block cluster of up to 4 CTAs when the partitions alone
 * leave the wave at least half empty).
 */
int pa_splitkv_num_partitions(int32_t batch, int32_t num_kv_heads, int32_t max_blocks);

/* ------------------------------------------------------------------------------------
 * Host-side KV block manager (no GPU involved).  "Qwen3-4B / 8B / 32B", "Architecture
 * Notes": the paged KV cache uses full-lifetime admission (a request that cannot fit is
 * rejected rather than left to hang under memory pressure) and a prefix cache, on by
 * default; "Qwen3-32B Serving Load": the KV budget is profiled at load (21.4 GB, 5360
 * blocks); "Warm Prefix-Cache TTFT": a warm request computes only what its cached prompt
 * prefix does not cover.
 *
 * Bytes of one block (K and V of every layer): num_layers * 2 * num_kv_heads * block_size
 * * head_dim * dtype_bytes.  Qwen3-32B (64 layers, 8 kv heads, d 128, bf16, 16-token blocks)
 * gives 4 MiB, so 5360 blocks are 22.48 GB (20.94 GiB).  0 on a non-positive argument.
 */
int64_t pa_kv_block_bytes(int32_t num_layers, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                          int32_t dtype_bytes);
/* Blocks a budget of budget_bytes holds (floor). */
int32_t pa_kv_budget_blocks(int64_t budget_bytes, int32_t num_layers, int32_t num_kv_heads, int32_t head_dim,
                            int32_t block_size, int32_t dtype_bytes);

/* Opaque manager of num_blocks pool blocks of block_size tokens; thread-safe.  NULL on a
 * bad argument or no memory.  Destroy with pa_bm_destroy. */
typedef struct pa_blockmgr pa_blockmgr;
pa_blockmgr *pa_bm_create(int32_t num_blocks, int32_t block_size, int32_t enable_prefix_cache);
void pa_bm_destroy(pa_blockmgr *bm);

/*
 * Admit request_id with its prompt tokens[0, n_tokens) and at most max_new_tokens tokens to
 * generate.  The blocks for its whole lifetime (n_tokens + max_new_tokens) are reserved now,
 * or nothing is and PA_ERR_REJECTED is returned.  With the prefix cache, the prompt's leading
 * full blocks whose token ids (and every token before them) match a cached block are shared
 * instead of reserved; at least the prompt's last token is always left to compute.
 *   block_table      out: the request's block ids, in token order (table_cap entries or more)
 *   n_blocks         out: ceil((n_tokens + max_new_tokens) / block_size)
 *   n_cached_tokens  out: prompt tokens whose K/V is already in the pool (a multiple of
 *                    block_size); compute tokens [n_cached_tokens, n_tokens) next.
 * PA_ERR_INVALID_ARG on a bad argument or a request id already admitted.
 */
int pa_bm_admit(pa_blockmgr *bm, int64_t request_id, const int32_t *tokens, int32_t n_tokens,
                int32_t max_new_tokens, int32_t *block_table, int32_t table_cap, int32_t *n_blocks,
                int32_t *n_cached_tokens);

/*
 * pa_bm_admit_cow -- pa_bm_admit that also reuses a prefix hit ending inside a block.  After
 * the prompt's matching full blocks, the cached block that follows the same prefix and whose
 * leading tokens match the prompt's next tokens longest (k of them, 1 <= k <= 15, leaving the
 * prompt's last token to compute) lends its first k rows: they are to be copied into the
 * request's own block at that position (its table entry n_cached_tokens / 16), a copy on
 * write, since a cached block is never written.
 *   copy_src, copy_dst  out: n_copy slot pairs (block_size - 1 entries of room) for pa_kv_copy,
 *                       which must run before the request's tokens [n_cached_tokens, ...) are
 *                       appended and attended; n_copy = 0 when there is no partial hit
 *   n_cached_tokens     out: tokens whose K/V is in the pool once that copy has run (any count)
 * The source block is held (one reference) until the request is released, so no other
 * request can take it before the copy.  Other arguments and results as pa_bm_admit.
 */
int pa_bm_admit_cow(pa_blockmgr *bm, int64_t request_id, const int32_t *tokens, int32_t n_tokens,
                    int32_t max_new_tokens, int32_t *block_table, int32_t table_cap, int32_t *n_blocks,
                    int32_t *n_cached_tokens, int64_t *copy_src, int64_t *copy_dst, int32_t *n_copy);

/*
 * Append n_new generated tokens to the request's token list (within its reserved lifetime)
 * and declare that the K/V of its first `computed` tokens is now in the pool.  Blocks that
 * are full within those tokens enter the prefix cache (one entry per distinct content).
 */
int pa_bm_commit(pa_blockmgr *bm, int64_t request_id, const int32_t *new_tokens, int32_t n_new, int32_t computed);

/* Release the request: its blocks lose a user; cached ones stay reusable until the allocator
 * needs them (the one released longest ago first), the rest are free at once. */
int pa_bm_release(pa_blockmgr *bm, int64_t request_id);

/* Pool slots of the request's tokens [start, start + n): the slot_mapping of pa_kv_append. */
int pa_bm_slots(pa_blockmgr *bm, int64_t request_id, int32_t start, int32_t n, int64_t *slots);

/* Free (never used or uncached), cached-but-idle, and in-use block counts (any may be NULL). */
int pa_bm_stats(pa_blockmgr *bm, int32_t *free_blocks, int32_t *cached_idle_blocks, int32_t *used_blocks);

/* Human-readable name of a status code (static string). */
const char *pa_status_str(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H */
