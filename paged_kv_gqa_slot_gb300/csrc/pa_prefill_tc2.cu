// pa_prefill_tc2.cu -- chunked prefill over a cached paged prefix on the 5th-generation
// tensor cores, with double-buffered scores and P kept in tensor memory.
//
// Method: "Qwen3-4B / 8B / 32B", sections "Warm Prefix-Cache TTFT" (a warm prefix hit:
// only the new chunk is computed, over the cached prefix) and "Architecture Notes" (GQA
// over a paged KV cache).  Chunk query i of sequence s sits at position L_s - C_s + i and
// attends causally to keys 0 .. L_s - C_s + i through the block table.
//
// Rows of a query tile are (query, head-of-the-group) pairs: row r = query r / g, head r % g,
// so one K/V tile serves all g heads; a tile holds 128 rows (128 / g queries).  One CTA holds
// ONE query tile, and two CTAs are resident on every SM (256 TMEM columns and 112 KB of shared
// memory each): the two run independently, so one's start-up and epilogue overlap the other's
// stages, and the hardware scheduler hands the next tile to whichever SM slot frees first.
// Tiles launch longest first (the last tile of every chunk, then the one before it, ...), so
// the short tiles fill in behind the long ones.  Per stage of 64 keys (four 16-token pool
// blocks, loaded by TMA with 128-byte swizzling):
//   S[128 x 64] = Q K^T       tcgen05.mma, M=128 N=64, Q (A) and K (B) from smem
//   softmax          one thread per row reads its S row from TMEM, masks causally (only in
//                    stages that cross the diagonal), keeps an online max / sum in base 2 and
//                    writes P (bf16, two keys per column) over the first 32 columns of S
//   O += P V         tcgen05.mma, M=128 N=128, P (A) from TMEM, V (B) from smem
// Tensor memory: two 64-column score buffers, stage j in buffer j % 2, and O at [128, 256).
// So S(j+1) is computed while the softmax works on stage j, and P V(j) only gates S(j+2),
// which reuses the buffer P(j) sits in: the tensor core runs one issuer's MMAs in order, and
// the MMA warp issues, per stage j, P V(j) then S(j+2).
// The running max is re-based lazily: a stage is first taken against the row's current base,
// and only a row's first visible stage, or a stage whose sum passes 2^16 in some row of the
// warp, takes the row maximum; O is then rescaled in TMEM for rows whose maximum grew by more
// than 2^8.  So every P <= 2^16, and both the maximum and the rescales are rare.
// Q tiles come in by TMA through a 3-D map of q (d, head, token) whose box is one tile; a tile
// cut short by the end of its chunk, one at a negative scale, or one past the rows the map
// covers is copied in row by row by its softmax threads instead.  O leaves the same way: a
// whole tile is staged in bf16 in the then free Q buffer -- the softmax warps the first column
// half of their rows, the four control warps (done with their roles) the second -- and stored
// by TMA through a map of out shaped like q's; the rows of a tile cut short are stored by
// their threads.
// Warp roles: 0-3 softmax (TMEM lanes 32w..32w+31), 4 MMA issue + TMEM owner, 5 TMA loads of
// K, 6 TMA loads of V, 7 only the epilogue.  Every CTA loads its own K/V; the CTAs of one (sequence, kv head) --
// and, with a shared prefix, of every sequence that shares it -- read the same pool blocks,
// the copies after the first from L2.
#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdlib>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kD = 128;
constexpr int kRows = 128;                      // MMA M: rows of the query tile
constexpr int kKeys = 64;                       // keys per stage (MMA N of S, K of P V)
constexpr int kKStages = 3, kVStages = 2;       // K and V ring slots (a third K slot measured 1% faster)
constexpr int kSoftmaxThreads = 128;
constexpr int kMmaWarp = kSoftmaxThreads / 32, kKLoadWarp = kMmaWarp + 1, kVLoadWarp = kMmaWarp + 2;
constexpr int kThreads = kSoftmaxThreads + 128;  // warp 7 helps only with the epilogue
constexpr int kCtasPerSm = 2;                   // resident CTAs an SM holds (tensor memory, shared memory)
constexpr int kTmemCols = 256;                  // half of an SM's tensor memory
constexpr uint32_t kTmemS = 0, kTmemO = 128;    // score buffers at 0 and 64, O at 128
constexpr int kQHalf = kRows * 128;             // [128 rows][64 columns] bf16 = 16 KB
constexpr int kQTile = 2 * kQHalf;              // the Q tile: two column halves
constexpr int kKVHalf = kKeys * 128;            // [64 keys][64 columns] bf16 = 8 KB
constexpr int kKVStage = 2 * kKVHalf;           // one K or V stage: two column halves
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kQTile;
constexpr int kOffV = kOffK + kKStages * kKVStage;
constexpr int kBarOff = kOffV + kVStages * kKVStage;
// The dynamic shared memory starts 1024-byte aligned (the swizzled tiles need it; the kernel
// checks), so no slack is added: two CTAs must fit an SM's 228 KB with 1 KB reserved each.
constexpr int kOffX = kBarOff + 256;           // [128] 1/l of every row, then the epilogue's path
constexpr int kSmemBytes = kOffX + 528;
constexpr float kRescaleThreshold = 8.f;        // log2 units: a re-base moves the base to the max
constexpr float kSpecSumLimit = 65536.f;        // a stage sum past this takes the maximum path
constexpr float kSplitScale = 2.f;              // |scale| sqrt(d) past this: P in two bf16 halves
constexpr int kFewKeys = 128;                   // a tile with a query that sees <= this: the same
constexpr float kLog2e = 1.44269504088896340736f;

struct Bars {
    uint64_t k_full[kKStages], k_empty[kKStages], v_full[kVStages], v_empty[kVStages];
    // scores and P of stage j use buffer j % 2 (the softmax may finish two stages before the
    // MMA warp waits for the first, so one barrier per buffer keeps their phases apart);
    // o_done completes after every P V, o_final after the last one
    uint64_t q_full, s_full[2], p_full[2], o_done, o_final;
    uint64_t drain;
    uint32_t tmem_base;
};
static_assert(sizeof(Bars) <= 256, "barrier block");
static_assert(kCtasPerSm * (kSmemBytes + 1024) <= 228 * 1024, "shared memory for two resident CTAs");
static_assert(kCtasPerSm * kTmemCols <= 512, "tensor memory for two resident CTAs");

struct Tc2Args {
    const __nv_bfloat16* q;
    const int32_t* block_tables;
    const int32_t* seq_lens;
    const int32_t* cu_q_lens;
    __nv_bfloat16* out;
    unsigned* status;
    int max_blocks, num_heads, num_kv_heads, num_blocks, group, batch;
    int tiles;         // tile ranks the grid holds per (sequence, kv head)
    int q_rows;        // tokens the q map covers (batch * max_chunk)
    float scale_log2;  // scale * log2(e), signed
};

// Keys a query tile needs: [0, kmax) with kmax the position of its last query + 1.
__device__ __forceinline__ int tile_key_count(int mt, int tpt, int C, int L) {
    const int tok0 = mt * tpt;
    if (mt < 0 || tok0 >= C) return 0;
    return L - C + tok0 + min(tpt, C - tok0);
}

// bar.red.and over the `count` threads of named barrier `id`: true iff every one has `pred`.
__device__ __forceinline__ bool named_sync_all(int id, int count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbarrier.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// Score c of a 64-key stage held in two 32-column loads.
__device__ __forceinline__ float score(const uint32_t (&s0)[32], const uint32_t (&s1)[32], int c) {
    return __uint_as_float(c < 32 ? s0[c] : s1[c - 32]);
}

// Maximum of the row's visible scores in one stage: keys c <= lim, or every key (kAll, a
// stage wholly below the diagonal, which is the common case and needs no mask).  Four
// independent chains of three-input max.
template <bool kAll>
__device__ __forceinline__ float stage_max(const uint32_t (&s0)[32], const uint32_t (&s1)[32], int lim) {
    float m[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
    for (int c = 0; c < kKeys; c += 2) {
        float a0 = score(s0, s1, c), a1 = score(s0, s1, c + 1);
        if (!kAll) {
            a0 = c > lim ? -INFINITY : a0;
            a1 = c + 1 > lim ? -INFINITY : a1;
        }
        m[(c >> 1) & 3] = fmax3(m[(c >> 1) & 3], a0, a1);
    }
    return fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3]));
}

// p = 2^(s scale log2(e) - base) for the stage's keys (0 for keys past lim unless kAll),
// rounded to bf16 two keys to a 32-bit word, the layout P V reads from tensor memory: one
// packed multiply-add per two keys, the special-function unit, bf16 packing.
template <bool kAll>
__device__ __forceinline__ void stage_exps(const uint32_t (&s0)[32], const uint32_t (&s1)[32], int lim, float sl,
                                           float nbase, uint32_t (&pw)[kKeys / 2]) {
#pragma unroll
    for (int c = 0; c < kKeys; c += 2) {
        float x0, x1;
        fma_x2(x0, x1, score(s0, s1, c), score(s0, s1, c + 1), sl, sl, nbase, nbase);
        if (!kAll) {
            x0 = c > lim ? -INFINITY : x0;  // 2^-inf = 0
            x1 = c + 1 > lim ? -INFINITY : x1;
        }
        pw[c / 2] = pack_bf16x2(fast_exp2(x0), fast_exp2(x1));
    }
}

// (a0, a1) += the two bf16 values of a packed word, each widened exactly: the mixed-precision
// add of sm_100 and later, in place of unpacking both halves into fp32 first.
__device__ __forceinline__ void add_bf16x2(float& a0, float& a1, uint32_t w) {
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "add.rn.f32.bf16 %0, lo, %0;\n\tadd.rn.f32.bf16 %1, hi, %1;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "r"(w));
}

// Prefetch one box of a 3-D tensor map into L2 (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap* map, int x, int y, int z) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z)
                 : "memory");
}

// P of a stage against base -nbase (stage_exps on the warp's path) and the sum of the rounded
// values, so that the weights P V uses sum to l.
__device__ __forceinline__ float stage_p(const uint32_t (&s0)[32], const uint32_t (&s1)[32], int lim, float sl,
                                         float nbase, bool unmasked, uint32_t (&pw)[kKeys / 2]) {
    if (unmasked)
        stage_exps<true>(s0, s1, lim, sl, nbase, pw);
    else
        stage_exps<false>(s0, s1, lim, sl, nbase, pw);
    float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int w = 0; w < kKeys / 2; w += 2) {
        add_bf16x2(ls[0], ls[1], pw[w]);
        add_bf16x2(ls[2], ls[3], pw[w + 1]);
    }
    return (ls[0] + ls[1]) + (ls[2] + ls[3]);
}

// The low halves of P for a large scale: p again (the same operations as stage_exps, so the same
// values), less its bf16 high half `pw`, rounded to bf16; written 8 words at a time to the
// 32 columns at `dst` (the second half of the stage's buffer, free once S is in registers).
// Returns the sum of the rounded low values.
template <bool kAll>
__device__ __forceinline__ float stage_lo(const uint32_t (&s0)[32], const uint32_t (&s1)[32], int lim, float sl,
                                          float nbase, const uint32_t (&pw)[kKeys / 2], uint32_t dst) {
    float ls[2] = {0.f, 0.f};
#pragma unroll
    for (int c0 = 0; c0 < kKeys; c0 += 16) {
        uint32_t lw[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int c = c0 + 2 * k;
            float x0, x1;
            fma_x2(x0, x1, score(s0, s1, c), score(s0, s1, c + 1), sl, sl, nbase, nbase);
            if (!kAll) {
                x0 = c > lim ? -INFINITY : x0;
                x1 = c + 1 > lim ? -INFINITY : x1;
            }
            const uint32_t h = pw[c / 2];
            lw[k] = pack_bf16x2(fast_exp2(x0) - bf16_lo(h), fast_exp2(x1) - bf16_hi(h));
            add_bf16x2(ls[0], ls[1], lw[k]);
        }
        tmem_st8_nowait(dst + c0 / 2, lw[0], lw[1], lw[2], lw[3], lw[4], lw[5], lw[6], lw[7]);
    }
    return ls[0] + ls[1];
}

// O (the row's 128 fp32 columns of tensor memory at `taddr`) *= f, in 8-column pieces.
__device__ __forceinline__ void scale_o(uint32_t taddr, float f) {
#pragma unroll 1
    for (int c = 0; c < kD; c += 8) {
        uint32_t o[8];
        tmem_ld8(taddr + c, o);
        tmem_st8_nowait(taddr + c, __float_as_uint(__uint_as_float(o[0]) * f), __float_as_uint(__uint_as_float(o[1]) * f),
                        __float_as_uint(__uint_as_float(o[2]) * f), __float_as_uint(__uint_as_float(o[3]) * f),
                        __float_as_uint(__uint_as_float(o[4]) * f), __float_as_uint(__uint_as_float(o[5]) * f),
                        __float_as_uint(__uint_as_float(o[6]) * f), __float_as_uint(__uint_as_float(o[7]) * f));
    }
    tmem_wait_st();
}

__device__ __noinline__ void tc2_tile_split(const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                            const CUtensorMap& tm_q, const CUtensorMap& tm_o, const Tc2Args& a);

// One CTA's query tile.  kSplit: P as bf16 high + low halves (two P V products).  The
// one-half form hands a tile with a query that sees at most kFewKeys keys (the first
// queries of a sequence) to the two-halves form.
template <bool kSplit>
__device__ __forceinline__ void tc2_tile(const CUtensorMap& tm_k, const CUtensorMap& tm_v, const CUtensorMap& tm_q,
                                         const CUtensorMap& tm_o, const Tc2Args& a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    Bars* bars = reinterpret_cast<Bars*>(smem + kBarOff);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // blockIdx.x = (rank * batch + b) * num_kv_heads + kvh, so the CTAs launch rank by rank:
    // rank 0 is every chunk's last (longest) tile, rank 1 the one before, ...
    const int kvh = (int)(blockIdx.x % (unsigned)a.num_kv_heads);
    const int rb = (int)(blockIdx.x / (unsigned)a.num_kv_heads);
    const int b = rb % a.batch, rank = rb / a.batch;
    pdl_wait();
    if (smem_u32(smem) & 1023u) {  // the swizzled layouts need the declared alignment
        if (threadIdx.x == 0) atomicOr(a.status, kDevOutOfRange);
        return;
    }
    const int g = a.group, tpt = kRows / g;
    const int q0 = a.cu_q_lens[b];
    const int C = a.cu_q_lens[b + 1] - q0;
    const int L = a.seq_lens[b];
    if (C < 0 || L < C || L > a.max_blocks * kBlockSize) {
        if (threadIdx.x == 0 && rank == 0 && kvh == 0) atomicOr(a.status, kDevOutOfRange);
        return;
    }
    const int T = (C + tpt - 1) / tpt;  // query tiles of this sequence
    // a chunk longer than max_chunk has more tiles than the grid: the grid covers its first
    // a.tiles tiles, and the rest is reported
    if (rank == 0 && kvh == 0 && threadIdx.x == 0 && T > a.tiles) atomicOr(a.status, kDevOutOfRange);
    const int covered = min(T, a.tiles);
    if (rank >= covered) return;  // the same for the whole CTA
    const int mt = covered - 1 - rank;
    const int nkeys = tile_key_count(mt, tpt, C, L);
    const int nst = (nkeys + kKeys - 1) / kKeys;               // key stages
    const int nblk = (nkeys + kBlockSize - 1) / kBlockSize;  // pool blocks read
    const int tok0 = mt * tpt;
    const int ntok = min(tpt, C - tok0);  // >= 1: the tile holds a query of the chunk
    if (!kSplit && L - C + tok0 + 1 <= kFewKeys) {
        tc2_tile_split(tm_k, tm_v, tm_q, tm_o, a);
        return;
    }
    // A negative scale enters as -Q (exact in bf16) against |scale|, so the row maximum is
    // always taken over the scores as they are; such Q is negated on the way in, by threads.
    const bool neg = a.scale_log2 < 0.f;
    // a whole tile inside the rows the q map covers (a chunk longer than max_chunk can put a
    // later sequence's tiles past them): Q by TMA at a positive scale
    const bool whole = ntok == tpt && q0 + tok0 + tpt <= a.q_rows;

    // The loads the first stage waits on start before the set-up below: the producers' first
    // block-table entries, and the Q tile and the tensor maps into L2 / the map cache.
    const int32_t* bt = a.block_tables + (size_t)b * a.max_blocks;
    int cur = 0, nxt = 0;
    if (warp == kKLoadWarp || warp == kVLoadWarp) {
        cur = lane < nblk ? __ldg(bt + lane) : 0;
        nxt = 32 + lane < nblk ? __ldg(bt + 32 + lane) : 0;
        if (lane == 0) prefetch_tensormap(warp == kKLoadWarp ? &tm_k : &tm_v);
    } else if (threadIdx.x == 32 && whole && !neg) {
        prefetch_tensormap(&tm_q);
        tma_prefetch_3d(&tm_q, 0, kvh * g, q0 + tok0);
        tma_prefetch_3d(&tm_q, 64, kvh * g, q0 + tok0);
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(&bars->k_full[s], 1);
            mbar_init(&bars->k_empty[s], 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(&bars->v_full[s], 1);
            mbar_init(&bars->v_empty[s], 1);
        }
        mbar_init(&bars->q_full, 1);
        mbar_init(&bars->s_full[0], 1);
        mbar_init(&bars->s_full[1], 1);
        mbar_init(&bars->p_full[0], 128);
        mbar_init(&bars->p_full[1], 128);
        mbar_init(&bars->o_done, 1);
        mbar_init(&bars->o_final, 1);
        mbar_init(&bars->drain, 1);
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&bars->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp >= kMmaWarp) {
        if (warp == kKLoadWarp || warp == kVLoadWarp) {
            // -------------------------------------------------------- TMA producers (K, V)
            // The 8 boxes of a stage (4 blocks x 2 column halves, 2 KB each) go out from lanes
            // 0-7, one each; a block past the keys the tile needs reads past the pool (zeros).
            const bool is_k = warp == kKLoadWarp;
            const CUtensorMap* map = is_k ? &tm_k : &tm_v;
            uint64_t* full = is_k ? bars->k_full : bars->v_full;
            uint64_t* empty = is_k ? bars->k_empty : bars->v_empty;
            uint8_t* ring = smem + (is_k ? kOffK : kOffV);
            const int nslots = is_k ? kKStages : kVStages;
            const uint64_t pol = l2_evict_last_policy();  // prefix blocks are shared across sequences
            const int oob_row = a.num_blocks * a.num_kv_heads * kBlockSize;
            int c0 = 0;
            const int box_t = lane >> 1, box_h = lane & 1;
            bool ok = true;
            int issued = 0;
            for (int j = 0; j < nst && ok; ++j) {
                if (4 * j >= c0 + 32) {
                    c0 += 32;
                    cur = nxt;
                    nxt = c0 + 32 + lane < nblk ? __ldg(bt + c0 + 32 + lane) : 0;
                }
                if (is_k && c0 + lane < nblk && (cur < 0 || cur >= a.num_blocks)) atomicOr(a.status, kDevOutOfRange);
                if (cur < 0 || cur >= a.num_blocks) cur = 0;
                const int lb = 4 * j + box_t;
                const int id = __shfl_sync(0xffffffffu, cur, (lb - c0) & 31);
                const int row = lb < nblk ? (id * a.num_kv_heads + kvh) * kBlockSize : oob_row;
                const int s = j % nslots;
                if (lane == 0) {
                    // the slot's previous stage, j - nslots, has been read
                    if (j >= nslots) ok = mbar_wait(&empty[s], ((j / nslots) & 1) ^ 1);
                    if (ok) mbar_arrive_expect_tx(&full[s], kKVStage);
                }
                ok = __shfl_sync(0xffffffffu, ok, 0) != 0;
                if (ok) {
                    if (lane < 8)
                        tma_load_2d(ring + s * kKVStage + box_h * kKVHalf + box_t * 2048, map, box_h * 64, row,
                                    &full[s], pol);
                    ++issued;
                }
            }
            if (lane == 0) {
                // before the CTA may leave: every box issued here has landed
                for (int j = max(0, issued - nslots); j < issued; ++j)
                    if (!mbar_wait(&full[j % nslots], (j / nslots) & 1)) ok = false;
                if (!ok) atomicOr(a.status, kDevTimeout);
            }
        } else if (warp == kMmaWarp) {
            // -------------------------------------------------------- MMA issue
            // The tile's chain -- P(j), then P V(j), then S(j+2) into the buffer P(j) held -- in
            // one warp; the other resident CTA's MMA warp keeps the tensor core busy while this
            // one waits (a waiting issuer leaves it idle: issue runs only a few MMAs ahead of
            // execution).  The warp runs the loop together and one elected lane issues, so
            // every operand is warp-uniform; waits give one verdict for the warp.  Operand
            // descriptors are built once; a stage or a k-step only moves the start address,
            // which adds (offset >> 4) to the low field (no carry: every shared address is
            // below 2^18).
            const int n = nst;
            constexpr uint32_t idesc_s = tc_idesc_bf16(kRows, kKeys, false);
            constexpr uint32_t idesc_o = tc_idesc_bf16(kRows, kD, true);
            const uint64_t qd = smem_desc_sw128(smem_u32(smem + kOffQ), 0, 1024);
            const uint64_t kdesc0 = smem_desc_sw128(smem_u32(smem + kOffK), 0, 1024);
            const uint64_t vdesc0 = smem_desc_sw128(smem_u32(smem + kOffV), kKVHalf, 1024);
            auto issue_qk = [&](int j) {  // S(j) = Q K(j)^T into score buffer j % 2
                const uint64_t kd = kdesc0 + (uint64_t)(((j % kKStages) * kKVStage) >> 4);
                const uint32_t tm_s = tmem + kTmemS + 64 * (j & 1);
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk)
                    tc_mma_ew(tm_s, qd + (uint64_t)(((kk >> 2) * kQHalf + (kk & 3) * 32) >> 4),
                              kd + (uint64_t)(((kk >> 2) * kKVHalf + (kk & 3) * 32) >> 4), idesc_s, kk > 0 ? 1u : 0u);
                tc_commit_ew(&bars->s_full[j & 1]);
                tc_commit_ew(&bars->k_empty[j % kKStages]);
            };
            auto issue_pv = [&](int j) {  // O += P(j) V(j), P(j) in score buffer j % 2
                const uint64_t vd = vdesc0 + (uint64_t)(((j % kVStages) * kKVStage) >> 4);
                const uint32_t tm_p = tmem + kTmemS + 64 * (j & 1);
#pragma unroll
                for (int kk = 0; kk < kKeys / 16; ++kk)
                    tc_mma_ts_ew(tmem + kTmemO, tm_p + kk * 8, vd + (uint64_t)((kk * 16 * 128) >> 4), idesc_o,
                                 (j > 0 || kk > 0) ? 1u : 0u);
                if (kSplit) {  // the low halves of P, against the same V
#pragma unroll
                    for (int kk = 0; kk < kKeys / 16; ++kk)
                        tc_mma_ts_ew(tmem + kTmemO, tm_p + 32 + kk * 8, vd + (uint64_t)((kk * 16 * 128) >> 4), idesc_o,
                                     1u);
                }
                tc_commit_ew(&bars->o_done);
                tc_commit_ew(&bars->v_empty[j % kVStages]);
                if (j + 1 == n) tc_commit_ew(&bars->o_final);
            };
            bool ok = mbar_wait_warp(&bars->q_full, 0);
            // stages 0 and 1 into the two score buffers
            for (int j = 0; j < 2 && j < n && ok; ++j) {
                ok = mbar_wait_warp(&bars->k_full[j], 0);
                if (!ok) break;
                tc_fence_after();
                issue_qk(j);
            }
            for (int j = 0; j < n && ok; ++j) {
                // The operands the stage needs besides P -- V(j) and K(j+2) -- are waited for
                // first (they are normally long in place), so that once P(j) is complete P V(j)
                // and S(j+2) go out back to back.
                ok = mbar_wait_warp(&bars->v_full[j % kVStages], (j / kVStages) & 1);
                if (ok && j + 2 < n) ok = mbar_wait_warp(&bars->k_full[(j + 2) % kKStages], ((j + 2) / kKStages) & 1);
                if (ok) ok = mbar_wait_warp(&bars->p_full[j & 1], (j >> 1) & 1);
                if (!ok) break;
                tc_fence_after();
                issue_pv(j);
                // S(j+2) reuses the buffer P(j) sits in: after P V(j) in this warp's issue order
                if (j + 2 < n) issue_qk(j + 2);
            }
            // every MMA this warp issued has finished before the tensor memory is released
            tc_commit_ew(&bars->drain);
            if (!mbar_wait_warp(&bars->drain, 0)) ok = false;
            if (!ok && lane == 0) atomicOr(a.status, kDevTimeout);
        }
        // Epilogue: for a whole tile, the second column half of O of the lanes this warp may
        // reach (quarter warp % 4), once the softmax warps have published 1/l of every row
        float* xinv = reinterpret_cast<float*>(smem + kOffX);
        const int* xflag = reinterpret_cast<const int*>(xinv + kRows);
        named_sync(3, 256);
        if (*xflag) {
            tc_fence_after();
            const int q = warp & 3, rr = 32 * q + lane;
            const float inv = xinv[rr];
            const uint32_t tm = tmem + ((uint32_t)(32 * q) << 16);
            uint8_t* qs = smem + kOffQ;
#pragma unroll
            for (int c = 64; c < kD; c += 32) {
                uint32_t o[32];
                tmem_ld32(tm + kTmemO + c, o);
#pragma unroll
                for (int e = 0; e < 32; e += 8) {
                    uint4 v;
                    v.x = pack_bf16x2(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv);
                    v.y = pack_bf16x2(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
                    v.z = pack_bf16x2(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv);
                    v.w = pack_bf16x2(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv);
                    const int cc = (c + e) >> 3;
                    *reinterpret_cast<uint4*>(qs + kQHalf + swz128(rr, cc & 7)) = v;
                }
            }
            fence_proxy_async_smem();
        }
        named_sync(3, 256);
        tc_fence_before();
    } else {
        // ------------------------------------------------------------ softmax: one row per thread
        const int r = threadIdx.x;                  // TMEM lane r, MMA row r
        const int nt = nst;
        const bool valid = r < ntok * g;
        const int qi = r / g, h = r % g;
        const int pos = valid ? L - C + tok0 + qi : -1;  // causal limit of the row (inclusive)
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tm_row = tmem + lane_base;
        uint8_t* qs = smem + kOffQ;
        constexpr int bar_id = 1;                   // named barrier of the softmax warps
        if (whole && !neg) {
            if (r == 0) {
                prefetch_tensormap(&tm_q);
                mbar_arrive_expect_tx(&bars->q_full, kQTile);
                tma_load_3d(qs, &tm_q, 0, kvh * g, q0 + tok0, &bars->q_full);
                tma_load_3d(qs + kQHalf, &tm_q, 64, kvh * g, q0 + tok0, &bars->q_full);
            }
        } else {
            // row by row into the same 128-byte swizzled layout (zeros past the chunk); the sign
            // bit of every bf16 flips for a negative scale
            const uint4* src = reinterpret_cast<const uint4*>(
                a.q + ((size_t)(q0 + tok0 + qi) * a.num_heads + (size_t)kvh * g + h) * kD);
            const uint32_t flip = neg ? 0x80008000u : 0u;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint4 v = valid ? __ldg(src + hh * 8 + c) : make_uint4(0u, 0u, 0u, 0u);
                    v.x ^= flip;
                    v.y ^= flip;
                    v.z ^= flip;
                    v.w ^= flip;
                    *reinterpret_cast<uint4*>(qs + hh * kQHalf + swz128(r, c)) = v;
                }
            fence_proxy_async_smem();
            named_sync(bar_id, 128);
            if (r == 0) mbar_arrive(&bars->q_full);
        }
        const float sl = fabsf(a.scale_log2);  // Q carries the sign
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        // tcgen05.ld / tcgen05.st are warp-collective: every decision that leads to one (a wait
        // that gave up, a rescale of O) is taken by the whole warp.
        for (int j = 0; j < nt; ++j) {
            const uint32_t sbuf = tm_row + kTmemS + 64 * (j & 1);
            if (__any_sync(0xffffffffu, !mbar_wait(&bars->s_full[j & 1], (j >> 1) & 1))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int k0 = j * kKeys;
            const int lim = pos - k0;  // keys c <= lim of this stage are visible to the row
            // Stages wholly below the diagonal (every row of the warp sees all 64 keys) take the
            // path without a mask; only they are common.  The path is the warp's vote, never a
            // row's own limit: the branches below hold warp-collective tensor-memory accesses.
            const bool unmasked = __all_sync(0xffffffffu, lim >= kKeys - 1);
            uint32_t s0[32], s1[32];
            tmem_ld32_async(sbuf, s0);
            tmem_ld32_async(sbuf + 32, s1);
            tmem_wait_ld(s0);
            tmem_wait_ld(s1);
            // The stage goes against the row's current base first.  Its maximum -- and with it a
            // possible re-base of O -- is taken only for a row's first visible stage, or when a
            // row's sum passes 2^16 (a score more than 10 above the base): otherwise every
            // p <= 2^16, far from overflow in P, l and O.  Both decisions are the warp's.
            uint32_t pw[kKeys / 2];
            float lsum = 0.f;
            bool full = __any_sync(0xffffffffu, m_used == -INFINITY && lim >= 0);
            if (!full) {
                lsum = stage_p(s0, s1, lim, sl, m_used == -INFINITY ? 0.f : -m_used, unmasked, pw);
                full = __any_sync(0xffffffffu, !(lsum <= kSpecSumLimit));
            }
            if (full) {
                const float mx = unmasked ? stage_max<true>(s0, s1, lim) : stage_max<false>(s0, s1, lim);
                const float mxs = mx == -INFINITY ? -INFINITY : mx * sl;  // log2 units
                const float m_new = fmaxf(m_used, mxs);
                const bool rebase = m_new > m_used + kRescaleThreshold;  // always for the first visible key
                if (__any_sync(0xffffffffu, rebase && m_used != -INFINITY)) {
                    // O changes only once P V(j-1) -- which may still run, since S(j) was ready
                    // long before -- has finished: its commit is o_done phase j-1 (phases up to
                    // j-2 are complete, as S(j) was issued after P V(j-2), and P V(j) waits for
                    // this stage's P, so the parity cannot alias)
                    if (j > 0 && __any_sync(0xffffffffu, !mbar_wait(&bars->o_done, (j - 1) & 1))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    scale_o(tm_row + kTmemO, rebase && m_used != -INFINITY ? fast_exp2(m_used - m_new) : 1.f);
                }
                if (rebase) {
                    l *= m_used == -INFINITY ? 0.f : fast_exp2(m_used - m_new);
                    m_used = m_new;
                }
                lsum = stage_p(s0, s1, lim, sl, m_used == -INFINITY ? 0.f : -m_used, unmasked, pw);
            }
            l += lsum;
            if (kSplit) {
                // the low halves go over the second 32 columns; l sums them too, so the weights
                // the two P V products apply still sum to l
                const float nbase = m_used == -INFINITY ? 0.f : -m_used;
                l += unmasked ? stage_lo<true>(s0, s1, lim, sl, nbase, pw, sbuf + 32)
                              : stage_lo<false>(s0, s1, lim, sl, nbase, pw, sbuf + 32);
            }
            // P goes over the first 32 columns of the stage's buffer
#pragma unroll
            for (int i = 0; i < kKeys / 16; ++i)
                tmem_st8_nowait(sbuf + 8 * i, pw[8 * i], pw[8 * i + 1], pw[8 * i + 2], pw[8 * i + 3], pw[8 * i + 4],
                                pw[8 * i + 5], pw[8 * i + 6], pw[8 * i + 7]);
            tmem_wait_st();
            if (k0 + kKeys > L) {
                // keys at or past the sequence end: zero their V rows, whatever the slots hold
                // (P is 0 there, but 0 times a NaN left in a slot is NaN).  Once V(j) has landed,
                // its slot's previous reader has finished (the refill waited for it); P V(j)
                // follows this stage's P.
                const int s = j % kVStages;
                if (__any_sync(0xffffffffu, !mbar_wait(&bars->v_full[s], (j / kVStages) & 1))) {
                    ok = false;
                    break;
                }
                uint8_t* vt = smem + kOffV + s * kKVStage;
                const int z0 = max(0, L - k0);
                const int nchunks = (kKeys - z0) * 16;  // 16-byte chunks over both column halves
                for (int c = r; c < nchunks; c += kRows) {
                    const int row = z0 + (c >> 4), half = (c >> 3) & 1, cc = c & 7;
                    *reinterpret_cast<uint4*>(vt + half * kKVHalf + row * 128 + cc * 16) = make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
            }
            tc_fence_before();
            mbar_arrive(&bars->p_full[j & 1]);
        }
        {
            if (ok) ok = !__any_sync(0xffffffffu, !mbar_wait(&bars->o_final, 0));
            // one verdict for the softmax warps, which then take the same path
            const bool all_ok = named_sync_all(bar_id, 128, ok);
            const float inv = l > 0.f ? 1.f / l : 0.f;
            float* xinv = reinterpret_cast<float*>(smem + kOffX);
            int* xflag = reinterpret_cast<int*>(xinv + kRows);
            // a whole tile: the control warps take the second column half of every quarter
            xinv[r] = inv;
            if (r == 0) *xflag = all_ok && whole;
            named_sync(3, 256);
            if (all_ok) {
                tc_fence_after();
                if (whole) {
#pragma unroll
                    for (int c = 0; c < 64; c += 32) {
                        uint32_t o[32];
                        tmem_ld32(tm_row + kTmemO + c, o);
#pragma unroll
                        for (int e = 0; e < 32; e += 8) {
                            uint4 v;
                            v.x = pack_bf16x2(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv);
                            v.y = pack_bf16x2(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
                            v.z = pack_bf16x2(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv);
                            v.w = pack_bf16x2(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv);
                            const int cc = (c + e) >> 3;  // 16-byte chunk of the row, 0..7
                            *reinterpret_cast<uint4*>(qs + swz128(r, cc)) = v;
                        }
                    }
                    fence_proxy_async_smem();
                } else {
                    // a tile cut short: each thread stores its own row (256 contiguous bytes)
                    __nv_bfloat16* dst = a.out + ((size_t)(q0 + tok0 + qi) * a.num_heads + (size_t)kvh * g + h) * kD;
#pragma unroll
                    for (int c = 0; c < kD; c += 32) {
                        uint32_t o[32];
                        tmem_ld32(tm_row + kTmemO + c, o);
                        if (valid) {
#pragma unroll
                            for (int e = 0; e < 32; e += 8) {
                                uint4 v;
                                v.x = pack_bf16x2(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv);
                                v.y = pack_bf16x2(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
                                v.z = pack_bf16x2(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv);
                                v.w = pack_bf16x2(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv);
                                *reinterpret_cast<uint4*>(dst + c + e) = v;
                            }
                        }
                    }
                }
            }
            named_sync(3, 256);  // both column halves staged
            if (all_ok && whole && r == 0) {
                tma_store_3d(&tm_o, 0, kvh * g, q0 + tok0, qs);
                tma_store_3d(&tm_o, 64, kvh * g, q0 + tok0, qs + kQHalf);
                bulk_commit();
                bulk_wait_read();  // the shared memory stays until the store has read it
            }
            if (!ok) atomicOr(a.status, kDevTimeout);
        }
        tc_fence_before();
    }
    __syncthreads();
    pdl_trigger();  // the next kernel may launch while this CTA leaves
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// The two-halves tile as a function of its own: its code stays out of the way of the
// one-half form's, whose instructions are fetched cold after an L2 flush (inlined side by
// side, the two forms made a cold launch of the one-half form about 10 us slower, with a
// fifth of the issue slots lost to instruction fetch).
__device__ __noinline__ void tc2_tile_split(const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                            const CUtensorMap& tm_q, const CUtensorMap& tm_o, const Tc2Args& a) {
    tc2_tile<true>(tm_k, tm_v, tm_q, tm_o, a);
}

// kSplitAll: every tile carries P as two halves (a large scale).  Otherwise only the tiles
// with a query that sees at most kFewKeys keys do -- the first queries of a sequence.
template <bool kSplitAll>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) prefill_tc2_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                                           const __grid_constant__ CUtensorMap tm_v,
                                                                           const __grid_constant__ CUtensorMap tm_q,
                                                                           const __grid_constant__ CUtensorMap tm_o,
                                                                           const __grid_constant__ Tc2Args a) {
    tc2_tile<kSplitAll>(tm_k, tm_v, tm_q, tm_o, a);
}

}  // namespace

cudaError_t launch_prefill_tc2(const PoolView& pool, const AttnArgs& a, cudaStream_t stream) {
    static OncePerDevice configured;
    const cudaError_t e = configured.run([] {
        cudaError_t r = cudaSuccess;
        for (const void* fn : {(const void*)prefill_tc2_kernel<false>, (const void*)prefill_tc2_kernel<true>}) {
            if (r == cudaSuccess) r = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
            // all of the SM's unified memory as shared memory, so that two CTAs fit
            if (r == cudaSuccess)
                r = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         (int)cudaSharedmemCarveoutMaxShared);
        }
        return r;
    });
    if (e != cudaSuccess) return e;
    const int g = a.num_heads / pool.num_kv_heads;
    const int tpt = kRows / g;
    // q as (d, head, token) with one query tile per box; a whole tile never reaches past the
    // chunk rows, whose total is at most batch * max_chunk
    const long long tokens = (long long)a.batch * a.max_chunk;
    CUtensorMap tm_q;
    if (!rows_map(&tm_q, a.q, tokens, a.num_heads, kD, g, tpt)) return cudaErrorInvalidValue;
    CUtensorMap tm_o;  // out, shaped like q: whole tiles are stored through it
    if (!rows_map(&tm_o, a.out, tokens, a.num_heads, kD, g, tpt)) return cudaErrorInvalidValue;
    Tc2Args t;
    t.q = static_cast<const __nv_bfloat16*>(a.q);
    t.block_tables = a.block_tables;
    t.seq_lens = a.seq_lens;
    t.cu_q_lens = a.cu_q_lens;
    t.out = static_cast<__nv_bfloat16*>(a.out);
    t.status = a.status;
    t.max_blocks = a.max_blocks;
    t.num_heads = a.num_heads;
    t.num_kv_heads = pool.num_kv_heads;
    t.num_blocks = pool.num_blocks;
    t.group = g;
    t.q_rows = (int)std::min<long long>(tokens, 0x7fffffffLL);
    t.scale_log2 = a.scale * kLog2e;
    const int tiles = std::max(1, (a.max_chunk + tpt - 1) / tpt);
    t.batch = a.batch;
    t.tiles = tiles;
    // Rounding P to bf16 perturbs each weight by up to 2^-9 of itself.  Where a few weights
    // dominate a row -- a peaked softmax (scores spread much wider than 1/sqrt(d) would make
    // them), or a query that sees only a few keys -- that error is not averaged away and
    // approaches the output tolerance, so P is then also carried as a low half: in every tile
    // at such a scale, else in the tiles that hold a sequence's first kFewKeys queries.
    const bool split = std::fabs(a.scale) * std::sqrt((float)kD) > kSplitScale;
    const long long ctas = (long long)tiles * a.batch * pool.num_kv_heads;
    if (ctas > 0x7fffffffLL) return cudaErrorInvalidValue;  // more CTAs than a grid holds
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return split ? cudaLaunchKernelEx(&cfg, prefill_tc2_kernel<true>, pool.tm_k, pool.tm_v, tm_q, tm_o, t)
                 : cudaLaunchKernelEx(&cfg, prefill_tc2_kernel<false>, pool.tm_k, pool.tm_v, tm_q, tm_o, t);
}

}  // namespace pa
