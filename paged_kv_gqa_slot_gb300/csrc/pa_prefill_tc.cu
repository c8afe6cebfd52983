// pa_prefill_tc.cu -- chunked prefill over a cached paged prefix on the 5th-generation
// tensor cores (tcgen05 MMA, accumulators in tensor memory).
//
// Method: "Qwen3-4B / 8B / 32B", sections "Warm Prefix-Cache TTFT" (a warm prefix hit:
// only the new chunk is computed, over the cached prefix) and "Architecture Notes" (GQA
// over a paged KV cache).  Chunk query i of sequence s sits at position L_s - C_s + i and
// attends causally to keys 0 .. L_s - C_s + i through the block table.
//
// Rows of a query tile are (query, head-of-the-group) pairs: row r = query r / g, head r % g,
// so one K/V tile serves all g heads; a tile holds 128 rows (128 / g queries).  One CTA per
// SM holds TWO query tiles of the same (sequence, kv head), the i-th longest with the i-th
// shortest (tiles T-1-i and i), so every CTA has about the same causal work.  Per stage of
// 64 keys (four 16-token pool blocks, loaded by TMA with 128-byte swizzling), for each tile:
//   S[128 x 64]  = Q K^T      tcgen05.mma, M=128 N=64, Q (A) from TMEM, K (B) from smem
//   softmax      one thread per row reads its S row from TMEM, masks causally (only in
//                tiles that cross the diagonal), keeps an online max / sum in base 2 and
//                writes P (bf16, 128-byte swizzled) to shared memory
//   O[128 x 128] += P V       tcgen05.mma, M=128 N=128, P (A) and V (B) from smem
// Each tile owns 256 TMEM columns: S [0,64), Q [64,128) (bf16 pairs), O [128,256).  The
// running max is re-based lazily: O is rescaled in TMEM only when a row's max grows by more
// than 2^8, which keeps every P <= 256 and makes rescales rare.
// Warp roles: 0-3 softmax of tile 0, 4-7 softmax of tile 1 (TMEM lanes 32(w%4)..+31),
// 8 MMA issue + TMEM owner, 9 TMA loads of K, 10 TMA loads of V.  While one tile's softmax
// runs, the other tile's MMAs do, so the tensor pipe and the special-function units
// overlap.  A warp issues only a few TMA boxes per microsecond, so K and V have a warp each
// and never wait on each other's ring.
// K and V have separate 4-slot rings: a K slot is handed back as soon as both tiles' Q K^T
// have run; 4 slots cover the L2 round trip of the next tiles.  P is double-buffered per
// tile, so the softmax of key tile j+1 waits for P V of tile j-1 only (long finished),
// unless O must be rescaled.
// Every CTA loads its own K/V boxes into its own shared memory.  The CTAs of one
// (sequence, kv head) -- and, with a shared prefix, of every sequence that shares it --
// read the same pool blocks; the copies after the first come from L2, which the loads ask
// to keep them (evict-last policy).
#include <algorithm>
#include <cmath>
#include <cstdlib>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kD = 128;
constexpr int kRows = 128;                      // MMA M: rows of one query tile
constexpr int kTiles = 2;                       // query tiles per CTA
constexpr int kKeys = 64;                       // keys per stage (MMA N of S)
constexpr int kKStages = 4, kVStages = 4, kPBufs = 2;
constexpr int kSoftmaxThreads = kTiles * 128;
constexpr int kMmaWarp = kSoftmaxThreads / 32, kKLoadWarp = kMmaWarp + 1, kVLoadWarp = kMmaWarp + 2;
constexpr int kThreads = kSoftmaxThreads + 96;
constexpr int kTmemCols = 512;
constexpr uint32_t kTmemTile = 256;             // columns owned by one tile
constexpr uint32_t kTmemS = 0, kTmemQ = 64, kTmemO = 128;
constexpr int kHalf = kKeys * 128;              // [64 keys][64 columns] bf16 = 8 KB
constexpr int kTileBytes = 2 * kHalf;           // one K or V stage (two column halves), 16 KB
constexpr int kPBytes = kRows * 128;            // [128 rows][64 keys] bf16 = 16 KB
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kKStages * kTileBytes;
constexpr int kOffP = kOffV + kVStages * kTileBytes;
constexpr int kBarOff = kOffP + kTiles * kPBufs * kPBytes;
constexpr int kSmemBytes = kBarOff + 512 + 1024;
constexpr float kLog2e = 1.44269504088896340736f;
constexpr float kRescaleThreshold = 8.f;        // log2 units

struct Bars {
    uint64_t k_full[kKStages], k_empty[kKStages], v_full[kVStages], v_empty[kVStages];
    uint64_t q_full[kTiles], s_full[kTiles], s_free[kTiles];
    uint64_t p_full[kTiles][kPBufs], o_done[kTiles][kPBufs];  // per P buffer: P written, P V done
    uint64_t drain;
    uint32_t tmem_base;
};
static_assert(sizeof(Bars) <= 512, "barrier block");
static_assert(kSmemBytes <= 227 * 1024, "shared memory");

struct TcArgs {
    const __nv_bfloat16* q;
    const int32_t* block_tables;
    const int32_t* seq_lens;
    const int32_t* cu_q_lens;
    __nv_bfloat16* out;
    unsigned* status;
    int max_blocks, num_heads, num_kv_heads, num_blocks, group;
    float scale_log2;  // |scale| log2(e)
    int negate_q;      // scale < 0: Q enters negated
};

// Keys a query tile needs: [0, kmax) with kmax the position of its last query + 1.
__device__ __forceinline__ int tile_key_count(int mt, int tpt, int C, int L) {
    const int tok0 = mt * tpt;
    if (mt < 0 || tok0 >= C) return 0;
    return L - C + tok0 + min(tpt, C - tok0);
}

// The two query tiles of pair p out of T: the (p+1)-th longest and the (p+1)-th shortest
// (-1: none).  Pairs p >= ceil(T / 2) hold nothing.
__device__ __forceinline__ void pair_tiles(int p, int T, int& t0, int& t1) {
    t0 = -1;
    t1 = -1;
    if (p < 0 || 2 * p >= T) return;
    t0 = T - 1 - p;
    t1 = p < t0 ? p : -1;
}

__device__ __forceinline__ int pair_key_count(int p, int T, int tpt, int C, int L) {
    int t0, t1;
    pair_tiles(p, T, t0, t1);
    return max(tile_key_count(t0, tpt, C, L), tile_key_count(t1, tpt, C, L));
}

// Score c of a 64-key stage held in two 32-column loads.
__device__ __forceinline__ float score(const uint32_t (&s0)[32], const uint32_t (&s1)[32], int c) {
    return __uint_as_float(c < 32 ? s0[c] : s1[c - 32]);
}

// Maximum of the row's visible raw scores in one stage: keys c <= lim, or every key (kAll: a
// stage wholly below the diagonal, the common case, needs no mask).  Four independent chains
// of three-input max: one row per thread leaves no other parallelism to hide a long chain.
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

// The row of P for one stage: p = 2^(s |scale| log2(e) - base) for keys c <= lim (every key
// when kAll), one packed multiply-add per two keys and the special-function unit, rounded to
// bf16 and stored as the row's 128 bytes of the 128-byte-swizzled P tile.  Returns the sum of
// the rounded values (so the weights P V uses sum to the normaliser), in independent chains.
template <bool kAll>
__device__ __forceinline__ float stage_p(const uint32_t (&s0)[32], const uint32_t (&s1)[32], int lim, float sl,
                                         float nbase, uint8_t* prow, int r) {
    float ls[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int cc = 0; cc < kKeys / 8; ++cc) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            const int c = cc * 8 + e;
            float x0, x1;
            fma_x2(x0, x1, score(s0, s1, c), score(s0, s1, c + 1), sl, sl, nbase, nbase);
            if (!kAll) {
                x0 = c > lim ? -INFINITY : x0;  // 2^-inf = 0
                x1 = c + 1 > lim ? -INFINITY : x1;
            }
            w[e / 2] = pack_bf16x2(fast_exp2(x0), fast_exp2(x1));
        }
        add_x2(ls[0], ls[1], bf16_lo(w[0]), bf16_hi(w[0]));
        add_x2(ls[2], ls[3], bf16_lo(w[1]), bf16_hi(w[1]));
        add_x2(ls[4], ls[5], bf16_lo(w[2]), bf16_hi(w[2]));
        add_x2(ls[6], ls[7], bf16_lo(w[3]), bf16_hi(w[3]));
        *reinterpret_cast<uint4*>(prow + swz128(r, cc)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    return ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
}

__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                                 const __grid_constant__ CUtensorMap tm_v,
                                                                 const __grid_constant__ TcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Bars* bars = reinterpret_cast<Bars*>(smem + kBarOff);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int p = blockIdx.x;  // tile pair
    const int kvh = blockIdx.y, b = blockIdx.z;
    pdl_wait();
    const int g = a.group, tpt = kRows / g;
    const int q0 = a.cu_q_lens[b];
    const int C = a.cu_q_lens[b + 1] - q0;
    const int L = a.seq_lens[b];
    if (C < 0 || L < C || L > a.max_blocks * kBlockSize) {
        if (threadIdx.x == 0 && p == 0 && kvh == 0) atomicOr(a.status, kDevOutOfRange);
        return;
    }
    const int T = (C + tpt - 1) / tpt;  // query tiles of this sequence
    // a chunk longer than max_chunk needs more tile pairs than the grid has: its middle tiles
    // would go unwritten, so it is reported
    if (p == 0 && kvh == 0 && threadIdx.x == 0 && (T + 1) / 2 > (int)gridDim.x) atomicOr(a.status, kDevOutOfRange);
    int mtile[kTiles], ntiles[kTiles];
    pair_tiles(p, T, mtile[0], mtile[1]);
#pragma unroll
    for (int t = 0; t < kTiles; ++t) ntiles[t] = (tile_key_count(mtile[t], tpt, C, L) + kKeys - 1) / kKeys;
    const int kmax = pair_key_count(p, T, tpt, C, L);             // keys either tile needs
    const int ntiles_cta = (kmax + kKeys - 1) / kKeys;             // key tiles loaded
    const int nblk = (kmax + kBlockSize - 1) / kBlockSize;         // pool blocks read

    if (threadIdx.x == 0) {
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(&bars->k_full[s], 1);
            mbar_init(&bars->k_empty[s], 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(&bars->v_full[s], 1);
            mbar_init(&bars->v_empty[s], 1);
        }
        for (int t = 0; t < kTiles; ++t) {
            mbar_init(&bars->q_full[t], 128);
            mbar_init(&bars->s_full[t], 1);
            mbar_init(&bars->s_free[t], 128);
            for (int s = 0; s < kPBufs; ++s) {
                mbar_init(&bars->p_full[t][s], 128);
                mbar_init(&bars->o_done[t][s], 1);
            }
        }
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

    if (warp == kKLoadWarp || warp == kVLoadWarp) {
        // ------------------------------------------------------------ TMA producers (K, V)
        // The 8 boxes of a stage (4 blocks x 2 column halves) go out from lanes 0-7, one each.
        const bool is_k = warp == kKLoadWarp;
        const CUtensorMap* map = is_k ? &tm_k : &tm_v;
        uint64_t* full = is_k ? bars->k_full : bars->v_full;
        uint64_t* empty = is_k ? bars->k_empty : bars->v_empty;
        uint8_t* ring = smem + (is_k ? kOffK : kOffV);
        constexpr int kStages = kKStages;
        static_assert(kKStages == kVStages, "one ring shape for both producers");
        if (lane == 0) prefetch_tensormap(map);
        const uint64_t pol = l2_evict_last_policy();  // prefix blocks are shared across sequences
        const int32_t* bt = a.block_tables + (size_t)b * a.max_blocks;
        const int oob_row = a.num_blocks * a.num_kv_heads * kBlockSize;  // past the pool: zero fill
        int c0 = 0;
        int cur = lane < nblk ? __ldg(bt + lane) : 0;
        int nxt = 32 + lane < nblk ? __ldg(bt + 32 + lane) : 0;
        const bool my_box = lane < 8;
        const int box_t = lane >> 1, box_h = lane & 1;
        bool ok = true;
        int issued = 0;
        for (int j = 0; j < ntiles_cta && ok; ++j) {
            // pool row of block 4j + box_t (for the issuing lanes)
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
            const int s = j % kStages;
            if (lane == 0) {
                if (j >= kStages) ok = mbar_wait(&empty[s], ((j / kStages) & 1) ^ 1);
                if (ok) mbar_arrive_expect_tx(&full[s], kTileBytes);
            }
            ok = __shfl_sync(0xffffffffu, ok, 0) != 0;
            if (ok) {
                if (my_box)
                    tma_load_2d(ring + s * kTileBytes + box_h * kHalf + box_t * 2048, map, box_h * 64, row, &full[s],
                                pol);
                ++issued;
            }
        }
        if (lane == 0) {
            // Before the CTA may leave: every box issued here has landed.
            for (int j = max(0, issued - kStages); j < issued; ++j)
                if (!mbar_wait(&full[j % kStages], (j / kStages) & 1)) ok = false;
            if (!ok) atomicOr(a.status, kDevTimeout);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issue (whole warp)
        // per key tile j: S_0 = Q_0 K_j^T, S_1 = Q_1 K_j^T, then O_0 += P_0 V_{j-1},
        // O_1 += P_1 V_{j-1}: each tile's Q K^T runs while the other tile's softmax does.
        // The warp runs the loop together and one elected lane issues, so every operand is
        // warp-uniform; waits give one verdict for the warp.
        constexpr uint32_t idesc_s = tc_idesc_bf16(kRows, kKeys, false);
        constexpr uint32_t idesc_o = tc_idesc_bf16(kRows, kD, true);
        // Operand descriptors are built once; a stage, a buffer or a k-step only moves the
        // start address, which adds (offset >> 4) to the low field (no carry: every shared
        // address is below 2^18).
        const uint64_t kdesc0 = smem_desc_sw128(smem_u32(smem + kOffK), 0, 1024);
        const uint64_t vdesc0 = smem_desc_sw128(smem_u32(smem + kOffV), kHalf, 1024);
        const uint64_t pdesc0 = smem_desc_sw128(smem_u32(smem + kOffP), 0, 1024);
        bool ok = true;
#pragma unroll
        for (int t = 0; t < kTiles; ++t)
            if (ok && ntiles[t] > 0) ok = mbar_wait_warp(&bars->q_full[t], 0);
        int ks_ = 0, kph = 0, vs_ = 0, vph = 0;  // ring slot and phase of K(j) and V(j-1)
        for (int j = 0; j <= ntiles_cta && ok; ++j) {
            if (j < ntiles_cta) {
                ok = mbar_wait_warp(&bars->k_full[ks_], kph);
                const uint64_t kd = kdesc0 + (uint64_t)((ks_ * kTileBytes) >> 4);
#pragma unroll
                for (int t = 0; t < kTiles; ++t) {
                    if (!ok || j >= ntiles[t]) continue;
                    if (j > 0) ok = mbar_wait_warp(&bars->s_free[t], (j - 1) & 1);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t tm_s = tmem + t * kTmemTile + kTmemS, tm_q = tmem + t * kTmemTile + kTmemQ;
#pragma unroll
                    for (int kk = 0; kk < kD / 16; ++kk)
                        tc_mma_ts_ew(tm_s, tm_q + kk * 8, kd + (uint64_t)(((kk >> 2) * kHalf + (kk & 3) * 32) >> 4),
                                     idesc_s, kk > 0 ? 1u : 0u);
                    tc_commit_ew(&bars->s_full[t]);
                }
                if (!ok) break;
                tc_commit_ew(&bars->k_empty[ks_]);  // release the K slot once both Q K^T have run
                if (++ks_ == kKStages) {
                    ks_ = 0;
                    kph ^= 1;
                }
            }
            if (j > 0) {
                const int jp = j - 1, pb = jp & (kPBufs - 1);
                ok = mbar_wait_warp(&bars->v_full[vs_], vph);
                const uint64_t vd = vdesc0 + (uint64_t)((vs_ * kTileBytes) >> 4);
#pragma unroll
                for (int t = 0; t < kTiles; ++t) {
                    if (!ok || jp >= ntiles[t]) continue;
                    ok = mbar_wait_warp(&bars->p_full[t][pb], (jp / kPBufs) & 1);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t pd = pdesc0 + (uint64_t)(((t * kPBufs + pb) * kPBytes) >> 4);
                    const uint32_t tm_o = tmem + t * kTmemTile + kTmemO;
                    tc_mma_ew(tm_o, pd, vd, idesc_o, jp > 0 ? 1u : 0u);
#pragma unroll
                    for (int ks = 1; ks < kKeys / 16; ++ks)
                        tc_mma_ew(tm_o, pd + (uint64_t)((ks * 32) >> 4), vd + (uint64_t)((ks * 16 * 128) >> 4), idesc_o,
                                  1u);
                    tc_commit_ew(&bars->o_done[t][pb]);
                }
                if (!ok) break;
                tc_commit_ew(&bars->v_empty[vs_]);
                if (++vs_ == kVStages) {
                    vs_ = 0;
                    vph ^= 1;
                }
            }
        }
        // every MMA issued above has finished before the tensor memory is released
        tc_commit_ew(&bars->drain);
        if (!mbar_wait_warp(&bars->drain, 0)) ok = false;
        if (!ok && lane == 0) atomicOr(a.status, kDevTimeout);
    } else {
        // ------------------------------------------------------------ softmax: one row per thread
        const int t = warp >> 2;                    // query tile of this warpgroup
        const int r = threadIdx.x & (kRows - 1);    // TMEM lane r, MMA row r
        const int mt = t == 0 ? mtile[0] : mtile[1], nt = t == 0 ? ntiles[0] : ntiles[1];
        const int tok0 = mt * tpt;
        const int ntok = (mt >= 0 && tok0 < C) ? min(tpt, C - tok0) : 0;
        const bool valid = r < ntok * g;
        const int qi = r / g, h = r % g;
        const int pos = valid ? L - C + tok0 + qi : -1;  // causal limit of the row (inclusive)
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tm_row = tmem + lane_base + t * kTmemTile;
        // this warpgroup zeroes V rows past the sequence end in key tile j unless tile 0 of
        // this CTA computes j too (it does so first: the MMA thread issues tile 0's P V first)
        const int zero_from = t == 0 ? 0 : ntiles[0];
        if (nt > 0) {
            // Q row -> TMEM columns [64, 128) as bf16 pairs (zeros for rows past the chunk).
            // A negative scale is carried by negating Q (exact in bf16), so the kernel works
            // with |scale| and the row maximum of the raw scores.
            const uint32_t sign = a.negate_q ? 0x80008000u : 0u;
            const uint4* src = reinterpret_cast<const uint4*>(
                a.q + ((size_t)(q0 + tok0 + qi) * a.num_heads + (size_t)kvh * g + h) * kD);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t w[32];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 v = valid ? __ldg(src + half * 8 + c) : make_uint4(0u, 0u, 0u, 0u);
                    w[4 * c] = v.x ^ sign;
                    w[4 * c + 1] = v.y ^ sign;
                    w[4 * c + 2] = v.z ^ sign;
                    w[4 * c + 3] = v.w ^ sign;
                }
                tmem_st32(tm_row + kTmemQ + half * 32, w);
            }
            tc_fence_before();
            mbar_arrive(&bars->q_full[t]);
        }
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        // tcgen05.ld / tcgen05.st are warp-collective: every decision that leads to one (a wait
        // that gave up, a rescale of O) is taken by the whole warp.
        for (int j = 0; j < nt; ++j) {
            if (__any_sync(0xffffffffu, !mbar_wait(&bars->s_full[t], j & 1))) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sr[2][32];
            tmem_ld64(tm_row + kTmemS, sr[0], sr[1]);
            tc_fence_before();
            mbar_arrive(&bars->s_free[t]);

            const int k0 = j * kKeys;
            const int lim = pos - k0;  // keys c <= lim of this tile are visible to the row
            // Tiles wholly below the diagonal (every row of the warp sees all 64 keys) take the
            // path without a mask; only they are common.  The warp's vote picks the path, so
            // the warp stays converged through the collective accesses below.
            const bool unmasked = __all_sync(0xffffffffu, lim >= kKeys - 1);
            const float mx = unmasked ? stage_max<true>(sr[0], sr[1], lim) : stage_max<false>(sr[0], sr[1], lim);
            const float mxs = mx == -INFINITY ? -INFINITY : mx * a.scale_log2;  // log2 units
            const float m_new = fmaxf(m_used, mxs);
            const bool rescale = m_new > m_used + kRescaleThreshold;  // always for the first visible key
            const int pb = j % kPBufs;
            // P buffer pb was last read by P V(j-2), which the MMA warp issued before Q K^T(j):
            // the commit behind s_full(j) covers every tcgen05 op issued before it, so that
            // P V has finished.  O is touched here only when it must be rescaled, and then
            // P V(j-1) (issued after Q K^T(j)) must have finished too; a buffer's barrier
            // cannot run two phases ahead of that wait, since P V(j) needs P(j) first.
            const bool warp_rescale = __any_sync(0xffffffffu, rescale && m_used != -INFINITY);
            if (warp_rescale && j >= 1) {
                if (__any_sync(0xffffffffu,
                               !mbar_wait(&bars->o_done[t][(j - 1) % kPBufs], ((j - 1) / kPBufs) & 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
            }
            // alpha = 2^(m_old - m_new) for rows that re-base (0 while nothing was visible), else 1
            const float alpha = rescale ? fast_exp2(m_used - m_new) : 1.f;
            if (warp_rescale) {
#pragma unroll
                for (int c = 0; c < kD; c += 32) {
                    uint32_t o[32];
                    tmem_ld32(tm_row + kTmemO + c, o);
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tmem_st32(tm_row + kTmemO + c, o);
                }
            }
            if (rescale) {
                l *= alpha;
                m_used = m_new;
            }
            const float nbase = m_used == -INFINITY ? 0.f : -m_used;
            uint8_t* prow = smem + kOffP + (t * kPBufs + pb) * kPBytes;
            l += unmasked ? stage_p<true>(sr[0], sr[1], lim, a.scale_log2, nbase, prow, r)
                          : stage_p<false>(sr[0], sr[1], lim, a.scale_log2, nbase, prow, r);
            if (k0 + kKeys > L && j >= zero_from) {
                // keys at or past the sequence end: zero their V rows, whatever the slots hold.
                // Once V(j) has landed, every earlier reader of the slot has finished (its
                // refill waited for all of them), and P V(j) of either tile is issued after
                // this warpgroup's P(j) is complete.
                const int s = j % kVStages;
                if (__any_sync(0xffffffffu, !mbar_wait(&bars->v_full[s], (j / kVStages) & 1))) {
                    ok = false;
                    break;
                }
                uint8_t* vt = smem + kOffV + s * kTileBytes;
                const int z0 = max(0, L - k0);
                const int nchunks = (kKeys - z0) * 16;  // 16-byte chunks over both column halves
                for (int c = r; c < nchunks; c += kRows) {
                    const int row = z0 + (c >> 4), half = (c >> 3) & 1, cc = c & 7;
                    *reinterpret_cast<uint4*>(vt + half * kHalf + row * 128 + cc * 16) = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bars->p_full[t][pb]);
        }
        if (ok && nt > 0)
            ok = !__any_sync(0xffffffffu, !mbar_wait(&bars->o_done[t][(nt - 1) % kPBufs], ((nt - 1) / kPBufs) & 1));
        if (ok && nt > 0) {
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
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
        if (!ok) atomicOr(a.status, kDevTimeout);
        tc_fence_before();
    }
    __syncthreads();
    pdl_trigger();  // the next kernel may launch while this CTA leaves
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

bool prefill_tc_supported(int head_dim, int group) {
    return head_dim == kD && group > 0 && group <= kRows && kRows % group == 0;
}

cudaError_t launch_prefill_tc(const PoolView& pool, const AttnArgs& a, cudaStream_t stream) {
    static OncePerDevice configured;
    const cudaError_t e = configured.run(
        [] { return cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes); });
    if (e != cudaSuccess) return e;
    TcArgs t;
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
    t.group = a.num_heads / pool.num_kv_heads;
    t.scale_log2 = std::fabs(a.scale) * kLog2e;
    t.negate_q = a.scale < 0.f ? 1 : 0;
    const int tpt = kRows / t.group;
    const int tiles = std::max(1, (a.max_chunk + tpt - 1) / tpt);
    const int pairs = (tiles + 1) / 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(pairs, pool.num_kv_heads, a.batch);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, prefill_tc_kernel, pool.tm_k, pool.tm_v, t);
}

}  // namespace pa
