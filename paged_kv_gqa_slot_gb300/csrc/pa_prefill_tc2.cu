// pa_prefill_tc2.cu -- chunked prefill over a cached paged prefix on the 5th-generation
// tensor cores, 128 keys per stage with P kept in tensor memory.
//
// Method: "Qwen3-4B / 8B / 32B", sections "Warm Prefix-Cache TTFT" (a warm prefix hit:
// only the new chunk is computed, over the cached prefix) and "Architecture Notes" (GQA
// over a paged KV cache).  Chunk query i of sequence s sits at position L_s - C_s + i and
// attends causally to keys 0 .. L_s - C_s + i through the block table.
//
// Rows of a query tile are (query, head-of-the-group) pairs: row r = query r / g, head r % g,
// so one K/V tile serves all g heads; a tile holds 128 rows (128 / g queries).  One CTA per
// SM holds TWO query tiles of the same (sequence, kv head), the i-th longest with the i-th
// shortest, so every CTA has about the same causal work.  Per stage of 128 keys (eight
// 16-token pool blocks, loaded by TMA with 128-byte swizzling), for each tile t:
//   S_t[128 x 128] = Q_t K^T    tcgen05.mma, M=128 N=128, Q_t (A) and K (B) from smem
//   softmax          one thread per row reads its S row from TMEM, masks causally (only in
//                    stages that cross the diagonal), keeps an online max / sum in base 2 and
//                    writes P (bf16) back into the first 64 columns of S_t in TMEM
//   O_t += P_t V     tcgen05.mma, M=128 N=128, P_t (A) from TMEM, V (B) from smem
// Tensor memory: tile t owns columns [256t, 256t+256): S_t (and P_t over its first half)
// [0, 128) and O_t [128, 256).  The tensor core runs the MMAs of one CTA in issue order, so
// the half of S_t(j+1) that P_t(j) shares, keys 0-63, is written only after P_t V(j) has read
// P_t(j); keys 64-127 are computed as soon as the softmax has read those columns of S_t(j).
// Per stage j the MMA warp issues, for each tile, S_t(j+1) keys 64-127, then P_t V(j) and S_t(j+1)
// keys 0-63, so one tile's softmax runs while the other tile's MMAs do.  The running max is
// re-based lazily: O is rescaled in TMEM only when a row's max grows by more than 2^8, which
// keeps every P <= 256 and makes rescales rare.
// Q tiles come in by TMA through a 3-D map of q (d, head, token) whose box is one tile (a tile
// cut short by the end of its chunk row by row instead); each row of O is stored by its thread.
// Warp roles: 0-3 softmax of tile 0, 4-7 softmax of tile 1 (TMEM lanes 32(w%4)..+31),
// 8 MMA issue + TMEM owner, 9 TMA loads of K, 10 TMA loads of V.  Every CTA loads its own
// K/V; the CTAs of one (sequence, kv head) -- and, with a shared prefix, of every sequence
// that shares it -- read the same pool blocks, the copies after the first from L2.
#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <type_traits>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kD = 128;
constexpr int kRows = 128;                      // MMA M: rows of one query tile
constexpr int kTiles = 2;                       // query tiles per CTA
constexpr int kKeys = 128;                      // keys per stage (MMA N of S, K of P V)
constexpr int kKStages = 3;                     // K ring slots: S(j+1)'s upper half starts early
constexpr int kVStages = 2;                     // V ring slots
constexpr int kSoftmaxThreads = kTiles * 128;
constexpr int kMmaWarp = kSoftmaxThreads / 32, kKLoadWarp = kMmaWarp + 1, kVLoadWarp = kMmaWarp + 2;
constexpr int kThreads = kSoftmaxThreads + 96;
constexpr int kTmemCols = 512;
constexpr uint32_t kTmemTile = 256;             // columns owned by one tile
constexpr uint32_t kTmemS = 0, kTmemO = 128;
constexpr int kHalfBytes = 128 * 128;           // [128 rows][64 columns] bf16 = 16 KB
constexpr int kTileBytes = 2 * kHalfBytes;      // a Q tile, or one K or V stage: two column halves
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kTiles * kTileBytes;
constexpr int kOffV = kOffK + kKStages * kTileBytes;
constexpr int kBarOff = kOffV + kVStages * kTileBytes;
constexpr int kSmemBytes = kBarOff + 256 + 1024;
constexpr float kLog2e = 1.44269504088896340736f;
constexpr float kRescaleThreshold = 8.f;        // log2 units

struct Bars {
    uint64_t k_full[kKStages], k_empty[kKStages], v_full[kVStages], v_empty[kVStages];
    uint64_t q_full[kTiles], s_full[kTiles], s_hi_free[kTiles], p_full[kTiles], o_done[kTiles];
    uint64_t drain;
    uint32_t tmem_base;
};
static_assert(sizeof(Bars) <= 256, "barrier block");
static_assert(kSmemBytes <= 227 * 1024, "shared memory");
static_assert(kRows == kKeys, "one 16 KB half layout for Q tiles and K/V stages");

struct Tc2Args {
    const __nv_bfloat16* q;
    const int32_t* block_tables;
    const int32_t* seq_lens;
    const int32_t* cu_q_lens;
    __nv_bfloat16* out;
    unsigned* status;
    int max_blocks, num_heads, num_kv_heads, num_blocks, group;
    float scale_log2;  // scale * log2(e), signed
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

__global__ void __launch_bounds__(kThreads, 1) prefill_tc2_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                                  const __grid_constant__ CUtensorMap tm_v,
                                                                  const __grid_constant__ CUtensorMap tm_q,
                                                                  const __grid_constant__ Tc2Args a) {
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
    int mtile[kTiles], nst[kTiles];
    pair_tiles(p, T, mtile[0], mtile[1]);
#pragma unroll
    for (int t = 0; t < kTiles; ++t) nst[t] = (tile_key_count(mtile[t], tpt, C, L) + kKeys - 1) / kKeys;
    const int nstage = nst[0];  // tile 0 is the later one: it needs the most keys
    if (nstage == 0) return;    // this pair holds no query of the chunk (the same for the whole CTA)
    const int nblk = (tile_key_count(mtile[0], tpt, C, L) + kBlockSize - 1) / kBlockSize;  // pool blocks read

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
            mbar_init(&bars->q_full[t], 1);
            mbar_init(&bars->s_full[t], 1);
            mbar_init(&bars->s_hi_free[t], 128);
            mbar_init(&bars->p_full[t], 128);
            mbar_init(&bars->o_done[t], 1);
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
        // The 16 boxes of a stage (8 blocks x 2 column halves, 2 KB each) go out from lanes
        // 0-15, one each; a block past the keys the pair needs reads past the pool (zeros).
        const bool is_k = warp == kKLoadWarp;
        const CUtensorMap* map = is_k ? &tm_k : &tm_v;
        uint64_t* full = is_k ? bars->k_full : bars->v_full;
        uint64_t* empty = is_k ? bars->k_empty : bars->v_empty;
        uint8_t* ring = smem + (is_k ? kOffK : kOffV);
        const int nslots = is_k ? kKStages : kVStages;
        if (lane == 0) prefetch_tensormap(map);
        const uint64_t pol = l2_evict_last_policy();  // prefix blocks are shared across sequences
        const int32_t* bt = a.block_tables + (size_t)b * a.max_blocks;
        const int oob_row = a.num_blocks * a.num_kv_heads * kBlockSize;
        int c0 = 0;
        int cur = lane < nblk ? __ldg(bt + lane) : 0;
        int nxt = 32 + lane < nblk ? __ldg(bt + 32 + lane) : 0;
        const int box_t = lane >> 1, box_h = lane & 1;
        bool ok = true;
        int issued = 0;
        for (int j = 0; j < nstage && ok; ++j) {
            if (8 * j >= c0 + 32) {
                c0 += 32;
                cur = nxt;
                nxt = c0 + 32 + lane < nblk ? __ldg(bt + c0 + 32 + lane) : 0;
            }
            if (is_k && c0 + lane < nblk && (cur < 0 || cur >= a.num_blocks)) atomicOr(a.status, kDevOutOfRange);
            if (cur < 0 || cur >= a.num_blocks) cur = 0;
            const int lb = 8 * j + box_t;
            const int id = __shfl_sync(0xffffffffu, cur, (lb - c0) & 31);
            const int row = lb < nblk ? (id * a.num_kv_heads + kvh) * kBlockSize : oob_row;
            const int s = j % nslots;
            if (lane == 0) {
                if (j >= nslots) ok = mbar_wait(&empty[s], ((j / nslots) & 1) ^ 1);
                if (ok) mbar_arrive_expect_tx(&full[s], kTileBytes);
            }
            ok = __shfl_sync(0xffffffffu, ok, 0) != 0;
            if (ok) {
                if (lane < 16)
                    tma_load_2d(ring + s * kTileBytes + box_h * kHalfBytes + box_t * 2048, map, box_h * 64, row,
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
        // ------------------------------------------------------------ MMA issue (whole warp)
        // The warp runs the loop together and one elected lane issues, so every operand is
        // warp-uniform; waits give one verdict for the warp.  Operand descriptors are built
        // once; a tile, a stage or a k-step only moves the start address, which adds
        // (offset >> 4) to the low field (no carry: every shared address is below 2^18).
        constexpr uint32_t idesc_s = tc_idesc_bf16(kRows, kKeys, false);
        constexpr uint32_t idesc_h = tc_idesc_bf16(kRows, kKeys / 2, false);
        constexpr uint32_t idesc_o = tc_idesc_bf16(kRows, kD, true);
        const uint64_t qdesc0 = smem_desc_sw128(smem_u32(smem + kOffQ), 0, 1024);
        const uint64_t kdesc0 = smem_desc_sw128(smem_u32(smem + kOffK), 0, 1024);
        const uint64_t vdesc0 = smem_desc_sw128(smem_u32(smem + kOffV), kHalfBytes, 1024);
        // S_t = Q_t K(j)^T over keys [64 h0, 64 (h0 + nh)): N = 64 nh, into S_t's columns from 64 h0
        auto issue_qk = [&](int t, int j, int h0, int nh) {
            const uint64_t qd = qdesc0 + (uint64_t)((t * kTileBytes) >> 4);
            const uint64_t kd = kdesc0 + (uint64_t)(((j % kKStages) * kTileBytes + h0 * (kHalfBytes / 2)) >> 4);
            const uint32_t tm_s = tmem + t * kTmemTile + kTmemS + 64 * h0;
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk) {
                const uint64_t off = (uint64_t)(((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4);
                tc_mma_ew(tm_s, qd + off, kd + off, nh == 2 ? idesc_s : idesc_h, kk > 0 ? 1u : 0u);
            }
        };
        auto issue_pv = [&](int t, int j) {  // O_t += P_t V(j), P_t from tensor memory
            const uint64_t vd = vdesc0 + (uint64_t)(((j % kVStages) * kTileBytes) >> 4);
            const uint32_t tm_p = tmem + t * kTmemTile + kTmemS, tm_o = tmem + t * kTmemTile + kTmemO;
#pragma unroll
            for (int kk = 0; kk < kKeys / 16; ++kk)
                tc_mma_ts_ew(tm_o, tm_p + kk * 8, vd + (uint64_t)((kk * 16 * 128) >> 4), idesc_o,
                             (j > 0 || kk > 0) ? 1u : 0u);
            tc_commit_ew(&bars->o_done[t]);
        };
        bool ok = true;
#pragma unroll
        for (int t = 0; t < kTiles; ++t)
            if (ok && nst[t] > 0) ok = mbar_wait_warp(&bars->q_full[t], 0);
        if (ok) ok = mbar_wait_warp(&bars->k_full[0], 0);
        if (ok) {
            tc_fence_after();
#pragma unroll
            for (int t = 0; t < kTiles; ++t)
                if (nst[t] > 0) {
                    issue_qk(t, 0, 0, 2);
                    tc_commit_ew(&bars->s_full[t]);
                }
            tc_commit_ew(&bars->k_empty[0]);  // S(0) is K(0)'s only reader
        }
        for (int j = 0; j < nstage && ok; ++j) {
            bool v_ready = false, k_next = false;
#pragma unroll
            for (int t = 0; t < kTiles; ++t) {
                if (!ok || j >= nst[t]) continue;
                const bool more = j + 1 < nst[t];
                if (more) {
                    // keys 64-127 of S_t(j+1) once the softmax has read those columns of S_t(j)
                    ok = mbar_wait_warp(&bars->s_hi_free[t], j & 1);
                    if (ok && !k_next) {
                        ok = mbar_wait_warp(&bars->k_full[(j + 1) % kKStages], ((j + 1) / kKStages) & 1);
                        k_next = true;
                    }
                    if (!ok) break;
                    tc_fence_after();
                    issue_qk(t, j + 1, 1, 1);
                }
                ok = mbar_wait_warp(&bars->p_full[t], j & 1);
                if (ok && !v_ready) {
                    ok = mbar_wait_warp(&bars->v_full[j % kVStages], (j / kVStages) & 1);
                    v_ready = true;
                }
                if (!ok) break;
                tc_fence_after();
                issue_pv(t, j);
                if (more) {
                    issue_qk(t, j + 1, 0, 1);  // keys 0-63, over P_t(j): after P_t V(j) in issue order
                    tc_commit_ew(&bars->s_full[t]);
                }
            }
            if (!ok) break;
            tc_commit_ew(&bars->v_empty[j % kVStages]);
            if (k_next) tc_commit_ew(&bars->k_empty[(j + 1) % kKStages]);  // K(j+1)'s last reader is issued
        }
        // every MMA issued above has finished before the tensor memory is released
        tc_commit_ew(&bars->drain);
        if (!mbar_wait_warp(&bars->drain, 0)) ok = false;
        if (!ok && lane == 0) atomicOr(a.status, kDevTimeout);
    } else {
        // ------------------------------------------------------------ softmax: one row per thread
        const int t = warp >> 2;                    // query tile of this warpgroup
        const int r = threadIdx.x & (kRows - 1);    // TMEM lane r, MMA row r
        const int mt = t == 0 ? mtile[0] : mtile[1], nt = t == 0 ? nst[0] : nst[1];
        const int tok0 = mt * tpt;
        const int ntok = (mt >= 0 && tok0 < C) ? min(tpt, C - tok0) : 0;
        const bool whole = ntok == tpt;             // the tile is whole: Q comes in by TMA
        const bool valid = r < ntok * g;
        const int qi = r / g, h = r % g;
        const int pos = valid ? L - C + tok0 + qi : -1;  // causal limit of the row (inclusive)
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tm_row = tmem + lane_base + t * kTmemTile;
        uint8_t* qs = smem + kOffQ + t * kTileBytes;
        const int bar_id = 1 + t;                   // named barrier of this warpgroup
        if (nt > 0) {
            if (whole) {
                if (r == 0) {
                    prefetch_tensormap(&tm_q);
                    mbar_arrive_expect_tx(&bars->q_full[t], kTileBytes);
                    tma_load_3d(qs, &tm_q, 0, kvh * g, q0 + tok0, &bars->q_full[t]);
                    tma_load_3d(qs + kHalfBytes, &tm_q, 64, kvh * g, q0 + tok0, &bars->q_full[t]);
                }
            } else {
                // row by row into the same 128-byte swizzled layout (zeros past the chunk)
                const uint4* src = reinterpret_cast<const uint4*>(
                    a.q + ((size_t)(q0 + tok0 + qi) * a.num_heads + (size_t)kvh * g + h) * kD);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<uint4*>(qs + hh * kHalfBytes + swz128(r, c)) =
                            valid ? __ldg(src + hh * 8 + c) : make_uint4(0u, 0u, 0u, 0u);
                fence_proxy_async_smem();
                named_sync(bar_id, 128);
                if (r == 0) mbar_arrive(&bars->q_full[t]);
            }
        }
        const float sl = a.scale_log2;
        const float sl_abs = fabsf(sl);
        const bool neg = sl < 0.f;  // the row maximum of scale * s is scale * min(s) then
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
            const int k0 = j * kKeys;
            const int lim = pos - k0;  // keys c <= lim of this stage are visible to the row
            // Stages wholly below the diagonal (every row of the warp sees all 128 keys) after
            // the first take the streaming path; the first stage and the diagonal ones the
            // careful path.  Both write P (rounded to bf16, two keys per tensor-memory column,
            // the layout P V reads) into the first 64 columns of S_t, and add the rounded
            // values to the row sum, so the weights P V uses sum to l.
            const bool stream = j > 0 && __all_sync(0xffffffffu, lim >= kKeys - 1);
            // p = 2^(s scale log2(e) - m) for 4 keys: one packed multiply-add per two keys, the
            // special-function unit, bf16 packing; the packed words' values go to the sum
            auto p4 = [&](float v0, float v1, float v2, float v3, float nbase, bool m0, bool m1, bool m2, bool m3,
                          uint32_t& w0, uint32_t& w1, float (&ls)[4]) {
                float x0, x1, x2, x3;
                fma_x2(x0, x1, v0, v1, sl, sl, nbase, nbase);
                fma_x2(x2, x3, v2, v3, sl, sl, nbase, nbase);
                float q0 = fast_exp2(x0), q1 = fast_exp2(x1), q2 = fast_exp2(x2), q3 = fast_exp2(x3);
                q0 = m0 ? 0.f : q0;
                q1 = m1 ? 0.f : q1;
                q2 = m2 ? 0.f : q2;
                q3 = m3 ? 0.f : q3;
                w0 = pack_bf16x2(q0, q1);
                w1 = pack_bf16x2(q2, q3);
                add_x2(ls[0], ls[1], bf16_lo(w0), bf16_hi(w0));
                add_x2(ls[2], ls[3], bf16_lo(w1), bf16_hi(w1));
            };
            float ls[4] = {0.f, 0.f, 0.f, 0.f};
            if (stream) {
                // S in 32-key pieces, the next piece's load in flight; the row maximum of the
                // (sign-adjusted) scores is tracked beside the exponentials, which use the
                // running base.  P is held in registers until the stage's maximum is known: a
                // row whose maximum outgrows the base recomputes it from S with the new base
                // (computing it against the old one and rescaling would round it twice).
                float nbase = -m_used;
                float m8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) m8[e] = -INFINITY;
                uint32_t pw[kKeys / 2];
                auto piece = [&](int c, const uint32_t (&sr)[32], bool with_max) {
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        const float v0 = __uint_as_float(sr[e]), v1 = __uint_as_float(sr[e + 1]);
                        const float v2 = __uint_as_float(sr[e + 2]), v3 = __uint_as_float(sr[e + 3]);
                        if (with_max) {
                            const int ch = (e >> 2) & 3;
                            m8[2 * ch] = fmax3(m8[2 * ch], neg ? -v0 : v0, neg ? -v1 : v1);
                            m8[2 * ch + 1] = fmax3(m8[2 * ch + 1], neg ? -v2 : v2, neg ? -v3 : v3);
                        }
                        float x0, x1, x2, x3;
                        fma_x2(x0, x1, v0, v1, sl, sl, nbase, nbase);
                        fma_x2(x2, x3, v2, v3, sl, sl, nbase, nbase);
                        pw[(c * 32 + e) / 2] = pack_bf16x2(fast_exp2(x0), fast_exp2(x1));
                        pw[(c * 32 + e) / 2 + 1] = pack_bf16x2(fast_exp2(x2), fast_exp2(x3));
                    }
                };
                auto pass = [&](bool with_max) {
                    uint32_t sa[32], sb[32];
                    tmem_ld32_async(tm_row + kTmemS, sa);
                    tmem_wait_ld(sa);
                    tmem_ld32_async(tm_row + kTmemS + 32, sb);
                    piece(0, sa, with_max);
                    tmem_wait_ld(sb);
                    tmem_ld32_async(tm_row + kTmemS + 64, sa);
                    piece(1, sb, with_max);
                    tmem_wait_ld(sa);
                    tmem_ld32_async(tm_row + kTmemS + 96, sb);
                    piece(2, sa, with_max);
                    tmem_wait_ld(sb);
                    piece(3, sb, with_max);
                };
                pass(true);
                const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                       fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
                const float m_new = fmaxf(m_used, mx * sl_abs);
                const bool rebase = m_new > m_used + kRescaleThreshold;
                if (__any_sync(0xffffffffu, rebase)) {
                    // Rare: some row's maximum outgrew its base.  O_t is still (P_t V(j-1) was
                    // issued before S_t(j), whose commit covers it), so rescale it; then P again,
                    // every row against its own base (unchanged rows get the same bits).
                    const float alpha = rebase ? fast_exp2(m_used - m_new) : 1.f;
#pragma unroll 1
                    for (int c = 0; c < kD; c += 8) {
                        uint32_t o[8];
                        tmem_ld8(tm_row + kTmemO + c, o);
                        tmem_st8_nowait(tm_row + kTmemO + c, __float_as_uint(__uint_as_float(o[0]) * alpha),
                                        __float_as_uint(__uint_as_float(o[1]) * alpha),
                                        __float_as_uint(__uint_as_float(o[2]) * alpha),
                                        __float_as_uint(__uint_as_float(o[3]) * alpha),
                                        __float_as_uint(__uint_as_float(o[4]) * alpha),
                                        __float_as_uint(__uint_as_float(o[5]) * alpha),
                                        __float_as_uint(__uint_as_float(o[6]) * alpha),
                                        __float_as_uint(__uint_as_float(o[7]) * alpha));
                    }
                    tmem_wait_st();
                    if (rebase) {
                        l *= alpha;
                        m_used = m_new;
                    }
                    nbase = -m_used;
                    pass(false);
                }
                tc_fence_before();
                mbar_arrive(&bars->s_hi_free[t]);  // S_t's columns 64-127 are read
                // the row sum adds the rounded values P V uses; P goes over S_t's first half
#pragma unroll
                for (int w = 0; w < kKeys / 2; w += 2) {
                    add_x2(ls[0], ls[1], bf16_lo(pw[w]), bf16_hi(pw[w]));
                    add_x2(ls[2], ls[3], bf16_lo(pw[w + 1]), bf16_hi(pw[w + 1]));
                }
#pragma unroll
                for (int i = 0; i < kKeys / 16; ++i)
                    tmem_st8_nowait(tm_row + kTmemS + 8 * i, pw[8 * i], pw[8 * i + 1], pw[8 * i + 2], pw[8 * i + 3],
                                    pw[8 * i + 4], pw[8 * i + 5], pw[8 * i + 6], pw[8 * i + 7]);
                tmem_wait_st();
            } else {
                // Two passes over S in 32-key pieces: the maximum over the visible keys, then
                // the exponentials against the (re-based if need be) base.
                float m8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) m8[e] = -INFINITY;
                // per-key masking only where some row of the warp sees part of the stage
                const bool masked = !__all_sync(0xffffffffu, lim >= kKeys - 1);
                const int mlim = masked ? lim : kKeys;
                auto max_piece = [&](int c, const uint32_t (&sr)[32]) {
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        const int kb = c * 32 + e;
                        float a0 = __uint_as_float(sr[e]), a1 = __uint_as_float(sr[e + 1]);
                        float a2 = __uint_as_float(sr[e + 2]), a3 = __uint_as_float(sr[e + 3]);
                        a0 = kb > mlim ? -INFINITY : (neg ? -a0 : a0);
                        a1 = kb + 1 > mlim ? -INFINITY : (neg ? -a1 : a1);
                        a2 = kb + 2 > mlim ? -INFINITY : (neg ? -a2 : a2);
                        a3 = kb + 3 > mlim ? -INFINITY : (neg ? -a3 : a3);
                        const int ch = (e >> 2) & 3;
                        m8[2 * ch] = fmax3(m8[2 * ch], a0, a1);
                        m8[2 * ch + 1] = fmax3(m8[2 * ch + 1], a2, a3);
                    }
                };
                {
                    uint32_t sa[32], sb[32];
                    tmem_ld32_async(tm_row + kTmemS, sa);
                    tmem_wait_ld(sa);
                    tmem_ld32_async(tm_row + kTmemS + 32, sb);
                    max_piece(0, sa);
                    tmem_wait_ld(sb);
                    tmem_ld32_async(tm_row + kTmemS + 64, sa);
                    max_piece(1, sb);
                    tmem_wait_ld(sa);
                    tmem_ld32_async(tm_row + kTmemS + 96, sb);
                    max_piece(2, sa);
                    tmem_wait_ld(sb);
                    max_piece(3, sb);
                }
                const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                       fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
                const float mxs = mx == -INFINITY ? -INFINITY : mx * sl_abs;  // log2 units
                const float m_new = fmaxf(m_used, mxs);
                const bool rescale = m_new > m_used + kRescaleThreshold;  // always for the first visible key
                const float alpha = rescale && m_used != -INFINITY ? fast_exp2(m_used - m_new) : 0.f;
                if (__any_sync(0xffffffffu, rescale && m_used != -INFINITY)) {
                    // O_t is still: see above
                    const float f = rescale ? alpha : 1.f;
#pragma unroll 1
                    for (int c = 0; c < kD; c += 8) {
                        uint32_t o[8];
                        tmem_ld8(tm_row + kTmemO + c, o);
                        tmem_st8_nowait(tm_row + kTmemO + c, __float_as_uint(__uint_as_float(o[0]) * f),
                                        __float_as_uint(__uint_as_float(o[1]) * f),
                                        __float_as_uint(__uint_as_float(o[2]) * f),
                                        __float_as_uint(__uint_as_float(o[3]) * f),
                                        __float_as_uint(__uint_as_float(o[4]) * f),
                                        __float_as_uint(__uint_as_float(o[5]) * f),
                                        __float_as_uint(__uint_as_float(o[6]) * f),
                                        __float_as_uint(__uint_as_float(o[7]) * f));
                    }
                    tmem_wait_st();
                }
                if (rescale) {
                    l *= alpha;  // 0 when nothing was visible before
                    m_used = m_new;
                }
                const float nbase = m_used == -INFINITY ? 0.f : -m_used;
                auto exp_piece = [&](int c, const uint32_t (&sr)[32]) {
                    uint32_t w[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        const int kb = c * 32 + e;
                        p4(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1]), __uint_as_float(sr[e + 2]),
                           __uint_as_float(sr[e + 3]), nbase, kb > mlim, kb + 1 > mlim, kb + 2 > mlim, kb + 3 > mlim,
                           w[e / 2], w[e / 2 + 1], ls);
                    }
                    tmem_st8_nowait(tm_row + kTmemS + 16 * c, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
                    tmem_st8_nowait(tm_row + kTmemS + 16 * c + 8, w[8], w[9], w[10], w[11], w[12], w[13], w[14], w[15]);
                };
                uint32_t sa[32], sb[32];
                tmem_ld32_async(tm_row + kTmemS, sa);
                tmem_wait_ld(sa);
                tmem_ld32_async(tm_row + kTmemS + 32, sb);
                exp_piece(0, sa);
                tmem_wait_ld(sb);
                tmem_ld32_async(tm_row + kTmemS + 64, sa);
                exp_piece(1, sb);
                tmem_wait_ld(sa);
                tmem_ld32_async(tm_row + kTmemS + 96, sb);
                exp_piece(2, sa);
                tmem_wait_ld(sb);
                tc_fence_before();
                mbar_arrive(&bars->s_hi_free[t]);  // S_t's columns 64-127 are read
                exp_piece(3, sb);
                tmem_wait_st();
            }
            l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
            if (t == 0 && k0 + kKeys > L) {
                // keys at or past the sequence end: zero their V rows, whatever the slots hold
                // (P is 0 there, but 0 times a NaN left in a slot is NaN).  Once V(j) has landed,
                // its slot's previous readers have finished (the refill waited for them), and
                // both tiles' P V(j) are issued after tile 0's P(j) is complete.
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
                    *reinterpret_cast<uint4*>(vt + half * kHalfBytes + row * 128 + cc * 16) = make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
            }
            tc_fence_before();
            mbar_arrive(&bars->p_full[t]);
        }
        if (nt > 0) {
            if (ok) ok = !__any_sync(0xffffffffu, !mbar_wait(&bars->o_done[t], (nt - 1) & 1));
            // one verdict for the warpgroup, which then takes the same path through its barriers
            const bool all_ok = named_sync_all(bar_id, 128, ok);
            if (all_ok) {
                tc_fence_after();
                const float inv = l > 0.f ? 1.f / l : 0.f;
                // each thread stores its own row (256 contiguous bytes; the g rows of a query
                // are one contiguous run)
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

}  // namespace

cudaError_t launch_prefill_tc2(const PoolView& pool, const AttnArgs& a, cudaStream_t stream) {
    static OncePerDevice configured;
    const cudaError_t e = configured.run(
        [] { return cudaFuncSetAttribute(prefill_tc2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes); });
    if (e != cudaSuccess) return e;
    const int g = a.num_heads / pool.num_kv_heads;
    const int tpt = kRows / g;
    // q as (d, head, token) with one query tile per box; a whole tile never reaches past the
    // chunk rows, whose total is at most batch * max_chunk
    const long long tokens = (long long)a.batch * a.max_chunk;
    CUtensorMap tm_q;
    if (!rows_map(&tm_q, a.q, tokens, a.num_heads, kD, g, tpt)) return cudaErrorInvalidValue;
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
    t.scale_log2 = a.scale * kLog2e;
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
    return cudaLaunchKernelEx(&cfg, prefill_tc2_kernel, pool.tm_k, pool.tm_v, tm_q, t);
}

}  // namespace pa
