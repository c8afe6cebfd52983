// pa_prefill_tc.cu -- chunked prefill over a cached paged prefix on the 5th-generation
// tensor cores (tcgen05 MMA, accumulators in tensor memory).
//
// Method: "Qwen3-4B / 8B / 32B", sections "Warm Prefix-Cache TTFT" (a warm prefix hit:
// only the new chunk is computed, over the cached prefix) and "Architecture Notes" (GQA
// over a paged KV cache).  Chunk query i of sequence s sits at position L_s - C_s + i and
// attends causally to keys 0 .. L_s - C_s + i through the block table.
//
// One CTA per (128-row tile, kv head, sequence).  Rows are (query, head-of-the-group)
// pairs, row r = query r / g, head r % g, so one K/V tile serves all g heads.  Per stage of
// 64 keys (four 16-token pool blocks, loaded by TMA with 128-byte swizzling):
//   S[128 x 64]  = Q K^T      tcgen05.mma, M=128 N=64, Q (A) from TMEM, K (B) from smem
//   softmax      one thread per row reads its S row from TMEM, masks causally (only in
//                tiles that cross the diagonal), keeps an online max / sum in base 2 and
//                writes P (bf16, 128-byte swizzled) to shared memory
//   O[128 x 128] += P V       tcgen05.mma, M=128 N=128, P (A) and V (B) from smem
// TMEM columns: S [0,64), Q [64,128) (bf16 pairs), O [128,256).  The running max is
// re-based lazily: O is rescaled in TMEM only when a row's max grows by more than 2^8,
// which keeps every P <= 256 and makes rescales rare.
// K and V have separate rings (3 and 2 slots): a K slot is handed back as soon as its
// Q K^T has run, so the next K tiles load while the softmax and P V of this one proceed.
// Warp roles: 0-3 softmax (TMEM lanes 32w..32w+31), 4 MMA issue + TMEM owner, 5 TMA.
// 96 KB of shared memory and 256 TMEM columns per CTA: two CTAs share an SM, so one's
// softmax overlaps the other's MMAs.
// The c CTAs that hold consecutive query tiles of one (sequence, kv head) form a
// thread-block cluster and read the same K/V: each issues 1/c of every stage's TMA boxes
// with multicast to all members, and every member's MMA thread releases a stage to all of
// them (multicast commit), so a stage refills once the whole cluster is done with it.  A
// TMA stream of small (2 KB) boxes is limited by boxes per second per SM, not bytes, so
// this divides the limiting cost by c.  Members walk the union of their key tiles (a tile
// some other member needs is received and released without compute).
#include <algorithm>
#include <cstdlib>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kD = 128;
constexpr int kRows = 128;                      // MMA M
constexpr int kKeys = 64;                       // keys per stage (MMA N of S)
constexpr int kKStages = 3, kVStages = 2;
constexpr int kThreads = 192;
constexpr int kTmemCols = 256;
constexpr uint32_t kTmemS = 0, kTmemQ = 64, kTmemO = 128;
constexpr int kHalf = kKeys * 128;              // [64 keys][64 columns] bf16 = 8 KB
constexpr int kTileBytes = 2 * kHalf;           // one K or V tile (two column halves), 16 KB
constexpr int kOffK = 0;
constexpr int kOffV = kKStages * kTileBytes;
constexpr int kOffP = kOffV + kVStages * kTileBytes;   // [128 rows][64 keys] bf16 = 16 KB
constexpr int kBarOff = kOffP + kRows * 128;
constexpr int kSmemBytes = kBarOff + 256 + 1024;
constexpr float kLog2e = 1.44269504088896340736f;
constexpr float kRescaleThreshold = 8.f;        // log2 units

struct Bars {
    uint64_t k_full[kKStages], k_empty[kKStages], v_full[kVStages], v_empty[kVStages];
    uint64_t q_full, s_full, s_free, p_full, o_done, drain;
    uint32_t tmem_base;
};

struct TcArgs {
    const __nv_bfloat16* q;
    const int32_t* block_tables;
    const int32_t* seq_lens;
    const int32_t* cu_q_lens;
    __nv_bfloat16* out;
    unsigned* status;
    int max_blocks, num_heads, num_kv_heads, num_blocks, group;
    float scale_log2;
};

// Key tiles a query tile needs: keys [0, kmax) with kmax the last query's position + 1.
__device__ __forceinline__ int tile_key_count(int mt, int tpt, int C, int L) {
    const int tok0 = mt * tpt;
    if (mt < 0 || tok0 >= C) return 0;
    return L - C + tok0 + min(tpt, C - tok0);
}

__global__ void __launch_bounds__(kThreads, 2) prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                                 const __grid_constant__ CUtensorMap tm_v,
                                                                 const __grid_constant__ TcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Bars* bars = reinterpret_cast<Bars*>(smem + kBarOff);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t crank, cnum;
    asm("mov.u32 %0, %%cluster_ctarank;" : "=r"(crank));
    asm("mov.u32 %0, %%cluster_nctarank;" : "=r"(cnum));
    const int rank = static_cast<int>(crank), csize = static_cast<int>(cnum);
    const uint16_t all_mask = static_cast<uint16_t>((1u << csize) - 1u);
    const int mt = gridDim.x - 1 - blockIdx.x;  // the latest (longest) query tiles first
    const int kvh = blockIdx.y, b = blockIdx.z;
    const int g = a.group, tpt = kRows / g;
    const int q0 = a.cu_q_lens[b];
    const int C = a.cu_q_lens[b + 1] - q0;
    const int L = a.seq_lens[b];
    if (C < 0 || L < C || L > a.max_blocks * kBlockSize) {  // the same for the whole cluster
        if (threadIdx.x == 0 && mt == gridDim.x - 1 && kvh == 0) atomicOr(a.status, kDevOutOfRange);
        return;
    }
    const int tok0 = mt * tpt;
    const int ntok = tok0 < C ? min(tpt, C - tok0) : 0;
    const int rows_valid = ntok * g;
    const int pos0 = L - C + tok0;                          // position of the tile's first query
    const int ntiles = (tile_key_count(mt, tpt, C, L) + kKeys - 1) / kKeys;  // this CTA's tiles
    int kmax_cl = 0;                                        // keys any member of the cluster needs
    for (int r = 0; r < csize; ++r) kmax_cl = max(kmax_cl, tile_key_count(mt + rank - r, tpt, C, L));
    const int ntiles_cl = (kmax_cl + kKeys - 1) / kKeys;
    const int nblk = (kmax_cl + kBlockSize - 1) / kBlockSize;  // pool blocks read

    if (threadIdx.x == 0) {
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(&bars->k_full[s], 1);
            mbar_init(&bars->k_empty[s], csize);  // one release from every member
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(&bars->v_full[s], 1);
            mbar_init(&bars->v_empty[s], csize);
        }
        mbar_init(&bars->q_full, 128);
        mbar_init(&bars->s_full, 1);
        mbar_init(&bars->s_free, 128);
        mbar_init(&bars->p_full, 128);
        mbar_init(&bars->o_done, 1);
        mbar_init(&bars->drain, 1);
        fence_mbar_init();
    }
    if (warp == 4) {
        tmem_alloc(&bars->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    // every member's barriers exist before any multicast box or release can reach them
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 5) {
        // ------------------------------------------------------------ TMA producer
        // issue order K(0), K(1), V(0), K(2), V(1), ...: K runs one tile ahead of V.  Of the
        // 8 boxes of a stage (4 blocks x 2 column halves) this member issues those with
        // index % csize == rank, multicast to the whole cluster.
        if (lane == 0) {
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
        }
        const uint64_t pol = l2_evict_last_policy();  // prefix blocks are shared across sequences
        const int32_t* bt = a.block_tables + (size_t)b * a.max_blocks;
        const int oob_row = a.num_blocks * a.num_kv_heads * kBlockSize;  // past the pool: zero fill
        int c0 = 0;
        int cur = lane < nblk ? __ldg(bt + lane) : 0;
        int nxt = 32 + lane < nblk ? __ldg(bt + 32 + lane) : 0;
        auto tile_rows = [&](int j, int (&rows)[4]) {
            if (4 * j >= c0 + 32) {
                c0 += 32;
                cur = nxt;
                nxt = c0 + 32 + lane < nblk ? __ldg(bt + c0 + 32 + lane) : 0;
            }
            if (c0 + lane < nblk && (cur < 0 || cur >= a.num_blocks)) {
                atomicOr(a.status, kDevOutOfRange);
                cur = 0;
            }
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int lb = 4 * j + t;
                const int id = __shfl_sync(0xffffffffu, cur, (lb - c0) & 31);
                rows[t] = lb < nblk ? (id * a.num_kv_heads + kvh) * kBlockSize : oob_row;
            }
        };
        const bool my_box = lane < 8 && (lane % csize) == rank;
        bool ok = true;
        int k_issued = 0, v_issued = 0;
        int rows_k[4], rows_v[4];
        for (int step = 0; step <= ntiles_cl && ok; ++step) {
            if (step < ntiles_cl) {
                tile_rows(step, rows_k);
                const int s = step % kKStages;
                if (lane == 0) {
                    if (step >= kKStages) ok = mbar_wait(&bars->k_empty[s], ((step / kKStages) & 1) ^ 1);
                    if (ok) mbar_arrive_expect_tx(&bars->k_full[s], kTileBytes);
                }
                ok = __shfl_sync(0xffffffffu, ok, 0) != 0;
                if (ok) {
                    if (my_box) {
                        const int t = lane >> 1, h = lane & 1;
                        const int row = t == 0 ? rows_k[0] : t == 1 ? rows_k[1] : t == 2 ? rows_k[2] : rows_k[3];
                        tma_load_2d_mc(smem + kOffK + s * kTileBytes + h * kHalf + t * 2048, &tm_k, h * 64, row,
                                       &bars->k_full[s], all_mask, pol);
                    }
                    ++k_issued;
                }
            }
            if (ok && step > 0) {
                const int j = step - 1, s = j % kVStages;
                if (lane == 0) {
                    if (j >= kVStages) ok = mbar_wait(&bars->v_empty[s], ((j / kVStages) & 1) ^ 1);
                    if (ok) mbar_arrive_expect_tx(&bars->v_full[s], kTileBytes);
                }
                ok = __shfl_sync(0xffffffffu, ok, 0) != 0;
                if (ok) {
                    if (my_box) {
                        const int t = lane >> 1, h = lane & 1;
                        const int row = t == 0 ? rows_v[0] : t == 1 ? rows_v[1] : t == 2 ? rows_v[2] : rows_v[3];
                        tma_load_2d_mc(smem + kOffV + s * kTileBytes + h * kHalf + t * 2048, &tm_v, h * 64, row,
                                       &bars->v_full[s], all_mask, pol);
                    }
                    ++v_issued;
                }
            }
#pragma unroll
            for (int t = 0; t < 4; ++t) rows_v[t] = rows_k[t];
        }
        if (lane == 0) {
            // Before the CTA may leave: every stage armed here has been filled (by every
            // member's boxes), and every member has released it (so no release can still be
            // on its way to this CTA's barriers).
            for (int j = max(0, k_issued - kKStages); j < k_issued; ++j) {
                if (!mbar_wait(&bars->k_full[j % kKStages], (j / kKStages) & 1)) ok = false;
                if (!mbar_wait(&bars->k_empty[j % kKStages], (j / kKStages) & 1)) ok = false;
            }
            for (int j = max(0, v_issued - kVStages); j < v_issued; ++j) {
                if (!mbar_wait(&bars->v_full[j % kVStages], (j / kVStages) & 1)) ok = false;
                if (!mbar_wait(&bars->v_empty[j % kVStages], (j / kVStages) & 1)) ok = false;
            }
            if (!ok) atomicOr(a.status, kDevTimeout);
        }
    } else if (warp == 4) {
        // ------------------------------------------------------------ MMA issue (one thread)
        if (lane == 0) {
            constexpr uint32_t idesc_s = tc_idesc_bf16(kRows, kKeys, false);
            constexpr uint32_t idesc_o = tc_idesc_bf16(kRows, kD, true);
            const uint32_t p_s = smem_u32(smem + kOffP);
            bool ok = mbar_wait(&bars->q_full, 0);
            for (int j = 0; j <= ntiles_cl && ok; ++j) {
                if (j < ntiles_cl) {
                    const int s = j % kKStages;
                    ok = mbar_wait(&bars->k_full[s], (j / kKStages) & 1);
                    if (ok && j < ntiles) {
                        if (j > 0) ok = mbar_wait(&bars->s_free, (j - 1) & 1);
                        if (!ok) break;
                        tc_fence_after();
                        const uint32_t k_s = smem_u32(smem + kOffK + s * kTileBytes);
#pragma unroll
                        for (int kk = 0; kk < kD / 16; ++kk) {
                            const uint64_t bd = smem_desc_sw128(k_s + (kk >> 2) * kHalf + (kk & 3) * 32, 0, 1024);
                            tc_mma_ts(tmem + kTmemS, tmem + kTmemQ + kk * 8, bd, idesc_s, kk > 0 ? 1u : 0u);
                        }
                        tc_commit(&bars->s_full);
                    }
                    if (!ok) break;
                    tc_commit_mc(&bars->k_empty[s], all_mask);  // release the K slot cluster-wide
                }
                if (j > 0) {
                    const int jp = j - 1, s = jp % kVStages;
                    ok = mbar_wait(&bars->v_full[s], (jp / kVStages) & 1);
                    if (ok && jp < ntiles) {
                        ok = mbar_wait(&bars->p_full, jp & 1);
                        if (!ok) break;
                        tc_fence_after();
                        const uint32_t v_s = smem_u32(smem + kOffV + s * kTileBytes);
#pragma unroll
                        for (int ks = 0; ks < kKeys / 16; ++ks) {
                            const uint64_t ad = smem_desc_sw128(p_s + ks * 32, 0, 1024);
                            const uint64_t bd = smem_desc_sw128(v_s + ks * 16 * 128, kHalf, 1024);
                            tc_mma(tmem + kTmemO, ad, bd, idesc_o, (jp > 0 || ks > 0) ? 1u : 0u);
                        }
                        tc_commit(&bars->o_done);
                    }
                    if (!ok) break;
                    tc_commit_mc(&bars->v_empty[s], all_mask);
                }
            }
            // every MMA issued above has finished before the tensor memory is released
            tc_commit(&bars->drain);
            if (!mbar_wait(&bars->drain, 0)) ok = false;
            if (!ok) atomicOr(a.status, kDevTimeout);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax: one row per thread
        const int r = threadIdx.x;  // TMEM lane r, MMA row r
        const bool valid = r < rows_valid;
        const int qi = r / g, h = r % g;
        const int pos = valid ? pos0 + qi : -1;  // causal limit of the row (inclusive)
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        {
            // Q row -> TMEM columns [64, 128) as bf16 pairs (zeros for rows past the chunk)
            const uint4* src = reinterpret_cast<const uint4*>(
                a.q + ((size_t)(q0 + tok0 + qi) * a.num_heads + (size_t)kvh * g + h) * kD);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t w[32];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 v = valid ? __ldg(src + half * 8 + c) : make_uint4(0u, 0u, 0u, 0u);
                    w[4 * c] = v.x;
                    w[4 * c + 1] = v.y;
                    w[4 * c + 2] = v.z;
                    w[4 * c + 3] = v.w;
                }
                tmem_st32(tmem + lane_base + kTmemQ + half * 32, w);
            }
            tc_fence_before();
            mbar_arrive(&bars->q_full);
        }
        uint8_t* prow = smem + kOffP;
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < ntiles; ++j) {
            if (!mbar_wait(&bars->s_full, j & 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sr[2][32];
            tmem_ld32(tmem + lane_base + kTmemS, sr[0]);
            tmem_ld32(tmem + lane_base + kTmemS + 32, sr[1]);
            tc_fence_before();
            mbar_arrive(&bars->s_free);

            const int k0 = j * kKeys;
            const bool need_mask = k0 + kKeys - 1 > pos;
            float x[kKeys];
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < kKeys; ++c) {
                const float v = __uint_as_float(sr[c >> 5][c & 31]) * a.scale_log2;
                x[c] = (need_mask && k0 + c > pos) ? -INFINITY : v;
                mx = fmaxf(mx, x[c]);
            }
            const float m_new = fmaxf(m_used, mx);
            const bool rescale = m_new > m_used + kRescaleThreshold;  // always for the first visible key
            if (j > 0) {
                // PV(j-1) has finished: O is stable and the P buffer is free (every phase, in order)
                if (!mbar_wait(&bars->o_done, (j - 1) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
            }
            if (rescale) {
                const float alpha = fast_exp2(m_used - m_new);
                if (m_used != -INFINITY) {
#pragma unroll
                    for (int c = 0; c < kD; c += 32) {
                        uint32_t o[32];
                        tmem_ld32(tmem + lane_base + kTmemO + c, o);
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st32(tmem + lane_base + kTmemO + c, o);
                    }
                }
                l *= alpha;
                m_used = m_new;
            }
            const float base = m_used == -INFINITY ? 0.f : m_used;
            float lsum = 0.f;
#pragma unroll
            for (int cc = 0; cc < kKeys / 8; ++cc) {
                float p[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    p[e] = fast_exp2(x[cc * 8 + e] - base);
                    lsum += p[e];
                }
                uint4 v;
                v.x = pack_bf16x2(p[0], p[1]);
                v.y = pack_bf16x2(p[2], p[3]);
                v.z = pack_bf16x2(p[4], p[5]);
                v.w = pack_bf16x2(p[6], p[7]);
                *reinterpret_cast<uint4*>(prow + swz128(r, cc)) = v;
            }
            l += lsum;
            if (k0 + kKeys > L) {
                // keys at or past the sequence end: zero their V rows, whatever the slots hold.
                // V(j) has landed: PV(j-2), the previous user of this slot, finished before
                // PV(j-1), so only this phase of the slot's barrier can be pending.  (The other
                // members need these rows zeroed too and zero them themselves: every member
                // that computes tile j reaches this point before releasing the slot.)
                const int s = j % kVStages;
                if (!mbar_wait(&bars->v_full[s], (j / kVStages) & 1)) {
                    ok = false;
                    break;
                }
                uint8_t* vt = smem + kOffV + s * kTileBytes;
                const int z0 = max(0, L - k0);
                const int nchunks = (kKeys - z0) * 16;  // 16-byte chunks over both column halves
                for (int c = r; c < nchunks; c += 128) {
                    const int row = z0 + (c >> 4), half = (c >> 3) & 1, cc = c & 7;
                    *reinterpret_cast<uint4*>(vt + half * kHalf + row * 128 + cc * 16) = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bars->p_full);
        }
        if (ok && ntiles > 0) ok = mbar_wait(&bars->o_done, (ntiles - 1) & 1);
        if (ok && ntiles > 0) {
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            __nv_bfloat16* dst = a.out + ((size_t)(q0 + tok0 + qi) * a.num_heads + (size_t)kvh * g + h) * kD;
#pragma unroll
            for (int c = 0; c < kD; c += 32) {
                uint32_t o[32];
                tmem_ld32(tmem + lane_base + kTmemO + c, o);
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
    if (warp == 4) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    // no member leaves while another may still multicast into its memory or release to it
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

}  // namespace

bool prefill_tc_supported(int head_dim, int group) {
    if (head_dim != kD || group <= 0 || group > kRows || kRows % group != 0) return false;
    static const bool disabled = [] {
        const char* e = std::getenv("PA_PREFILL_IMPL");
        return e && e[0] == 'm';  // "mma": the warp-MMA kernel, for A/B comparisons
    }();
    return !disabled;
}

cudaError_t launch_prefill_tc(const PoolView& pool, const AttnArgs& a, cudaStream_t stream) {
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        configured = true;
    }
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
    t.scale_log2 = a.scale * kLog2e;
    const int tpt = kRows / t.group;
    const int tiles = std::max(1, (a.max_chunk + tpt - 1) / tpt);
    // cluster over consecutive query tiles of one (sequence, kv head): up to 4 members
    static const int forced = [] {
        const char* e = std::getenv("PA_PREFILL_CLUSTER");
        return e ? std::atoi(e) : 0;
    }();
    int cs = forced > 0 ? forced : 4;
    cs = std::max(1, std::min(cs, 8));
    while (cs > 1 && cs > tiles) cs >>= 1;
    const int gx = (tiles + cs - 1) / cs * cs;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(gx, pool.num_kv_heads, a.batch);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, prefill_tc_kernel, pool.tm_k, pool.tm_v, t);
}

}  // namespace pa
