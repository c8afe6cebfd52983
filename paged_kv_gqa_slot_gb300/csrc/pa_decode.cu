// pa_decode.cu -- paged GQA decode (one query token per sequence), its split-KV
// (flash-decoding) variant, and the log-sum-exp combine.
//
// Method: "Qwen3-4B / 8B / 32B", section "Architecture Notes" -- full attention with
// grouped-query attention (32 query heads over 8 KV heads, head dim 128; Qwen3-32B
// group 8) served from a paged KV cache; 16-token blocks per section "Qwen3-32B
// Serving Load" (21.4 GB = 5360 blocks).
//
// One CTA serves one (sequence, kv head, split): the g query heads of the group are the
// rows of one 16-row MMA tile, so each K/V byte is read from HBM once for all of them.
// Three consumer warps take the split's blocks round-robin, each with its own running
// softmax, fed by one TMA producer warp; the CTA merges the three, and then
//   * pa_decode with one split writes bf16 O;
//   * pa_decode with S > 1 splits runs the S CTAs of a sequence/head as one thread-block
//     cluster and merges their partials through distributed shared memory (no
//     workspace, one launch) -- used when batch x kv heads is too small to fill the GPU;
//   * pa_decode_splitkv writes each partition's normalised O_p and lse_p to the caller's
//     workspace for pa_combine.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <type_traits>

#include <cooperative_groups.h>

#include "pa_block_attn.cuh"
#include "pa_internal.h"

namespace cg = cooperative_groups;

namespace pa {
namespace {

// 3 consumer warps + 1 producer warp, 6 ring slots of one 16-token block each: at <= 128
// registers and ~50 KB of shared memory four CTAs fit on an SM, so a batch of 64
// sequences x 8 kv heads (512 CTAs) is resident in one wave on 152 SMs.
constexpr int kConsumerWarps = 3;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;

// The ring depth is chosen per launch (a multiple of the consumer warp count, so each
// warp owns the slots i with i % kConsumerWarps == warp and observes every phase of its
// slots in order, which an mbarrier parity wait relies on): shallow when many CTAs share
// an SM, deep when the grid is small and each CTA must keep more bytes in flight.
template <int D>
struct DecodeShape {
    static constexpr int kMinStages = 6;
    static constexpr int kMaxStages = 24;
    // epilogue scratch, overlaid on the ring once it is drained
    static constexpr int kWarpPartFloats = 32 + 16 * D;  // m[16], l[16], O[16][D]
    static constexpr int kCtaPartFloats = 32 + 16 * D;
    static constexpr int kEpiBytes = (kConsumerWarps * kWarpPartFloats + kCtaPartFloats) * 4;
    __host__ __device__ static constexpr int data_bytes(int stages) {
        return stages * KvTile<D>::kStageBytes > kEpiBytes ? stages * KvTile<D>::kStageBytes : kEpiBytes;
    }
    __host__ __device__ static constexpr int smem_bytes(int stages) { return data_bytes(stages) + 2 * stages * 8 + 1024; }
};

struct DecodeArgs {
    const __nv_bfloat16* q;
    const int32_t* block_tables;
    const int32_t* seq_lens;
    __nv_bfloat16* out;
    float* ws_o;
    float* ws_lse;
    unsigned* status;
    int max_blocks, num_heads, num_kv_heads, num_blocks, group;
    int stages;  // ring slots, a multiple of kConsumerWarps
    float scale_log2;
    int p_two_parts;  // |scale| sqrt(d) is large: P in two bf16 parts in every CTA
    const uint4* k_new;  // fused append (decode only): [B, Hkv, D] bf16, or null
    const uint4* v_new;
    const int64_t* slots;  // [B]
    const int32_t* cu_q_lens;  // multi-query: chunk of query tokens of each sequence [B+1]
    void* k_pool;  // the pool, for the fused append's row write
    void* v_pool;
};

// Where a multi-query chunk may keep P as one bf16 part: every row sees more than kFewKeys
// keys and |scale| sqrt(d) <= kTwoPartScale (the same bounds as the tensor-core prefill's).
constexpr int kFewKeys = 128;
constexpr float kTwoPartScale = 2.f;

template <int D, int NT, bool SPLIT, bool MQ>
__global__ void __launch_bounds__(kThreads, 4) decode_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                          const __grid_constant__ CUtensorMap tm_v,
                                                          const __grid_constant__ DecodeArgs a) {
    using Sh = DecodeShape<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int stages = a.stages;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Sh::data_bytes(stages));
    uint64_t* empty = full + stages;

    // The `sub` CTAs of a thread-block cluster (1 without one) share one result: a partition
    // of split-KV, or the whole sequence of a clustered decode.  x = result * sub + rank.
    uint32_t ncl;
    asm("mov.u32 %0, %%cluster_nctarank;" : "=r"(ncl));
    const int sub = static_cast<int>(ncl);
    const int parts = gridDim.x / sub;                      // partitions (split-KV) or 1
    const int unit = blockIdx.x / sub, sub_rank = blockIdx.x % sub;
    const int kvh = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = a.group;
    pdl_wait();
    // The producer loads its first 32 table entries now, in parallel with seq_lens, instead of
    // after it, which takes one dependent memory round trip off the first copy.  A CTA that
    // alone covers its sequence starts at block 0; a partition or cluster member's first block
    // depends on the length, so it guesses the length that fills the table (the common case of
    // a long context) and keeps the guess only if it gives the same first block.
    const bool whole = parts == 1 && sub == 1;
    int first_entry = 0, guess0 = 0;
    if (warp == kConsumerWarps) {
        if (!whole) {
            const int nb_g = a.max_blocks;
            const int per_ug = (nb_g + parts - 1) / parts;
            const int nu_g = max(0, min(per_ug, nb_g - unit * per_ug));
            const int per_g = (nu_g + sub - 1) / sub;
            guess0 = unit * per_ug + sub_rank * per_g;
        }
        if (guess0 + lane < a.max_blocks) first_entry = __ldg(a.block_tables + (size_t)b * a.max_blocks + guess0 + lane);
    }

    int L = a.seq_lens[b];
    if (L < 0 || L > a.max_blocks * kBlockSize) {
        if (threadIdx.x == 0) atomicOr(a.status, kDevOutOfRange);
        L = L < 0 ? 0 : a.max_blocks * kBlockSize;
    }
    // Multi-query (MQ): the last C tokens of the sequence are queries (a short causal chunk,
    // e.g. the draft tokens of a speculative-decoding verify); the MMA columns are its C x g
    // (query, head) rows.  Otherwise one query, the g heads.
    int C = 1, q0 = b;
    if (MQ) {
        q0 = a.cu_q_lens[b];
        C = a.cu_q_lens[b + 1] - q0;
        if (C < 0 || C > L || C * g > 8 * NT) {
            if (threadIdx.x == 0) atomicOr(a.status, kDevOutOfRange);
            C = 0;
        }
    }
    const int R = MQ ? C * g : g;  // columns in use
    const int nb = (L + kBlockSize - 1) / kBlockSize;
    // partition `unit` covers blocks [unit * per_u, (unit + 1) * per_u) (ceil(nb / parts) each);
    // its sub CTAs take equal consecutive shares of them
    const int per_u = (nb + parts - 1) / parts;
    const int u0 = unit * per_u;
    const int nu = max(0, min(per_u, nb - u0));
    const int per = (nu + sub - 1) / sub;
    const int blk0 = u0 + sub_rank * per;
    const int n = R == 0 ? 0 : max(0, min(per, nu - sub_rank * per));

    if (a.k_new != nullptr && warp == 0 && nb > 0 && blk0 + n == nb && n > 0) {
        // Fused append: the CTA that reads the sequence's last block first writes the new K/V
        // row of its kv head into the slot (token L-1 of the sequence), so the result equals an
        // append followed by the decode.  The row must land in that very slot; any other slot
        // is reported and not written.  The proxy fence and the barrier below order the write
        // before this CTA's TMA loads of the block.
        const int64_t slot = a.slots[b];
        if (slot >= 0) {
            const int lb = (L - 1) / kBlockSize, off = (L - 1) % kBlockSize;
            const int32_t blk = a.block_tables[(size_t)b * a.max_blocks + lb];
            const bool ok_slot = blk >= 0 && blk < a.num_blocks && slot == (int64_t)blk * kBlockSize + off;
            constexpr int kChunks = D * 2 / 16;  // 16-byte chunks of one row
            if (!ok_slot) {
                if (lane == 0) atomicOr(a.status, kDevOutOfRange);
            } else if (lane < 2 * kChunks) {
                const int c = lane % kChunks;
                const bool is_v = lane >= kChunks;
                const size_t src = ((size_t)b * a.num_kv_heads + kvh) * kChunks + c;
                const size_t dst = (((size_t)blk * a.num_kv_heads + kvh) * kBlockSize + off) * kChunks + c;
                uint4* pool = static_cast<uint4*>(is_v ? a.v_pool : a.k_pool);
                pool[dst] = __ldg((is_v ? a.v_new : a.k_new) + src);
                asm volatile("fence.proxy.async.global;" ::: "memory");
            }
        }
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        fence_mbar_init();
    }
    __syncthreads();

    float ot[NT][D / 16][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) ot[nt][mt][0] = ot[nt][mt][1] = ot[nt][mt][2] = ot[nt][mt][3] = 0.f;
    HeadState<NT> hs;
    hs.init();

    if (warp == kConsumerWarps) {
        if (lane == 0) {
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
        }
        produce_kv_blocks<D>(smem, stages, full, empty, &tm_k, &tm_v,
                             a.block_tables + (size_t)b * a.max_blocks + blk0, n, a.num_blocks, a.num_kv_heads, kvh,
                             a.status, l2_evict_first_policy(), first_entry, blk0 == guess0);
    } else {
        uint32_t qb[NT][D / 16][2];
        int colpos[NT][2];  // MQ: causal limit of this thread's two columns per n-tile
        if (MQ) {
            load_q_rows<D, NT>(qb, a.q, q0, C, g, a.num_heads, kvh);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int col = nt * 8 + (lane & 3) * 2 + j;
                    colpos[nt][j] = col < R ? L - C + col / g : -1;
                }
        } else {
            load_q_heads<D, NT>(qb, a.q + ((size_t)b * a.num_heads + (size_t)kvh * g) * D, g);
        }
        bool ok = true;
        auto consume = [&](auto two) {
            for (int i = warp; i < n; i += kConsumerWarps) {
                const int st = i % stages;
                ok = __all_sync(0xffffffffu, mbar_wait(&full[st], (i / stages) & 1));
                if (!ok) break;
                uint8_t* kt = smem + st * KvTile<D>::kStageBytes;
                uint8_t* vt = kt + KvTile<D>::kTileBytes;
                const int valid = min(kBlockSize, L - (blk0 + i) * kBlockSize);
                block_step_heads<D, NT, MQ, decltype(two)::value>(smem_u32(kt), smem_u32(vt), qb, ot, hs, valid,
                                                                  a.scale_log2, colpos, (blk0 + i) * kBlockSize);
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[st]);
            }
        };
        // P in two bf16 parts, except in a multi-query chunk whose every row sees more than
        // kFewKeys keys at the usual scale: there the one-part rounding averages away, and the
        // chunk's extra columns make the second P V product cost (the same CTA-uniform choice
        // in every CTA of the sequence).
        if (MQ && !a.p_two_parts && L - C + 1 > kFewKeys)
            consume(std::false_type{});
        else
            consume(std::true_type{});
        if (!ok && lane == 0) atomicOr(a.status, kDevTimeout);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float l = hs.l[nt][j];
                l += __shfl_xor_sync(0xffffffffu, l, 4);
                l += __shfl_xor_sync(0xffffffffu, l, 8);
                l += __shfl_xor_sync(0xffffffffu, l, 16);
                hs.l[nt][j] = l;
            }
    }
    __syncthreads();  // ring drained: every issued copy has landed and been consumed
    pdl_trigger();    // the next kernel may launch while this one merges and writes

    // ---- per-warp partials -> one CTA partial (unnormalised O, max m, sum l per head)
    float* part = reinterpret_cast<float*>(smem);
    float* cta = part + kConsumerWarps * Sh::kWarpPartFloats;  // m[16], l[16], O[16][D]
    if (warp < kConsumerWarps) {
        const int gid = lane >> 2, h0 = (lane & 3) * 2;
        float* pm = part + warp * Sh::kWarpPartFloats;
        float* po = pm + 32;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int ha = nt * 8 + h0;
            if (gid == 0) {
                pm[ha] = hs.m[nt][0];
                pm[ha + 1] = hs.m[nt][1];
                pm[16 + ha] = hs.l[nt][0];
                pm[16 + ha + 1] = hs.l[nt][1];
            }
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                const int d0 = mt * 16 + gid;
                po[ha * D + d0] = ot[nt][mt][0];
                po[(ha + 1) * D + d0] = ot[nt][mt][1];
                po[ha * D + d0 + 8] = ot[nt][mt][2];
                po[(ha + 1) * D + d0 + 8] = ot[nt][mt][3];
            }
        }
    }
    __syncthreads();
    const int E = R * D;
    for (int e = threadIdx.x; e < E; e += kThreads) {
        const int h = e / D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, part[w * Sh::kWarpPartFloats + h]);
        float num = 0.f, den = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float* pm = part + w * Sh::kWarpPartFloats;
                if (pm[h] == -INFINITY) continue;
                const float wt = fast_exp2(pm[h] - M);
                num += wt * pm[32 + e];
                den += wt * pm[16 + h];
            }
        }
        cta[32 + e] = num;
        if (e % D == 0) {
            cta[h] = M;
            cta[16 + h] = den;
        }
    }
    __syncthreads();

    if (SPLIT && sub == 1) {
        // partition `unit` of parts: normalised O_p and natural-log lse_p
        for (int e = threadIdx.x; e < E; e += kThreads) {
            const int h = e / D, dd = e % D;
            const size_t row = ((size_t)b * a.num_heads + (size_t)kvh * g + h) * parts + unit;
            const float den = cta[16 + h];
            a.ws_o[row * D + dd] = den > 0.f ? cta[32 + e] / den : 0.f;
            if (dd == 0) a.ws_lse[row] = den > 0.f ? (cta[h] + log2f(den)) * kLn2 : -INFINITY;
        }
        return;
    }
    // element e = row * D + d of this CTA's output -> its place in out
    auto out_at = [&](int e) -> __nv_bfloat16* {
        const int row = e / D;
        const size_t tok = MQ ? (size_t)q0 + row / g : (size_t)b;
        return a.out + (tok * a.num_heads + (size_t)kvh * g + (MQ ? row % g : row)) * D + e % D;
    };
    if (sub == 1) {
        for (int e = threadIdx.x; e < E; e += kThreads) {
            const float den = cta[16 + e / D];
            *out_at(e) = __float2bfloat16_rn(den > 0.f ? cta[32 + e] / den : 0.f);
        }
        return;
    }
    // ---- cluster merge: CTA `rank` finalises a slice of the g x D outputs from every CTA's
    // partial, read through distributed shared memory in two rounds: first all (m, l) pairs
    // (one remote load per thread), then the O slices as independent 16-byte loads.
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    float* wgt = part;  // [sub][16] merge weights, then den[16], max[16] (the warp partials are done)
    float* den = part + 16 * 16;
    float* mrow = part + 16 * 16 + 16;
    const int rank = static_cast<int>(cluster.block_rank());
    for (int t = threadIdx.x; t < sub * R; t += kThreads) {
        const int r = t / R, h = t % R;
        const float* rc = cluster.map_shared_rank(cta, r);
        wgt[r * 16 + h] = rc[h];
        wgt[256 + 32 + r * 16 + h] = rc[16 + h];
    }
    __syncthreads();
    if (threadIdx.x < R) {
        const int h = threadIdx.x;
        float M = -INFINITY;
        for (int r = 0; r < sub; ++r) M = fmaxf(M, wgt[r * 16 + h]);
        float dsum = 0.f;
        for (int r = 0; r < sub; ++r) {
            const float m = wgt[r * 16 + h];
            const float w = m == -INFINITY ? 0.f : fast_exp2(m - M);
            wgt[r * 16 + h] = w;
            dsum += w * wgt[256 + 32 + r * 16 + h];
        }
        den[h] = dsum;
        mrow[h] = M;
    }
    __syncthreads();
    const int quads = E / 4;
    const int qper = (quads + sub - 1) / sub;
    for (int qd = rank * qper + threadIdx.x; qd < min(quads, (rank + 1) * qper); qd += kThreads) {
        const int e = qd * 4, h = e / D;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int r = 0; r < sub; ++r) {
            const float w = wgt[r * 16 + h];
            const float4 v = *reinterpret_cast<const float4*>(cluster.map_shared_rank(cta, r) + 32 + e);
            acc.x += w * v.x;
            acc.y += w * v.y;
            acc.z += w * v.z;
            acc.w += w * v.w;
        }
        const float inv = den[h] > 0.f ? 1.f / den[h] : 0.f;
        if (SPLIT) {
            // the partition's normalised O_p slice and (once per row) its natural-log lse_p
            const size_t row = ((size_t)b * a.num_heads + (size_t)kvh * g + h) * parts + unit;
            float* wo = a.ws_o + row * D + e % D;
            wo[0] = acc.x * inv;
            wo[1] = acc.y * inv;
            wo[2] = acc.z * inv;
            wo[3] = acc.w * inv;
            if (e % D == 0) a.ws_lse[row] = den[h] > 0.f ? (mrow[h] + log2f(den[h])) * kLn2 : -INFINITY;
        } else {
            __nv_bfloat16* dst = out_at(e);  // 4 consecutive d of one row (D is a multiple of 4)
            *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
            *reinterpret_cast<__nv_bfloat162*>(dst + 2) = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
        }
    }
    cluster.sync();  // keep this CTA's partial alive until every reader is done
}

// out[r, :] = sum_p exp(lse_p - M) O_p / sum_p exp(lse_p - M) with M = max_p lse_p.
// One CTA of 8 warps per (sequence, head) row: every warp finds M from the row's lse values
// (one load per lane), then warp w accumulates partitions p = w, w+8, ... with lane l
// owning elements 4l..4l+3; the eight partial sums meet in shared memory.
constexpr int kCombineWarps = 8;

template <int D>
__global__ void __launch_bounds__(kCombineWarps * 32) combine_kernel(const float* __restrict__ ws_o,
                                                                     const float* __restrict__ ws_lse, int P,
                                                                     __nv_bfloat16* __restrict__ out) {
    constexpr int kQuads = D / 4;
    __shared__ float4 part[kCombineWarps][kQuads];
    __shared__ float dpart[kCombineWarps];
    const int r = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_trigger();
    pdl_wait();
    const float* lse = ws_lse + (size_t)r * P;
    const float4* op = reinterpret_cast<const float4*>(ws_o + (size_t)r * P * D) + lane;
    // This warp's first partitions (p = warp + 8k) are loaded together with the lse values:
    // the O slices do not depend on the maximum, so both round trips overlap.
    constexpr int kPre = 4;  // covers P <= 32 in one go
    float4 vpre[kPre];
    float lpre[kPre];
#pragma unroll
    for (int k = 0; k < kPre; ++k) {
        const int p = warp + k * kCombineWarps;
        const bool in = p < P && lane < kQuads;
        vpre[k] = in ? __ldg(op + (size_t)p * kQuads) : make_float4(0.f, 0.f, 0.f, 0.f);
        lpre[k] = p < P ? __ldg(lse + p) : -INFINITY;
    }
    float M = -INFINITY;
    for (int p = lane; p < P; p += 32) M = fmaxf(M, __ldg(lse + p));
    M = warp_max(M);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float den = 0.f;
    if (M != -INFINITY) {
        auto add = [&](float lp, const float4& v) {
            const float w = lp == -INFINITY ? 0.f : fast_exp2((lp - M) * kLog2e);  // empty partitions hold zeros
            den += w;
            acc.x += w * v.x;
            acc.y += w * v.y;
            acc.z += w * v.z;
            acc.w += w * v.w;
        };
#pragma unroll
        for (int k = 0; k < kPre; ++k) add(lpre[k], vpre[k]);
        for (int p = warp + kPre * kCombineWarps; p < P; p += kCombineWarps)
            add(__ldg(lse + p), lane < kQuads ? __ldg(op + (size_t)p * kQuads) : make_float4(0.f, 0.f, 0.f, 0.f));
    }
    if (lane < kQuads) part[warp][lane] = acc;
    if (lane == 0) dpart[warp] = den;
    __syncthreads();
    if (warp == 0 && lane < kQuads) {
        float4 t = part[0][lane];
        float dt = dpart[0];
#pragma unroll
        for (int w = 1; w < kCombineWarps; ++w) {
            t.x += part[w][lane].x;
            t.y += part[w][lane].y;
            t.z += part[w][lane].z;
            t.w += part[w][lane].w;
            dt += dpart[w];
        }
        const float inv = dt > 0.f ? 1.f / dt : 0.f;
        __nv_bfloat162* dst = reinterpret_cast<__nv_bfloat162*>(out + (size_t)r * D + lane * 4);
        dst[0] = __floats2bfloat162_rn(t.x * inv, t.y * inv);
        dst[1] = __floats2bfloat162_rn(t.z * inv, t.w * inv);
    }
}

// Ring slots per CTA.  Measured on GB300: 6 slots of 8 KB (three per consumer warp pair of
// K+V blocks) with four CTAs per SM beat deeper rings at every grid size tried -- a deeper
// ring costs residency (fewer CTAs per SM) more than it gains in bytes in flight.
template <int D>
int stages_for(int /*ctas*/) {
    using Sh = DecodeShape<D>;
    // PA_DECODE_STAGES=n forces the ring depth (rounded to the warp count, clamped), for tuning
    static const int forced = [] {
        const char* e = std::getenv("PA_DECODE_STAGES");
        return e ? std::atoi(e) : 0;
    }();
    if (forced > 0)
        return std::max(Sh::kMinStages, std::min(Sh::kMaxStages, (forced / kConsumerWarps) * kConsumerWarps));
    return D == 128 ? 6 : 12;
}

template <int D, int NT, bool SPLIT, bool MQ = false>
// grid_x CTAs per (sequence, kv head), in thread-block clusters of `cluster` (1: none)
cudaError_t launch_one(const PoolView& pool, const AttnArgs& a, int grid_x, int cluster, cudaStream_t stream) {
    using Sh = DecodeShape<D>;
    auto kern = decode_kernel<D, NT, SPLIT, MQ>;
    static OncePerDevice configured;  // per instantiation
    cudaError_t se = configured.run([&] {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             Sh::smem_bytes(Sh::kMaxStages));
        if (e != cudaSuccess) return e;
        // one carveout (all shared memory) for every ring depth, so launches of different
        // depths do not reconfigure the SMs between kernels
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e != cudaSuccess) return e;
        if (!SPLIT) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        return e;
    });
    if (se != cudaSuccess) return se;
    DecodeArgs da;
    da.q = static_cast<const __nv_bfloat16*>(a.q);
    da.block_tables = a.block_tables;
    da.seq_lens = a.seq_lens;
    da.out = static_cast<__nv_bfloat16*>(a.out);
    da.ws_o = a.ws_o;
    da.ws_lse = a.ws_lse;
    da.status = a.status;
    da.max_blocks = a.max_blocks;
    da.num_heads = a.num_heads;
    da.num_kv_heads = pool.num_kv_heads;
    da.num_blocks = pool.num_blocks;
    da.group = a.num_heads / pool.num_kv_heads;
    da.scale_log2 = a.scale * kLog2e;
    da.p_two_parts = std::fabs(a.scale) * std::sqrt((float)D) > kTwoPartScale ? 1 : 0;
    da.stages = stages_for<D>(grid_x * pool.num_kv_heads * a.batch);
    da.k_new = static_cast<const uint4*>(a.k_new);
    da.v_new = static_cast<const uint4*>(a.v_new);
    da.slots = a.slots;
    da.k_pool = pool.k;
    da.v_pool = pool.v;
    da.cu_q_lens = MQ ? a.cu_q_lens : nullptr;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid_x, pool.num_kv_heads, a.batch);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Sh::smem_bytes(da.stages);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2] = {pdl_attribute(), {}};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cluster > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = cluster;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelEx(&cfg, kern, pool.tile_k, pool.tile_v, da);
}

template <bool SPLIT>
cudaError_t dispatch(const PoolView& pool, const AttnArgs& a, int grid_x, int cluster, cudaStream_t stream) {
    const int g = a.num_heads / pool.num_kv_heads;
    if (pool.head_dim == 128)
        return g > 8 ? launch_one<128, 2, SPLIT, false>(pool, a, grid_x, cluster, stream)
                     : launch_one<128, 1, SPLIT, false>(pool, a, grid_x, cluster, stream);
    return g > 8 ? launch_one<64, 2, SPLIT, false>(pool, a, grid_x, cluster, stream)
                 : launch_one<64, 1, SPLIT, false>(pool, a, grid_x, cluster, stream);
}

int max_cluster_splits() {
    // Largest cluster the decode kernel can run with on the current device (16 needs the
    // non-portable opt-in), asked once per device.
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 8;
    if (const int c = cached[dev].load(std::memory_order_relaxed)) return c;
    int best = 8;
    auto kern = decode_kernel<128, 1, false, false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             DecodeShape<128>::smem_bytes(DecodeShape<128>::kMaxStages)) == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(16, 1, 1);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = DecodeShape<128>::smem_bytes(DecodeShape<128>::kMinStages);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 16;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int nclusters = 0;
        if (cudaOccupancyMaxActiveClusters(&nclusters, kern, &cfg) == cudaSuccess && nclusters > 0) best = 16;
    }
    cudaGetLastError();
    cached[dev].store(best, std::memory_order_relaxed);
    return best;
}

}  // namespace

int decode_splits_for(int batch, int num_kv_heads, int max_blocks) {
    // PA_DECODE_SPLITS=n forces the split count (clamped to the cluster limit), for tuning
    static const int forced = [] {
        const char* e = std::getenv("PA_DECODE_SPLITS");
        return e ? std::atoi(e) : 0;
    }();
    if (forced > 0) return std::min(forced, max_cluster_splits());
    const int items = batch * num_kv_heads;
    const int sms = device_info().num_sms;
    if (items >= sms) return 1;
    int s = std::max(1, (4 * sms) / items);  // fill one wave of four CTAs per SM
    s = std::min(s, max_cluster_splits());
    s = std::min(s, std::max(1, max_blocks / 4));  // at least ~4 blocks per split
    return std::max(1, s);
}

int splitkv_partitions_for(int batch, int num_kv_heads, int max_blocks) {
    // Partitions per (sequence, kv head) pair: as many as fill four fifths of one wave of four
    // CTAs per SM, up to 16; a thread-block cluster per partition takes the rest of the wave
    // when the partitions alone leave it at least half empty (splitkv_cluster_for).  Measured
    // on GB300 (152 SMs, 134 MB of KV, per call with the merge, means of 60 in-graph samples):
    // 4 x 8192 over 8 kv heads runs 28.4-28.7 us at P = 15 (480 CTAs), 28.9-29.2 at 14 and
    // 29.3-30.4 at 16 (512), about 30.5 at 10; P = 19 (608, the whole wave) ran 28.7 against
    // 27.2 at 16 in an earlier sweep, 24 and 32 slower still.  1 x 32768 runs its 16
    // partitions on 4-CTA clusters (512 CTAs); 13-15 partitions there measured within half a
    // microsecond of it, and 19 partitions on 4-CTA clusters (608 CTAs, which do not all fit
    // as clusters at once) 40.6 us.  At least 8 blocks per partition.
    const int items = std::max(1, batch * num_kv_heads);
    int p = std::max(1, std::min(16, (16 * device_info().num_sms) / (5 * items)));
    while (p > 1 && max_blocks / p < 8) --p;
    return p;
}

cudaError_t launch_decode(const PoolView& pool, const AttnArgs& a, cudaStream_t stream) {
    const int nsplit = decode_splits_for(a.batch, pool.num_kv_heads, a.max_blocks);
    return dispatch<false>(pool, a, nsplit, nsplit, stream);
}

bool decode_mq_supported(int group, int max_chunk) { return max_chunk >= 1 && (long long)max_chunk * group <= 16; }

cudaError_t launch_decode_mq(const PoolView& pool, const AttnArgs& a, cudaStream_t stream) {
    const int g = a.num_heads / pool.num_kv_heads;
    const int nsplit = decode_splits_for(a.batch, pool.num_kv_heads, a.max_blocks);
    const bool two = a.max_chunk * g > 8;
    if (pool.head_dim == 128)
        return two ? launch_one<128, 2, false, true>(pool, a, nsplit, nsplit, stream)
                   : launch_one<128, 1, false, true>(pool, a, nsplit, nsplit, stream);
    return two ? launch_one<64, 2, false, true>(pool, a, nsplit, nsplit, stream)
               : launch_one<64, 1, false, true>(pool, a, nsplit, nsplit, stream);
}

// CTAs per split-KV partition: when the partitions of all (sequence, kv head) pairs leave
// the GPU's four-per-SM wave at least half empty, each partition runs on a cluster of 2-4
// CTAs that split its blocks and merge on chip (the partition boundaries do not change).
int splitkv_cluster_for(int batch, int num_kv_heads, int num_partitions, int max_blocks) {
    static const int forced = [] {
        const char* e = std::getenv("PA_SPLITKV_CLUSTER");
        return e ? std::atoi(e) : 0;
    }();
    const long long ctas = (long long)std::max(1, batch) * num_kv_heads * num_partitions;
    int c = forced > 0 ? forced : (int)std::min<long long>(4, (4LL * device_info().num_sms) / ctas);
    c = std::max(1, std::min(c, 8));
    if (forced <= 0)
        while (c & (c - 1)) --c;  // a power of two: clusters of 3 place worse than of 2 or 4
    while (c > 1 && max_blocks / ((long long)num_partitions * c) < 4) --c;  // >= ~4 blocks per CTA
    return c;
}

cudaError_t launch_decode_splitkv(const PoolView& pool, const AttnArgs& a, cudaStream_t stream) {
    const int c = splitkv_cluster_for(a.batch, pool.num_kv_heads, a.num_partitions, a.max_blocks);
    return dispatch<true>(pool, a, a.num_partitions * c, c, stream);
}

cudaError_t launch_combine(const float* ws_o, const float* ws_lse, int batch, int num_heads, int head_dim,
                           int num_partitions, void* out, cudaStream_t stream) {
    const int rows = batch * num_heads;
    auto* o = static_cast<__nv_bfloat16*>(out);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(rows);
    cfg.blockDim = dim3(kCombineWarps * 32);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (head_dim == 128) return cudaLaunchKernelEx(&cfg, combine_kernel<128>, ws_o, ws_lse, num_partitions, o);
    return cudaLaunchKernelEx(&cfg, combine_kernel<64>, ws_o, ws_lse, num_partitions, o);
    return cudaGetLastError();
}

}  // namespace pa
