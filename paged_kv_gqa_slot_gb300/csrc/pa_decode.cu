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
// Four consumer warps take the split's blocks round-robin, each with its own running
// softmax; the CTA merges the four, and then
//   * pa_decode with one split writes bf16 O;
//   * pa_decode with S > 1 splits runs the S CTAs of a sequence/head as one thread-block
//     cluster and merges their partials through distributed shared memory (no
//     workspace, one launch) -- used when batch x kv heads is too small to fill the GPU;
//   * pa_decode_splitkv writes each partition's normalised O_p and lse_p to the caller's
//     workspace for pa_combine.
#include <algorithm>
#include <cstdlib>

#include <cooperative_groups.h>

#include "pa_block_attn.cuh"
#include "pa_internal.h"

namespace cg = cooperative_groups;

namespace pa {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;

template <int D>
struct DecodeShape {
    // each consumer warp owns the slots i with i % kConsumerWarps == warp, so it observes
    // every phase of its slots in order (what an mbarrier parity wait relies on)
    static constexpr int kStages = 8;
    static_assert(kStages % kConsumerWarps == 0, "slots must divide evenly among consumer warps");
    static constexpr int kRingBytes = kStages * KvTile<D>::kStageBytes;
    // epilogue scratch, overlaid on the ring once it is drained
    static constexpr int kWarpPartFloats = 32 + 16 * D;  // m[16], l[16], O[16][D]
    static constexpr int kCtaPartFloats = 32 + 16 * D;
    static constexpr int kEpiBytes = (kConsumerWarps * kWarpPartFloats + kCtaPartFloats) * 4;
    static constexpr int kDataBytes = kRingBytes > kEpiBytes ? kRingBytes : kEpiBytes;
    static constexpr int kSmemBytes = kDataBytes + 2 * kStages * 8 + 1024;
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
    float scale_log2;
};

template <int D, bool TWO_ROWS, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 3) decode_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                          const __grid_constant__ CUtensorMap tm_v,
                                                          const __grid_constant__ DecodeArgs a) {
    using Sh = DecodeShape<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Sh::kDataBytes);
    uint64_t* empty = full + Sh::kStages;

    const int split = blockIdx.x, nsplit = gridDim.x, kvh = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = a.group;

    int L = a.seq_lens[b];
    if (L < 0 || L > a.max_blocks * kBlockSize) {
        if (threadIdx.x == 0) atomicOr(a.status, kDevOutOfRange);
        L = L < 0 ? 0 : a.max_blocks * kBlockSize;
    }
    const int nb = (L + kBlockSize - 1) / kBlockSize;
    const int per = (nb + nsplit - 1) / nsplit;
    const int blk0 = split * per;
    const int n = max(0, min(per, nb - blk0));

    if (threadIdx.x == 0) {
        for (int s = 0; s < Sh::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        fence_mbar_init();
    }
    __syncthreads();

    constexpr int kC = Rows<TWO_ROWS>::kC;
    float o[D / 8][kC];
#pragma unroll
    for (int j = 0; j < D / 8; ++j)
#pragma unroll
        for (int c = 0; c < kC; ++c) o[j][c] = 0.f;
    RowState rs;
    rs.init();

    if (warp == kConsumerWarps) {
        if (lane == 0) {
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
        }
        produce_kv_blocks<D, Sh::kStages>(smem, full, empty, &tm_k, &tm_v,
                                          a.block_tables + (size_t)b * a.max_blocks + blk0, n, a.num_blocks,
                                          a.num_kv_heads, kvh, a.status, l2_evict_first_policy());
    } else {
        const int r0 = lane >> 2;
        const __nv_bfloat16* qg = a.q + ((size_t)b * a.num_heads + (size_t)kvh * g) * D;
        uint32_t qa[D / 16][Rows<TWO_ROWS>::kA];
        load_q_frags<D, TWO_ROWS>(qa, r0 < g ? qg + r0 * D : nullptr,
                                  (TWO_ROWS && r0 + 8 < g) ? qg + (r0 + 8) * D : nullptr);
        bool ok = true;
        for (int i = warp; i < n; i += kConsumerWarps) {
            const int st = i % Sh::kStages;
            ok = __all_sync(0xffffffffu, mbar_wait(&full[st], (i / Sh::kStages) & 1));
            if (!ok) break;
            uint8_t* kt = smem + st * KvTile<D>::kStageBytes;
            uint8_t* vt = kt + KvTile<D>::kTileBytes;
            const int valid = min(kBlockSize, L - (blk0 + i) * kBlockSize);
            block_step<D, TWO_ROWS>(smem_u32(kt), smem_u32(vt), qa, o, rs, valid, valid, valid, a.scale_log2);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
        }
        if (!ok && lane == 0) atomicOr(a.status, kDevTimeout);
        rs.l_a += __shfl_xor_sync(0xffffffffu, rs.l_a, 1);
        rs.l_a += __shfl_xor_sync(0xffffffffu, rs.l_a, 2);
        rs.l_b += __shfl_xor_sync(0xffffffffu, rs.l_b, 1);
        rs.l_b += __shfl_xor_sync(0xffffffffu, rs.l_b, 2);
    }
    __syncthreads();  // ring drained: every issued copy has landed and been consumed

    // ---- per-warp partials -> one CTA partial (unnormalised O, max m, sum l per row)
    float* part = reinterpret_cast<float*>(smem);
    float* cta = part + kConsumerWarps * Sh::kWarpPartFloats;  // m[16], l[16], O[16][D]
    if (warp < kConsumerWarps) {
        const int r0 = lane >> 2, c = (lane & 3) * 2;
        float* pm = part + warp * Sh::kWarpPartFloats;
        if ((lane & 3) == 0) {
            pm[r0] = rs.m_a;
            pm[16 + r0] = rs.l_a;
            if (TWO_ROWS) {
                pm[r0 + 8] = rs.m_b;
                pm[16 + r0 + 8] = rs.l_b;
            }
        }
        float* po = pm + 32;
#pragma unroll
        for (int j = 0; j < D / 8; ++j) {
            *reinterpret_cast<float2*>(po + r0 * D + j * 8 + c) = make_float2(o[j][0], o[j][1]);
            if constexpr (TWO_ROWS)
                *reinterpret_cast<float2*>(po + (r0 + 8) * D + j * 8 + c) = make_float2(o[j][2], o[j][3]);
        }
    }
    __syncthreads();
    const int E = g * D;
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

    if (SPLIT) {
        // partition `split` of nsplit: normalised O_p and natural-log lse_p
        for (int e = threadIdx.x; e < E; e += kThreads) {
            const int h = e / D, dd = e % D;
            const size_t row = ((size_t)b * a.num_heads + (size_t)kvh * g + h) * nsplit + split;
            const float den = cta[16 + h];
            a.ws_o[row * D + dd] = den > 0.f ? cta[32 + e] / den : 0.f;
            if (dd == 0) a.ws_lse[row] = den > 0.f ? (cta[h] + log2f(den)) * kLn2 : -INFINITY;
        }
        return;
    }
    __nv_bfloat16* outg = a.out + ((size_t)b * a.num_heads + (size_t)kvh * g) * D;
    if (nsplit == 1) {
        for (int e = threadIdx.x; e < E; e += kThreads) {
            const float den = cta[16 + e / D];
            outg[e] = __float2bfloat16_rn(den > 0.f ? cta[32 + e] / den : 0.f);
        }
        return;
    }
    // ---- cluster merge: CTA `rank` finalises a slice of the g x D outputs, reading every
    // CTA's partial through distributed shared memory (lane r reads CTA r).
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    const int rank = static_cast<int>(cluster.block_rank());
    const int slice = (E + nsplit - 1) / nsplit;
    const int e0 = rank * slice, e1 = min(E, e0 + slice);
    for (int e = e0 + warp; e < e1; e += kThreads / 32) {
        const int h = e / D;
        float mr = -INFINITY, lr = 0.f, orr = 0.f;
        if (lane < nsplit) {
            const float* rc = cluster.map_shared_rank(cta, lane);
            mr = rc[h];
            lr = rc[16 + h];
            orr = rc[32 + e];
        }
        const float M = warp_max(mr);
        const float wt = (mr != -INFINITY) ? fast_exp2(mr - M) : 0.f;
        const float num = warp_sum(wt * orr);
        const float den = warp_sum(wt * lr);
        if (lane == 0) outg[e] = __float2bfloat16_rn(den > 0.f ? num / den : 0.f);
    }
    cluster.sync();  // keep this CTA's partial alive until every reader is done
}

// out[r, :] = sum_p exp(lse_p - M) O_p / sum_p exp(lse_p - M), one warp per (seq, head).
template <int D>
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ ws_o,
                                                      const float* __restrict__ ws_lse, int rows, int P,
                                                      __nv_bfloat16* __restrict__ out) {
    const int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (r >= rows) return;
    constexpr int kPer = D / 32;
    const float* lse = ws_lse + (size_t)r * P;
    const float* op = ws_o + (size_t)r * P * D + lane * kPer;
    float M = -INFINITY;
    for (int p = lane; p < P; p += 32) M = fmaxf(M, lse[p]);
    M = warp_max(M);
    float acc[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) acc[j] = 0.f;
    float den = 0.f;
    if (M != -INFINITY) {
        for (int p = 0; p < P; ++p) {
            const float lp = lse[p];
            if (lp == -INFINITY) continue;
            const float w = fast_exp2((lp - M) * kLog2e);
            den += w;
            if (kPer == 4) {
                const float4 v = *reinterpret_cast<const float4*>(op + (size_t)p * D);
                acc[0] += w * v.x;
                acc[1] += w * v.y;
                acc[2] += w * v.z;
                acc[3] += w * v.w;
            } else {
                const float2 v = *reinterpret_cast<const float2*>(op + (size_t)p * D);
                acc[0] += w * v.x;
                acc[1] += w * v.y;
            }
        }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    __nv_bfloat16* dst = out + (size_t)r * D + lane * kPer;
#pragma unroll
    for (int j = 0; j < kPer; j += 2)
        *reinterpret_cast<__nv_bfloat162*>(dst + j) = __floats2bfloat162_rn(acc[j] * inv, acc[j + 1] * inv);
}

template <int D, bool TWO_ROWS, bool SPLIT>
cudaError_t launch_one(const PoolView& pool, const AttnArgs& a, int nsplit, cudaStream_t stream) {
    using Sh = DecodeShape<D>;
    auto kern = decode_kernel<D, TWO_ROWS, SPLIT>;
    static bool configured = false;  // per instantiation; attribute setting is idempotent
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::kSmemBytes);
        if (e != cudaSuccess) return e;
        if (!SPLIT) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess) return e;
        }
        configured = true;
    }
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

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(nsplit, pool.num_kv_heads, a.batch);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Sh::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (!SPLIT && nsplit > 1) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = nsplit;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kern, pool.tm_k, pool.tm_v, da);
}

template <bool SPLIT>
cudaError_t dispatch(const PoolView& pool, const AttnArgs& a, int nsplit, cudaStream_t stream) {
    const int g = a.num_heads / pool.num_kv_heads;
    if (pool.head_dim == 128)
        return g > 8 ? launch_one<128, true, SPLIT>(pool, a, nsplit, stream)
                     : launch_one<128, false, SPLIT>(pool, a, nsplit, stream);
    return g > 8 ? launch_one<64, true, SPLIT>(pool, a, nsplit, stream)
                 : launch_one<64, false, SPLIT>(pool, a, nsplit, stream);
}

int max_cluster_splits() {
    // Largest cluster the decode kernel can run with (16 needs the non-portable opt-in).
    static int cached = 0;
    if (cached) return cached;
    int best = 8;
    auto kern = decode_kernel<128, false, false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, DecodeShape<128>::kSmemBytes) ==
            cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(16, 1, 1);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = DecodeShape<128>::kSmemBytes;
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
    cached = best;
    return cached;
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
    int s = (2 * sms + items - 1) / items;  // aim for about two CTAs per SM
    s = std::min(s, max_cluster_splits());
    s = std::min(s, std::max(1, max_blocks / 4));  // at least ~4 blocks per split
    return std::max(1, s);
}

cudaError_t launch_decode(const PoolView& pool, const AttnArgs& a, cudaStream_t stream) {
    const int nsplit = decode_splits_for(a.batch, pool.num_kv_heads, a.max_blocks);
    return dispatch<false>(pool, a, nsplit, stream);
}

cudaError_t launch_decode_splitkv(const PoolView& pool, const AttnArgs& a, cudaStream_t stream) {
    return dispatch<true>(pool, a, a.num_partitions, stream);
}

cudaError_t launch_combine(const float* ws_o, const float* ws_lse, int batch, int num_heads, int head_dim,
                           int num_partitions, void* out, cudaStream_t stream) {
    const int rows = batch * num_heads;
    const int blocks = (rows * 32 + 255) / 256;
    auto* o = static_cast<__nv_bfloat16*>(out);
    if (head_dim == 128)
        combine_kernel<128><<<blocks, 256, 0, stream>>>(ws_o, ws_lse, rows, num_partitions, o);
    else
        combine_kernel<64><<<blocks, 256, 0, stream>>>(ws_o, ws_lse, rows, num_partitions, o);
    return cudaGetLastError();
}

}  // namespace pa
