// pa_prefill.cu -- chunked prefill over a cached paged prefix (warp-MMA kernel, used for the
// shapes the tcgen05 kernel in pa_prefill_tc.cu does not take: head_dim 64, or a group size
// that does not divide 128).
//
// Method: "Qwen3-4B / 8B / 32B", sections "Warm Prefix-Cache TTFT" (most of a prompt
// is a warm prefix-cache hit; only the new chunk is computed) and "Architecture Notes"
// (GQA over a paged KV cache).  Query i of sequence s's chunk of C_s tokens sits at
// position L_s - C_s + i (seq_lens counts the chunk, whose K/V the append has already
// written) and attends causally to keys 0 .. L_s - C_s + i through the block table.
//
// Work unit: one CTA per (128-row tile, kv head, sequence), where the rows are the
// chunk's (query, head-of-the-group) pairs -- row r is query r / g, head r % g -- so
// every K/V tile read from L2 serves all g heads of the group.  Eight consumer warps own
// 16 rows each and all consume every block; one producer warp streams the blocks
// [0, keys needed by the tile's last query) through TMA.  A warp skips the MMAs of a
// block that lies wholly past its last row's causal limit, so the diagonal costs only
// the masking of the blocks it straddles.
#include <algorithm>
#include <cstdlib>

#include "pa_block_attn.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kWarps = 8;  // consumer warps
constexpr int kThreads = (kWarps + 1) * 32;
constexpr int kRows = kWarps * 16;  // (query, head) rows per CTA
constexpr float kLog2e = 1.44269504088896340736f;

template <int D>
struct PrefillShape {
    static constexpr int kStages = D == 128 ? 8 : 12;
    static constexpr int kRingBytes = kStages * KvTile<D>::kStageBytes;
    static constexpr int kSmemBytes = kRingBytes + 2 * kStages * 8 + 1024;
};

struct PrefillArgs {
    const __nv_bfloat16* q;
    const int32_t* block_tables;
    const int32_t* seq_lens;
    const int32_t* cu_q_lens;
    __nv_bfloat16* out;
    unsigned* status;
    int max_blocks, num_heads, num_kv_heads, num_blocks, group;
    float scale_log2;
};

template <int D>
__global__ void __launch_bounds__(kThreads) prefill_mma_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                               const __grid_constant__ CUtensorMap tm_v,
                                                               const __grid_constant__ PrefillArgs a) {
    using Sh = PrefillShape<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Sh::kRingBytes);
    uint64_t* empty = full + Sh::kStages;

    const int mt = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_trigger();
    pdl_wait();
    const int g = a.group;
    const int q0 = a.cu_q_lens[b];
    const int C = a.cu_q_lens[b + 1] - q0;
    const int L = a.seq_lens[b];
    if (C < 0 || L < C || L > a.max_blocks * kBlockSize) {
        if (threadIdx.x == 0 && mt == 0 && kvh == 0) atomicOr(a.status, kDevOutOfRange);
        return;
    }
    const int rows = C * g;
    const int row0 = mt * kRows;
    // a chunk longer than max_chunk would leave rows past the grid unwritten: reported
    if (mt == 0 && kvh == 0 && threadIdx.x == 0 && (long long)(rows + kRows - 1) / kRows > gridDim.x)
        atomicOr(a.status, kDevOutOfRange);
    if (row0 >= rows) return;  // this sequence's chunk is shorter than the grid allows
    const int last_row = min(rows, row0 + kRows) - 1;
    const int kmax = L - C + last_row / g + 1;  // keys the tile's last query sees
    const int nb = (kmax + kBlockSize - 1) / kBlockSize;

    if (threadIdx.x == 0) {
        for (int s = 0; s < Sh::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kWarps) {
        if (lane == 0) {
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
        }
        // the prefix blocks are shared by every sequence of a prefix-cache hit: keep them in L2
        produce_kv_blocks<D>(smem, Sh::kStages, full, empty, &tm_k, &tm_v, a.block_tables + (size_t)b * a.max_blocks,
                                          nb, a.num_blocks, a.num_kv_heads, kvh, a.status, l2_evict_last_policy());
        return;
    }

    const int r0 = lane >> 2;
    const int ra = row0 + warp * 16 + r0, rb = ra + 8;
    const bool va = ra < rows, vb = rb < rows;
    const int pos_a = va ? L - C + ra / g : -1;  // causal limit (inclusive) of each row
    const int pos_b = vb ? L - C + rb / g : -1;
    const int wfirst = row0 + warp * 16;
    const bool warp_active = wfirst < rows;
    const int wpos_max = warp_active ? L - C + (min(rows - 1, wfirst + 15)) / g : -1;

    auto row_ptr = [&](int r) -> const __nv_bfloat16* {
        return a.q + ((size_t)(q0 + r / g) * a.num_heads + (size_t)kvh * g + r % g) * D;
    };
    uint32_t qa[D / 16][4];
    load_q_frags<D, true>(qa, va ? row_ptr(ra) : nullptr, vb ? row_ptr(rb) : nullptr);
    float o[D / 8][4];
#pragma unroll
    for (int j = 0; j < D / 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    RowState rs;
    rs.init();

    bool ok = true;
    for (int i = 0; i < nb; ++i) {
        const int st = i % Sh::kStages;
        const int tok0 = i * kBlockSize;
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&full[st], (i / Sh::kStages) & 1));
        if (ok && warp_active && tok0 <= wpos_max) {
            uint8_t* kt = smem + st * KvTile<D>::kStageBytes;
            uint8_t* vt = kt + KvTile<D>::kTileBytes;
            block_step<D, true>(smem_u32(kt), smem_u32(vt), qa, o, rs, pos_a - tok0 + 1, pos_b - tok0 + 1,
                                L - tok0, a.scale_log2);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
    }
    if (!ok && lane == 0) atomicOr(a.status, kDevTimeout);
    rs.l_a += __shfl_xor_sync(0xffffffffu, rs.l_a, 1);
    rs.l_a += __shfl_xor_sync(0xffffffffu, rs.l_a, 2);
    rs.l_b += __shfl_xor_sync(0xffffffffu, rs.l_b, 1);
    rs.l_b += __shfl_xor_sync(0xffffffffu, rs.l_b, 2);

    const int c = (lane & 3) * 2;
    if (va) {
        const float inv = rs.l_a > 0.f ? 1.f / rs.l_a : 0.f;
        __nv_bfloat16* dst = a.out + ((size_t)(q0 + ra / g) * a.num_heads + (size_t)kvh * g + ra % g) * D + c;
#pragma unroll
        for (int j = 0; j < D / 8; ++j)
            *reinterpret_cast<__nv_bfloat162*>(dst + j * 8) = __floats2bfloat162_rn(o[j][0] * inv, o[j][1] * inv);
    }
    if (vb) {
        const float inv = rs.l_b > 0.f ? 1.f / rs.l_b : 0.f;
        __nv_bfloat16* dst = a.out + ((size_t)(q0 + rb / g) * a.num_heads + (size_t)kvh * g + rb % g) * D + c;
#pragma unroll
        for (int j = 0; j < D / 8; ++j)
            *reinterpret_cast<__nv_bfloat162*>(dst + j * 8) = __floats2bfloat162_rn(o[j][2] * inv, o[j][3] * inv);
    }
}

template <int D>
cudaError_t launch_mma(const PoolView& pool, const AttnArgs& a, cudaStream_t stream) {
    using Sh = PrefillShape<D>;
    auto kern = prefill_mma_kernel<D>;
    static OncePerDevice configured;
    cudaError_t e = configured.run(
        [&] { return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::kSmemBytes); });
    if (e != cudaSuccess) return e;
    PrefillArgs pa_;
    pa_.q = static_cast<const __nv_bfloat16*>(a.q);
    pa_.block_tables = a.block_tables;
    pa_.seq_lens = a.seq_lens;
    pa_.cu_q_lens = a.cu_q_lens;
    pa_.out = static_cast<__nv_bfloat16*>(a.out);
    pa_.status = a.status;
    pa_.max_blocks = a.max_blocks;
    pa_.num_heads = a.num_heads;
    pa_.num_kv_heads = pool.num_kv_heads;
    pa_.num_blocks = pool.num_blocks;
    pa_.group = a.num_heads / pool.num_kv_heads;
    pa_.scale_log2 = a.scale * kLog2e;
    const long long rows = (long long)a.max_chunk * pa_.group;
    const int tiles = static_cast<int>((rows + kRows - 1) / kRows);
    dim3 grid(std::max(1, tiles), pool.num_kv_heads, a.batch);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Sh::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, pool.tile_k, pool.tile_v, pa_);
}

}  // namespace

cudaError_t launch_prefill(const PoolView& pool, const AttnArgs& a, cudaStream_t stream) {
    const int g = a.num_heads / pool.num_kv_heads;
    // A chunk of a few queries (a speculative-decoding verify, one decode token) is a
    // bandwidth-bound decode with a causal mask: it runs on the decode kernel, its
    // (query, head) rows on the MMA N dimension.  Longer chunks run on the tensor-core
    // kernel with scores and P in tensor memory (pa_prefill_tc2.cu).  PA_PREFILL_IMPL forces a
    // kernel for A/B comparisons: 2 that one, t the tensor-core kernel with Q in tensor memory
    // and P in shared memory (pa_prefill_tc.cu), m the warp-MMA kernel.
    static const char forced = [] {
        const char* e = std::getenv("PA_PREFILL_IMPL");
        return e ? e[0] : '\0';
    }();
    if (forced != 't' && forced != 'm' && forced != '2' && decode_mq_supported(g, a.max_chunk))
        return launch_decode_mq(pool, a, stream);
    if (forced != 'm' && prefill_tc_supported(pool.head_dim, g))
        return forced == 't' ? launch_prefill_tc(pool, a, stream) : launch_prefill_tc2(pool, a, stream);
    if (pool.head_dim == 128) return launch_mma<128>(pool, a, stream);
    return launch_mma<64>(pool, a, stream);
}

}  // namespace pa
