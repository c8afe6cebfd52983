// pa_append.cu -- scatter of new K/V rows into pool slots through a slot mapping.
//
// k_cache[slot / 16, h, slot % 16, :] = k_new[t, h, :] (and V) for every t with
// slot_mapping[t] >= 0.  This is how a decode step's newest token, or a prefill
// chunk, enters the paged cache before attention reads it ("Qwen3-4B / 8B / 32B",
// section "Architecture Notes": paged KV cache; section "Warm Prefix-Cache TTFT":
// a warm prefix is reused and only the new tokens are written).
//
// One thread moves one 16-byte chunk; consecutive threads take consecutive chunks
// of a (token, head) row, so both the read of k_new and the write into the pool row
// are coalesced 256-byte runs (d = 128).  A slot past the pool is skipped and
// reported in the device status word.
#include <algorithm>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

__global__ void __launch_bounds__(256) kv_append_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                                                        const uint4* __restrict__ k_new,
                                                        const uint4* __restrict__ v_new,
                                                        const int64_t* __restrict__ slots, int num_tokens,
                                                        int num_kv_heads, int chunks, long long pool_slots,
                                                        unsigned* status) {
    pdl_trigger();
    pdl_wait();
    const int row = num_kv_heads * chunks;  // 16-byte chunks of one token's K (or V) row
    const int per_tok = 2 * row;
    const int total = num_tokens * per_tok;  // < 2^31, checked by the launcher
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
        const int t = i / per_tok, r = i - t * per_tok;
        const bool is_v = r >= row;
        const int j = is_v ? r - row : r;  // h * chunks + c
        // the source chunk does not depend on the slot: both loads are in flight together
        const uint4 val = __ldg((is_v ? v_new : k_new) + (size_t)t * row + j);
        const int64_t slot = __ldg(slots + t);
        if (slot < 0) continue;
        if (slot >= pool_slots) {
            if (j == 0 && !is_v) atomicOr(status, kDevOutOfRange);
            continue;
        }
        const int h = j / chunks, c = j - h * chunks;
        const size_t dst = (((size_t)(slot / kBlockSize) * num_kv_heads + h) * kBlockSize + slot % kBlockSize) * chunks + c;
        (is_v ? v_cache : k_cache)[dst] = val;
    }
}

// Copy of whole (slot, every kv head) rows inside the pool: row src_slots[t] -> row
// dst_slots[t] of K and of V (a prefix-cache hit that ends inside a cached block copies that
// block's leading rows into the request's own block).  Same chunk-per-thread layout as the
// append: consecutive threads move consecutive 16-byte chunks of one row.
__global__ void __launch_bounds__(256) kv_copy_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                                                      const int64_t* __restrict__ src_slots,
                                                      const int64_t* __restrict__ dst_slots, int n, int num_kv_heads,
                                                      int chunks, long long pool_slots, unsigned* status) {
    pdl_trigger();
    pdl_wait();
    const int row = num_kv_heads * chunks;
    const int per_tok = 2 * row;
    const int total = n * per_tok;  // < 2^31, checked by the launcher
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
        const int t = i / per_tok, r = i - t * per_tok;
        const bool is_v = r >= row;
        const int j = is_v ? r - row : r;
        const int64_t src = __ldg(src_slots + t), dst = __ldg(dst_slots + t);
        if (src < 0 || dst < 0) continue;
        if (src >= pool_slots || dst >= pool_slots) {
            if (j == 0 && !is_v) atomicOr(status, kDevOutOfRange);
            continue;
        }
        const int h = j / chunks, c = j - h * chunks;
        auto at = [&](int64_t slot) {
            return (((size_t)(slot / kBlockSize) * num_kv_heads + h) * kBlockSize + slot % kBlockSize) * chunks + c;
        };
        uint4* pool = is_v ? v_cache : k_cache;
        pool[at(dst)] = pool[at(src)];
    }
}

}  // namespace

cudaError_t launch_kv_copy(const PoolView& pool, const int64_t* src_slots, const int64_t* dst_slots, int n,
                           unsigned* status, cudaStream_t stream) {
    const int chunks = pool.head_dim * 2 / 16;
    const long long total = (long long)n * 2 * pool.num_kv_heads * chunks;
    if (total >= (1LL << 31)) return cudaErrorInvalidValue;
    const long long want = (total + 255) / 256;
    const int blocks = static_cast<int>(std::max(1LL, std::min<long long>(want, (long long)device_info().num_sms * 16)));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kv_copy_kernel, static_cast<uint4*>(pool.k), static_cast<uint4*>(pool.v),
                              src_slots, dst_slots, n, pool.num_kv_heads, chunks,
                              (long long)pool.num_blocks * kBlockSize, status);
}

cudaError_t launch_kv_append(const PoolView& pool, const void* k_new, const void* v_new, const int64_t* slots,
                             int num_tokens, unsigned* status, cudaStream_t stream) {
    const int chunks = pool.head_dim * 2 / 16;
    const long long total = (long long)num_tokens * 2 * pool.num_kv_heads * chunks;
    if (total >= (1LL << 31)) return cudaErrorInvalidValue;
    const long long want = (total + 255) / 256;
    const int blocks = static_cast<int>(std::max(1LL, std::min<long long>(want, (long long)device_info().num_sms * 16)));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kv_append_kernel, static_cast<uint4*>(pool.k), static_cast<uint4*>(pool.v),
                              static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), slots, num_tokens,
                              pool.num_kv_heads, chunks, (long long)pool.num_blocks * kBlockSize, status);
}

}  // namespace pa
