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
                                                        const int64_t* __restrict__ slots, long long per_tensor,
                                                        int num_kv_heads, int chunks, long long pool_slots,
                                                        unsigned* status) {
    pdl_trigger();
    pdl_wait();
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < 2 * per_tensor; i += stride) {
        const bool is_v = i >= per_tensor;
        const long long j = is_v ? i - per_tensor : i;
        const int c = static_cast<int>(j % chunks);
        const long long th = j / chunks;
        const int h = static_cast<int>(th % num_kv_heads);
        const long long t = th / num_kv_heads;
        const int64_t slot = __ldg(slots + t);
        if (slot < 0) continue;
        if (slot >= pool_slots) {
            if (c == 0 && h == 0 && !is_v) atomicOr(status, kDevOutOfRange);
            continue;
        }
        const long long dst = (((slot / kBlockSize) * num_kv_heads + h) * kBlockSize + slot % kBlockSize) * chunks + c;
        if (is_v)
            v_cache[dst] = __ldg(v_new + j);
        else
            k_cache[dst] = __ldg(k_new + j);
    }
}

}  // namespace

cudaError_t launch_kv_append(const PoolView& pool, const void* k_new, const void* v_new, const int64_t* slots,
                             int num_tokens, unsigned* status, cudaStream_t stream) {
    const int chunks = pool.head_dim * 2 / 16;
    const long long per_tensor = (long long)num_tokens * pool.num_kv_heads * chunks;
    const long long want = (2 * per_tensor + 255) / 256;
    const int blocks = static_cast<int>(std::max(1LL, std::min<long long>(want, (long long)device_info().num_sms * 16)));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kv_append_kernel, static_cast<uint4*>(pool.k), static_cast<uint4*>(pool.v),
                              static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), slots, per_tensor,
                              pool.num_kv_heads, chunks, (long long)pool.num_blocks * kBlockSize, status);
}

}  // namespace pa
