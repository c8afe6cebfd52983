// pa_noalloc.cu -- long-context decode for callers that cannot allocate device memory.
//
// pa_decode_splitkv needs a caller-provided workspace for the per-partition results.
// Some callers have no way to provide one: an engine whose device memory is a fixed arena
// owned by someone else, a plugin inside a host framework that exposes no allocator, or a
// serving loop that must never call cudaMalloc on its hot path (an allocation there can
// synchronise the device and stall every stream).  pa_decode_splitkv_noalloc runs the same
// split-KV decode and log-sum-exp combine, but keeps the partition results in one
// statically sized device array that is part of the library image (every GPU that loads
// the library holds it until the process exits).
#include <mutex>

#include "pagedattn.h"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr size_t kScratchBytes = size_t(8) << 20;  // 8 MiB: ws_o + ws_lse of one call

__device__ __align__(256) unsigned char g_splitkv_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code the array's
// name is only a host-side stand-in, so the real address is looked up once per device
// (with that device current) and cached for the life of the process; a cudaDeviceReset
// could move the module, which is why the header rules out calls after one.
void* scratch_on_current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_splitkv_scratch) != cudaSuccess || !p) return nullptr;
        g_scratch_addr[dev] = p;
    }
    return g_scratch_addr[dev];
}

}  // namespace
}  // namespace pa

extern "C" {

size_t pa_noalloc_scratch_bytes(void) { return pa::kScratchBytes; }

int pa_decode_splitkv_noalloc(const pa_pool* pool, const void* q, const int32_t* block_tables, int32_t max_blocks,
                              const int32_t* seq_lens, int32_t batch, int32_t num_heads, float scale,
                              int32_t num_partitions, void* out, pa_stream_t stream) {
    if (!pool) return PA_ERR_INVALID_ARG;
    if (pool->head_dim != 64 && pool->head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (batch < 0 || num_heads <= 0 || num_partitions < 1 || num_partitions > 4096) return PA_ERR_INVALID_ARG;
    if (batch == 0) return PA_OK;
    if (!out) return PA_ERR_INVALID_ARG;
    const size_t need = pa_splitkv_workspace_bytes(batch, num_heads, pool->head_dim, num_partitions);
    if (need == 0 || need > pa::kScratchBytes) return PA_ERR_TOO_LARGE;
    void* base = pa::scratch_on_current_device();
    if (!base) return PA_ERR_CUDA;
    // ws_o first, then ws_lse at the next 16-byte boundary (the layout the size above counts)
    const size_t o_bytes = (size_t)batch * num_heads * num_partitions * pool->head_dim * sizeof(float);
    float* ws_o = static_cast<float*>(base);
    float* ws_lse = reinterpret_cast<float*>(static_cast<unsigned char*>(base) + ((o_bytes + 15) & ~size_t(15)));
    // every partition slot is written by the split kernel (empty ones as O = 0, lse = -inf),
    // so nothing left over from an earlier call is ever read
    int rc = pa_decode_splitkv(pool, q, block_tables, max_blocks, seq_lens, batch, num_heads, scale,
                               num_partitions, ws_o, ws_lse, stream);
    if (rc != PA_OK) return rc;
    return pa_combine(ws_o, ws_lse, batch, num_heads, pool->head_dim, num_partitions, out, stream);
}

}  // extern "C"
