// pa_internal.h -- what the C-ABI layer (pa_capi.cu) hands to the kernel launchers.
// Host-side only; no torch types anywhere in the library.
#pragma once

#include <cuda.h>
#include <atomic>
#include <cstdlib>
#include <cuda_runtime.h>
#include <mutex>
#include <stdint.h>

namespace pa {

// A validated pool: [num_blocks, num_kv_heads, 16, head_dim] bf16 for K and for V, with
// two TMA maps per tensor, both with 128-byte swizzling:
//   tm_k / tm_v   2-D [rows = num_blocks*num_kv_heads*16, head_dim], box 64 columns x 16 rows
//                 (one 64-column half of a (block, head) tile, 2 KB);
//   tile_k/tile_v 4-D (64 columns, 16 rows, head_dim/64 halves, num_blocks*num_kv_heads tiles)
//                 with the halves dimension strided 128 B and the rows 2*head_dim B, box =
//                 one whole (block, head) tile, which lands as [half][16 rows][128 B].
struct PoolView {
    void* k;
    void* v;
    int num_blocks;
    int num_kv_heads;
    int head_dim;
    CUtensorMap tm_k;
    CUtensorMap tm_v;
    CUtensorMap tile_k;
    CUtensorMap tile_v;
};

struct DeviceInfo {
    int device;
    int num_sms;
    int max_smem_optin;
};

// Per-call arguments of the attention kernels (decode, split-KV, prefill).
struct AttnArgs {
    const void* q;               // decode [B, Hq, D]; prefill [sum C, Hq, D] bf16
    const int32_t* block_tables; // [B, max_blocks]
    const int32_t* seq_lens;     // [B]
    const int32_t* cu_q_lens;    // prefill only, [B+1]
    void* out;                   // bf16, same shape as q
    float* ws_o;                 // split-KV partial outputs [B, Hq, P, D] fp32
    float* ws_lse;               // split-KV partial log-sum-exp [B, Hq, P] fp32
    unsigned* status;            // device status word
    int batch;
    int num_heads;
    int max_blocks;
    int num_partitions;          // split-KV only
    int max_chunk;               // prefill only
    float scale;
    // decode only, fused append (null: none): one new K/V row per sequence [B, Hkv, D] bf16
    // and its slot [B]; written by the kernel before it reads the sequence's last block
    const void* k_new;
    const void* v_new;
    const int64_t* slots;
};

const DeviceInfo& device_info();
// 3-D TMA map (d, head, token) over a [tokens, heads, d] bf16 tensor (d = 128), 128-byte
// swizzled, box (64, box_heads, box_tokens); false if it cannot be encoded.
bool rows_map(CUtensorMap* out, const void* base, long long tokens, int heads, int d, int box_heads, int box_tokens);
unsigned* device_status_ptr();

// One-time set-up of a kernel (function attributes, occupancy queries) on each device:
// function attributes are per device, and library calls may come from several host threads
// at once.  `run` calls `setup` on the current device's first use, under a lock, and
// remembers success; a failed set-up is retried by the next call.
class OncePerDevice {
  public:
    template <typename F>
    cudaError_t run(F&& setup) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevices) return cudaErrorInvalidDevice;
        if (done_[dev].load(std::memory_order_acquire)) return cudaSuccess;
        std::lock_guard<std::mutex> lk(mu_);
        if (done_[dev].load(std::memory_order_relaxed)) return cudaSuccess;
        const cudaError_t e = setup();
        if (e == cudaSuccess) done_[dev].store(true, std::memory_order_release);
        return e;
    }

  private:
    static constexpr int kDevices = 64;
    std::mutex mu_;
    std::atomic<bool> done_[kDevices] = {};
};

// Launch attribute that lets a kernel overlap its launch with the previous kernel's tail
// (every kernel waits for that kernel to complete before touching memory, so results do not
// depend on it).  On unless PA_PDL=0: with a serving step's independent workloads on
// parallel streams it measured 139 us per step against 147 without, and 164 against 165
// with the calls one after another on one stream.
inline cudaLaunchAttribute pdl_attribute() {
    static const int allowed = [] {
        const char* e = std::getenv("PA_PDL");
        return (e && e[0] == '0') ? 0 : 1;
    }();
    cudaLaunchAttribute at = {};
    at.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at.val.programmaticStreamSerializationAllowed = allowed;
    return at;
}

cudaError_t launch_kv_append(const PoolView& pool, const void* k_new, const void* v_new, const int64_t* slots,
                             int num_tokens, unsigned* status, cudaStream_t stream);
cudaError_t launch_selftest_wait(unsigned* status, long long limit_cycles, cudaStream_t stream);
cudaError_t launch_kv_copy(const PoolView& pool, const int64_t* src_slots, const int64_t* dst_slots, int n,
                           unsigned* status, cudaStream_t stream);
cudaError_t launch_decode(const PoolView& pool, const AttnArgs& a, cudaStream_t stream);
cudaError_t launch_decode_splitkv(const PoolView& pool, const AttnArgs& a, cudaStream_t stream);
// Multi-query decode: a chunk of <= max_chunk queries per sequence over its cache, on the
// decode kernel (columns = query x head), when max_chunk x group <= 16.
bool decode_mq_supported(int group, int max_chunk);
cudaError_t launch_decode_mq(const PoolView& pool, const AttnArgs& a, cudaStream_t stream);
cudaError_t launch_combine(const float* ws_o, const float* ws_lse, int batch, int num_heads, int head_dim,
                           int num_partitions, void* out, cudaStream_t stream);
cudaError_t launch_prefill(const PoolView& pool, const AttnArgs& a, cudaStream_t stream);
// tcgen05 chunked prefill: head_dim 128 and a group size dividing 128
bool prefill_tc_supported(int head_dim, int group);
cudaError_t launch_prefill_tc(const PoolView& pool, const AttnArgs& a, cudaStream_t stream);
// the same shapes, 128-key stages with P in tensor memory
cudaError_t launch_prefill_tc2(const PoolView& pool, const AttnArgs& a, cudaStream_t stream);

// Split count the decode launcher picks for a problem (exposed for tests and tuning).
int decode_splits_for(int batch, int num_kv_heads, int max_blocks);
// Partition count suggested for pa_decode_splitkv.
int splitkv_partitions_for(int batch, int num_kv_heads, int max_blocks);

}  // namespace pa
