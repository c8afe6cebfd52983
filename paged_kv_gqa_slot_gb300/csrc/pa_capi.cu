// pa_capi.cu -- the C ABI of libpagedattn: argument validation, the device status
// word, the per-device launch facts and the cache of TMA descriptors over the pool.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "pagedattn.h"
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

__device__ unsigned g_status_word;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;

int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    return dev;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

struct MapKey {
    const void* base;
    long long rows;
    int d;
    int kind;   // 0: 2-D half-tile boxes, 1: 4-D whole-tile boxes, 2: 3-D (d, head, token) rows
    int extra;  // kind 2: heads * 65536 + box heads
    bool operator==(const MapKey& o) const {
        return base == o.base && rows == o.rows && d == o.d && kind == o.kind && extra == o.extra;
    }
};
struct MapKeyHash {
    size_t operator()(const MapKey& k) const {
        return std::hash<const void*>()(k.base) ^ (std::hash<long long>()(k.rows) * 31u) ^ (size_t)k.d ^
               ((size_t)k.kind << 20) ^ ((size_t)k.extra << 24);
    }
};
std::unordered_map<MapKey, CUtensorMap, MapKeyHash>& map_cache() {
    static std::unordered_map<MapKey, CUtensorMap, MapKeyHash> cache;
    return cache;
}

// TMA maps over one pool tensor, 128-byte swizzled (see PoolView).  A map depends only on
// (address, rows, head_dim, kind), so cached maps never go stale.
//   kind 0: [rows = num_blocks*num_kv_heads*16, head_dim], box 64 x 16 (a tile half, 2 KB);
//   kind 1: (64, 16, head_dim/64, rows/16) with strides (2*head_dim, 128, 32*head_dim) bytes,
//           box (64, 16, head_dim/64, 1): a whole (block, head) tile landing half-major.
bool pool_map(CUtensorMap* out, void* base, long long rows, int d, int kind) {
    auto& cache = map_cache();
    const MapKey key{base, rows, d, kind, 0};
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = cache.find(key);
        if (it != cache.end()) {
            *out = it->second;
            return true;
        }
    }
    auto fn = encode_fn();
    if (!fn) return false;
    CUtensorMap m;
    CUresult r;
    if (kind == 0) {
        const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
        const cuuint64_t strides[1] = {(cuuint64_t)d * 2};
        const cuuint32_t box[2] = {64, 16};
        const cuuint32_t estr[2] = {1, 1};
        r = fn(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        const cuuint64_t dims[4] = {64, (cuuint64_t)kBlockSize, (cuuint64_t)(d / 64), (cuuint64_t)(rows / kBlockSize)};
        const cuuint64_t strides[3] = {(cuuint64_t)d * 2, 128, (cuuint64_t)kBlockSize * d * 2};
        const cuuint32_t box[4] = {64, (cuuint32_t)kBlockSize, (cuuint32_t)(d / 64), 1};
        const cuuint32_t estr[4] = {1, 1, 1, 1};
        r = fn(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (r != CUDA_SUCCESS) return false;
    std::lock_guard<std::mutex> lk(g_mu);
    if (cache.size() > 256) cache.clear();
    cache[key] = m;
    *out = m;
    return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_pool(const pa_pool* p, PoolView* v, bool need_maps) {
    if (!p || !p->k_cache || !p->v_cache) return PA_ERR_INVALID_ARG;
    if (p->num_blocks <= 0 || p->num_kv_heads <= 0 || p->block_size <= 0 || p->head_dim <= 0)
        return PA_ERR_INVALID_ARG;
    if (p->block_size != kBlockSize) return PA_ERR_UNSUPPORTED;
    if (p->head_dim != 64 && p->head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (!aligned16(p->k_cache) || !aligned16(p->v_cache)) return PA_ERR_INVALID_ARG;
    const long long rows = (long long)p->num_blocks * p->num_kv_heads * kBlockSize;
    if (rows > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;  // TMA row coordinates are int32
    v->k = p->k_cache;
    v->v = p->v_cache;
    v->num_blocks = p->num_blocks;
    v->num_kv_heads = p->num_kv_heads;
    v->head_dim = p->head_dim;
    if (need_maps) {
        if (!pool_map(&v->tm_k, p->k_cache, rows, p->head_dim, 0)) return PA_ERR_CUDA;
        if (!pool_map(&v->tm_v, p->v_cache, rows, p->head_dim, 0)) return PA_ERR_CUDA;
        if (!pool_map(&v->tile_k, p->k_cache, rows, p->head_dim, 1)) return PA_ERR_CUDA;
        if (!pool_map(&v->tile_v, p->v_cache, rows, p->head_dim, 1)) return PA_ERR_CUDA;
    }
    return PA_OK;
}

int check_heads(const PoolView& v, int num_heads) {
    if (num_heads <= 0 || num_heads % v.num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    return PA_OK;
}

int from_cuda(cudaError_t e) { return e == cudaSuccess ? PA_OK : PA_ERR_CUDA; }

}  // namespace

// 3-D map (d, head, token) over a [tokens, heads, d] bf16 tensor, 128-byte swizzled, whose
// box is (64 columns, box_heads heads, box_tokens tokens): one column half of a query tile
// whose rows are (token, head) pairs.  Cached like the pool maps.
bool rows_map(CUtensorMap* out, const void* base, long long tokens, int heads, int d, int box_heads, int box_tokens) {
    if (tokens <= 0 || heads <= 0 || d != 128 || box_heads <= 0 || box_heads > 256 || box_tokens <= 0 ||
        box_tokens > 256 || box_heads > heads)
        return false;
    auto& cache = map_cache();
    const MapKey key{base, tokens, d, 2, heads * 65536 + box_heads};
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = cache.find(key);
        if (it != cache.end()) {
            *out = it->second;
            return true;
        }
    }
    auto fn = encode_fn();
    if (!fn) return false;
    CUtensorMap m;
    const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)tokens};
    const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)heads * d * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)box_heads, (cuuint32_t)box_tokens};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    std::lock_guard<std::mutex> lk(g_mu);
    if (cache.size() > 256) cache.clear();
    cache[key] = m;
    *out = m;
    return true;
}

const DeviceInfo& device_info() {
    static DeviceInfo infos[kMaxDevices];
    static bool ready[kMaxDevices] = {};
    int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) dev = 0;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!ready[dev]) {
        DeviceInfo d{};
        d.device = dev;
        cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
        cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (d.num_sms <= 0) d.num_sms = 1;
        infos[dev] = d;
        ready[dev] = true;
    }
    return infos[dev];
}

unsigned* device_status_ptr() {
    static unsigned* ptrs[kMaxDevices] = {};
    int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!ptrs[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        ptrs[dev] = static_cast<unsigned*>(p);
    }
    return ptrs[dev];
}

}  // namespace pa

using namespace pa;

extern "C" {

int pa_kv_append(const pa_pool* pool, const void* k_new, const void* v_new, const int64_t* slot_mapping,
                 int32_t num_tokens, pa_stream_t stream) {
    PoolView v;
    int rc = check_pool(pool, &v, false);
    if (rc) return rc;
    if (num_tokens < 0) return PA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PA_OK;
    if (!k_new || !v_new || !slot_mapping || !aligned16(k_new) || !aligned16(v_new)) return PA_ERR_INVALID_ARG;
    if ((long long)num_tokens * 2 * v.num_kv_heads * (v.head_dim / 8) >= (1LL << 31)) return PA_ERR_INVALID_ARG;
    unsigned* st = device_status_ptr();
    if (!st) return PA_ERR_CUDA;
    return from_cuda(launch_kv_append(v, k_new, v_new, slot_mapping, num_tokens, st, (cudaStream_t)stream));
}

int pa_kv_copy(const pa_pool* pool, const int64_t* src_slots, const int64_t* dst_slots, int32_t n,
               pa_stream_t stream) {
    PoolView v;
    int rc = check_pool(pool, &v, false);
    if (rc) return rc;
    if (n < 0) return PA_ERR_INVALID_ARG;
    if (n == 0) return PA_OK;
    if (!src_slots || !dst_slots) return PA_ERR_INVALID_ARG;
    if ((long long)n * 2 * v.num_kv_heads * (v.head_dim / 8) >= (1LL << 31)) return PA_ERR_INVALID_ARG;
    unsigned* st = device_status_ptr();
    if (!st) return PA_ERR_CUDA;
    return from_cuda(launch_kv_copy(v, src_slots, dst_slots, n, st, (cudaStream_t)stream));
}

static int check_attn(const pa_pool* pool, PoolView* v, const void* q, const int32_t* block_tables,
                      int32_t max_blocks, const int32_t* seq_lens, int32_t batch, int32_t num_heads, float scale,
                      const void* out) {
    int rc = check_pool(pool, v, false);
    if (rc) return rc;
    rc = check_heads(*v, num_heads);
    if (rc) return rc;
    if (batch < 0 || batch > 65535) return PA_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return PA_ERR_INVALID_ARG;
    if (batch == 0) return PA_OK;
    if (!q || !block_tables || !seq_lens || !out || !aligned16(q) || !aligned16(out)) return PA_ERR_INVALID_ARG;
    if (max_blocks <= 0 || (long long)max_blocks * kBlockSize > 0x7fffffffLL) return PA_ERR_INVALID_ARG;
    return PA_OK;
}

int pa_decode(const pa_pool* pool, const void* q, const int32_t* block_tables, int32_t max_blocks,
              const int32_t* seq_lens, int32_t batch, int32_t num_heads, float scale, void* out,
              pa_stream_t stream) {
    PoolView v;
    int rc = check_attn(pool, &v, q, block_tables, max_blocks, seq_lens, batch, num_heads, scale, out);
    if (rc || batch == 0) return rc;
    if (num_heads / v.num_kv_heads > 16) return PA_ERR_UNSUPPORTED;
    rc = check_pool(pool, &v, true);
    if (rc) return rc;
    AttnArgs a{};
    a.q = q;
    a.block_tables = block_tables;
    a.seq_lens = seq_lens;
    a.out = out;
    a.status = device_status_ptr();
    if (!a.status) return PA_ERR_CUDA;
    a.batch = batch;
    a.num_heads = num_heads;
    a.max_blocks = max_blocks;
    a.scale = scale;
    return from_cuda(launch_decode(v, a, (cudaStream_t)stream));
}

int pa_append_decode(const pa_pool* pool, const void* k_new, const void* v_new, const int64_t* slot_mapping,
                     const void* q, const int32_t* block_tables, int32_t max_blocks, const int32_t* seq_lens,
                     int32_t batch, int32_t num_heads, float scale, void* out, pa_stream_t stream) {
    PoolView v;
    int rc = check_attn(pool, &v, q, block_tables, max_blocks, seq_lens, batch, num_heads, scale, out);
    if (rc || batch == 0) return rc;
    if (num_heads / v.num_kv_heads > 16) return PA_ERR_UNSUPPORTED;
    if (!k_new || !v_new || !slot_mapping || !aligned16(k_new) || !aligned16(v_new)) return PA_ERR_INVALID_ARG;
    rc = check_pool(pool, &v, true);
    if (rc) return rc;
    AttnArgs a{};
    a.q = q;
    a.block_tables = block_tables;
    a.seq_lens = seq_lens;
    a.out = out;
    a.status = device_status_ptr();
    if (!a.status) return PA_ERR_CUDA;
    a.batch = batch;
    a.num_heads = num_heads;
    a.max_blocks = max_blocks;
    a.scale = scale;
    a.k_new = k_new;
    a.v_new = v_new;
    a.slots = slot_mapping;
    return from_cuda(launch_decode(v, a, (cudaStream_t)stream));
}

size_t pa_splitkv_workspace_bytes(int32_t batch, int32_t num_heads, int32_t head_dim, int32_t num_partitions) {
    if (batch < 0 || num_heads < 0 || head_dim < 0 || num_partitions < 0) return 0;
    const size_t rows = (size_t)batch * num_heads * num_partitions;
    const size_t o = rows * head_dim * sizeof(float);
    const size_t lse = rows * sizeof(float);
    return ((o + 15) & ~size_t(15)) + lse;
}

int pa_decode_splitkv(const pa_pool* pool, const void* q, const int32_t* block_tables, int32_t max_blocks,
                      const int32_t* seq_lens, int32_t batch, int32_t num_heads, float scale,
                      int32_t num_partitions, float* ws_o, float* ws_lse, pa_stream_t stream) {
    PoolView v;
    int rc = check_attn(pool, &v, q, block_tables, max_blocks, seq_lens, batch, num_heads, scale, ws_o);
    if (rc) return rc;
    if (num_partitions < 1 || num_partitions > 4096) return PA_ERR_INVALID_ARG;
    if (batch == 0) return PA_OK;
    if (!ws_lse || !aligned16(ws_o)) return PA_ERR_INVALID_ARG;
    if (num_heads / v.num_kv_heads > 16) return PA_ERR_UNSUPPORTED;
    rc = check_pool(pool, &v, true);
    if (rc) return rc;
    AttnArgs a{};
    a.q = q;
    a.block_tables = block_tables;
    a.seq_lens = seq_lens;
    a.ws_o = ws_o;
    a.ws_lse = ws_lse;
    a.status = device_status_ptr();
    if (!a.status) return PA_ERR_CUDA;
    a.batch = batch;
    a.num_heads = num_heads;
    a.max_blocks = max_blocks;
    a.num_partitions = num_partitions;
    a.scale = scale;
    return from_cuda(launch_decode_splitkv(v, a, (cudaStream_t)stream));
}

int pa_combine(const float* ws_o, const float* ws_lse, int32_t batch, int32_t num_heads, int32_t head_dim,
               int32_t num_partitions, void* out, pa_stream_t stream) {
    if (batch < 0 || num_heads <= 0 || num_partitions < 1 || num_partitions > 4096) return PA_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
    if ((long long)batch * num_heads > 0x3fffffffLL) return PA_ERR_INVALID_ARG;
    if (batch == 0) return PA_OK;
    if (!ws_o || !ws_lse || !out || !aligned16(ws_o) || !aligned16(out)) return PA_ERR_INVALID_ARG;
    return from_cuda(launch_combine(ws_o, ws_lse, batch, num_heads, head_dim, num_partitions, out,
                                    (cudaStream_t)stream));
}

int pa_prefill_chunked(const pa_pool* pool, const void* q, const int32_t* cu_q_lens, const int32_t* block_tables,
                       int32_t max_blocks, const int32_t* seq_lens, int32_t batch, int32_t num_heads,
                       int32_t max_chunk, float scale, void* out, pa_stream_t stream) {
    PoolView v;
    int rc = check_attn(pool, &v, q, block_tables, max_blocks, seq_lens, batch, num_heads, scale, out);
    if (rc) return rc;
    if (max_chunk < 0) return PA_ERR_INVALID_ARG;
    if (batch == 0 || max_chunk == 0) return PA_OK;
    if (!cu_q_lens) return PA_ERR_INVALID_ARG;
    if ((long long)max_chunk * (num_heads / v.num_kv_heads) > 0x3fffffffLL) return PA_ERR_INVALID_ARG;
    rc = check_pool(pool, &v, true);
    if (rc) return rc;
    AttnArgs a{};
    a.q = q;
    a.cu_q_lens = cu_q_lens;
    a.block_tables = block_tables;
    a.seq_lens = seq_lens;
    a.out = out;
    a.status = device_status_ptr();
    if (!a.status) return PA_ERR_CUDA;
    a.batch = batch;
    a.num_heads = num_heads;
    a.max_blocks = max_blocks;
    a.max_chunk = max_chunk;
    a.scale = scale;
    return from_cuda(launch_prefill(v, a, (cudaStream_t)stream));
}

int pa_device_status(uint32_t* flags, int32_t clear, pa_stream_t stream) {
    if (!flags) return PA_ERR_INVALID_ARG;
    unsigned* p = device_status_ptr();
    if (!p) return PA_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    unsigned host = 0;
    if (cudaMemcpyAsync(&host, p, sizeof host, cudaMemcpyDeviceToHost, s) != cudaSuccess) return PA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_CUDA;
    if (clear) {
        if (cudaMemsetAsync(p, 0, sizeof(unsigned), s) != cudaSuccess) return PA_ERR_CUDA;
        if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_CUDA;
    }
    *flags = host;
    if (host & PA_DEV_TIMEOUT) return PA_ERR_TIMEOUT;
    if (host & PA_DEV_OUT_OF_RANGE) return PA_ERR_OUT_OF_RANGE;
    return PA_OK;
}

int pa_selftest_wait_timeout(uint64_t limit_cycles, pa_stream_t stream) {
    if (limit_cycles < 1 || limit_cycles > (1ull << 40)) return PA_ERR_INVALID_ARG;
    unsigned* p = device_status_ptr();
    if (!p) return PA_ERR_CUDA;
    return from_cuda(launch_selftest_wait(p, (long long)limit_cycles, (cudaStream_t)stream));
}

int pa_decode_num_splits(int32_t batch, int32_t num_kv_heads, int32_t max_blocks) {
    if (batch <= 0 || num_kv_heads <= 0 || max_blocks <= 0) return 1;
    return decode_splits_for(batch, num_kv_heads, max_blocks);
}

int pa_splitkv_num_partitions(int32_t batch, int32_t num_kv_heads, int32_t max_blocks) {
    if (batch <= 0 || num_kv_heads <= 0 || max_blocks <= 0) return 1;
    return splitkv_partitions_for(batch, num_kv_heads, max_blocks);
}

const char* pa_status_str(int status) {
    switch (status) {
        case PA_OK: return "PA_OK";
        case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
        case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
        case PA_ERR_CUDA: return "PA_ERR_CUDA";
        case PA_ERR_OUT_OF_RANGE: return "PA_ERR_OUT_OF_RANGE";
        case PA_ERR_TIMEOUT: return "PA_ERR_TIMEOUT";
        case PA_ERR_TOO_LARGE: return "PA_ERR_TOO_LARGE";
        case PA_ERR_REJECTED: return "PA_ERR_REJECTED";
        default: return "PA_ERR_UNKNOWN";
    }
}

int pa_version(void) { return 100; }

}  // extern "C"
