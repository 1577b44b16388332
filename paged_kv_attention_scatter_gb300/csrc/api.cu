// Library-wide entry points of libpagedattn: version, error text, device facts.
#include "common.cuh"

int pkv_num_sms() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            n <= 0)
            n = 1;
        cached[dev] = n;
    }
    return cached[dev];
}

namespace {
std::atomic<uint32_t> g_wait_polls{PKV_DEFAULT_WAIT_POLLS};
}  // namespace

uint32_t pkv_wait_polls() { return g_wait_polls.load(std::memory_order_relaxed); }

extern "C" int pkv_set_wait_poll_limit(uint32_t polls) {
    g_wait_polls.store(polls, std::memory_order_relaxed);
    return PKV_OK;
}

extern "C" int pkv_version(void) { return 100; }

extern "C" const char* pkv_error_string(int code) {
    switch (code) {
        case PKV_OK: return "ok";
        case PKV_ERR_NULL_POINTER: return "a required pointer is null";
        case PKV_ERR_BAD_DIMENSION: return "a size argument is out of range";
        case PKV_ERR_UNSUPPORTED_HEAD_DIM: return "head_dim is not supported (64 or 128)";
        case PKV_ERR_MISALIGNED: return "a pointer is not aligned as required";
        case PKV_ERR_WORKSPACE_TOO_SMALL: return "the workspace is smaller than required";
        case PKV_ERR_CUDA: return "a CUDA launch failed";
        case PKV_ERR_UNSUPPORTED: return "no kernel supports these shapes";
        default: return "unknown error code";
    }
}

extern "C" const char* pkv_status_string(uint32_t bits) {
    if (bits == 0) return "ok";
    if (bits & PKV_STATUS_SLOT_OUT_OF_RANGE) return "slot outside the pool";
    if (bits & PKV_STATUS_BAD_BLOCK_ID) return "block table entry outside the pool";
    if (bits & PKV_STATUS_BAD_CONTEXT_LEN) return "context length out of range";
    if (bits & PKV_STATUS_BAD_SEQLENS) return "inconsistent cu_seqlens";
    if (bits & PKV_STATUS_BAD_TEMPERATURE) return "temperature not positive and finite";
    if (bits & PKV_STATUS_NO_FINITE_KEY) return "every sampling key of a row is NaN";
    if (bits & PKV_STATUS_WORKSPACE_OVERFLOW) return "more work items than the workspace holds";
    if (bits & PKV_STATUS_WAIT_TIMEOUT) return "a bounded in-kernel wait gave up";
    return "unknown status bit";
}

extern "C" int pkv_layer_cache(const void* kv_pool, int32_t num_layers, int32_t layer,
                               pkv_cache_desc cache, const void** k_cache,
                               const void** v_cache) {
    if (!kv_pool || !k_cache || !v_cache) return PKV_ERR_NULL_POINTER;
    if (num_layers <= 0 || layer < 0 || layer >= num_layers || cache.num_blocks <= 0 ||
        cache.block_size <= 0 || cache.num_kv_heads <= 0 || cache.head_dim <= 0)
        return PKV_ERR_BAD_DIMENSION;
    const size_t layer_bytes = (size_t)cache.num_blocks * cache.block_size *
                               cache.num_kv_heads * cache.head_dim * 2;
    const char* base = (const char*)kv_pool;
    *k_cache = base + (size_t)layer * layer_bytes;
    *v_cache = base + ((size_t)num_layers + layer) * layer_bytes;
    return PKV_OK;
}
