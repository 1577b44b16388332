// kv_store: scatter each new token's K and V rows into the paged cache.
//
// The per-layer cache write of a Nano-vLLM-style engine (uml.org.cn
// walk-through §2.4 and "KV cache的写入函数"; "一个 prompt 的一生" §3.3.2, §4):
// slot_mapping[i] is the physical slot of flattened token i, a slot being
// row block_id*block_size + offset of the pool viewed as
// [num_blocks*block_size, Hkv, D].  The writer needs no other paging logic, so
// the kernel is a row scatter: token i's K row (Hkv*D bf16, contiguous) goes
// to pool row slot_mapping[i], and the same for V.
//
// Design: one 16-byte vector per thread per tensor; a warp covers 512
// contiguous bytes of a row, so both the read of k/v and the write of the
// cache row are fully coalesced.  Loads are issued for K and V before either
// store to keep two requests in flight per thread.  When a row is a
// power-of-two number of vectors (every usual Hkv x D) the token / column
// split of the flat index is a shift and a mask on 32-bit indices instead of
// a 64-bit division.  HBM traffic = 2 reads + 2 writes of Hkv*D*2 bytes per
// token: the roofline is pure bandwidth.
#include "common.cuh"

namespace {

// kRowShift >= 0: a row is 2^kRowShift vectors and every index fits in 32
// bits, so the row / column split is a shift and a mask; -1: the general case.
template <int kRowShift>
__global__ void __launch_bounds__(256) kv_store_kernel(
        const uint4* __restrict__ k, const uint4* __restrict__ v,
        uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
        const int32_t* __restrict__ slot_mapping, int32_t num_tokens,
        int32_t row_vecs, int64_t num_slots, uint32_t* status) {
    // a decode launched after this store may start its set-up now; it waits
    // for this grid's stores before reading the cache
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if constexpr (kRowShift >= 0) {
        const uint32_t total = (uint32_t)num_tokens << kRowShift;
        const uint32_t stride = gridDim.x * blockDim.x;
        for (uint32_t idx = blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += stride) {
            const uint32_t t = idx >> kRowShift, c = idx & ((1u << kRowShift) - 1u);
            const int32_t s = __ldg(slot_mapping + t);
            if (s < 0) continue;                              // padding row
            if ((int64_t)s >= num_slots) {
                if (c == 0) pkv::report(status, PKV_STATUS_SLOT_OUT_OF_RANGE);
                continue;
            }
            const uint4 kv = pkv::ld_stream16(k + idx);
            const uint4 vv = pkv::ld_stream16(v + idx);
            const int64_t dst = ((int64_t)s << kRowShift) + c;
            k_cache[dst] = kv;
            v_cache[dst] = vv;
        }
    } else {
        const int64_t total = (int64_t)num_tokens * row_vecs;
        const int64_t stride = (int64_t)gridDim.x * blockDim.x;
        for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
             idx += stride) {
            const int32_t t = (int32_t)(idx / row_vecs);
            const int32_t c = (int32_t)(idx - (int64_t)t * row_vecs);
            const int32_t s = __ldg(slot_mapping + t);
            if (s < 0) continue;                              // padding row
            if ((int64_t)s >= num_slots) {
                if (c == 0) pkv::report(status, PKV_STATUS_SLOT_OUT_OF_RANGE);
                continue;
            }
            const uint4 kv = pkv::ld_stream16(k + idx);
            const uint4 vv = pkv::ld_stream16(v + idx);
            const int64_t dst = (int64_t)s * row_vecs + c;
            k_cache[dst] = kv;
            v_cache[dst] = vv;
        }
    }
}

}  // namespace

int pkv_store_rows_args(const void* k, const void* v, void* k_cache, void* v_cache,
                        const int32_t* slot_mapping, int32_t num_tokens,
                        const pkv_cache_desc& cache, uint32_t* status, pkv::StoreRows& st) {
    if (num_tokens < 0) return PKV_ERR_BAD_DIMENSION;
    if (cache.num_blocks <= 0 || cache.block_size <= 0 || cache.num_kv_heads <= 0 ||
        cache.head_dim <= 0)
        return PKV_ERR_BAD_DIMENSION;
    st = pkv::StoreRows{};
    st.num_tokens = num_tokens;
    if (num_tokens == 0) return PKV_OK;
    if (!k || !v || !k_cache || !v_cache || !slot_mapping) return PKV_ERR_NULL_POINTER;
    const int64_t row_bytes = (int64_t)cache.num_kv_heads * cache.head_dim * 2;
    if (row_bytes % 16 != 0) return PKV_ERR_UNSUPPORTED_HEAD_DIM;
    if (((uintptr_t)k | (uintptr_t)v | (uintptr_t)k_cache | (uintptr_t)v_cache) & 15)
        return PKV_ERR_MISALIGNED;
    if (((uintptr_t)slot_mapping) & 3) return PKV_ERR_MISALIGNED;
    st.k = (const uint4*)k;
    st.v = (const uint4*)v;
    st.kc = (uint4*)k_cache;
    st.vc = (uint4*)v_cache;
    st.slots = slot_mapping;
    st.row_vecs = (int32_t)(row_bytes / 16);
    st.num_slots = (int64_t)cache.num_blocks * cache.block_size;
    st.status = status;
    return PKV_OK;
}

extern "C" int pkv_kv_store(const void* k, const void* v, void* k_cache, void* v_cache,
                            const int32_t* slot_mapping, int32_t num_tokens,
                            pkv_cache_desc cache, uint32_t* status, void* stream) {
    pkv::StoreRows st;
    const int rc = pkv_store_rows_args(k, v, k_cache, v_cache, slot_mapping, num_tokens, cache,
                                       status, st);
    if (rc != PKV_OK || num_tokens == 0) return rc;
    const int32_t row_vecs = st.row_vecs;
    const int64_t total = (int64_t)num_tokens * row_vecs;
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    const int64_t cap = (int64_t)pkv_num_sms() * 16;
    if (blocks > cap) blocks = cap;
    const int64_t num_slots = st.num_slots;
    // the shift-and-mask form when a row is a power-of-two number of vectors
    // and every index fits in 32 bits (always, at these sizes)
    int shift = -1;
    if ((row_vecs & (row_vecs - 1)) == 0 && total + (int64_t)blocks * threads < (1LL << 31))
        shift = __builtin_ctz((unsigned)row_vecs);
    auto launch = [&](auto kernel) {
        kernel<<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(
            (const uint4*)k, (const uint4*)v, (uint4*)k_cache, (uint4*)v_cache, slot_mapping,
            num_tokens, row_vecs, num_slots, status);
    };
    switch (shift) {
        case 3: launch(kv_store_kernel<3>); break;     // 128-byte rows (e.g. 1 x 64)
        case 4: launch(kv_store_kernel<4>); break;     // 256-byte rows (e.g. 1 x 128)
        case 5: launch(kv_store_kernel<5>); break;
        case 6: launch(kv_store_kernel<6>); break;
        case 7: launch(kv_store_kernel<7>); break;     // 2 KiB rows (8 x 128)
        case 8: launch(kv_store_kernel<8>); break;
        default: launch(kv_store_kernel<-1>); break;
    }
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
