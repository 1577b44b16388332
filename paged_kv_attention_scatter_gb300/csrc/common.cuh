// Shared device helpers of libpagedattn (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/pagedattn.h"

// Raises a kernel's dynamic shared memory limit to `bytes` on the current
// device, once per device (the attribute is per device, so one flag per
// process would leave a second GPU of the same process unset).  `done` is the
// call site's mask of devices already set.
inline bool pkv_dynamic_smem_once(const void* fn, int bytes, std::atomic<uint64_t>& done) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0;
    if (bit != 0 && (done.load(std::memory_order_acquire) & bit)) return true;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
        cudaSuccess)
        return false;
    done.fetch_or(bit, std::memory_order_acq_rel);
    return true;
}

namespace pkv {

__device__ __forceinline__ void report(uint32_t* status, uint32_t bit) {
    if (status != nullptr) atomicOr(status, bit);
}

// 16-byte global load that bypasses L1 allocation (streamed K/V, logits).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ float4 ld_stream16f(const void* p) {
    float4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
                 : "l"(p));
    return r;
}

// One kv_store call as a device-side row scatter: token i's K and V rows
// (row_vecs 16-byte vectors each) go to pool row slots[i]; a negative slot is
// a padding row, one past the pool is reported and skipped.
struct StoreRows {
    const uint4* k;
    const uint4* v;
    uint4* kc;
    uint4* vc;
    const int32_t* slots;
    int32_t num_tokens, row_vecs;
    int64_t num_slots;
    uint32_t* status;
};

// The scatter over flat vector indices first, first + stride, ... (any split
// of the grid; the index is divided by the row length).
__device__ __forceinline__ void store_rows(const StoreRows& st, int64_t first, int64_t stride) {
    const int64_t total = (int64_t)st.num_tokens * st.row_vecs;
    for (int64_t idx = first; idx < total; idx += stride) {
        const int32_t t = (int32_t)(idx / st.row_vecs);
        const int32_t c = (int32_t)(idx - (int64_t)t * st.row_vecs);
        const int32_t s = __ldg(st.slots + t);
        if (s < 0) continue;
        if ((int64_t)s >= st.num_slots) {
            if (c == 0) report(st.status, PKV_STATUS_SLOT_OUT_OF_RANGE);
            continue;
        }
        const uint4 kv = ld_stream16(st.k + idx);
        const uint4 vv = ld_stream16(st.v + idx);
        const int64_t dst = (int64_t)s * st.row_vecs + c;
        st.kc[dst] = kv;
        st.vc[dst] = vv;
    }
}

// Two floats -> packed bf16x2 (round to nearest even), lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// D = A*B + D for one m16n8k16 bf16 tile with fp32 accumulation.
__device__ __forceinline__ void mma_bf16_16816(float d[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

constexpr float kLog2e = 1.4426950408889634f;

}  // namespace pkv

// Host side: per-device SM count (cached).
int pkv_num_sms();

// Checks pkv_kv_store's arguments and fills `st` (enqueues nothing); the
// return code is the one pkv_kv_store gives for them.  num_tokens == 0 passes.
int pkv_store_rows_args(const void* k, const void* v, void* k_cache, void* v_cache,
                        const int32_t* slot_mapping, int32_t num_tokens,
                        const pkv_cache_desc& cache, uint32_t* status, pkv::StoreRows& st);

// Polls a bounded in-kernel mbarrier wait makes before it gives up (the
// unwinding drains use their own, fixed limit).  pkv_set_wait_poll_limit
// changes it for calls enqueued afterwards.
uint32_t pkv_wait_polls();
