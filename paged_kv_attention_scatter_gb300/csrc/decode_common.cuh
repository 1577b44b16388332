// Declarations shared by the two paged_decode split kernels (paged_decode.cu:
// loads straight into registers, any block size; paged_decode_tma.cu: a TMA
// producer warp feeding a shared-memory ring, block sizes that are multiples
// of 64) and by the plan and combine kernels they share.
#pragma once

#include "common.cuh"

namespace pkv {

constexpr int kMaxGroup = 8;         // q heads per unit (mma rows 0..7)

struct DecodeArgs {
    const __nv_bfloat16* q;
    const __nv_bfloat16* kc;
    const __nv_bfloat16* vc;
    const int32_t* bt;
    const int32_t* ctx;
    __nv_bfloat16* out;
    int32_t* chunk_prefix;           // [B+1] exclusive prefix of chunk counts
    int4* chunk_info;                // [cap]: (sequence, first key, end key, chunks of it)
    float2* part_ml;                 // [cap * Hq]: (max, sum) in base 2
    float* part_o;                   // [cap * Hq * D]
    int32_t B, Hq, Hkv, G, n_hg, MB, NB, bs, max_ctx, chunk_keys, cap;
    float scale_log2;
    uint32_t* status;
    // A varlen batch (mixed prefill and decode): when cu_q is set, sequence b
    // is a decode row only if cu_q[b+1] - cu_q[b] == 1; its q and out row is
    // cu_q[b] and its context cu_k[b+1] - cu_k[b].  Other sequences get no
    // chunks and their out rows are left alone.
    const int32_t* cu_q;
    const int32_t* cu_k;
    int32_t total_q;                 // rows of q / out (varlen batch only)
    int32_t b0;                      // first sequence of a combine launch
    uint32_t wait_polls;             // polls of a bounded mbarrier wait
};

// q / out row of sequence b
__device__ __forceinline__ int64_t row_of(const DecodeArgs& a, int32_t b) {
    return a.cu_q != nullptr ? (int64_t)a.cu_q[b] : (int64_t)b;
}

__device__ __forceinline__ uint32_t word(const uint4& v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// pack (lo = element e of a, hi = element e of b), e in 0..7 of a 16-byte chunk
__device__ __forceinline__ uint32_t pair(const uint4& a, const uint4& b, int e) {
    return __byte_perm(word(a, e >> 1), word(b, e >> 1), (e & 1) ? 0x7632 : 0x5410);
}

__device__ __forceinline__ void allow_dependent_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void wait_for_predecessor() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace pkv

// The TMA split kernel (paged_decode_tma.cu).  `supported` returns PKV_OK when
// the shapes are its own; `launch` enqueues the split kernel only, as a
// programmatic dependent of the plan kernel.
int pkv_decode_tma_supported(const pkv::DecodeArgs& a, int head_dim);
int pkv_launch_decode_tma(pkv::DecodeArgs& a, int head_dim, cudaStream_t s);
