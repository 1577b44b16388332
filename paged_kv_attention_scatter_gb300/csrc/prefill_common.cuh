// Shared pieces of the varlen prefill kernels: arguments, the tile schedule.
#pragma once

#include "common.cuh"

namespace pkv {

constexpr int kPrefillTileQ = 128;    // queries per tile of the prefill kernel
constexpr int kPrefillTileK = 128;    // keys per tile

struct PrefillArgs {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    const __nv_bfloat16* kc;
    const __nv_bfloat16* vc;
    const int32_t* cu_q;
    const int32_t* cu_k;
    const int32_t* bt;               // may be null
    __nv_bfloat16* out;
    int32_t* sched;                  // [0]=tile count, [1]=dispatch counter, [2..3] spare
    int2* tiles;                     // (sequence, q tile) pairs, heaviest first
    int32_t B, total_q, max_sq, max_sk, Hq, Hkv, G, MB, NB, bs, max_tiles;
    int32_t tile_m, tile_n;          // tile shape the schedule is built for
    float scale_log2;
    uint32_t* status;
    int32_t skip_single;             // sequences of one query are left to the decode kernels
    uint32_t wait_polls;             // polls of a bounded mbarrier wait
};

// Lengths of sequence b; returns false (and reports) when they are inconsistent.
__device__ __forceinline__ bool seq_lengths(const PrefillArgs& a, int32_t b, int32_t& q0,
                                            int32_t& lq, int32_t& lk, bool report_bad) {
    q0 = a.cu_q[b];
    lq = a.cu_q[b + 1] - q0;
    lk = a.cu_k[b + 1] - a.cu_k[b];
    const int32_t c = lk - lq;
    bool ok = lq >= 0 && c >= 0 && q0 >= 0 && q0 + lq <= a.total_q;
    if (c > 0) ok = ok && a.bt != nullptr && (int64_t)(c + a.bs - 1) / a.bs <= a.MB;
    if (!ok && report_bad) report(a.status, PKV_STATUS_BAD_SEQLENS);
    return ok;
}

}  // namespace pkv

struct PrefillLayout {
    size_t off_sched, off_tiles, total;
    int32_t max_tiles;
};

PrefillLayout pkv_prefill_layout(int32_t batch, int32_t total_q);

// Work a fused entry point enqueues ahead of the prefill on the same stream
// (the chunk's kv_store).  The launchers run it after every host-side step
// that can fail, so a rejected call enqueues nothing.  When it launched a
// grid, the tile plan is launched as that grid's programmatic dependent and
// finishes only after it (the attention kernels wait for the plan).
struct PrefillPrologue {
    int (*enqueue)(void* ctx, bool* launched);
    void* ctx;
};

// Enqueues `pre` (may be null), then the tile plan.
int pkv_launch_prefill_plan(pkv::PrefillArgs& a, cudaStream_t s, const PrefillPrologue* pre);

// Checks pkv_paged_prefill_varlen's arguments and fills `a` (enqueues nothing),
// and enqueues `pre` (may be null) then the prefill of `a`; used by the entry
// points that add a kv_store or decode rows around a prefill.
int pkv_prefill_make_args(const void* q, const void* k, const void* v, const void* k_cache,
                          const void* v_cache, const int32_t* cu_seqlens_q,
                          const int32_t* cu_seqlens_k, int32_t batch, int32_t total_q,
                          int32_t max_seqlen_q, int32_t max_seqlen_k, int32_t num_q_heads,
                          const int32_t* block_tables, int32_t max_blocks_per_seq, float scale,
                          void* out, void* workspace, size_t workspace_bytes,
                          pkv_cache_desc cache, uint32_t* status, pkv::PrefillArgs& a);
int pkv_prefill_launch(pkv::PrefillArgs& a, int head_dim, cudaStream_t s,
                       const PrefillPrologue* pre);

namespace pkv {
// A kv_store to run as the prologue of a fused call (its arguments, as
// pkv_kv_store takes them).
struct StoreCall {
    const void* k;
    const void* v;
    void* k_cache;
    void* v_cache;
    const int32_t* slot_mapping;
    int32_t num_tokens;
    pkv_cache_desc cache;
    uint32_t* status;
    void* stream;
};
}  // namespace pkv

// PrefillPrologue::enqueue for a pkv::StoreCall.
int pkv_enqueue_store(void* store_call, bool* launched);
