// paged_prefill_varlen: causal prefill over a flattened varlen batch whose
// first tokens may already sit in the paged cache (prefix caching, chunked
// prefill).
//
// What it computes (uml.org.cn walk-through §2.4 / §3.2: the varlen prefill
// attention op with cu_seqlens_q/k and, for a cached prefix, block_tables;
// "一个 prompt 的一生" §3.1 and the Sequence walkthrough of "《Nano-vLLM源码逐行解析》
// 第2篇": a round computes num_scheduled_tokens tokens from num_cached_tokens):
// sequence b has Lq queries and Lk keys, c = Lk - Lq of them cached.  Query i
// sits at position c + i and attends keys j <= c + i; keys j < c are read
// from the cache through block_tables[b], keys j >= c are rows of this call's
// k / v.
//
// This file holds the tile scheduler (the plan kernel that lists the
// (sequence, q tile) pairs of a call, longest first), the argument checks and
// the entry points; the attention itself is the tcgen05 kernel of
// prefill_tc.cu (head_dim 64 or 128, any block size).
#include "prefill_common.cuh"

using pkv::PrefillArgs;

namespace {

constexpr int kBins = 4096;
constexpr int kPlanThreads = 1024;

// Lengths of the sequences base .. base+kPlanThreads-1 into shared memory, one
// sequence per thread (one load round trip for the whole group); lq = -1 marks
// a sequence that gets no tiles (inconsistent lengths, reported when `report`,
// or a one-query sequence left to the decode kernels).
__device__ __forceinline__ void load_lengths(const PrefillArgs& a, int32_t base, bool report,
                                             int32_t* s_lq, int32_t* s_lk) {
    const int32_t b = base + (int32_t)threadIdx.x;
    int32_t q0 = 0, lq = -1, lk = 0;
    if (b < a.B) {
        if (!pkv::seq_lengths(a, b, q0, lq, lk, report) || (a.skip_single && lq == 1)) {
            lq = -1;
        } else if (report && (lq > a.max_sq || lk > a.max_sk)) {
            pkv::report(a.status, PKV_STATUS_BAD_SEQLENS);
        }
    }
    s_lq[threadIdx.x] = lq;
    s_lk[threadIdx.x] = lk;
}

// One CTA: the (sequence, q tile) list ordered by decreasing number of key
// tiles (a counting sort), so the longest tiles start first.  Each pass reads
// the lengths of up to 1024 sequences at once, then a warp takes a sequence
// and its lanes the sequence's q tiles.  The main kernel is launched as a
// programmatic dependent and waits for this grid before reading the list.
__global__ void __launch_bounds__(kPlanThreads) prefill_plan_kernel(PrefillArgs a) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __shared__ int32_t hist[kBins];
    __shared__ int32_t warp_sums[32];
    __shared__ int32_t total;
    __shared__ int32_t s_lq[kPlanThreads], s_lk[kPlanThreads];
    for (int i = threadIdx.x; i < kBins; i += kPlanThreads) hist[i] = 0;
    if (threadIdx.x == 0) total = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    constexpr int nwarps = kPlanThreads / 32;
    for (int32_t base = 0; base < a.B; base += kPlanThreads) {
        load_lengths(a, base, true, s_lq, s_lk);
        __syncthreads();
        const int32_t nb = min(kPlanThreads, a.B - base);
        for (int32_t i = w; i < nb; i += nwarps) {
            const int32_t lq = s_lq[i], lk = s_lk[i];
            if (lq < 0) continue;
            const int32_t c = lk - lq;
            const int32_t nt = (lq + a.tile_m - 1) / a.tile_m;
            for (int32_t m = lane; m < nt; m += 32) {
                const int32_t lim = min(lk, c + (m + 1) * a.tile_m);
                const int32_t cost = min((lim + a.tile_n - 1) / a.tile_n, kBins - 1);
                atomicAdd(&hist[kBins - 1 - cost], 1);
            }
            if (lane == 0) atomicAdd(&total, nt);
        }
        __syncthreads();
    }
    // exclusive scan of hist: 4 bins per thread
    constexpr int per = kBins / kPlanThreads;
    int32_t local[per];
    int32_t sum = 0;
#pragma unroll
    for (int i = 0; i < per; ++i) {
        local[i] = hist[threadIdx.x * per + i];
        sum += local[i];
    }
    int32_t x = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) warp_sums[w] = x;
    __syncthreads();
    if (w == 0) {
        int32_t s = warp_sums[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, s, off);
            if (lane >= off) s += y;
        }
        warp_sums[lane] = s;
    }
    __syncthreads();
    int32_t run = x - sum + (w > 0 ? warp_sums[w - 1] : 0);
#pragma unroll
    for (int i = 0; i < per; ++i) {
        hist[threadIdx.x * per + i] = run;
        run += local[i];
    }
    __syncthreads();
    bool overflow = false;
    for (int32_t base = 0; base < a.B; base += kPlanThreads) {
        load_lengths(a, base, false, s_lq, s_lk);
        __syncthreads();
        const int32_t nb = min(kPlanThreads, a.B - base);
        for (int32_t i = w; i < nb; i += nwarps) {
            const int32_t lq = s_lq[i], lk = s_lk[i];
            if (lq < 0) continue;
            const int32_t c = lk - lq;
            const int32_t nt = (lq + a.tile_m - 1) / a.tile_m;
            for (int32_t m = lane; m < nt; m += 32) {
                const int32_t lim = min(lk, c + (m + 1) * a.tile_m);
                const int32_t cost = min((lim + a.tile_n - 1) / a.tile_n, kBins - 1);
                const int32_t pos = atomicAdd(&hist[kBins - 1 - cost], 1);
                if (pos < a.max_tiles) a.tiles[pos] = make_int2(base + i, m);
                else overflow = true;
            }
        }
        __syncthreads();
    }
    if (overflow) pkv::report(a.status, PKV_STATUS_WORKSPACE_OVERFLOW);
    if (threadIdx.x == 0) {
        a.sched[0] = min(total, a.max_tiles);
        a.sched[1] = 0;
    }
    // Launched after a store, the plan completes only once the store's writes
    // are visible, so the attention kernels' wait on the plan covers both.
    // Without a programmatic predecessor this returns at once.
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace

PrefillLayout pkv_prefill_layout(int32_t batch, int32_t total_q) {
    PrefillLayout L{};
    // sequence b has ceil(lq_b / 128) q tiles <= lq_b / 128 + 1
    L.max_tiles = (int32_t)(((int64_t)total_q + pkv::kPrefillTileQ - 1) / pkv::kPrefillTileQ +
                            batch);
    L.off_sched = 0;
    L.off_tiles = 256;
    L.total = (L.off_tiles + sizeof(int2) * (size_t)L.max_tiles + 255) & ~(size_t)255;
    return L;
}

int pkv_launch_prefill_plan(PrefillArgs& a, cudaStream_t s, const PrefillPrologue* pre) {
    bool chained = false;
    if (pre) {
        const int rc = pre->enqueue(pre->ctx, &chained);
        if (rc != PKV_OK) return rc;
    }
    if (!chained) {
        prefill_plan_kernel<<<1, kPlanThreads, 0, s>>>(a);
    } else {
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1, 1, 1);
        cfg.blockDim = dim3(kPlanThreads, 1, 1);
        cfg.stream = s;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, prefill_plan_kernel, a) != cudaSuccess) return PKV_ERR_CUDA;
    }
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

// The tcgen05 kernel (prefill_tc.cu).  PKV_ERR_UNSUPPORTED: head_dim other
// than 64 / 128, a pool of 2^31 rows or more, or no tensor-map encoder in the
// driver.
int pkv_prefill_tc_supported(const PrefillArgs& a, int head_dim);
int pkv_launch_prefill_tc(PrefillArgs& a, int head_dim, cudaStream_t s,
                         const PrefillPrologue* pre);

// Checks every argument and fills the kernel arguments; enqueues nothing.
int pkv_prefill_make_args(const void* q, const void* k, const void* v, const void* k_cache,
                      const void* v_cache, const int32_t* cu_seqlens_q,
                      const int32_t* cu_seqlens_k, int32_t batch, int32_t total_q,
                      int32_t max_seqlen_q, int32_t max_seqlen_k, int32_t num_q_heads,
                      const int32_t* block_tables, int32_t max_blocks_per_seq, float scale,
                      void* out, void* workspace, size_t workspace_bytes, pkv_cache_desc cache,
                      uint32_t* status, PrefillArgs& a) {
    if (batch < 0 || total_q < 0 || num_q_heads <= 0 || cache.num_kv_heads <= 0 ||
        max_seqlen_q < 0 || max_seqlen_k < 0)
        return PKV_ERR_BAD_DIMENSION;
    if (num_q_heads % cache.num_kv_heads != 0) return PKV_ERR_BAD_DIMENSION;
    if (!(scale > 0.f) || !isfinite(scale)) return PKV_ERR_BAD_DIMENSION;
    if (cache.head_dim != 64 && cache.head_dim != 128) return PKV_ERR_UNSUPPORTED_HEAD_DIM;
    if (block_tables && (max_blocks_per_seq <= 0 || cache.num_blocks <= 0 ||
                         cache.block_size <= 0))
        return PKV_ERR_BAD_DIMENSION;
    if (batch == 0 || total_q == 0) return PKV_OK;
    if (!q || !k || !v || !cu_seqlens_q || !cu_seqlens_k || !out || !workspace)
        return PKV_ERR_NULL_POINTER;
    if (block_tables && (!k_cache || !v_cache)) return PKV_ERR_NULL_POINTER;
    if (((uintptr_t)q | (uintptr_t)k | (uintptr_t)v | (uintptr_t)k_cache |
         (uintptr_t)v_cache | (uintptr_t)out | (uintptr_t)workspace) & 15)
        return PKV_ERR_MISALIGNED;
    if (((uintptr_t)cu_seqlens_q | (uintptr_t)cu_seqlens_k | (uintptr_t)block_tables) & 3)
        return PKV_ERR_MISALIGNED;
    const PrefillLayout L = pkv_prefill_layout(batch, total_q);
    if (workspace_bytes < L.total) return PKV_ERR_WORKSPACE_TOO_SMALL;
    char* ws = (char*)workspace;
    a.q = (const __nv_bfloat16*)q;
    a.k = (const __nv_bfloat16*)k;
    a.v = (const __nv_bfloat16*)v;
    a.kc = (const __nv_bfloat16*)k_cache;
    a.vc = (const __nv_bfloat16*)v_cache;
    a.cu_q = cu_seqlens_q;
    a.cu_k = cu_seqlens_k;
    a.bt = block_tables;
    a.out = (__nv_bfloat16*)out;
    a.sched = (int32_t*)(ws + L.off_sched);
    a.tiles = (int2*)(ws + L.off_tiles);
    a.B = batch;
    a.total_q = total_q;
    a.max_sq = max_seqlen_q;
    a.max_sk = max_seqlen_k;
    a.Hq = num_q_heads;
    a.Hkv = cache.num_kv_heads;
    a.G = num_q_heads / cache.num_kv_heads;
    a.MB = block_tables ? max_blocks_per_seq : 0;
    a.NB = cache.num_blocks;
    a.bs = cache.block_size > 0 ? cache.block_size : 1;
    a.max_tiles = L.max_tiles;
    a.scale_log2 = scale * pkv::kLog2e;
    a.status = status;
    a.skip_single = 0;
    a.wait_polls = pkv_wait_polls();
    return PKV_OK;
}

int pkv_prefill_launch(PrefillArgs& a, int head_dim, cudaStream_t s, const PrefillPrologue* pre) {
    const int rc = pkv_prefill_tc_supported(a, head_dim);
    if (rc != PKV_OK) return rc;
    return pkv_launch_prefill_tc(a, head_dim, s, pre);
}

int pkv_enqueue_store(void* ctx, bool* launched) {
    const pkv::StoreCall& c = *(const pkv::StoreCall*)ctx;
    *launched = c.num_tokens > 0;                 // an empty store launches nothing
    return pkv_kv_store(c.k, c.v, c.k_cache, c.v_cache, c.slot_mapping, c.num_tokens, c.cache,
                        c.status, c.stream);
}

extern "C" size_t pkv_paged_prefill_workspace_bytes(int32_t batch, int32_t total_q,
                                                    int32_t num_q_heads, pkv_cache_desc cache) {
    (void)num_q_heads;
    (void)cache;
    if (batch < 0 || total_q < 0) return 0;
    return pkv_prefill_layout(batch, total_q).total;
}

extern "C" int pkv_paged_prefill_varlen(
        const void* q, const void* k, const void* v, const void* k_cache, const void* v_cache,
        const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t batch,
        int32_t total_q, int32_t max_seqlen_q, int32_t max_seqlen_k, int32_t num_q_heads,
        const int32_t* block_tables, int32_t max_blocks_per_seq, float scale, void* out,
        void* workspace, size_t workspace_bytes, pkv_cache_desc cache, uint32_t* status,
        void* stream) {
    PrefillArgs a;
    const int rc = pkv_prefill_make_args(q, k, v, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k,
                                     batch, total_q, max_seqlen_q, max_seqlen_k, num_q_heads,
                                     block_tables, max_blocks_per_seq, scale, out, workspace,
                                     workspace_bytes, cache, status, a);
    if (rc != PKV_OK || batch == 0 || total_q == 0) return rc;
    return pkv_prefill_launch(a, cache.head_dim, (cudaStream_t)stream, nullptr);
}

extern "C" int pkv_kv_store_paged_prefill_varlen(
        const void* q, const void* k, const void* v, void* k_cache, void* v_cache,
        const int32_t* slot_mapping, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
        int32_t batch, int32_t total_q, int32_t max_seqlen_q, int32_t max_seqlen_k,
        int32_t num_q_heads, const int32_t* block_tables, int32_t max_blocks_per_seq,
        float scale, void* out, void* workspace, size_t workspace_bytes, pkv_cache_desc cache,
        uint32_t* status, void* stream) {
    PrefillArgs a;
    const int rc = pkv_prefill_make_args(q, k, v, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k,
                                     batch, total_q, max_seqlen_q, max_seqlen_k, num_q_heads,
                                     block_tables, max_blocks_per_seq, scale, out, workspace,
                                     workspace_bytes, cache, status, a);
    if (rc != PKV_OK) return rc;                              // nothing enqueued
    pkv::StoreCall store{k, v, k_cache, v_cache, slot_mapping, total_q, cache, status, stream};
    if (batch == 0 || total_q == 0) {
        bool launched = false;
        return pkv_enqueue_store(&store, &launched);
    }
    const PrefillPrologue pre{pkv_enqueue_store, &store};
    return pkv_prefill_launch(a, cache.head_dim, (cudaStream_t)stream, &pre);
}
