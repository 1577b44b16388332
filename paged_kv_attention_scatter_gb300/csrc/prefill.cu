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
// This file holds the tile scheduler shared by both prefill kernels, the
// entry point, and the general kernel (any block size, head_dim 64 or 128):
// FlashAttention-2-style tiles of 64 queries x 64 keys on mma.sync, four warps
// of 16 query rows, K/V tiles gathered row by row through the block table with
// cp.async into XOR-swizzled shared memory (double-buffered), ldmatrix
// fragments, online softmax in registers.  The tcgen05/TMA kernel in
// prefill_tc.cu takes over when the block size is a multiple of 128 and
// head_dim is 128.
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

// ---------------------------------------------------------------------------
// general kernel (mma.sync)
// ---------------------------------------------------------------------------
constexpr int kBM = 64, kBN = 64, kThreadsG = 128;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// 16-byte chunk cc of tile row r, XOR-swizzled so ldmatrix rows hit distinct banks
template <int CH>
__device__ __forceinline__ int swz(int r, int cc) {
    return r * CH + (cc ^ (r & 7));
}

template <int D>
__global__ void __launch_bounds__(kThreadsG) prefill_general_kernel(PrefillArgs a,
                                                                    int32_t slot_base) {
    constexpr int CH = D / 8;
    extern __shared__ uint4 smem[];
    uint4* sQ = smem;
    uint4* sK = sQ + kBM * CH;
    uint4* sV = sK + 2 * kBN * CH;

    asm volatile("griddepcontrol.wait;" ::: "memory");    // the plan's tile list
    const int h = blockIdx.x;
    const int32_t slot = slot_base + (int32_t)blockIdx.y;
    if (slot >= a.sched[0]) return;
    const int2 tile = a.tiles[slot];
    const int32_t b = tile.x, m = tile.y;
    int32_t q0, lq, lk;
    pkv::seq_lengths(a, b, q0, lq, lk, false);
    const int32_t c = lk - lq;
    const int32_t kvh = h / a.G;
    const int32_t row0 = m * kBM;
    const int32_t rows = min(kBM, lq - row0);
    const int32_t kv_limit = min(lk, c + row0 + kBM);
    const int32_t n_tiles = (kv_limit + kBN - 1) / kBN;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int32_t* bt_row = a.bt ? a.bt + (int64_t)b * a.MB : nullptr;

    // ---- Q tile ----
    for (int idx = tid; idx < kBM * CH; idx += kThreadsG) {
        const int r = idx / CH, cc = idx - r * CH;
        const bool ok = r < rows;
        const __nv_bfloat16* src =
            ok ? a.q + ((int64_t)(q0 + row0 + r) * a.Hq + h) * D + cc * 8 : a.q;
        cp_async16(smem_u32(sQ + swz<CH>(r, cc)), src, ok ? 16 : 0);
    }
    cp_async_commit();

    bool bad_block = false;
    auto load_kv = [&](int n, int st) {
        uint4* dk = sK + st * kBN * CH;
        uint4* dv = sV + st * kBN * CH;
        for (int idx = tid; idx < kBN * CH; idx += kThreadsG) {
            const int r = idx / CH, cc = idx - r * CH;
            const int32_t j = n * kBN + r;
            const __nv_bfloat16* ks = nullptr;
            const __nv_bfloat16* vs = nullptr;
            if (j < kv_limit) {
                if (j < c) {
                    const int32_t blk = bt_row[j / a.bs];
                    if ((unsigned)blk < (unsigned)a.NB) {
                        const int64_t off =
                            (((int64_t)blk * a.bs + j % a.bs) * a.Hkv + kvh) * D + cc * 8;
                        ks = a.kc + off;
                        vs = a.vc + off;
                    } else {
                        bad_block = true;
                    }
                } else {
                    const int64_t off = ((int64_t)(q0 + j - c) * a.Hkv + kvh) * D + cc * 8;
                    ks = a.k + off;
                    vs = a.v + off;
                }
            }
            cp_async16(smem_u32(dk + swz<CH>(r, cc)), ks ? ks : a.k, ks ? 16 : 0);
            cp_async16(smem_u32(dv + swz<CH>(r, cc)), vs ? vs : a.v, vs ? 16 : 0);
        }
    };
    load_kv(0, 0);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();

    // ---- Q fragments ----
    uint32_t qf[D / 16][4];
    {
        const int mi = lane >> 3, rr = lane & 7;
        const int r = warp * 16 + (mi & 1) * 8 + rr;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
            ldsm_x4(smem_u32(sQ + swz<CH>(r, 2 * kk + (mi >> 1))), qf[kk][0], qf[kk][1],
                    qf[kk][2], qf[kk][3]);
    }
    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m_i[2] = {-INFINITY, -INFINITY}, l_i[2] = {0.f, 0.f};
    const int32_t pos_lo = c + row0 + warp * 16 + g;     // query positions of rows g, g+8
    const int32_t pos_hi = pos_lo + 8;

    for (int n = 0; n < n_tiles; ++n) {
        if (n + 1 < n_tiles) {
            load_kv(n + 1, (n + 1) & 1);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const uint4* tk = sK + (n & 1) * kBN * CH;
        const uint4* tv = sV + (n & 1) * kBN * CH;
        float s[kBN / 8][4];
#pragma unroll
        for (int i = 0; i < kBN / 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
        {
            const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
                for (int np = 0; np < kBN / 16; ++np) {
                    const int r = np * 16 + (mi >> 1) * 8 + rr;
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(smem_u32(tk + swz<CH>(r, 2 * kk + (mi & 1))), b0, b1, b2, b3);
                    pkv::mma_bf16_16816(s[2 * np], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3],
                                        b0, b1);
                    pkv::mma_bf16_16816(s[2 * np + 1], qf[kk][0], qf[kk][1], qf[kk][2],
                                        qf[kk][3], b2, b3);
                }
            }
        }
        // ---- mask, online softmax (base 2) ----
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int nt = 0; nt < kBN / 8; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int32_t j = n * kBN + nt * 8 + 2 * t + (e & 1);
                const int32_t p = (e < 2) ? pos_lo : pos_hi;
                const float x = (j <= p && j < lk) ? s[nt][e] * a.scale_log2 : -INFINITY;
                s[nt][e] = x;
                mx[e >> 1] = fmaxf(mx[e >> 1], x);
            }
        }
        float alpha[2], muse[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
            const float mn = fmaxf(m_i[r], mx[r]);
            muse[r] = (mn == -INFINITY) ? 0.f : mn;
            alpha[r] = (m_i[r] == -INFINITY) ? 0.f : pkv::fast_exp2(m_i[r] - muse[r]);
            m_i[r] = mn;
            l_i[r] *= alpha[r];
        }
#pragma unroll
        for (int nt = 0; nt < kBN / 8; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float p = pkv::fast_exp2(s[nt][e] - muse[e >> 1]);
                s[nt][e] = p;
                l_i[e >> 1] += p;
            }
        }
#pragma unroll
        for (int i = 0; i < D / 8; ++i) {
            o[i][0] *= alpha[0]; o[i][1] *= alpha[0];
            o[i][2] *= alpha[1]; o[i][3] *= alpha[1];
        }
        // ---- O += P V ----
        {
            const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
            for (int kc = 0; kc < kBN / 16; ++kc) {
                const uint32_t a0 = pkv::pack_bf16(s[2 * kc][0], s[2 * kc][1]);
                const uint32_t a1 = pkv::pack_bf16(s[2 * kc][2], s[2 * kc][3]);
                const uint32_t a2 = pkv::pack_bf16(s[2 * kc + 1][0], s[2 * kc + 1][1]);
                const uint32_t a3 = pkv::pack_bf16(s[2 * kc + 1][2], s[2 * kc + 1][3]);
                const int r = kc * 16 + (mi & 1) * 8 + rr;
#pragma unroll
                for (int dp = 0; dp < D / 16; ++dp) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(smem_u32(tv + swz<CH>(r, 2 * dp + (mi >> 1))), b0, b1, b2, b3);
                    pkv::mma_bf16_16816(o[2 * dp], a0, a1, a2, a3, b0, b1);
                    pkv::mma_bf16_16816(o[2 * dp + 1], a0, a1, a2, a3, b2, b3);
                }
            }
        }
        __syncthreads();
    }
    if (bad_block) pkv::report(a.status, PKV_STATUS_BAD_BLOCK_ID);
    // ---- epilogue ----
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        l_i[r] += __shfl_xor_sync(0xffffffffu, l_i[r], 1);
        l_i[r] += __shfl_xor_sync(0xffffffffu, l_i[r], 2);
        l_i[r] = l_i[r] > 0.f ? 1.f / l_i[r] : 0.f;
    }
    const int r_lo = warp * 16 + g, r_hi = r_lo + 8;
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
        const int d = i * 8 + 2 * t;
        if (r_lo < rows)
            *reinterpret_cast<uint32_t*>(a.out + ((int64_t)(q0 + row0 + r_lo) * a.Hq + h) * D +
                                         d) = pkv::pack_bf16(o[i][0] * l_i[0], o[i][1] * l_i[0]);
        if (r_hi < rows)
            *reinterpret_cast<uint32_t*>(a.out + ((int64_t)(q0 + row0 + r_hi) * a.Hq + h) * D +
                                         d) = pkv::pack_bf16(o[i][2] * l_i[1], o[i][3] * l_i[1]);
    }
}

template <int D>
int launch_general(PrefillArgs& a, cudaStream_t s, const PrefillPrologue* pre) {
    const size_t smem = (size_t)(kBM + 4 * kBN) * (D / 8) * 16;
    static std::atomic<uint64_t> configured{0};
    if (!pkv_dynamic_smem_once((const void*)prefill_general_kernel<D>, (int)smem, configured))
        return PKV_ERR_CUDA;
    a.tile_m = kBM;
    a.tile_n = kBN;
    const int rc = pkv_launch_prefill_plan(a, s, pre);
    if (rc != PKV_OK) return rc;
    for (int32_t base = 0; base < a.max_tiles; base += 65535) {
        const int32_t n = a.max_tiles - base < 65535 ? a.max_tiles - base : 65535;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)a.Hq, (unsigned)n, 1);
        cfg.blockDim = dim3(kThreadsG, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = s;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, prefill_general_kernel<D>, a, base) != cudaSuccess)
            return PKV_ERR_CUDA;
    }
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace

PrefillLayout pkv_prefill_layout(int32_t batch, int32_t total_q) {
    PrefillLayout L{};
    // the smallest q tile of either kernel (64) bounds the tile count
    L.max_tiles = (int32_t)(((int64_t)total_q + kBM - 1) / kBM + batch);
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

// tcgen05 fast path (prefill_tc.cu): returns PKV_ERR_UNSUPPORTED when the
// shapes are not its own.
int pkv_prefill_tc_supported(const PrefillArgs& a, int head_dim);
int pkv_launch_prefill_tc(PrefillArgs& a, int head_dim, cudaStream_t s,
                         const PrefillPrologue* pre);

namespace {

}  // namespace

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
    if (pkv_prefill_tc_supported(a, head_dim) == PKV_OK)
        return pkv_launch_prefill_tc(a, head_dim, s, pre);
    return head_dim == 128 ? launch_general<128>(a, s, pre) : launch_general<64>(a, s, pre);
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
