// paged_decode split kernel fed by TMA (block sizes that are multiples of 64).
//
// Same computation and work units as the register-load split kernel in
// paged_decode.cu (uml.org.cn walk-through §2.4: decode attention through
// block_tables; a unit is (chunk of a sequence's keys, kv head, group of <= 8
// q heads)), with the K/V stream decoupled from the arithmetic:
//
//  * One CTA per SM, 5 warps.  Warp 4 is the producer: it walks this CTA's
//    units and, for each 64-key stage of a unit, waits for a free slot of a
//    ring in shared memory and issues TMA tile loads of the stage's K and V
//    rows (one kv head, 64 consecutive keys of one cache block; 128-byte
//    swizzle) plus, on a unit's first stage, a bulk copy of the unit's q rows.
//    It keeps the next unit's chunk record and block ids in flight while it
//    streams the current one, so the ring stays full across unit boundaries.
//  * Warps 0-3 consume: warp w takes keys 16w..16w+15 of every stage and runs
//    the same mma.sync fragments as the register kernel (S = Q K^T with a
//    permuted head_dim order, O^T = V^T P^T with P kept in registers), online
//    softmax in base 2.  A stage slot is released as soon as its rows have been
//    read.  At a unit's last stage the four warps merge through shared memory
//    (two mbarriers of the consumers only) while the producer keeps loading.
//  * Inside a warp's 16 keys, fragment key k sits at stage row
//    16w + (k ^ ((k & 1) << 2)): with the 128-byte swizzle this makes every
//    16-byte fragment load of K and of V free of shared-memory bank conflicts.
//  * Keys past a sequence's end are loaded (they are rows of the same cache
//    block) but their scores are -inf and their V registers are zero, so stale
//    or NaN cache contents never reach the output.  A block id outside the
//    pool masks its stage and sets PKV_STATUS_BAD_BLOCK_ID.
//  * Every wait on a barrier is bounded; on expiry the kernel sets
//    PKV_STATUS_WAIT_TIMEOUT and returns.  The producer leaves last: it waits
//    at a named barrier for the consumers to finish (normally or by giving
//    up), and when any role gave up it lets every copy it issued land before
//    the CTA can exit, since a consumer may give up after the producer has
//    issued its last stage.
#include <cudaTypedefs.h>

#include "decode_common.cuh"
#include "tc_utils.cuh"
#include "tma_host.cuh"

using pkv::DecodeArgs;
using pkv::kMaxGroup;

namespace {

namespace tc = pkv::tc;

constexpr int kStageKeys = 64;
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kTileBytes = kStageKeys * 128;      // 64 rows x 64 bf16 (one swizzle atom wide)

enum : int32_t { kFirst = 1, kLast = 2, kEnd = 4, kMasked = 8 };

struct StageMeta {
    int32_t b, key0, key_end, flags;   // key0: first key of the stage
    int32_t sc, h0, nh, nch;
};

template <int D>
struct Cfg {
    static constexpr int kHalves = D / 64;
    static constexpr int kStageBytes = 2 * kHalves * kTileBytes;    // K halves, then V halves
    static constexpr int kQBytes = kMaxGroup * D * 2;
    static constexpr int kStages = D == 128 ? 5 : 10;   // 5 x 32 KB measured faster than 6
};

template <int D>
struct DecodeSmem {
    uint8_t kv[Cfg<D>::kStages][Cfg<D>::kStageBytes];   // 1024-byte aligned tiles
    uint8_t qs[Cfg<D>::kStages][Cfg<D>::kQBytes];
    StageMeta meta[Cfg<D>::kStages];
    uint64_t full[Cfg<D>::kStages];
    uint64_t empty[Cfg<D>::kStages];
    uint64_t merge_full;                                // the four warps' partials written
    uint64_t merge_free;                                // ... and read by the merge
    float m[kConsumerWarps][kMaxGroup];
    float l[kConsumerWarps][kMaxGroup];
    float o[kConsumerWarps][kMaxGroup][D];
    int abort_flag;
};

__device__ __forceinline__ uint4 lds16(const uint8_t* p) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(tc::saddr(p)));
    return r;
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(tc::saddr(dst)), "l"(src), "r"(bytes), "r"(tc::saddr(bar))
        : "memory");
}

// Stage row of fragment key k (0..15) inside a warp's 16 rows.
__device__ __forceinline__ int key_row(int k) { return k ^ ((k & 1) << 2); }

// Byte offset of 16-byte chunk c (0..7) of row r in a 128-byte-swizzled tile.
__device__ __forceinline__ int swz(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

// q / out row of sequence b: b itself, or cu_q[b] in a varlen batch.  A
// template flag rather than a run-time test: the test alone, in the producer
// and the merge, cost the ordinary decode about 4%.
template <bool kVarlen>
__device__ __forceinline__ int64_t qrow_of(const DecodeArgs& a, int32_t b) {
    if constexpr (kVarlen) return (int64_t)a.cu_q[b];
    return (int64_t)b;
}

// kPolls: the waits take their poll limit from the arguments
// (pkv_set_wait_poll_limit) rather than the compile-time default, in
// instantiations of their own.
template <int D, bool kVarlen, bool kPolls>
__global__ void __launch_bounds__(kThreads, 1)
    decode_tma_kernel(const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, DecodeArgs a) {
    const uint32_t polls = kPolls ? a.wait_polls : (uint32_t)PKV_DEFAULT_WAIT_POLLS;
    using C = Cfg<D>;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    DecodeSmem<D>& sm = *reinterpret_cast<DecodeSmem<D>*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            tc::mbar_init(&sm.full[s], 1);
            tc::mbar_init(&sm.empty[s], kConsumerWarps);
        }
        tc::mbar_init(&sm.merge_full, kConsumerWarps * 32);
        tc::mbar_init(&sm.merge_free, kConsumerWarps * 32);
        sm.abort_flag = 0;
        tc::mbar_init_fence();
    }
    __syncthreads();
    pkv::wait_for_predecessor();                 // the plan kernel's chunk records
    // The combine may launch from here on: every CTA has seen the plan done,
    // so the combine can read the chunk prefix before its own wait.
    pkv::allow_dependent_launch();

    const int units_per_sc = a.Hkv * a.n_hg;
    const int64_t units = (int64_t)a.chunk_prefix[a.B] * units_per_sc;

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tc::tma_prefetch_desc(&kmap);
            tc::tma_prefetch_desc(&vmap);
        }
        int slot = 0;
        uint32_t phase = 0;
        int issued = 0;
        bool ok = true;
        int64_t u = blockIdx.x;
        int4 info_next = make_int4(0, 0, 0, 0);
        if (u < units) info_next = a.chunk_info[u / units_per_sc];
        while (u < units && ok) {
            const int32_t sc = (int32_t)(u / units_per_sc);
            const int32_t rem = (int32_t)(u - (int64_t)sc * units_per_sc);
            const int32_t kvh = rem / a.n_hg, hg = rem - kvh * a.n_hg;
            const int4 info = info_next;
            const int64_t un = u + gridDim.x;
            if (un < units) info_next = a.chunk_info[un / units_per_sc];
            const int32_t b = info.x, key0 = info.y, key_end = info.z, nch = info.w;
            const int32_t blk0 = key0 / a.bs;
            const int32_t nblk = (key_end - 1) / a.bs - blk0 + 1;
            const int32_t my_blk = lane < nblk ? a.bt[(int64_t)b * a.MB + blk0 + lane] : -1;
            const int32_t h0 = kvh * a.G + hg * kMaxGroup;
            const int32_t nh = min(kMaxGroup, a.G - hg * kMaxGroup);
            const int64_t qrow = qrow_of<kVarlen>(a, b);
            for (int32_t k = key0; k < key_end; k += kStageKeys) {
                if (!tc::mbar_wait(&sm.empty[slot], phase ^ 1, &sm.abort_flag, polls)) {
                    ok = false;
                    break;
                }
                const int32_t blk = __shfl_sync(0xffffffffu, my_blk, k / a.bs - blk0);
                if (lane == 0) {
                    const bool first = k == key0;
                    const bool good = (unsigned)blk < (unsigned)a.NB;
                    int32_t flags = (first ? kFirst : 0) |
                                    (k + kStageKeys >= key_end ? kLast : 0);
                    if (!good) {
                        flags |= kMasked;
                        pkv::report(a.status, PKV_STATUS_BAD_BLOCK_ID);
                    }
                    StageMeta& m = sm.meta[slot];
                    m.b = b;
                    m.key0 = k;
                    m.key_end = key_end;
                    m.flags = flags;
                    m.sc = sc;
                    m.h0 = h0;
                    m.nh = nh;
                    m.nch = nch;
                    const uint32_t bytes = (good ? (uint32_t)C::kStageBytes : 0u) +
                                           (first ? (uint32_t)(nh * D * 2) : 0u);
                    if (bytes == 0) {
                        tc::mbar_arrive(&sm.full[slot]);
                    } else {
                        tc::mbar_expect_tx(&sm.full[slot], bytes);
                        if (good) {
                            const int32_t row = blk * a.bs + (k % a.bs);
#pragma unroll
                            for (int h = 0; h < C::kHalves; ++h) {
                                tc::tma_load_3d(sm.kv[slot] + h * kTileBytes, &kmap,
                                                &sm.full[slot], h * 64, kvh, row);
                                tc::tma_load_3d(sm.kv[slot] + (C::kHalves + h) * kTileBytes,
                                                &vmap, &sm.full[slot], h * 64, kvh, row);
                            }
                        }
                        if (first)
                            bulk_load(sm.qs[slot], a.q + (qrow * a.Hq + h0) * D,
                                      (uint32_t)(nh * D * 2), &sm.full[slot]);
                    }
                }
                __syncwarp();
                ++issued;
                if (++slot == S) {
                    slot = 0;
                    phase ^= 1;
                }
            }
            u = un;
        }
        if (ok && tc::mbar_wait(&sm.empty[slot], phase ^ 1, &sm.abort_flag, polls)) {
            if (lane == 0) {
                sm.meta[slot].flags = kEnd;
                tc::mbar_arrive(&sm.full[slot]);
            }
            __syncwarp();
        } else {
            if (lane == 0) {
                sm.abort_flag = 1;
                pkv::report(a.status, PKV_STATUS_WAIT_TIMEOUT);
            }
        }
        // wait until the consumers are done (they arrive at barrier 1 on every
        // way out); if any role gave up, let every copy still in flight land
        // before the CTA can exit
        asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory");
        if (sm.abort_flag) {
            for (int i = 1; i <= min(issued, S); ++i) {
                int s = slot - i;
                uint32_t ph = phase;
                if (s < 0) {
                    s += S;
                    ph ^= 1;
                }
                tc::mbar_drain(&sm.full[s], ph);
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    constexpr int NQ = D / 32;       // 16-byte chunks per thread of a Q / K row
    constexpr int KK = D / 16;       // k-steps of S = Q K^T
    constexpr int MT = D / 16;       // m-tiles of O^T
    constexpr int VC = D == 128 ? 2 : 1;
    const int g = lane >> 2, t = lane & 3;
    int kr_row[2], v_row[4], v_key[4];
#pragma unroll
    for (int r = 0; r < 2; ++r) kr_row[r] = 16 * warp + key_row(8 * r + g);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        v_key[r] = 2 * t + (r & 1) + 8 * (r >> 1);
        v_row[r] = 16 * warp + key_row(v_key[r]);
    }

    uint4 qv[NQ];
    float o[MT][4];
    float m_run = -INFINITY, l_run = 0.f;
#pragma unroll
    for (int i = 0; i < NQ; ++i) qv[i] = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

    int slot = 0;
    uint32_t phase = 0;
    uint32_t merged = 0;                         // units merged so far
    while (true) {
        if (!tc::mbar_wait(&sm.full[slot], phase, &sm.abort_flag, polls)) {
            if (lane == 0) {
                sm.abort_flag = 1;
                pkv::report(a.status, PKV_STATUS_WAIT_TIMEOUT);
            }
            break;
        }
        const StageMeta st = sm.meta[slot];
        if (st.flags & kEnd) break;
        const uint8_t* kv = sm.kv[slot];
        if (st.flags & kFirst) {
            const uint8_t* qs = sm.qs[slot];
#pragma unroll
            for (int i = 0; i < NQ; ++i)
                qv[i] = g < st.nh ? lds16(qs + g * D * 2 + (i * 4 + t) * 16)
                                  : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
            m_run = -INFINITY;
            l_run = 0.f;
        }
        const int32_t lim = (st.flags & kMasked) ? 0 : st.key_end - st.key0;   // valid rows
        // ---- fragments from the stage: K rows of fragment keys g, 8+g ----
        uint4 kr[2][NQ];
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int i = 0; i < NQ; ++i) {
                const int j = i * 4 + t;
                kr[r][i] = lds16(kv + (j >> 3) * kTileBytes + swz(kr_row[r], j & 7));
            }
        bool valid[4];
        uint4 vr[4][VC];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            valid[r] = v_row[r] < lim;
#pragma unroll
            for (int c = 0; c < VC; ++c)
                vr[r][c] = valid[r] ? lds16(kv + (C::kHalves + c) * kTileBytes + swz(v_row[r], g))
                                    : make_uint4(0, 0, 0, 0);
        }
        // ---- S = Q K^T for two 8-key tiles ----
        float s[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < KK; ++kk) {
                const int i = kk >> 1, w0 = 2 * (kk & 1);
                pkv::mma_bf16_16816(s[nt], pkv::word(qv[i], w0), 0u, pkv::word(qv[i], w0 + 1),
                                    0u, pkv::word(kr[nt][i], w0), pkv::word(kr[nt][i], w0 + 1));
            }
        }
        // ---- online softmax (base 2) over fragment keys 2t, 2t+1, 8+2t, 9+2t ----
        float x[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) x[j] = valid[j] ? s[j >> 1][j & 1] * a.scale_log2 : -INFINITY;
        float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(m_run, mx);
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = (m_run == -INFINITY) ? 0.f : pkv::fast_exp2(m_run - m_use);
        float p[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) p[j] = pkv::fast_exp2(x[j] - m_use);
        l_run = l_run * alpha + (p[0] + p[1]) + (p[2] + p[3]);
        m_run = m_new;
        const float alpha_a = __shfl_sync(0xffffffffu, alpha, (2 * t) * 4);
        const float alpha_b = __shfl_sync(0xffffffffu, alpha, (2 * t + 1) * 4);
        const uint32_t b0 = pkv::pack_bf16(p[0], p[1]);
        const uint32_t b1 = pkv::pack_bf16(p[2], p[3]);
        // ---- O^T = V^T P^T ----
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            o[mt][0] *= alpha_a; o[mt][1] *= alpha_b;
            o[mt][2] *= alpha_a; o[mt][3] *= alpha_b;
            uint32_t a0, a1, a2, a3;
            if (D == 128) {
                a0 = pkv::pair(vr[0][0], vr[1][0], mt);
                a1 = pkv::pair(vr[0][VC - 1], vr[1][VC - 1], mt);
                a2 = pkv::pair(vr[2][0], vr[3][0], mt);
                a3 = pkv::pair(vr[2][VC - 1], vr[3][VC - 1], mt);
            } else {
                a0 = pkv::pair(vr[0][0], vr[1][0], mt);
                a1 = pkv::pair(vr[0][0], vr[1][0], 4 + mt);
                a2 = pkv::pair(vr[2][0], vr[3][0], mt);
                a3 = pkv::pair(vr[2][0], vr[3][0], 4 + mt);
            }
            pkv::mma_bf16_16816(o[mt], a0, a1, a2, a3, b0, b1);
        }
        // every register read from the slot has been consumed: release it
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&sm.empty[slot]);
        if (++slot == S) {
            slot = 0;
            phase ^= 1;
        }
        if (!(st.flags & kLast)) continue;

        // ---- end of a unit: merge the four warps (bounded mbarrier waits, so a
        // warp that gave up can never leave the others blocked) ----
        if (merged > 0 &&
            !tc::mbar_wait(&sm.merge_free, (merged - 1) & 1, &sm.abort_flag, polls)) {
            sm.abort_flag = 1;
            pkv::report(a.status, PKV_STATUS_WAIT_TIMEOUT);
            break;
        }
        float lr = l_run;
        lr += __shfl_xor_sync(0xffffffffu, lr, 1);
        lr += __shfl_xor_sync(0xffffffffu, lr, 2);
        if (t == 0) {
            sm.m[warp][g] = m_run;
            sm.l[warp][g] = lr;
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const int d_lo = 8 * g + mt;
            const int d_hi = (D == 128) ? 64 + 8 * g + mt : 8 * g + 4 + mt;
            sm.o[warp][2 * t][d_lo] = o[mt][0];
            sm.o[warp][2 * t + 1][d_lo] = o[mt][1];
            sm.o[warp][2 * t][d_hi] = o[mt][2];
            sm.o[warp][2 * t + 1][d_hi] = o[mt][3];
        }
        tc::mbar_arrive(&sm.merge_full);
        if (!tc::mbar_wait(&sm.merge_full, merged & 1, &sm.abort_flag, polls)) {
            sm.abort_flag = 1;
            pkv::report(a.status, PKV_STATUS_WAIT_TIMEOUT);
            break;
        }
        for (int idx = threadIdx.x; idx < st.nh * D; idx += kConsumerWarps * 32) {
            const int h = idx / D, d = idx - h * D;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, sm.m[w][h]);
            float L = 0.f, O = 0.f;
            if (M != -INFINITY) {
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) {
                    const float mw = sm.m[w][h];
                    if (mw == -INFINITY) continue;
                    const float f = pkv::fast_exp2(mw - M);
                    L += sm.l[w][h] * f;
                    O += sm.o[w][h][d] * f;
                }
            }
            const int64_t qh = qrow_of<kVarlen>(a, st.b) * a.Hq + st.h0 + h;
            if (st.nch == 1) {
                a.out[qh * D + d] = __float2bfloat16_rn(L > 0.f ? O / L : 0.f);
            } else {
                const int64_t pslot = (int64_t)st.sc * a.Hq + st.h0 + h;
                a.part_o[pslot * D + d] = O;
                if (d == 0) a.part_ml[pslot] = make_float2(M, L);
            }
        }
        tc::mbar_arrive(&sm.merge_free);
        ++merged;
    }
    // the consumers are done: let the producer check for copies in flight
    asm volatile("bar.arrive 1, %0;" ::"n"(kThreads) : "memory");
}

template <int D>
int launch(DecodeArgs& a, cudaStream_t s) {
    CUtensorMap kmap, vmap;
    const int64_t rows = (int64_t)a.NB * a.bs;
    if (!pkv::tma_encode_rows(&kmap, a.kc, rows, a.Hkv, D, kStageKeys) ||
        !pkv::tma_encode_rows(&vmap, a.vc, rows, a.Hkv, D, kStageKeys))
        return PKV_ERR_CUDA;
    const int smem = (int)sizeof(DecodeSmem<D>) + 1024;
    static std::atomic<uint64_t> configured[4] = {0, 0, 0, 0};
    const bool varlen = a.cu_q != nullptr;
    const bool custom = a.wait_polls != (uint32_t)PKV_DEFAULT_WAIT_POLLS;
    void (*kernel)(const CUtensorMap, const CUtensorMap, DecodeArgs) =
        varlen ? (custom ? decode_tma_kernel<D, true, true> : decode_tma_kernel<D, true, false>)
               : (custom ? decode_tma_kernel<D, false, true> : decode_tma_kernel<D, false, false>);
    if (!pkv_dynamic_smem_once((const void*)kernel, smem, configured[(varlen ? 2 : 0) + custom]))
        return PKV_ERR_CUDA;
    int64_t grid = pkv_num_sms();
    const int64_t upper = (int64_t)a.cap * a.Hkv * a.n_hg;
    if (grid > upper) grid = upper;
    if (grid < 1) grid = 1;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kernel, kmap, vmap, a) != cudaSuccess)
        return PKV_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace

int pkv_decode_tma_supported(const DecodeArgs& a, int head_dim) {
    if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (a.bs % kStageKeys != 0) return PKV_ERR_UNSUPPORTED;
    if ((int64_t)a.NB * a.bs >= (1LL << 31)) return PKV_ERR_UNSUPPORTED;
    if (a.chunk_keys % kStageKeys != 0) return PKV_ERR_UNSUPPORTED;
    if (pkv::tma_encode_fn() == nullptr) return PKV_ERR_UNSUPPORTED;
    return PKV_OK;
}

int pkv_launch_decode_tma(DecodeArgs& a, int head_dim, cudaStream_t s) {
    return head_dim == 128 ? launch<128>(a, s) : launch<64>(a, s);
}
