// paged_decode: split-KV (flash-decoding) attention for one query token per
// sequence, K/V read through a per-sequence block table.
//
// What it computes (uml.org.cn walk-through §2.4: the decode attention op over
// the paged cache with cache_seqlens and block_tables; §3.2 tensor formats):
// out[b,h] = sum_{j < ctx_b} softmax_j(scale * q[b,h] . K_j) V_j, where key j
// of sequence b is row j % bs of physical block block_tables[b][j / bs] and
// q head h reads kv head h / G (G = Hq / Hkv, grouped-query attention).
//
// Design for GB300 (HBM-bound: every cache byte is read once):
//  * Work unit = (sequence, kv head, group of <= 8 q heads, chunk of keys).  A
//    one-CTA plan kernel writes each sequence's chunk count as a prefix sum,
//    and one record per chunk (sequence, key range, chunk count), into the
//    workspace; the persistent main grid (SMs x resident CTAs) walks the
//    units round-robin, reading a unit's record with one load, so empty units
//    cost nothing and nothing depends on a host-side length (the launch is
//    graph-capturable).  Block sizes that are multiples of 64 take the TMA-fed
//    split kernel of paged_decode_tma.cu; this file's split kernel takes the
//    others.
//  * Inside a unit each of the 4 warps takes 16-key steps.  K and V rows are
//    loaded straight from HBM into mma.sync fragments with 16-byte loads (a
//    warp reads 8 rows x 64 B of K and 4 rows x 128 B of V per instruction):
//      S   = Q K^T   : M = the q heads of the group (rows 0..7 of m16), N = 8
//                      keys, K = head_dim.  The head_dim order of the K
//                      fragment is a fixed permutation applied to Q as well,
//                      so each thread loads contiguous 16-byte chunks.
//      O^T = V^T P^T : M = head_dim (16 per tile), N = the q heads, K = 16
//                      keys.  The S accumulator of two key tiles is exactly
//                      the P^T operand, so P never leaves registers; V's
//                      transpose is done by byte permutes of row pairs.
//    The dot products run on the tensor pipe, which keeps the kernel
//    memory-bound even for a group of 8 (8 flop per cache byte).
//  * Online softmax in base 2 with warp-shuffle row maxima; the 4 warps of a
//    CTA merge through shared memory; units of a sequence with more than one
//    chunk write (m, l, unnormalised o) to the workspace and a combine kernel
//    merges them.  A sequence with a single chunk is written directly.
//  * plan -> split -> combine are chained as programmatic dependent launches:
//    each kernel lets the next one launch as soon as it starts, and the next
//    one waits (griddepcontrol.wait) for its predecessor's results, so launch
//    latency is hidden.  (Folding the combine into the split kernel with
//    per-group tickets was measured slower: the ticket round trip per unit
//    stalls the K/V stream.)
//  * Keys past ctx_b are never loaded (their registers are zero and their
//    scores -inf), so NaN in unused cache slots cannot reach the output.
#include "decode_common.cuh"
#include "prefill_common.cuh"

namespace {

using pkv::DecodeArgs;
using pkv::kMaxGroup;
using pkv::allow_dependent_launch;
using pkv::pair;
using pkv::wait_for_predecessor;
using pkv::word;

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kStep = 16;            // keys per warp step

// The chunk schedule of one decode batch, written by one CTA of up to 1024
// threads: each sequence's chunk count as a prefix sum, and one record per
// chunk (sequence, key range, chunk count).
__device__ __forceinline__ void plan_body(const DecodeArgs& a) {
    __shared__ int32_t warp_sums[32];
    __shared__ int32_t carry;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    const int64_t cap_keys = (int64_t)a.MB * a.bs;
    for (int32_t base = 0; base < a.B; base += blockDim.x) {
        const int32_t b = base + threadIdx.x;
        int32_t n = 0;
        int32_t c = 0;
        if (b < a.B) {
            if (a.cu_q != nullptr) {
                // varlen batch: one-query rows only, with the prefill's checks
                // (query row inside q, at least its own key, blocks inside the table)
                const int32_t q0 = a.cu_q[b];
                c = a.cu_k[b + 1] - a.cu_k[b];
                if (a.cu_q[b + 1] - q0 == 1) {
                    if (q0 < 0 || q0 >= a.total_q || c < 1 || c > cap_keys || c > a.max_ctx)
                        pkv::report(a.status, PKV_STATUS_BAD_SEQLENS);
                    else
                        n = (c + a.chunk_keys - 1) / a.chunk_keys;
                }
            } else {
                c = a.ctx[b];
                if (c < 0 || c > cap_keys || c > a.max_ctx)
                    pkv::report(a.status, PKV_STATUS_BAD_CONTEXT_LEN);
                else
                    n = (c + a.chunk_keys - 1) / a.chunk_keys;
            }
        }
        // block-wide inclusive scan of n
        int32_t x = n;
        const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        if (lane == 31) warp_sums[w] = x;
        __syncthreads();
        if (w == 0) {
            int32_t s = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int32_t y = __shfl_up_sync(0xffffffffu, s, off);
                if (lane >= off) s += y;
            }
            warp_sums[lane] = s;
        }
        __syncthreads();
        const int32_t incl = x + (w > 0 ? warp_sums[w - 1] : 0) + carry;
        if (b < a.B) {
            a.chunk_prefix[b + 1] = incl;
            // one record per chunk: what the split kernels need to start it
            for (int32_t i = 0; i < n; ++i)
                a.chunk_info[incl - n + i] =
                    make_int4(b, i * a.chunk_keys, min(c, (i + 1) * a.chunk_keys), n);
        }
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) carry = incl;
        __syncthreads();
    }
    if (threadIdx.x == 0) a.chunk_prefix[0] = 0;
}

__global__ void __launch_bounds__(1024) decode_plan_kernel(DecodeArgs a) {
    allow_dependent_launch();
    plan_body(a);
}

// kv_store and the decode plan as one grid (pkv_kv_store_paged_decode): block
// 0 writes the chunk schedule while the other blocks store the step's K/V
// rows, so the pair costs one launch and the longer of the two.  The split
// kernel is this grid's programmatic dependent and waits for all of it, so it
// reads the stored rows.
__global__ void __launch_bounds__(1024) decode_store_plan_kernel(DecodeArgs a,
                                                                 pkv::StoreRows st) {
    allow_dependent_launch();
    if (blockIdx.x == 0) {
        plan_body(a);
        return;
    }
    pkv::store_rows(st, (int64_t)(blockIdx.x - 1) * blockDim.x + threadIdx.x,
                    (int64_t)(gridDim.x - 1) * blockDim.x);
}

template <int D>
__global__ void __launch_bounds__(kThreads) decode_split_kernel(DecodeArgs a) {
    constexpr int NQ = D / 32;       // 16-byte chunks per thread of a Q / K row
    constexpr int KK = D / 16;       // k-steps of S = Q K^T
    constexpr int MT = D / 16;       // m-tiles of O^T
    __shared__ float sm_m[kWarps][kMaxGroup];
    __shared__ float sm_l[kWarps][kMaxGroup];
    __shared__ float sm_o[kWarps][kMaxGroup][D];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    wait_for_predecessor();                  // the plan kernel's prefix sums
    allow_dependent_launch();                // after the wait: see the TMA kernel
    const int units_per_sc = a.Hkv * a.n_hg;
    const int32_t total_sc = a.chunk_prefix[a.B];
    const int64_t units = (int64_t)total_sc * units_per_sc;
    const bool fast_bs = (a.bs % kStep) == 0;
    const int64_t row_elems = (int64_t)a.Hkv * D;

    for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
        const int32_t sc = (int32_t)(u / units_per_sc);
        const int32_t rem = (int32_t)(u - (int64_t)sc * units_per_sc);
        const int32_t kvh = rem / a.n_hg, hg = rem - kvh * a.n_hg;
        // the plan's record of chunk slot sc: sequence, key range, chunk count
        const int4 info = a.chunk_info[sc];
        const int32_t b = info.x, key0 = info.y, key_end = info.z, nch = info.w;
        const int32_t h0 = kvh * a.G + hg * kMaxGroup;
        const int32_t nh = min(kMaxGroup, a.G - hg * kMaxGroup);
        const int32_t* bt_row = a.bt + (int64_t)b * a.MB;
        const __nv_bfloat16* kbase = a.kc + (int64_t)kvh * D;
        const __nv_bfloat16* vbase = a.vc + (int64_t)kvh * D;

        // Q fragment: row g = head h0+g, chunks i*4+t (the fixed head_dim order)
        uint4 qv[NQ];
#pragma unroll
        for (int i = 0; i < NQ; ++i) {
            qv[i] = make_uint4(0, 0, 0, 0);
            if (g < nh)
                qv[i] = *reinterpret_cast<const uint4*>(
                    a.q + (pkv::row_of(a, b) * a.Hq + h0 + g) * D + (i * 4 + t) * 8);
        }
        float o[MT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
        float m_run = -INFINITY, l_run = 0.f;
        bool bad_block = false;

        // Block sizes that are multiples of 16: one block-table entry covers a
        // warp step.  Others: lane l resolves key step + (l & 15) to its row
        // offset (-1 past the chunk or for a bad block id), one lookup and one
        // division per lane, and each fragment row is shuffled from the lane
        // that holds it (six lookups per lane were 20% slower at block size 8).
        auto lookup_row = [&](int32_t st) {
            const int32_t key = st + (lane & 15);
            int64_t row = -1;
            if (key < key_end) {
                const int32_t blk = bt_row[key / a.bs];
                if ((unsigned)blk < (unsigned)a.NB)
                    row = ((int64_t)blk * a.bs + key % a.bs) * row_elems;
                else
                    bad_block = true;
            }
            return row;
        };

        for (int32_t step = key0 + warp * kStep; step < key_end; step += kWarps * kStep) {
            // ---- row addresses (nullptr: not loaded, treated as masked) ----
            const __nv_bfloat16* krow[2];
            const __nv_bfloat16* vrow[4];
            const int vkey[4] = {step + 2 * t, step + 2 * t + 1, step + 2 * t + 8,
                                 step + 2 * t + 9};
            if (fast_bs) {
                const int32_t blk = bt_row[step / a.bs];
                const int32_t off = step % a.bs;
                const bool ok = (unsigned)blk < (unsigned)a.NB;
                bad_block |= !ok;
                const int64_t r0 = ((int64_t)blk * a.bs + off) * row_elems;
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int key = step + r * 8 + g;
                    krow[r] = (ok && key < key_end) ? kbase + r0 + (int64_t)(r * 8 + g) * row_elems
                                                    : nullptr;
                }
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    vrow[r] = (ok && vkey[r] < key_end)
                                  ? vbase + r0 + (int64_t)(vkey[r] - step) * row_elems
                                  : nullptr;
            } else {
                const int64_t row = lookup_row(step);
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int64_t rr = __shfl_sync(0xffffffffu, row, r * 8 + g);
                    krow[r] = rr >= 0 ? kbase + rr : nullptr;
                }
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int64_t rr = __shfl_sync(0xffffffffu, row, vkey[r] - step);
                    vrow[r] = rr >= 0 ? vbase + rr : nullptr;
                }
            }
            // ---- loads: K rows step+g, step+8+g; V rows 2t, 2t+1, 2t+8, 2t+9 ----
            uint4 kr[2][NQ];
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int i = 0; i < NQ; ++i)
                    kr[r][i] = krow[r] ? pkv::ld_stream16(krow[r] + (i * 4 + t) * 8)
                                       : make_uint4(0, 0, 0, 0);
            constexpr int VC = (D == 128) ? 2 : 1;          // chunks per V row
            uint4 vr[4][VC];
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c = 0; c < VC; ++c)
                    vr[r][c] = vrow[r] ? pkv::ld_stream16(vrow[r] + (g + 8 * c) * 8)
                                       : make_uint4(0, 0, 0, 0);
            // ---- S = Q K^T for two 8-key tiles ----
            float s[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
                for (int kk = 0; kk < KK; ++kk) {
                    const int i = kk >> 1, w0 = 2 * (kk & 1);
                    pkv::mma_bf16_16816(s[nt], word(qv[i], w0), 0u, word(qv[i], w0 + 1), 0u,
                                        word(kr[nt][i], w0), word(kr[nt][i], w0 + 1));
                }
            }
            // ---- online softmax (base 2) for head g over keys 2t,2t+1,8+2t,9+2t ----
            float x[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int nt = j >> 1, e = j & 1;
                x[j] = vrow[j] ? s[nt][e] * a.scale_log2 : -INFINITY;
            }
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
                    a0 = pair(vr[0][0], vr[1][0], mt);
                    a1 = pair(vr[0][VC - 1], vr[1][VC - 1], mt);
                    a2 = pair(vr[2][0], vr[3][0], mt);
                    a3 = pair(vr[2][VC - 1], vr[3][VC - 1], mt);
                } else {
                    a0 = pair(vr[0][0], vr[1][0], mt);
                    a1 = pair(vr[0][0], vr[1][0], 4 + mt);
                    a2 = pair(vr[2][0], vr[3][0], mt);
                    a3 = pair(vr[2][0], vr[3][0], 4 + mt);
                }
                pkv::mma_bf16_16816(o[mt], a0, a1, a2, a3, b0, b1);
            }
        }
        if (bad_block) pkv::report(a.status, PKV_STATUS_BAD_BLOCK_ID);

        // ---- per-warp results to shared memory ----
        l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
        l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
        if (t == 0) {
            sm_m[warp][g] = m_run;
            sm_l[warp][g] = l_run;
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            // O^T rows: d of fragment row g and row g+8 of m-tile mt
            const int d_lo = (D == 128) ? 8 * g + mt : 8 * g + mt;
            const int d_hi = (D == 128) ? 64 + 8 * g + mt : 8 * g + 4 + mt;
            sm_o[warp][2 * t][d_lo] = o[mt][0];
            sm_o[warp][2 * t + 1][d_lo] = o[mt][1];
            sm_o[warp][2 * t][d_hi] = o[mt][2];
            sm_o[warp][2 * t + 1][d_hi] = o[mt][3];
        }
        __syncthreads();
        // ---- merge the 4 warps: thread -> (head, d) ----
        for (int idx = threadIdx.x; idx < nh * D; idx += kThreads) {
            const int h = idx / D, d = idx - h * D;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w][h]);
            float L = 0.f, O = 0.f;
            if (M != -INFINITY) {
#pragma unroll
                for (int w = 0; w < kWarps; ++w) {
                    const float mw = sm_m[w][h];
                    if (mw == -INFINITY) continue;
                    const float f = pkv::fast_exp2(mw - M);
                    L += sm_l[w][h] * f;
                    O += sm_o[w][h][d] * f;
                }
            }
            const int64_t qh = pkv::row_of(a, b) * a.Hq + h0 + h;
            if (nch == 1) {
                a.out[qh * D + d] = __float2bfloat16_rn(L > 0.f ? O / L : 0.f);
            } else {
                const int64_t slot = (int64_t)sc * a.Hq + h0 + h;
                a.part_o[slot * D + d] = O;
                if (d == 0) a.part_ml[slot] = make_float2(M, L);
            }
        }
        __syncthreads();
    }
}

constexpr int kCombineBatch = 16;    // chunks whose partials are loaded at once
constexpr int kCombineHeads = 4;     // q heads per combine CTA, one warp each

// One warp per (sequence, q head); lane l owns head_dim elements
// [l*D/32, (l+1)*D/32).  The chunks' (max, sum) pairs and partial outputs of up
// to 16 chunks are loaded at once and merged online (base 2), so a sequence of
// up to 16 chunks costs one round trip; no block-wide reduction.
template <int D>
__global__ void __launch_bounds__(32 * kCombineHeads) decode_combine_kernel(DecodeArgs a) {
    constexpr int E = D / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int32_t h = blockIdx.x * kCombineHeads + warp, b = a.b0 + (int32_t)blockIdx.y;
    // The plan's prefix is final before this grid launches (the split kernels
    // allow it only after their own wait for the plan), so it is read ahead
    // of the wait for the split kernel's partials.
    const int32_t p0 = a.chunk_prefix[b], n = a.chunk_prefix[b + 1] - p0;
    wait_for_predecessor();                  // the split kernel's partials
    if (h >= a.Hq) return;
    if (n == 1) return;                                  // written by the split kernel
    if (n == 0 && a.cu_q != nullptr) return;             // not a decode row of a varlen batch
    const int d0 = lane * E;
    float M = -INFINITY, L = 0.f, O[E];
#pragma unroll
    for (int e = 0; e < E; ++e) O[e] = 0.f;
    for (int32_t c0 = 0; c0 < n; c0 += kCombineBatch) {
        const int cn = min(kCombineBatch, n - c0);
        float2 ml[kCombineBatch];
        float ov[kCombineBatch][E];
#pragma unroll
        for (int c = 0; c < kCombineBatch; ++c) {
            ml[c] = make_float2(-INFINITY, 0.f);
#pragma unroll
            for (int e = 0; e < E; ++e) ov[c][e] = 0.f;
            if (c < cn) {
                const int64_t slot = (int64_t)(p0 + c0 + c) * a.Hq + h;
                ml[c] = a.part_ml[slot];
                const float* po = a.part_o + slot * D + d0;
                if constexpr (E == 4) {
                    const float4 v = *reinterpret_cast<const float4*>(po);
                    ov[c][0] = v.x;
                    ov[c][1] = v.y;
                    ov[c][2] = v.z;
                    ov[c][3] = v.w;
                } else {
                    const float2 v = *reinterpret_cast<const float2*>(po);
                    ov[c][0] = v.x;
                    ov[c][1] = v.y;
                }
            }
        }
        float mb = M;
#pragma unroll
        for (int c = 0; c < kCombineBatch; ++c) mb = fmaxf(mb, ml[c].x);
        if (mb == -INFINITY) continue;                   // nothing visible yet
        const float r = (M == -INFINITY) ? 0.f : pkv::fast_exp2(M - mb);
        L *= r;
#pragma unroll
        for (int e = 0; e < E; ++e) O[e] *= r;
#pragma unroll
        for (int c = 0; c < kCombineBatch; ++c) {
            if (ml[c].x == -INFINITY) continue;
            const float f = pkv::fast_exp2(ml[c].x - mb);
            L += ml[c].y * f;
#pragma unroll
            for (int e = 0; e < E; ++e) O[e] += ov[c][e] * f;
        }
        M = mb;
    }
    __nv_bfloat16* dst = a.out + (pkv::row_of(a, b) * a.Hq + h) * D + d0;
#pragma unroll
    for (int e = 0; e < E; e += 2)
        *reinterpret_cast<uint32_t*>(dst + e) =
            pkv::pack_bf16(L > 0.f ? O[e] / L : 0.f, L > 0.f ? O[e + 1] / L : 0.f);
}

template <typename... Args>
cudaError_t launch_dependent(void (*kernel)(Args...), dim3 grid, dim3 block, cudaStream_t s,
                             Args... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Keys per work unit: the multiple of 64 nearest to the length that gives
// about 16 units per SM (of 152) for a typical context of half the stated
// maximum, within 64..1024; chosen from the sizes alone so the workspace
// query and the call agree.  Longer units cut the partial results and the
// per-unit merges, shorter ones keep the persistent grid's last round short.
// (Measured on decode-0.6b: powers of two only, 256-key chunks, 6188 GB/s;
// 320: 6287; 384: 6241; 448: 6357; 512: 5969.  The long workloads keep 1024.)
int32_t choose_chunk_keys(int32_t batch, int32_t units_per_seq_chunk, int32_t max_ctx) {
    const double typical = (double)max_ctx / 2.0;
    const double want_units = 16.0 * 152;
    const double keys = typical * (double)batch * (double)units_per_seq_chunk / want_units;
    int64_t chunk = (int64_t)(keys / 64.0 + 0.5) * 64;
    if (chunk < 64) chunk = 64;
    if (chunk > 1024) chunk = 1024;
    return (int32_t)chunk;
}

struct DecodeLayout {
    int32_t chunk_keys, cap;
    size_t off_prefix, off_info, off_ml, off_o, total;
};

DecodeLayout decode_layout(int32_t batch, int32_t num_q_heads, int32_t max_ctx,
                           const pkv_cache_desc& c) {
    DecodeLayout L{};
    const int32_t G = num_q_heads / (c.num_kv_heads > 0 ? c.num_kv_heads : 1);
    const int32_t n_hg = (G + kMaxGroup - 1) / kMaxGroup;
    L.chunk_keys = choose_chunk_keys(batch, c.num_kv_heads * n_hg, max_ctx);
    const int64_t per_seq = ((int64_t)max_ctx + L.chunk_keys - 1) / L.chunk_keys;
    L.cap = (int32_t)((int64_t)batch * per_seq);
    auto align = [](size_t x) { return (x + 255) & ~(size_t)255; };
    L.off_prefix = 0;
    L.off_info = align(L.off_prefix + sizeof(int32_t) * ((size_t)batch + 1));
    L.off_ml = align(L.off_info + sizeof(int4) * (size_t)L.cap);
    L.off_o = align(L.off_ml + sizeof(float2) * (size_t)L.cap * num_q_heads);
    L.total = align(L.off_o + sizeof(float) * (size_t)L.cap * num_q_heads * c.head_dim);
    return L;
}

// Resident CTAs per SM of the register-load split kernel, cached per device
// (occupancy depends on the device's limits, so a process driving GPUs of
// different kinds sizes each one's grid from its own answer).
template <int D>
int max_resident(const void* fn) {
    static int cached[64][2] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
    int& slot = cached[dev][D == 128 ? 1 : 0];
    if (slot <= 0) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kThreads, 0) != cudaSuccess ||
            n < 1)
            n = 1;
        slot = n;
    }
    return slot;
}

// How a decode's plan kernel is launched: on its own, in one grid with the
// step's kv_store (`store`), or not at all (a plan already in the workspace).
enum class PlanLaunch { kPlain, kWithStore, kNone };

template <int D>
int launch_decode(DecodeArgs& a, cudaStream_t s, PlanLaunch plan = PlanLaunch::kPlain,
                  const pkv::StoreRows* store = nullptr) {
    if (plan == PlanLaunch::kWithStore) {
        // one vector per thread and tensor, blocks of 1024, at most 2 per SM
        const int64_t vecs = (int64_t)store->num_tokens * store->row_vecs;
        int64_t blocks = (vecs + 1023) / 1024;
        const int64_t cap = 2LL * pkv_num_sms();
        if (blocks > cap) blocks = cap;
        if (blocks < 1) blocks = 1;
        decode_store_plan_kernel<<<(unsigned)(1 + blocks), 1024, 0, s>>>(a, *store);
    } else if (plan == PlanLaunch::kPlain) {
        decode_plan_kernel<<<1, 1024, 0, s>>>(a);
    }
    if (pkv_decode_tma_supported(a, D) == PKV_OK) {
        const int rc = pkv_launch_decode_tma(a, D, s);
        if (rc != PKV_OK) return rc;
    } else {
        const int per_sm = max_resident<D>((const void*)decode_split_kernel<D>);
        const int64_t upper = (int64_t)a.cap * a.Hkv * a.n_hg;
        int64_t grid = (int64_t)pkv_num_sms() * per_sm;
        if (grid > upper) grid = upper;
        if (grid < 1) grid = 1;
        if (launch_dependent(decode_split_kernel<D>, dim3((unsigned)grid), dim3(kThreads), s,
                             a) != cudaSuccess)
            return PKV_ERR_CUDA;
    }
    for (int32_t b0 = 0; b0 < a.B; b0 += 65535) {
        DecodeArgs sub = a;
        const int32_t rows = a.B - b0 < 65535 ? a.B - b0 : 65535;
        sub.b0 = b0;
        const unsigned hblocks = (unsigned)((a.Hq + kCombineHeads - 1) / kCombineHeads);
        if (launch_dependent(decode_combine_kernel<D>, dim3(hblocks, (unsigned)rows),
                             dim3(32 * kCombineHeads), s, sub) != cudaSuccess)
            return PKV_ERR_CUDA;
    }
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace

extern "C" size_t pkv_paged_decode_workspace_bytes(int32_t batch, int32_t num_q_heads,
                                                   int32_t max_context_len,
                                                   pkv_cache_desc cache) {
    if (batch < 0 || num_q_heads <= 0 || max_context_len < 0 || cache.num_kv_heads <= 0 ||
        cache.head_dim <= 0)
        return 0;
    return decode_layout(batch, num_q_heads, max_context_len, cache).total;
}

namespace {

// Checks what the plan depends on (context lengths, sizes, workspace) and
// fills the corresponding fields of `a`.
int make_plan_args(const int32_t* context_lens, int32_t batch, int32_t num_q_heads,
                   int32_t max_context_len, int32_t max_blocks_per_seq, void* workspace,
                   size_t workspace_bytes, const pkv_cache_desc& cache, uint32_t* status,
                   DecodeArgs& a) {
    if (batch < 0 || max_context_len < 0 || max_blocks_per_seq <= 0 || num_q_heads <= 0 ||
        cache.num_blocks <= 0 || cache.block_size <= 0 || cache.num_kv_heads <= 0)
        return PKV_ERR_BAD_DIMENSION;
    if (num_q_heads % cache.num_kv_heads != 0) return PKV_ERR_BAD_DIMENSION;
    if (cache.head_dim != 64 && cache.head_dim != 128) return PKV_ERR_UNSUPPORTED_HEAD_DIM;
    if (!context_lens || !workspace) return PKV_ERR_NULL_POINTER;
    if ((uintptr_t)workspace & 15) return PKV_ERR_MISALIGNED;
    if ((uintptr_t)context_lens & 3) return PKV_ERR_MISALIGNED;
    const DecodeLayout L = decode_layout(batch, num_q_heads, max_context_len, cache);
    if (workspace_bytes < L.total) return PKV_ERR_WORKSPACE_TOO_SMALL;
    char* ws = (char*)workspace;
    a.ctx = context_lens;
    a.chunk_prefix = (int32_t*)(ws + L.off_prefix);
    a.chunk_info = (int4*)(ws + L.off_info);
    a.part_ml = (float2*)(ws + L.off_ml);
    a.part_o = (float*)(ws + L.off_o);
    a.B = batch;
    a.Hq = num_q_heads;
    a.Hkv = cache.num_kv_heads;
    a.G = num_q_heads / cache.num_kv_heads;
    a.n_hg = (a.G + kMaxGroup - 1) / kMaxGroup;
    a.MB = max_blocks_per_seq;
    a.NB = cache.num_blocks;
    a.bs = cache.block_size;
    a.max_ctx = max_context_len;
    a.chunk_keys = L.chunk_keys;
    a.cap = L.cap;
    a.status = status;
    a.cu_q = nullptr;
    a.cu_k = nullptr;
    a.total_q = 0;
    a.b0 = 0;
    a.wait_polls = pkv_wait_polls();
    return PKV_OK;
}

// Checks the arguments and fills `a`; PKV_OK means the decode may be launched.
int make_decode_args(const void* q, const void* k_cache, const void* v_cache,
                     const int32_t* block_tables, int32_t max_blocks_per_seq,
                     const int32_t* context_lens, int32_t batch, int32_t num_q_heads,
                     int32_t max_context_len, float scale, void* out, void* workspace,
                     size_t workspace_bytes, const pkv_cache_desc& cache, uint32_t* status,
                     DecodeArgs& a) {
    if (batch < 0 || max_context_len < 0 || max_blocks_per_seq <= 0 || num_q_heads <= 0 ||
        cache.num_blocks <= 0 || cache.block_size <= 0 || cache.num_kv_heads <= 0)
        return PKV_ERR_BAD_DIMENSION;
    if (num_q_heads % cache.num_kv_heads != 0) return PKV_ERR_BAD_DIMENSION;
    if (cache.head_dim != 64 && cache.head_dim != 128) return PKV_ERR_UNSUPPORTED_HEAD_DIM;
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out || !workspace)
        return PKV_ERR_NULL_POINTER;
    if (((uintptr_t)q | (uintptr_t)k_cache | (uintptr_t)v_cache | (uintptr_t)out |
         (uintptr_t)workspace) & 15)
        return PKV_ERR_MISALIGNED;
    if (((uintptr_t)block_tables | (uintptr_t)context_lens) & 3) return PKV_ERR_MISALIGNED;
    const int rc = make_plan_args(context_lens, batch, num_q_heads, max_context_len,
                                  max_blocks_per_seq, workspace, workspace_bytes, cache, status,
                                  a);
    if (rc != PKV_OK) return rc;
    a.q = (const __nv_bfloat16*)q;
    a.kc = (const __nv_bfloat16*)k_cache;
    a.vc = (const __nv_bfloat16*)v_cache;
    a.bt = block_tables;
    a.out = (__nv_bfloat16*)out;
    a.scale_log2 = scale * pkv::kLog2e;
    return PKV_OK;
}

}  // namespace

extern "C" int pkv_paged_decode(const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* block_tables, int32_t max_blocks_per_seq,
                                const int32_t* context_lens, int32_t batch,
                                int32_t num_q_heads, int32_t max_context_len, float scale,
                                void* out, void* workspace, size_t workspace_bytes,
                                pkv_cache_desc cache, uint32_t* status, void* stream) {
    if (batch == 0 && max_context_len >= 0 && num_q_heads > 0) return PKV_OK;
    DecodeArgs a;
    const int rc = make_decode_args(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                    context_lens, batch, num_q_heads, max_context_len, scale, out,
                                    workspace, workspace_bytes, cache, status, a);
    if (rc != PKV_OK) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    return cache.head_dim == 128 ? launch_decode<128>(a, s) : launch_decode<64>(a, s);
}

extern "C" int pkv_paged_decode_plan(const int32_t* context_lens, int32_t batch,
                                     int32_t num_q_heads, int32_t max_context_len,
                                     int32_t max_blocks_per_seq, void* workspace,
                                     size_t workspace_bytes, pkv_cache_desc cache,
                                     uint32_t* status, void* stream) {
    if (batch == 0 && max_context_len >= 0 && num_q_heads > 0) return PKV_OK;
    DecodeArgs a{};
    const int rc = make_plan_args(context_lens, batch, num_q_heads, max_context_len,
                                  max_blocks_per_seq, workspace, workspace_bytes, cache, status,
                                  a);
    if (rc != PKV_OK) return rc;
    decode_plan_kernel<<<1, 1024, 0, (cudaStream_t)stream>>>(a);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" int pkv_paged_decode_run(const void* q, const void* k_cache, const void* v_cache,
                                    const int32_t* block_tables, int32_t max_blocks_per_seq,
                                    const int32_t* context_lens, int32_t batch,
                                    int32_t num_q_heads, int32_t max_context_len, float scale,
                                    void* out, void* workspace, size_t workspace_bytes,
                                    pkv_cache_desc cache, uint32_t* status, void* stream) {
    if (batch == 0 && max_context_len >= 0 && num_q_heads > 0) return PKV_OK;
    DecodeArgs a{};
    const int rc = make_decode_args(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                    context_lens, batch, num_q_heads, max_context_len, scale, out,
                                    workspace, workspace_bytes, cache, status, a);
    if (rc != PKV_OK) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    return cache.head_dim == 128 ? launch_decode<128>(a, s, PlanLaunch::kNone)
                                 : launch_decode<64>(a, s, PlanLaunch::kNone);
}

extern "C" int pkv_kv_store_paged_decode(
        const void* k, const void* v, const int32_t* slot_mapping, int32_t num_tokens,
        const void* q, void* k_cache, void* v_cache, const int32_t* block_tables,
        int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t batch,
        int32_t num_q_heads, int32_t max_context_len, float scale, void* out, void* workspace,
        size_t workspace_bytes, pkv_cache_desc cache, uint32_t* status, void* stream) {
    if (batch == 0 && max_context_len >= 0 && num_q_heads > 0)
        return pkv_kv_store(k, v, k_cache, v_cache, slot_mapping, num_tokens, cache, status,
                            stream);
    DecodeArgs a;
    int rc = make_decode_args(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                              context_lens, batch, num_q_heads, max_context_len, scale, out,
                              workspace, workspace_bytes, cache, status, a);
    if (rc != PKV_OK) return rc;                 // nothing enqueued
    pkv::StoreRows st;
    rc = pkv_store_rows_args(k, v, k_cache, v_cache, slot_mapping, num_tokens, cache, status,
                             st);
    if (rc != PKV_OK) return rc;                 // nothing enqueued
    cudaStream_t s = (cudaStream_t)stream;
    // the store and the plan in one grid (an empty store: the plan alone)
    const PlanLaunch plan = num_tokens > 0 ? PlanLaunch::kWithStore : PlanLaunch::kPlain;
    return cache.head_dim == 128 ? launch_decode<128>(a, s, plan, &st)
                                 : launch_decode<64>(a, s, plan, &st);
}

// ---------------------------------------------------------------------------
// Decode without a caller-provided workspace.
//
// For callers that cannot allocate device memory at the point of the call --
// for example a plugin inside a host engine that owns and budgets all device
// memory up front, or a latency-critical serving loop where cudaMalloc's
// implicit device-wide synchronisation is unacceptable -- this variant keeps
// the split-KV scratch in a fixed array compiled into the library.  Every GPU
// that loads the library holds the array until the process exits.
// ---------------------------------------------------------------------------
#include <mutex>

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[PKV_STATIC_DECODE_WORKSPACE_BYTES];

// Device address of g_decode_scratch on each device.  In host code the
// symbol's name is only a host-side handle, never a device address, so it is
// resolved with cudaGetSymbolAddress once per device while that device is
// current.
void* static_scratch_for_current_device(int* err) {
    static std::mutex mu;
    static void* ptr[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        *err = PKV_ERR_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) {
            *err = PKV_ERR_CUDA;
            return nullptr;
        }
        ptr[dev] = p;
    }
    return ptr[dev];
}

}  // namespace

extern "C" int pkv_paged_decode_static_workspace(
        const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
        int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t batch,
        int32_t num_q_heads, int32_t max_context_len, float scale, void* out,
        pkv_cache_desc cache, uint32_t* status, void* stream) {
    if (batch < 0 || max_context_len < 0 || max_blocks_per_seq <= 0 || num_q_heads <= 0 ||
        cache.num_blocks <= 0 || cache.block_size <= 0 || cache.num_kv_heads <= 0)
        return PKV_ERR_BAD_DIMENSION;
    if (num_q_heads % cache.num_kv_heads != 0) return PKV_ERR_BAD_DIMENSION;
    if (cache.head_dim != 64 && cache.head_dim != 128) return PKV_ERR_UNSUPPORTED_HEAD_DIM;
    if (batch == 0) return PKV_OK;
    const DecodeLayout L = decode_layout(batch, num_q_heads, max_context_len, cache);
    if (L.total > (size_t)PKV_STATIC_DECODE_WORKSPACE_BYTES) return PKV_ERR_WORKSPACE_TOO_SMALL;
    int err = PKV_OK;
    void* scratch = static_scratch_for_current_device(&err);
    if (scratch == nullptr) return err;
    return pkv_paged_decode(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                            batch, num_q_heads, max_context_len, scale, out, scratch,
                            (size_t)PKV_STATIC_DECODE_WORKSPACE_BYTES, cache, status, stream);
}

// ---------------------------------------------------------------------------
// Mixed prefill and decode batches (continuous batching).
//
// A step of a continuous-batching engine carries prefill chunks and decode
// rows in one varlen batch.  The causal varlen prefill computes every row
// correctly, but a one-query sequence would take a whole 128-query tile (and
// one CTA's worth of K/V streaming per head group); routing those rows to the
// split-KV decode kernels gives them the decode path's parallelism and
// bandwidth instead.  Order on the stream: the store, the prefill plan (its
// programmatic dependent) and kernel over the multi-query sequences, then the
// decode plan, split and combine over the one-query sequences.  The two sets
// of rows are disjoint, so neither pass touches the other's output.
// ---------------------------------------------------------------------------
namespace {

struct MixedLayout {
    size_t off_decode, total;
};

MixedLayout mixed_layout(int32_t batch, int32_t total_q, int32_t num_q_heads,
                         int32_t max_seqlen_k, const pkv_cache_desc& c) {
    MixedLayout L{};
    const size_t pre = pkv_paged_prefill_workspace_bytes(batch, total_q, num_q_heads, c);
    L.off_decode = (pre + 255) & ~(size_t)255;
    L.total = L.off_decode + decode_layout(batch, num_q_heads, max_seqlen_k, c).total;
    return L;
}

}  // namespace

extern "C" size_t pkv_paged_attention_varlen_workspace_bytes(int32_t batch, int32_t total_q,
                                                             int32_t num_q_heads,
                                                             int32_t max_seqlen_k,
                                                             pkv_cache_desc cache) {
    if (batch < 0 || total_q < 0 || num_q_heads <= 0 || max_seqlen_k < 0 ||
        cache.num_kv_heads <= 0 || cache.head_dim <= 0)
        return 0;
    return mixed_layout(batch, total_q, num_q_heads, max_seqlen_k, cache).total;
}

extern "C" int pkv_kv_store_paged_attention_varlen(
        const void* q, const void* k, const void* v, void* k_cache, void* v_cache,
        const int32_t* slot_mapping, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
        int32_t batch, int32_t total_q, int32_t max_seqlen_q, int32_t max_seqlen_k,
        int32_t num_q_heads, const int32_t* block_tables, int32_t max_blocks_per_seq,
        float scale, void* out, void* workspace, size_t workspace_bytes, pkv_cache_desc cache,
        uint32_t* status, void* stream) {
    pkv::PrefillArgs p;
    int rc = pkv_prefill_make_args(q, k, v, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, batch,
                                   total_q, max_seqlen_q, max_seqlen_k, num_q_heads,
                                   block_tables, max_blocks_per_seq, scale, out, workspace,
                                   workspace_bytes, cache, status, p);
    if (rc != PKV_OK) return rc;                              // nothing enqueued
    pkv::StoreCall store{k, v, k_cache, v_cache, slot_mapping, total_q, cache, status, stream};
    if (batch == 0 || total_q == 0) {
        bool launched = false;
        return pkv_enqueue_store(&store, &launched);
    }
    // one-query sequences read every key, their own included, from the cache
    if (!block_tables || !k_cache || !v_cache) return PKV_ERR_NULL_POINTER;
    const MixedLayout L = mixed_layout(batch, total_q, num_q_heads, max_seqlen_k, cache);
    if (workspace_bytes < L.total) return PKV_ERR_WORKSPACE_TOO_SMALL;
    DecodeArgs d{};
    // cu_seqlens_k stands in for context_lens in the checks; the plan reads
    // the lengths from cu_seqlens_q/k below.
    rc = make_decode_args(q, k_cache, v_cache, block_tables, max_blocks_per_seq, cu_seqlens_k,
                          batch, num_q_heads, max_seqlen_k, scale, out,
                          (char*)workspace + L.off_decode, L.total - L.off_decode, cache, status,
                          d);
    if (rc != PKV_OK) return rc;
    d.ctx = nullptr;
    d.cu_q = cu_seqlens_q;
    d.cu_k = cu_seqlens_k;
    d.total_q = total_q;
    p.skip_single = 1;
    cudaStream_t s = (cudaStream_t)stream;
    const PrefillPrologue pre{pkv_enqueue_store, &store};
    rc = pkv_prefill_launch(p, cache.head_dim, s, &pre);
    if (rc != PKV_OK) return rc;
    return cache.head_dim == 128 ? launch_decode<128>(d, s) : launch_decode<64>(d, s);
}
