// sample: temperature, softmax and Gumbel-max, one token per row.
//
// The uml.org.cn walk-through (§2.4 Model Runner) states the sampler as
// temperature, then softmax, then a Gumbel-max draw; "一个 prompt 的一生" §4
// applies it to each sequence's last-position logits.  With Exp(1) noise E
// supplied, the draw argmax_i softmax(x)_i / E_i (x = logits / T) equals
// argmax_i (x_i - ln E_i): softmax is a monotone map of x within a row and its
// normaliser is common to the row.  So one streaming pass per row suffices:
// no max, no exp, no sum -- each element costs one multiply, one log and one
// compare, and the row is read exactly once (8 bytes per vocabulary entry).
//
// Design: a thread-block cluster of up to 8 CTAs owns one row at a time (as
// many clusters as can be resident, each walking rows); each CTA scans a
// contiguous segment with 16-byte streaming loads, reduces its best
// (key, index) by warp shuffles and shared memory, and rank 0 of the cluster
// gathers the CTAs' results over distributed shared memory.  Ties keep the
// lowest index at every level, so the result does not depend on the split.
// No workspace and no second launch: the cluster barrier is a hardware
// barrier of co-scheduled CTAs, not a spin on memory.
//
// A second entry point draws the noise in the kernel instead of reading it:
// Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as
// easy as 1, 2, 3", SC 2011) keyed by a 64-bit seed, with counter
// (n / 4 as 64 bits, offset as 64 bits) for entry n = row * vocab + i, word
// n % 4 of the four outputs; U = (word / 2^8 + 1) / 2^24 in (0, 1] and
// E = -ln U.  The row then costs 4 bytes per entry instead of 8.
//
// There the two logarithms of the key, not the bytes, set the pace, so they
// are computed only for entries that can still matter.  The key
// x - ln(-ln U) grows with U, so an entry can reach a bound T0 only if
// U >= exp(-exp(x - T0)).  Taking T0 a little below the best key the warp has
// found so far, that threshold costs two fast exp2 evaluations; it is lowered
// by margins larger than its own error (about 1e-5 relative), and the word is
// compared with room for its float conversion, so the test never turns away
// an entry whose exact key reaches the warp's best.  Entries that pass get the
// exact key (the same float formula as with supplied noise), so the chosen
// token is the one the unfiltered computation picks.  After a row's first
// few entries almost none pass.
#include <cooperative_groups.h>
#include <math_constants.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace {

constexpr int kThreads = 256;
constexpr float kNoiseFloor = 1e-10f;

struct Cand {
    float key;
    int idx;
};

__device__ __forceinline__ void take_if_better(Cand& a, float key, int idx) {
    if (key > a.key || (key == a.key && idx < a.idx)) {
        a.key = key;
        a.idx = idx;
    }
}

__device__ __forceinline__ float gumbel_key(float logit, float inv_t, float e) {
    return logit * inv_t - __logf(fmaxf(e, kNoiseFloor));
}

// ---- Philox4x32-10 (the published round function and key schedule) ----
constexpr uint32_t kPhiloxM0 = 0xD2511F53u, kPhiloxM1 = 0xCD9E8D57u;
constexpr uint32_t kPhiloxW0 = 0x9E3779B9u, kPhiloxW1 = 0xBB67AE85u;

// Exp(1) noise from one Philox output word: U = (w / 2^8 + 1) / 2^24, E = -ln U.
// logf (not the fast log): U close to 1 gives a tiny E that needs relative accuracy.
__device__ __forceinline__ float exp_noise_of(uint32_t w) {
    const float u = (float)((w >> 8) + 1u) * 5.9604644775390625e-8f;   // 2^-24
    return -logf(u);
}

__device__ __forceinline__ uint32_t word_of(const uint4& w, int j) {
    return j == 0 ? w.x : j == 1 ? w.y : j == 2 ? w.z : w.w;
}

// The key schedule of one seed, computed once per thread: round r uses the
// seed's two words plus r times the Weyl increments.
struct PhiloxKeys {
    uint32_t k0[10], k1[10];
};

__device__ __forceinline__ PhiloxKeys philox_keys(uint64_t seed) {
    PhiloxKeys k;
    uint32_t a = (uint32_t)seed, b = (uint32_t)(seed >> 32);
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        // kept in registers (an opaque copy is not recomputed at each use,
        // which would cost an add per round and key)
        asm volatile("mov.b32 %0, %1;" : "=r"(k.k0[r]) : "r"(a));
        asm volatile("mov.b32 %0, %1;" : "=r"(k.k1[r]) : "r"(b));
        a += kPhiloxW0;
        b += kPhiloxW1;
    }
    return k;
}

// Philox4x32-10 of counter (n4 low, n4 high, offset low, offset high): each
// round multiplies words 0 and 2 by the two constants and mixes the products'
// high words with words 1 and 3 and the round key.
__device__ __forceinline__ uint4 philox_block_keys(uint64_t n4, uint64_t offset,
                                                   const PhiloxKeys& k) {
    uint4 c = make_uint4((uint32_t)n4, (uint32_t)(n4 >> 32), (uint32_t)offset,
                         (uint32_t)(offset >> 32));
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t hi0 = __umulhi(kPhiloxM0, c.x), lo0 = kPhiloxM0 * c.x;
        const uint32_t hi1 = __umulhi(kPhiloxM1, c.z), lo1 = kPhiloxM1 * c.z;
        c = make_uint4(hi1 ^ c.y ^ k.k0[r], lo1, hi0 ^ c.w ^ k.k1[r], lo0);
    }
    return c;
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Order-preserving map of floats (not NaN) to signed ints, and back.
__device__ __forceinline__ int ordered(float f) {
    const int i = __float_as_int(f);
    return i >= 0 ? i : i ^ 0x7fffffff;
}
__device__ __forceinline__ float unordered(int i) {
    return __int_as_float(i >= 0 ? i : i ^ 0x7fffffff);
}

constexpr float kLog2e = 1.4426950408889634f;
// The smallest noise term of any key: -ln E >= -ln(24 ln 2) = -2.8116 because
// U >= 2^-24 gives E = -ln U <= 24 ln 2.  Rounded up.
constexpr float kMinBonus = 2.8117f;

__device__ __forceinline__ float max4(const float4& v) {
    return fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
}
__device__ __forceinline__ uint32_t max4u(const uint4& w) {
    return max(max(w.x, w.y), max(w.z, w.w));
}

// The smallest Philox word with which an entry of scaled logit x (or any
// smaller one) may still reach a key T0, given a = (x - T0) * log2(e).
// Exactly: U >= thr = exp(-exp(x - T0)), and U = (w/2^8 + 1) / 2^24 makes that
// w >= thr * 2^32 - 256.  thr comes from two fast exp2 (relative error below
// 2e-5 wherever thr * 2^32 exceeds 512), is lowered by the factor 2^(-1/4096)
// (1.7e-4) and truncated to an integer, and 512 more is taken off (0 if that
// goes below 0), so the bound never exceeds the exact one.  An entry with a
// smaller x needs a larger U, so the bound of a block's largest x serves the
// whole block.  A NaN exponent gives 0 (every word passes: the exact key
// decides); +inf gives 0 as well.
__device__ __forceinline__ uint32_t reach_floor(float a) {
    const float z = fast_exp2(a);                                      // exp(x - T0)
    const float thr32 = fast_exp2(fmaf(z, -kLog2e, 32.0f - 1.0f / 4096.0f));
    uint32_t t;
    asm("cvt.rzi.sat.u32.f32 %0, %1;" : "=r"(t) : "f"(thr32));          // NaN -> 0
    return t > 512u ? t - 512u : 0u;
}

// The exact keys of the entries of one block whose word reaches `floor_w`
// (called behind a test that some word does, which is rare once a row's best
// has settled).
__device__ __forceinline__ void exact_block(Cand& best, const float4& l, const uint4& w,
                                            uint32_t floor_w, float inv_t, int i0) {
    const float lj[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
    for (int j = 0; j < 4; ++j)
        if (word_of(w, j) >= floor_w)
            take_if_better(best, gumbel_key(lj[j], inv_t, exp_noise_of(word_of(w, j))), i0 + j);
}

template <bool kPhilox>
__global__ void __launch_bounds__(kThreads, 8) sample_kernel(
        const float* __restrict__ logits, const float* __restrict__ temperatures,
        const float* __restrict__ noise, uint64_t seed, uint64_t offset, int32_t num_rows,
        int32_t vocab, bool vec_ok, int32_t* __restrict__ out, uint32_t* status) {
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int csize = (int)cluster.num_blocks();

    __shared__ float warp_key[kThreads / 32];
    __shared__ int warp_idx[kThreads / 32];
    __shared__ Cand cta_best[2];          // by row parity: one cluster barrier per row
    // in-kernel noise: the CTA's floor (an ordered int, see `ordered`) by row
    // parity; the slot of the next row is reset during this one, after the
    // last row that used it has passed its cluster barrier
    __shared__ int cta_floor[2];
    if (kPhilox && threadIdx.x < 2) cta_floor[threadIdx.x] = ordered(-CUDART_INF_F);
    __syncthreads();

    PhiloxKeys keys;
    if constexpr (kPhilox) keys = philox_keys(seed);
    // persistent: a cluster per resident slot walks rows blockIdx.y, +gridDim.y, ...
    int par = 0;
    for (int64_t row = blockIdx.y; row < num_rows; row += gridDim.y, par ^= 1) {
    if (kPhilox && threadIdx.x == 0) cta_floor[par ^ 1] = ordered(-CUDART_INF_F);
    const float temp = temperatures[row];
    const bool t_ok = isfinite(temp) && temp > 0.f;
    Cand best{-CUDART_INF_F, INT_MAX};
    if (t_ok) {
        const float inv_t = 1.0f / temp;
        const float* lrow = logits + row * vocab;
        const float* nrow = kPhilox ? nullptr : noise + row * vocab;
        // contiguous segment of this CTA, a multiple of 4 entries long
        int seg = (vocab + csize - 1) / csize;
        seg = (seg + 3) & ~3;
        const int lo = min(vocab, rank * seg);
        const int hi = min(vocab, lo + seg);
        const uint64_t n_row = (uint64_t)row * (uint64_t)vocab;
        if (vec_ok) {
            // rows start 16-byte aligned: lo is a multiple of 4 (and so is n_row)
            const int nvec = (hi - lo) >> 2;
            int v0 = threadIdx.x;
            if (!kPhilox) {
                // four vectors of logits and noise in flight per thread: all
                // loads issued before any key is compared
                for (; v0 + 3 * kThreads < nvec; v0 += 4 * kThreads) {
                    float4 l4[4], e4[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int i = lo + 4 * (v0 + u * kThreads);
                        l4[u] = pkv::ld_stream16f(lrow + i);
                        e4[u] = pkv::ld_stream16f(nrow + i);
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int i = lo + 4 * (v0 + u * kThreads);
                        take_if_better(best, gumbel_key(l4[u].x, inv_t, e4[u].x), i);
                        take_if_better(best, gumbel_key(l4[u].y, inv_t, e4[u].y), i + 1);
                        take_if_better(best, gumbel_key(l4[u].z, inv_t, e4[u].z), i + 2);
                        take_if_better(best, gumbel_key(l4[u].w, inv_t, e4[u].w), i + 3);
                    }
                }
            }
            if constexpr (kPhilox) {
                // One vector (4 entries) per lane and iteration: lane l of
                // warp w takes vectors 32w + l, + 256, ...; the trip count is
                // warp-uniform (the floor below is a warp-wide maximum).
                // Entry lo + 4v has Philox counter n4 = base4 + v.  Few
                // registers, so 8 CTAs fit per SM and their loads hide each
                // other's latency.
                //
                // The floor T0 an entry must reach is a lower bound on the
                // key of some entry that is (or will be) taken exactly: the
                // CTA's floor so far (each warp publishes its own through
                // shared memory), or x - kMinBonus for the largest scaled logit
                // x of this lane's block (every key is at least x - ln(24 ln 2),
                // as E <= 24 ln 2), lowered by margins for the float rounding
                // of either.  The entry that gives a bound always reaches it,
                // so it is taken.
                const int lane = threadIdx.x & 31;
                const float c1 = inv_t * kLog2e;
                const uint64_t base4 = (n_row + (uint64_t)lo) >> 2;
                float wfloor = -CUDART_INF_F;              // floor known to this warp
                int k = 0;                                 // iterations done
                for (int vb = threadIdx.x & ~31; vb < nvec; vb += kThreads, ++k) {
                    const int v = vb + lane;
                    const bool in = v < nvec;
                    float4 l4 = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (in) l4 = pkv::ld_stream16f(lrow + lo + 4 * v);
                    const uint4 w = philox_block_keys(base4 + (uint64_t)v, offset, keys);
                    const float m = in ? max4(l4) : -CUDART_INF_F;
                    const float x = m * inv_t;
                    const float own = x - (kMinBonus + 1e-4f * fabsf(x));
                    const float f = fmaxf(wfloor, own);         // NaN bounds are ignored
                    const float t0 = f - (1e-3f + 1e-4f * fabsf(f));
                    const uint32_t fw = reach_floor(fmaf(m, c1, -t0 * kLog2e));
                    if (in && max4u(w) >= fw) exact_block(best, l4, w, fw, inv_t, lo + 4 * v);
                    // a lane's own bound and best enter the floor at once;
                    // the warp and the CTA exchange theirs every 4 iterations
                    wfloor = fmaxf(wfloor, fmaxf(best.key, own));
                    if ((k & 3) == 3) {
                        const int wf = __reduce_max_sync(0xffffffffu, ordered(wfloor));
                        if (lane == 0) atomicMax(&cta_floor[par], wf);
                        wfloor = unordered(max(wf, *(volatile int*)&cta_floor[par]));
                    }
                }
            } else {
                for (int v = v0; v < nvec; v += kThreads) {
                    const int i = lo + 4 * v;
                    const float4 l4 = pkv::ld_stream16f(lrow + i);
                    const float4 e4 = pkv::ld_stream16f(nrow + i);
                    take_if_better(best, gumbel_key(l4.x, inv_t, e4.x), i);
                    take_if_better(best, gumbel_key(l4.y, inv_t, e4.y), i + 1);
                    take_if_better(best, gumbel_key(l4.z, inv_t, e4.z), i + 2);
                    take_if_better(best, gumbel_key(l4.w, inv_t, e4.w), i + 3);
                }
            }
            for (int i = lo + 4 * nvec + threadIdx.x; i < hi; i += kThreads) {
                const float e = kPhilox ? exp_noise_of(word_of(
                                              philox_block_keys((n_row + i) >> 2, offset, keys),
                                              (int)((n_row + i) & 3)))
                                        : nrow[i];
                take_if_better(best, gumbel_key(lrow[i], inv_t, e), i);
            }
        } else {
            for (int i = lo + threadIdx.x; i < hi; i += kThreads) {
                const float e = kPhilox ? exp_noise_of(word_of(
                                              philox_block_keys((n_row + i) >> 2, offset, keys),
                                              (int)((n_row + i) & 3)))
                                        : nrow[i];
                take_if_better(best, gumbel_key(lrow[i], inv_t, e), i);
            }
        }
    }
    // warp, then CTA
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float k2 = __shfl_xor_sync(0xffffffffu, best.key, off);
        const int i2 = __shfl_xor_sync(0xffffffffu, best.idx, off);
        take_if_better(best, k2, i2);
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        warp_key[warp] = best.key;
        warp_idx[warp] = best.idx;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        Cand c{warp_key[0], warp_idx[0]};
        for (int w = 1; w < kThreads / 32; ++w) take_if_better(c, warp_key[w], warp_idx[w]);
        cta_best[par] = c;
    }
    // every CTA's cta_best[par] is written; the slot is written again two rows
    // later, after the next barrier, which rank 0 reaches only once it has read it
    cluster.sync();
    if (rank == 0 && threadIdx.x == 0) {
        Cand c = cta_best[par];
        for (int r = 1; r < csize; ++r) {
            const Cand* other = cluster.map_shared_rank(&cta_best[par], r);
            take_if_better(c, other->key, other->idx);
        }
        int32_t tok = 0;
        if (!t_ok) {
            pkv::report(status, PKV_STATUS_BAD_TEMPERATURE);
        } else if (c.idx == INT_MAX) {
            pkv::report(status, PKV_STATUS_NO_FINITE_KEY);
        } else {
            tok = c.idx;
        }
        out[row] = tok;
    }
    }
    cluster.sync();                       // keep shared memory alive for rank 0
}

// Clusters of `csize` CTAs of sample_kernel<kPhilox> that fit on the current
// device at once, cached per device (65535 if the query fails).
template <bool kPhilox>
int resident_clusters(int csize) {
    static int cache[64][9] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
    int& n_res = cache[dev][csize];
    if (n_res == 0) {
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)csize;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)csize, 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, sample_kernel<kPhilox>, &cfg) != cudaSuccess ||
            n < 1) {
            cudaGetLastError();
            n = 65535;
        }
        n_res = n;
    }
    return n_res;
}

template <bool kPhilox>
int launch_sample(const float* logits, const float* temperatures, const float* exp_noise,
                  uint64_t seed, uint64_t offset, int32_t batch, int32_t vocab,
                  int32_t* out_token_ids, uint32_t* status, void* stream) {
    const bool vec_ok = (vocab % 4 == 0) &&
                        ((((uintptr_t)logits) | ((uintptr_t)exp_noise)) & 15) == 0;
    int csize;
    if (!kPhilox) {
        // reading the noise is bandwidth-bound: about 16K entries per CTA, at
        // most 8 CTAs per row
        csize = (vocab + 16383) / 16384;
        if (csize > 8) csize = 8;
        if (csize < 1) csize = 1;
    } else {
        // drawing it is arithmetic-bound, so a partial last wave of clusters
        // costs time in proportion: take a cluster size c (at most 8, at
        // least 4096 entries per CTA) with the fewest waves of row segments,
        // ceil(batch / resident clusters(c)) / c, and among those the middle
        // one: more CTAs per row pay more row ends (cluster barriers, start-up
        // latency), fewer leave SMs unevenly loaded.  (B=512 x V=151936, 8 CTAs
        // per SM: c = 2, 4 and 8 tie; measured 123, 113 and 132 us.)
        int c_max = (vocab + 4095) / 4096;
        if (c_max > 8) c_max = 8;
        if (c_max < 1) c_max = 1;
        int tied[8], n_tied = 0;
        double best = 1e30;
        for (int c = 1; c <= c_max; ++c) {
            const int n = resident_clusters<true>(c);
            const double cost = (double)((batch + n - 1) / n) / c;
            if (cost < best * (1.0 - 1e-9)) {
                best = cost;
                n_tied = 0;
            }
            if (cost <= best * (1.0 + 1e-9)) tied[n_tied++] = c;
        }
        csize = tied[(n_tied - 1) / 2];
    }
    const int n_res = resident_clusters<kPhilox>(csize);
    const int32_t clusters = batch < n_res ? batch : n_res;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)csize, (unsigned)clusters, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = (cudaStream_t)stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, sample_kernel<kPhilox>, logits, temperatures,
                                       exp_noise, seed, offset, batch, vocab, vec_ok,
                                       out_token_ids, status);
    if (e != cudaSuccess) return PKV_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace

extern "C" int pkv_sample(const float* logits, const float* temperatures,
                          const float* exp_noise, int32_t batch, int32_t vocab,
                          int32_t* out_token_ids, uint32_t* status, void* stream) {
    if (batch < 0 || vocab <= 0) return PKV_ERR_BAD_DIMENSION;
    if (batch == 0) return PKV_OK;
    if (!logits || !temperatures || !exp_noise || !out_token_ids) return PKV_ERR_NULL_POINTER;
    if (((uintptr_t)logits | (uintptr_t)temperatures | (uintptr_t)exp_noise |
         (uintptr_t)out_token_ids) & 3)
        return PKV_ERR_MISALIGNED;
    return launch_sample<false>(logits, temperatures, exp_noise, 0, 0, batch, vocab,
                                out_token_ids, status, stream);
}

extern "C" int pkv_sample_philox(const float* logits, const float* temperatures,
                                 uint64_t seed, uint64_t offset, int32_t batch, int32_t vocab,
                                 int32_t* out_token_ids, uint32_t* status, void* stream) {
    if (batch < 0 || vocab <= 0) return PKV_ERR_BAD_DIMENSION;
    if (batch == 0) return PKV_OK;
    if (!logits || !temperatures || !out_token_ids) return PKV_ERR_NULL_POINTER;
    if (((uintptr_t)logits | (uintptr_t)temperatures | (uintptr_t)out_token_ids) & 3)
        return PKV_ERR_MISALIGNED;
    return launch_sample<true>(logits, temperatures, nullptr, seed, offset, batch, vocab,
                               out_token_ids, status, stream);
}
