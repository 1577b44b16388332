// paged_prefill_varlen on the 5th-generation tensor cores: tcgen05.mma with
// TMEM accumulators, Q/K/V tiles staged by TMA (cached tiles gathered row by
// row with cp.async, in part or whole, when the block size is not a multiple
// of 128), for head_dim 128 or 64 and any block size.
//
// What it computes is stated in prefill.cu (causal varlen prefill over a
// prefix-cached paged cache, uml.org.cn walk-through §2.4 / §3.2).
//
// Work item = (sequence, 128-query tile, q head); the persistent grid takes
// items of the plan kernel's cost-sorted list dynamically (the producer warp
// draws the next index from a counter and hands it to the other roles
// through a small ring in shared memory), heads innermost, so the G heads of
// a kv group read the same K/V tiles out of L2 at about the same time.  The keys of a q tile are covered by
//   * cached tiles u = 0 .. ceil(c/128)-1: keys 128u .. 128u+127 of the
//     prefix, per half of head_dim one TMA box at row
//     block_tables[b][128u / bs] * bs + (128u % bs) of the pool when bs is a
//     multiple of 128.  For block sizes 8, 16, 32 and 64 the K tile is one
//     box per cache block (bs rows, stacked at row offsets that are multiples
//     of 8, the swizzle atom), and so are the first 96 (bs 16, 32) or 64
//     (bs 8, 64) rows of the V tile, whose other rows the V producer warp
//     gathers with 16-byte cp.async copies into the same swizzled layout: the
//     copy unit and the load path share the bytes.  For any other block size
//     both producer warps gather (keys past the prefix read zeros in every
//     mode).  Boxes for everything, or the gather for everything, measured
//     15-30% slower at 16..64, and a box below 8 rows would start inside a
//     swizzle atom;
//   * new tiles t = 0 .. m: the chunk's own k/v rows q0 + 128t ..; tile t == m
//     is the diagonal (causal mask col <= row), tiles t > m are never visible.
// Masked keys get -inf scores; V rows of masked cached keys are zeroed in
// shared memory because unused cache slots may hold NaN.
//
// Roles (256 threads, one CTA per SM):
//   warps 0-3  softmax: thread i owns query row i = TMEM lane i.  It loads S,
//              masks (diagonal and partial tiles only) and stores
//              P = exp2(S - m) as packed bf16 back into the first 64 columns of
//              the same S buffer; at the end it normalises O and writes it out
//              (32-byte stores when the output allows).  m is a running
//              row maximum: the first tile of an item takes its maximum first,
//              every later tile computes P against m straight away and is
//              redone -- maximum taken, m raised and O, l rescaled when it grew
//              by more than 2^8 -- only if its row sum passed 2^16.  The
//              exponent argument and the row sum use packed f32x2 instructions
//              (one per column pair).
//   warp 4     TMA producer (one thread): Q once per item, K tiles into a
//              three-stage ring, a stage refilled as soon as its Q K^T is done.
//   warp 7     TMA producer of the V tiles (one thread, three stages), a stage
//              refilled once its P V is done; on its own warp so that wait
//              never holds back a K tile.  When cached tiles are gathered,
//              all 32 lanes of warps 4 and 7 take part (K and V respectively;
//              with per-block boxes, lane u looks up block u and issues its
//              boxes; a V stage's barrier then expects the boxes' bytes and is
//              arrived once the gathered rows have landed).
//   warp 5     Q K^T issuer (one thread): S = Q K^T (both operands K-major in
//              shared memory) into one of three TMEM S buffers, running up to
//              two tiles ahead of the softmax; Q K^T into a buffer waits for
//              the P V that last read P from it.  Also owns TMEM.
//   warp 6     P V issuer (one thread): O += P V with P read from TMEM and V
//              MN-major in shared memory, as soon as the softmax has stored P.
//   Two issuers, because one thread that also waits on four barriers and
//   commits three times per tile leaves the tensor pipe idle between its
//   groups of MMAs (a 128x128x16 MMA takes 64 cycles when the pipe is fed);
//   with two, the waits of one overlap the MMAs of the other.  Descriptors are
//   built once: a later stage or K slice only adds a constant to the address
//   field.
// Keeping P in TMEM means shared memory only carries Q, K and V: an SS MMA of
// 128x128x16 already reads 128 bytes per clock from it.
// TMEM columns: S0 [0,128), S1 [128,256), S2 [256,384), O [384,512); stage,
// S buffer and the barriers of tile t all use index t % 3.  Every mbarrier wait
// is bounded; a wait that gives up sets PKV_STATUS_WAIT_TIMEOUT and the CTA
// unwinds: the issuers wait for their MMAs, and after the CTA's last barrier
// both producers (which may have finished normally) wait for every copy they
// issued -- Q, K and V -- to land before TMEM is freed and the CTA exits.
#include <cudaTypedefs.h>

#include "prefill_common.cuh"
#include "tc_utils.cuh"
#include "tma_host.cuh"

using pkv::PrefillArgs;
using namespace pkv::tc;

namespace {

constexpr int kBM = pkv::kPrefillTileQ;  // queries per tile
constexpr int kBN = pkv::kPrefillTileK;  // keys per tile
// head_dim D is 128 or 64: a tile is D/64 column blocks of 64 bf16 (one
// 128-byte swizzle atom wide), each 128 rows x 128 B
constexpr int kHalf = kBM * 128;         // one 64-column block of a tile
constexpr int kThreads = 256;
// How a cached 128-key tile reaches shared memory, by block size: one TMA box
// per 64-column block (a multiple of 128); K as one box per cache block and
// the first 64 (block sizes 8, 64) or 96 (16, 32) rows of V the same way, the
// rest of V gathered with cp.async, so the copy unit and the load path share
// the bytes; or both tensors gathered by the producer warps (any other block
// size).
constexpr int kLoadTile = 0, kLoadGather = 1, kLoadSplit64 = 2, kLoadSplit96 = 3;
constexpr int kStages = 3;               // K/V ring depth
constexpr int kItemRing = 4;             // work items handed from the producer to the others
constexpr int kItemReaders = 7;          // V producer, Q K^T and P V issuers, 4 softmax warps
constexpr uint32_t kColS0 = 0, kColO = 384;
constexpr float kRescaleThreshold = 8.0f;  // log2 of the tolerated growth
// A tile computed against the running maximum is redone (maximum taken, O and
// l rescaled) when its row sum of P passes 2^16, i.e. when some exponent may
// exceed 9; P stays below 2^16 otherwise, far inside the fp32 / bf16 range.
constexpr float kSumTrigger = 65536.0f;

template <int D>
struct __align__(1024) TcSmem {
    static constexpr int kTile = kBM * D * 2;     // bytes of one bf16 tile
    unsigned char q[kTile];
    unsigned char k[kStages][kTile];
    unsigned char v[kStages][kTile];
    uint64_t q_full, q_free;
    uint64_t k_full[kStages], v_full[kStages], k_empty[kStages], v_empty[kStages];
    uint64_t s_full[kStages], p_full[kStages], pv_done[kStages];
    uint64_t o_free, mma_done;
    uint64_t item_full[kItemRing], item_empty[kItemRing];
    int32_t item_ring[kItemRing];        // item index, or -1 when the CTA is done
    uint32_t tmem_base;
    int abort_flag;
};

struct TcMaps {
    CUtensorMap q, k, v, kc, vc;
};

struct Item {
    int32_t b, m, h, q0, lq, lk, c, n_cached, n_tiles, rows;
};

__device__ __forceinline__ Item item_at(const PrefillArgs& a, int64_t it) {
    Item x;
    const int32_t tile = (int32_t)(it / a.Hq);
    x.h = (int32_t)(it - (int64_t)tile * a.Hq);
    const int2 tm = a.tiles[tile];
    x.b = tm.x;
    x.m = tm.y;
    x.q0 = a.cu_q[x.b];
    x.lq = a.cu_q[x.b + 1] - x.q0;
    x.lk = a.cu_k[x.b + 1] - a.cu_k[x.b];
    x.c = x.lk - x.lq;
    x.n_cached = (x.c + kBN - 1) / kBN;
    x.n_tiles = x.n_cached + x.m + 1;
    x.rows = min(kBM, x.lq - x.m * kBM);
    return x;
}

// max(a, b, c) in one instruction (sm_100 and later).
__device__ __forceinline__ float max3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Packed pairs of fp32 (one 64-bit register pair): fma.rn.f32x2 and add.f32x2
// do two lanes' worth of work per instruction, each lane rounded as the scalar
// instruction would be.
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void up2(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// 32 bytes to global memory in one instruction (address 32-byte aligned).
__device__ __forceinline__ void st_global_32b(void* p, const uint32_t (&w)[8]) {
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(w[0]), "r"(w[1]),
                 "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

// All 32 lanes wait on the same barrier; the result is made warp-uniform so
// the warp-wide TMEM instructions that follow never see a diverged warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const int* abort_flag,
                                          uint32_t polls) {
    const bool r = mbar_wait(bar, parity, abort_flag, polls);
    return __all_sync(0xffffffffu, r);
}

// Item I of this CTA from the producer's ring (-1: no more).  A whole warp
// calls it when `warp_wide`, else one thread; the slot is released after the
// read.
template <class Smem>
__device__ __forceinline__ bool next_item(Smem& s, uint32_t I, int32_t& it, uint32_t polls,
                                          bool warp_wide = false) {
    const int qs = I % kItemRing;
    const uint32_t par = (I / kItemRing) & 1;
    const bool got = warp_wide ? warp_wait(&s.item_full[qs], par, &s.abort_flag, polls)
                               : mbar_wait(&s.item_full[qs], par, &s.abort_flag, polls);
    if (!got) return false;
    it = s.item_ring[qs];
    if (warp_wide) {
        __syncwarp();
        if ((threadIdx.x & 31) == 0) mbar_arrive(&s.item_empty[qs]);
    } else {
        mbar_arrive(&s.item_empty[qs]);
    }
    return true;
}

template <class Smem>
__device__ __forceinline__ void give_up(Smem& s, uint32_t* status) {
    s.abort_flag = 1;
    pkv::report(status, PKV_STATUS_WAIT_TIMEOUT);
}

// Where tile j of item x comes from (one TMA box per 64-column block at
// `row`): the chunk's own rows of k/v, or the pool row of key 128j through
// the block table (keys past the prefix, or a block id outside the pool, read
// the zeros TMA fills past the pool; the latter sets `bad`).  Returns whether
// it is a cached tile.
__device__ __forceinline__ bool tile_source(const PrefillArgs& a, const Item& x, int32_t j,
                                            int32_t& row, bool& bad) {
    if (j >= x.n_cached) {
        row = x.q0 + (j - x.n_cached) * kBN;
        return false;
    }
    const int32_t key0 = j * kBN;
    const int32_t blk = a.bt[(int64_t)x.b * a.MB + key0 / a.bs];
    row = a.NB * a.bs;                     // past the pool: TMA fills zeros
    if ((unsigned)blk < (unsigned)a.NB)
        row = blk * a.bs + key0 % a.bs;
    else
        bad = true;
    return true;
}

// One tile (K or V) into a stage: one box per 64-column block.
template <int D>
__device__ __forceinline__ void load_tile(unsigned char* dst, const CUtensorMap* map,
                                          uint64_t* bar, int kvh, int32_t row) {
    for (int hf = 0; hf < D / 64; ++hf)
        tma_load_3d(dst + hf * kHalf, map, bar, hf * 64, kvh, row);
}

// 16 bytes global -> shared with cp.async; `bytes` 0 writes zeros and reads
// nothing.
__device__ __forceinline__ void cp_async16_zfill(void* smem, const void* gmem, uint32_t bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(saddr(smem)), "l"(gmem),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int kPending>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(kPending) : "memory");
}

// Gathers cached tile j of item x (keys 128j .. 128j+127 of the prefix) of
// one pool (K or V) into a stage, each 16-byte chunk c of row r where a
// 128-byte-swizzled TMA box would put it (64-column block c/8, row r, chunk
// (c%8) ^ (r%8)).  Lane l resolves rows l, l+32, l+64, l+96 through the block
// table; then each warp instruction copies whole rows (D/8 consecutive lanes
// per row).  Keys past the prefix or in a block outside the pool read zeros;
// the latter set `bad`.  kG0 > 0 gathers only rows 32 kG0 .. 127.
template <int D, int kG0 = 0>
__device__ __forceinline__ void gather_cached_rows(const PrefillArgs& a, const Item& x, int32_t j,
                                                   int32_t kvh, const __nv_bfloat16* pool,
                                                   unsigned char* dst, int lane, bool& bad) {
    constexpr int kChunks = D / 8;              // 16-byte chunks of a row
    constexpr int kRowsPer = 32 / kChunks;      // rows one warp instruction covers
    int64_t src[kBN / 32];                      // element offset of the row, or -1
#pragma unroll
    for (int g = kG0; g < kBN / 32; ++g) {
        const int32_t key = j * kBN + g * 32 + lane;
        src[g] = -1;
        if (key < x.c) {
            const int32_t blk = a.bt[(int64_t)x.b * a.MB + key / a.bs];
            if ((unsigned)blk < (unsigned)a.NB)
                src[g] = (((int64_t)blk * a.bs + key % a.bs) * a.Hkv + kvh) * D;
            else
                bad = true;
        }
    }
    const int c = lane % kChunks, sub = lane / kChunks;
#pragma unroll
    for (int g = kG0; g < kBN / 32; ++g) {
#pragma unroll 4
        for (int i = 0; i < 32 / kRowsPer; ++i) {
            const int rl = i * kRowsPer + sub;
            const int64_t e = __shfl_sync(0xffffffffu, src[g], rl);
            const int r = g * 32 + rl;
            const uint32_t bytes = e >= 0 ? 16u : 0u;
            const int64_t eo = (e >= 0 ? e : 0) + c * 8;
            const int off = (c >> 3) * kHalf + r * 128 + (((c & 7) ^ (r & 7)) << 4);
            cp_async16_zfill(dst + off, pool + eo, bytes);
        }
    }
}

// kLoad: how cached tiles are loaded (see kLoadTile); the gather is an
// instantiation of its own so the one-box producer loops carry none of its
// code.  kPolls: the waits take their
// poll limit from the arguments (pkv_set_wait_poll_limit) instead of the
// compile-time default, in instantiations of their own (a run-time limit in
// the tight waits of the issuers cost the default kernel about 5%).
// Adds `bytes` to the transaction count of the barrier's current phase
// without arriving on it.
__device__ __forceinline__ void mbar_expect_tx_only(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(saddr(bar)),
                 "r"(bytes)
                 : "memory");
}

template <int D, int kLoad, bool kPolls>
__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(
        const __grid_constant__ TcMaps maps, const PrefillArgs a) {
    constexpr bool kGather = kLoad != kLoadTile;  // the producer warps' lanes gather
    // rows of a cached V tile loaded as per-block boxes (K: all of them)
    constexpr int kVBoxRows = kLoad == kLoadSplit64 ? 64 : kLoad == kLoadSplit96 ? 96 : 0;
    constexpr bool kBoxK = kVBoxRows > 0;
    const uint32_t polls = kPolls ? a.wait_polls : (uint32_t)PKV_DEFAULT_WAIT_POLLS;
    constexpr int kTile = TcSmem<D>::kTile;
    constexpr int kBlocks = D / 64;               // 64-column blocks of a tile
    extern __shared__ unsigned char smem_raw[];
    TcSmem<D>& s =
        *reinterpret_cast<TcSmem<D>*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        s.abort_flag = 0;
        mbar_init(&s.q_full, 1);
        mbar_init(&s.q_free, 1);
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&s.k_full[i], 1);
            mbar_init(&s.v_full[i], 1);
            mbar_init(&s.k_empty[i], 1);
            mbar_init(&s.v_empty[i], 1);
            mbar_init(&s.s_full[i], 1);
            mbar_init(&s.p_full[i], 4);
            mbar_init(&s.pv_done[i], 1);
        }
        mbar_init(&s.o_free, 128);
        for (int q = 0; q < kItemRing; ++q) {
            mbar_init(&s.item_full[q], 1);
            mbar_init(&s.item_empty[q], kItemReaders);
        }
        mbar_init(&s.mma_done, 2);
        mbar_init_fence();
    }
    if (warp == 5) tmem_alloc(&s.tmem_base, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s.tmem_base;
    asm volatile("griddepcontrol.wait;" ::: "memory");    // the plan's tile list
    const int64_t n_items = (int64_t)a.sched[0] * a.Hq;
    // copies issued by this producer (its lane 0, or with per-block boxes and
    // gathers any of its lanes), drained at the end through the barriers they
    // complete if any role gave up: tiles into the ring, and Q tiles
    uint32_t tiles_issued = 0, q_issued = 0;

    if (kGather && (warp == 4 || warp == 7)) {
        // ------------------------------------------------------ gather producers
        // Warp 4 takes K (and claims the items and loads Q), warp 7 takes V.
        // Each loads its tensor's tiles of the chunk's own rows by TMA (lane
        // 0).  Cached tiles: with per-block boxes (kVBoxRows > 0) K is all
        // boxes and V's first kVBoxRows rows too, lane u issuing block u's;
        // the rows left (all of them without boxes) are gathered with
        // cp.async by every lane, one commit group per tile.  A gathered
        // tile's barrier is arrived once its group has landed (wait_group,
        // then a proxy fence so the tensor core sees the writes, then lane 0
        // arrives), one tile behind the copies being issued so two tiles are
        // in flight; the boxes complete their bytes on the same barrier.
        const bool k_side = warp == 4;
        uint64_t* full = k_side ? s.k_full : s.v_full;
        uint64_t* empty = k_side ? s.k_empty : s.v_empty;
        const CUtensorMap* own = k_side ? &maps.k : &maps.v;
        const __nv_bfloat16* pool = k_side ? a.kc : a.vc;
        const bool boxes = kBoxK && k_side;     // cached K tiles as per-block boxes
        if (lane == 0) {
            if (k_side) tma_prefetch_desc(&maps.q);
            if (kBoxK) tma_prefetch_desc(k_side ? &maps.kc : &maps.vc);
            tma_prefetch_desc(own);
        }
        uint32_t& T = tiles_issued;               // tiles whose barriers will complete
        uint32_t I = 0;
        bool ok = true, bad_block = false;
        int pend = -1;                            // stage of a gathered tile in flight
        auto land = [&](int st_) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&full[st_]);
        };
        for (; ok; ++I) {
            int32_t it = 0;
            if (k_side) {
                const int qs = I % kItemRing;
                if (I >= kItemRing &&
                    !(ok = warp_wait(&s.item_empty[qs], (I / kItemRing - 1) & 1,
                                     &s.abort_flag, polls)))
                    break;
                if (lane == 0) {
                    it = atomicAdd(&a.sched[1], 1);
                    s.item_ring[qs] = it < n_items ? it : -1;
                    mbar_arrive(&s.item_full[qs]);
                }
                it = __shfl_sync(0xffffffffu, it, 0);
                if (it >= n_items) break;
            } else {
                if (!(ok = next_item(s, I, it, polls, true))) break;
                if (it < 0) break;
            }
            const Item x = item_at(a, it);
            const int32_t kvh = x.h / a.G;
            if (k_side) {
                if (I > 0 && !(ok = warp_wait(&s.q_free, (I - 1) & 1, &s.abort_flag, polls)))
                    break;
                if (lane == 0) {
                    mbar_expect_tx(&s.q_full, kTile);
                    for (int hf = 0; hf < kBlocks; ++hf)
                        tma_load_3d(s.q + hf * kHalf, &maps.q, &s.q_full, hf * 64, x.h,
                                    x.q0 + x.m * kBM);
                }
                ++q_issued;
            }
            for (int32_t j = 0; j < x.n_tiles; ++j, ++T) {
                const int st = T % kStages;
                const uint32_t use = T / kStages;
                if (use > 0 && !(ok = warp_wait(&empty[st], (use - 1) & 1, &s.abort_flag, polls)))
                    break;
                unsigned char* dst = k_side ? s.k[st] : s.v[st];
                if (boxes && j < x.n_cached) {
                    // lane u resolves cache block u of the tile (128 / bs of
                    // them, each a box of bs rows stacked at row u * bs, an
                    // 8-row swizzle atom boundary); keys past the prefix, or a
                    // block id outside the pool, read the zeros past the pool
                    const int nbox = kBN / a.bs;
                    int32_t my_row = a.NB * a.bs;
                    if (lane < nbox) {
                        const int32_t key = j * kBN + lane * a.bs;
                        if (key < x.c) {
                            const int32_t blk = a.bt[(int64_t)x.b * a.MB + key / a.bs];
                            if ((unsigned)blk < (unsigned)a.NB)
                                my_row = blk * a.bs;
                            else
                                bad_block = true;
                        }
                    }
                    if (lane == 0) mbar_expect_tx(&full[st], kTile);
                    __syncwarp();
                    if (lane < nbox)                  // each lane its own block's boxes
                        for (int hf = 0; hf < kBlocks; ++hf)
                            tma_load_3d(dst + hf * kHalf + lane * a.bs * 128, &maps.kc,
                                        &full[st], hf * 64, kvh, my_row);
                } else if (kBoxK && j < x.n_cached) {
                    // V: rows 0 .. kVBoxRows-1 as per-block boxes (the barrier
                    // expects their bytes, the gathered rows' arrival completes
                    // it), the rest gathered
                    const int nbox = kVBoxRows / a.bs;
                    int32_t my_row = a.NB * a.bs;
                    if (lane < nbox) {
                        const int32_t key = j * kBN + lane * a.bs;
                        if (key < x.c) {
                            const int32_t blk = a.bt[(int64_t)x.b * a.MB + key / a.bs];
                            if ((unsigned)blk < (unsigned)a.NB)
                                my_row = blk * a.bs;
                            else
                                bad_block = true;
                        }
                    }
                    if (lane == 0) mbar_expect_tx_only(&full[st], (uint32_t)(kVBoxRows * D * 2));
                    __syncwarp();
                    if (lane < nbox)
                        for (int hf = 0; hf < kBlocks; ++hf)
                            tma_load_3d(dst + hf * kHalf + lane * a.bs * 128, &maps.vc,
                                        &full[st], hf * 64, kvh, my_row);
                    gather_cached_rows<D, kVBoxRows / 32>(a, x, j, kvh, pool, dst, lane,
                                                          bad_block);
                    cp_async_commit();
                    if (pend >= 0) {
                        cp_async_wait<1>();
                        land(pend);
                    }
                    pend = st;
                } else if (j < x.n_cached) {
                    gather_cached_rows<D>(a, x, j, kvh, pool, dst, lane, bad_block);
                    cp_async_commit();
                    if (pend >= 0) {
                        cp_async_wait<1>();          // the tile before this one has landed
                        land(pend);
                    }
                    pend = st;
                } else {
                    // cached tiles come first in an item: the last one lands now
                    if (pend >= 0) {
                        cp_async_wait<0>();
                        land(pend);
                        pend = -1;
                    }
                    if (lane == 0) {
                        const int32_t row = x.q0 + (j - x.n_cached) * kBN;
                        mbar_expect_tx(&full[st], kTile);
                        for (int hf = 0; hf < kBlocks; ++hf)
                            tma_load_3d(dst + hf * kHalf, own, &full[st], hf * 64, kvh, row);
                    }
                }
            }
        }
        // copies still in flight land, and complete their barriers, before
        // anything else (on every way out)
        if (pend >= 0) {
            cp_async_wait<0>();
            land(pend);
        }
        if (__any_sync(0xffffffffu, bad_block) && lane == 0)
            pkv::report(a.status, PKV_STATUS_BAD_BLOCK_ID);
        if (!ok && lane == 0) give_up(s, a.status);
    } else if (warp == 4) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&maps.q);
            tma_prefetch_desc(&maps.k);
            tma_prefetch_desc(&maps.v);
            if (a.bt) {
                tma_prefetch_desc(&maps.kc);
                tma_prefetch_desc(&maps.vc);
            }
            uint32_t& T = tiles_issued;
            uint32_t I = 0;
            bool ok = true, bad_block = false;
            for (; ok; ++I) {
                // the next item of the cost-sorted list, taken dynamically so
                // the CTAs finish together; the other roles read it from the ring
                const int qs = I % kItemRing;
                if (I >= kItemRing &&
                    !(ok = mbar_wait(&s.item_empty[qs], (I / kItemRing - 1) & 1,
                            &s.abort_flag, polls)))
                    break;
                const int32_t it = atomicAdd(&a.sched[1], 1);
                s.item_ring[qs] = it < n_items ? it : -1;
                mbar_arrive(&s.item_full[qs]);
                if (it >= n_items) break;
                const Item x = item_at(a, it);
                const int32_t kvh = x.h / a.G;
                if (I > 0 && !(ok = mbar_wait(&s.q_free, (I - 1) & 1,
                        &s.abort_flag, polls))) break;
                mbar_expect_tx(&s.q_full, kTile);
                for (int hf = 0; hf < kBlocks; ++hf)
                    tma_load_3d(s.q + hf * kHalf, &maps.q, &s.q_full, hf * 64, x.h,
                                x.q0 + x.m * kBM);
                ++q_issued;
                for (int32_t j = 0; j < x.n_tiles; ++j, ++T) {
                    const int st = T % kStages;
                    const uint32_t use = T / kStages;
                    if (use > 0 && !(ok = mbar_wait(&s.k_empty[st], (use - 1) & 1,
                            &s.abort_flag, polls)))
                        break;
                    int32_t row;
                    const bool cached = tile_source(a, x, j, row, bad_block);
                    mbar_expect_tx(&s.k_full[st], kTile);
                    load_tile<D>(s.k[st], cached ? &maps.kc : &maps.k, &s.k_full[st], kvh, row);
                }
            }
            if (bad_block) pkv::report(a.status, PKV_STATUS_BAD_BLOCK_ID);
            if (!ok) give_up(s, a.status);
        }
    } else if (warp == 7) {
        // ------------------------------------------------------------ V producer
        // V tiles on their own thread: a V stage waits for its P V, and in
        // the producer's loop that wait held back the next K tile
        if (lane == 0) {
            uint32_t& T = tiles_issued;
            uint32_t I = 0;
            bool ok = true, bad_block = false;
            for (; ok; ++I) {
                int32_t it = -1;
                if (!(ok = next_item(s, I, it, polls))) break;
                if (it < 0) break;
                const Item x = item_at(a, it);
                const int32_t kvh = x.h / a.G;
                for (int32_t j = 0; j < x.n_tiles; ++j, ++T) {
                    const int st = T % kStages;
                    const uint32_t use = T / kStages;
                    if (use > 0 && !(ok = mbar_wait(&s.v_empty[st], (use - 1) & 1,
                            &s.abort_flag, polls)))
                        break;
                    int32_t row;
                    const bool cached = tile_source(a, x, j, row, bad_block);
                    mbar_expect_tx(&s.v_full[st], kTile);
                    load_tile<D>(s.v[st], cached ? &maps.vc : &maps.v, &s.v_full[st], kvh, row);
                }
            }
            if (!ok) give_up(s, a.status);
        }
    } else if (warp == 5 || warp == 6) {
        // ------------------------------------------------------------ MMA issuers
        // warp 5 issues Q K^T, warp 6 issues P V: the barrier waits of one
        // overlap the MMAs of the other, so the tensor pipe stays fed
        if (lane == 0) {
            const uint32_t id_qk = umma_idesc_bf16(kBM, kBN, false);
            const uint32_t id_pv = umma_idesc_bf16(kBM, D, true);
            const uint64_t qd0 = umma_desc_sw128(saddr(s.q), 16, 1024);
            const uint64_t kd0 = umma_desc_sw128(saddr(s.k[0]), 16, 1024);
            const uint64_t vd0 = umma_desc_sw128(saddr(s.v[0]), kHalf, 1024);
            uint32_t T = 0, I = 0;
            bool ok = true;
            for (; ok; ++I) {
                int32_t it = -1;
                if (!(ok = next_item(s, I, it, polls))) break;
                if (it < 0) break;
                const Item x = item_at(a, it);
                if (warp == 5) {
                    if (!(ok = mbar_wait(&s.q_full, I & 1, &s.abort_flag, polls))) break;
                    for (int32_t j = 0; j < x.n_tiles; ++j) {
                        const uint32_t t = T + j;
                        const int st = t % kStages;
                        if (!(ok = mbar_wait(&s.k_full[st], (t / kStages) & 1,
                                &s.abort_flag, polls))) break;
                        // the S buffer still holds P of tile t-3 until its P V is done
                        if (t >= kStages &&
                            !(ok = mbar_wait(&s.pv_done[st], (t / kStages - 1) & 1,
                                    &s.abort_flag, polls)))
                            break;
                        tc_fence_after();
                        const uint64_t kd = kd0 + (uint64_t)(st * (kTile >> 4));
                        const uint32_t d_s = tmem + kColS0 + st * kBN;
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint32_t off = ((kk >> 2) * kHalf + (kk & 3) * 32) >> 4;
                            umma_bf16(d_s, qd0 + off, kd + off, id_qk, kk > 0);
                        }
                        umma_commit(&s.s_full[st]);
                        umma_commit(&s.k_empty[st]);      // K stage free once Q K^T is done
                    }
                    if (!ok) break;
                    umma_commit(&s.q_free);              // every Q K^T of the item issued
                } else {
                    for (int32_t j = 0; j < x.n_tiles; ++j) {
                        const uint32_t t = T + j;
                        const int st = t % kStages;
                        if (!(ok = mbar_wait(&s.p_full[st], (t / kStages) & 1,
                                &s.abort_flag, polls))) break;
                        if (j == 0 && I > 0 && !(ok = mbar_wait(&s.o_free, (I - 1) & 1,
                                &s.abort_flag, polls)))
                            break;
                        if (!(ok = mbar_wait(&s.v_full[st], (t / kStages) & 1,
                                &s.abort_flag, polls))) break;
                        tc_fence_after();
                        const uint64_t vd = vd0 + (uint64_t)(st * (kTile >> 4));
                        const uint32_t a_p = tmem + kColS0 + st * kBN;
                        const uint32_t acc0 = j > 0 ? 1u : 0u;
#pragma unroll
                        for (int kk = 0; kk < kBN / 16; ++kk)
                            umma_bf16_tmem_a(tmem + kColO, a_p + kk * 8, vd + (kk * 2048 >> 4), id_pv,
                                             kk > 0 ? 1u : acc0);
                        umma_commit(&s.pv_done[st]);
                        umma_commit(&s.v_empty[st]);
                    }
                    if (!ok) break;
                }
                T += x.n_tiles;
            }
            if (!ok) give_up(s, a.status);
            // every MMA of both issuers has finished before TMEM is freed
            umma_commit(&s.mma_done);
            mbar_drain(&s.mma_done, 0);
        }
    } else {
        // ------------------------------------------------------------ softmax
        const int i = tid;                          // query row == TMEM lane
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        uint32_t T = 0, I = 0;
        bool ok = true;
        for (; ok; ++I) {
            int32_t it = -1;
            if (!(ok = next_item(s, I, it, polls, true))) break;
            if (it < 0) break;
            const Item x = item_at(a, it);
            float m_run = -INFINITY, l_run = 0.f;
            for (int32_t j = 0; j < x.n_tiles && ok; ++j) {
                const uint32_t t = T + j;
                const int st = t % kStages;
                const uint32_t s_col = lane_base + kColS0 + st * kBN;
                if (!(ok = warp_wait(&s.s_full[st], (t / kStages) & 1,
                        &s.abort_flag, polls))) break;
                tc_fence_after();
                float sv[kBN];
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) tmem_ld32(s_col + cc * 32, sv + cc * 32);
                tmem_wait_ld();
                // visible keys of this tile for row i: col < lim
                int32_t lim = kBN;
                bool partial_cached = false, masked = false;
                if (j < x.n_cached) {
                    lim = min(kBN, x.c - j * kBN);
                    partial_cached = masked = lim < kBN;
                } else if (j - x.n_cached == x.m) {
                    lim = i + 1;
                    masked = true;
                }
                if (masked) {
#pragma unroll
                    for (int col = 0; col < kBN; ++col) sv[col] = col < lim ? sv[col] : -INFINITY;
                }
                // P = exp2(S*scale - m) into the first 64 columns of the S
                // buffer, with the row sum in two packed pairs of chains (the
                // exponent and the sum take one f32x2 instruction per column
                // pair).
                float ls[4];
                auto exp_pass = [&](float neg_m) {
                    const uint64_t scale2 = pk2(a.scale_log2, a.scale_log2);
                    const uint64_t neg_m2 = pk2(neg_m, neg_m);
                    uint64_t l2[2] = {pk2(0.f, 0.f), pk2(0.f, 0.f)};
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        float pw[32];                           // packed bf16 pairs
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const int col = half * 64 + 2 * e;
                            float x0, x1;
                            up2(fma2(pk2(sv[col], sv[col + 1]), scale2, neg_m2), x0, x1);
                            const float p0 = pkv::fast_exp2(x0);
                            const float p1 = pkv::fast_exp2(x1);
                            l2[e & 1] = add2(l2[e & 1], pk2(p0, p1));
                            pw[e] = __uint_as_float(pkv::pack_bf16(p0, p1));
                        }
                        tmem_st32(s_col + half * 32, pw);       // P aliases S columns 0..63
                    }
                    up2(l2[0], ls[0], ls[1]);
                    up2(l2[1], ls[2], ls[3]);
                };
                // After the first tile, P is computed straight away against the
                // running maximum; only when some row's sum passes kSumTrigger
                // (rare: the maximum grew by more than 2^9) is the tile's
                // maximum taken and P recomputed.  The first tile of an item
                // takes the maximum first.
                bool redo = j == 0;
                if (!redo) {
                    exp_pass(-m_run);
                    const float lt = (ls[0] + ls[1]) + (ls[2] + ls[3]);
                    redo = __any_sync(0xffffffffu, !(lt <= kSumTrigger));
                    if (redo) tmem_wait_st();                   // before P is stored again
                }
                if (redo) {
                    // eight independent partial maxima (no 128-long dependency
                    // chain), two new columns per three-input max
                    float mxp[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) mxp[e] = fmaxf(sv[e], sv[8 + e]);
#pragma unroll
                    for (int col = 16; col < kBN; col += 16)
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            mxp[e] = max3(mxp[e], sv[col + e], sv[col + 8 + e]);
                    float mx = fmaxf(fmaxf(fmaxf(mxp[0], mxp[1]), fmaxf(mxp[2], mxp[3])),
                                     fmaxf(fmaxf(mxp[4], mxp[5]), fmaxf(mxp[6], mxp[7])));
                    mx *= a.scale_log2;                     // scale > 0 keeps the order
                    const bool raise = mx > m_run + kRescaleThreshold;
                    float alpha = 1.f;
                    if (raise) {
                        alpha = (m_run == -INFINITY) ? 0.f : pkv::fast_exp2(m_run - mx);
                        m_run = mx;
                        l_run *= alpha;
                    }
                    if (j > 0 && __any_sync(0xffffffffu, raise)) {
                        // O may only be rescaled once the previous P V has finished
                        const uint32_t tp = t - 1;
                        if (!(ok = warp_wait(&s.pv_done[tp % kStages], (tp / kStages) & 1,
                                             &s.abort_flag, polls)))
                            break;
                        tc_fence_after();
#pragma unroll
                        for (int cc = 0; cc < D / 32; ++cc) {
                            float ov[32];
                            tmem_ld32(lane_base + kColO + cc * 32, ov);
                            tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 32; ++e) ov[e] *= alpha;
                            tmem_st32(lane_base + kColO + cc * 32, ov);
                        }
                    }
                    exp_pass((m_run == -INFINITY) ? 0.f : -m_run);
                }
                l_run += (ls[0] + ls[1]) + (ls[2] + ls[3]);
                tmem_wait_st();
                if (partial_cached) {
                    // masked cached slots may hold NaN: zero their V rows
                    if (!(ok = warp_wait(&s.v_full[st], (t / kStages) & 1,
                            &s.abort_flag, polls))) break;
                    if (i >= lim) {
#pragma unroll
                        for (int hf = 0; hf < kBlocks; ++hf)
#pragma unroll
                            for (int qc = 0; qc < 8; ++qc)
                                *reinterpret_cast<uint4*>(s.v[st] + hf * kHalf + i * 128 + qc * 16) =
                                    make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s.p_full[st]);   // one arrival per softmax warp
            }
            if (!ok) break;
            // ---- epilogue: O / l to global ----
            const uint32_t tl = T + x.n_tiles - 1;
            if (!(ok = warp_wait(&s.pv_done[tl % kStages], (tl / kStages) & 1,
                    &s.abort_flag, polls)))
                break;
            tc_fence_after();
            const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
            __nv_bfloat16* orow = a.out + ((int64_t)(x.q0 + x.m * kBM + i) * a.Hq + x.h) * D;
            // a row is 32-byte aligned when `out` is (rows are D*2 bytes):
            // then 32 bytes per store, a whole sector each (each store of a
            // warp lands in 32 different rows, so the store count sets the
            // cost)
            const bool wide = ((uintptr_t)a.out & 31) == 0;
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                float ov[32];
                tmem_ld32(lane_base + kColO + cc * 32, ov);
                tmem_wait_ld();
                if (i < x.rows) {
                    if (wide) {
#pragma unroll
                        for (int q2 = 0; q2 < 2; ++q2) {
                            uint32_t w8[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                w8[e] = pkv::pack_bf16(ov[q2 * 16 + 2 * e] * inv,
                                                       ov[q2 * 16 + 2 * e + 1] * inv);
                            st_global_32b(orow + cc * 32 + q2 * 16, w8);
                        }
                    } else {
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            uint4 pk;
                            pk.x = pkv::pack_bf16(ov[q4 * 8 + 0] * inv, ov[q4 * 8 + 1] * inv);
                            pk.y = pkv::pack_bf16(ov[q4 * 8 + 2] * inv, ov[q4 * 8 + 3] * inv);
                            pk.z = pkv::pack_bf16(ov[q4 * 8 + 4] * inv, ov[q4 * 8 + 5] * inv);
                            pk.w = pkv::pack_bf16(ov[q4 * 8 + 6] * inv, ov[q4 * 8 + 7] * inv);
                            *reinterpret_cast<uint4*>(orow + cc * 32 + q4 * 8) = pk;
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&s.o_free);
            T += x.n_tiles;
        }
        if (!ok) give_up(s, a.status);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (s.abort_flag && lane == 0 && (warp == 4 || warp == 7)) {
        // some role gave up: every copy this producer issued lands before the
        // CTA exits (a consumer may have given up after the last one was issued)
        const bool k_side = warp == 4;
        for (uint32_t back = 1; back <= (uint32_t)kStages && back <= tiles_issued; ++back) {
            const uint32_t t = tiles_issued - back;
            mbar_drain(k_side ? &s.k_full[t % kStages] : &s.v_full[t % kStages],
                       (t / kStages) & 1);
        }
        if (k_side && q_issued > 0) mbar_drain(&s.q_full, (q_issued - 1) & 1);
    }
    if (warp == 5) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------- host side
// [rows, heads, D] bf16, box 64 x 1 head x box_rows rows.
bool encode_rows(CUtensorMap* m, const void* base, int64_t rows, int heads, int head_dim,
                 int box_rows = kBN) {
    return pkv::tma_encode_rows(m, base, rows, heads, head_dim, box_rows);
}

// The load mode of a call's cached tiles (see kLoadTile).
int load_mode(const PrefillArgs& a) {
    if (a.bt == nullptr || a.bs % kBN == 0) return kLoadTile;
    if (a.bs == 16 || a.bs == 32) return kLoadSplit96;
    if (a.bs == 8 || a.bs == 64) return kLoadSplit64;
    return kLoadGather;
}

template <int D>
int launch_tc(PrefillArgs& a, const TcMaps& maps, cudaStream_t s, const PrefillPrologue* pre) {
    using Kernel = void (*)(const TcMaps, const PrefillArgs);
    static const Kernel kernels[4][2] = {
        {prefill_tc_kernel<D, kLoadTile, false>, prefill_tc_kernel<D, kLoadTile, true>},
        {prefill_tc_kernel<D, kLoadGather, false>, prefill_tc_kernel<D, kLoadGather, true>},
        {prefill_tc_kernel<D, kLoadSplit64, false>, prefill_tc_kernel<D, kLoadSplit64, true>},
        {prefill_tc_kernel<D, kLoadSplit96, false>, prefill_tc_kernel<D, kLoadSplit96, true>}};
    const int smem = (int)sizeof(TcSmem<D>) + 1024;
    const int mode = load_mode(a);
    const int custom = a.wait_polls != (uint32_t)PKV_DEFAULT_WAIT_POLLS ? 1 : 0;
    const Kernel kernel = kernels[mode][custom];
    static std::atomic<uint64_t> configured[8];
    if (!pkv_dynamic_smem_once((const void*)kernel, smem, configured[mode * 2 + custom]))
        return PKV_ERR_CUDA;
    a.tile_m = kBM;
    a.tile_n = kBN;
    const int rc = pkv_launch_prefill_plan(a, s, pre);
    if (rc != PKV_OK) return rc;
    int64_t grid = pkv_num_sms();
    const int64_t upper = (int64_t)a.max_tiles * a.Hq;
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
    if (cudaLaunchKernelEx(&cfg, kernel, maps, a) != cudaSuccess) return PKV_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace

int pkv_prefill_tc_supported(const PrefillArgs& a, int head_dim) {
    if (head_dim != 128 && head_dim != 64) return PKV_ERR_UNSUPPORTED;
    if ((int64_t)a.NB * a.bs >= (1LL << 31)) return PKV_ERR_UNSUPPORTED;
    if (pkv::tma_encode_fn() == nullptr) return PKV_ERR_UNSUPPORTED;
    return PKV_OK;
}

int pkv_launch_prefill_tc(PrefillArgs& a, int head_dim, cudaStream_t s,
                         const PrefillPrologue* pre) {
    TcMaps maps;
    if (!encode_rows(&maps.q, a.q, a.total_q, a.Hq, head_dim) ||
        !encode_rows(&maps.k, a.k, a.total_q, a.Hkv, head_dim) ||
        !encode_rows(&maps.v, a.v, a.total_q, a.Hkv, head_dim))
        return PKV_ERR_CUDA;
    const int mode = a.bt ? load_mode(a) : kLoadTile;
    if (a.bt && mode == kLoadTile) {
        if (!encode_rows(&maps.kc, a.kc, (int64_t)a.NB * a.bs, a.Hkv, head_dim) ||
            !encode_rows(&maps.vc, a.vc, (int64_t)a.NB * a.bs, a.Hkv, head_dim))
            return PKV_ERR_CUDA;
    } else if (mode == kLoadSplit64 || mode == kLoadSplit96) {
        // boxes of one cache block
        if (!encode_rows(&maps.kc, a.kc, (int64_t)a.NB * a.bs, a.Hkv, head_dim, a.bs) ||
            !encode_rows(&maps.vc, a.vc, (int64_t)a.NB * a.bs, a.Hkv, head_dim, a.bs))
            return PKV_ERR_CUDA;
    } else {
        maps.kc = maps.k;
        maps.vc = maps.v;
    }
    return head_dim == 128 ? launch_tc<128>(a, maps, s, pre) : launch_tc<64>(a, maps, s, pre);
}
