/*
 * pagedattn.h -- C ABI of libpagedattn.so, attention over a paged KV cache on
 * one NVIDIA GB300 (sm_103a).
 *
 * The four operations are the per-layer GPU hot path of a Nano-vLLM-style
 * serving engine, as described on these pages:
 *   [LIFE] "一个 prompt 的一生：nano-vllm 从起服务到吐出 token" (violet-quartz.github.io)
 *   [UML]  the Nano-vLLM walk-through at uml.org.cn
 *   [SRC2] "《Nano-vLLM源码逐行解析》第2篇 sequence.py、scheduler.py" (yeyulingfeng.com)
 *
 * Data layout (all row-major, contiguous):
 *   k_cache, v_cache  [num_blocks, block_size, num_kv_heads, head_dim] bf16: one
 *                     layer's view of the KV pool ([LIFE] §2.2.3; [UML] §3.2).
 *                     A slot s is row s of the pool viewed as
 *                     [num_blocks*block_size, num_kv_heads, head_dim].
 *   block_tables      [batch, max_blocks_per_seq] int32: logical block i of a
 *                     sequence -> physical block id ([UML] §1 Step2, §3.2).
 *                     Entries past a sequence's last block are never read.
 *   q                 [tokens, num_q_heads, head_dim] bf16; k, v [tokens,
 *                     num_kv_heads, head_dim] bf16 ([UML] §3.2 formats).
 *   Grouped-query attention: q head h reads kv head h / (num_q_heads/num_kv_heads).
 *
 * Ownership: every pointer argument is caller-owned memory; the library keeps
 * no pointer past the call, allocates nothing and never synchronises.  Device
 * pointers must be device memory of the current CUDA device.  All work is
 * enqueued on `stream` (a cudaStream_t passed as void*; NULL = legacy default
 * stream) and runs asynchronously.
 *
 * Errors, two kinds:
 *   - the return value: PKV_OK (0) or a negative PKV_ERR_* code for a problem
 *     the host can see (null pointer, bad size, unsupported head_dim,
 *     misaligned pointer, workspace too small, launch failure).  Nothing is
 *     enqueued when a call returns an error.
 *   - `status`: an optional device uint32 into which kernels OR the
 *     PKV_STATUS_* bits of data-dependent problems (a slot or block id outside
 *     the pool, a bad context length, ...).  The offending item is skipped
 *     (its outputs are zeros where the entry point says so); nothing traps.
 *     The caller clears the word; NULL disables reporting.
 */
#ifndef PAGEDATTN_H
#define PAGEDATTN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes ------------------------------------------------------ */
#define PKV_OK                        0
#define PKV_ERR_NULL_POINTER         -1
#define PKV_ERR_BAD_DIMENSION        -2
#define PKV_ERR_UNSUPPORTED_HEAD_DIM -3
#define PKV_ERR_MISALIGNED           -4
#define PKV_ERR_WORKSPACE_TOO_SMALL  -5
#define PKV_ERR_CUDA                 -6
#define PKV_ERR_UNSUPPORTED          -7

/* ---- device status bits ------------------------------------------------ */
#define PKV_STATUS_SLOT_OUT_OF_RANGE  (1u << 0) /* kv_store: slot >= num_blocks*block_size   */
#define PKV_STATUS_BAD_BLOCK_ID       (1u << 1) /* a block table entry outside [0,num_blocks) */
#define PKV_STATUS_BAD_CONTEXT_LEN    (1u << 2) /* context len < 0, > table capacity or > max */
#define PKV_STATUS_BAD_SEQLENS        (1u << 3) /* cu_seqlens not monotone, Lk < Lq, ...       */
#define PKV_STATUS_BAD_TEMPERATURE    (1u << 4) /* sample: temperature not positive & finite  */
#define PKV_STATUS_NO_FINITE_KEY      (1u << 5) /* sample: every key of a row is NaN           */
#define PKV_STATUS_WORKSPACE_OVERFLOW (1u << 6) /* more work items than the workspace holds   */
#define PKV_STATUS_WAIT_TIMEOUT       (1u << 7) /* a bounded in-kernel wait gave up           */

/* One layer's KV cache geometry: k_cache/v_cache are [num_blocks, block_size,
 * num_kv_heads, head_dim] bf16. */
typedef struct pkv_cache_desc {
    int32_t num_blocks;
    int32_t block_size;
    int32_t num_kv_heads;
    int32_t head_dim;
} pkv_cache_desc;

/* Library version, major*10000 + minor*100 + patch. */
PKV_API int pkv_version(void);

/* Text for a PKV_ERR_* return code (static storage). */
PKV_API const char* pkv_error_string(int code);

/* Text naming the lowest PKV_STATUS_* bit set in `bits` ("ok" for 0). */
PKV_API const char* pkv_status_string(uint32_t bits);

/*
 * Diagnostics (no counterpart on the pages).  Every in-kernel wait on a
 * shared-memory barrier polls at most `polls` times, then gives up: the kernel
 * sets PKV_STATUS_WAIT_TIMEOUT, lets the copies and tensor-core operations it
 * already issued finish, frees what it holds and returns (its outputs are then
 * unspecified).  The setting is process-wide and applies to calls enqueued
 * after it.  The default, PKV_DEFAULT_WAIT_POLLS, is far beyond any wait of a
 * healthy kernel; 0 makes every such wait give up at once, which is how the
 * tests exercise the unwinding path.  Returns PKV_OK.
 */
#define PKV_DEFAULT_WAIT_POLLS (1u << 20)
PKV_API int pkv_set_wait_poll_limit(uint32_t polls);

/*
 * kv_store -- the per-layer KV cache write ("store_kvcache").
 * [UML] §2.4 (KV written into the cache before attention), §1 Step2 (slot =
 * blockID*blockSize + loc); [LIFE] §3.3.2 / §4 (slot_mapping holds one
 * physical slot per flattened token, so the writer needs no paging logic).
 *
 *   k, v           device, [num_tokens, num_kv_heads, head_dim] bf16, 16-byte aligned
 *   k_cache/v_cache device, the pool, written in place, 16-byte aligned
 *   slot_mapping   device, [num_tokens] int32; slot < 0 skips the token (padding
 *                  rows of a fixed-shape batch); slot >= num_blocks*block_size
 *                  sets PKV_STATUS_SLOT_OUT_OF_RANGE and skips it
 * Row i of k and of v is copied bit for bit into slot slot_mapping[i].  Two
 * tokens with the same slot in one call: the surviving row is one of them.
 * Needs num_kv_heads*head_dim*2 to be a multiple of 16.  num_tokens == 0 is a
 * no-op.
 */
PKV_API int pkv_kv_store(const void* k, const void* v, void* k_cache, void* v_cache,
                 const int32_t* slot_mapping, int32_t num_tokens,
                 pkv_cache_desc cache, uint32_t* status, void* stream);

/*
 * Bytes of device workspace pkv_paged_decode needs for these sizes (a pure
 * host function; the same arguments give the same answer).  The split into
 * key chunks depends on the batch, so the size is not monotone in it: a
 * workspace shared by several batch sizes (e.g. one CUDA graph per size)
 * must be as large as the largest of their answers.
 */
PKV_API size_t pkv_paged_decode_workspace_bytes(int32_t batch, int32_t num_q_heads,
                                        int32_t max_context_len, pkv_cache_desc cache);

/*
 * paged_decode -- decode attention, one query token per sequence, K/V read
 * through the block table ([UML] §2.4: the decode attention op; §3.2: Q as
 * (batch, 1, heads, head_dim), cache_seqlens, block_tables).
 *
 *   q             device, [batch, num_q_heads, head_dim] bf16
 *   k_cache/v_cache device, the pool (read only)
 *   block_tables  device, [batch, max_blocks_per_seq] int32
 *   context_lens  device, [batch] int32: keys of sequence b are its logical
 *                 positions 0..context_lens[b]-1 (the new token's K/V must
 *                 already be stored).  0 gives a zero output row.  A value < 0,
 *                 > max_blocks_per_seq*block_size or > max_context_len sets
 *                 PKV_STATUS_BAD_CONTEXT_LEN and gives zeros.
 *   max_context_len host upper bound of context_lens, sizes the split-KV grid
 *   scale         softmax scale (e.g. 1/sqrt(head_dim))
 *   out           device, [batch, num_q_heads, head_dim] bf16
 *   workspace     device, >= pkv_paged_decode_workspace_bytes(...) bytes,
 *                 16-byte aligned; holds the split-KV partial results
 * out[b,h] = sum_j softmax_j(scale * q[b,h].K_j) V_j, fp32 accumulation.
 * head_dim 64 or 128; num_q_heads a multiple of num_kv_heads.
 */
PKV_API int pkv_paged_decode(const void* q, const void* k_cache, const void* v_cache,
                     const int32_t* block_tables, int32_t max_blocks_per_seq,
                     const int32_t* context_lens, int32_t batch, int32_t num_q_heads,
                     int32_t max_context_len, float scale, void* out,
                     void* workspace, size_t workspace_bytes,
                     pkv_cache_desc cache, uint32_t* status, void* stream);

/*
 * paged_decode split into a plan and a run, for a caller that attends many
 * layers over the same sequences: in a model's decode step every layer has the
 * same context_lens and block_tables, so the chunk schedule is the same for
 * all of them.  (No counterpart on the pages: it divides pkv_paged_decode's
 * work; the result is the same.)
 *
 * pkv_paged_decode_plan checks context_lens (a length outside
 * [0, min(max_context_len, max_blocks_per_seq * block_size)] sets
 * PKV_STATUS_BAD_CONTEXT_LEN and that sequence attends to nothing) and writes
 * the chunk schedule into the workspace.  pkv_paged_decode_run then attends with
 * it: the split-KV and combine kernels only.  A run must get the same
 * context_lens contents, batch, num_q_heads, max_context_len,
 * max_blocks_per_seq, cache geometry and workspace as the plan it follows, and
 * the plan must be enqueued earlier on the same stream (or have completed).  Any
 * number of runs may follow one plan; a run overwrites the workspace's partial
 * results, so runs sharing a workspace must not overlap.  Arguments have the
 * meaning they have in pkv_paged_decode.
 */
PKV_API int pkv_paged_decode_plan(const int32_t* context_lens, int32_t batch,
                                  int32_t num_q_heads, int32_t max_context_len,
                                  int32_t max_blocks_per_seq, void* workspace,
                                  size_t workspace_bytes, pkv_cache_desc cache,
                                  uint32_t* status, void* stream);
PKV_API int pkv_paged_decode_run(const void* q, const void* k_cache, const void* v_cache,
                                 const int32_t* block_tables, int32_t max_blocks_per_seq,
                                 const int32_t* context_lens, int32_t batch, int32_t num_q_heads,
                                 int32_t max_context_len, float scale, void* out, void* workspace,
                                 size_t workspace_bytes, pkv_cache_desc cache, uint32_t* status,
                                 void* stream);

/*
 * paged_decode without a caller-provided workspace.  (Not an operation of the
 * pages: it exists for callers that cannot allocate device memory where they
 * call -- e.g. a plugin inside a host engine that owns and budgets all device
 * memory up front, or a latency-critical loop that must not pay for
 * cudaMalloc's implicit device-wide synchronisation.)
 *
 * Same arguments and results as pkv_paged_decode, minus workspace and
 * workspace_bytes.  The split-KV scratch is a fixed array of
 * PKV_STATIC_DECODE_WORKSPACE_BYTES compiled into the library; every GPU that
 * loads the library holds it until the process exits.  The call allocates
 * nothing (no cudaMalloc, no allocating library routine).
 *   - When pkv_paged_decode_workspace_bytes(batch, num_q_heads,
 *     max_context_len, cache) exceeds PKV_STATIC_DECODE_WORKSPACE_BYTES the
 *     call returns PKV_ERR_WORKSPACE_TOO_SMALL and enqueues nothing.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - All calls share the one array, which keeps the last call's contents
 *     (the kernels write every scratch entry they read, so no state carries
 *     over).  Calls that may overlap on the GPU -- on different streams, or
 *     from different host threads -- race on it: serialise them.
 */
#define PKV_STATIC_DECODE_WORKSPACE_BYTES (16u * 1024u * 1024u)
PKV_API int pkv_paged_decode_static_workspace(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t batch,
    int32_t num_q_heads, int32_t max_context_len, float scale, void* out,
    pkv_cache_desc cache, uint32_t* status, void* stream);

/*
 * kv_store then paged_decode, enqueued as one call: the per-layer pair the
 * engine runs every decode step ([LIFE] §2.2.4: store_kvcache, then the
 * attention op; [UML] §2.4).  Arguments are those of pkv_kv_store (k, v,
 * slot_mapping, num_tokens) followed by those of pkv_paged_decode; k_cache
 * and v_cache are written by the store and read by the decode.  The store and
 * the decode's set-up (its chunk schedule) run as one grid, so the pair costs
 * one launch and the longer of the two; the attention kernels wait for that
 * whole grid, so they read the stored rows whatever slots slot_mapping names.
 * Arguments are all checked before anything is enqueued.
 */
PKV_API int pkv_kv_store_paged_decode(
    const void* k, const void* v, const int32_t* slot_mapping, int32_t num_tokens,
    const void* q, void* k_cache, void* v_cache, const int32_t* block_tables,
    int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t batch,
    int32_t num_q_heads, int32_t max_context_len, float scale, void* out, void* workspace,
    size_t workspace_bytes, pkv_cache_desc cache, uint32_t* status, void* stream);

/*
 * One layer's k_cache / v_cache inside the whole KV pool the engine allocates
 * once, [2, num_layers, num_blocks, block_size, num_kv_heads, head_dim] bf16
 * ([LIFE] §2.2.3: kv_cache[0, l] and kv_cache[1, l] are views, not copies).
 * Pure host pointer arithmetic; nothing is read or enqueued.
 */
PKV_API int pkv_layer_cache(const void* kv_pool, int32_t num_layers, int32_t layer,
                            pkv_cache_desc cache, const void** k_cache, const void** v_cache);

/*
 * Bytes of device workspace pkv_paged_prefill_varlen needs (pure host function).
 */
PKV_API size_t pkv_paged_prefill_workspace_bytes(int32_t batch, int32_t total_q,
                                         int32_t num_q_heads, pkv_cache_desc cache);

/*
 * paged_prefill_varlen -- causal prefill over a flattened batch of
 * variable-length sequences whose first tokens may already be in the cache
 * (prefix caching, chunked prefill).  [UML] §2.4 and §3.2 (the varlen prefill
 * attention op: cu_seqlens_q/k, max_seqlen_q/k, block_tables when a prefix is
 * cached); [LIFE] §3.1 / [SRC2] Sequence walkthrough (a round computes
 * num_scheduled_tokens tokens starting at num_cached_tokens).
 *
 *   q             device, [total_q, num_q_heads, head_dim] bf16
 *   k, v          device, [total_q, num_kv_heads, head_dim] bf16: this call's
 *                 own keys/values, one row per query token
 *   k_cache/v_cache device, the pool (read only)
 *   cu_seqlens_q/k device, [batch+1] int32 prefix sums.  Sequence b has
 *                 Lq = cu_q[b+1]-cu_q[b] queries and Lk = cu_k[b+1]-cu_k[b] keys.
 *                 Keys j < Lk-Lq (the cached prefix) are read from the cache
 *                 through block_tables[b]; keys j >= Lk-Lq are rows
 *                 cu_q[b]+j-(Lk-Lq) of k/v.  Query i sits at position Lk-Lq+i
 *                 and attends keys j <= Lk-Lq+i (bottom-right causal).
 *   max_seqlen_q/k host upper bounds of Lq/Lk
 *   block_tables  device [batch, max_blocks_per_seq] int32, or NULL when no
 *                 sequence has a cached prefix (then Lk must equal Lq)
 *   scale         softmax scale, positive and finite (e.g. 1/sqrt(head_dim))
 *   out           device, [total_q, num_q_heads, head_dim] bf16
 *   workspace     device, >= pkv_paged_prefill_workspace_bytes(...) bytes,
 *                 16-byte aligned; holds the tile schedule
 * A sequence with inconsistent lengths sets PKV_STATUS_BAD_SEQLENS and is
 * skipped (its output rows are not written).  head_dim 64 or 128, any
 * block_size.  PKV_ERR_UNSUPPORTED: num_blocks*block_size >= 2^31 (no such
 * pool fits in device memory) or a driver without cuTensorMapEncodeTiled.
 */
PKV_API int pkv_paged_prefill_varlen(const void* q, const void* k, const void* v,
                             const void* k_cache, const void* v_cache,
                             const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                             int32_t batch, int32_t total_q, int32_t max_seqlen_q,
                             int32_t max_seqlen_k, int32_t num_q_heads,
                             const int32_t* block_tables, int32_t max_blocks_per_seq,
                             float scale, void* out, void* workspace, size_t workspace_bytes,
                             pkv_cache_desc cache, uint32_t* status, void* stream);

/*
 * kv_store followed by paged_prefill_varlen on the same stream: the per-layer
 * pair of a prefill round, cache write then attention ([LIFE] §2.2.4 and §4
 * store_kvcache before the attention op; [UML] §2.4).  The store writes this
 * call's k/v rows (total_q of them) to slot_mapping's slots (negative =
 * padding, skipped); the other arguments are those of
 * pkv_paged_prefill_varlen, with k_cache/v_cache written by the store and
 * required even when block_tables is NULL.  The prefill's tile plan is launched
 * as a programmatic dependent of the store, and the attention reads nothing
 * until both are done.  Every argument is checked before anything is
 * enqueued.
 */
PKV_API int pkv_kv_store_paged_prefill_varlen(
    const void* q, const void* k, const void* v, void* k_cache, void* v_cache,
    const int32_t* slot_mapping, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
    int32_t batch, int32_t total_q, int32_t max_seqlen_q, int32_t max_seqlen_k,
    int32_t num_q_heads, const int32_t* block_tables, int32_t max_blocks_per_seq, float scale,
    void* out, void* workspace, size_t workspace_bytes, pkv_cache_desc cache, uint32_t* status,
    void* stream);

/*
 * Bytes of device workspace pkv_kv_store_paged_attention_varlen needs (pure
 * host function): the prefill's tile schedule followed by the decode's chunk
 * plan and partial results, the latter sized for max_seqlen_k keys.
 */
PKV_API size_t pkv_paged_attention_varlen_workspace_bytes(int32_t batch, int32_t total_q,
                                                  int32_t num_q_heads, int32_t max_seqlen_k,
                                                  pkv_cache_desc cache);

/*
 * kv_store then attention over a mixed batch: prefill chunks and decode
 * tokens in one step.  The pages' scheduler never mixes the two ([LIFE] §3.2),
 * but a step's sequences each compute num_scheduled_tokens tokens from
 * num_cached_tokens on ([LIFE] §3.1), so a decode row is a chunk of one token
 * and continuous batching ([UML] §2.1) can take both in one call.  The
 * arguments and the result are those of pkv_kv_store_paged_prefill_varlen
 * (bottom-right causal attention of every query row), computed in two passes:
 * sequences with Lq != 1 by the varlen prefill kernels, sequences with Lq == 1
 * by the split-KV decode kernels.  The second pass reads all Lk keys of a
 * one-query sequence from the cache through block_tables[b], its own key
 * included, so slot_mapping must store that row at position Lk-1 of
 * block_tables[b] (as an engine's slot mapping does); block_tables and the
 * cache are required.
 *   workspace     device, >= pkv_paged_attention_varlen_workspace_bytes(...)
 *                 bytes, 16-byte aligned
 * A one-query sequence whose lengths are inconsistent (Lk < 1, its row outside
 * q, more keys than max_seqlen_k or than its table holds) sets
 * PKV_STATUS_BAD_SEQLENS and its output row is not written.  Every argument
 * is checked before anything is enqueued.
 */
PKV_API int pkv_kv_store_paged_attention_varlen(
    const void* q, const void* k, const void* v, void* k_cache, void* v_cache,
    const int32_t* slot_mapping, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
    int32_t batch, int32_t total_q, int32_t max_seqlen_q, int32_t max_seqlen_k,
    int32_t num_q_heads, const int32_t* block_tables, int32_t max_blocks_per_seq, float scale,
    void* out, void* workspace, size_t workspace_bytes, pkv_cache_desc cache, uint32_t* status,
    void* stream);

/*
 * sample -- temperature, softmax and Gumbel-max sampling of one token per row
 * ([UML] §2.4: "温度、softmax和gumbel max"; [LIFE] §4: the sampler runs on each
 * sequence's last-position logits).  With supplied Exp(1) noise E the draw is
 * argmax_i softmax(logits/T)_i / E_i, computed as the equal
 * argmax_i (logits_i/T - ln max(E_i, 1e-10)); ties go to the lowest index.
 *
 *   logits        device, [batch, vocab] fp32
 *   temperatures  device, [batch] fp32; a value that is not positive and finite
 *                 sets PKV_STATUS_BAD_TEMPERATURE and the row returns 0
 *   exp_noise     device, [batch, vocab] fp32 Exp(1) draws
 *   out_token_ids device, [batch] int32
 * NaN keys never win; a row of NaN keys returns 0 and sets
 * PKV_STATUS_NO_FINITE_KEY.
 */
PKV_API int pkv_sample(const float* logits, const float* temperatures, const float* exp_noise,
               int32_t batch, int32_t vocab, int32_t* out_token_ids,
               uint32_t* status, void* stream);

/*
 * sample with the Exp(1) noise drawn inside the kernel instead of read from
 * memory (halves the sampler's HBM bytes).  The noise of entry n = row*vocab+i
 * comes from Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel random
 * numbers: as easy as 1, 2, 3", SC 2011) with key = seed (low word first) and
 * counter = (n/4 low, n/4 high, offset low, offset high), output word n%4:
 * U = ((w >> 8) + 1) * 2^-24 in (0, 1], E = -ln U.  Everything else is as in
 * pkv_sample (temperature, lowest-index ties, status bits).  The same (seed,
 * offset) gives the same draw; advance `offset` per step for fresh noise.
 */
PKV_API int pkv_sample_philox(const float* logits, const float* temperatures, uint64_t seed,
                              uint64_t offset, int32_t batch, int32_t vocab,
                              int32_t* out_token_ids, uint32_t* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H */
