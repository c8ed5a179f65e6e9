/*
 * pagedkv.h -- C ABI of the B300 (sm_103a) paged KV-cache hot path: KV store, paged decode
 * attention, varlen paged prefill attention.
 *
 * The operations follow the PagedAttention scheme described on the source pages:
 *  [P1] "DeepSeek研究员1200行代码复刻vLLM，H800硬件实测性能反超原版" (QbitAI), section "vLLM是什么？":
 *       the KV cache is divided into fixed-size blocks; a per-sequence block table maps logical
 *       blocks to physical blocks; keys and values of one sequence live in blocks that need not be
 *       contiguous; the attention kernel fetches the blocks one by one; KV may be shared within
 *       and across requests.
 *  [P3] "nano-vllm 深度分析报告": table "可复用的模式与技巧", row "slot_mapping -1 padding"
 *       (slots padded for CUDA graphs are -1 and the store skips them); table "关键设计决策"
 *       (block_size 256 versus vLLM's 16); section "创新之处" (prefix-cache hits share physical
 *       blocks; CUDA graphs captured for a ladder of batch sizes).
 *
 * Conventions for every entry point:
 *  - Pointers marked "device" are CUDA device pointers owned by the caller; the library never
 *    allocates, frees or retains them. bf16 tensors are passed as `uint16_t*` holding bf16 bit
 *    patterns. All device pointers must be 16-byte aligned.
 *  - `stream` is a cudaStream_t passed as `void*` (NULL = the legacy default stream). Work is only
 *    enqueued; no call synchronises the device, so the calls can be captured into a CUDA graph.
 *  - Cache layout: k_cache and v_cache are [num_blocks, block_size, num_kv_heads, head_dim] bf16,
 *    row-major. The token at slot s lives at block s / block_size, offset s % block_size.
 *  - Grouped-query attention: query head h reads kv head h / (num_q_heads / num_kv_heads).
 *  - Return value: PKV_OK (0) or a negative PKV_ERR_* code. On error nothing is enqueued and a
 *    message is available from pkv_last_error() (thread-local). No exception crosses the ABI.
 *  - Bad data inside device buffers (a slot or block id out of range, a context longer than its
 *    block table) cannot be checked on the host without a synchronisation. The kernels check it,
 *    skip the offending access (they never read or write out of range) and set a bit in a device
 *    error word that pkv_get_device_error() reads back.
 *  - Supported shapes: head_dim 64 or 128; block_size a power of two from 16 to 256;
 *    num_q_heads a multiple of num_kv_heads with group size 1, 2, 4 or 8;
 *    num_blocks * block_size < 2^31.
 */
#ifndef PAGEDKV_H_
#define PAGEDKV_H_

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

#define PKV_OK 0
#define PKV_ERR_INVALID_ARG (-1)        /* null pointer, bad size, misaligned pointer */
#define PKV_ERR_UNSUPPORTED (-2)        /* valid but unsupported shape (see above) */
#define PKV_ERR_WORKSPACE_TOO_SMALL (-3) /* workspace_bytes below what the plan needs */
#define PKV_ERR_CUDA (-4)               /* a CUDA runtime / driver call failed */

/* Bits of the device error word (pkv_get_device_error). */
#define PKV_DEVERR_BAD_SLOT 1       /* kv_store: slot neither -1 nor in [0, num_blocks*block_size) */
#define PKV_DEVERR_BAD_BLOCK 2      /* a block table entry outside [0, num_blocks) was needed */
#define PKV_DEVERR_CTX_CLAMPED 4    /* a context longer than its block table or the decode plan */
#define PKV_DEVERR_TIMEOUT 8        /* an internal pipeline wait gave up after one second */
#define PKV_DEVERR_BAD_LENGTHS 16   /* prefill: cu_seqlens not increasing or k_len < q_len */
#define PKV_DEVERR_INTERNAL 32      /* an internal layout invariant failed (nothing written) */

/* Geometry of one layer's paged cache. */
typedef struct pkv_cache_desc {
  int32_t num_blocks;
  int32_t block_size;
  int32_t num_kv_heads;
  int32_t head_dim;
} pkv_cache_desc;

/*
 * KV store [P3 "slot_mapping -1 padding"; P1 fixed-size blocks].
 * For t in [0, num_tokens): s = slot_mapping[t]; if s == -1 the token is skipped; otherwise
 * k[t] is copied bit for bit to k_cache[s / block_size][s % block_size] and v[t] likewise.
 *   k, v          device, [num_tokens, num_kv_heads, head_dim] bf16
 *   slot_mapping  device, [num_tokens] int32
 *   k_cache, v_cache  device, cache layout above (written in place)
 * Duplicate slots in one call are a caller error (which row wins is unspecified).
 * num_tokens == 0 is a no-op.
 */
PKV_API int pkv_kv_store(const uint16_t* k, const uint16_t* v, const int32_t* slot_mapping,
                 int32_t num_tokens, uint16_t* k_cache, uint16_t* v_cache, pkv_cache_desc cache,
                 void* stream);

/*
 * Decode plan: how pkv_paged_decode cuts contexts into chunks (flash-decoding split) and how much
 * device workspace it needs. A pure host computation (no CUDA call).
 *   max_context_len    an upper bound of every context length the plan will be used with
 *   split_tokens_hint  0 = automatic: contexts longer than 512 tokens may be split, and the
 *                      device picks the chunk length (>= 512) from the actual lengths so that
 *                      the work spreads over all SMs; a large batch is then not split at all.
 *                      > 0 = fixed chunk length (rounded up to a multiple of 128).
 *                      < 0 = never split.
 * Outputs: split_tokens (fixed chunk length, or the smallest chunk length when auto_split is 1),
 * max_splits (the most chunks any sequence can have), workspace_bytes (device workspace the
 * decode call needs for these num_seqs and num_q_heads), and engine. The plan picks
 * PKV_DECODE_ENGINE_TENSOR_CORE when head_dim is 128, block_size >= 128 and the group size
 * G = num_q_heads / num_kv_heads is 4 or 8, and PKV_DECODE_ENGINE_CUDA_CORE otherwise. The caller
 * may change engine before the decode call:
 *   PKV_DECODE_ENGINE_CUDA_CORE    the persistent decode kernel: CUDA-core fp32 arithmetic,
 *                                  any supported shape.
 *   PKV_DECODE_ENGINE_TENSOR_CORE  tcgen05 MMAs with 128 keys of one kv head on the M dimension
 *                                  and that kv head's G query heads on N (P in bf16, fp32
 *                                  accumulation); head_dim 128 only (PKV_ERR_UNSUPPORTED
 *                                  otherwise), any group size, chunked contexts as above.
 * Both give the same results within bf16 rounding. Measured on a B300 (1024 sequences, 32/8
 * heads, block_size 256): the tensor-core engine streams K/V at the copy bandwidth and runs a
 * sustained decode loop at full SM clock; the CUDA-core engine issues about twice the
 * instructions per byte at G >= 4 and is ~5% slower there. At G <= 2 the CUDA-core engine is
 * the faster one, and below block_size 128 the TMA boxes of the tensor-core engine (one per
 * block and 64-dim half) become too small to keep HBM busy.
 */
#define PKV_DECODE_ENGINE_CUDA_CORE 1
#define PKV_DECODE_ENGINE_TENSOR_CORE 2

/*
 * flags (0 from pkv_decode_plan_make; the caller may set):
 *   PKV_DECODE_PLAN_REUSE  the decode call launches no plan kernel and runs on the device plan
 *                          (chunk length, work list) already in its workspace. Valid when the
 *                          previous decode call on that workspace used this plan, the same
 *                          num_seqs, num_q_heads and cache geometry, and context_lens with the
 *                          same values, e.g. every layer of a decode step after the first, as
 *                          the per-step attention metadata of ["nano-vllm 深度分析报告", table
 *                          "可复用的模式与技巧"] is set once per step. Every decode call leaves
 *                          its workspace's work counters reset for such a call. With
 *                          pkv_paged_decode_store the step's store still runs, in a grid of
 *                          its own before the decode kernel. A reuse that breaks these
 *                          conditions gives wrong outputs (never an access outside the caches
 *                          or the workspace: every table entry and context is still
 *                          bounds-checked, a work list longer than this call's batch allows is
 *                          dropped and one naming a sequence outside it is skipped, both
 *                          raising PKV_DEVERR_INTERNAL).
 */
#define PKV_DECODE_PLAN_REUSE 1

typedef struct pkv_decode_plan {
  int32_t split_tokens;
  int32_t max_splits;
  int32_t auto_split;
  int32_t max_context_len;
  size_t workspace_bytes;
  int32_t engine;
  int32_t flags;
} pkv_decode_plan;

PKV_API int pkv_decode_plan_make(int32_t num_seqs, int32_t num_q_heads, pkv_cache_desc cache,
                         int32_t max_context_len, int32_t split_tokens_hint,
                         pkv_decode_plan* plan);

/*
 * Paged decode attention [P1 PagedAttention].
 * For sequence b and query head h (kv head g = h / G):
 *   out[b][h] = softmax(scale * q[b][h] . K_b^T) V_b
 * over the context_lens[b] tokens at positions 0 .. context_lens[b]-1, where position p of
 * sequence b lives at block block_tables[b][p / block_size], offset p % block_size. A sequence
 * with context_lens[b] == 0 (a padded batch entry) gets zeros. Chunks of a split context are
 * merged with their log-sum-exp weights inside the same launch sequence.
 *   q             device, [num_seqs, num_q_heads, head_dim] bf16
 *   block_tables  device, [num_seqs, max_blocks_per_seq] int32 (entries past the context unused)
 *   context_lens  device, [num_seqs] int32, each <= plan->max_context_len and
 *                 <= max_blocks_per_seq * block_size (longer contexts are clamped and flagged)
 *   scale         softmax scale applied to q.k (e.g. 1/sqrt(head_dim))
 *   plan          host, from pkv_decode_plan_make with the same num_seqs, num_q_heads, cache
 *   out           device, [num_seqs, num_q_heads, head_dim] bf16 (fp32 accumulation, RNE)
 *   workspace     device scratch of at least plan->workspace_bytes, 256-byte aligned, owned by
 *                 the caller. Every call rewrites it, so calls that share one workspace must be
 *                 ordered on one stream.
 * Launches: a one-CTA plan kernel (chunking, work list) and the persistent decode kernel of the
 * plan's engine, launched as its programmatic dependent; with PKV_DECODE_PLAN_REUSE in
 * plan->flags, the decode kernel alone.
 */
PKV_API int pkv_paged_decode(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                     pkv_cache_desc cache, const int32_t* block_tables,
                     int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t num_seqs,
                     int32_t num_q_heads, float scale, const pkv_decode_plan* plan,
                     uint16_t* out, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Whole-block moves ["nano-vllm 深度分析报告", section "解法哲学": swap (CPU offload) and
 * copy-on-write are the block-level features Nano-vLLM leaves out and vLLM keeps].
 * A block of one cache is block_size * num_kv_heads * head_dim bf16, contiguous; every call moves
 * the K and the V block alike. Block ids outside [0, num_blocks) are skipped and flagged
 * (PKV_DEVERR_BAD_BLOCK). n == 0 is a no-op.
 *
 * pkv_copy_blocks: copy-on-write. For i in [0, n): block pairs[2i+1] := block pairs[2i].
 *   pairs   device, [n, 2] int32 (source, destination). A block that is a destination must not
 *           also be a source in the same call (the result would be unspecified).
 * pkv_gather_blocks: swap out. out_k[i] := k_cache[ids[i]], out_v[i] := v_cache[ids[i]].
 *   ids     device, [n] int32;  out_k, out_v  device, [n, block_size, num_kv_heads, head_dim]
 * pkv_scatter_blocks: swap in. k_cache[ids[i]] := in_k[i], v_cache[ids[i]] := in_v[i].
 *   ids must be distinct.
 */
PKV_API int pkv_copy_blocks(uint16_t* k_cache, uint16_t* v_cache, pkv_cache_desc cache,
                            const int32_t* pairs, int32_t n, void* stream);
PKV_API int pkv_gather_blocks(const uint16_t* k_cache, const uint16_t* v_cache,
                              pkv_cache_desc cache, const int32_t* ids, int32_t n,
                              uint16_t* out_k, uint16_t* out_v, void* stream);
PKV_API int pkv_scatter_blocks(const uint16_t* in_k, const uint16_t* in_v, const int32_t* ids,
                               int32_t n, uint16_t* k_cache, uint16_t* v_cache,
                               pkv_cache_desc cache, void* stream);

/*
 * Chained block hashes for prefix-cache lookup ["nano-vllm 深度分析报告", section "创新之处" and
 * table "可复用的模式与技巧": each full block is content-addressed by an xxhash64 that includes the
 * hash of the preceding blocks, which makes the position part of the identity].
 * For sequence b (tokens token_ids[cu_seqlens[b] .. cu_seqlens[b+1])) and each of its full blocks
 * i < len_b / block_size:
 *   out[b * max_blocks + i] = XXH64(seed 0) of [8-byte little-endian out[b*max_blocks + i-1],
 *                              omitted for i = 0] ++ [the block's token ids, 4-byte little-endian]
 * Entries for i >= the number of full blocks are set to 0. A sequence with more than max_blocks
 * full blocks has the rest ignored and raises PKV_DEVERR_CTX_CLAMPED.
 *   token_ids   device, int32;  cu_seqlens  device, [num_seqs + 1] int32, non-decreasing
 *   block_size  even, 2..256;   out  device, [num_seqs, max_blocks] uint64
 */
PKV_API int pkv_block_hashes(const int32_t* token_ids, const int32_t* cu_seqlens,
                             int32_t num_seqs, int32_t block_size, int32_t max_blocks,
                             uint64_t* out, void* stream);

/*
 * Paged decode without any device allocation by the caller (no counterpart in the source pages:
 * it exists for callers of this library that cannot allocate device memory).
 * Some callers cannot call cudaMalloc for the decode workspace: a process that has given all of
 * a GPU's memory to its own pool allocator, or code that must not enter an allocator where it
 * runs attention (for example a plugin invoked inside another runtime's execution loop). This
 * entry point computes exactly what pkv_paged_decode computes, with the same arguments minus
 * workspace and workspace_bytes: its workspace is a fixed array of PKV_STATIC_WS_BYTES (8 MiB)
 * in the library's own device memory, which every GPU that loads the library holds until the
 * process exits. It calls no allocating routine.
 *  - A plan whose workspace_bytes exceeds PKV_STATIC_WS_BYTES is rejected with
 *    PKV_ERR_WORKSPACE_TOO_SMALL (pkv_last_error() gives both sizes) before anything is enqueued;
 *    a plan with fewer splits (split_tokens_hint < 0 never splits) needs far less.
 *  - The array exists once per CUDA context (normally once per device, in its primary context).
 *    The first call in a context looks up the array's device address with that context current
 *    and keeps it under the driver's unique context id; make that first call before any stream
 *    capture. A context the caller creates itself, or the device's new primary context after
 *    cudaDeviceReset, has a new id and gets a fresh lookup, so no stale address is ever used.
 *  - All calls in a context share the array, which keeps the previous call's contents; each call
 *    re-initialises what must start at zero itself. Calls that overlap on the GPU (unordered
 *    streams) race on the array: order them, e.g. on one stream.
 * The caller still owns and passes every input and the output.
 */
#define PKV_STATIC_WS_BYTES ((size_t)8 << 20)

PKV_API int pkv_paged_decode_static_ws(const uint16_t* q, const uint16_t* k_cache,
                                       const uint16_t* v_cache, pkv_cache_desc cache,
                                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                                       const int32_t* context_lens, int32_t num_seqs,
                                       int32_t num_q_heads, float scale,
                                       const pkv_decode_plan* plan, uint16_t* out,
                                       void* stream);

/*
 * Decode step with the KV store fused in ["nano-vllm 深度分析报告", table "可复用的模式与技巧":
 * the store of the step's new tokens precedes attention; fusing the two removes one launch].
 * Equivalent to pkv_kv_store(k_new, v_new, slot_mapping, num_seqs, ...) followed by
 * pkv_paged_decode(...) when, as in a decode step, slot_mapping[b] is the slot of position
 * context_lens[b] - 1 of sequence b (or -1 for a padded entry with context 0):
 *   - k_new[b], v_new[b] are written to slot_mapping[b] (skipped when -1) by the call's first
 *     grid, which also plans the attention work unless the plan is reused; the attention grid
 *     starts once that grid is complete and reads all ctx positions from the cache, so the
 *     result equals store-then-decode bit for bit, with one launch fewer than store, plan and
 *     decode. (With a reused plan, pkv_kv_store then pkv_paged_decode measured ~0.4% faster on
 *     a B300: this call's store also checks every slot against the block table.)
 *   - a slot outside the cache is skipped and raises PKV_DEVERR_BAD_SLOT; a slot that is not
 *     the block table's slot of position ctx-1 (or any slot other than -1 for a sequence of
 *     context 0) is still written and raises PKV_DEVERR_BAD_SLOT; the output row of that
 *     sequence is then unspecified.
 *   k_new, v_new  device, [num_seqs, num_kv_heads, head_dim] bf16 (one new token per sequence)
 *   slot_mapping  device, [num_seqs] int32
 * Other arguments as pkv_paged_decode; k_cache and v_cache are written.
 */
PKV_API int pkv_paged_decode_store(const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                                   const int32_t* slot_mapping, uint16_t* k_cache,
                                   uint16_t* v_cache, pkv_cache_desc cache,
                                   const int32_t* block_tables, int32_t max_blocks_per_seq,
                                   const int32_t* context_lens, int32_t num_seqs,
                                   int32_t num_q_heads, float scale, const pkv_decode_plan* plan,
                                   uint16_t* out, void* workspace, size_t workspace_bytes,
                                   void* stream);

/* Device workspace bytes pkv_paged_prefill needs (a work counter, padded). */
#define PKV_PREFILL_WORKSPACE_BYTES 256

/*
 * Varlen causal paged prefill [P1 PagedAttention; P3 prefix-cache hits share blocks].
 * Sequence b has q_len = cu_seqlens_q[b+1] - cu_seqlens_q[b] new tokens (rows cu_seqlens_q[b] ..
 * of q, k, v) and k_len = cu_seqlens_k[b+1] - cu_seqlens_k[b] keys. The first P = k_len - q_len
 * keys are a cached prefix (possibly blocks shared with other sequences); the rest are the new
 * tokens. New query i attends keys 0 .. P + i (causal, aligned to the end).
 *   q             device, [total_q, num_q_heads, head_dim] bf16
 *   k, v          device, [total_q, num_kv_heads, head_dim] bf16: the new tokens
 *   cu_seqlens_q, cu_seqlens_k  device, [num_seqs + 1] int32, non-decreasing, starting at 0
 *   max_seqlen_q  host int, >= every q_len
 *   block_tables  device [num_seqs, max_blocks_per_seq] int32, or NULL.
 *       Non-NULL: every key (prefix and new) is read through the block table, so the new tokens
 *       must already have been stored with pkv_kv_store (as the engine does before attention).
 *       NULL: there is no prefix (cu_seqlens_k must equal cu_seqlens_q) and keys are read from
 *       k and v directly; k_cache and v_cache may then be NULL.
 *   out           device, [total_q, num_q_heads, head_dim] bf16
 *   workspace     device, >= PKV_PREFILL_WORKSPACE_BYTES, 16-byte aligned, owned by the caller;
 *                 need not be initialised (the call resets what must start at zero on `stream`
 *                 before the attention grid runs). Calls that may run at the same time need
 *                 distinct workspaces. Fewer bytes return PKV_ERR_WORKSPACE_TOO_SMALL before
 *                 anything is enqueued. With workspace_bytes >= pkv_prefill_workspace_bytes(
 *                 num_seqs), a one-CTA plan kernel first numbers only the query tiles each
 *                 sequence has, so that the attention grid claims no empty work (a decode row
 *                 in a batch with long prefill rows would otherwise cost ceil(max_seqlen_q /
 *                 tile) claims), and puts sequences whose tiles are at least half full (prefill
 *                 rows) in one queue and the rest (decode rows) in another; half the grid starts
 *                 on each queue, so tensor work and K/V streaming overlap on every SM. The
 *                 attention grid is the plan's programmatic dependent.
 * Runs on the tcgen05 tensor cores (bf16 operands, fp32 accumulation in tensor memory); supports
 * head_dim 128 and group sizes 1, 2, 4, 8 (other shapes return PKV_ERR_UNSUPPORTED). A persistent
 * grid (two CTAs per SM) claims (sequence, kv head, query tile) items from the counter.
 */
/*
 * Workspace bytes with which pkv_paged_prefill numbers a call's work densely (see above):
 * PKV_PREFILL_WORKSPACE_BYTES plus two ints per sequence and one more, rounded up to 256 bytes.
 * Pure host function; returns PKV_PREFILL_WORKSPACE_BYTES for num_seqs < 0.
 */
PKV_API size_t pkv_prefill_workspace_bytes(int32_t num_seqs);

PKV_API int pkv_paged_prefill(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                      const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t num_seqs,
                      int32_t total_q, int32_t max_seqlen_q, const int32_t* block_tables,
                      int32_t max_blocks_per_seq, const uint16_t* k_cache,
                      const uint16_t* v_cache, pkv_cache_desc cache, int32_t num_q_heads,
                      float scale, uint16_t* out, void* workspace, size_t workspace_bytes,
                      void* stream);

/*
 * Read and clear the device error word of the current CUDA context (PKV_DEVERR_* bits; one word
 * per context, normally one per device). Synchronises the device first; not for use inside stream
 * capture. The library keeps its per-context state (this word's address, kernel attributes) under
 * the driver's unique context id, so a context created by the caller, or the primary context that
 * replaces one destroyed by cudaDeviceReset, gets its own.
 */
PKV_API int pkv_get_device_error(int32_t* flags);

/*
 * Diagnostic for the failure-detection path: launches one CTA that waits on a barrier nothing will
 * ever complete. The wait is bounded like every pipeline wait in the kernels: after one second it
 * gives up, sets PKV_DEVERR_TIMEOUT in the device error word and the CTA exits, so the context
 * stays usable. Enqueued on `stream`; read the result with pkv_get_device_error().
 */
PKV_API int pkv_selftest_bounded_wait(void* stream);

/* Text for a PKV_* status code (static storage). */
PKV_API const char* pkv_status_string(int status);

/* Message for the last failing call on this thread ("" if none). */
PKV_API const char* pkv_last_error(void);

/* ABI version: major * 10000 + minor * 100 + patch. 0.2.0 added the prefill workspace. */
#define PKV_VERSION 202
PKV_API int pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H_ */
