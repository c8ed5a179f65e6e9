// kernels.h -- launchers of the paged KV-cache kernels (internal to libpagedkv.so).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pagedkv.h"

namespace pkv {

// Tokens per decode tile for a given number of query heads per CTA; split chunks are multiples
// of the largest tile (128 tokens).
constexpr int kSplitQuantum = 128;

// Decode kernel instances: head_dim {128, 64} x query heads per CTA {4, 2, 1}.
constexpr int kDecodeInstances = 6;

// State of the library in one CUDA context. Module globals (the device error word, the static
// decode workspace) and kernel attributes exist once per context, so they are looked up or set
// once per context and kept under the driver's unique context id: a context the caller created
// itself, or the new primary context after cudaDeviceReset, gets an entry of its own.
struct ContextState {
  unsigned long long ctx_id = 0;
  int device = 0;
  int num_sms = 0;
  int* flags = nullptr;                   // this context's copy of the device error word
  int decode_ctas[kDecodeInstances] = {};  // resident CTAs per SM of each decode instance
};

// The calling thread's current context (its primary context is bound first if none is). The
// first call in a context sets it up: symbol lookups, shared-memory opt-ins, occupancy queries.
// Returns PKV_OK or a PKV_ERR_* status with the message in pkv_last_error().
int context_state(const ContextState** out);

// Unique id of the calling thread's current context (binding the device's primary context if
// none is current yet). Returns PKV_OK or a PKV_ERR_* status.
int current_context_id(unsigned long long* id, int* device);

// Records "what: <CUDA error>" as the message pkv_last_error() returns; returns PKV_ERR_CUDA.
int report_cuda_error(cudaError_t e, const char* what);

// One-time attributes of the attention kernels in the current context (shared-memory opt-in,
// carve-out); the decode call also reports each instance's resident CTAs per SM.
cudaError_t configure_decode_kernels(int (&ctas_per_sm)[kDecodeInstances]);
cudaError_t configure_prefill_kernel();

struct DecodeWorkspace {
  uint32_t* header;    // [0] claim counter, [1] number of items, [2] chunk length (tokens)
  int2* items;         // (sequence, chunk) pairs, B * max_splits entries at most
  uint32_t* counters;  // chunks finished per (sequence, head group, consumer warp)
  float* part_acc;     // [B, max_splits, Hq, D] un-normalised partial outputs
  float2* part_ml;     // [B, max_splits, Hq, D / 64] (running max in log2 units, denominator)
};

size_t decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                              int32_t max_splits, DecodeWorkspace* carve, void* base);

cudaError_t launch_kv_store(const uint16_t* k, const uint16_t* v, const int32_t* slot_mapping,
                            int32_t num_tokens, uint16_t* k_cache, uint16_t* v_cache,
                            const pkv_cache_desc& cache, int num_sms, int* flags,
                            cudaStream_t stream);

struct DecodeArgs {
  const uint16_t* q;
  const uint16_t* k_cache;
  const uint16_t* v_cache;
  pkv_cache_desc cache;
  const int32_t* block_tables;
  int32_t max_blocks;
  const int32_t* context_lens;
  int32_t num_seqs;
  int32_t num_q_heads;
  float scale;
  int32_t split_tokens;  // chunk length (fixed) or smallest chunk length (auto), multiple of 128
  int32_t max_splits;    // ceil(max_context_len / split_tokens)
  bool auto_split;       // choose the chunk length on the device from the actual lengths
  uint16_t* out;
  DecodeWorkspace ws;
  int* flags;
  // the step's store (all null for a plain decode): newest token of sequence b, [B, Hkv, D],
  // written to slot_mapping[b] by the plan grid before the decode grid reads the cache
  const uint16_t* k_new = nullptr;
  const uint16_t* v_new = nullptr;
  const int32_t* slot_mapping = nullptr;
  const int* ctas_per_sm = nullptr;  // ContextState::decode_ctas of the current context
  // The workspace holds the device plan of an earlier call with the same plan and lengths: no
  // plan kernel (with a store, a store-only grid runs before the decode kernel instead).
  bool reuse_plan = false;
};

// Whole-block moves: mode 0 copies (src, dst) pairs inside the caches, mode 1 gathers blocks
// into buf_k/buf_v, mode 2 scatters them back from buf_k/buf_v.
cudaError_t launch_block_move(int mode, uint16_t* k_cache, uint16_t* v_cache,
                              const int32_t* ids, int32_t n, const pkv_cache_desc& cache,
                              uint16_t* buf_k, uint16_t* buf_v, int num_sms, int* flags,
                              cudaStream_t stream);

// Chained xxhash64 of every full block of each sequence (one thread per sequence).
cudaError_t launch_block_hashes(const int32_t* token_ids, const int32_t* cu_seqlens,
                                int32_t num_seqs, int32_t block_size, int32_t max_blocks,
                                uint64_t* out, int* flags, cudaStream_t stream);

// Rows of the K/V TMA box the decode kernel expects (tile tokens, or the block size if smaller).
int decode_box_rows(int head_dim, int group, int block_size);

// The plan grid of a decode call: one CTA turns context_lens into the chunk length and the
// longest-first list of (sequence, chunk) items for a decode grid with `slots` resident CTAs and
// head_groups items per (sequence, chunk), and resets the claim counter and the first
// counters_per_seq merge counters of every split sequence; with a.k_new, more CTAs store the
// step's new rows. The decode grid is launched after it as a programmatic dependent.
cudaError_t launch_decode_plan(const DecodeArgs& a, int32_t head_groups, int32_t slots,
                               int32_t counters_per_seq, int32_t cap_tokens, int num_sms,
                               cudaStream_t stream);

// Decode on the tensor cores with keys on the MMA's M dimension (head_dim 128, any group size):
// its shared-memory opt-in, the rows of its K/V TMA boxes (128-byte swizzle, 64 dims wide), and
// the plan plus decode launch. q is read through tmap_q (boxes of 64 dims x G heads x 1 row),
// K/V through tmap_k/tmap_v (boxes of decode_tc_box_rows rows) and, for a chunk's partial last
// tile, through tail[] = {K, V with 64-row boxes, K, V with 32-row boxes}.
cudaError_t configure_decode_tc_kernels();
int decode_tc_box_rows(int block_size);
cudaError_t launch_paged_decode_tc(const DecodeArgs& a, const CUtensorMap& tmap_q,
                                   const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                                   const CUtensorMap* tail, int num_sms, cudaStream_t stream);

// Returns a CUDA error, or cudaErrorNotSupported for shapes without an instance.
cudaError_t launch_paged_decode(const DecodeArgs& a, const CUtensorMap& tmap_k,
                                const CUtensorMap& tmap_v, int num_sms, cudaStream_t stream);

struct PrefillArgs {
  const uint16_t* q;
  const uint16_t* k;
  const uint16_t* v;
  const int32_t* cu_seqlens_q;
  const int32_t* cu_seqlens_k;
  int32_t num_seqs;
  int32_t total_q;
  int32_t max_seqlen_q;
  const int32_t* block_tables;
  int32_t max_blocks;
  pkv_cache_desc cache;
  int32_t num_q_heads;
  float scale;
  uint16_t* out;
  int* flags;
  int32_t* item_counter;  // device, in the caller's workspace
  // Dense item numbering (nullptr: ids run over num_seqs x num_kv_heads x ceil(max_seqlen_q /
  // positions per tile), and the grid skips the ids of query tiles a sequence does not have):
  // 2 x num_seqs + 1 ints in the caller's workspace, which a one-CTA plan kernel fills before
  // the attention grid starts: each position's first item id (num_seqs + 1 ints), then the
  // sequence at each position (heavy sequences first). item_counter then holds four ints.
  int32_t* item_prefix = nullptr;
};

// Query positions per 128-row prefill tile, and rows per K/V TMA box.
int prefill_positions_per_tile(int group);
int prefill_kv_box_rows(int block_size, bool paged);

// The store of a decode step alone (the plan grid's store CTAs): row b of a.k_new / a.v_new to
// slot a.slot_mapping[b], checked against the block table.
cudaError_t launch_decode_store_rows(const DecodeArgs& a, int num_sms, cudaStream_t stream);

cudaError_t launch_paged_prefill(const PrefillArgs& a, const CUtensorMap& tmap_q,
                                 const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                                 int num_sms, cudaStream_t stream);

}  // namespace pkv
