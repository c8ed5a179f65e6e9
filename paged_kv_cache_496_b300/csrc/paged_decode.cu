// paged_decode.cu -- paged decode attention (one query per sequence) for sm_103a.
//
// Source: "DeepSeek研究员1200行代码复刻vLLM，H800硬件实测性能反超原版" (QbitAI), section
// "vLLM是什么？": keys and values of a sequence sit in fixed-size blocks found through its block
// table, and the attention kernel fetches the blocks one by one. The result is ordinary softmax
// attention over the sequence's tokens; only the addressing is paged.
//
// Design (B300-first, not a translation of any earlier kernel):
//  * Work item = (sequence b, group of GH query heads sharing one kv head, context chunk s).
//    A one-CTA plan kernel turns context_lens into a list of (b, s) items on the device, so the
//    host never synchronises; a persistent grid claims items with an atomic counter and keeps
//    its TMA pipeline full across item boundaries.
//  * Warp specialisation: one producer warp walks the block table (32 entries per coalesced
//    load, kept in registers, the next 32 prefetched) and issues one 3-D TMA box per (block, tile)
//    for K and for V into a multi-stage shared-memory ring guarded by mbarriers (three stages at
//    D=128 with two CTAs per SM); four consumer warps compute.
//  * Consumers: eight lanes share one token row (each lane owns D/8 of the dims). A lane group
//    holds N (token, head) pairs (16 for groups of four heads, else 8); their q.k partial sums are
//    reduced with a reduce-scatter that leaves N/8 full scores per lane. q comes from a per-warp
//    bf16 copy and the scale is applied to the reduced scores. Online softmax runs in log2 units
//    in fp32 with a lazy rescale (only when a head's max grows by more than 2^8); products use
//    the packed fp32x2 FMA. The four warps' partial (max, sum, acc) are merged through one
//    shared-memory buffer, guarded so that no warp overwrites it before all have read it.
//  * Long contexts are cut into chunks (flash-decoding split). The plan kernel picks the chunk
//    length from the actual total work (so a few long sequences are spread over all SMs while a
//    large batch is not split at all). A chunk writes fp32 partials (un-normalised acc, running
//    max, denominator) to the caller's workspace; the CTA that finishes the last chunk of a
//    (sequence, head group) merges them with log-sum-exp weights, so no extra launch is needed.
#include "common.cuh"
#include "kernels.h"

namespace pkv {

namespace {

constexpr int kMetaFirst = 1;  // first tile of an item: load q, reset the running state
constexpr int kMetaLast = 2;   // last tile of an item: merge warps and write the result
constexpr int kMetaZero = 4;   // an item with no tokens (context 0): write zeros
constexpr int kMetaDone = 8;   // no more items
constexpr float kTau = 8.0f;   // lazy-rescale threshold (log2 units)

struct alignas(16) StageMeta {
  int32_t b, x, split, nsplit;
  int32_t tok0, tok_end, flags, pad;
};

struct DecodeParams {
  const uint16_t* q;
  const int32_t* block_tables;
  const int32_t* context_lens;
  uint16_t* out;
  float* part_acc;
  float2* part_ml;
  const int2* items;
  uint32_t* header;    // [0] claim counter, [1] item count, [2] chunk length in tokens
  uint32_t* counters;  // per (sequence, head group, consumer warp): chunks finished
  int* flags;
  int32_t max_blocks;
  int32_t num_seqs;
  int32_t num_q_heads;
  int32_t head_groups;     // groups of GH query heads: num_q_heads / GH
  int32_t groups_per_kv;   // head groups that share one kv head: (Hq / Hkv) / GH
  int32_t block_size;
  int32_t num_blocks;
  int32_t max_splits;
  int32_t cap_tokens;  // contexts are clamped to this many tokens (table and plan capacity)
  float qk_scale_log2;
};

template <int D, int GH>
struct Traits {
  static constexpr int kWarps = 4;
  static constexpr int kThreads = (kWarps + 1) * 32;
  // Each lane starts with kN partial scores, one per (token, head) pair of its lane group, and
  // ends the reduce-scatter holding kVPL full scores. Four-head groups take 16 pairs (4 tokens),
  // which doubles the independent work per softmax step; smaller groups take 8.
  static constexpr int kN = GH == 4 ? 16 : 8;
  static constexpr int kVPL = kN / 8;
  static constexpr int kTPG = kN / GH;                 // tokens per lane group per tile
  static constexpr int kTokPerWarp = 4 * kTPG;
  static constexpr int kTileT = kWarps * kTokPerWarp;  // tokens per tile (64 or 128)
  static constexpr int kChunks = D / 64;               // 16-byte chunks per lane per row
  static constexpr int kPairs = D / 16;                // fp32 pairs per lane per row
  static constexpr int kRowBytes = D * 2;
  static constexpr int kTileBytes = kTileT * kRowBytes;
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kQBytes = GH * D * 2;
  // acc [GH][D], then m [GH], then l [GH]; padded so every warp's slot is 16-byte aligned
  static constexpr int kCbFloats = (GH * D + 2 * GH + 3) / 4 * 4;
  // Two CTAs per SM: keep each CTA within 113 KB of shared memory (three K+V stages at D=128).
  static constexpr int kSmemBudget = 113 * 1024;
  static constexpr int kFixedBytes =
      kWarps * kCbFloats * 4 + kWarps * kChunks * 4 * 8 * GH * 4 + 8 * 32 + 160;
  static constexpr int kStagesRaw = (kSmemBudget - kFixedBytes) / (kStageBytes + kQBytes);
  static constexpr int kStages = kStagesRaw < 2 ? 2 : (kStagesRaw > 8 ? 8 : kStagesRaw);
  static constexpr int kMaxSub = kTileT / 16;        // TMA boxes per tile at block_size 16
  // Per-warp copy of the item's q as bf16 pairs: for (chunk c, word w) lane j of a group reads
  // the GH heads' pairs as one 4*GH-byte slot; the 8 slots are consecutive, conflict-free.
  static constexpr int kQfBytesPerWarp = kChunks * 4 * 8 * GH * 4;
  static constexpr int kOffTiles = 0;
  static constexpr int kOffQ = kOffTiles + kStages * kStageBytes;
  static constexpr int kOffQf = kOffQ + kStages * kQBytes;
  static constexpr int kOffCb = kOffQf + kWarps * kQfBytesPerWarp;
  static constexpr int kOffMeta = kOffCb + kWarps * kCbFloats * 4;
  static constexpr int kOffBar = (kOffMeta + kStages * (int)sizeof(StageMeta) + 15) / 16 * 16;
  static constexpr int kSmemBytes = kOffBar + (2 * kStages + 2) * 8;
  static_assert(kTPG * GH == kN && (kN == 8 || kN == 16), "lane-group pair layout");
  static_assert(kCbFloats % 4 == 0, "float4 stores into the combine slots");
  static_assert(kQBytes % 16 == 0 && kOffQ % 128 == 0 && kOffCb % 16 == 0, "smem alignment");
  static_assert(kOffMeta % 16 == 0 && kOffBar % 16 == 0, "smem alignment");
  static_assert(kStageBytes % 1024 == 0 && kTileBytes % 1024 == 0, "TMA destinations");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
};

// ---------------------------------------------------------------------------------------------
// Plan: context_lens -> chunk length and list of (sequence, chunk) items; resets the counters.
// ---------------------------------------------------------------------------------------------

constexpr int kPlanThreads = 1024;
// Chunk length when splitting: about 2/5 of one resident CTA's share of the work, so every CTA
// takes two or three chunks. Finer chunks pay the per-item cost (q load, warp combine, partial
// write, final merge) more often than they gain in balance: on a B300, 4 x 32768 + 60 short
// sequences run 16% faster at 2048-token chunks than at 512.
constexpr double kChunkShare = 0.4;
constexpr int kSizeBuckets = 32;  // length classes of the remainder items (longest-first order)

struct PlanParams {
  const int32_t* context_lens;
  int2* items;
  uint32_t* header;
  uint32_t* counters;
  int* flags;
  int32_t num_seqs;
  int32_t cap_tokens;
  int32_t split_floor;   // smallest chunk length (tokens, multiple of 128)
  int32_t fixed_split;   // > 0: use exactly this chunk length
  int32_t head_groups;
  int32_t slots;         // resident CTAs of the decode grid
  int32_t counters_per_seq;  // merge counters per sequence (0 when nothing can be split)
  // The store of a decode step (pkv_paged_decode_store; k_new == nullptr otherwise): the CTAs
  // after the first write row b of k_new / v_new ([B, Hkv, D]) to slot slot_mapping[b].
  const uint16_t* k_new;
  const uint16_t* v_new;
  const int32_t* slot_mapping;
  uint16_t* k_cache;
  uint16_t* v_cache;
  const int32_t* block_tables;
  int32_t max_blocks;
  int32_t block_size;
  int32_t num_blocks;
  int32_t row_chunks;  // 16-byte chunks in one token row of all kv heads (Hkv * D / 8)
  int32_t do_plan;     // 0: the grid only stores (CTA 0 has nothing to do)
};

// The store of a decode step, in the CTAs of the plan grid after the first: row b of k_new / v_new
// goes to cache slot slot_mapping[b] (-1 is skipped; any other slot outside the cache is skipped
// and flagged), copied in 16-byte chunks across the grid. A slot that is not the block table's
// slot of position context_lens[b] - 1 is still written and flagged. The decode grid waits for
// this whole grid, so its copies read the new rows.
__device__ void store_new_rows(const PlanParams& pp) {
  const int rc = pp.row_chunks;
  const int64_t total = (int64_t)pp.num_seqs * rc;
  const int64_t stride = (int64_t)(gridDim.x - 1) * blockDim.x;
  const int64_t cap = (int64_t)pp.num_blocks * pp.block_size;
  const int lbs = __ffs(pp.block_size) - 1;
  for (int64_t i = (int64_t)(blockIdx.x - 1) * blockDim.x + threadIdx.x; i < total; i += stride) {
    const int b = (int)(i / rc);
    const int c = (int)(i - (int64_t)b * rc);
    const int slot = __ldg(pp.slot_mapping + b);
    if (slot == -1) continue;
    const bool writes = slot >= 0 && slot < cap;
    if (c == 0) {
      int ctx = __ldg(pp.context_lens + b);
      ctx = ctx < pp.cap_tokens ? ctx : pp.cap_tokens;
      bool on_table = false;
      if (writes && ctx > 0) {
        const int pos = ctx - 1;
        const int e = pos >> lbs;
        const int blk = e < pp.max_blocks ? __ldg(pp.block_tables + (int64_t)b * pp.max_blocks + e)
                                          : -1;
        on_table = slot == blk * pp.block_size + (pos & (pp.block_size - 1));
      }
      if (!on_table) raise_flag(pp.flags, PKV_DEVERR_BAD_SLOT);
    }
    if (!writes) continue;
    const int64_t src = (int64_t)b * rc + c, dst = (int64_t)slot * rc + c;
    reinterpret_cast<uint4*>(pp.k_cache)[dst] = __ldg(reinterpret_cast<const uint4*>(pp.k_new) + src);
    reinterpret_cast<uint4*>(pp.v_cache)[dst] = __ldg(reinterpret_cast<const uint4*>(pp.v_new) + src);
  }
}

__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* warp_sums,
                                                         uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kFullMask, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(kFullMask, w, o);
      if (lane >= o) w += y;
    }
    warp_sums[lane] = w;
  }
  __syncthreads();
  const uint32_t r = incl - v + (warp > 0 ? warp_sums[warp - 1] : 0u);
  *total = warp_sums[31];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kPlanThreads) decode_plan_kernel(const PlanParams pp) {
  // the decode grid may be scheduled now: it sets up its barriers, then waits for this grid
  allow_dependent_launch();
  // this grid is itself a programmatic dependent of the previous work in the stream
  grid_dependency_wait();
  if (blockIdx.x > 0) {
    store_new_rows(pp);
    return;
  }
  if (!pp.do_plan) return;
  __shared__ uint32_t warp_sums[32];
  __shared__ int32_t split_sh;
  const int tid = threadIdx.x;
  const int per = (pp.num_seqs + kPlanThreads - 1) / kPlanThreads;
  const int b0 = min(pp.num_seqs, tid * per);
  const int b1 = min(pp.num_seqs, b0 + per);
  // total tokens (for the chunk length) -- in units of 16 tokens to stay within 32 bits
  uint32_t local_tok = 0;
  for (int b = b0; b < b1; ++b) {
    int ctx = pp.context_lens[b];
    if (ctx > pp.cap_tokens) {
      raise_flag(pp.flags, PKV_DEVERR_CTX_CLAMPED);
      ctx = pp.cap_tokens;
    }
    local_tok += ctx > 0 ? (uint32_t)((ctx + 15) / 16) : 0u;
  }
  uint32_t total16 = 0;
  block_exclusive_scan(local_tok, warp_sums, &total16);
  if (tid == 0) {
    int32_t S = pp.fixed_split;
    if (S <= 0) {
      // a chunk of about kChunkShare of a resident CTA's share, to the nearest 256 tokens
      const double per_slot = (double)total16 * 16.0 * pp.head_groups / (double)pp.slots;
      double want = per_slot * kChunkShare;
      if (want > (double)pp.cap_tokens) want = (double)pp.cap_tokens;
      int64_t w = ((int64_t)want + 128) / 256 * 256;
      if (w < pp.split_floor) w = pp.split_floor;
      S = (int32_t)w;
    }
    split_sh = S;
    pp.header[2] = (uint32_t)S;
  }
  __syncthreads();
  const int32_t S = split_sh;
  // Items in roughly longest-first order, so the last claims are the smallest: first every
  // full-length chunk, then the remainders (a split sequence's last, partial chunk and every
  // unsplit sequence) by decreasing length, in kSizeBuckets buckets; items of context 0 last.
  __shared__ uint32_t bucket_count[kSizeBuckets + 1], bucket_next[kSizeBuckets + 1];
  if (tid <= kSizeBuckets) bucket_count[tid] = 0u;
  uint32_t local_full = 0;
  for (int b = b0; b < b1; ++b) {
    const int ctx = min(pp.context_lens[b], pp.cap_tokens);
    if (ctx <= 0) continue;
    const int full = ctx / S;
    local_full += (uint32_t)full;
    // only split sequences use merge counters
    if ((ctx + S - 1) / S > 1)
      for (int i = 0; i < pp.counters_per_seq; ++i)
        pp.counters[(int64_t)b * pp.counters_per_seq + i] = 0u;
  }
  uint32_t total_full = 0;
  uint32_t pos = block_exclusive_scan(local_full, warp_sums, &total_full);
  // bucket of a sequence's remainder: kSizeBuckets - 1 (longest) .. 0; context 0 -> kSizeBuckets
  auto bucket_of = [&](int ctx) -> int {
    if (ctx <= 0) return kSizeBuckets;
    const int rem = ctx - (ctx / S) * S;
    if (rem == 0) return -1;  // no remainder: all chunks are full
    return (int)(((int64_t)rem * kSizeBuckets - 1) / S);
  };
  for (int b = b0; b < b1; ++b) {
    const int ctx = min(pp.context_lens[b], pp.cap_tokens);
    const int full = ctx > 0 ? ctx / S : 0;
    for (int s = 0; s < full; ++s) pp.items[pos++] = make_int2(b, s);
    const int k = bucket_of(ctx);
    if (k >= 0) atomicAdd(&bucket_count[k], 1u);
  }
  __syncthreads();
  if (tid == 0) {
    uint32_t at = total_full;
    for (int k = kSizeBuckets - 1; k >= 0; --k) {
      bucket_next[k] = at;
      at += bucket_count[k];
    }
    bucket_next[kSizeBuckets] = at;
  }
  __syncthreads();
  for (int b = b0; b < b1; ++b) {
    const int ctx = min(pp.context_lens[b], pp.cap_tokens);
    const int k = bucket_of(ctx);
    if (k < 0) continue;
    const uint32_t at = atomicAdd(&bucket_next[k], 1u);
    pp.items[at] = make_int2(b, ctx > 0 ? ctx / S : 0);
  }
  uint32_t total = total_full;
  for (int k = 0; k <= kSizeBuckets; ++k) total += bucket_count[k];
  if (tid == 0) {
    pp.header[1] = total;  // number of (sequence, chunk) items
    pp.header[0] = 0u;     // claim counter
    pp.header[3] = 0u;     // producers done (release_claims)
  }
}

// ---------------------------------------------------------------------------------------------
// Register-level pieces of the consumer
// ---------------------------------------------------------------------------------------------

// N partial sums per lane, one per (token, head) pair idx = token * GH + head of the lane group,
// summed over the group's eight lanes by three halving exchanges (lane masks 4, 2, 1). Afterwards
// lane j holds the full sums of pairs j*N/8 .. j*N/8 + N/8 - 1 in v[0 .. N/8 - 1].
template <int N>
__device__ __forceinline__ void reduce_scatter(float (&v)[N], int j) {
#pragma unroll
  for (int step = 0; step < 3; ++step) {
    const int m = 4 >> step;
    const int half = N >> (step + 1);
    const bool up = j & m;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = up ? v[i] : v[i + half];
      const float keep = up ? v[i + half] : v[i];
      v[i] = keep + __shfl_xor_sync(kFullMask, send, m);
    }
  }
}

// After the reduce-scatter, lane bit b (< 3) moves a held pair index by 2^b * N/8 and the group
// bits (3, 4) select other tokens. A lane bit that moves the index by a multiple of GH keeps the
// head and changes only the token, so reducing over those bits combines one head's tokens.
template <int N, int GH>
__device__ __forceinline__ float max_over_tokens(float x) {
#pragma unroll
  for (int b = 0; b < 5; ++b)
    if (b >= 3 || ((1 << b) * (N / 8)) % GH == 0)
      x = fmaxf(x, __shfl_xor_sync(kFullMask, x, 1 << b));
  return x;
}

template <int N, int GH>
__device__ __forceinline__ float sum_over_tokens(float x) {
#pragma unroll
  for (int b = 0; b < 5; ++b)
    if (b >= 3 || ((1 << b) * (N / 8)) % GH == 0) x += __shfl_xor_sync(kFullMask, x, 1 << b);
  return x;
}

// The last warp to finish a (sequence, head group, output slice) of a split sequence merges all
// chunk partials: o = sum_s 2^(m_s - M) acc_s / sum_s 2^(m_s - M) l_s, with a running max over
// batches of chunks. A batch is one round of loads for all of the warp's outputs: lane u holds
// chunk s0 + u's (m, l) and every lane the accumulators of its output pairs for all chunks of the
// batch (16 loads in flight per lane); the batch maximum and the weights travel by shuffles. The
// merge ends the launch for the sequence whose last chunk is claimed late, so its dependent L2
// round trips (partials written by other SMs) are kept few. Out of line: it runs once per split
// sequence, and the decode loop runs faster with less code in it.
template <int D, int GH, int kWarps>
__device__ __noinline__ void merge_chunks(const DecodeParams& p, int b, int x, int nsplit, int warp,
                                          int lane) {
  constexpr int kO = (GH * D + kWarps * 64 - 1) / (kWarps * 64);  // output pairs per lane
  constexpr int kB = 16 / kO;  // chunks per batch: 16 accumulator loads in flight per lane
  const int o0 = 64 * warp + 2 * lane;
  if (o0 >= GH * D) return;  // warp-uniform: GH * D is a multiple of 64
  int64_t pbase[kO];  // partial index of chunk 0 for output k: (b, split 0, head)
  int dd[kO];
  float M[kO], dl[kO], n0[kO], n1[kO];
#pragma unroll
  for (int k = 0; k < kO; ++k) {
    const int o = min(o0 + k * kWarps * 64, GH * D - 2);  // past the end: a harmless duplicate
    dd[k] = o % D;
    pbase[k] = (int64_t)b * p.max_splits * p.num_q_heads + x * GH + o / D;
    M[k] = -INFINITY;
    dl[k] = 0.f;
    n0[k] = 0.f;
    n1[k] = 0.f;
  }
  for (int s0 = 0; s0 < nsplit; s0 += kB) {
    float2 ml[kO], a[kO][kB];
#pragma unroll
    for (int k = 0; k < kO; ++k) {
      ml[k] = make_float2(-INFINITY, 0.f);
      if (lane < kB && s0 + lane < nsplit)
        ml[k] = __ldcg(p.part_ml + (pbase[k] + (int64_t)(s0 + lane) * p.num_q_heads) * (D / 64) +
                       dd[k] / 64);
#pragma unroll
      for (int u = 0; u < kB; ++u) {
        a[k][u] = make_float2(0.f, 0.f);
        if (s0 + u < nsplit)
          a[k][u] = __ldcg(reinterpret_cast<const float2*>(
              p.part_acc + (pbase[k] + (int64_t)(s0 + u) * p.num_q_heads) * D + dd[k]));
      }
    }
#pragma unroll
    for (int k = 0; k < kO; ++k) {
      float mb = ml[k].x;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mb = fmaxf(mb, __shfl_xor_sync(kFullMask, mb, off));
      const float mnew = fmaxf(M[k], mb);
      if (mnew == -INFINITY) continue;  // nothing seen yet (warp-uniform)
      const float keep = M[k] == -INFINITY ? 0.f : fast_exp2(M[k] - mnew);
      const float w = ml[k].x == -INFINITY ? 0.f : fast_exp2(ml[k].x - mnew);
      dl[k] = dl[k] * keep + w * ml[k].y;
      float s_0 = n0[k] * keep, s_1 = n1[k] * keep;
#pragma unroll
      for (int u = 0; u < kB; ++u) {
        const float wu = __shfl_sync(kFullMask, w, u);
        s_0 += wu * a[k][u].x;
        s_1 += wu * a[k][u].y;
      }
      n0[k] = s_0;
      n1[k] = s_1;
      M[k] = mnew;
    }
  }
#pragma unroll
  for (int k = 0; k < kO; ++k) {
    float den = dl[k];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(kFullMask, den, off);
    const int o = o0 + k * kWarps * 64;
    if (o >= GH * D) continue;
    const float inv = den > 0.f ? 1.f / den : 0.f;
    *reinterpret_cast<__nv_bfloat162*>(
        p.out + ((int64_t)b * p.num_q_heads + x * GH + o / D) * D + o % D) =
        __floats2bfloat162_rn(n0[k] * inv, n1[k] * inv);
  }
}

// ---------------------------------------------------------------------------------------------
// The decode kernel
// ---------------------------------------------------------------------------------------------

template <int D, int GH>
__global__ void __maxnreg__(168)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v,
                        const __grid_constant__ DecodeParams p) {
  using T = Traits<D, GH>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* tiles = smem + T::kOffTiles;
  uint8_t* qbuf = smem + T::kOffQ;
  float* cb = reinterpret_cast<float*>(smem + T::kOffCb);
  StageMeta* meta = reinterpret_cast<StageMeta*>(smem + T::kOffMeta);
  const uint32_t full0 = smem_addr(smem + T::kOffBar);
  const uint32_t empty0 = full0 + T::kStages * 8;
  // combine: all warps wrote their partials (cmb) / all warps finished reading them (cmr)
  const uint32_t cmb = empty0 + T::kStages * 8;
  const uint32_t cmr = cmb + 8;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < T::kStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, T::kWarps);
    }
    mbar_init(cmb, T::kWarps);
    mbar_init(cmr, T::kWarps);
    fence_barrier_init();
  }
  __syncthreads();
  // Launched as a programmatic dependent of the plan kernel: everything above overlaps the plan;
  // nothing below reads memory before the plan (and all earlier work) has completed. The next
  // work in the stream may then be scheduled; it waits for this grid before touching memory.
  grid_dependency_wait();
  allow_dependent_launch();

  if (warp == T::kWarps) {
    // =============================== producer warp ===============================
    if (lane == 0) {
      tma_prefetch_desc(&tmap_k);
      tma_prefetch_desc(&tmap_v);
    }
    // The header and the work list come from this call's plan kernel or, with a reused plan,
    // from an earlier call on the same workspace. The count is clamped to the list's capacity and
    // items outside this call's batch are skipped (and flagged), so a reuse on the wrong
    // workspace gives wrong outputs but never reaches memory outside the workspace or caches.
    uint32_t n_items = p.header[1];
    const int split = (int)p.header[2];
    if (n_items > (uint32_t)p.num_seqs * (uint32_t)p.max_splits || split < kSplitQuantum) {
      if (lane == 0) raise_flag(p.flags, PKV_DEVERR_INTERNAL);
      n_items = 0;
    }
    const uint32_t total = n_items * (uint32_t)p.head_groups;
    const int bs = p.block_size;
    // block_size is a power of two: shifts and masks instead of divisions by a runtime value
    const int lbs = __ffs(bs) - 1;
    const int box_t = bs < T::kTileT ? bs : T::kTileT;
    const int nsub = T::kTileT / box_t;
    const int ent_per_tile = (T::kTileT + bs - 1) >> lbs;
    uint32_t issue = 0;
    bool ok = true;
    // Block-table window: entries [win_base, win_base + 32) of sequence win_b, one per lane, and
    // the next 32 entries prefetched so that walking on does not stall the pipeline.
    int win_b = -1, win_base = 0, win_val = -1, nxt_val = -1;

    auto claim = [&]() -> uint32_t {
      uint32_t c = 0;
      if (lane == 0) c = atomicAdd(p.header, 1u);
      return __shfl_sync(kFullMask, c, 0);
    };
    // Each stage slot has its own issuing lane (lane == stage): one thread's bulk copies complete
    // one barrier phase at a time, so copies of several stages issued from one thread would
    // queue behind each other (at block size 16 a stage is eight 4 KB boxes plus q). The slot's
    // lane waits until the consumers have released it, then fills it.
    auto acquire = [&](int stage) -> bool {
      int good = 1;
      if (lane == stage)
        good = mbar_wait(empty0 + 8 * stage, ((issue / T::kStages) & 1) ^ 1) ? 1 : 0;
      return __shfl_sync(kFullMask, good, stage) != 0;
    };

    uint32_t c = claim();
    while (ok) {
      const int stage = issue % T::kStages;
      if (c >= total) {
        ok = acquire(stage);
        if (ok && lane == stage) {
          meta[stage].flags = kMetaDone;
          mbar_arrive(full0 + 8 * stage);
        }
        ++issue;
        break;
      }
      const int2 it = p.items[c / (uint32_t)p.head_groups];
      const int x = (int)(c % (uint32_t)p.head_groups);
      const uint32_t c_next = claim();
      const int b = it.x, s = it.y;
      if ((unsigned)b >= (unsigned)p.num_seqs || (unsigned)s >= (unsigned)p.max_splits) {
        if (lane == 0) raise_flag(p.flags, PKV_DEVERR_INTERNAL);
        c = c_next;
        continue;
      }
      int ctx = p.context_lens[b];
      ctx = ctx < p.cap_tokens ? ctx : p.cap_tokens;
      if (ctx <= 0) {
        ok = acquire(stage);
        if (ok && lane == stage) {
          StageMeta m;
          m.b = b; m.x = x; m.split = 0; m.nsplit = 1;
          m.tok0 = 0; m.tok_end = 0; m.flags = kMetaZero; m.pad = 0;
          meta[stage] = m;
          mbar_arrive(full0 + 8 * stage);
        }
        ++issue;
        c = c_next;
        continue;
      }
      const int nsplit = (ctx + split - 1) / split;
      const int tok_begin = s * split;
      const int tok_end = min(ctx, tok_begin + split);
      const int need_ent = (ctx + bs - 1) >> lbs;  // table entries of the whole sequence
      const int32_t* bt_row = p.block_tables + (int64_t)b * p.max_blocks;
      const uint16_t* qsrc = p.q + ((int64_t)b * p.num_q_heads + x * GH) * D;
      const int kv_head = x / p.groups_per_kv;

      for (int tok0 = tok_begin; tok0 < tok_end && ok; tok0 += T::kTileT) {
        const int st = issue % T::kStages;
        const int e0 = tok0 >> lbs;
        if (win_b != b || e0 < win_base || e0 + ent_per_tile > win_base + 32) {
          if (win_b == b && e0 >= win_base + 32 && e0 + ent_per_tile <= win_base + 64) {
            win_base += 32;  // step into the prefetched window
            win_val = nxt_val;
          } else {
            win_b = b;
            win_base = e0;
            const int e = e0 + lane;
            win_val = e < need_ent ? __ldg(bt_row + e) : -1;
          }
          const int e = win_base + 32 + lane;
          nxt_val = e < need_ent ? __ldg(bt_row + e) : -1;
        }
        int rows[T::kMaxSub];
        uint32_t bytes = 0;
#pragma unroll
        for (int sb = 0; sb < T::kMaxSub; ++sb) {
          rows[sb] = -1;
          if (sb < nsub) {
            const int t = tok0 + sb * box_t;
            const int blk = __shfl_sync(kFullMask, win_val, ((t >> lbs) - win_base) & 31);
            if (t < tok_end) {
              if (blk >= 0 && blk < p.num_blocks) {
                rows[sb] = blk * bs + (t & (bs - 1));
                bytes += 2u * (uint32_t)box_t * T::kRowBytes;
              } else if (lane == 0) {
                raise_flag(p.flags, PKV_DEVERR_BAD_BLOCK);
              }
            }
          }
        }
        const bool first = tok0 == tok_begin;
        if (first) bytes += T::kQBytes;
        ok = acquire(st);
        if (ok && lane == st) {
          StageMeta m;
          m.b = b; m.x = x; m.split = s; m.nsplit = nsplit;
          m.tok0 = tok0; m.tok_end = tok_end;
          m.flags = (first ? kMetaFirst : 0) | (tok0 + T::kTileT >= tok_end ? kMetaLast : 0);
          m.pad = 0;
          meta[st] = m;
          const uint32_t fb = full0 + 8 * st;
          mbar_arrive_expect_tx(fb, bytes);
          uint8_t* kdst = tiles + st * T::kStageBytes;
          uint8_t* vdst = kdst + T::kTileBytes;
#pragma unroll
          for (int sb = 0; sb < T::kMaxSub; ++sb) {
            if (sb < nsub && rows[sb] >= 0) {
              const int off = sb * box_t * T::kRowBytes;
              tma_load_3d(smem_addr(kdst + off), &tmap_k, 0, kv_head, rows[sb], fb);
              tma_load_3d(smem_addr(vdst + off), &tmap_v, 0, kv_head, rows[sb], fb);
            }
          }
          if (first) bulk_load(smem_addr(qbuf + st * T::kQBytes), qsrc, T::kQBytes, fb);
        }
        ++issue;
      }
      c = c_next;
    }
    if (!ok && lane == 0) raise_flag(p.flags, PKV_DEVERR_TIMEOUT);
    if (lane == 0) release_claims(p.header);
    // Drain: never leave while a copy into this CTA's shared memory may be in flight.
    if (lane == 0) {
      const uint32_t n = issue < (uint32_t)T::kStages ? issue : (uint32_t)T::kStages;
      for (uint32_t i = issue - n; i < issue; ++i) {
        if (!mbar_wait(full0 + 8 * (i % T::kStages), (i / T::kStages) & 1)) {
          raise_flag(p.flags, PKV_DEVERR_TIMEOUT);
          break;
        }
      }
    }
    return;
  }

  // ================================= consumer warps =================================
  constexpr int VPL = T::kVPL;
  const int g = lane >> 3;  // lane group: tokens [g*TPG, (g+1)*TPG) of this warp's share
  const int j = lane & 7;   // dims [(j + 8c) * 8, +8) for chunk c
  // after the reduce-scatter this lane holds pairs idx = j*VPL + r: token idx/GH, head idx%GH
  auto my_h = [j](int r) { return (j * VPL + r) % GH; };
  auto my_t = [j](int r) { return (j * VPL + r) / GH; };
  const int tbase = warp * T::kTokPerWarp + g * T::kTPG;

  uint8_t* qfw = smem + T::kOffQf + warp * T::kQfBytesPerWarp;  // this warp's q copy
  uint64_t acc[GH][T::kPairs];
  float m_ref[GH];
  float l_lane[VPL];
#pragma unroll
  for (int r = 0; r < VPL; ++r) l_lane[r] = 0.f;
  uint32_t use = 0;
  uint32_t item = 0;

  while (true) {
    const int st = use % T::kStages;
    if (!mbar_wait(full0 + 8 * st, (use / T::kStages) & 1)) {
      if (lane == 0) raise_flag(p.flags, PKV_DEVERR_TIMEOUT);
      return;
    }
    const int mflags = meta[st].flags;
    if (mflags & kMetaDone) break;

    if (mflags & (kMetaFirst | kMetaZero)) {
#pragma unroll
      for (int h = 0; h < GH; ++h) {
        m_ref[h] = -INFINITY;
#pragma unroll
        for (int i = 0; i < T::kPairs; ++i) acc[h][i] = 0ull;
      }
#pragma unroll
      for (int r = 0; r < VPL; ++r) l_lane[r] = 0.f;
    }
    if (mflags & kMetaFirst) {
      // q of this item into this warp's copy, regrouped so that a lane reads the GH heads'
      // pairs of one (chunk, word) at once (lanes of group 0 write)
      if (lane < 8) {
        const uint8_t* qs = qbuf + st * T::kQBytes;
#pragma unroll
        for (int c = 0; c < T::kChunks; ++c) {
          uint32_t qv[GH][4];
#pragma unroll
          for (int h = 0; h < GH; ++h) {
            const uint4 w = *reinterpret_cast<const uint4*>(qs + (h * D + (j + 8 * c) * 8) * 2);
            qv[h][0] = w.x;
            qv[h][1] = w.y;
            qv[h][2] = w.z;
            qv[h][3] = w.w;
          }
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            uint8_t* base = qfw + (c * 4 + w) * (32 * GH) + j * (4 * GH);
            if constexpr (GH == 1) {
              *reinterpret_cast<uint32_t*>(base) = qv[0][w];
            } else if constexpr (GH == 2) {
              *reinterpret_cast<uint2*>(base) = make_uint2(qv[0][w], qv[1][w]);
            } else {
              *reinterpret_cast<uint4*>(base) = make_uint4(qv[0][w], qv[1][w], qv[2][w], qv[3][w]);
            }
          }
        }
      }
      __syncwarp();
    }

    if (!(mflags & kMetaZero)) {
      const uint8_t* kt = tiles + st * T::kStageBytes;
      const uint8_t* vt = kt + T::kTileBytes;
      const int n_valid = meta[st].tok_end - meta[st].tok0;  // tokens that count (may exceed)

      // ---- scores: partial q.k over this lane's dims for its TPG tokens x GH heads ----
      uint64_t s2[T::kTPG][GH];
#pragma unroll
      for (int tt = 0; tt < T::kTPG; ++tt)
#pragma unroll
        for (int h = 0; h < GH; ++h) s2[tt][h] = 0ull;
#pragma unroll
      for (int c = 0; c < T::kChunks; ++c) {
        uint4 kw[T::kTPG];
#pragma unroll
        for (int tt = 0; tt < T::kTPG; ++tt)
          kw[tt] = *reinterpret_cast<const uint4*>(kt + (tbase + tt) * T::kRowBytes +
                                                   (j + 8 * c) * 16);
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          uint64_t qv[GH];
          const uint8_t* base = qfw + (c * 4 + w) * (32 * GH) + j * (4 * GH);
          if constexpr (GH == 1) {
            qv[0] = bf16x2_to_f32x2(*reinterpret_cast<const uint32_t*>(base));
          } else if constexpr (GH == 2) {
            const uint2 v = *reinterpret_cast<const uint2*>(base);
            qv[0] = bf16x2_to_f32x2(v.x);
            qv[1] = bf16x2_to_f32x2(v.y);
          } else {
            const uint4 v = *reinterpret_cast<const uint4*>(base);
            qv[0] = bf16x2_to_f32x2(v.x);
            qv[1] = bf16x2_to_f32x2(v.y);
            qv[2] = bf16x2_to_f32x2(v.z);
            qv[3] = bf16x2_to_f32x2(v.w);
          }
#pragma unroll
          for (int tt = 0; tt < T::kTPG; ++tt) {
            const uint32_t word = w == 0 ? kw[tt].x : w == 1 ? kw[tt].y : w == 2 ? kw[tt].z
                                                                                   : kw[tt].w;
            const uint64_t kp = bf16x2_to_f32x2(word);
#pragma unroll
            for (int h = 0; h < GH; ++h) s2[tt][h] = ffma2(qv[h], kp, s2[tt][h]);
          }
        }
      }
      float part[T::kN];
#pragma unroll
      for (int tt = 0; tt < T::kTPG; ++tt)
#pragma unroll
        for (int h = 0; h < GH; ++h) {
          const float2 f = unpack2(s2[tt][h]);
          part[tt * GH + h] = f.x + f.y;
        }
      reduce_scatter<T::kN>(part, j);
      float sc[VPL], mx[VPL];
      bool valid[VPL];
#pragma unroll
      for (int r = 0; r < VPL; ++r) {
        valid[r] = (tbase + my_t(r)) < n_valid;
        sc[r] = valid[r] ? part[r] * p.qk_scale_log2 : -INFINITY;  // log2 units
        mx[r] = max_over_tokens<T::kN, GH>(sc[r]);
      }

      // ---- online softmax (log2 units), lazy rescale ----
      float mt_all[GH];  // head h sits in lane h / VPL of group 0, slot h % VPL
#pragma unroll
      for (int h = 0; h < GH; ++h) mt_all[h] = __shfl_sync(kFullMask, mx[h % VPL], h / VPL);
      bool need = false;
#pragma unroll
      for (int h = 0; h < GH; ++h) need |= mt_all[h] > m_ref[h] + kTau;
      if (need) {
#pragma unroll
        for (int h = 0; h < GH; ++h) {
          if (mt_all[h] > m_ref[h] + kTau) {
            const float alpha = fast_exp2(m_ref[h] - mt_all[h]);
            const uint64_t a2 = pack2(alpha, alpha);
#pragma unroll
            for (int i = 0; i < T::kPairs; ++i) acc[h][i] = fmul2(acc[h][i], a2);
#pragma unroll
            for (int r = 0; r < VPL; ++r)
              if (my_h(r) == h) l_lane[r] *= alpha;
            m_ref[h] = mt_all[h];
          }
        }
      }
      float pr[VPL];
#pragma unroll
      for (int r = 0; r < VPL; ++r) {
        float my_m = m_ref[0];
#pragma unroll
        for (int h = 1; h < GH; ++h)
          if (my_h(r) == h) my_m = m_ref[h];
        pr[r] = valid[r] ? fast_exp2(sc[r] - my_m) : 0.f;
        l_lane[r] += pr[r];
      }

      // ---- acc += p * V over this lane group's tokens ----
#pragma unroll
      for (int tt = 0; tt < T::kTPG; ++tt) {
        uint64_t pp[GH];
#pragma unroll
        for (int h = 0; h < GH; ++h) {
          const int idx = tt * GH + h;  // held by lane idx / VPL of this group, slot idx % VPL
          const float pv = __shfl_sync(kFullMask, pr[idx % VPL], (lane & ~7) | (idx / VPL));
          pp[h] = pack2(pv, pv);
        }
        // stale shared memory past the end of the context must not reach the products
        const uint32_t keep = (tbase + tt) < n_valid ? 0xffffffffu : 0u;
        const uint8_t* row = vt + (tbase + tt) * T::kRowBytes;
#pragma unroll
        for (int c = 0; c < T::kChunks; ++c) {
          const uint4 w = *reinterpret_cast<const uint4*>(row + (j + 8 * c) * 16);
          const uint64_t v0 = bf16x2_to_f32x2(w.x & keep), v1 = bf16x2_to_f32x2(w.y & keep);
          const uint64_t v2 = bf16x2_to_f32x2(w.z & keep), v3 = bf16x2_to_f32x2(w.w & keep);
#pragma unroll
          for (int h = 0; h < GH; ++h) {
            acc[h][4 * c + 0] = ffma2(pp[h], v0, acc[h][4 * c + 0]);
            acc[h][4 * c + 1] = ffma2(pp[h], v1, acc[h][4 * c + 1]);
            acc[h][4 * c + 2] = ffma2(pp[h], v2, acc[h][4 * c + 2]);
            acc[h][4 * c + 3] = ffma2(pp[h], v3, acc[h][4 * c + 3]);
          }
        }
      }
    }
    if (!(mflags & (kMetaLast | kMetaZero))) {
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * st);
      ++use;
      continue;
    }
    // Last tile of the item: take its identity from the stage before releasing the stage.
    StageMeta mt;
    mt.b = meta[st].b;
    mt.x = meta[st].x;
    mt.split = meta[st].split;
    mt.nsplit = meta[st].nsplit;
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * st);
    ++use;

    // ---- item finished: merge the lane groups, then the warps, then write ----
#pragma unroll
    for (int h = 0; h < GH; ++h)
#pragma unroll
      for (int i = 0; i < T::kPairs; ++i) {
        float2 v = unpack2(acc[h][i]);
        v.x += __shfl_xor_sync(kFullMask, v.x, 8);
        v.y += __shfl_xor_sync(kFullMask, v.y, 8);
        v.x += __shfl_xor_sync(kFullMask, v.x, 16);
        v.y += __shfl_xor_sync(kFullMask, v.y, 16);
        acc[h][i] = pack2(v.x, v.y);
      }
    float l_sum[VPL];
#pragma unroll
    for (int r = 0; r < VPL; ++r) l_sum[r] = sum_over_tokens<T::kN, GH>(l_lane[r]);
    float l_all[GH];
#pragma unroll
    for (int h = 0; h < GH; ++h) l_all[h] = __shfl_sync(kFullMask, l_sum[h % VPL], h / VPL);
    float* cbw = cb + warp * T::kCbFloats;
    // every warp has finished reading the previous item's partials before this slot is reused
    if (item > 0 && !mbar_wait(cmr, (item - 1) & 1)) {
      if (lane == 0) raise_flag(p.flags, PKV_DEVERR_TIMEOUT);
      return;
    }
    if (g == 0) {
#pragma unroll
      for (int h = 0; h < GH; ++h)
#pragma unroll
        for (int c = 0; c < T::kChunks; ++c) {
          float* dst = cbw + h * D + (j + 8 * c) * 8;
          const float2 a0 = unpack2(acc[h][4 * c + 0]), a1 = unpack2(acc[h][4 * c + 1]);
          const float2 a2 = unpack2(acc[h][4 * c + 2]), a3 = unpack2(acc[h][4 * c + 3]);
          reinterpret_cast<float4*>(dst)[0] = make_float4(a0.x, a0.y, a1.x, a1.y);
          reinterpret_cast<float4*>(dst)[1] = make_float4(a2.x, a2.y, a3.x, a3.y);
        }
    }
    if (lane == 0) {
#pragma unroll
      for (int h = 0; h < GH; ++h) {
        cbw[GH * D + h] = m_ref[h];
        cbw[GH * D + GH + h] = l_all[h];
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(cmb);
    if (!mbar_wait(cmb, item & 1)) {
      if (lane == 0) raise_flag(p.flags, PKV_DEVERR_TIMEOUT);
      return;
    }
    const float* cbp = cb;
    const bool final_out = mt.nsplit == 1;
    // Warp w writes outputs o = 64 w + 2 lane + 256 k: one (head, 64-dim slice) per k.
    for (int o = 64 * warp + 2 * lane; o < GH * D; o += T::kWarps * 64) {
      const int h = o / D, d = o % D;
      float mw[T::kWarps];
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < T::kWarps; ++w) {
        mw[w] = cbp[w * T::kCbFloats + GH * D + h];
        M = fmaxf(M, mw[w]);
      }
      float den = 0.f, n0 = 0.f, n1 = 0.f;
#pragma unroll
      for (int w = 0; w < T::kWarps; ++w) {
        const float wt = mw[w] == -INFINITY ? 0.f : fast_exp2(mw[w] - M);
        den += wt * cbp[w * T::kCbFloats + GH * D + GH + h];
        const float2 a = *reinterpret_cast<const float2*>(cbp + w * T::kCbFloats + h * D + d);
        n0 += wt * a.x;
        n1 += wt * a.y;
      }
      const int head = mt.x * GH + h;
      if (final_out) {
        const float inv = den > 0.f ? 1.f / den : 0.f;
        *reinterpret_cast<__nv_bfloat162*>(p.out + ((int64_t)mt.b * p.num_q_heads + head) * D +
                                           d) = __floats2bfloat162_rn(n0 * inv, n1 * inv);
      } else {
        const int64_t pi = ((int64_t)mt.b * p.max_splits + mt.split) * p.num_q_heads + head;
        *reinterpret_cast<float2*>(p.part_acc + pi * D + d) = make_float2(n0, n1);
        if (lane == 0) p.part_ml[pi * (D / 64) + d / 64] = make_float2(M, den);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(cmr);  // this warp no longer reads the partials
    if (!final_out) {
      // Chunk partials are out; the warp that finishes last for this (sequence, head group,
      // slice) merges all chunks: o = sum_s 2^(m_s - M) acc_s / sum_s 2^(m_s - M) l_s.
      __threadfence();
      __syncwarp();
      uint32_t* ctr = p.counters + ((int64_t)mt.b * p.head_groups + mt.x) * T::kWarps + warp;
      uint32_t done = 0;
      if (lane == 0) done = atomicAdd(ctr, 1u);
      done = __shfl_sync(kFullMask, done, 0);
      if (done == (uint32_t)mt.nsplit - 1) {
        __threadfence();
        merge_chunks<D, GH, T::kWarps>(p, mt.b, mt.x, mt.nsplit, warp, lane);
        if (lane == 0) *ctr = 0u;  // all chunks counted: ready for the next call
      }
    }
    ++item;
  }
}

template <int D, int GH>
cudaError_t configure_instance(int* ctas_per_sm) {
  using T = Traits<D, GH>;
  cudaError_t e = cudaFuncSetAttribute(paged_decode_kernel<D, GH>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, T::kSmemBytes);
  if (e != cudaSuccess) return e;
  // the largest shared-memory carve-out, so that two CTAs fit on an SM
  e = cudaFuncSetAttribute(paged_decode_kernel<D, GH>,
                           cudaFuncAttributePreferredSharedMemoryCarveout,
                           (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  int n = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, paged_decode_kernel<D, GH>,
                                                    T::kThreads, T::kSmemBytes);
  if (e != cudaSuccess) return e;
  *ctas_per_sm = n < 1 ? 1 : n;
  return cudaSuccess;
}

// Index of an instance in ContextState::decode_ctas.
constexpr int decode_instance(int D, int GH) { return (D == 128 ? 0 : 3) + (GH == 4 ? 0 : GH == 2 ? 1 : 2); }

template <int D, int GH>
cudaError_t launch_instance(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                            int num_sms, cudaStream_t stream) {
  using T = Traits<D, GH>;
  const int ctas_per_sm = a.ctas_per_sm[decode_instance(D, GH)];
  if (ctas_per_sm <= 0) return cudaErrorInvalidConfiguration;
  const int G = a.num_q_heads / a.cache.num_kv_heads;
  DecodeParams p;
  p.q = a.q;
  p.block_tables = a.block_tables;
  p.context_lens = a.context_lens;
  p.out = a.out;
  p.part_acc = a.ws.part_acc;
  p.part_ml = a.ws.part_ml;
  p.items = a.ws.items;
  p.header = a.ws.header;
  p.counters = a.ws.counters;
  p.flags = a.flags;
  p.max_blocks = a.max_blocks;
  p.num_seqs = a.num_seqs;
  p.num_q_heads = a.num_q_heads;
  p.head_groups = a.num_q_heads / GH;
  p.groups_per_kv = G / GH;
  p.block_size = a.cache.block_size;
  p.num_blocks = a.cache.num_blocks;
  p.max_splits = a.max_splits;
  const int64_t cap_table = (int64_t)a.max_blocks * a.cache.block_size;
  const int64_t cap_plan = (int64_t)a.max_splits * a.split_tokens;
  int64_t cap = cap_table < cap_plan ? cap_table : cap_plan;
  if (cap > 0x7fffffff) cap = 0x7fffffff;
  p.cap_tokens = (int32_t)cap;
  p.qk_scale_log2 = a.scale * 1.4426950408889634f;

  const int64_t upper = (int64_t)a.num_seqs * a.max_splits * p.head_groups;
  int64_t grid = (int64_t)num_sms * ctas_per_sm;
  if (grid > upper) grid = upper;
  if (grid < 1) grid = 1;

  cudaError_t e =
      a.reuse_plan ? (a.k_new != nullptr ? launch_decode_store_rows(a, num_sms, stream)
                                         : cudaSuccess)
                   : launch_decode_plan(a, p.head_groups, (int32_t)((int64_t)num_sms * ctas_per_sm),
                                        a.max_splits > 1 ? p.head_groups * T::kWarps : 0,
                                        p.cap_tokens, num_sms, stream);
  if (e != cudaSuccess) return e;
  // The decode grid is a programmatic dependent of the plan: it is scheduled while the plan runs
  // and waits for it in-kernel, which hides the launch gap between the two.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(T::kThreads);
  cfg.dynamicSmemBytes = T::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, paged_decode_kernel<D, GH>, tk, tv, p);
}

}  // namespace

cudaError_t launch_decode_plan(const DecodeArgs& a, int32_t head_groups, int32_t slots,
                               int32_t counters_per_seq, int32_t cap_tokens, int num_sms,
                               cudaStream_t stream) {
  PlanParams pp;
  pp.context_lens = a.context_lens;
  pp.items = a.ws.items;
  pp.header = a.ws.header;
  pp.counters = a.ws.counters;
  pp.flags = a.flags;
  pp.num_seqs = a.num_seqs;
  pp.cap_tokens = cap_tokens;
  pp.split_floor = a.split_tokens;
  pp.fixed_split = a.auto_split ? 0 : a.split_tokens;
  pp.head_groups = head_groups;
  pp.slots = slots;
  pp.counters_per_seq = counters_per_seq;
  pp.k_new = a.k_new;
  pp.v_new = a.v_new;
  pp.slot_mapping = a.slot_mapping;
  pp.k_cache = const_cast<uint16_t*>(a.k_cache);
  pp.v_cache = const_cast<uint16_t*>(a.v_cache);
  pp.block_tables = a.block_tables;
  pp.max_blocks = a.max_blocks;
  pp.block_size = a.cache.block_size;
  pp.num_blocks = a.cache.num_blocks;
  pp.row_chunks = a.cache.num_kv_heads * a.cache.head_dim / 8;
  pp.do_plan = 1;
  // One CTA plans; with a store (pkv_paged_decode_store) more CTAs copy the new rows, about four
  // 16-byte chunks of K and of V per thread.
  int store_ctas = 0;
  if (a.k_new != nullptr) {
    const int64_t chunks = (int64_t)a.num_seqs * pp.row_chunks;
    const int64_t want = (chunks + 4 * kPlanThreads - 1) / (4 * kPlanThreads);
    store_ctas = (int)(want < num_sms ? want : num_sms);
    if (store_ctas < 1) store_ctas = 1;
  }
  return launch_dependent(decode_plan_kernel, dim3(1 + store_ctas), dim3(kPlanThreads), 0, stream,
                          pp);
}

size_t decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                              int32_t max_splits, DecodeWorkspace* carve, void* base) {
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t n_items = (size_t)num_seqs * max_splits;
  size_t off = 0;
  const size_t header = off;
  off += 256;
  const size_t items = off;
  off += up(n_items * sizeof(int2));
  size_t counters = 0, acc = 0, ml = 0;
  if (max_splits > 1) {
    // one counter per (sequence, query head, consumer warp) bounds every head grouping
    counters = off;
    off += up((size_t)num_seqs * num_q_heads * 4 * sizeof(uint32_t));
    acc = off;
    off += up(n_items * num_q_heads * head_dim * sizeof(float));
    ml = off;
    off += up(n_items * num_q_heads * (head_dim / 64) * sizeof(float2));
  }
  if (carve != nullptr) {
    uint8_t* b8 = static_cast<uint8_t*>(base);
    carve->header = reinterpret_cast<uint32_t*>(b8 + header);
    carve->items = reinterpret_cast<int2*>(b8 + items);
    carve->counters = max_splits > 1 ? reinterpret_cast<uint32_t*>(b8 + counters) : nullptr;
    carve->part_acc = max_splits > 1 ? reinterpret_cast<float*>(b8 + acc) : nullptr;
    carve->part_ml = max_splits > 1 ? reinterpret_cast<float2*>(b8 + ml) : nullptr;
  }
  return off;
}

cudaError_t configure_decode_kernels(int (&ctas)[kDecodeInstances]) {
  cudaError_t e = cudaSuccess;
#define PKV_CONFIGURE(D, GH) \
  if (e == cudaSuccess) e = configure_instance<D, GH>(&ctas[decode_instance(D, GH)]);
  PKV_CONFIGURE(128, 4)
  PKV_CONFIGURE(128, 2)
  PKV_CONFIGURE(128, 1)
  PKV_CONFIGURE(64, 4)
  PKV_CONFIGURE(64, 2)
  PKV_CONFIGURE(64, 1)
#undef PKV_CONFIGURE
  return e;
}

cudaError_t launch_decode_store_rows(const DecodeArgs& a, int num_sms, cudaStream_t stream) {
  PlanParams pp = {};
  pp.context_lens = a.context_lens;
  pp.flags = a.flags;
  pp.num_seqs = a.num_seqs;
  const int64_t cap = (int64_t)a.max_blocks * a.cache.block_size;
  pp.cap_tokens = (int32_t)(cap > 0x7fffffff ? 0x7fffffff : cap);
  pp.k_new = a.k_new;
  pp.v_new = a.v_new;
  pp.slot_mapping = a.slot_mapping;
  pp.k_cache = const_cast<uint16_t*>(a.k_cache);
  pp.v_cache = const_cast<uint16_t*>(a.v_cache);
  pp.block_tables = a.block_tables;
  pp.max_blocks = a.max_blocks;
  pp.block_size = a.cache.block_size;
  pp.num_blocks = a.cache.num_blocks;
  pp.row_chunks = a.cache.num_kv_heads * a.cache.head_dim / 8;
  pp.do_plan = 0;
  const int64_t chunks = (int64_t)a.num_seqs * pp.row_chunks;
  int64_t ctas = (chunks + 4 * kPlanThreads - 1) / (4 * kPlanThreads);
  if (ctas > num_sms) ctas = num_sms;
  if (ctas < 1) ctas = 1;
  return launch_dependent(decode_plan_kernel, dim3((unsigned)(1 + ctas)), dim3(kPlanThreads), 0,
                          stream, pp);
}

int decode_box_rows(int head_dim, int group, int block_size) {
  const int GH = group >= 4 ? 4 : group;
  int tile = 0;
  if (head_dim == 128) {
    tile = GH == 4 ? Traits<128, 4>::kTileT : GH == 2 ? Traits<128, 2>::kTileT
                                                     : Traits<128, 1>::kTileT;
  } else {
    tile = GH == 4 ? Traits<64, 4>::kTileT : GH == 2 ? Traits<64, 2>::kTileT
                                                    : Traits<64, 1>::kTileT;
  }
  return block_size < tile ? block_size : tile;
}

cudaError_t launch_paged_decode(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                                int num_sms, cudaStream_t stream) {
  const int G = a.num_q_heads / a.cache.num_kv_heads;
  const int GH = G >= 4 ? 4 : G;
  if (a.cache.head_dim == 128) {
    if (GH == 4) return launch_instance<128, 4>(a, tk, tv, num_sms, stream);
    if (GH == 2) return launch_instance<128, 2>(a, tk, tv, num_sms, stream);
    if (GH == 1) return launch_instance<128, 1>(a, tk, tv, num_sms, stream);
  } else if (a.cache.head_dim == 64) {
    if (GH == 4) return launch_instance<64, 4>(a, tk, tv, num_sms, stream);
    if (GH == 2) return launch_instance<64, 2>(a, tk, tv, num_sms, stream);
    if (GH == 1) return launch_instance<64, 1>(a, tk, tv, num_sms, stream);
  }
  return cudaErrorNotSupported;
}

}  // namespace pkv
