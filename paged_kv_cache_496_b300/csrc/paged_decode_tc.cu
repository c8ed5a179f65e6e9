// paged_decode_tc.cu -- paged decode attention on tcgen05 tensor cores with the keys on the MMA's
// M dimension (sm_103a).
//
// Source: "DeepSeek研究员1200行代码复刻vLLM，H800硬件实测性能反超原版" (QbitAI), section
// "vLLM是什么？": keys and values of a sequence sit in fixed-size blocks found through its block
// table, and the attention kernel fetches the blocks one by one. The result is ordinary softmax
// attention over the sequence's tokens; only the addressing is paged.
//
// Design (B300-first):
//  * A decode step has one query row per sequence. With the queries on the MMA's M dimension a
//    128-row tile would carry G useful rows of 128. Here the roles are swapped: for each tile of
//    128 keys of one (sequence, kv head), S^T = K Q^T (M = 128 keys, N = 16 columns holding the G
//    query heads of that kv head, K = 128 dims) and O^T += V^T P^T (M = 128 dims, N = 16,
//    K = 128 keys, V read MN-major). Every MMA row carries data, and the tensor work per byte of
//    K/V is small: the kernel is bound by HBM, not by the tensor pipe or its power.
//  * Work item = (sequence, kv head, context chunk) from the same device-side plan as the CUDA-core
//    decode kernel: chunk length from the actual lengths, items longest first. The warp of each
//    output-dim quarter that finishes a split sequence's last chunk merges the chunk partials.
//  * One CTA per SM, 192 threads. Warp 0 claims items, walks the block table and fills a
//    three-stage ring (68 KB a stage): K and V of 128 keys as 3-D TMA boxes in 128-byte swizzle
//    (two 64-dim halves each) and the G rows of q in each half (rows G..15 stay zero). Warp 1
//    allocates 64 TMEM columns (two S^T slots and two O^T slots of 16 columns) and issues the MMAs
//    from one thread. Warps 2-5 own one TMEM lane quarter each: thread = key for the scores,
//    thread = output dim for O^T.
//  * Online softmax in log2 units with a lazy rescale. Per tile each warp reduces its keys'
//    scores to a maximum per head; the four warps swap them through shared memory under an
//    mbarrier, so every thread holds the same tile maximum. The running maximum moves, and O^T in
//    TMEM is rescaled, only when a head's tile maximum passes it by more than 2^8. Each thread
//    keeps partial denominators for its keys, summed once per item. P^T goes to shared memory as
//    bf16 in the K-major swizzled layout the MMA reads.
//  * Every wait is bounded (one second) and warp-uniform; the CTA always frees its TMEM.
#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace pkv {

namespace {

constexpr int kTK = 128;  // keys per tile: M of S^T = K Q^T, K of O^T += V^T P^T
constexpr int kDT = 128;  // head_dim: M of O^T
constexpr int kNT = 16;   // MMA N: the G query heads of a kv head, padded with zero rows
constexpr int kStagesT = 3;
constexpr int kThreadsT = 192;
constexpr int kTmemColsT = 64;
constexpr int kColST = 0;   // S^T slots: columns [0, 16) and [16, 32)
constexpr int kColOT = 32;  // O^T slots: columns [32, 48) and [48, 64)
constexpr float kTauT = 8.0f;

constexpr int kKVHalf = kTK * 128;                  // 64 dims of 128 keys: 16 KB
constexpr int kKVTile = 2 * kKVHalf;                // 32 KB
constexpr int kQHalfT = kNT * 128;                  // 64 dims of 16 head rows: 2 KB
constexpr int kOffKS = 0;                           // offsets inside a stage
constexpr int kOffVS = kKVTile;
constexpr int kOffQS = 2 * kKVTile;
constexpr int kStageT = 2 * kKVTile + 2 * kQHalfT;  // 68 KB
constexpr int kOffPT = kStagesT * kStageT;          // P^T: two halves of 16 rows x 64 keys
constexpr int kOffRedT = kOffPT + 2 * kQHalfT;      // two slots of [4 warps][8 heads] floats
constexpr int kOffMetaT = kOffRedT + 2 * 4 * 8 * 4;

struct alignas(16) TileMeta {
  int32_t b, x, split, nsplit;
  int32_t tok0, tok_end, flags, pad;
};
constexpr int kTFirst = 1;  // first tile of an item: new running state, new O^T slot
constexpr int kTLast = 2;   // last tile of an item: normalise or write partials
constexpr int kTDone = 4;   // no more items

// barriers: full[], empty[] (ring), s_full[2], s_free[2], p_full, o_done, o_free[2], vote,
// mma_done
constexpr int kBFull = 0, kBEmpty = kBFull + kStagesT, kBSFull = kBEmpty + kStagesT,
              kBSFree = kBSFull + 2, kBPFull = kBSFree + 2, kBODone = kBPFull + 1,
              kBOFree = kBODone + 1, kBVote = kBOFree + 2, kBMmaT = kBVote + 1,
              kNumBarsT = kBMmaT + 1;
constexpr int kOffBarT = kOffMetaT + kStagesT * (int)sizeof(TileMeta);
constexpr int kOffTmemT = kOffBarT + kNumBarsT * 8;
constexpr int kSmemT = kOffTmemT + 16;
static_assert(kStageT % 1024 == 0 && kOffQS % 1024 == 0 && kOffPT % 1024 == 0,
              "swizzle atoms need 1024-byte alignment");
static_assert(kOffMetaT % 16 == 0 && kOffBarT % 8 == 0, "shared memory alignment");
static_assert(kSmemT <= 227 * 1024, "shared memory per CTA");

struct TcDecodeParams {
  const int32_t* block_tables;
  const int32_t* context_lens;
  uint16_t* out;
  float* part_acc;
  float2* part_ml;
  const int2* items;
  uint32_t* header;    // [0] claim counter, [1] item count, [2] chunk length in tokens
  uint32_t* counters;  // per (sequence, kv head, output-dim quarter): chunks finished
  int* flags;
  int32_t max_blocks;
  int32_t num_seqs;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t block_size;
  int32_t num_blocks;
  int32_t max_splits;
  int32_t cap_tokens;  // contexts are clamped to this many tokens (table and plan capacity)
  int32_t box_rows;    // rows of a K/V TMA box: min(block_size, 128)
  float qk_scale_log2;
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFullMask, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFullMask, v, o);
  return v;
}

// A bounded mbarrier wait whose result is the same on every lane of the warp.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity) {
  return __all_sync(kFullMask, mbar_wait(bar, parity)) != 0;
}

template <int G>
__global__ void __launch_bounds__(kThreadsT, 1)
    paged_decode_tc_kernel(const __grid_constant__ CUtensorMap tmap_q,
                           const __grid_constant__ CUtensorMap tmap_k,
                           const __grid_constant__ CUtensorMap tmap_v,
                           const __grid_constant__ CUtensorMap tmap_k64,
                           const __grid_constant__ CUtensorMap tmap_v64,
                           const __grid_constant__ CUtensorMap tmap_k32,
                           const __grid_constant__ CUtensorMap tmap_v32,
                           const __grid_constant__ TcDecodeParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if ((smem_addr(smem) & 1023u) != 0) {  // the swizzled layouts need a 1024-byte aligned base
    if (threadIdx.x == 0) raise_flag(p.flags, PKV_DEVERR_INTERNAL);
    return;
  }
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bar0 = sbase + kOffBarT;
  auto bar = [bar0](int i) { return bar0 + 8u * (uint32_t)i; };
  TileMeta* meta = reinterpret_cast<TileMeta*>(smem + kOffMetaT);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + kOffTmemT);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesT; ++s) {
      mbar_init(bar(kBFull + s), 1);
      mbar_init(bar(kBEmpty + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kBSFull + i), 1);
      mbar_init(bar(kBSFree + i), 4);
      mbar_init(bar(kBOFree + i), 4);
    }
    mbar_init(bar(kBPFull), 4);
    mbar_init(bar(kBODone), 1);
    mbar_init(bar(kBVote), 4);
    mbar_init(bar(kBMmaT), 1);
    fence_barrier_init();
  }
  // The q slots' rows G..15 and P^T's rows G..15 hold zeros that nothing overwrites: the q boxes
  // fill rows 0..G-1 only, and the softmax writes rows 0..G-1 only.
  {
    constexpr int kChunks = 2 * kQHalfT / 16;
    for (int i = threadIdx.x; i < (kStagesT + 1) * kChunks; i += kThreadsT) {
      const int st = i / kChunks, c = i % kChunks;
      uint8_t* base = st < kStagesT ? smem + st * kStageT + kOffQS : smem + kOffPT;
      *reinterpret_cast<uint4*>(base + c * 16) = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_async_shared();
  }
  if (warp == 1) {
    tmem_alloc(sbase + kOffTmemT, kTmemColsT);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  // Launched as a programmatic dependent of the plan grid: everything above overlaps it; nothing
  // below reads memory before the plan (and all earlier work) has completed. The next work in
  // the stream may then be scheduled; it waits for this grid before touching memory.
  grid_dependency_wait();
  allow_dependent_launch();
  const int nkv = p.num_kv_heads;

  if (warp == 0) {
    // =============================== producer warp ===============================
    if (lane == 0) {
      tma_prefetch_desc(&tmap_q);
      tma_prefetch_desc(&tmap_k);
      tma_prefetch_desc(&tmap_v);
      tma_prefetch_desc(&tmap_k64);
      tma_prefetch_desc(&tmap_v64);
      tma_prefetch_desc(&tmap_k32);
      tma_prefetch_desc(&tmap_v32);
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
    const uint32_t total = n_items * (uint32_t)nkv;
    auto in_batch = [&](int2 r) {
      return (unsigned)r.x < (unsigned)p.num_seqs && (unsigned)r.y < (unsigned)p.max_splits;
    };
    const int bs = p.block_size;
    const int lbs = __ffs(bs) - 1;  // block_size is a power of two
    // Full tiles use boxes of min(block_size, 128) rows. A chunk's partial last tile of n rows
    // uses 32-row boxes when n <= 32 and 64-row boxes when n <= 64 (if those are smaller), so it
    // fetches fewer rows past its end without issuing more boxes: every box carries a fixed cost
    // in the TMA unit, and many small boxes cost more than the rows they save.
    const int box_full = p.box_rows;
    const int ent_per_tile = (kTK + bs - 1) >> lbs;
    uint32_t issue = 0;
    bool ok = true;
    auto claim = [&]() -> uint32_t {
      uint32_t c = 0;
      if (lane == 0) c = atomicAdd(p.header, 1u);
      return __shfl_sync(kFullMask, c, 0);
    };
    // Each stage has its own issuing lane (lane == stage): one thread's bulk copies complete one
    // barrier phase at a time, so a thread with several stages in flight would queue them.
    auto acquire = [&](int stage) -> bool {
      int good = 1;
      if (lane == stage)
        good = mbar_wait(bar(kBEmpty + stage), ((issue / kStagesT) & 1) ^ 1) ? 1 : 0;
      return __shfl_sync(kFullMask, good, stage) != 0;
    };

    // Claims run one item ahead, and the next item's record, length and first two table windows
    // are loaded while the current item's first tile goes out: no chain of dependent global loads
    // sits between the last tile of one item and the first tile of the next.
    auto window = [&](int b, int e) -> int {
      return e < p.max_blocks ? __ldg(p.block_tables + (int64_t)b * p.max_blocks + e) : -1;
    };
    uint32_t c = claim();
    int2 it = make_int2(0, 0);
    int ctx_raw = 0, w_lo = -1, w_hi = -1;
    if (c < total) {
      it = p.items[c / (uint32_t)nkv];
      if (in_batch(it)) {
        ctx_raw = p.context_lens[it.x];
        const int e0 = (it.y * split) >> lbs;
        w_lo = window(it.x, e0 + lane);
        w_hi = window(it.x, e0 + 32 + lane);
      }
    }
    uint32_t c_ahead = lane == 0 ? atomicAdd(p.header, 1u) : 0u;  // read one item later
    while (ok) {
      if (c >= total) {
        const int st = issue % kStagesT;
        ok = acquire(st);
        if (ok && lane == st) {
          meta[st].flags = kTDone;
          mbar_arrive(bar(kBFull + st));
        }
        ++issue;
        break;
      }
      const int b = it.x, s = it.y;
      const int x = (int)(c % (uint32_t)nkv);
      const bool valid = in_batch(it);
      if (!valid && lane == 0) raise_flag(p.flags, PKV_DEVERR_INTERNAL);
      const int ctx = !valid ? -1 : ctx_raw < p.cap_tokens ? ctx_raw : p.cap_tokens;
      // the next item: its id was claimed during the previous item; its record is loaded now
      const uint32_t c_nx = __shfl_sync(kFullMask, c_ahead, 0);
      const int2 it_nx = c_nx < total ? p.items[c_nx / (uint32_t)nkv] : make_int2(0, 0);
      c_ahead = lane == 0 ? atomicAdd(p.header, 1u) : 0u;
      int ctx_nx = 0, w_lo_nx = -1, w_hi_nx = -1;
      bool nx_loaded = false;
      auto load_next = [&]() {
        if (nx_loaded) return;
        nx_loaded = true;
        if (c_nx < total && in_batch(it_nx)) {
          ctx_nx = p.context_lens[it_nx.x];
          const int e0 = (it_nx.y * split) >> lbs;
          w_lo_nx = window(it_nx.x, e0 + lane);
          w_hi_nx = window(it_nx.x, e0 + 32 + lane);
        }
      };
      if (!valid) {
        // outside this call's batch: nothing to read or write
      } else if (ctx <= 0) {
        // no keys: the item's G output rows are zeros, written here without using a stage
        uint4* o = reinterpret_cast<uint4*>(p.out + ((int64_t)b * p.num_q_heads + x * G) * kDT);
        for (int i = lane; i < G * kDT / 8; i += 32) o[i] = make_uint4(0u, 0u, 0u, 0u);
      } else {
        const int nsplit = (ctx + split - 1) / split;
        const int tok_begin = s * split;
        const int tok_end = min(ctx, tok_begin + split);
        // Block-table window: entries [win_base, win_base + 32) of this sequence, one per lane,
        // and the next 32 entries prefetched (entries past the sequence's end are never used).
        int win_base = tok_begin >> lbs, win_val = w_lo, nxt_val = w_hi;
        for (int tok0 = tok_begin; tok0 < tok_end && ok; tok0 += kTK) {
          const int st = issue % kStagesT;
          const int e0 = tok0 >> lbs;
          if (e0 + ent_per_tile > win_base + 32) {
            win_base += 32;  // step into the prefetched window, and fetch the one after it
            win_val = nxt_val;
            nxt_val = window(b, win_base + 32 + lane);
          }
          const int n_left = tok_end - tok0;
          const bool t32 = n_left <= 32 && box_full > 32;
          const bool t64 = !t32 && n_left <= 64 && box_full > 64;
          const int box = t32 ? 32 : t64 ? 64 : box_full;
          const int nsub = kTK / box;
          const CUtensorMap* mk = t32 ? &tmap_k32 : t64 ? &tmap_k64 : &tmap_k;
          const CUtensorMap* mv = t32 ? &tmap_v32 : t64 ? &tmap_v64 : &tmap_v;
          int rows[kTK / 16];
          uint32_t bytes = 2u * G * 128u;  // q: G rows of each 64-dim half
#pragma unroll
          for (int sb = 0; sb < kTK / 16; ++sb) {
            rows[sb] = -1;
            if (sb < nsub) {
              const int t = tok0 + sb * box;
              const int blk = __shfl_sync(kFullMask, win_val, ((t >> lbs) - win_base) & 31);
              if (t < tok_end) {
                if (blk >= 0 && blk < p.num_blocks) {
                  rows[sb] = blk * bs + (t & (bs - 1));
                  bytes += 4u * (uint32_t)box * 128u;  // K and V, two halves each
                } else if (lane == 0) {
                  raise_flag(p.flags, PKV_DEVERR_BAD_BLOCK);
                }
              }
            }
          }
          ok = acquire(st);
          if (ok && lane == st) {
            TileMeta m;
            m.b = b; m.x = x; m.split = s; m.nsplit = nsplit;
            m.tok0 = tok0; m.tok_end = tok_end;
            m.flags = (tok0 == tok_begin ? kTFirst : 0) | (tok0 + kTK >= tok_end ? kTLast : 0);
            m.pad = 0;
            meta[st] = m;
            const uint32_t fb = bar(kBFull + st);
            mbar_arrive_expect_tx(fb, bytes);
            const uint32_t kdst = sbase + st * kStageT + kOffKS;
            const uint32_t vdst = sbase + st * kStageT + kOffVS;
            const uint32_t qdst = sbase + st * kStageT + kOffQS;
#pragma unroll
            for (int sb = 0; sb < kTK / 16; ++sb) {
              if (sb < nsub && rows[sb] >= 0) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  const uint32_t off = h * kKVHalf + sb * box * 128;
                  tma_load_3d(kdst + off, mk, 64 * h, x, rows[sb], fb);
                  tma_load_3d(vdst + off, mv, 64 * h, x, rows[sb], fb);
                }
              }
            }
            tma_load_3d(qdst, &tmap_q, 0, x * G, b, fb);
            tma_load_3d(qdst + kQHalfT, &tmap_q, 64, x * G, b, fb);
          }
          ++issue;
          load_next();  // after the item's first tile: its record has arrived by now
        }
      }
      load_next();
      c = c_nx;
      it = it_nx;
      ctx_raw = ctx_nx;
      w_lo = w_lo_nx;
      w_hi = w_hi_nx;
    }
    if (!ok && lane == 0) raise_flag(p.flags, PKV_DEVERR_TIMEOUT);
    if (lane == 0) release_claims(p.header);  // after the claim issued one item ahead
    // Drain: never leave while a copy into this CTA's shared memory may be in flight.
    if (lane == 0) {
      const uint32_t n = issue < (uint32_t)kStagesT ? issue : (uint32_t)kStagesT;
      for (uint32_t i = issue - n; i < issue; ++i) {
        if (!mbar_wait(bar(kBFull + i % kStagesT), (i / kStagesT) & 1)) {
          raise_flag(p.flags, PKV_DEVERR_TIMEOUT);
          break;
        }
      }
    }
  } else if (warp == 1) {
    // ============================ MMA issuer (one thread) ============================
    // Global tile t: S^T(t) = K Q^T into S slot t & 1, then O^T += V^T P^T for the previous tile,
    // so the tensor core computes the next scores while the softmax warps work. An item's last
    // P V goes out right after its S, so the item's output is not held up by the next item's
    // loads. O^T of item n accumulates in slot n & 1.
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32_t(kTK, kNT, false, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32_t(kDT, kNT, true, false);
      const uint64_t pdesc0 = sdesc_kmajor_sw128(sbase + kOffPT);
      bool ok = true;
      auto issue_pv = [&](int tv, int stv, bool first, int nv) {
        if (!ok) return;
        ok = mbar_wait(bar(kBPFull), tv & 1);
        // the first tile of item nv reuses the O^T slot of item nv - 2, once it has been read
        if (ok && first && nv >= 2) ok = mbar_wait(bar(kBOFree + (nv & 1)), ((nv >> 1) - 1) & 1);
        if (!ok) return;
        tc_fence_after_sync();
        // descriptors advance by address / 16 in their low 14 bits (shared addresses < 256 KB)
        const uint64_t vdesc0 = sdesc_mnmajor_sw128(sbase + stv * kStageT + kOffVS, kKVHalf);
        const uint32_t dcol = tmem + kColOT + (nv & 1) * kNT;
#pragma unroll
        for (int kk = 0; kk < kTK / 16; ++kk) {
          const uint64_t ad = vdesc0 + (uint64_t)(kk * 16 * 128 / 16);
          const uint64_t bd = pdesc0 + (uint64_t)(((kk >> 2) * kQHalfT + (kk & 3) * 32) / 16);
          tc_mma_f16(dcol, ad, bd, idesc_o, (!first || kk > 0) ? 1u : 0u);
        }
        tc_commit(bar(kBODone));
        tc_commit(bar(kBEmpty + stv));
      };
      uint32_t use = 0;
      int t = 0, n = -1;
      bool pend = false, pend_first = false;
      int pend_t = 0, pend_st = 0, pend_n = 0;
      while (ok) {
        const int st = use % kStagesT;
        ok = mbar_wait(bar(kBFull + st), (use / kStagesT) & 1);
        if (!ok) break;
        const int fl = meta[st].flags;
        if (fl & kTDone) break;
        if (fl & kTFirst) ++n;
        // S slot t & 1 was last read by the softmax of tile t - 2
        if (t >= 2) ok = mbar_wait(bar(kBSFree + (t & 1)), ((t >> 1) - 1) & 1);
        if (!ok) break;
        tc_fence_after_sync();
        const uint32_t kb = sbase + st * kStageT + kOffKS;
        const uint32_t qb = sbase + st * kStageT + kOffQS;
#pragma unroll
        for (int kk = 0; kk < kDT / 16; ++kk) {
          const uint32_t ok_ = (kk >> 2) * kKVHalf + (kk & 3) * 32;
          const uint32_t oq = (kk >> 2) * kQHalfT + (kk & 3) * 32;
          tc_mma_f16(tmem + kColST + (t & 1) * kNT, sdesc_kmajor_sw128(kb + ok_),
                     sdesc_kmajor_sw128(qb + oq), idesc_s, kk > 0 ? 1u : 0u);
        }
        tc_commit(bar(kBSFull + (t & 1)));
        if (pend) {
          issue_pv(pend_t, pend_st, pend_first, pend_n);
          pend = false;
        }
        if (fl & kTLast) {
          issue_pv(t, st, (fl & kTFirst) != 0, n);
        } else {
          pend = true;
          pend_t = t;
          pend_st = st;
          pend_first = (fl & kTFirst) != 0;
          pend_n = n;
        }
        ++t;
        ++use;
      }
      if (pend) issue_pv(pend_t, pend_st, pend_first, pend_n);
      if (!ok) raise_flag(p.flags, PKV_DEVERR_TIMEOUT);
      // all MMAs of this CTA are complete before TMEM is released
      tc_commit(bar(kBMmaT));
      if (!mbar_wait(bar(kBMmaT), 0)) raise_flag(p.flags, PKV_DEVERR_TIMEOUT);
    }
    __syncwarp();
  } else {
    // ================= softmax warps: thread = key (scores), thread = dim (output) =================
    const int quarter = warp & 3;  // the TMEM lane quarter this warp may access
    const int row = quarter * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
    float* red = reinterpret_cast<float*>(smem + kOffRedT);
    bool ok = true;
    uint32_t use = 0, vr = 0;
    int t = 0, n = -1;
    float m_run[G], l_part[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      m_run[h] = -INFINITY;
      l_part[h] = 0.f;
    }
    // The four warps swap one value per head: lane 0 writes this warp's, and after the exchange
    // the returned slot holds [warp quarter][head] for all four. Slots alternate, so a fast warp
    // never overwrites values a slow one is still reading.
    auto exchange = [&](const float (&v)[G], const float*& slot) -> bool {
      float* sl = red + (vr & 1) * 32;
      if (lane == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) sl[quarter * 8 + h] = v[h];
        mbar_arrive(bar(kBVote));
      }
      const bool good = warp_wait(bar(kBVote), vr & 1);
      ++vr;
      slot = sl;
      return good;
    };

    while (true) {
      const int st = use % kStagesT;
      ok = warp_wait(bar(kBFull + st), (use / kStagesT) & 1);
      if (!ok) break;
      const TileMeta m = meta[st];
      if (m.flags & kTDone) break;
      if (m.flags & kTFirst) {
        ++n;
#pragma unroll
        for (int h = 0; h < G; ++h) {
          m_run[h] = -INFINITY;
          l_part[h] = 0.f;
        }
      }
      ok = warp_wait(bar(kBSFull + (t & 1)), (t >> 1) & 1);
      if (!ok) break;
      tc_fence_after_sync();
      uint32_t sr[G];
      tmem_ld_cols<G>(tl + kColST + (t & 1) * kNT, sr);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBSFree + (t & 1)));

      // keys tok0 + row with row < nvalid count (the chunk's last tile may be partial)
      const bool kvalid = row < m.tok_end - m.tok0;
      float s[G], wm[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        s[h] = kvalid ? __uint_as_float(sr[h]) * p.qk_scale_log2 : -INFINITY;
        wm[h] = warp_max(s[h]);
      }
      const float* slot = nullptr;
      ok = exchange(wm, slot);
      if (!ok) break;
      float alpha[G];
      bool resc = false;  // the same on every thread: all read the same tile maxima
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float mt = fmaxf(fmaxf(slot[h], slot[8 + h]), fmaxf(slot[16 + h], slot[24 + h]));
        alpha[h] = 1.f;
        if (mt > m_run[h] + kTauT) {
          alpha[h] = fast_exp2(m_run[h] - mt);  // 0 when nothing was seen yet
          m_run[h] = mt;
          resc = true;
        }
      }
      float pr[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        pr[h] = kvalid ? fast_exp2(s[h] - m_run[h]) : 0.f;
        l_part[h] = l_part[h] * alpha[h] + pr[h];
      }
      // P^T(t) replaces P^T(t - 1) once P V(t - 1) has finished; O^T is stable then too
      if (t > 0) {
        ok = warp_wait(bar(kBODone), (t - 1) & 1);
        if (!ok) break;
        tc_fence_after_sync();
      }
      {
        // row h of P^T, key `row`: half row / 64, 16-byte chunk (row % 64) / 8 swizzled by h
        const int c = (row & 63) >> 3;
        uint8_t* pt = smem + kOffPT + (row >> 6) * kQHalfT + (row & 7) * 2;
#pragma unroll
        for (int h = 0; h < G; ++h)
          *reinterpret_cast<__nv_bfloat16*>(pt + h * 128 + ((c ^ h) << 4)) =
              __float2bfloat16_rn(pr[h]);
      }
      if (resc && !(m.flags & kTFirst)) {
        // thread = dim: scale this dim's accumulated O^T of each head
        uint32_t o[G];
        const uint32_t oc = tl + kColOT + (n & 1) * kNT;
        tmem_ld_cols<G>(oc, o);
#pragma unroll
        for (int h = 0; h < G; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * alpha[h]);
        tmem_st_cols<G>(oc, o);
        tmem_st_wait();
      }
      if (!kvalid) {
        // a key past the chunk's end: its V row holds whatever the stage held; zero it so that
        // p = 0 times it stays 0 (the stage's copies have landed: S of this tile is done)
        uint8_t* vrow = smem + st * kStageT + kOffVS + row * 128;
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
          for (int cc = 0; cc < 8; ++cc)
            *reinterpret_cast<uint4*>(vrow + h2 * kKVHalf + cc * 16) = make_uint4(0u, 0u, 0u, 0u);
      }
      fence_async_shared();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBPFull));

      if (m.flags & kTLast) {
        // ---- item finished: denominators, O^T, then the output or the chunk's partials ----
        float ls[G];
#pragma unroll
        for (int h = 0; h < G; ++h) ls[h] = warp_sum(l_part[h]);
        ok = exchange(ls, slot);
        if (!ok) break;
        float l[G];
#pragma unroll
        for (int h = 0; h < G; ++h) l[h] = (slot[h] + slot[8 + h]) + (slot[16 + h] + slot[24 + h]);
        ok = warp_wait(bar(kBODone), t & 1);
        if (!ok) break;
        tc_fence_after_sync();
        uint32_t o[G];
        tmem_ld_cols<G>(tl + kColOT + (n & 1) * kNT, o);
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBOFree + (n & 1)));
        const int head0 = m.x * G;
        if (m.nsplit == 1) {
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float inv = l[h] > 0.f ? 1.f / l[h] : 0.f;
            p.out[((int64_t)m.b * p.num_q_heads + head0 + h) * kDT + row] =
                __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(o[h]) * inv));
          }
        } else {
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const int64_t pi =
                ((int64_t)m.b * p.max_splits + m.split) * p.num_q_heads + head0 + h;
            p.part_acc[pi * kDT + row] = __uint_as_float(o[h]);
            // both quarters of a 64-dim half write its (max, denominator): the same values
            if (lane == 0) p.part_ml[pi * 2 + (quarter >> 1)] = make_float2(m_run[h], l[h]);
          }
          // The warp of this dim quarter that finishes the sequence's last chunk merges all of
          // them: o = sum_s 2^(m_s - M) acc_s / sum_s 2^(m_s - M) l_s.
          __threadfence();
          __syncwarp();
          uint32_t* ctr = p.counters + ((int64_t)m.b * nkv + m.x) * 4 + quarter;
          uint32_t done = 0;
          if (lane == 0) done = atomicAdd(ctr, 1u);
          done = __shfl_sync(kFullMask, done, 0);
          if (done == (uint32_t)m.nsplit - 1) {
            __threadfence();
#pragma unroll 1
            for (int h = 0; h < G; ++h) {
              const int64_t base = (int64_t)m.b * p.max_splits * p.num_q_heads + head0 + h;
              float M = -INFINITY, den = 0.f, num = 0.f;
#pragma unroll 1
              for (int sp0 = 0; sp0 < m.nsplit; sp0 += 4) {
                float2 ml[4];
                float a[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  ml[u] = make_float2(-INFINITY, 0.f);
                  a[u] = 0.f;
                  if (sp0 + u < m.nsplit) {
                    const int64_t pi = base + (int64_t)(sp0 + u) * p.num_q_heads;
                    ml[u] = __ldcg(p.part_ml + pi * 2 + (quarter >> 1));
                    a[u] = __ldcg(p.part_acc + pi * kDT + row);
                  }
                }
                float mnew = M;
#pragma unroll
                for (int u = 0; u < 4; ++u) mnew = fmaxf(mnew, ml[u].x);
                if (mnew == -INFINITY) continue;
                const float keep = M == -INFINITY ? 0.f : fast_exp2(M - mnew);
                den *= keep;
                num *= keep;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  const float wt = ml[u].x == -INFINITY ? 0.f : fast_exp2(ml[u].x - mnew);
                  den += wt * ml[u].y;
                  num += wt * a[u];
                }
                M = mnew;
              }
              const float inv = den > 0.f ? 1.f / den : 0.f;
              p.out[((int64_t)m.b * p.num_q_heads + head0 + h) * kDT + row] =
                  __bfloat16_as_ushort(__float2bfloat16_rn(num * inv));
            }
            if (lane == 0) *ctr = 0u;  // all chunks counted: ready for the next call
          }
        }
      }
      ++t;
      ++use;
    }
    if (!ok && lane == 0) raise_flag(p.flags, PKV_DEVERR_TIMEOUT);
    if (!ok && lane == 0) raise_flag(p.flags, PKV_DEVERR_TIMEOUT);
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemColsT);
  }
}

template <int G>
cudaError_t configure_tc_instance() {
  return cudaFuncSetAttribute(paged_decode_tc_kernel<G>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemT);
}

template <int G>
cudaError_t launch_tc_instance(const TcDecodeParams& p, int grid, const CUtensorMap& tq,
                               const CUtensorMap& tk, const CUtensorMap& tv,
                               const CUtensorMap* tail, cudaStream_t stream) {
  // a programmatic dependent of the plan grid, which it waits for in-kernel
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreadsT);
  cfg.dynamicSmemBytes = kSmemT;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, paged_decode_tc_kernel<G>, tq, tk, tv, tail[0], tail[1],
                            tail[2], tail[3], p);
}

}  // namespace

cudaError_t configure_decode_tc_kernels() {
  cudaError_t e = configure_tc_instance<1>();
  if (e == cudaSuccess) e = configure_tc_instance<2>();
  if (e == cudaSuccess) e = configure_tc_instance<4>();
  if (e == cudaSuccess) e = configure_tc_instance<8>();
  return e;
}

int decode_tc_box_rows(int block_size) { return block_size < kTK ? block_size : kTK; }

cudaError_t launch_paged_decode_tc(const DecodeArgs& a, const CUtensorMap& tq,
                                   const CUtensorMap& tk, const CUtensorMap& tv,
                                   const CUtensorMap* tail, int num_sms, cudaStream_t stream) {
  const int nkv = a.cache.num_kv_heads;
  const int G = a.num_q_heads / nkv;
  if (a.cache.head_dim != kDT || (G != 1 && G != 2 && G != 4 && G != 8))
    return cudaErrorNotSupported;
  TcDecodeParams p;
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
  p.num_kv_heads = nkv;
  p.block_size = a.cache.block_size;
  p.num_blocks = a.cache.num_blocks;
  p.max_splits = a.max_splits;
  const int64_t cap_table = (int64_t)a.max_blocks * a.cache.block_size;
  const int64_t cap_plan = (int64_t)a.max_splits * a.split_tokens;
  int64_t cap = cap_table < cap_plan ? cap_table : cap_plan;
  if (cap > 0x7fffffff) cap = 0x7fffffff;
  p.cap_tokens = (int32_t)cap;
  p.box_rows = decode_tc_box_rows(a.cache.block_size);
  p.qk_scale_log2 = a.scale * 1.4426950408889634f;

  const int64_t upper = (int64_t)a.num_seqs * a.max_splits * nkv;
  int64_t grid = num_sms;  // one CTA per SM
  if (grid > upper) grid = upper;
  if (grid < 1) grid = 1;
  // Chunks are sized as for two CTAs per SM although one runs: with one CTA per SM a chunk of
  // 0.4 of its share leaves a coarse tail (4 x 32768 + 60 short sequences at block_size 256:
  // 5064 GB/s, against 5147 with this sizing and 4332 with four CTAs' sizing).
  cudaError_t e =
      a.reuse_plan ? (a.k_new != nullptr ? launch_decode_store_rows(a, num_sms, stream)
                                         : cudaSuccess)
                   : launch_decode_plan(a, nkv, 2 * num_sms, a.max_splits > 1 ? nkv * 4 : 0,
                                        p.cap_tokens, num_sms, stream);
  if (e != cudaSuccess) return e;
  switch (G) {
    case 1: return launch_tc_instance<1>(p, (int)grid, tq, tk, tv, tail, stream);
    case 2: return launch_tc_instance<2>(p, (int)grid, tq, tk, tv, tail, stream);
    case 4: return launch_tc_instance<4>(p, (int)grid, tq, tk, tv, tail, stream);
    default: return launch_tc_instance<8>(p, (int)grid, tq, tk, tv, tail, stream);
  }
}

}  // namespace pkv
