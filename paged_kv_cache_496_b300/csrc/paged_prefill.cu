// paged_prefill.cu -- varlen causal paged prefill attention on tcgen05 tensor cores (sm_103a).
//
// Source: "DeepSeek研究员1200行代码复刻vLLM，H800硬件实测性能反超原版" (QbitAI), section
// "vLLM是什么？" (KV in fixed-size blocks reached through a block table; KV shared within and
// across requests) and "nano-vllm 深度分析报告", section "创新之处" (prefix-cache hits reuse
// physical blocks). A sequence's new queries attend to its cached prefix, which may sit in blocks
// shared with other sequences, plus its own new tokens, causally and aligned to the end.
//
// Design (per CTA: one sequence, one kv head, one tile of 128 query rows):
//  * The 128 rows are 128/G positions x the G query heads that share the kv head, so each K/V
//    tile feeds all of them (rows ordered position-major, as the Q TMA box delivers them).
//  * Warp 0 claims items and streams 64-key K and V tiles through the block table with 3-D TMA
//    boxes in 128-byte swizzle (the layout the tensor core reads). K and V have their own
//    three-deep rings and barriers, and K runs one tile ahead of V: a K buffer is free as soon as
//    its S = Q K^T is done. An item's Q travels through the K ring too, as two 16 KB slots of 64
//    dims each, ahead of its first key tile. Each ring slot has its own issuing lane: one
//    thread's bulk copies complete one barrier phase at a time (a few hundred nanoseconds each,
//    whatever their size), so a thread with several phases in flight would queue them.
//  * Warp 1 allocates 256 TMEM columns and, from one thread, copies Q from the ring into TMEM
//    columns [192, 256) (tcgen05.cp), issues S = Q K^T (M=128, N=64, K=128: eight kind::f16
//    MMAs, A from TMEM, K K-major in shared memory) into columns [0, 64) and O += P V (M=128,
//    N=128, K=64: four MMAs, V read MN-major) into columns [64, 192). With A in TMEM an N=64 MMA
//    reads 2 KB of shared memory instead of 6 KB and is no longer limited by that read.
//  * Warps 2-5 (one TMEM lane quarter each, thread = query row) load S rows, apply the causal
//    mask and an online softmax in log2 units with a lazy rescale (O in TMEM is rescaled only when
//    a row's max grows by more than 2^8), write P as bf16 into shared memory in the swizzled
//    K-major layout, and finally normalise O and store it.
//  * The tensor core computes S for the next tile while the softmax warps work on the current
//    one. Every wait is bounded; the CTA always frees its TMEM.
//  * Items are claimed from a counter. With a large enough workspace a one-CTA plan kernel first
//    numbers only the query tiles each sequence has, and orders a batch that mixes prefill rows
//    with decode rows so that the two kinds alternate in the claims: a decode row costs this
//    kernel a full tile's MMAs and softmax, so memory-bound and compute-bound work overlap only
//    when they are claimed side by side.
#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace pkv {

namespace {

constexpr int kRows = 128;  // MMA M: query rows per CTA
constexpr int kKeys = 64;   // keys per tile
constexpr int kHD = 128;    // head_dim
constexpr int kThreadsP = 192;
constexpr int kTmemCols = 256;
constexpr int kColS = 0;
constexpr int kColO = 64;
constexpr int kColQ = 192;  // Q as the MMA A operand: 128 lanes x 64 columns of bf16 pairs
constexpr float kTauP = 8.0f;

constexpr int kQHalf = kRows * 128;          // 16 KB: 64 dims of Q, one K-ring slot
constexpr int kKTile = kKeys * kHD * 2;      // 16 KB: two 8 KB halves
constexpr int kKHalf = kKeys * 128;          // 8 KB
constexpr int kKStages = 3;
constexpr int kVStages = 3;
constexpr int kPBytes = kRows * kKeys * 2;
constexpr int kOffP = 0;
constexpr int kOffK = kOffP + kPBytes;
constexpr int kOffV = kOffK + kKStages * kKTile;
constexpr int kOffBar = kOffV + kVStages * kKTile;
static_assert(kQHalf == kKTile, "a Q half fills one K-ring slot");
// barriers: k_full[], k_empty[], v_full[], v_empty[], s_full, s_free, p_full, o_done, o_free,
// mma_done, item_full[2], item_empty[2]
constexpr int kBarFullK = 0, kBarEmptyK = kBarFullK + kKStages,
              kBarFullV = kBarEmptyK + kKStages, kBarEmptyV = kBarFullV + kVStages,
              kBarSFull = kBarEmptyV + kVStages, kBarSFree = kBarSFull + 1,
              kBarPFull = kBarSFree + 1, kBarODone = kBarPFull + 1, kBarOFree = kBarODone + 1,
              kBarMma = kBarOFree + 1, kBarItemFull = kBarMma + 1, kBarItemEmpty = kBarItemFull + 2,
              kNumBars = kBarItemEmpty + 2;
constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
// Two item slots of kItemInts ints: the claimed id (-1 = no more work) and the item's fields
constexpr int kItemInts = 12;
constexpr int kOffItem = kOffTmemSlot + 16;
constexpr int kSmemBytes = kOffItem + 2 * kItemInts * 4;
constexpr int kItemReaders = 5;  // the MMA thread and the four softmax warps
static_assert(kOffK % 1024 == 0 && kOffV % 1024 == 0 && kOffP % 1024 == 0 && kKTile % 1024 == 0,
              "swizzle atoms need 1024-byte alignment");
static_assert(2 * (kSmemBytes + 1024) <= 228 * 1024, "two CTAs per SM");

struct PrefillParams {
  const int32_t* cu_q;
  const int32_t* cu_k;
  const int32_t* block_tables;  // nullptr: keys come from k / v directly
  uint16_t* out;
  int* flags;
  int32_t max_blocks;
  int32_t num_seqs;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t group;         // G = num_q_heads / num_kv_heads
  int32_t pos_per_tile;  // 128 / G
  int32_t num_q_tiles;   // ceil(max_seqlen_q / pos_per_tile)
  int32_t num_items;     // num_seqs * num_kv_heads * num_q_tiles
  int32_t* item_counter; // zero at launch; CTAs claim item ids from it
  int32_t block_size;
  int32_t num_blocks;
  int32_t box_rows;      // rows per K/V TMA box
  int32_t oob_row;       // a row coordinate past the end of the K/V tensors (zero fill)
  float qk_scale_log2;
  // Dense numbering when non-null: the sequence at position pos is item_perm[pos] (heavy ones
  // spread among light ones) and its items are ids item_prefix[pos] .. item_prefix[pos + 1] - 1
  // (its kv heads x its own query tiles), item_prefix[num_seqs] of them in all; written by
  // prefill_plan_kernel, with the counters, before this grid reads them.
  const int32_t* item_prefix;
  const int32_t* item_perm;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// One unit of work: a tile of pos_per_tile query positions x G heads of one (sequence, kv head).
struct Item {
  int b, g, q_start, q_len, k_len, q0, P, n_kt;
};
static_assert(sizeof(Item) / 4 + 1 <= kItemInts, "item slot size");

constexpr int kItemSkip = 0;  // no work (a tile past the sequence's end, or invalid lengths)
constexpr int kItemWork = 1;

// Items are numbered so that the query tiles of one (sequence, kv head) are adjacent, longest
// first: CTAs that run at the same time then share that head's K/V through L2. Without a plan
// (sparse numbering) id = (sequence x kv heads + kv head) x num_q_tiles + tile, and ids past a
// sequence's tiles or with invalid lengths have no work; invalid lengths are flagged once per
// sequence. The dense numbering's lookup runs inside the producer (below).
__device__ __forceinline__ int load_item(const PrefillParams& p, int id, Item& it) {
  const int qt = p.num_q_tiles - 1 - id % p.num_q_tiles;
  const int t = id / p.num_q_tiles;
  it.g = t % p.num_kv_heads;
  it.b = t / p.num_kv_heads;
  it.q_start = __ldg(p.cu_q + it.b);
  it.q_len = __ldg(p.cu_q + it.b + 1) - it.q_start;
  it.k_len = __ldg(p.cu_k + it.b + 1) - __ldg(p.cu_k + it.b);
  if (it.q_len < 0 || it.k_len < it.q_len) {
    if (threadIdx.x == 0 && qt == 0 && it.g == 0) raise_flag(p.flags, PKV_DEVERR_BAD_LENGTHS);
    return kItemSkip;
  }
  it.q0 = qt * p.pos_per_tile;
  if (it.q0 >= it.q_len) return kItemSkip;
  it.P = it.k_len - it.q_len;  // cached prefix length
  const int last_pos = min(it.q_len, it.q0 + p.pos_per_tile) - 1;
  it.n_kt = (it.P + last_pos + 1 + kKeys - 1) / kKeys;
  return kItemWork;
}

// Persistent: the producer claims item ids in increasing order from a global counter (skipping
// items without work) and hands each to the MMA thread and the softmax warps through a two-slot
// ring in shared memory. All ring and barrier phases count tiles over the CTA's whole life, so the
// producer loads the next item's Q and first K while the current item finishes, and the tensor
// core computes the next item's first S while the softmax warps write out the current item's O.
__global__ void __launch_bounds__(kThreadsP, 2)
    paged_prefill_kernel(const __grid_constant__ CUtensorMap tmap_q,
                         const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v, const PrefillParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if ((smem_addr(smem) & 1023u) != 0) {  // the swizzled layouts need a 1024-byte aligned base
    if (threadIdx.x == 0) raise_flag(p.flags, PKV_DEVERR_INTERNAL);
    return;
  }
  const int G = p.group;

  const uint32_t sbase = smem_addr(smem);
  const uint32_t bar0 = sbase + kOffBar;
  auto bar = [bar0](int i) { return bar0 + 8u * (uint32_t)i; };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + kOffTmemSlot);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(bar(kBarFullK + s), 1);
      mbar_init(bar(kBarEmptyK + s), 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(bar(kBarFullV + s), 1);
      mbar_init(bar(kBarEmptyV + s), 1);
    }
    mbar_init(bar(kBarSFull), 1);
    mbar_init(bar(kBarSFree), 4);
    mbar_init(bar(kBarPFull), 4);
    mbar_init(bar(kBarODone), 1);
    mbar_init(bar(kBarOFree), 4);
    mbar_init(bar(kBarMma), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kBarItemFull + s), 1);
      mbar_init(bar(kBarItemEmpty + s), kItemReaders);
    }
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(sbase + kOffTmemSlot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  // With dense numbering this grid is a programmatic dependent of the plan kernel: everything
  // above overlapped the plan; nothing below reads memory before the plan (and all earlier work)
  // has completed. Without a plan the wait returns at once.
  grid_dependency_wait();
  // The producer decodes each claimed item once and passes its fields to the other warps through
  // a two-slot ring in shared memory, so that no consumer reloads the sequence lengths from
  // global memory when it moves to the next item.
  volatile int* item_slots = reinterpret_cast<volatile int*>(smem + kOffItem);
  auto read_slot = [&](int n, Item& it) -> int {
    volatile int* sl = item_slots + (n & 1) * kItemInts;
    it.b = sl[1]; it.g = sl[2]; it.q_start = sl[3]; it.q_len = sl[4];
    it.k_len = sl[5]; it.q0 = sl[6]; it.P = sl[7]; it.n_kt = sl[8];
    return sl[0];
  };
  // one consumer thread: the id of the n-th item this CTA works on (-1: none left, or a timeout)
  auto take_item_thread = [&](int n, Item& it) -> int {
    int id = -1;
    if (mbar_wait(bar(kBarItemFull + (n & 1)), (n >> 1) & 1)) {
      id = read_slot(n, it);
    } else {
      raise_flag(p.flags, PKV_DEVERR_TIMEOUT);
    }
    mbar_arrive(bar(kBarItemEmpty + (n & 1)));
    return id;
  };
  // a whole consumer warp: lane 0 waits, every lane reads the slot, then lane 0 releases it
  auto take_item_warp = [&](int n, Item& it) -> int {
    int full = 0;
    if (lane == 0) {
      full = mbar_wait(bar(kBarItemFull + (n & 1)), (n >> 1) & 1) ? 1 : 0;
      if (!full) raise_flag(p.flags, PKV_DEVERR_TIMEOUT);
    }
    full = __shfl_sync(kFullMask, full, 0);
    const int id = full ? read_slot(n, it) : -1;
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(kBarItemEmpty + (n & 1)));
    return id;
  };

  if (warp == 0) {
    // =============================== producer ===============================
    // Per item: its two Q halves into the K ring, then for global tile t: K(t) and V(t-1); K runs
    // one tile ahead of V. kr counts K-ring slots used (Q halves and key tiles). All lanes run
    // the loop (the block-table window is spread over them); each ring slot has its own issuing
    // lane, so that a thread never has more than one barrier phase of copies in flight.
    bool ok = true;
    if (lane == 0) {
      tma_prefetch_desc(&tmap_q);
      tma_prefetch_desc(&tmap_k);
      tma_prefetch_desc(&tmap_v);
    }
    const bool paged = p.block_tables != nullptr;
    // block_size is a power of two: positions map to table entries by shifts and masks (a
    // division by a runtime value would cost the producer tens of instructions per tile)
    const int bs = p.block_size;
    const int lbs = __ffs(bs) - 1;
    const int ent = (kKeys + bs - 1) >> lbs;  // table entries one key tile spans
    const int box = p.box_rows;
    const int nsub = kKeys / box;
    int t = 0, n = 0, kr = 0;
    // cache rows and kv head of key tile t - 1
    int prev_rows[kKeys / 16];
#pragma unroll
    for (int sb = 0; sb < kKeys / 16; ++sb) prev_rows[sb] = 0;
    int prev_g = 0;
    // Lane s (s < kKStages) owns K-ring slot s and lane kKStages + s owns V-ring slot s: it waits
    // for the slot and issues the copies into it. Unless k_on is false, the owner of K-ring slot
    // use kr puts K of the current key tile (cache rows k_rows, kv head gk) there; unless v_on is
    // false, the owner of the slot of V tile tv puts V (rows prev_rows, head prev_g) there.
    // Returns the lane's success.
    auto issue_kv = [&](const int (&k_rows)[kKeys / 16], int gk, bool k_on, int tv,
                        bool v_on) -> bool {
      const bool isk = k_on && lane == kr % kKStages;
      const bool isv = v_on && lane == kKStages + tv % kVStages;
      if (!isk && !isv) return true;
      const int u = isk ? kr : tv;
      const int st = isk ? u % kKStages : u % kVStages;
      const int use = isk ? u / kKStages : u / kVStages;
      if (!mbar_wait(bar((isk ? kBarEmptyK : kBarEmptyV) + st), (use & 1) ^ 1)) return false;
      const uint32_t full = bar((isk ? kBarFullK : kBarFullV) + st);
      mbar_arrive_expect_tx(full, kKTile);
      const uint32_t d = sbase + (isk ? kOffK : kOffV) + st * kKTile;
      const CUtensorMap* map = isk ? &tmap_k : &tmap_v;
      const int g = isk ? gk : prev_g;
#pragma unroll
      for (int sb = 0; sb < kKeys / 16; ++sb) {
        if (sb < nsub) {
          const uint32_t off = (uint32_t)(sb * box * 128);
          const int r = isk ? k_rows[sb] : prev_rows[sb];
          tma_load_3d(d + off, map, 0, g, r, full);
          tma_load_3d(d + kKHalf + off, map, 64, g, r, full);
        }
      }
      return true;
    };
    const bool dense = p.item_prefix != nullptr;
    const int num_items = dense ? __ldg(p.item_prefix + p.num_seqs) : p.num_items;
    // positions are permuted (heavy sequences spread among light ones) only when the batch
    // holds both kinds of sequence
    const int n_heavy_seqs = dense ? __ldg(p.item_counter + 1) : 0;
    const bool permuted = n_heavy_seqs > 0 && n_heavy_seqs < p.num_seqs;
    int claimed = lane == 0 ? atomicAdd(p.item_counter, 1) : 0;
    // Dense numbering: the position holding a claimed id is found by a 128-way search over
    // item_prefix: each lane probes four points and ballots narrow the range 129-fold (one round
    // of loads for up to 128 sequences, two for up to 16,641). The sequence's lengths and its
    // first block-table window (entries 0..31, masked by the need at use) are then loaded
    // together, so a lookup costs two or three dependent loads (one more when the positions are
    // permuted) instead of a bisection's log2(num_seqs) + 2.
    auto find_dense = [&](int id, Item& it, int& w) {
      int lo = 0, hi = p.num_seqs;  // item_prefix[lo] <= id < item_prefix[hi]
      int b = lo;
      while (hi - lo > 1) {
        const int step = (hi - lo + 127) >> 7;
        // the last round probes single positions (step 1): with permuted positions it also
        // loads the sequence at every probe and at lo, so the answer costs no extra round trip
        const bool with_perm = permuted && step == 1;
        int v[4], pv[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int idx = lo + (q * 32 + lane + 1) * step;
          v[q] = idx < hi ? __ldg(p.item_prefix + idx) : 0x7fffffff;
          pv[q] = with_perm && idx < hi ? __ldg(p.item_perm + idx) : 0;
        }
        const int p_lo = with_perm ? __ldg(p.item_perm + lo) : 0;
        // probes are non-decreasing in (q, lane) order: the ones at or below id lead
        int k = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) k += __popc(__ballot_sync(kFullMask, v[q] <= id));
        if (with_perm) {  // the answer is lo + k: position lo itself, or probe k - 1
          const int slot = (k - 1) >> 5;  // uniform over the warp
          const int mine = slot <= 0 ? pv[0] : slot == 1 ? pv[1] : slot == 2 ? pv[2] : pv[3];
          const int from = __shfl_sync(kFullMask, mine, (k - 1) & 31);
          b = k == 0 ? p_lo : from;
        }
        hi = min(hi, lo + (k + 1) * step);
        lo += k * step;
      }
      const int pos = lo;
      if (!permuted) b = pos;
      // lanes 0-4: cu_q[b], cu_q[b + 1], cu_k[b], cu_k[b + 1], item_prefix[pos]
      const int32_t* src = lane < 2 ? p.cu_q + b + lane
                                    : (lane < 4 ? p.cu_k + b + lane - 2 : p.item_prefix + pos);
      const int f = lane < 5 ? __ldg(src) : 0;
      w = paged && lane < p.max_blocks ? __ldg(p.block_tables + (int64_t)b * p.max_blocks + lane)
                                       : -1;
      it.b = b;
      it.q_start = __shfl_sync(kFullMask, f, 0);
      it.q_len = __shfl_sync(kFullMask, f, 1) - it.q_start;
      it.k_len = __shfl_sync(kFullMask, f, 3) - __shfl_sync(kFullMask, f, 2);
      const int local = id - __shfl_sync(kFullMask, f, 4);
      const int tiles = (it.q_len + p.pos_per_tile - 1) / p.pos_per_tile;  // >= 1: listed
      it.g = local / tiles;
      it.q0 = (tiles - 1 - local % tiles) * p.pos_per_tile;
      it.P = it.k_len - it.q_len;
      const int last_pos = min(it.q_len, it.q0 + p.pos_per_tile) - 1;
      it.n_kt = (it.P + last_pos + 1 + kKeys - 1) / kKeys;
    };
    while (ok) {
      // next item with work, or -1; the claim after it is issued now and used later
      int id = -1, w0 = -1;
      Item it;
      if (dense) {
        id = __shfl_sync(kFullMask, claimed, 0);
        if (id < num_items) {
          if (lane == 0) claimed = atomicAdd(p.item_counter, 1);
          find_dense(id, it, w0);
        } else {
          id = -1;
        }
      } else if (lane == 0) {
        while (claimed < num_items) {
          const int c = claimed;
          claimed = atomicAdd(p.item_counter, 1);
          if (load_item(p, c, it) == kItemWork) {
            id = c;
            break;
          }
        }
      }
      if (lane == 0) {
        ok = mbar_wait(bar(kBarItemEmpty + (n & 1)), ((n >> 1) & 1) ^ 1);
        if (ok) {
          volatile int* sl = item_slots + (n & 1) * kItemInts;
          sl[0] = id;
          if (id >= 0) {
            sl[1] = it.b; sl[2] = it.g; sl[3] = it.q_start; sl[4] = it.q_len;
            sl[5] = it.k_len; sl[6] = it.q0; sl[7] = it.P; sl[8] = it.n_kt;
          }
          mbar_arrive(bar(kBarItemFull + (n & 1)));
        }
      }
      ok = __shfl_sync(kFullMask, ok ? 1 : 0, 0) != 0;
      id = __shfl_sync(kFullMask, id, 0);
      if (!ok || id < 0) break;
      if (!dense) {
        it.b = __shfl_sync(kFullMask, it.b, 0);
        it.g = __shfl_sync(kFullMask, it.g, 0);
        it.q_start = __shfl_sync(kFullMask, it.q_start, 0);
        it.q_len = __shfl_sync(kFullMask, it.q_len, 0);
        it.k_len = __shfl_sync(kFullMask, it.k_len, 0);
        it.q0 = __shfl_sync(kFullMask, it.q0, 0);
        it.P = __shfl_sync(kFullMask, it.P, 0);
        it.n_kt = __shfl_sync(kFullMask, it.n_kt, 0);
      }
      int need_ent = 0;
      const int32_t* bt_row = nullptr;
      int win_base = -1000000, win_val = -1;
      if (paged) {
        need_ent = (it.k_len + bs - 1) >> lbs;
        if (need_ent > p.max_blocks) {
          if (lane == 0) raise_flag(p.flags, PKV_DEVERR_CTX_CLAMPED);
          need_ent = p.max_blocks;
        }
        bt_row = p.block_tables + (int64_t)it.b * p.max_blocks;
        if (dense) {  // entries 0..31, loaded by the lookup
          win_base = 0;
          win_val = w0;
        }
      }
      // Q half h into K-ring slot use kr + h, from that slot's lane
      const int hq = (lane + kKStages - kr % kKStages) % kKStages;
      if (lane < kKStages && hq < 2) {
        const int u = kr + hq, st = u % kKStages;
        ok = mbar_wait(bar(kBarEmptyK + st), ((u / kKStages) & 1) ^ 1);
        if (ok) {
          const uint32_t full = bar(kBarFullK + st);
          mbar_arrive_expect_tx(full, kKTile);
          tma_load_3d(sbase + kOffK + st * kKTile, &tmap_q, 64 * hq, it.g * G,
                      it.q_start + it.q0, full);
        }
      }
      kr += 2;
      ok = __all_sync(kFullMask, ok);
      for (int j = 0; j < it.n_kt && ok; ++j, ++t) {
        int rows[kKeys / 16];
#pragma unroll
        for (int sb = 0; sb < kKeys / 16; ++sb) rows[sb] = p.oob_row;
        const int key0 = j * kKeys;
        if (paged) {
          const int e0 = key0 >> lbs;
          if (e0 < win_base || e0 + ent > win_base + 32) {
            win_base = e0;
            const int e = e0 + lane;
            win_val = e < need_ent ? __ldg(bt_row + e) : -1;
          }
#pragma unroll
          for (int sb = 0; sb < kKeys / 16; ++sb) {
            if (sb < nsub) {
              const int key = key0 + sb * box;
              const int blk = __shfl_sync(kFullMask, win_val, ((key >> lbs) - win_base) & 31);
              if (key < it.k_len && (key >> lbs) < need_ent) {
                if (blk >= 0 && blk < p.num_blocks) {
                  rows[sb] = blk * bs + (key & (bs - 1));
                } else if (lane == 0) {
                  raise_flag(p.flags, PKV_DEVERR_BAD_BLOCK);
                }
              }
            }
          }
        } else {
#pragma unroll
          for (int sb = 0; sb < kKeys / 16; ++sb)
            if (sb < nsub) rows[sb] = it.q_start + key0 + sb * box;
        }
        if (lane < kKStages + kVStages) ok = issue_kv(rows, it.g, true, t - 1, j > 0);
        ++kr;
        ok = __all_sync(kFullMask, ok);
#pragma unroll
        for (int sb = 0; sb < kKeys / 16; ++sb) prev_rows[sb] = rows[sb];
        prev_g = it.g;
      }
      // V of the item's last key tile goes out now, so that the item's last P V (issued as soon
      // as its P is ready) does not wait for the next item's claim and Q
      if (ok && lane < kKStages + kVStages) ok = issue_kv(prev_rows, prev_g, false, t - 1, true);
      ok = __all_sync(kFullMask, ok);
      ++n;
    }
    if (lane == 0) {
      if (!ok) raise_flag(p.flags, PKV_DEVERR_TIMEOUT);
      // never leave while a copy into this CTA's shared memory may be in flight: wait for the
      // last uses of each ring's slots (earlier ones completed before their slot was reused).
      // After a timeout some of these were never issued; their waits then also time out, which
      // is harmless.
      bool drained = true;
      for (int i = (kr > kKStages ? kr - kKStages : 0); i < kr && drained; ++i)
        drained = mbar_wait(bar(kBarFullK + i % kKStages), (i / kKStages) & 1);
      for (int i = (t > kVStages ? t - kVStages : 0); i < t && drained; ++i)
        drained = mbar_wait(bar(kBarFullV + i % kVStages), (i / kVStages) & 1);
      if (!drained) raise_flag(p.flags, PKV_DEVERR_TIMEOUT);
    }
  } else if (warp == 1) {
    // ============================ MMA issuer (one thread) ============================
    // Per item: Q from its two K-ring slots into TMEM; then for global tile t: S(t) = Q K(t)^T,
    // then O += P(t-1) V(t-1), so the tensor core computes the next S while the softmax warps work
    // on the current one, across item boundaries too.
    if (lane == 0) {
      const uint32_t idesc_s = idesc_bf16_f32(kRows, kKeys, false);
      const uint32_t idesc_o = idesc_bf16_f32(kRows, kHD, true);
      const uint64_t adesc_p = sdesc_kmajor_sw128(sbase + kOffP);
      bool ok = true;
      // O += P V for global tile tv; `first`: the first tile of item number nv (O starts at 0,
      // after the previous item's O has been read out)
      auto issue_pv = [&](int tv, bool first, int nv) {
        if (!ok) return;
        ok = mbar_wait(bar(kBarFullV + tv % kVStages), (tv / kVStages) & 1);
        if (ok) ok = mbar_wait(bar(kBarPFull), tv & 1);
        if (ok && first && nv > 0) ok = mbar_wait(bar(kBarOFree), (nv - 1) & 1);
        if (!ok) return;
        tc_fence_after_sync();
        // descriptors advance by address / 16 in their low 14 bits (shared addresses < 256 KB)
        const uint64_t bdesc0 =
            sdesc_mnmajor_sw128(sbase + kOffV + (tv % kVStages) * kKTile, kKHalf);
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk) {
          tc_mma_f16(tmem + kColO, adesc_p + (uint64_t)(kk * 32 / 16),
                     bdesc0 + (uint64_t)(kk * 16 * 128 / 16), idesc_o,
                     (!first || kk > 0) ? 1u : 0u);
        }
        tc_commit(bar(kBarODone));
        tc_commit(bar(kBarEmptyV + tv % kVStages));
      };
      int t = 0, n = 0, kr = 0;
      bool pending = false, pend_first = false;
      int pend_n = 0;
      while (ok) {
        Item it;
        if (take_item_thread(n, it) < 0) break;
        // the previous item's S MMAs read Q's TMEM columns: they are complete before the copy
        // below overwrites them (an MMA followed by a copy is not ordered by the tensor core)
        if (ok && t > 0) ok = mbar_wait(bar(kBarSFull), (t - 1) & 1);
        for (int h = 0; h < 2 && ok; ++h, ++kr) {
          const int st = kr % kKStages;
          ok = mbar_wait(bar(kBarFullK + st), (kr / kKStages) & 1);
          if (!ok) break;
          tc_fence_after_sync();
          const uint32_t qs = sbase + kOffK + st * kKTile;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_cp_128x256b(tmem + kColQ + (h * 4 + kk) * 8, sdesc_kmajor_sw128(qs + kk * 32));
          tc_commit(bar(kBarEmptyK + st));
        }
        for (int j = 0; j < it.n_kt && ok; ++j, ++t, ++kr) {
          const int st = kr % kKStages;
          ok = mbar_wait(bar(kBarFullK + st), (kr / kKStages) & 1);
          if (ok && t > 0) ok = mbar_wait(bar(kBarSFree), (t - 1) & 1);
          if (!ok) break;
          tc_fence_after_sync();
          const uint64_t kdesc0 = sdesc_kmajor_sw128(sbase + kOffK + st * kKTile);
#pragma unroll
          for (int kk = 0; kk < kHD / 16; ++kk) {
            const uint64_t bdesc = kdesc0 + (uint64_t)(((kk >> 2) * kKHalf + (kk & 3) * 32) / 16);
            tc_mma_f16_ts(tmem + kColS, tmem + kColQ + kk * 8, bdesc, idesc_s, kk > 0 ? 1u : 0u);
          }
          tc_commit(bar(kBarSFull));
          tc_commit(bar(kBarEmptyK + st));
          if (pending) issue_pv(t - 1, pend_first, pend_n);
          pending = true;
          pend_first = j == 0;
          pend_n = n;
        }
        // The item's last P V goes out as soon as its P is ready, ahead of the next item's Q
        // copy and first S: the softmax warps can then write out O while the next item's Q and
        // first K tile are still arriving.
        if (pending) issue_pv(t - 1, pend_first, pend_n);
        pending = false;
        ++n;
      }
      if (pending) issue_pv(t - 1, pend_first, pend_n);
      if (!ok) raise_flag(p.flags, PKV_DEVERR_TIMEOUT);
      // all MMAs of this CTA are complete before TMEM is released
      tc_commit(bar(kBarMma));
      if (!mbar_wait(bar(kBarMma), 0)) raise_flag(p.flags, PKV_DEVERR_TIMEOUT);
    }
    __syncwarp();
  } else {
    // ======================== softmax warps: thread = query row ========================
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
    bool ok = true;
    int t = 0;
    for (int n = 0; ok; ++n) {
      Item it;
      if (take_item_warp(n, it) < 0) break;
      const int pos = it.q0 + r / G;
      const bool row_valid = pos < it.q_len;
      const int limit = it.P + pos;  // last key this row may see
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; j < it.n_kt; ++j, ++t) {
        ok = mbar_wait(bar(kBarSFull), t & 1);
        if (!ok) break;
        tc_fence_after_sync();
        uint32_t sr[64];
        tmem_ld64(trow + kColS, sr);
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarSFree));

        const int kbase = j * kKeys;
        // Tiles below every row's causal limit and inside k_len need no mask (CTA-uniform
        // test); there, with a positive scale, max and exp take the raw scores:
        // p = 2^(s*c - m). Arithmetic runs on pairs (fp32x2 FMA and add) and the max takes
        // three inputs per instruction, in four chains.
        const bool full = kbase + kKeys - 1 <= it.P + it.q0 && kbase + kKeys <= it.k_len &&
                          p.qk_scale_log2 > 0.f;
        if (!full) {
          // keys kbase + c with c < nv are unmasked for this row (c <= limit - kbase, inside k_len)
          const int nv = max(0, min(kKeys, min(limit + 1, it.k_len) - kbase));
#pragma unroll
          for (int c = 0; c < 64; ++c)
            sr[c] = __float_as_uint(c < nv ? __uint_as_float(sr[c]) * p.qk_scale_log2
                                           : -INFINITY);
        }
        float mt;
        {
          auto sv = [&sr](int c) { return __uint_as_float(sr[c]); };
          float mx[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) mx[u] = fmax3(sv(u), sv(u + 4), sv(u + 8));
#pragma unroll
          for (int k = 3; k < 15; k += 2)
#pragma unroll
            for (int u = 0; u < 4; ++u) mx[u] = fmax3(mx[u], sv(u + 4 * k), sv(u + 4 * k + 4));
#pragma unroll
          for (int u = 0; u < 4; ++u) mx[u] = fmaxf(mx[u], sv(u + 60));
          mt = fmaxf(fmax3(mx[0], mx[1], mx[2]), mx[3]);
        }
        if (full) mt *= p.qk_scale_log2;
        const bool resc = mt > m_run + kTauP;
        float alpha = 1.f;
        if (resc) {
          alpha = fast_exp2(m_run - mt);  // 0 when nothing was seen yet
          m_run = mt;
        }
        uint32_t pk[32];
        uint64_t sum2[4] = {0ull, 0ull, 0ull, 0ull};  // pair sums of p
        {
          // full tiles: x = s*c - m; masked tiles: x = s - m, where masked scores are -inf and
          // 2^-inf = 0 (a row with no unmasked key yet has m_run = -inf and only masked scores
          // here, so any finite offset gives its zeros)
          const float mm = m_run == -INFINITY ? 0.f : m_run;
          const uint64_t mul = full ? pack2(p.qk_scale_log2, p.qk_scale_log2) : pack2(1.f, 1.f);
          const uint64_t off = pack2(-mm, -mm);
#pragma unroll
          for (int c = 0; c < 64; c += 2) {
            const float2 x = unpack2(ffma2(
                pack2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), mul, off));
            const float p0 = fast_exp2(x.x), p1 = fast_exp2(x.y);
            sum2[(c >> 1) & 3] = fadd2(sum2[(c >> 1) & 3], pack2(p0, p1));
            pk[c / 2] = pack_bf16x2(p0, p1);
          }
        }
        const float2 s01 = unpack2(fadd2(sum2[0], sum2[1]));
        const float2 s23 = unpack2(fadd2(sum2[2], sum2[3]));
        const float sum = (s01.x + s01.y) + (s23.x + s23.y);
        l_run = l_run * alpha + sum;

        if (t > 0) {  // the previous P V is done: P buffer free, O stable
          ok = mbar_wait(bar(kBarODone), (t - 1) & 1);
          if (!ok) break;
          tc_fence_after_sync();
        }
        {
          uint8_t* pbuf = smem + kOffP;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint4 v = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
            *reinterpret_cast<uint4*>(pbuf + r * 128 + ((c ^ (r & 7)) << 4)) = v;
          }
        }
        if (j > 0 && __any_sync(kFullMask, resc)) {
#pragma unroll 1
          for (int cc = 0; cc < kHD / 32; ++cc) {
            uint32_t o[32];
            tmem_ld32(trow + kColO + cc * 32, o);
            const uint64_t a2 = pack2(alpha, alpha);
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
              const float2 v = unpack2(
                  fmul2(pack2(__uint_as_float(o[c]), __uint_as_float(o[c + 1])), a2));
              o[c] = __float_as_uint(v.x);
              o[c + 1] = __float_as_uint(v.y);
            }
            tmem_st32(trow + kColO + cc * 32, o);
          }
        }
        tmem_st_wait();
        if (j == it.n_kt - 1 && kbase + kKeys > it.k_len) {
          // V rows past the last key hold whatever the cache holds there: zero them (after the
          // stage's copy has landed)
          ok = mbar_wait(bar(kBarFullV + t % kVStages), (t / kVStages) & 1);
          if (!ok) break;
          const int first = it.k_len - kbase;
          uint8_t* vt = smem + kOffV + (t % kVStages) * kKTile;
          const int nrow = kKeys - first;
          for (int i = threadIdx.x - 64; i < nrow * 16; i += 128) {
            const int row = first + i / 16, part16 = i % 16;  // 16 x 16 bytes = both halves
            *reinterpret_cast<uint4*>(vt + (part16 >> 3) * kKHalf + row * 128 +
                                      (part16 & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        fence_async_shared();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarPFull));
      }
      if (ok) ok = mbar_wait(bar(kBarODone), (t - 1) & 1);
      if (!ok) break;
      tc_fence_after_sync();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      uint16_t* orow =
          p.out + ((int64_t)(it.q_start + pos) * p.num_q_heads + it.g * G + r % G) * kHD;
      uint32_t w[64];  // the row's O as bf16 pairs, normalised
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t o[64];
        tmem_ld64(trow + kColO + cc * 64, o);
        const uint64_t inv2 = pack2(inv, inv);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float2 v = unpack2(
              fmul2(pack2(__uint_as_float(o[2 * c]), __uint_as_float(o[2 * c + 1])), inv2));
          w[cc * 32 + c] = pack_bf16x2(v.x, v.y);
        }
      }
      // O is in registers: the next item's P V may overwrite it
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarOFree));
      if (row_valid) {
        uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
        for (int c = 0; c < 16; ++c)
          dst[c] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
      }
    }
    if (!ok && lane == 0) raise_flag(p.flags, PKV_DEVERR_TIMEOUT);
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

// Dense item numbering with heavy sequences spread among light ones. A sequence is heavy when
// its query tiles are at least half full (q_len >= positions per tile / 2: prefill rows,
// compute-bound) and light otherwise (decode rows and short chunks, bound by their K/V read).
// The grid claims items in position order; heavy sequence i (of H, in batch order) and light
// sequence j (of L) are merged by the keys (i + 1/2) / H and (j + 1/2) / L, heavy first on a
// tie, so every stretch of claims mixes the two kinds in the batch's proportion and the
// prefill tiles' tensor work fills the time the decode rows wait on memory. item_perm[pos] is
// the sequence at position pos, item_prefix[pos] its first item id (kv heads x its own query
// tiles, longest first), item_prefix[num_seqs] = all items. counter[0] is zeroed for the
// claims and counter[1] = H (no permutation when H is 0 or num_seqs). Sequences with invalid
// lengths have no items and are flagged here. One CTA; the attention grid is its programmatic
// dependent.
constexpr int kPlanThreadsP = 1024;
// Heavy sequence i's merge key is (kMixA / kMixB) (i + 1/2) / H. Spreading the prefill rows over
// the whole run of decode rows (1/1) measured best on a mixed batch: 5743 GB/s of K/V, against
// 5684 with them over the first three quarters (3/4) and 5605 over the first half (1/2).
constexpr int64_t kMixA = 1, kMixB = 1;
__device__ __forceinline__ int64_t plan_block_scan(int64_t v, int64_t* warp_sums, int64_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int64_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t y = __shfl_up_sync(kFullMask, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int64_t w = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(kFullMask, w, o);
      if (lane >= o) w += y;
    }
    warp_sums[lane] = w;
  }
  __syncthreads();
  const int64_t r = incl - v + (warp > 0 ? warp_sums[warp - 1] : 0);
  *total = warp_sums[31];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kPlanThreadsP, 1) prefill_plan_kernel(
    const int32_t* cu_q, const int32_t* cu_k, int32_t num_seqs, int32_t pos_per_tile,
    int32_t num_kv_heads, int32_t* item_prefix, int32_t* item_perm, int32_t* item_counter,
    int* flags) {
  allow_dependent_launch();
  __shared__ int64_t warp_sums[32];
  const int tid = threadIdx.x;
  const int per = (num_seqs + kPlanThreadsP - 1) / kPlanThreadsP;
  const int b0 = min(num_seqs, tid * per), b1 = min(num_seqs, b0 + per);
  // items of sequence b; *heavy: its query tiles are at least half full
  auto items_of = [&](int b, bool* heavy) -> int32_t {
    const int q_len = __ldg(cu_q + b + 1) - __ldg(cu_q + b);
    const int k_len = __ldg(cu_k + b + 1) - __ldg(cu_k + b);
    *heavy = false;
    if (q_len < 0 || k_len < q_len) {
      raise_flag(flags, PKV_DEVERR_BAD_LENGTHS);
      return 0;
    }
    *heavy = 2 * q_len >= pos_per_tile;
    return ((q_len + pos_per_tile - 1) / pos_per_tile) * num_kv_heads;
  };
  // one scan for both: items in the low 40 bits, heavy sequences above them (batches of 2^22
  // sequences or more keep the batch order, so that the count fits)
  const bool may_mix = num_seqs < (1 << 22);
  int64_t mine = 0;
  for (int b = b0; b < b1; ++b) {
    bool h;
    const int32_t n = items_of(b, &h);
    mine += (int64_t)n + (h && may_mix ? (int64_t)1 << 40 : 0);
  }
  int64_t both = 0;
  const int64_t before = plan_block_scan(mine, warp_sums, &both);
  const int64_t H = both >> 40;
  const int64_t L = num_seqs - H;
  const bool mix = H > 0 && L > 0;
  auto clamp32 = [](int64_t v) { return (int32_t)(v < 0x7fffffff ? v : 0x7fffffff); };
  if (!mix) {
    // one kind only: positions are the batch order, and the scan above numbers the items
    int64_t at = before & (((int64_t)1 << 40) - 1);
    for (int b = b0; b < b1; ++b) {
      bool h;
      item_prefix[b] = clamp32(at);
      at += items_of(b, &h);
    }
    if (tid == 0) {
      const int64_t total = both & (((int64_t)1 << 40) - 1);
      item_prefix[num_seqs] = clamp32(total);
      if (total > 0x7fffffff) raise_flag(flags, PKV_DEVERR_BAD_LENGTHS);
      item_counter[0] = 0;
      item_counter[1] = (int32_t)H;
    }
    return;
  }
  int64_t i = before >> 40;  // heavy rank of my first heavy one
  int64_t j = b0 - i;        // light rank of my first light one
  // positions: heavy i goes after the light j with (2j + 1) H < (2i + 1) L; light j after the
  // heavy i with (2i + 1) L <= (2j + 1) H. Item counts go to item_prefix for the scan below.
  for (int b = b0; b < b1; ++b) {
    bool h;
    const int32_t n = items_of(b, &h);
    int64_t pos;
    if (h) {  // light ones before it: ceil(num / 2BH)
      const int64_t num = kMixA * (2 * i + 1) * L - kMixB * H;
      pos = i + (num <= 0 ? 0 : min(L, (num + 2 * kMixB * H - 1) / (2 * kMixB * H)));
      ++i;
    } else {  // heavy ones before it: floor(num / 2AL) + 1
      const int64_t num = kMixB * (2 * j + 1) * H - kMixA * L;
      pos = j + (num < 0 ? 0 : min(H, num / (2 * kMixA * L) + 1));
      ++j;
    }
    item_perm[pos] = b;
    item_prefix[pos] = n;
  }
  __syncthreads();  // every position's count is written (and visible to the CTA)
  // first item id of each position: an exclusive scan of the counts in position order
  int64_t local = 0;
  for (int pos = b0; pos < b1; ++pos) local += item_prefix[pos];
  int64_t total = 0;
  int64_t at = plan_block_scan(local, warp_sums, &total);
  for (int pos = b0; pos < b1; ++pos) {
    const int32_t n = item_prefix[pos];
    item_prefix[pos] = clamp32(at);
    at += n;
  }
  if (tid == 0) {
    item_prefix[num_seqs] = clamp32(total);
    if (total > 0x7fffffff) raise_flag(flags, PKV_DEVERR_BAD_LENGTHS);
    item_counter[0] = 0;
    item_counter[1] = (int32_t)H;
  }
}

int prefill_positions_per_tile(int group) { return kRows / group; }

cudaError_t configure_prefill_kernel() {
  cudaError_t e = cudaFuncSetAttribute(paged_prefill_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(paged_prefill_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                              (int)cudaSharedmemCarveoutMaxShared);
}

int prefill_kv_box_rows(int block_size, bool paged) {
  return paged ? (block_size < kKeys ? block_size : kKeys) : kKeys;
}

cudaError_t launch_paged_prefill(const PrefillArgs& a, const CUtensorMap& tq,
                                 const CUtensorMap& tk, const CUtensorMap& tv, int num_sms,
                                 cudaStream_t stream) {
  const int G = a.num_q_heads / a.cache.num_kv_heads;
  PrefillParams p;
  p.cu_q = a.cu_seqlens_q;
  p.cu_k = a.cu_seqlens_k;
  p.block_tables = a.block_tables;
  p.out = a.out;
  p.flags = a.flags;
  p.max_blocks = a.max_blocks;
  p.num_seqs = a.num_seqs;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.cache.num_kv_heads;
  p.group = G;
  p.pos_per_tile = kRows / G;
  p.num_q_tiles = (a.max_seqlen_q + p.pos_per_tile - 1) / p.pos_per_tile;
  p.block_size = a.cache.block_size;
  p.num_blocks = a.cache.num_blocks;
  const bool paged = a.block_tables != nullptr;
  p.box_rows = prefill_kv_box_rows(a.cache.block_size, paged);
  p.oob_row = paged ? a.cache.num_blocks * a.cache.block_size : a.total_q;
  p.qk_scale_log2 = a.scale * 1.4426950408889634f;
  p.item_prefix = a.item_prefix;
  p.item_perm = a.item_prefix != nullptr ? a.item_prefix + a.num_seqs + 1 : nullptr;
  // upper bound of the item count (the exact count, with dense numbering, is on the device)
  const int64_t items = (int64_t)p.num_q_tiles * p.num_kv_heads * a.num_seqs;
  if (items <= 0) return cudaSuccess;
  if (items > 0x7fffffff) return cudaErrorInvalidConfiguration;
  p.num_items = (int32_t)items;
  p.item_counter = a.item_counter;
  // two CTAs fit on an SM (registers, shared memory, 2 x 256 TMEM columns)
  const int64_t slots = 2 * (int64_t)(num_sms > 0 ? num_sms : 148);
  const unsigned grid = (unsigned)(items < slots ? items : slots);
  if (a.item_prefix == nullptr) {
    cudaError_t e = cudaMemsetAsync(a.item_counter, 0, sizeof(int32_t), stream);
    if (e != cudaSuccess) return e;
    paged_prefill_kernel<<<grid, kThreadsP, kSmemBytes, stream>>>(tq, tk, tv, p);
    return cudaGetLastError();
  }
  prefill_plan_kernel<<<1, kPlanThreadsP, 0, stream>>>(a.cu_seqlens_q, a.cu_seqlens_k,
                                                       a.num_seqs, p.pos_per_tile,
                                                       p.num_kv_heads, a.item_prefix,
                                                       a.item_prefix + a.num_seqs + 1,
                                                       a.item_counter, a.flags);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // the attention grid is a programmatic dependent of the plan: scheduled while the plan runs,
  // it waits for it in-kernel
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreadsP);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, paged_prefill_kernel, tq, tk, tv, p);
}

}  // namespace pkv
