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
//  * Warp 0 loads Q once and streams 64-key K and V tiles through the block table with 3-D TMA
//    boxes in 128-byte swizzle (the layout the tensor core reads). K and V have their own
//    two-deep rings and barriers, and K runs one tile ahead of V: a K buffer is free as soon as
//    its S = Q K^T is done, so the next K is in flight while the softmax of the current tile runs.
//  * Warp 1 allocates 256 TMEM columns and, from one thread, issues S = Q K^T (M=128, N=64,
//    K=128: eight kind::f16 MMAs, K-major operands) into TMEM columns [0, 64) and O += P V
//    (M=128, N=128, K=64: four MMAs, V read MN-major) into columns [64, 192).
//  * Warps 2-5 (one TMEM lane quarter each, thread = query row) load S rows, apply the causal
//    mask and an online softmax in log2 units with a lazy rescale (O in TMEM is rescaled only when
//    a row's max grows by more than 2^8), write P as bf16 into shared memory in the swizzled
//    K-major layout, and finally normalise O and store it.
//  * The tensor core computes S for the next tile while the softmax warps work on the current
//    one. Every wait is bounded; the CTA always frees its TMEM.
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
constexpr float kTauP = 8.0f;

constexpr int kQBytes = kRows * kHD * 2;     // two 16 KB halves of 64 dims
constexpr int kQHalf = kRows * 128;          // 16 KB
constexpr int kKTile = kKeys * kHD * 2;      // 16 KB: two 8 KB halves
constexpr int kKHalf = kKeys * 128;          // 8 KB
constexpr int kStage = 2 * kKTile;           // K then V
constexpr int kNStage = 2;
constexpr int kPBytes = kRows * kKeys * 2;   // 16 KB
constexpr int kOffQ = 0;
constexpr int kOffKV = kOffQ + kQBytes;
constexpr int kOffP = kOffKV + kNStage * kStage;
constexpr int kOffBar = kOffP + kPBytes;
// barriers: q, k_full[2], k_empty[2], v_full[2], v_empty[2], s_full, s_free, p_full, o_done,
// mma_done
constexpr int kBarQ = 0, kBarFullK = 1, kBarEmptyK = 3, kBarFullV = 5, kBarEmptyV = 7,
              kBarSFull = 9, kBarSFree = 10, kBarPFull = 11, kBarODone = 12, kBarMma = 13,
              kNumBars = 14;
constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffTmemSlot + 16;
static_assert(kOffKV % 1024 == 0 && kOffP % 1024 == 0, "swizzle atoms need 1024-byte alignment");

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
  int32_t block_size;
  int32_t num_blocks;
  int32_t box_rows;      // rows per K/V TMA box
  int32_t oob_row;       // a row coordinate past the end of the K/V tensors (zero fill)
  float qk_scale_log2;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__global__ void __launch_bounds__(kThreadsP, 2)
    paged_prefill_kernel(const __grid_constant__ CUtensorMap tmap_q,
                         const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v, const PrefillParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- which (sequence, kv head, query tile): the query tiles of one (sequence, kv head) are
  // adjacent, longest first, so they run together and share that head's K/V through L2 ----
  const int id = blockIdx.x;
  const int qt = p.num_q_tiles - 1 - id % p.num_q_tiles;
  const int t = id / p.num_q_tiles;
  const int g = t % p.num_kv_heads;
  const int b = t / p.num_kv_heads;
  const int q_start = p.cu_q[b];
  const int q_len = p.cu_q[b + 1] - q_start;
  const int k_len = p.cu_k[b + 1] - p.cu_k[b];
  if (q_len < 0 || k_len < q_len) {
    if (threadIdx.x == 0 && qt == 0) raise_flag(p.flags, PKV_DEVERR_BAD_LENGTHS);
    return;
  }
  const int G = p.group;
  const int q0 = qt * p.pos_per_tile;
  if (q0 >= q_len) return;
  if ((smem_addr(smem) & 1023u) != 0) {  // the swizzled layouts need a 1024-byte aligned base
    if (threadIdx.x == 0) raise_flag(p.flags, PKV_DEVERR_INTERNAL);
    return;
  }
  const int P = k_len - q_len;  // cached prefix length
  const int last_pos = min(q_len, q0 + p.pos_per_tile) - 1;
  const int n_kt = (P + last_pos + 1 + kKeys - 1) / kKeys;

  const uint32_t sbase = smem_addr(smem);
  const uint32_t bar0 = sbase + kOffBar;
  auto bar = [bar0](int i) { return bar0 + 8u * (uint32_t)i; };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + kOffTmemSlot);

  if (threadIdx.x == 0) {
    mbar_init(bar(kBarQ), 1);
    for (int s = 0; s < kNStage; ++s) {
      mbar_init(bar(kBarFullK + s), 1);
      mbar_init(bar(kBarEmptyK + s), 1);
      mbar_init(bar(kBarFullV + s), 1);
      mbar_init(bar(kBarEmptyV + s), 1);
    }
    mbar_init(bar(kBarSFull), 1);
    mbar_init(bar(kBarSFree), 4);
    mbar_init(bar(kBarPFull), 4);
    mbar_init(bar(kBarODone), 1);
    mbar_init(bar(kBarMma), 1);
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

  if (warp == 0) {
    // =============================== producer ===============================
    bool ok = true;
    if (lane == 0) {
      tma_prefetch_desc(&tmap_q);
      tma_prefetch_desc(&tmap_k);
      tma_prefetch_desc(&tmap_v);
      mbar_arrive_expect_tx(bar(kBarQ), kQBytes);
      tma_load_3d(sbase + kOffQ, &tmap_q, 0, g * G, q_start + q0, bar(kBarQ));
      tma_load_3d(sbase + kOffQ + kQHalf, &tmap_q, 64, g * G, q_start + q0, bar(kBarQ));
    }
    const bool paged = p.block_tables != nullptr;
    const int bs = p.block_size;
    const int box = p.box_rows;
    const int nsub = kKeys / box;
    int need_ent = 0;
    const int32_t* bt_row = nullptr;
    if (paged) {
      need_ent = (k_len + bs - 1) / bs;
      if (need_ent > p.max_blocks) {
        if (lane == 0) raise_flag(p.flags, PKV_DEVERR_CTX_CLAMPED);
        need_ent = p.max_blocks;
      }
      bt_row = p.block_tables + (int64_t)b * p.max_blocks;
    }
    int win_base = -1000000, win_val = -1;
    int issued_k = 0, issued_v = 0;
    int prev_rows[kKeys / 16];
    // Issue order K0, K1, V0, K2, V1, ...: step j loads K(j) (if j < n_kt), then V(j-1).
    for (int j = 0; j <= n_kt && ok; ++j) {
      int rows[kKeys / 16];
#pragma unroll
      for (int sb = 0; sb < kKeys / 16; ++sb) rows[sb] = p.oob_row;
      const int key0 = j * kKeys;
      if (j < n_kt) {
        if (paged) {
          const int e0 = key0 / bs;
          const int ent = (kKeys + bs - 1) / bs;
          if (e0 < win_base || e0 + ent > win_base + 32) {
            win_base = e0;
            const int e = e0 + lane;
            win_val = e < need_ent ? __ldg(bt_row + e) : -1;
          }
#pragma unroll
          for (int sb = 0; sb < kKeys / 16; ++sb) {
            if (sb < nsub) {
              const int key = key0 + sb * box;
              const int blk = __shfl_sync(kFullMask, win_val, (key / bs - win_base) & 31);
              if (key < k_len && key / bs < need_ent) {
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
            if (sb < nsub) rows[sb] = q_start + key0 + sb * box;
        }
      }
      if (lane == 0) {
        if (j < n_kt) {
          const int st = j & 1;
          ok = mbar_wait(bar(kBarEmptyK + st), ((j >> 1) & 1) ^ 1);
          if (ok) {
            const uint32_t full = bar(kBarFullK + st);
            mbar_arrive_expect_tx(full, kKTile);
            const uint32_t kd = sbase + kOffKV + st * kStage;
#pragma unroll
            for (int sb = 0; sb < kKeys / 16; ++sb) {
              if (sb < nsub) {
                const uint32_t off = (uint32_t)(sb * box * 128);
                tma_load_3d(kd + off, &tmap_k, 0, g, rows[sb], full);
                tma_load_3d(kd + kKHalf + off, &tmap_k, 64, g, rows[sb], full);
              }
            }
            ++issued_k;
          }
        }
        if (ok && j > 0) {
          const int jv = j - 1, st = jv & 1;
          ok = mbar_wait(bar(kBarEmptyV + st), ((jv >> 1) & 1) ^ 1);
          if (ok) {
            const uint32_t full = bar(kBarFullV + st);
            mbar_arrive_expect_tx(full, kKTile);
            const uint32_t vd = sbase + kOffKV + st * kStage + kKTile;
#pragma unroll
            for (int sb = 0; sb < kKeys / 16; ++sb) {
              if (sb < nsub) {
                const uint32_t off = (uint32_t)(sb * box * 128);
                tma_load_3d(vd + off, &tmap_v, 0, g, prev_rows[sb], full);
                tma_load_3d(vd + kKHalf + off, &tmap_v, 64, g, prev_rows[sb], full);
              }
            }
            ++issued_v;
          }
        }
        if (!ok) raise_flag(p.flags, PKV_DEVERR_TIMEOUT);
      }
#pragma unroll
      for (int sb = 0; sb < kKeys / 16; ++sb) prev_rows[sb] = rows[sb];
      ok = __shfl_sync(kFullMask, ok ? 1 : 0, 0) != 0;
    }
    if (lane == 0) {
      // never leave while a copy into this CTA's shared memory may be in flight
      if (!mbar_wait(bar(kBarQ), 0)) raise_flag(p.flags, PKV_DEVERR_TIMEOUT);
      bool drained = true;
      for (int i = (issued_k > kNStage ? issued_k - kNStage : 0); i < issued_k && drained; ++i)
        drained = mbar_wait(bar(kBarFullK + (i & 1)), (i >> 1) & 1);
      for (int i = (issued_v > kNStage ? issued_v - kNStage : 0); i < issued_v && drained; ++i)
        drained = mbar_wait(bar(kBarFullV + (i & 1)), (i >> 1) & 1);
      if (!drained) raise_flag(p.flags, PKV_DEVERR_TIMEOUT);
    }
  } else if (warp == 1) {
    // ============================ MMA issuer (one thread) ============================
    if (lane == 0) {
      const uint32_t idesc_s = idesc_bf16_f32(kRows, kKeys, false);
      const uint32_t idesc_o = idesc_bf16_f32(kRows, kHD, true);
      bool ok = mbar_wait(bar(kBarQ), 0);
      auto issue_pv = [&](int jj) {
        if (!ok) return;
        ok = mbar_wait(bar(kBarFullV + (jj & 1)), (jj >> 1) & 1);
        if (ok) ok = mbar_wait(bar(kBarPFull), jj & 1);
        if (!ok) return;
        tc_fence_after_sync();
        const uint32_t vbase = sbase + kOffKV + (jj & 1) * kStage + kKTile;
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk) {
          const uint64_t a = sdesc_kmajor_sw128(sbase + kOffP + kk * 32);
          const uint64_t bdesc = sdesc_mnmajor_sw128(vbase + kk * 16 * 128, kKHalf);
          tc_mma_f16(tmem + kColO, a, bdesc, idesc_o, (jj > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(bar(kBarODone));
        tc_commit(bar(kBarEmptyV + (jj & 1)));
      };
      for (int j = 0; j < n_kt && ok; ++j) {
        const int st = j & 1;
        ok = mbar_wait(bar(kBarFullK + st), (j >> 1) & 1);
        if (ok && j > 0) ok = mbar_wait(bar(kBarSFree), (j - 1) & 1);
        if (!ok) break;
        tc_fence_after_sync();
        const uint32_t kbase = sbase + kOffKV + st * kStage;
#pragma unroll
        for (int kk = 0; kk < kHD / 16; ++kk) {
          const uint32_t off = (uint32_t)((kk & 3) * 32);
          const uint64_t a = sdesc_kmajor_sw128(sbase + kOffQ + (kk >> 2) * kQHalf + off);
          const uint64_t bdesc = sdesc_kmajor_sw128(kbase + (kk >> 2) * kKHalf + off);
          tc_mma_f16(tmem + kColS, a, bdesc, idesc_s, kk > 0 ? 1u : 0u);
        }
        tc_commit(bar(kBarSFull));
        tc_commit(bar(kBarEmptyK + st));
        if (j > 0) issue_pv(j - 1);
      }
      if (ok) issue_pv(n_kt - 1);
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
    const int pos = q0 + r / G;
    const bool row_valid = pos < q_len;
    const int limit = P + pos;  // last key this row may see
    const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
    uint8_t* pbuf = smem + kOffP;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kt; ++j) {
      ok = mbar_wait(bar(kBarSFull), j & 1);
      if (!ok) break;
      tc_fence_after_sync();
      uint32_t sr[64];
      tmem_ld64(trow + kColS, sr);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarSFree));

      const int kbase = j * kKeys;
      // Tiles below every row's causal limit and inside k_len need no mask (CTA-uniform test);
      // there, with a positive scale, max and exp take the raw scores: p = 2^(s*c - m).
      // Max and sum use eight partial accumulators to keep dependency chains short.
      const bool full = kbase + kKeys - 1 <= P + q0 && kbase + kKeys <= k_len &&
                        p.qk_scale_log2 > 0.f;
      float part[8];
      if (full) {
#pragma unroll
        for (int u = 0; u < 8; ++u) part[u] = __uint_as_float(sr[u]);
#pragma unroll
        for (int c = 8; c < 64; ++c) part[c & 7] = fmaxf(part[c & 7], __uint_as_float(sr[c]));
      } else {
#pragma unroll
        for (int u = 0; u < 8; ++u) part[u] = -INFINITY;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const int key = kbase + c;
          const float s = (key <= limit && key < k_len)
                              ? __uint_as_float(sr[c]) * p.qk_scale_log2
                              : -INFINITY;
          sr[c] = __float_as_uint(s);
          part[c & 7] = fmaxf(part[c & 7], s);
        }
      }
      float mt = fmaxf(fmaxf(fmaxf(part[0], part[1]), fmaxf(part[2], part[3])),
                       fmaxf(fmaxf(part[4], part[5]), fmaxf(part[6], part[7])));
      if (full) mt *= p.qk_scale_log2;
      const bool resc = mt > m_run + kTauP;
      float alpha = 1.f;
      if (resc) {
        alpha = fast_exp2(m_run - mt);  // 0 when nothing was seen yet
        m_run = mt;
      }
      uint32_t pk[32];
#pragma unroll
      for (int u = 0; u < 8; ++u) part[u] = 0.f;
      if (full) {
        const float c2 = p.qk_scale_log2, nm = -m_run;
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          const float p0 = fast_exp2(fmaf(__uint_as_float(sr[c]), c2, nm));
          const float p1 = fast_exp2(fmaf(__uint_as_float(sr[c + 1]), c2, nm));
          part[(c >> 1) & 7] += p0 + p1;
          pk[c / 2] = pack_bf16x2(p0, p1);
        }
      } else {
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          const float s0 = __uint_as_float(sr[c]), s1 = __uint_as_float(sr[c + 1]);
          const float p0 = s0 == -INFINITY ? 0.f : fast_exp2(s0 - m_run);
          const float p1 = s1 == -INFINITY ? 0.f : fast_exp2(s1 - m_run);
          part[(c >> 1) & 7] += p0 + p1;
          pk[c / 2] = pack_bf16x2(p0, p1);
        }
      }
      const float sum = ((part[0] + part[1]) + (part[2] + part[3])) +
                        ((part[4] + part[5]) + (part[6] + part[7]));
      l_run = l_run * alpha + sum;

      if (j > 0) {  // the previous P V is done: P buffer free, O stable
        ok = mbar_wait(bar(kBarODone), (j - 1) & 1);
        if (!ok) break;
        tc_fence_after_sync();
      }
      // P row r, K-major with 128-byte swizzle: 16-byte chunk c lands at chunk c ^ (r % 8)
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint4 v = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        *reinterpret_cast<uint4*>(pbuf + r * 128 + ((c ^ (r & 7)) << 4)) = v;
      }
      if (j > 0 && __any_sync(kFullMask, resc)) {
#pragma unroll 1
        for (int cc = 0; cc < kHD / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32(trow + kColO + cc * 32, o);
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
          tmem_st32(trow + kColO + cc * 32, o);
        }
        tmem_st_wait();
      }
      if (j == n_kt - 1 && kbase + kKeys > k_len) {
        // V rows past the last key hold whatever the cache holds there: zero them (after the
        // stage's copy has landed)
        ok = mbar_wait(bar(kBarFullV + (j & 1)), (j >> 1) & 1);
        if (!ok) break;
        const int first = k_len - kbase;
        uint8_t* vt = smem + kOffKV + (j & 1) * kStage + kKTile;
        const int nrow = kKeys - first;
        for (int i = threadIdx.x - 64; i < nrow * 16; i += 128) {
          const int row = first + i / 16, part = i % 16;  // 16 x 16 bytes = both halves
          *reinterpret_cast<uint4*>(vt + (part >> 3) * kKHalf + row * 128 + (part & 7) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
      }
      fence_async_shared();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarPFull));
    }
    if (ok) ok = mbar_wait(bar(kBarODone), (n_kt - 1) & 1);
    if (ok) {
      tc_fence_after_sync();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      uint16_t* orow = p.out + ((int64_t)(q_start + pos) * p.num_q_heads + g * G + r % G) * kHD;
#pragma unroll 1
      for (int cc = 0; cc < kHD / 64; ++cc) {
        uint32_t o[64];
        tmem_ld64(trow + kColO + cc * 64, o);
        uint32_t w[32];
#pragma unroll
        for (int c = 0; c < 32; ++c)
          w[c] = pack_bf16x2(__uint_as_float(o[2 * c]) * inv, __uint_as_float(o[2 * c + 1]) * inv);
        if (row_valid) {
          uint4* dst = reinterpret_cast<uint4*>(orow + cc * 64);
#pragma unroll
          for (int c = 0; c < 8; ++c)
            dst[c] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
        }
      }
    } else if (lane == 0) {
      raise_flag(p.flags, PKV_DEVERR_TIMEOUT);
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

int prefill_positions_per_tile(int group) { return kRows / group; }

int prefill_kv_box_rows(int block_size, bool paged) {
  return paged ? (block_size < kKeys ? block_size : kKeys) : kKeys;
}

cudaError_t launch_paged_prefill(const PrefillArgs& a, const CUtensorMap& tq,
                                 const CUtensorMap& tk, const CUtensorMap& tv, int num_sms,
                                 cudaStream_t stream) {
  (void)num_sms;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(paged_prefill_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(paged_prefill_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    configured = true;
  }
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
  const int64_t grid = (int64_t)p.num_q_tiles * p.num_kv_heads * a.num_seqs;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffff) return cudaErrorInvalidConfiguration;
  paged_prefill_kernel<<<(unsigned)grid, kThreadsP, kSmemBytes, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace pkv
