// block_hash.cu -- chained xxhash64 of full token blocks, for prefix-cache lookup.
//
// Source: "nano-vllm 深度分析报告", section "创新之处" and table "可复用的模式与技巧": prefix
// caching content-addresses each full block with an xxhash64 that includes the hash of the
// blocks before it, so equal hashes identify equal prefixes (position included).
//
// Byte string of block i of a sequence: [8-byte little-endian hash of block i-1, omitted for
// block 0] ++ [block_size token ids, 4-byte little-endian]. Hash: XXH64 with seed 0, as the
// xxHash specification defines it. With an even block size the string is a whole number of
// 8-byte lanes: lane 0 is the parent hash (when present) and every other lane packs two
// consecutive token ids (low id in the low 32 bits). The kernel builds those lanes from the block's
// tokens staged in shared memory (no byte buffer): 4-lane stripes through the accumulators,
// leftover lanes through the 8-byte tail step, then the avalanche.
//
// The chain is sequential within a sequence; sequences are independent, one warp each.
#include "common.cuh"
#include "kernels.h"

namespace pkv {

namespace {

constexpr uint64_t kP1 = 0x9E3779B185EBCA87ull;
constexpr uint64_t kP2 = 0xC2B2AE3D27D4EB4Full;
constexpr uint64_t kP3 = 0x165667B19E3779F9ull;
constexpr uint64_t kP4 = 0x85EBCA77C2B2AE63ull;
constexpr uint64_t kP5 = 0x27D4EB2F165667C5ull;

__device__ __forceinline__ uint64_t rotl(uint64_t x, int r) { return (x << r) | (x >> (64 - r)); }

__device__ __forceinline__ uint64_t lane_round(uint64_t acc, uint64_t lane) {
  return rotl(acc + lane * kP2, 31) * kP1;
}

constexpr int kWarpsPerCta = 4;
constexpr int kMaxBlockSize = 256;

// The i-th 8-byte lane of the block's byte string, tokens taken from shared memory.
__device__ __forceinline__ uint64_t lane_at(const int32_t* tok, bool has_parent, uint64_t parent,
                                            int i) {
  if (has_parent) {
    if (i == 0) return parent;
    i -= 1;
  }
  return (uint64_t)(uint32_t)tok[2 * i] | ((uint64_t)(uint32_t)tok[2 * i + 1] << 32);
}

// One warp per sequence. Each block's tokens are loaded into shared memory by the whole warp
// (coalesced); lanes 0-3 each run one of the four XXH64 accumulators over the 32-byte stripes,
// and lane 0 merges them, runs the 8-byte tail steps and the avalanche. The result is the parent
// of the next block.
__global__ void __launch_bounds__(kWarpsPerCta * 32)
    block_hash_kernel(const int32_t* __restrict__ token_ids, const int32_t* __restrict__ cu,
                      int32_t num_seqs, int32_t block_size, int32_t max_blocks,
                      uint64_t* __restrict__ out, int* flags) {
  __shared__ int32_t stage[kWarpsPerCta][kMaxBlockSize];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x * kWarpsPerCta + warp;
  if (b >= num_seqs) return;
  int32_t* tok = stage[warp];
  const int32_t start = cu[b];
  const int32_t len = cu[b + 1] - start;
  int32_t nfull = len > 0 ? len / block_size : 0;
  if (nfull > max_blocks) {
    if (lane == 0) raise_flag(flags, PKV_DEVERR_CTX_CLAMPED);
    nfull = max_blocks;
  }
  uint64_t* row = out + (int64_t)b * max_blocks;
  uint64_t parent = 0;
  for (int i = 0; i < nfull; ++i) {
    const int32_t* src = token_ids + start + (int64_t)i * block_size;
    __syncwarp();
    for (int t = lane; t < block_size; t += 32) tok[t] = __ldg(src + t);
    __syncwarp();
    const bool has_parent = i > 0;
    const int lanes = block_size / 2 + (has_parent ? 1 : 0);
    const int stripes = lanes / 4;
    uint64_t v = 0;
    if (lane < 4 && stripes > 0) {
      v = lane == 0 ? kP1 + kP2 : lane == 1 ? kP2 : lane == 2 ? 0ull : 0ull - kP1;  // seed 0
      for (int s = 0; s < stripes; ++s)
        v = lane_round(v, lane_at(tok, has_parent, parent, 4 * s + lane));
    }
    const uint64_t v1 = __shfl_sync(kFullMask, v, 0), v2 = __shfl_sync(kFullMask, v, 1);
    const uint64_t v3 = __shfl_sync(kFullMask, v, 2), v4 = __shfl_sync(kFullMask, v, 3);
    if (lane == 0) {
      uint64_t acc;
      if (stripes > 0) {
        acc = rotl(v1, 1) + rotl(v2, 7) + rotl(v3, 12) + rotl(v4, 18);
        acc = (acc ^ lane_round(0, v1)) * kP1 + kP4;
        acc = (acc ^ lane_round(0, v2)) * kP1 + kP4;
        acc = (acc ^ lane_round(0, v3)) * kP1 + kP4;
        acc = (acc ^ lane_round(0, v4)) * kP1 + kP4;
      } else {
        acc = kP5;
      }
      acc += (uint64_t)lanes * 8;
      for (int l = 4 * stripes; l < lanes; ++l) {
        acc ^= lane_round(0, lane_at(tok, has_parent, parent, l));
        acc = rotl(acc, 27) * kP1 + kP4;
      }
      acc ^= acc >> 33;
      acc *= kP2;
      acc ^= acc >> 29;
      acc *= kP3;
      acc ^= acc >> 32;
      parent = acc;
      row[i] = acc;
    }
    parent = __shfl_sync(kFullMask, parent, 0);
  }
  for (int i = nfull + lane; i < max_blocks; i += 32) row[i] = 0;  // no full block: no hash
}

}  // namespace

cudaError_t launch_block_hashes(const int32_t* token_ids, const int32_t* cu_seqlens,
                                int32_t num_seqs, int32_t block_size, int32_t max_blocks,
                                uint64_t* out, int* flags, cudaStream_t stream) {
  if (num_seqs == 0) return cudaSuccess;
  if (block_size > kMaxBlockSize) return cudaErrorNotSupported;
  block_hash_kernel<<<(num_seqs + kWarpsPerCta - 1) / kWarpsPerCta, kWarpsPerCta * 32, 0,
                      stream>>>(
      token_ids, cu_seqlens, num_seqs, block_size, max_blocks, out, flags);
  return cudaGetLastError();
}

}  // namespace pkv
