// block_ops.cu -- whole-block moves in the paged cache: copy-on-write copies and swap-style
// gather / scatter of blocks.
//
// Source: "nano-vllm 深度分析报告", section "解法哲学": Nano-vLLM keeps PagedAttention and prefix
// caching but drops swap (CPU offload) and copy-on-write, which vLLM has. Both act on whole
// physical blocks: copy-on-write duplicates a shared block before one sequence writes into it;
// swapping moves a sequence's blocks out to a staging buffer and back into (other) free blocks.
//
// One physical block of one cache is block_size * num_kv_heads * head_dim bf16, contiguous. Each
// kernel moves 16-byte vectors with a grid-stride loop, reading once (L1 bypassed) and writing
// once; a block id outside [0, num_blocks) is skipped and flagged, never dereferenced.
#include "common.cuh"
#include "kernels.h"

namespace pkv {

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ uint4 ld_once(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// mode 0: cache[dst] = cache[src] for (src, dst) = (pairs[2i], pairs[2i+1])
// mode 1: out[i] = cache[ids[i]]   (gather, swap out)
// mode 2: cache[ids[i]] = in[i]    (scatter, swap in)
__global__ void __launch_bounds__(kThreads)
    block_move_kernel(int mode, uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                      const int32_t* __restrict__ ids, int32_t n, int64_t block_vecs,
                      int32_t num_blocks, uint4* __restrict__ buf_k, uint4* __restrict__ buf_v,
                      int* flags) {
  const int64_t total = (int64_t)n * block_vecs;
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  for (int64_t idx = (int64_t)blockIdx.x * kThreads + threadIdx.x; idx < total; idx += stride) {
    const int64_t i = idx / block_vecs;
    const int64_t c = idx - i * block_vecs;
    if (mode == 0) {
      const int32_t src = __ldg(ids + 2 * i), dst = __ldg(ids + 2 * i + 1);
      if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (c == 0) raise_flag(flags, PKV_DEVERR_BAD_BLOCK);
        continue;
      }
      k_cache[dst * block_vecs + c] = ld_once(k_cache + src * block_vecs + c);
      v_cache[dst * block_vecs + c] = ld_once(v_cache + src * block_vecs + c);
    } else {
      const int32_t blk = __ldg(ids + i);
      if (blk < 0 || blk >= num_blocks) {
        if (c == 0) raise_flag(flags, PKV_DEVERR_BAD_BLOCK);
        continue;
      }
      if (mode == 1) {
        buf_k[idx] = ld_once(k_cache + blk * block_vecs + c);
        buf_v[idx] = ld_once(v_cache + blk * block_vecs + c);
      } else {
        k_cache[blk * block_vecs + c] = ld_once(buf_k + idx);
        v_cache[blk * block_vecs + c] = ld_once(buf_v + idx);
      }
    }
  }
}

}  // namespace

cudaError_t launch_block_move(int mode, uint16_t* k_cache, uint16_t* v_cache,
                              const int32_t* ids, int32_t n, const pkv_cache_desc& cache,
                              uint16_t* buf_k, uint16_t* buf_v, int num_sms, int* flags,
                              cudaStream_t stream) {
  const int64_t block_vecs =
      (int64_t)cache.block_size * cache.num_kv_heads * cache.head_dim * 2 / 16;
  const int64_t total = (int64_t)n * block_vecs;
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + kThreads - 1) / kThreads;
  const int64_t cap = (int64_t)num_sms * 8;
  if (blocks > cap) blocks = cap;
  block_move_kernel<<<(unsigned)blocks, kThreads, 0, stream>>>(
      mode, reinterpret_cast<uint4*>(k_cache), reinterpret_cast<uint4*>(v_cache), ids, n,
      block_vecs, cache.num_blocks, reinterpret_cast<uint4*>(buf_k),
      reinterpret_cast<uint4*>(buf_v), flags);
  return cudaGetLastError();
}

}  // namespace pkv
