// kv_store.cu -- scatter new K/V rows into the paged cache through slot_mapping.
//
// Source: "nano-vllm 深度分析报告", table "可复用的模式与技巧", row "slot_mapping -1 padding": the
// store kernel writes each token's K/V at its slot and skips positions padded with -1 for CUDA
// graphs; "DeepSeek研究员1200行代码复刻vLLM..." section "vLLM是什么？": the cache is made of
// fixed-size blocks.
//
// One token row (num_kv_heads * head_dim bf16, 2 KB at 8 x 128) is contiguous in both the source
// and the cache, so the copy is a gather of 16-byte vectors: each thread moves vector c of token t
// for K and for V. Source loads bypass L1 (read once); cache stores stay in L2 for the attention
// kernel that follows. Slots outside [0, num_slots) other than -1 are skipped and flagged.
#include "common.cuh"
#include "kernels.h"

namespace pkv {

namespace {

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

constexpr int kStoreThreads = 256;
constexpr int kStoreUnroll = 4;

__global__ void __launch_bounds__(kStoreThreads)
    kv_store_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                    const int32_t* __restrict__ slot_mapping, int64_t total_vecs,
                    int32_t row_vecs, int64_t num_slots, uint4* __restrict__ k_cache,
                    uint4* __restrict__ v_cache, int* flags) {
  // a programmatic dependent of the previous work: wait for it before any memory access
  allow_dependent_launch();
  grid_dependency_wait();
  const int64_t stride = (int64_t)gridDim.x * kStoreThreads;
  int64_t i = (int64_t)blockIdx.x * kStoreThreads + threadIdx.x;
  for (; i < total_vecs; i += stride * kStoreUnroll) {
    uint4 kv[kStoreUnroll], vv[kStoreUnroll];
    int64_t dst[kStoreUnroll];
#pragma unroll
    for (int u = 0; u < kStoreUnroll; ++u) {
      const int64_t idx = i + u * stride;
      dst[u] = -1;
      if (idx < total_vecs) {
        const int64_t t = idx / row_vecs;
        const int32_t c = (int32_t)(idx - t * row_vecs);
        const int64_t s = __ldg(slot_mapping + t);
        if (s >= 0 && s < num_slots) {
          dst[u] = s * row_vecs + c;
          kv[u] = ld_stream(k + idx);
          vv[u] = ld_stream(v + idx);
        } else if (s != -1 && c == 0) {
          raise_flag(flags, PKV_DEVERR_BAD_SLOT);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kStoreUnroll; ++u) {
      if (dst[u] >= 0) {
        k_cache[dst[u]] = kv[u];
        v_cache[dst[u]] = vv[u];
      }
    }
  }
}

}  // namespace

cudaError_t launch_kv_store(const uint16_t* k, const uint16_t* v, const int32_t* slot_mapping,
                            int32_t num_tokens, uint16_t* k_cache, uint16_t* v_cache,
                            const pkv_cache_desc& cache, int num_sms, int* flags,
                            cudaStream_t stream) {
  const int32_t row_vecs = cache.num_kv_heads * cache.head_dim * 2 / 16;
  const int64_t total = (int64_t)num_tokens * row_vecs;
  if (total == 0) return cudaSuccess;
  const int64_t per_block = (int64_t)kStoreThreads * kStoreUnroll;
  int64_t blocks = (total + per_block - 1) / per_block;
  const int64_t cap = (int64_t)num_sms * 8;
  if (blocks > cap) blocks = cap;
  return launch_dependent(kv_store_kernel, dim3((unsigned)blocks), dim3(kStoreThreads), 0, stream,
                          reinterpret_cast<const uint4*>(k), reinterpret_cast<const uint4*>(v),
                          slot_mapping, total, row_vecs,
                          (int64_t)cache.num_blocks * cache.block_size,
                          reinterpret_cast<uint4*>(k_cache), reinterpret_cast<uint4*>(v_cache),
                          flags);
}

}  // namespace pkv
