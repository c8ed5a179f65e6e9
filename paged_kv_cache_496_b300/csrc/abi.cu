// abi.cu -- the extern "C" entry points of libpagedkv.so (declared in include/pagedkv.h).
//
// Host-side argument validation, TMA descriptor encoding, the per-context library state (device
// error word, kernel attributes) and status strings. Every entry point only enqueues work on the caller's stream; nothing here allocates
// device memory.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>
#include <vector>

#include "common.cuh"
#include "kernels.h"

namespace pkv {
namespace {

thread_local char g_last_error[512] = "";

int fail(int status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return status;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(PKV_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// Device error word: one copy per CUDA context (a __device__ variable exists once per loaded
// module, and each context loads its own).
__device__ int g_device_flags = 0;

// Driver entry points, fetched through the runtime (no link to libcuda).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

struct DriverFns {
  EncodeTiledFn encode = nullptr;
  CtxGetCurrentFn ctx_get_current = nullptr;
  CtxGetIdFn ctx_get_id = nullptr;
  cudaError_t err = cudaSuccess;
};

const DriverFns& driver_fns() {
  static std::once_flag once;
  static DriverFns fns;
  std::call_once(once, [] {
    auto get = [](const char* name) -> void* {
      void* f = nullptr;
      cudaDriverEntryPointQueryResult q;
      const cudaError_t e = cudaGetDriverEntryPointByVersion(name, &f, 12000, cudaEnableDefault, &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess) {
        if (fns.err == cudaSuccess) fns.err = e != cudaSuccess ? e : cudaErrorSymbolNotFound;
        return nullptr;
      }
      return f;
    };
    fns.encode = reinterpret_cast<EncodeTiledFn>(get("cuTensorMapEncodeTiled"));
    fns.ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(get("cuCtxGetCurrent"));
    fns.ctx_get_id = reinterpret_cast<CtxGetIdFn>(get("cuCtxGetId"));
  });
  return fns;
}

int get_encoder(EncodeTiledFn* fn) {
  const DriverFns& f = driver_fns();
  if (f.encode == nullptr)
    return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled unavailable (%s)", cudaGetErrorName(f.err));
  *fn = f.encode;
  return PKV_OK;
}

// One entry per context this process has used; entries are never freed (there are only a few).
std::mutex g_context_mutex;
std::vector<ContextState*> g_contexts;

}  // namespace

int report_cuda_error(cudaError_t e, const char* what) { return cuda_fail(e, what); }

int current_context_id(unsigned long long* id, int* device) {
  const DriverFns& f = driver_fns();
  if (f.ctx_get_current == nullptr || f.ctx_get_id == nullptr)
    return fail(PKV_ERR_CUDA, "cuCtxGetCurrent / cuCtxGetId unavailable (%s)",
                cudaGetErrorName(f.err));
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  CUcontext c = nullptr;
  if (f.ctx_get_current(&c) != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "cuCtxGetCurrent failed");
  if (c == nullptr) {
    // nothing bound to this thread yet: cudaSetDevice initialises and binds the primary context
    e = cudaSetDevice(dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
    if (f.ctx_get_current(&c) != CUDA_SUCCESS || c == nullptr)
      return fail(PKV_ERR_CUDA, "no CUDA context is current");
  }
  unsigned long long v = 0;
  if (f.ctx_get_id(c, &v) != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "cuCtxGetId failed");
  *id = v;
  if (device != nullptr) *device = dev;
  return PKV_OK;
}

int context_state(const ContextState** out) {
  unsigned long long id = 0;
  int dev = 0;
  int st = current_context_id(&id, &dev);
  if (st != PKV_OK) return st;
  std::lock_guard<std::mutex> lock(g_context_mutex);
  for (const ContextState* s : g_contexts)
    if (s->ctx_id == id) {
      *out = s;
      return PKV_OK;
    }
  ContextState s;
  s.ctx_id = id;
  s.device = dev;
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_device_flags);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(device error word)");
  s.flags = static_cast<int*>(p);
  e = cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
  e = configure_prefill_kernel();
  if (e != cudaSuccess) return cuda_fail(e, "prefill kernel attributes");
  e = configure_decode_kernels(s.decode_ctas);
  if (e != cudaSuccess) return cuda_fail(e, "decode kernel attributes");
  e = configure_decode_tc_kernels();
  if (e != cudaSuccess) return cuda_fail(e, "tensor-core decode kernel attributes");
  g_contexts.push_back(new ContextState(s));
  *out = g_contexts.back();
  return PKV_OK;
}

namespace {

// 3-D view {D, heads, rows} of a row-major [rows, heads, D] bf16 tensor;
// box {box_d, box_heads, box_rows}.
int encode_rows_map(CUtensorMap* map, const void* base, int64_t rows, int heads, int head_dim,
                    int box_d, int box_rows, CUtensorMapSwizzle swizzle, int box_heads = 1) {
  EncodeTiledFn enc;
  int st = get_encoder(&enc);
  if (st != PKV_OK) return st;
  const cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)heads, (cuuint64_t)rows};
  const cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, (cuuint64_t)heads * head_dim * 2};
  const cuuint32_t box[3] = {(cuuint32_t)box_d, (cuuint32_t)box_heads, (cuuint32_t)box_rows};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return PKV_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

int check_cache(const pkv_cache_desc& c) {
  if (c.num_blocks <= 0 || c.block_size <= 0 || c.num_kv_heads <= 0 || c.head_dim <= 0)
    return fail(PKV_ERR_INVALID_ARG, "cache geometry must be positive");
  if (c.head_dim != 64 && c.head_dim != 128)
    return fail(PKV_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", c.head_dim);
  if (!is_pow2(c.block_size) || c.block_size < 16 || c.block_size > 256)
    return fail(PKV_ERR_UNSUPPORTED, "block_size %d (supported: powers of two 16..256)",
                c.block_size);
  if ((int64_t)c.num_blocks * c.block_size >= ((int64_t)1 << 31))
    return fail(PKV_ERR_UNSUPPORTED, "num_blocks * block_size must be below 2^31");
  return PKV_OK;
}

int check_heads(int num_q_heads, int num_kv_heads) {
  if (num_q_heads <= 0 || num_q_heads % num_kv_heads != 0)
    return fail(PKV_ERR_INVALID_ARG, "num_q_heads %d not a multiple of num_kv_heads %d",
                num_q_heads, num_kv_heads);
  const int G = num_q_heads / num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8)
    return fail(PKV_ERR_UNSUPPORTED, "group size %d (supported: 1, 2, 4, 8)", G);
  return PKV_OK;
}

constexpr int32_t kAutoSplitFloor = 512;

// One CTA waits on an mbarrier that nothing ever completes, with the same bounded wait the
// kernels' pipelines use; the wait gives up after its time limit and reports a timeout.
__global__ void bounded_wait_selftest_kernel(int* flags) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(smem_addr(&bar), 0)) raise_flag(flags, PKV_DEVERR_TIMEOUT);
}

int32_t round_up(int64_t x, int64_t q) { return (int32_t)((x + q - 1) / q * q); }

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" {

int pkv_version(void) { return PKV_VERSION; }

const char* pkv_last_error(void) { return g_last_error; }

const char* pkv_status_string(int status) {
  switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported shape";
    case PKV_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case PKV_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

int pkv_get_device_error(int32_t* flags) {
  if (flags == nullptr) return fail(PKV_ERR_INVALID_ARG, "flags is NULL");
  const ContextState* d = nullptr;
  int st = context_state(&d);
  if (st != PKV_OK) return st;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  int v = 0;
  e = cudaMemcpy(&v, d->flags, sizeof v, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read device error word");
  const int zero = 0;
  e = cudaMemcpy(d->flags, &zero, sizeof zero, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "clear device error word");
  *flags = v;
  return PKV_OK;
}

int pkv_selftest_bounded_wait(void* stream) {
  g_last_error[0] = 0;
  const ContextState* d = nullptr;
  int st = context_state(&d);
  if (st != PKV_OK) return st;
  bounded_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(d->flags);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "selftest launch");
  return PKV_OK;
}

int pkv_kv_store(const uint16_t* k, const uint16_t* v, const int32_t* slot_mapping,
                 int32_t num_tokens, uint16_t* k_cache, uint16_t* v_cache, pkv_cache_desc cache,
                 void* stream) {
  g_last_error[0] = 0;
  int st = check_cache(cache);
  if (st != PKV_OK) return st;
  if (num_tokens < 0) return fail(PKV_ERR_INVALID_ARG, "num_tokens %d < 0", num_tokens);
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache)
    return fail(PKV_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(PKV_ERR_INVALID_ARG, "k, v, k_cache and v_cache must be 16-byte aligned");
  const ContextState* d = nullptr;
  st = context_state(&d);
  if (st != PKV_OK) return st;
  cudaError_t e = launch_kv_store(k, v, slot_mapping, num_tokens, k_cache, v_cache, cache,
                                  d->num_sms, d->flags, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kv_store launch");
  return PKV_OK;
}

int block_move(int mode, uint16_t* k_cache, uint16_t* v_cache, const pkv_cache_desc& cache,
               const int32_t* ids, int32_t n, uint16_t* buf_k, uint16_t* buf_v, void* stream) {
  g_last_error[0] = 0;
  int st = check_cache(cache);
  if (st != PKV_OK) return st;
  if (n < 0) return fail(PKV_ERR_INVALID_ARG, "n %d < 0", n);
  if (n == 0) return PKV_OK;
  if (!k_cache || !v_cache || !ids || (mode != 0 && (!buf_k || !buf_v)))
    return fail(PKV_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(k_cache) || !aligned16(v_cache) ||
      (mode != 0 && (!aligned16(buf_k) || !aligned16(buf_v))))
    return fail(PKV_ERR_INVALID_ARG, "caches and buffers must be 16-byte aligned");
  const ContextState* d = nullptr;
  st = context_state(&d);
  if (st != PKV_OK) return st;
  cudaError_t e = launch_block_move(mode, k_cache, v_cache, ids, n, cache, buf_k, buf_v,
                                    d->num_sms, d->flags, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "block move launch");
  return PKV_OK;
}

int pkv_copy_blocks(uint16_t* k_cache, uint16_t* v_cache, pkv_cache_desc cache,
                    const int32_t* pairs, int32_t n, void* stream) {
  return block_move(0, k_cache, v_cache, cache, pairs, n, nullptr, nullptr, stream);
}

int pkv_gather_blocks(const uint16_t* k_cache, const uint16_t* v_cache, pkv_cache_desc cache,
                      const int32_t* ids, int32_t n, uint16_t* out_k, uint16_t* out_v,
                      void* stream) {
  return block_move(1, const_cast<uint16_t*>(k_cache), const_cast<uint16_t*>(v_cache), cache,
                    ids, n, out_k, out_v, stream);
}

int pkv_scatter_blocks(const uint16_t* in_k, const uint16_t* in_v, const int32_t* ids, int32_t n,
                       uint16_t* k_cache, uint16_t* v_cache, pkv_cache_desc cache,
                       void* stream) {
  return block_move(2, k_cache, v_cache, cache, ids, n, const_cast<uint16_t*>(in_k),
                    const_cast<uint16_t*>(in_v), stream);
}

int pkv_block_hashes(const int32_t* token_ids, const int32_t* cu_seqlens, int32_t num_seqs,
                     int32_t block_size, int32_t max_blocks, uint64_t* out, void* stream) {
  g_last_error[0] = 0;
  if (num_seqs < 0 || max_blocks < 0)
    return fail(PKV_ERR_INVALID_ARG, "num_seqs and max_blocks must be >= 0");
  if (block_size < 2 || (block_size & 1) || block_size > 256)
    return fail(PKV_ERR_UNSUPPORTED, "block_size %d (must be even, 2..256)", block_size);
  if (num_seqs == 0 || max_blocks == 0) return PKV_OK;
  if (!token_ids || !cu_seqlens || !out) return fail(PKV_ERR_INVALID_ARG, "null pointer");
  const ContextState* d = nullptr;
  int st = context_state(&d);
  if (st != PKV_OK) return st;
  cudaError_t e = launch_block_hashes(token_ids, cu_seqlens, num_seqs, block_size, max_blocks,
                                      out, d->flags, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "block hash launch");
  return PKV_OK;
}

int pkv_decode_plan_make(int32_t num_seqs, int32_t num_q_heads, pkv_cache_desc cache,
                         int32_t max_context_len, int32_t split_tokens_hint,
                         pkv_decode_plan* plan) {
  g_last_error[0] = 0;
  if (plan == nullptr) return fail(PKV_ERR_INVALID_ARG, "plan is NULL");
  int st = check_cache(cache);
  if (st != PKV_OK) return st;
  st = check_heads(num_q_heads, cache.num_kv_heads);
  if (st != PKV_OK) return st;
  if (num_seqs < 0 || max_context_len < 0)
    return fail(PKV_ERR_INVALID_ARG, "num_seqs and max_context_len must be >= 0");
  const int64_t ctx = max_context_len > 0 ? max_context_len : 1;
  pkv_decode_plan pl;
  memset(&pl, 0, sizeof pl);
  pl.max_context_len = max_context_len;
  if (split_tokens_hint < 0 || (split_tokens_hint == 0 && ctx <= kAutoSplitFloor)) {
    pl.split_tokens = round_up(ctx, kSplitQuantum);
    pl.max_splits = 1;
    pl.auto_split = 0;
  } else if (split_tokens_hint > 0) {
    pl.split_tokens = round_up(split_tokens_hint, kSplitQuantum);
    pl.max_splits = (int32_t)((ctx + pl.split_tokens - 1) / pl.split_tokens);
    pl.auto_split = 0;
  } else {
    pl.split_tokens = kAutoSplitFloor;
    pl.max_splits = (int32_t)((ctx + kAutoSplitFloor - 1) / kAutoSplitFloor);
    pl.auto_split = 1;
  }
  pl.workspace_bytes =
      decode_workspace_bytes(num_seqs, num_q_heads, cache.head_dim, pl.max_splits, nullptr,
                             nullptr);
  // The tensor-core engine where it is the faster one on a B300: head_dim 128, blocks of at least
  // 128 rows (one TMA box per block and 64-dim half stays large) and G >= 4 (the CUDA-core
  // kernel's arithmetic per byte grows with G and it becomes issue-bound).
  const int G = num_q_heads / cache.num_kv_heads;
  pl.engine = cache.head_dim == 128 && cache.block_size >= 128 && G >= 4
                  ? PKV_DECODE_ENGINE_TENSOR_CORE
                  : PKV_DECODE_ENGINE_CUDA_CORE;
  *plan = pl;
  return PKV_OK;
}

static int decode_impl(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                       pkv_cache_desc cache, const int32_t* block_tables,
                       int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t num_seqs,
                       int32_t num_q_heads, float scale, const pkv_decode_plan* plan,
                       uint16_t* out, void* workspace, size_t workspace_bytes, void* stream,
                       const uint16_t* k_new, const uint16_t* v_new,
                       const int32_t* slot_mapping) {
  g_last_error[0] = 0;
  int st = check_cache(cache);
  if (st != PKV_OK) return st;
  st = check_heads(num_q_heads, cache.num_kv_heads);
  if (st != PKV_OK) return st;
  if (num_seqs < 0) return fail(PKV_ERR_INVALID_ARG, "num_seqs %d < 0", num_seqs);
  if (num_seqs == 0) return PKV_OK;
  if (plan == nullptr) return fail(PKV_ERR_INVALID_ARG, "plan is NULL");
  if (plan->split_tokens <= 0 || plan->split_tokens % kSplitQuantum != 0 ||
      plan->max_splits <= 0)
    return fail(PKV_ERR_INVALID_ARG, "malformed decode plan");
  if (plan->engine != PKV_DECODE_ENGINE_CUDA_CORE && plan->engine != PKV_DECODE_ENGINE_TENSOR_CORE)
    return fail(PKV_ERR_INVALID_ARG, "decode plan engine %d", plan->engine);
  if ((plan->flags & ~PKV_DECODE_PLAN_REUSE) != 0)
    return fail(PKV_ERR_INVALID_ARG, "decode plan flags %#x", (unsigned)plan->flags);
  const int G = num_q_heads / cache.num_kv_heads;
  const bool tc = plan->engine == PKV_DECODE_ENGINE_TENSOR_CORE;
  if (tc && cache.head_dim != 128)
    return fail(PKV_ERR_UNSUPPORTED, "tensor-core decode needs head_dim 128 (got %d)",
                cache.head_dim);
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out || !workspace)
    return fail(PKV_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return fail(PKV_ERR_INVALID_ARG, "q, caches and out must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(PKV_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (max_blocks_per_seq <= 0)
    return fail(PKV_ERR_INVALID_ARG, "max_blocks_per_seq %d <= 0", max_blocks_per_seq);
  if (!(scale == scale) || scale > 3.0e38f || scale < -3.0e38f)
    return fail(PKV_ERR_INVALID_ARG, "scale is not finite");
  DecodeArgs a;
  const size_t need = decode_workspace_bytes(num_seqs, num_q_heads, cache.head_dim,
                                             plan->max_splits, &a.ws, workspace);
  if (workspace_bytes < need)
    return fail(PKV_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes, plan needs %zu",
                workspace_bytes, need);
  const ContextState* d = nullptr;
  st = context_state(&d);
  if (st != PKV_OK) return st;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.cache = cache;
  a.block_tables = block_tables;
  a.max_blocks = max_blocks_per_seq;
  a.context_lens = context_lens;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.scale = scale;
  a.split_tokens = plan->split_tokens;
  a.max_splits = plan->max_splits;
  a.auto_split = plan->auto_split != 0;
  a.out = out;
  a.flags = d->flags;
  a.k_new = k_new;
  a.v_new = v_new;
  a.slot_mapping = slot_mapping;
  a.ctas_per_sm = d->decode_ctas;
  a.reuse_plan = (plan->flags & PKV_DECODE_PLAN_REUSE) != 0;
  const int64_t rows = (int64_t)cache.num_blocks * cache.block_size;
  CUtensorMap tk, tv;
  cudaError_t e = cudaSuccess;
  if (tc) {
    // keys on the MMA's M dimension: 128-byte swizzled boxes of 64 dims; q as G rows per box
    CUtensorMap tq;
    st = encode_rows_map(&tq, q, num_seqs, num_q_heads, 128, 64, 1, CU_TENSOR_MAP_SWIZZLE_128B, G);
    if (st != PKV_OK) return st;
    const int box = decode_tc_box_rows(cache.block_size);
    st = encode_rows_map(&tk, k_cache, rows, cache.num_kv_heads, 128, 64, box,
                         CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != PKV_OK) return st;
    st = encode_rows_map(&tv, v_cache, rows, cache.num_kv_heads, 128, 64, box,
                         CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != PKV_OK) return st;
    // boxes of 64 and 32 rows for partial last tiles (only used where smaller than `box`)
    CUtensorMap tail[4];
    for (int i = 0; i < 4; ++i) {
      const int r = (i < 2 ? 64 : 32) < box ? (i < 2 ? 64 : 32) : box;
      st = encode_rows_map(&tail[i], (i & 1) ? v_cache : k_cache, rows, cache.num_kv_heads, 128,
                           64, r, CU_TENSOR_MAP_SWIZZLE_128B);
      if (st != PKV_OK) return st;
    }
    e = launch_paged_decode_tc(a, tq, tk, tv, tail, d->num_sms, static_cast<cudaStream_t>(stream));
  } else {
    const int box_t = decode_box_rows(cache.head_dim, G, cache.block_size);
    st = encode_rows_map(&tk, k_cache, rows, cache.num_kv_heads, cache.head_dim, cache.head_dim,
                         box_t, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st != PKV_OK) return st;
    st = encode_rows_map(&tv, v_cache, rows, cache.num_kv_heads, cache.head_dim, cache.head_dim,
                         box_t, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st != PKV_OK) return st;
    e = launch_paged_decode(a, tk, tv, d->num_sms, static_cast<cudaStream_t>(stream));
  }
  if (e == cudaErrorNotSupported) return fail(PKV_ERR_UNSUPPORTED, "no decode instance");
  if (e != cudaSuccess) return cuda_fail(e, "paged_decode launch");
  return PKV_OK;
}

int pkv_paged_decode(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                     pkv_cache_desc cache, const int32_t* block_tables,
                     int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t num_seqs,
                     int32_t num_q_heads, float scale, const pkv_decode_plan* plan,
                     uint16_t* out, void* workspace, size_t workspace_bytes, void* stream) {
  return decode_impl(q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq, context_lens,
                     num_seqs, num_q_heads, scale, plan, out, workspace, workspace_bytes, stream,
                     nullptr, nullptr, nullptr);
}

int pkv_paged_decode_store(const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                           const int32_t* slot_mapping, uint16_t* k_cache, uint16_t* v_cache,
                           pkv_cache_desc cache, const int32_t* block_tables,
                           int32_t max_blocks_per_seq, const int32_t* context_lens,
                           int32_t num_seqs, int32_t num_q_heads, float scale,
                           const pkv_decode_plan* plan, uint16_t* out, void* workspace,
                           size_t workspace_bytes, void* stream) {
  g_last_error[0] = 0;
  if (num_seqs > 0 && (!k_new || !v_new || !slot_mapping))
    return fail(PKV_ERR_INVALID_ARG, "null pointer");
  if (num_seqs > 0 && (!aligned16(k_new) || !aligned16(v_new)))
    return fail(PKV_ERR_INVALID_ARG, "k_new and v_new must be 16-byte aligned");
  return decode_impl(q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq, context_lens,
                     num_seqs, num_q_heads, scale, plan, out, workspace, workspace_bytes, stream,
                     k_new, v_new, slot_mapping);
}

int pkv_paged_prefill(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                      const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t num_seqs,
                      int32_t total_q, int32_t max_seqlen_q, const int32_t* block_tables,
                      int32_t max_blocks_per_seq, const uint16_t* k_cache,
                      const uint16_t* v_cache, pkv_cache_desc cache, int32_t num_q_heads,
                      float scale, uint16_t* out, void* workspace, size_t workspace_bytes,
                      void* stream) {
  g_last_error[0] = 0;
  if (num_seqs < 0 || total_q < 0 || max_seqlen_q < 0)
    return fail(PKV_ERR_INVALID_ARG, "num_seqs, total_q and max_seqlen_q must be >= 0");
  if (cache.num_kv_heads <= 0 || cache.head_dim <= 0)
    return fail(PKV_ERR_INVALID_ARG, "num_kv_heads and head_dim must be positive");
  if (cache.head_dim != 128)
    return fail(PKV_ERR_UNSUPPORTED, "paged_prefill supports head_dim 128 (got %d)",
                cache.head_dim);
  int st = check_heads(num_q_heads, cache.num_kv_heads);
  if (st != PKV_OK) return st;
  if (num_seqs == 0 || total_q == 0 || max_seqlen_q == 0) return PKV_OK;
  if (!q || !k || !v || !cu_seqlens_q || !cu_seqlens_k || !out)
    return fail(PKV_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return fail(PKV_ERR_INVALID_ARG, "q, k, v and out must be 16-byte aligned");
  if (!workspace || !aligned16(workspace))
    return fail(PKV_ERR_INVALID_ARG, "workspace must be a 16-byte aligned device pointer");
  if (workspace_bytes < PKV_PREFILL_WORKSPACE_BYTES)
    return fail(PKV_ERR_WORKSPACE_TOO_SMALL, "workspace_bytes %zu < %d", workspace_bytes,
                PKV_PREFILL_WORKSPACE_BYTES);
  const bool paged = block_tables != nullptr;
  if (paged) {
    st = check_cache(cache);
    if (st != PKV_OK) return st;
    if (!k_cache || !v_cache) return fail(PKV_ERR_INVALID_ARG, "null cache pointer");
    if (!aligned16(k_cache) || !aligned16(v_cache))
      return fail(PKV_ERR_INVALID_ARG, "caches must be 16-byte aligned");
    if (max_blocks_per_seq <= 0)
      return fail(PKV_ERR_INVALID_ARG, "max_blocks_per_seq %d <= 0", max_blocks_per_seq);
  }
  if (!(scale == scale) || scale > 3.0e38f || scale < -3.0e38f)
    return fail(PKV_ERR_INVALID_ARG, "scale is not finite");
  const ContextState* d = nullptr;
  st = context_state(&d);
  if (st != PKV_OK) return st;
  const int G = num_q_heads / cache.num_kv_heads;
  CUtensorMap tq, tk, tv;
  st = encode_rows_map(&tq, q, total_q, num_q_heads, 128, 64, prefill_positions_per_tile(G),
                       CU_TENSOR_MAP_SWIZZLE_128B, G);
  if (st != PKV_OK) return st;
  const int box = prefill_kv_box_rows(cache.block_size, paged);
  if (paged) {
    const int64_t rows = (int64_t)cache.num_blocks * cache.block_size;
    st = encode_rows_map(&tk, k_cache, rows, cache.num_kv_heads, 128, 64, box,
                         CU_TENSOR_MAP_SWIZZLE_128B);
    if (st == PKV_OK)
      st = encode_rows_map(&tv, v_cache, rows, cache.num_kv_heads, 128, 64, box,
                           CU_TENSOR_MAP_SWIZZLE_128B);
  } else {
    st = encode_rows_map(&tk, k, total_q, cache.num_kv_heads, 128, 64, box,
                         CU_TENSOR_MAP_SWIZZLE_128B);
    if (st == PKV_OK)
      st = encode_rows_map(&tv, v, total_q, cache.num_kv_heads, 128, 64, box,
                           CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (st != PKV_OK) return st;
  PrefillArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.cu_seqlens_q = cu_seqlens_q;
  a.cu_seqlens_k = cu_seqlens_k;
  a.num_seqs = num_seqs;
  a.total_q = total_q;
  a.max_seqlen_q = max_seqlen_q;
  a.block_tables = block_tables;
  a.max_blocks = paged ? max_blocks_per_seq : 0;
  a.cache = cache;
  a.num_q_heads = num_q_heads;
  a.scale = scale;
  a.out = out;
  a.flags = d->flags;
  a.item_counter = static_cast<int32_t*>(workspace);
  // dense item numbering when the workspace holds the per-sequence prefix after the counter
  if (workspace_bytes >= pkv_prefill_workspace_bytes(num_seqs))
    a.item_prefix = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) +
                                               PKV_PREFILL_WORKSPACE_BYTES);
  cudaError_t e = launch_paged_prefill(a, tq, tk, tv, d->num_sms,
                                       static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "paged_prefill launch");
  return PKV_OK;
}

size_t pkv_prefill_workspace_bytes(int32_t num_seqs) {
  if (num_seqs < 0) return PKV_PREFILL_WORKSPACE_BYTES;
  const size_t prefix = (2 * (size_t)num_seqs + 1) * sizeof(int32_t);  // prefix + permutation
  return PKV_PREFILL_WORKSPACE_BYTES + (prefix + 255) / 256 * 256;
}

}  // extern "C"
