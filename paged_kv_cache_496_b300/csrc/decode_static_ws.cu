// decode_static_ws.cu -- paged decode for callers that cannot allocate device memory.
//
// pkv_paged_decode needs a device workspace (work list, claim counter, chunk partials) that the
// caller allocates. Some callers cannot do that: a host process that has handed all of a GPU's
// memory to its own pool allocator (so a cudaMalloc would fail or fragment that pool), or code
// that must not enter an allocator at the point where it runs attention, such as a plugin called
// from inside another runtime's execution loop. pkv_paged_decode_static_ws serves them: it runs
// the same decode with the workspace placed in a fixed-size array in the library's own device
// memory, PKV_STATIC_WS_BYTES long (a file-scope __device__ array that every GPU which loads the
// library holds until the process exits). It calls no allocating routine.
//
// Sharing: every call on a device uses the same array, which keeps what the previous call left
// in it. The decode's one-CTA plan kernel resets everything that must start at zero (the claim
// counter and the per-chunk merge counters) at the start of each call, so nothing has to be
// cleared here. Two calls that overlap on the GPU (different streams, no ordering between them)
// race on the array and corrupt each other's results: order them, for example on one stream.
#include <mutex>
#include <vector>

#include "common.cuh"
#include "kernels.h"

namespace {

static __device__ __align__(256) unsigned char g_static_workspace[PKV_STATIC_WS_BYTES];

// Device address of the array in each CUDA context seen so far, keyed by the driver's unique
// context id. Host code cannot use the symbol itself (it names a host-side stand-in), and each
// context (normally one per device: its primary context) holds its own copy of the array, so the
// first call in a context looks the address up with that context current and keeps it. After
// cudaDeviceReset the device's new primary context has a new id and gets a fresh lookup.
struct WorkspaceAddr {
  unsigned long long ctx_id;
  void* addr;
};
std::mutex g_workspace_mutex;
std::vector<WorkspaceAddr> g_workspace_addrs;

int static_workspace(void** out) {
  unsigned long long id = 0;
  int st = pkv::current_context_id(&id, nullptr);
  if (st != PKV_OK) return st;
  std::lock_guard<std::mutex> lock(g_workspace_mutex);
  for (const WorkspaceAddr& w : g_workspace_addrs)
    if (w.ctx_id == id) {
      *out = w.addr;
      return PKV_OK;
    }
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_static_workspace);
  if (e != cudaSuccess) return pkv::report_cuda_error(e, "cudaGetSymbolAddress(static workspace)");
  if (p == nullptr)
    return pkv::report_cuda_error(cudaErrorInvalidSymbol, "cudaGetSymbolAddress(static workspace)");
  g_workspace_addrs.push_back(WorkspaceAddr{id, p});
  *out = p;
  return PKV_OK;
}

}  // namespace

extern "C" PKV_API int pkv_paged_decode_static_ws(
    const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache, pkv_cache_desc cache,
    const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* context_lens,
    int32_t num_seqs, int32_t num_q_heads, float scale, const pkv_decode_plan* plan,
    uint16_t* out, void* stream) {
  void* ws = nullptr;
  const int st = static_workspace(&ws);
  if (st != PKV_OK) return st;
  // pkv_paged_decode validates every argument and rejects a plan whose workspace exceeds
  // PKV_STATIC_WS_BYTES (PKV_ERR_WORKSPACE_TOO_SMALL, with both sizes in pkv_last_error())
  // before anything is enqueued.
  return pkv_paged_decode(q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq,
                          context_lens, num_seqs, num_q_heads, scale, plan, out, ws,
                          (size_t)PKV_STATIC_WS_BYTES, stream);
}
