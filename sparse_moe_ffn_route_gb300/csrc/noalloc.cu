// moe_ffn_forward_noalloc: the whole layer with its scratch memory taken from a
// fixed array that the library itself holds in device memory, for callers that
// cannot allocate device memory.
//
// Who needs this: code that is handed only its input and output buffers, such
// as a plug-in kernel inside a host program or serving framework that owns all
// device memory through its own pool (a cudaMalloc there would fail, or take
// memory the pool has already reserved), or a latency-critical loop that must
// not make a call which may synchronise the device.  Such callers cannot
// provide the workspace that moe_ffn_forward asks for.
//
// The array is file-scope device memory of the library: every GPU that loads
// libmoe.so holds kStaticWorkspaceBytes of it until the process exits.  Host
// code cannot use the array's name as a device address.  A __device__ symbol
// has its own address in every CUDA context (the device's primary context, a
// context the host program made with the driver API, the primary context
// re-created after cudaDeviceReset), so the address is looked up with
// cudaGetSymbolAddress once per context, with that context current, and kept
// under the context's unique id.
#include <mutex>

#include "../../include/moe.h"
#include "internal.h"

namespace {

constexpr size_t kStaticWorkspaceBytes = MOE_NOALLOC_WORKSPACE_BYTES;
constexpr int kCachedContexts = 16;

__device__ __align__(256) unsigned char g_static_ws[kStaticWorkspaceBytes];

// Driver entry points, resolved through the runtime (no link-time libcuda).
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

struct CachedAddress {
  unsigned long long ctx_id;   // 0: unused (context ids start at 1)
  void* addr;
};

std::mutex g_ws_mutex;
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;
CachedAddress g_ws_cache[kCachedContexts] = {};
int g_ws_next = 0;

bool resolve_driver_calls() {
  if (g_ctx_get_current && g_ctx_get_id) return true;
  void* a = nullptr;
  void* b = nullptr;
  cudaDriverEntryPointQueryResult qa, qb;
  if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) != cudaSuccess ||
      qa != cudaDriverEntryPointSuccess || !a)
    return false;
  if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) != cudaSuccess ||
      qb != cudaDriverEntryPointSuccess || !b)
    return false;
  g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(a);
  g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(b);
  return true;
}

// Unique id of the calling thread's current context; 0 when none is current.
unsigned long long current_context_id() {
  CUcontext ctx = nullptr;
  if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  unsigned long long id = 0;
  if (g_ctx_get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of g_static_ws in the current context.
int static_workspace(void** out) {
  std::lock_guard<std::mutex> lock(g_ws_mutex);
  if (!resolve_driver_calls()) {
    (void)cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  unsigned long long id = current_context_id();
  void* p = nullptr;
  if (id == 0) {
    // No context is current on this thread yet: the runtime's lookup makes the
    // current device's primary context current, and the address belongs to it.
    if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || !p) {
      (void)cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    id = current_context_id();
    if (id == 0) return MOE_ERR_CUDA;
  } else {
    for (const CachedAddress& c : g_ws_cache)
      if (c.ctx_id == id) {
        *out = c.addr;
        return MOE_OK;
      }
    if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || !p) {
      (void)cudaGetLastError();
      return MOE_ERR_CUDA;
    }
  }
  for (const CachedAddress& c : g_ws_cache)
    if (c.ctx_id == id) {
      *out = c.addr;
      return MOE_OK;
    }
  g_ws_cache[g_ws_next] = CachedAddress{id, p};
  g_ws_next = (g_ws_next + 1) % kCachedContexts;
  *out = p;
  return MOE_OK;
}

}  // namespace

extern "C" size_t moe_noalloc_workspace_bytes(void) { return kStaticWorkspaceBytes; }

extern "C" int moe_ffn_forward_noalloc(const moe_cfg_t* cfg, const void* x, int32_t T,
                                       const moe_router_t* router, const moe_experts_t* experts,
                                       const moe_shared_t* shared, void* y, int32_t* topk_ids,
                                       float* topk_w, void* stream) {
  const size_t need = moe_workspace_bytes(cfg, T);
  if (need == 0) return MOE_ERR_INVALID_ARG;           // invalid cfg or T < 0
  if (need > kStaticWorkspaceBytes) return MOE_ERR_WORKSPACE;
  if (T == 0) return MOE_OK;
  void* ws = nullptr;
  const int st = static_workspace(&ws);
  if (st != MOE_OK) return st;
  // Every kernel of the forward pass writes the scratch it later reads, and the
  // call's first kernel (the router logits, or the RMSNorm when cfg.rms_norm)
  // clears the device status word, so what the previous call left in the array
  // needs no clearing.
  return moe_ffn_forward(cfg, x, T, router, experts, shared, y, topk_ids, topk_w, ws,
                         kStaticWorkspaceBytes, stream);
}

extern "C" int moe_noalloc_device_status(void* stream, uint32_t* detail) {
  void* ws = nullptr;
  const int st = static_workspace(&ws);
  if (st != MOE_OK) return st;
  return moe_device_status(ws, stream, detail);
}
