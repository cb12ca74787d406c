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
// code cannot use the array's name as a device address, so the first call on a
// device (with that device current) looks the address up with
// cudaGetSymbolAddress and keeps it; later calls on that device reuse it.
#include <mutex>

#include "../../include/moe.h"
#include "internal.h"

namespace {

constexpr size_t kStaticWorkspaceBytes = MOE_NOALLOC_WORKSPACE_BYTES;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_static_ws[kStaticWorkspaceBytes];

void* g_ws_addr[kMaxDevices] = {};
std::mutex g_ws_mutex;

// Device address of g_static_ws on the current device (looked up once per device).
int static_workspace(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_ws_mutex);
  if (!g_ws_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
    g_ws_addr[dev] = p;
  }
  *out = g_ws_addr[dev];
  return MOE_OK;
}

}  // namespace

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
  // Every kernel of the forward pass writes the scratch it later reads (the
  // grouping kernel also clears the device status word first), so what the
  // previous call left in the array needs no clearing.
  return moe_ffn_forward(cfg, x, T, router, experts, shared, y, topk_ids, topk_w, ws,
                         kStaticWorkspaceBytes, stream);
}
