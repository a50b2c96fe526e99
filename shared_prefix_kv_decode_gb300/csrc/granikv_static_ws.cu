// granikv_static_ws.cu -- decode attention for callers that cannot allocate device memory.
//
// granikv_decode_attention needs a caller-provided workspace (the step's work list, the partial
// attention records and the per-row merge tickets).  Some callers cannot provide one: a serving
// engine that has reserved nearly all of the GPU's memory for its own KV pools and allocator up
// front, or a plain C host that only holds pointers to buffers someone else allocated.  For
// them this file keeps one workspace in a file-scope device array, sized at build time, and
// offers granikv_decode_attention_static, which runs the regular entry point on it.
//
// The array is a module global: every GPU that loads the library holds its kStaticWorkspaceBytes
// until the process exits, and every call on a device shares it.  Host code cannot use the
// array's name as a device address, so the first call on each device looks the address up with
// cudaGetSymbolAddress (with that device current) and caches it.
#include <mutex>

#include "../../include/granikv.h"
#include "internal.h"

namespace granikv {
namespace {

constexpr size_t kStaticWorkspaceBytes = size_t(16) << 20;  // 16 MiB

static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

constexpr int kMaxDevices = 64;
std::mutex g_addr_mutex;
void* g_addr[kMaxDevices] = {};

// Device address of g_static_workspace on `device` (looked up once, that device current).
cudaError_t static_workspace_address(int device, void** out) {
  if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_addr_mutex);
  if (!g_addr[device]) {
    int prev = -1;
    cudaError_t e = cudaGetDevice(&prev);
    if (e != cudaSuccess) return e;
    if (prev != device && (e = cudaSetDevice(device)) != cudaSuccess) return e;
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_static_workspace);
    if (prev != device) cudaSetDevice(prev);
    if (e != cudaSuccess) return e;
    g_addr[device] = ptr;
  }
  *out = g_addr[device];
  return cudaSuccess;
}

}  // namespace
}  // namespace granikv

extern "C" granikv_status granikv_decode_attention_static(granikv_ctx* ctx, int32_t layer, const void* q,
                                                          const granikv_batch* batch, granikv_plan* plan,
                                                          void* o, float* lse, granikv_stream_t stream) {
  using namespace granikv;
  if (!ctx || !plan || !batch) return GRANIKV_ERR_INVALID;
  size_t need = 0;
  granikv_status st = granikv_workspace_size(ctx, plan, &need);
  if (st != GRANIKV_OK) return st;
  if (need > kStaticWorkspaceBytes) return GRANIKV_ERR_STATIC_WORKSPACE_TOO_SMALL;
  int device = -1;
  st = granikv_internal_device(ctx, &device);
  if (st != GRANIKV_OK) return st;
  void* ws = nullptr;
  if (static_workspace_address(device, &ws) != cudaSuccess) return GRANIKV_ERR_CUDA;
  // The array may hold another plan's work list and tickets from an earlier call (of any
  // context): make this call copy its own work list in and zero its tickets again.
  granikv_internal_forget_workspace(ws);
  return granikv_decode_attention(ctx, layer, q, batch, plan, o, lse, ws, kStaticWorkspaceBytes, stream);
}
