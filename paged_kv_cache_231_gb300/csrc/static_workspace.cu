// pkv_paged_attention_static_workspace: the paged attention call for callers that may
// not allocate device memory themselves (for example an engine plugin whose enqueue
// step is not allowed to allocate, or a host framework that has handed all device
// memory to its own pool). Its scratch lives in a file-scope __device__ array of
// PKV_STATIC_WORKSPACE_BYTES that every GPU loading this library keeps until exit.
//
// The array's name is a host-side stand-in in host code, not a device address, so the
// host resolves the real address once per device with cudaGetSymbolAddress (with that
// device current) and passes it to the unchanged paged attention path. The first call
// on a device performs that look-up; make it before any stream capture. Under lazy module
// loading (CUDA's default) that look-up also loads the module and commits the array, so
// the first call must come before a caller's pool takes the device's memory. The cached
// address is not refreshed after a device reset, which is therefore not supported.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

constexpr size_t kStaticBytes = PKV_STATIC_WORKSPACE_BYTES;

// Keeps the previous call's contents; nothing needs clearing, because the planner of every
// call rewrites the counters and piece tickets it later reads.
static __device__ __align__(256) unsigned char g_static_workspace[kStaticBytes];

namespace {

constexpr int kMaxDevices = 64;

std::mutex g_mutex;
void* g_device_address[kMaxDevices] = {};

// Device address of g_static_workspace on the current device (looked up once).
int static_workspace_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return PKV_ERR_LAUNCH;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_device_address[dev]) {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_static_workspace) != cudaSuccess || !addr)
      return PKV_ERR_LAUNCH;
    g_device_address[dev] = addr;
  }
  *out = g_device_address[dev];
  return PKV_OK;
}

}  // namespace

extern "C" int pkv_paged_attention_static_workspace(const pkv_paged_attention_args* args,
                                                    void* stream) {
  size_t need = 0;
  const int st = pkv_paged_attention_workspace_size(args, &need);
  if (st != PKV_OK) return st;
  if (need > kStaticBytes) return PKV_ERR_WORKSPACE;
  if (args->num_tokens == 0) return PKV_OK;
  void* ws = nullptr;
  const int got = static_workspace_address(&ws);
  if (got != PKV_OK) return got;
  return pkv_paged_attention(args, ws, kStaticBytes, stream);
}
