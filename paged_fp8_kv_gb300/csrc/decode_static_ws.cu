// mj_decode_attn_static_ws: decode attention whose split-KV workspace lives in
// a fixed device array compiled into this library, so the call allocates no
// memory at all.
//
// Who needs it: code that may not ask the CUDA allocator for memory at call
// time, for example a serving runtime that hands every byte of the device to
// its own arena up front, a plugin loaded into a host framework that owns the
// allocator, or a latency-critical thread that must not take the driver's
// allocation locks.  Such callers can still provide their inputs and outputs;
// only the scratch for the split partials is taken off their hands.
//
// The array below is reserved on every GPU that loads libmj.so for as long
// as the process lives, so it is kept small (MJ_STATIC_WORKSPACE_BYTES).

#include <cuda_runtime.h>

#include <mutex>

#include "mj.h"

namespace {

constexpr size_t kStaticWorkspaceBytes = MJ_STATIC_WORKSPACE_BYTES;
constexpr int kMaxDevices = 64;

// The shared scratch.  Host code must not use this name as an address: in
// host code it is only a stand-in for the device symbol.
static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

std::mutex g_mutex;
void* g_device_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per
// device (with that device current) and cached.
mj_status static_workspace_ptr(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return MJ_ERR_CUDA;
  if (dev >= kMaxDevices) return MJ_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_device_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || !p) return MJ_ERR_CUDA;
    g_device_ptr[dev] = p;
  }
  *out = g_device_ptr[dev];
  return MJ_OK;
}

}  // namespace

extern "C" mj_status mj_decode_attn_static_ws(const mj_decode_params* params, const mj_decode_args* args,
                                              mj_stream_t stream) {
  if (!params || !args) return MJ_ERR_INVALID_ARG;
  const size_t need = mj_decode_workspace_bytes(params);
  if (need > kStaticWorkspaceBytes) return MJ_ERR_CAPACITY;  // problem too large for the fixed scratch
  mj_decode_args a = *args;
  if (need > 0) {
    void* ws = nullptr;
    const mj_status st = static_workspace_ptr(&ws);
    if (st != MJ_OK) return st;
    a.workspace = ws;
    a.workspace_bytes = kStaticWorkspaceBytes;
  } else {
    a.workspace = nullptr;
    a.workspace_bytes = 0;
  }
  return mj_decode_attn(params, &a, stream);
}
