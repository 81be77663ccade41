// attn_bwd_noalloc: the backward with its scratch memory inside the library.
//
// attn_bwd needs device scratch beyond its inputs and outputs: the row
// statistics it precomputes (L * log2 e and D), the fp32 dQ accumulator and,
// with a block mask, the compacted tile lists.  Normally the caller passes
// that scratch as a workspace it allocated.  Some callers cannot allocate
// device memory: a plug-in running inside a host application that owns every
// device allocation itself, a runtime with a fixed device-memory budget
// handed out at start-up, or a latency-critical loop where a cudaMalloc could
// synchronise the device.  For them this entry point keeps the scratch in a
// fixed-size array that is part of the library's own device code: every GPU
// that loads the library holds kNoAllocScratchBytes of it until the process
// exits.
//
// Everything else is the ordinary attn_bwd path: the entry point looks up
// the array's device address and calls attn_bwd with it as the workspace.
#include <cstdio>
#include <mutex>

#include "attn.h"
#include "attn_kernels.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t{64} << 20;   // 64 MiB

// The scratch.  In host code this name is only a host-side stand-in: the
// kernels get the device address looked up below.
static __device__ __align__(256) unsigned char g_bwd_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

}  // namespace

// Device address of the scratch on the current device; looked up once per
// device (with that device current) and cached.  attn_check(NULL, ...)
// reads the status words at its start through it.
int attn::builtin_scratch(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof(msg), "cudaGetDevice: %s", cudaGetErrorString(e));
    return static_cast<attn_status>(attn::record_error(ATTN_ERR_CUDA, msg));
  }
  if (dev < 0 || dev >= kMaxDevices)
    return static_cast<attn_status>(
        attn::record_error(ATTN_ERR_UNSUPPORTED, "device index beyond the scratch table"));
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_bwd_scratch);
    if (e != cudaSuccess || ptr == nullptr) {
      char msg[256];
      snprintf(msg, sizeof(msg), "cudaGetSymbolAddress of the built-in scratch: %s",
               cudaGetErrorString(e));
      return static_cast<attn_status>(attn::record_error(ATTN_ERR_CUDA, msg));
    }
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return ATTN_OK;
}

extern "C" attn_status attn_bwd_noalloc(const attn_params* p, const void* q, const void* k,
                                        const void* v, const void* o, const float* lse,
                                        const void* dout, void* dq, void* dk, void* dv,
                                        void* stream) {
  const size_t need = attn_workspace_size(p, 1);
  if (need == 0)   // invalid parameters: let the ordinary entry point say why
    return attn_bwd(p, q, k, v, o, lse, dout, dq, dk, dv, nullptr, 0, stream);
  if (need > kNoAllocScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "attn_bwd_noalloc: this problem needs %zu bytes of scratch; the built-in scratch "
             "holds %zu (use attn_bwd with a caller workspace)",
             need, kNoAllocScratchBytes);
    return static_cast<attn_status>(attn::record_error(ATTN_ERR_WORKSPACE, msg));
  }
  void* ws = nullptr;
  const attn_status st = static_cast<attn_status>(attn::builtin_scratch(&ws));
  if (st != ATTN_OK) return st;
  // the status words must start at zero; a previous call may have left a
  // time-out recorded there (every other part of the scratch is rewritten)
  const cudaError_t e = cudaMemsetAsync(ws, 0, 256, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof(msg), "attn_bwd_noalloc: status clear: %s", cudaGetErrorString(e));
    return static_cast<attn_status>(attn::record_error(ATTN_ERR_CUDA, msg));
  }
  return attn_bwd(p, q, k, v, o, lse, dout, dq, dk, dv, ws, kNoAllocScratchBytes, stream);
}
