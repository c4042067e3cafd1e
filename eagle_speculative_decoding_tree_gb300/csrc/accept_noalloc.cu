// accept_noalloc.cu -- eagle_accept_noalloc: the acceptance step with its scratch in a
// fixed device buffer, so the call needs no workspace from the caller.
//
// Who needs it: callers that cannot allocate device memory at the point where they
// verify a draft -- a runtime that reserved all of the GPU's memory up front and
// hands none out per call, an inference server whose allocator is not reachable from
// the thread that runs acceptance, or C code linked against the library without any
// device allocator of its own.  eagle_accept asks them for a workspace (row
// statistics exchanged between its two kernels); this entry point keeps that scratch
// in a file-scope device array of EAGLE_ACCEPT_NOALLOC_SCRATCH_BYTES instead and
// makes no allocation itself.  It runs the very same kernels as eagle_accept.
//
// The scratch needs no clearing: each call zeroes the barrier counters it uses and
// writes every chunk record before reading it.  There is one buffer per device, so
// calls on the same device must not overlap in time (two streams, or two host
// threads, running it at once would race on the buffer).
#include <mutex>

#include "launch.h"

namespace {

// One device-resident scratch buffer, 256-byte aligned (the kernels need 16).
static __device__ __align__(256) unsigned char g_accept_scratch[EAGLE_ACCEPT_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// Device address of g_accept_scratch on the current device, looked up once per
// device (the first call on a device does it) and cached.  nullptr on failure, with
// the CUDA error in *err.
void* scratch_on_current_device(cudaError_t* err) {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    *err = e;
    return nullptr;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_accept_scratch);
    if (e != cudaSuccess || !p) {
      *err = (e != cudaSuccess) ? e : cudaErrorInvalidSymbol;
      return nullptr;
    }
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

extern "C" int eagle_accept_noalloc(const eagle_accept_desc* d, const void* target_logits,
                                    const void* draft_logits, const int32_t* tree_tokens,
                                    const int32_t* tree_parent, const float* u_accept, const float* u_final,
                                    const eagle_accept_out* out, void* stream) {
  const size_t need = eagle_workspace_size(EAGLE_WS_ACCEPT, d);
  if (need == 0)  // a bad descriptor: eagle_accept reports it before using any scratch
    return eagle_accept(d, target_logits, draft_logits, tree_tokens, tree_parent, u_accept, u_final, out, nullptr,
                        0, stream);
  if (need > EAGLE_ACCEPT_NOALLOC_SCRATCH_BYTES) return EAGLE_ERR_WORKSPACE;
  cudaError_t e = cudaSuccess;
  void* ws = scratch_on_current_device(&e);
  if (!ws) return eagle::report_cuda_error(e);
  return eagle_accept(d, target_logits, draft_logits, tree_tokens, tree_parent, u_accept, u_final, out, ws,
                      EAGLE_ACCEPT_NOALLOC_SCRATCH_BYTES, stream);
}
