// kda_noalloc.cu -- kda_fwd for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) when they run the
// forward: for example a plugin or callback executing inside another engine
// that owns all device memory and hands it only the inputs and outputs, or a
// latency-critical path that cannot afford cudaMalloc's implicit device
// synchronisation. kda_fwd_no_alloc serves them: its scratch lives in one
// file-scope device array of fixed size, so the call allocates nothing.
//
// Rules (also stated in include/kda.h):
//  * the array holds KDA_NO_ALLOC_SCRATCH_BYTES; larger problems are rejected
//    with KDA_ERR_INVALID_ARG before anything is enqueued;
//  * each device that loads this code keeps the array until the process exits;
//  * the first call on a device looks up the array's device address (with that
//    device current) and caches it; make that first call before any stream
//    capture;
//  * every call uses the same array, so calls whose work overlaps on the GPU
//    (other streams, other host threads) race; the array keeps the previous
//    call's contents -- the forward writes every scratch byte it reads before
//    reading it, so nothing needs clearing. That is why skip_prep (which reads
//    chunk records left in the scratch by an earlier call) is rejected here:
//    the earlier call may have been another caller's problem;
//  * the cached address belongs to the device's current context: after
//    cudaDeviceReset (or a release and re-creation of the primary context) the
//    array is loaded again elsewhere, so the entry point must not be used
//    across a reset.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "../../include/kda.h"
#include "kda_internal.h"

namespace {

__device__ __align__(256) unsigned char g_kda_fwd_scratch[KDA_NO_ALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 256;
void *g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

// Device address of the scratch array on the current device (set up once per device).
cudaError_t scratch_ptr(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_kda_fwd_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" kda_status kda_fwd_no_alloc(const kda_fwd_args *args, cudaStream_t stream) {
  if (!args) return kda_fwd(args, stream);   // reports the NULL-args error
  if (args->skip_prep) {
    kda::set_last_error(
        "kda_fwd_no_alloc: skip_prep is not supported (the shared static scratch may hold another call's chunk records)");
    return KDA_ERR_UNSUPPORTED;
  }
  // the caller's workspace fields are ignored: size and run a copy without them
  kda_fwd_args a = *args;
  a.workspace = nullptr;
  a.workspace_bytes = 0;
  const size_t need = kda_fwd_workspace_size(&a);
  if (need == 0) return kda_fwd(&a, stream);   // invalid arguments: kda_fwd reports which
  if (need > (size_t)KDA_NO_ALLOC_SCRATCH_BYTES) {
    char msg[256];
    std::snprintf(msg, sizeof msg,
                  "kda_fwd_no_alloc: this problem needs %zu bytes of scratch, more than the %zu-byte static scratch",
                  need, (size_t)KDA_NO_ALLOC_SCRATCH_BYTES);
    kda::set_last_error(msg);
    return KDA_ERR_INVALID_ARG;
  }
  void *ptr = nullptr;
  const cudaError_t e = scratch_ptr(&ptr);
  if (e != cudaSuccess) {
    char msg[256];
    std::snprintf(msg, sizeof msg, "kda_fwd_no_alloc: cudaGetSymbolAddress of the static scratch failed: %s",
                  cudaGetErrorString(e));
    kda::set_last_error(msg);
    return KDA_ERR_CUDA;
  }
  a.workspace = ptr;
  a.workspace_bytes = KDA_NO_ALLOC_SCRATCH_BYTES;
  return kda_fwd(&a, stream);
}
