// kda_noalloc.cu -- kda_chunk_fwd for callers that cannot allocate device memory.
//
// Some callers of a prefill kernel are not allowed to call cudaMalloc (or any
// allocator) at the point where they run it: a serving engine that reserved all
// device memory at start-up and hands none out on the request path, a plugin
// host that gives its plugins no allocator, or a latency-critical loop that
// cannot afford an allocation's implicit synchronization.  kda_chunk_fwd needs a
// scratch workspace; this entry point supplies it from a fixed array that the
// library declares in device memory, so the caller passes only inputs and
// outputs.
//
// The array has a fixed capacity (KDA_NOALLOC_SCRATCH_BYTES) and exists on every
// GPU that loads the library until the process exits.  All calls share it and it
// keeps the last call's contents; the kernels write every workspace byte they
// later read, so nothing needs clearing between calls.  Two calls whose work
// overlaps on the GPU (different streams without ordering) race on the array.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/kda.h"
#include "kda_internal.cuh"

namespace kda {
void set_error_message(const char* msg);
}

namespace {

constexpr size_t kScratchBytes = KDA_NOALLOC_SCRATCH_BYTES;

__device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of the array on the current device, resolved once per device
// (cudaGetSymbolAddress with that device current).  Host code must not use the
// symbol itself: on the host it names a stand-in object, not device memory.
void* scratch_address(cudaError_t* err) {
  static void* addr[64] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 64) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (*err != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

extern "C" {

size_t kda_chunk_fwd_noalloc_capacity(void) { return kScratchBytes; }

kda_status_t kda_chunk_fwd_noalloc(const void* q, const void* k, const void* v, int dtype,
                                   const float* g, const void* beta, const float* h0,
                                   const int32_t* cu_seqlens, int n_seqs, int B, int64_t T,
                                   int H, int dk, int dv, void* o, float* hT,
                                   kda_stream_t stream) {
  cudaError_t e = cudaSuccess;
  void* ws = scratch_address(&e);
  if (!ws) {
    kda::set_error_message("kda_chunk_fwd_noalloc: cannot resolve the scratch array's address");
    return KDA_ERR_CUDA;
  }
  // kda_chunk_fwd checks every argument first (shapes, dtypes, pointers, alignment)
  // and only then compares its workspace need with the array's capacity, so a
  // malformed call gets its own error and a well-formed one that is too large
  // gets KDA_ERR_WORKSPACE_TOO_SMALL; either way nothing has been enqueued.
  const kda_status_t st = kda_chunk_fwd(q, k, v, dtype, g, beta, h0, cu_seqlens, n_seqs, B, T,
                                        H, dk, dv, o, hT, ws, kScratchBytes, stream);
  if (st == KDA_ERR_WORKSPACE_TOO_SMALL)
    kda::set_error_message(
        "kda_chunk_fwd_noalloc: this problem needs more scratch than the library's fixed "
        "device array holds (KDA_NOALLOC_SCRATCH_BYTES); use kda_chunk_fwd with a workspace");
  return st;
}

}  // extern "C"
