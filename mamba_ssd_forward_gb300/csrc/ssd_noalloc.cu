// ssd_forward_noalloc: the forward pass with its workspace in a fixed,
// statically sized device array of this library, for callers that cannot
// allocate device memory at call time (see include/ssd.h for who and why).
//
// Nothing here calls cudaMalloc, cudaFree or a library routine that
// allocates.  The only set-up is cudaGetSymbolAddress, once per device,
// guarded by a mutex; its result is cached, so later calls make no CUDA call
// besides cudaGetDevice before handing the array to ssd_forward.
#include <mutex>

#include "ssd_internal.cuh"

namespace {

// The scratch array.  Its size is part of the ABI (SSD_NOALLOC_SCRATCH_BYTES);
// 256-byte alignment is what ssd_forward asks of a workspace.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SSD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 256;
std::mutex g_setup_mutex;
void *g_scratch_addr[kMaxDevices];  // device address of the array, per device ordinal

// Device address of the array on device `dev`; nullptr if the lookup failed.
void *scratch_address(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" ssd_status ssd_forward_noalloc(const ssd_dims *dims, ssd_dtype dtype, const void *x,
                                          const void *dt, const float *A, const void *B,
                                          const void *C, const float *D, const float *h0,
                                          void *y, float *final_state, void *stream) {
  const size_t need = ssd_forward_workspace_size(dims, dtype);
  if (need == 0)  // invalid dims or dtype: ssd_forward reports which, launching nothing
    return ssd_forward(dims, dtype, x, dt, A, B, C, D, h0, y, final_state, nullptr, 0, stream);
  if (need > (size_t)SSD_NOALLOC_SCRATCH_BYTES) return SSD_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SSD_ERR_CUDA;
  void *ws = scratch_address(dev);
  if (!ws) return SSD_ERR_CUDA;
  // Every byte of the workspace that ssd_forward reads is written earlier in
  // the same call, so the array needs no clearing between calls.
  return ssd_forward(dims, dtype, x, dt, A, B, C, D, h0, y, final_state, ws,
                     (size_t)SSD_NOALLOC_SCRATCH_BYTES, stream);
}
