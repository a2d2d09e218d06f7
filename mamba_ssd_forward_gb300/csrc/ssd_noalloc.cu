// ssd_forward_noalloc: the forward pass with its workspace in a fixed,
// statically sized device array of this library, for callers that cannot
// allocate device memory at call time (see include/ssd.h for who and why).
//
// Nothing here calls cudaMalloc, cudaFree or a library routine that
// allocates.  The only set-up is cudaGetSymbolAddress, once per (device,
// context) pair, guarded by a mutex; its result is cached under that pair, so
// a device reset or a different context current on the same device looks the
// array up afresh instead of reusing an address from an unloaded module.
#include <cuda.h>

#include <mutex>
#include <vector>

#include "ssd_internal.cuh"

namespace {

// The scratch array.  Its size is part of the ABI (SSD_NOALLOC_SCRATCH_BYTES);
// 256-byte alignment is what ssd_forward asks of a workspace.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SSD_NOALLOC_SCRATCH_BYTES];

using GetCtx = CUresult (*)(CUcontext *);

// cuCtxGetCurrent through the runtime's driver entry-point query (the library
// does not link libcuda directly); null if unavailable.
GetCtx get_ctx_fn() {
  static GetCtx fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<GetCtx>(p);
  });
  return fn;
}

struct CacheEntry {
  int dev;
  CUcontext ctx;
  void *addr;
};
std::mutex g_setup_mutex;
std::vector<CacheEntry> g_cache;  // guarded by g_setup_mutex

// Device address of the array in the current context; nullptr if the look-up
// failed.
void *scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  GetCtx fn = get_ctx_fn();
  if (!fn) return nullptr;
  CUcontext ctx = nullptr;
  if (fn(&ctx) != CUDA_SUCCESS) return nullptr;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (ctx)
    for (const CacheEntry &c : g_cache)
      if (c.dev == dev && c.ctx == ctx) return c.addr;
  // the look-up also makes the device's primary context current when no
  // context is yet (nothing is allocated); the key is then read again
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
  if (!ctx && (fn(&ctx) != CUDA_SUCCESS || !ctx)) return nullptr;
  g_cache.push_back(CacheEntry{dev, ctx, p});
  return p;
}

}  // namespace

extern "C" ssd_status ssd_forward_noalloc(const ssd_dims *dims, ssd_dtype dtype, const void *x,
                                          const void *dt, const float *A, const void *B,
                                          const void *C, const float *D, const float *h0,
                                          void *y, float *final_state, void *stream) {
  // dims, dtype and pointers first, with ssd_forward's codes; then the size
  ssd::Dims d;
  const ssd_status s =
      ssd::check_forward_args(dims, dtype, x, dt, A, B, C, D, h0, y, final_state, &d);
  if (s != SSD_OK) return s;
  const size_t need = ssd_forward_workspace_size(dims, dtype);
  if (need == 0 || need > (size_t)SSD_NOALLOC_SCRATCH_BYTES) return SSD_ERR_UNSUPPORTED;
  void *ws = scratch_address();
  if (!ws) return SSD_ERR_CUDA;
  int *err = ssd::device_error_word();
  if (!err) return SSD_ERR_CUDA;
  // Every byte of the workspace that the kernels read is written earlier in
  // the same call, so the array needs no clearing between calls; bounded
  // waits that give up report to the library-wide error word
  // (ssd_device_error), since the array is not the caller's.
  return ssd::forward_impl(dims, dtype, x, dt, A, B, C, D, h0, y, final_state, ws,
                           (size_t)SSD_NOALLOC_SCRATCH_BYTES, nullptr, err, (cudaStream_t)stream,
                           nullptr, 0, nullptr);
}
