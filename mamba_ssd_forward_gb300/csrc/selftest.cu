// Self-test of the bounded device-side waits every kernel of the library
// uses: one CTA waits on an mbarrier that nothing ever arrives on.  The wait
// gives up after the caller's limit, records its code in the given error
// word and returns, so the kernel ends and the context stays usable; the
// next read of that word (ssd_workspace_error, or ssd_device_error for the
// library-wide word) reports SSD_ERR_TIMEOUT and clears it.
#include "tc_common.cuh"

namespace ssd {
namespace {

constexpr int kSelftestCode = 199;

__global__ void bounded_wait_selftest(int *err, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t never;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&never, 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) ptx::mbar_wait(&never, 0, err, kSelftestCode, limit_ns);
  __syncthreads();
}

}  // namespace
}  // namespace ssd

extern "C" ssd_status ssd_selftest_bounded_wait(uint64_t limit_ns, int *err_word, void *stream) {
  if (limit_ns < 1000 || limit_ns > 1000000000ull) return SSD_ERR_INVALID_ARG;
  if (err_word && (reinterpret_cast<uintptr_t>(err_word) & 3u)) return SSD_ERR_INVALID_ARG;
  int *err = err_word ? err_word : ssd::device_error_word();
  if (!err) return SSD_ERR_CUDA;
  ssd::bounded_wait_selftest<<<1, 32, 0, (cudaStream_t)stream>>>(
      err, (unsigned long long)limit_ns);
  return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}
