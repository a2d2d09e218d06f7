// Internal declarations shared by the kernels and the C ABI of libssd_gb300.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ssd.h"

namespace ssd {

constexpr float kLog2e = 1.4426950408889634f;

// Dimensions after validation, with derived sizes.
struct Dims {
  int64_t b, L, nh, P, S, ng, T;
  int64_t nc;   // number of chunks, ceil(L / T)
  int64_t hpg;  // heads per group
};

// Element access for the two I/O types.
__device__ __forceinline__ float ld_io(const float *p) { return *p; }
__device__ __forceinline__ float ld_io(const __nv_bfloat16 *p) {
  return __bfloat162float(*p);
}
__device__ __forceinline__ void st_io(float *p, float v) { *p = v; }
__device__ __forceinline__ void st_io(__nv_bfloat16 *p, float v) {
  *p = __float2bfloat16_rn(v);
}

// Address of the device error word (current device); kernels that give up a
// bounded wait write a nonzero code there.
int *device_error_word();
// Copy the device error word to *code and clear it; synchronises `st`.
cudaError_t read_and_clear_device_error(cudaStream_t st, int *code);

// Launchers (one per step).  Each enqueues its kernel(s) on `st` and returns
// the cudaGetLastError() of the launch.
cudaError_t launch_chunk_cumsum(const Dims &d, ssd_dtype io, const void *dt,
                                const float *A, float *G, cudaStream_t st);
cudaError_t launch_chunk_state(const Dims &d, ssd_dtype io, const void *x,
                               const void *B, const void *dt, const float *G,
                               float *dstates, cudaStream_t st);
cudaError_t launch_state_passing(const Dims &d, const float *dstates,
                                 const float *G, const float *h0,
                                 float *states, float *final_state,
                                 cudaStream_t st);
cudaError_t launch_chunk_scan(const Dims &d, ssd_dtype io, const void *x,
                              const void *B, const void *C, const void *dt,
                              const float *G, const float *states,
                              const float *D, void *y, cudaStream_t st);

// Single-token decode step (decode_step.cu).
cudaError_t launch_decode_step(int64_t b, int64_t nh, int64_t P, int64_t S, int64_t ng,
                               ssd_dtype io, const void *x, const void *dt, const float *A,
                               const void *B, const void *C, const float *D, float *state,
                               void *y, cudaStream_t st);

}  // namespace ssd
