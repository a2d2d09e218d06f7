// Kernels of the bf16 forward path (ssd_forward): a state pass over chunks
// and a warp-specialised output pass.  See fwd_state.cu and fwd_scan.cu.
#pragma once

#include "tc_common.cuh"

namespace ssd {

// Per-chunk start states (bf16, [b, nh, nc, S, P]) and the final state.
cudaError_t launch_fwd_state(const Dims &d, const void *x, const void *B, const void *dt,
                             const float *A, const float *h0, void *states, float *final_state,
                             cudaStream_t st);

// y from x, B, C, dt, A, D and the bf16 per-chunk states.
cudaError_t launch_fwd_scan(const Dims &d, const void *x, const void *B, const void *C,
                            const void *dt, const float *A, const void *states, const float *D,
                            void *y, cudaStream_t st);

// Heads per CTA of the output pass: the largest divisor of nheads/ngroups
// that is at most 4 and keeps heads * P <= 256 tensor-memory columns.
inline int fwd_scan_heads(const Dims &d) {
  const int hmax = (int)std::min<int64_t>(4, 256 / d.P);
  for (int h = hmax; h > 1; --h)
    if (d.hpg % h == 0) return h;
  return 1;
}

}  // namespace ssd
