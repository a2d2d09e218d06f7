// Kernels of the bf16 forward path (ssd_forward): the chunk jump terms (all
// chunks in parallel), the sequential pass over chunks, and the
// warp-specialised output pass.  See fwd_chunk_state.cu, fwd_state_pass.cu
// and fwd_scan.cu.
#pragma once

#include "tc_common.cuh"

namespace ssd {

// Jump term of every chunk (bf16, [b, nh, nc, S, P]) and its decay
// exp2(G_last) (fp32, [b, nh, nc]); all chunks in parallel.
cudaError_t launch_fwd_chunk_state(const Dims &d, const void *x, const void *B, const void *dt,
                                   const float *A, void *dH, float *gamma, cudaStream_t st);
// Sequential pass over chunks: per-chunk start states (bf16, [b, nh, nc, S,
// P]) and the final state (fp32, [b, nh, P, S]) from the jump terms.
cudaError_t launch_fwd_state_pass(const Dims &d, const void *dH, const float *gamma,
                                  const float *h0, void *states, float *final_state,
                                  cudaStream_t st);
// Heads per CTA of fwd_chunk_state (B shared by the heads of a group).
int fwd_state_heads(const Dims &d);

// y from x, B, C, dt, A, D and the bf16 per-chunk states.
cudaError_t launch_fwd_scan(const Dims &d, const void *x, const void *B, const void *C,
                            const void *dt, const float *A, const void *states, const float *D,
                            void *y, cudaStream_t st);

// Output pass with C B^T of a whole chunk shared by a slice of heads (P = 64,
// S in {64, 128}, T in {128, 256}); fwd_scan_chunk_supported says whether
// the dims qualify.
bool fwd_scan_chunk_supported(const Dims &d);
cudaError_t launch_fwd_scan_chunk(const Dims &d, const void *x, const void *B, const void *C,
                                  const void *dt, const float *A, const void *states,
                                  const float *D, void *y, cudaStream_t st);

// Heads per CTA of the output pass: the largest divisor of nheads/ngroups
// that is at most 4 and keeps heads * P <= 256 tensor-memory columns.
inline int fwd_scan_heads(const Dims &d) {
  const int hmax = (int)std::min<int64_t>(4, 256 / d.P);
  for (int h = hmax; h > 1; --h)
    if (d.hpg % h == 0) return h;
  return 1;
}

}  // namespace ssd
