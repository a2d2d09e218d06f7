// Kernels of the bf16 forward path (ssd_forward): the chunk jump terms (all
// chunks in parallel), the sequential pass over chunks, and the
// warp-specialised output passes.  See fwd_chunk_state.cu, fwd_state_pass.cu,
// fwd_scan_chunk.cu and fwd_scan.cu; ssd_plan.cu holds the launch plans.
#pragma once

#include <vector>

#include "tc_common.cuh"

namespace ssd {

// Sequential pass over chunks: per-chunk start states (bf16, [b, nh, nc, S,
// P]) and the final state (fp32, [b, nh, P, S]) from the jump terms and the
// (decay, scale) pairs of fwd_chunk_state: each stored start state is the
// carried state times its chunk's scale (a power of two: exact).
cudaError_t launch_fwd_state_pass(const Dims &d, const void *dH, const float2 *gamma,
                                  const float *h0, void *states, float *final_state, int *err,
                                  cudaStream_t st);

// Launch plans: knobs that change the speed of a kernel, never its results.

// fwd_chunk_state: jump term of every chunk (bf16, [b, nh, nc, S, P]) and its
// decay exp2(G_last) with the scale of its stored start state (fp32 pairs,
// [b, nh, nc]; the scale is 1 unless the anchors are written), all chunks
// in parallel, with H
// heads per work item (sharing one load of B) and `ctas` CTAs per SM.  With
// u, v, anchor not null it also writes the factored-decay inputs of
// fwd_out: u, v fp32 [b, nh, nc * T] and anchor [b, nh, nc] = (alpha,
// steep ? 1 : 0).
struct CsPlan {
  int H, ctas;
};
CsPlan chunk_state_plan(const Dims &d);  // the cost-model choice
bool chunk_state_plan_ok(const Dims &d, const CsPlan &plan);
cudaError_t launch_fwd_chunk_state(const Dims &d, const void *x, const void *B, const void *dt,
                                   const float *A, void *dH, float2 *gamma, float *u, float *v,
                                   float2 *anchor, const CsPlan &plan, int *err,
                                   cudaStream_t st);

// Output pass, y from x, B, C, dt, A, D and the bf16 per-chunk states, by
// one of two kernels with an explicit number of heads per CTA.
// fwd_scan: any shape, H heads per CTA.
// fwd_scan_chunk: C B^T of a whole chunk (fwd_scan_chunk_supported: P = 64,
// S in {64, 128}, T in {128, 256}) or, split, of one 128-row tile of a chunk
// (fwd_scan_chunk_split_supported: P = 64, S up to 256, T in {128, 256})
// shared by a slice of hs heads.
// fwd_scan_heads(d) and fwd_scan_chunk_heads(d, split) are the cost-model
// choices; the _ok functions say which values a launch accepts.
bool fwd_scan_chunk_supported(const Dims &d);
bool fwd_scan_chunk_split_supported(const Dims &d);
int fwd_scan_chunk_heads(const Dims &d, bool split);
bool fwd_scan_heads_ok(const Dims &d, int H);
bool fwd_scan_chunk_heads_ok(const Dims &d, int hs, bool split);
cudaError_t launch_fwd_scan(const Dims &d, const void *x, const void *B, const void *C,
                            const void *dt, const float *A, const void *states, const float *D,
                            void *y, int H, int *err, cudaStream_t st);
cudaError_t launch_fwd_scan_chunk(const Dims &d, const void *x, const void *B, const void *C,
                                  const void *dt, const float *A, const void *states,
                                  const float *D, void *y, int hs, bool split, int *err,
                                  cudaStream_t st);

// fwd_out: the output pass with the decay factored about one anchor per
// chunk and head, so that the masked C B^T of a chunk is shared unchanged by
// a slice of hs heads (P = 64, S a multiple of 64 up to 256, T in {128,
// 256}).
bool fwd_out_supported(const Dims &d);
bool fwd_out_heads_ok(const Dims &d, int hs);
int fwd_out_heads(const Dims &d);  // the cost-model choice
cudaError_t launch_fwd_out(const Dims &d, const void *x, const void *B, const void *C,
                           const void *dt, const float *A, const void *states, const float *D,
                           const float *u, const float *v, const float2 *anchor, void *y,
                           int hs, int *err, cudaStream_t st);

// fwd_out_tf32: the output pass for fp32 I/O (kind::tf32), one 128-row tile
// of a chunk and a slice of hs heads per CTA, the masked C B^T of the tile
// shared by the slice's heads with the decay factored about one anchor per
// chunk and head (P = 64, S a multiple of 32 up to 256, T in {128, 256}).
// It reads G (fp32, log2 units, [b, nh, nc * T]) and the fp32 start states
// [b, nh, nc, P, S] times 2^alpha_k rounded to tf32 (state_passing with
// tf32_out).
bool fwd_out_tf32_supported(const Dims &d);
bool fwd_out_tf32_heads_ok(const Dims &d, int hs);
int fwd_out_tf32_heads(const Dims &d);  // the cost-model choice
cudaError_t launch_fwd_out_tf32(const Dims &d, const float *x, const float *B, const float *C,
                                const float *dt, const float *G, const float *states,
                                const float *D, float *y, int hs, int *err, cudaStream_t st);

// fwd_chunk_state_tf32: the chunk jump terms for fp32 I/O (kind::tf32),
// dstates [b, nh, nc, P, S] fp32 from x, B, dt and A, writing the in-chunk
// cumsums G (fp32, log2 units, [b, nh, nc * T]) it forms on the way; P = 64,
// S a multiple of 64, T in {128, 256}.
bool fwd_chunk_state_tf32_supported(const Dims &d);
cudaError_t launch_fwd_chunk_state_tf32(const Dims &d, const float *x, const float *B,
                                        const float *dt, const float *A, float *G,
                                        float *dstates, int *err, cudaStream_t st);

// Heads per CTA of fwd_scan: the largest divisor of nheads/ngroups that is
// at most 4 and keeps heads * P <= 256 tensor-memory columns.
inline int fwd_scan_heads(const Dims &d) {
  const int hmax = (int)std::min<int64_t>(4, 256 / d.P);
  for (int h = hmax; h > 1; --h)
    if (d.hpg % h == 0) return h;
  return 1;
}

// Launch plan of the whole bf16 forward path (the public ssd_plan): the
// chunk-jump plan, and the output kernel (0 = fwd_scan, 1 = fwd_scan_chunk,
// 2 = fwd_scan_chunk with one row tile per CTA, 3 = fwd_out) with its heads
// per CTA.
struct FwdPlan {
  CsPlan cs;
  int scan_kernel, scan_heads;
};
FwdPlan fwd_default_plan(const Dims &d);
// Valid chunk-jump plans and output-kernel plans (as FwdPlan with only the
// relevant fields meaningful), appended to the vectors.
void fwd_cs_candidates(const Dims &d, std::vector<CsPlan> *out);
void fwd_scan_candidates(const Dims &d, std::vector<FwdPlan> *out);
bool fwd_plan_ok(const Dims &d, const FwdPlan &p);

}  // namespace ssd
