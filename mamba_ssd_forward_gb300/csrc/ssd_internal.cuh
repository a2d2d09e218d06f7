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

// Debug-bounds builds (compiled with -DSSD_DEBUG_BOUNDS; the release library
// never is): SSD_IN_BOUNDS(cond, err, site) evaluates `cond`, the index of a
// global access checked against its buffer's extent; a false condition
// records kErrBoundsBase + site in the error word `err` (when not null and
// still clear) and the caller skips the access.  In release builds it is the
// constant true and `cond` is not evaluated.  The host reports such a code as
// SSD_ERR_BOUNDS.
constexpr int kErrBoundsBase = 2000;
#ifdef SSD_DEBUG_BOUNDS
__device__ __forceinline__ bool in_bounds_check(bool ok, int *err, int site) {
  if (!ok && err) atomicCAS(err, 0, kErrBoundsBase + site);
  return ok;
}
#define SSD_IN_BOUNDS(cond, err, site) (::ssd::in_bounds_check((cond), (err), (site)))
#else
#define SSD_IN_BOUNDS(cond, err, site) (true)
#endif

// Element access for the two I/O types.
__device__ __forceinline__ float ld_io(const float *p) { return *p; }
__device__ __forceinline__ float ld_io(const __nv_bfloat16 *p) {
  return __bfloat162float(*p);
}
__device__ __forceinline__ void st_io(float *p, float v) { *p = v; }
__device__ __forceinline__ void st_io(__nv_bfloat16 *p, float v) {
  *p = __float2bfloat16_rn(v);
}

// Address of the library-wide device error word (current device), used by
// the calls that have no workspace of their own (the step-wise entry points,
// ssd_forward_noalloc, the self-test by default); kernels that give up a
// bounded wait write a nonzero code there.  Null if the look-up failed.
int *device_error_word();
// Copy the error word at `word` (device) to *code and clear it; synchronises
// `st`.
cudaError_t read_and_clear_error(int *word, cudaStream_t st, int *code);
// The status an error-word code stands for: 0 -> SSD_OK, a debug-bounds
// code (kErrBoundsBase and up) -> SSD_ERR_BOUNDS, any other -> the code of a
// bounded wait that gave up, SSD_ERR_TIMEOUT.
inline ssd_status status_of_error_code(int code) {
  if (code == 0) return SSD_OK;
  return code >= kErrBoundsBase ? SSD_ERR_BOUNDS : SSD_ERR_TIMEOUT;
}

// SM count of the current device, looked up once per device and cached
// (race-free under concurrent callers).
int sm_count();

// Workspace header of ssd_forward and the host-buffer calls: the first
// SSD_WS_HEADER_BYTES bytes.  Word 0 is the call's error word.
constexpr size_t kWsHeader = SSD_WS_HEADER_BYTES;

// Argument checks of ssd_forward (dims, dtype and tensor pointers; not the
// workspace), with the validated dims in *out.
ssd_status check_forward_args(const ssd_dims *dims, ssd_dtype dtype, const void *x,
                              const void *dt, const float *A, const void *B, const void *C,
                              const float *D, const float *h0, const void *y,
                              const float *final_state, Dims *out);
// The forward pass behind ssd_forward, ssd_forward_ex and ssd_forward_profiled:
// plan NULL = the default plan; err NULL = the workspace's own error word;
// events / n_events / n_launches as for ssd_forward_profiled.
ssd_status forward_impl(const ssd_dims *dims, ssd_dtype dtype, const void *x, const void *dt,
                        const float *A, const void *B, const void *C, const float *D,
                        const float *h0, void *y, float *final_state, void *workspace,
                        size_t ws_bytes, const ssd_plan *plan, int *err, cudaStream_t st,
                        void *const *events, int n_events, int *n_launches);

// SSD_OK if `plan` (NULL = the default) can run these dims and dtype, else
// the code ssd_forward_ex would return for it.
ssd_status plan_status(const ssd_dims *dims, ssd_dtype dtype, const ssd_plan *plan);

// Launchers (one per step).  Each enqueues its kernel(s) on `st` and returns
// the cudaGetLastError() of the launch; `err` is the device error word its
// kernels report to.
cudaError_t launch_chunk_cumsum(const Dims &d, ssd_dtype io, const void *dt,
                                const float *A, float *G, int *err, cudaStream_t st);
cudaError_t launch_chunk_state(const Dims &d, ssd_dtype io, const void *x,
                               const void *B, const void *dt, const float *G,
                               float *dstates, int *err, cudaStream_t st);
cudaError_t launch_state_passing(const Dims &d, const float *dstates,
                                 const float *G, const float *h0,
                                 float *states, float *final_state, int *err,
                                 cudaStream_t st, bool tf32_out = false, bool reverse = false,
                                 bool chunk_major = false);
cudaError_t launch_chunk_scan(const Dims &d, ssd_dtype io, const void *x,
                              const void *B, const void *C, const void *dt,
                              const float *G, const float *states,
                              const float *D, void *y, int *err, cudaStream_t st);

// Single-token decode step (decode_step.cu).
cudaError_t launch_decode_step(int64_t b, int64_t nh, int64_t P, int64_t S, int64_t ng,
                               ssd_dtype io, const void *x, const void *dt, const float *A,
                               const void *B, const void *C, const float *D, float *state,
                               void *y, int *err, cudaStream_t st);

// bf16 <-> fp32 conversion of up to five tensors in one launch (the bf16
// I/O of ssd_backward): to_bf16 = 0 reads bf16 and writes fp32, 1 the
// reverse; n elements per segment, 16-byte aligned pointers.
struct BwdConvert {
  struct Seg {
    const void *src;
    void *dst;
    int64_t n;
  } seg[5];
  int nseg, to_bf16;
};
cudaError_t launch_bwd_convert(const BwdConvert &a, cudaStream_t st);

// Backward pass for fp32 I/O (bwd.cu), CUDA cores.  bwd_supported: P = 64,
// S in {64, 128, 256}, T a multiple of 32 up to 256.  Shapes (fp32):
// dR, R [b, nh, nc, P, S]; dB, dC [b, L, ng, S]; qB, dG, gyx [b, nh, nc*T];
// part float2 [b, nh, nc].
bool bwd_supported(const Dims &d);
// the backward's GEMMs on the tensor cores in split TF32 (bwd_gemm.cu),
// nprod (1 or 2) products per launch: product i reads Ai and Si and writes
// outi.  R and H: the start states, chunk-major [b, nc, nh, P, S].
//   mode 2, jump terms: A = x~ or gy~, S = B or C ([b, L, ng, S]), out
//     [b, nh, nc, P, S] = per chunk and head sum_t A_t^T S_t;
//   mode 0, before bwd_main: A = B or C, S = R or H, out = dxS = B R^T or
//     ysmS = C H^T per (batch, chunk, group), in the layout of x;
//   mode 1, after it: A = x~ or gy~, S = R or H, out = dB += x~ R or
//     dC += gy~ H;
//   mode 3, A = C, S = B: out = Kcb [b, ng, nc, T, T], c_i . B_j of every
//     chunk and group on and below the diagonal (128 x 128 token tiles).
bool bwd_state_gemm_supported(const Dims &d);
cudaError_t launch_bwd_gemm(const Dims &d, int mode, int nprod, const float *A0, const float *A1,
                            const float *S0, const float *S1, float *out0, float *out1, int *err,
                            cudaStream_t st);
// x~ = dt exp2(G_last - G_t) x and gy~ = exp2(G_t) gy, in the layout of x
cudaError_t launch_bwd_scale(const Dims &d, const float *x, const float *gy, const float *dt,
                             const float *G, float *xs, float *gys, int *err, cudaStream_t st);
// per (row tile, chunk, group): dx of its heads, the group's dB and dC
// in-chunk parts, and per token and head q . B, dL/dG, gy . x
cudaError_t launch_bwd_main(const Dims &d, const float *x, const float *dt, const float *B,
                            const float *C, const float *D, const float *gy, const float *G,
                            const float *dxS, const float *ysmS, const float *Kcb, float *dx,
                            float *dB, float *dC, float *qB, float *dG, float *gyx, int *err,
                            cudaStream_t st);
// ddt, and the per-chunk shares of dA and dD
cudaError_t launch_bwd_finish(const Dims &d, const float *dt, const float *A, const float *R,
                              const float *states, const float *final_state, const float *qB,
                              const float *dG, const float *gyx, float *ddt, float2 *part,
                              int *err, cudaStream_t st);
// heads of a group per bwd_main CTA are hpg / bwd_head_slices(d); with more
// than one slice bwd_main writes each slice's share of dB and dC (slice-major,
// [nslice, b, L, ng, S]) for bwd_reduce to add up
int bwd_head_slices(const Dims &d);
// dB, dC from the slices' shares sB, sC (when there are several slices),
// then dA, dD (nullable): every sum in a fixed order
cudaError_t launch_bwd_reduce(const Dims &d, const float *sB, const float *sC, float *dB,
                              float *dC, const float2 *part, float *dA, float *dD, int *err,
                              cudaStream_t st);

}  // namespace ssd
