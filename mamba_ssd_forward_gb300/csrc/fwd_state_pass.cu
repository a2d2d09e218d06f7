// Forward path, sequential pass over chunks (bf16 I/O): the loop of the
// page's fwd_pass_state ("Kernel 2" of "Accelerating Mamba-2 with
// High-Performance Forward Pass Kernels in NVIDIA CUDA Tile"), given every
// chunk's jump term and decay from fwd_chunk_state.cu:
//
//   h = h0;  for k:  states[k] = h;  h = gamma[k] h + dH[k];   final = h
//
// A bandwidth kernel: each thread owns eight consecutive elements of one
// (batch, head) state in the [S][P] layout, keeps them in fp32 registers, and
// walks the chunks with the next group of eight chunks' loads in flight.  dH
// and the stored states are bf16 [b, nh, nc, S, P]; h0 and the final state
// are fp32 [b, nh, P, S] (the public layout).  gamma holds per chunk the
// decay and the scale of its stored start state (1, or 2^alpha_k for the
// factored output pass: a power of two, so the scaling is exact); the
// carried state stays unscaled.
#include "fwd.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 256;
constexpr int kDepth = 8;  // chunks per prefetch group

// two CTAs per SM (at most 128 registers a thread)
__global__ void __launch_bounds__(kThreads, 2)
fwd_state_pass_bf16(const uint4 *__restrict__ dH, const float2 *__restrict__ gamma,
                    const float *__restrict__ h0, uint4 *__restrict__ states,
                    float *__restrict__ final_state, int P, int S, int nc, int64_t nbh,
                    int *err) {
  // the CTA's (decay, scale) pairs, 256 chunks at a time
  __shared__ float2 gsm[256];
  const int n8 = S * P / 8;
  const int e8x = blockIdx.x * kThreads + threadIdx.x;
  // every index below lies in [0, nbh nc n8) (dH, states), [0, nbh nc)
  // (gamma) or [0, nbh P S) (h0, final state) when bh < nbh and e8 < n8; a
  // failed check works on element 0 of head 0 without storing, so that the
  // thread still takes part in the barriers
  const bool ok = SSD_IN_BOUNDS((int64_t)blockIdx.y < nbh, err, 30);
  const int64_t bh = ok ? blockIdx.y : 0;
  // threads past the state (a partial last CTA) take part in the barriers
  // only, working on element 0 without storing
  const bool live = e8x < n8 && ok;
  const int e8 = live ? e8x : 0;
  const int s = (e8 * 8) / P, p0 = (e8 * 8) % P;
  ptx::griddep_launch_dependents();  // the output pass may be scheduled now
  float h[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) h[i] = h0 ? h0[(bh * P + p0 + i) * S + s] : 0.f;
  ptx::griddep_wait();  // dH and gamma come from the preceding kernel
  const uint4 *src = dH + bh * nc * n8 + e8;
  uint4 *dst = states + bh * nc * n8 + e8;
  const float2 *gm = gamma + bh * nc;
  // Two groups of kDepth chunks: the next group's loads are issued before the
  // current group is consumed, so up to 2 kDepth 16-byte loads are in flight.
  // Every thread of the CTA works on the same (batch, head), so the group's
  // per-chunk decays and anchors are the same for all: they are loaded
  // together at the start of the group and come from L1.
  uint4 cur[kDepth], nxt[kDepth];
#pragma unroll
  for (int i = 0; i < kDepth; ++i)
    if (i < nc) cur[i] = src[(int64_t)i * n8];
  for (int k0 = 0; k0 < nc; k0 += kDepth) {
    if ((k0 & 255) == 0) {
      // the next 256 chunks' (decay, scale) pairs into shared memory
      __syncthreads();
      if (k0 + (int)threadIdx.x < nc) gsm[threadIdx.x] = gm[k0 + threadIdx.x];
      __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < kDepth; ++i)
      if (k0 + kDepth + i < nc) nxt[i] = src[(int64_t)(k0 + kDepth + i) * n8];
#pragma unroll
    for (int i = 0; i < kDepth; ++i)
      if (k0 + i < nc) {
        const float2 g = gsm[(k0 + i) & 255];  // (decay, stored-state scale)
        float hs[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) hs[j] = g.y * h[j];
        if (live) dst[(int64_t)(k0 + i) * n8] = pack_io16(hs, (__nv_bfloat16 *)nullptr);
        float d[8];
        unpack16(cur[i], d, (__nv_bfloat16 *)nullptr);
#pragma unroll
        for (int j = 0; j < 8; ++j) h[j] = fmaf(g.x, h[j], d[j]);
      }
#pragma unroll
    for (int i = 0; i < kDepth; ++i) cur[i] = nxt[i];
  }
  if (final_state && live) {
#pragma unroll
    for (int i = 0; i < 8; ++i) final_state[(bh * P + p0 + i) * S + s] = h[i];
  }
}

}  // namespace

cudaError_t launch_fwd_state_pass(const Dims &d, const void *dH, const float2 *gamma,
                                  const float *h0, void *states, float *final_state, int *err,
                                  cudaStream_t st) {
  const int n8 = (int)(d.S * d.P / 8);
  dim3 grid((unsigned)((n8 + kThreads - 1) / kThreads), (unsigned)(d.b * d.nh));
  // programmatic stream serialisation: this kernel may start while
  // fwd_chunk_state finishes; it waits on the device before reading dH
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fwd_state_pass_bf16, static_cast<const uint4 *>(dH), gamma,
                            h0, static_cast<uint4 *>(states), final_state, (int)d.P,
                            (int)d.S, (int)d.nc, (int64_t)(d.b * d.nh), err);
}

}  // namespace ssd
