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
// are fp32 [b, nh, P, S] (the public layout).
#include "fwd.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 256;
constexpr int kDepth = 8;  // chunks per prefetch group

__global__ void __launch_bounds__(kThreads)
fwd_state_pass_bf16(const uint4 *__restrict__ dH, const float *__restrict__ gamma,
                    const float *__restrict__ h0, uint4 *__restrict__ states,
                    float *__restrict__ final_state, int P, int S, int nc) {
  const int64_t bh = blockIdx.y;
  const int n8 = S * P / 8;
  const int e8 = blockIdx.x * kThreads + threadIdx.x;
  if (e8 >= n8) return;
  const int s = (e8 * 8) / P, p0 = (e8 * 8) % P;
  ptx::griddep_launch_dependents();  // the output pass may be scheduled now
  float h[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) h[i] = h0 ? h0[(bh * P + p0 + i) * S + s] : 0.f;
  ptx::griddep_wait();  // dH and gamma come from the preceding kernel
  const uint4 *src = dH + bh * nc * n8 + e8;
  uint4 *dst = states + bh * nc * n8 + e8;
  const float *gm = gamma + bh * nc;
  // Two groups of kDepth chunks: the next group's loads are issued before the
  // current group is consumed, so up to 2 kDepth 16-byte loads are in flight.
  uint4 cur[kDepth], nxt[kDepth];
  float gcur[kDepth], gnxt[kDepth];
#pragma unroll
  for (int i = 0; i < kDepth; ++i)
    if (i < nc) {
      cur[i] = src[(int64_t)i * n8];
      gcur[i] = gm[i];
    }
  for (int k0 = 0; k0 < nc; k0 += kDepth) {
#pragma unroll
    for (int i = 0; i < kDepth; ++i)
      if (k0 + kDepth + i < nc) {
        nxt[i] = src[(int64_t)(k0 + kDepth + i) * n8];
        gnxt[i] = gm[k0 + kDepth + i];
      }
#pragma unroll
    for (int i = 0; i < kDepth; ++i)
      if (k0 + i < nc) {
        dst[(int64_t)(k0 + i) * n8] = pack_io16(h, (__nv_bfloat16 *)nullptr);
        float d[8];
        unpack16(cur[i], d, (__nv_bfloat16 *)nullptr);
#pragma unroll
        for (int j = 0; j < 8; ++j) h[j] = fmaf(gcur[i], h[j], d[j]);
      }
#pragma unroll
    for (int i = 0; i < kDepth; ++i) {
      cur[i] = nxt[i];
      gcur[i] = gnxt[i];
    }
  }
  if (final_state) {
#pragma unroll
    for (int i = 0; i < 8; ++i) final_state[(bh * P + p0 + i) * S + s] = h[i];
  }
}

}  // namespace

cudaError_t launch_fwd_state_pass(const Dims &d, const void *dH, const float *gamma,
                                  const float *h0, void *states, float *final_state,
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
                            (int)d.S, (int)d.nc);
}

}  // namespace ssd
