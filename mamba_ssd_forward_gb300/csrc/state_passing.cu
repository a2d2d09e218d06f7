// Step 3: the sequential pass over chunks (the loop of the page's
// fwd_pass_state, "Kernel 2"), given every chunk's jump term:
//
//   h = h0;  for k: states[k] = h;  h = exp2(G_last,k) h + dstates[k]
//   final_state = h
//
// A bandwidth kernel: each thread owns four consecutive elements of one
// (batch, head) state and walks the chunks; one read of dstates, one write
// of states.  The chunks go in groups of eight, the next group's loads in
// flight while the current group is consumed; the CTA's (decay, scale) pairs
// are formed once per 256 chunks in shared memory.  Launched with
// programmatic stream serialisation: it waits on the device before reading
// what the chunk-state step wrote.
// With tf32_out (the fp32 forward, whose output kernel fwd_out_tf32 reads
// the stored states as tf32 MMA operands with the decay factored about
// alpha_k = rint(G_last,k / 2)) each stored state is the carried state times
// 2^alpha_k (alpha_k = 0 when the chunk decays by more than 2^-180; a power
// of two, so exact), rounded to tf32 (nearest); the carried state and the
// final state stay unscaled fp32.
// With reverse (the backward pass) the chunks are walked from the last to
// the first: from h0 = dL/dfinal_state it stores R_k = dL/dh_{k+1} for every
// chunk and leaves R_{-1} = dL/dh0 in final_state, R_{k-1} = exp2(G_last,k)
// R_k + dstates[k] (dstates holding the adjoint's jump terms).
// With chunk_major the stored states are laid out [b, nc, nh, P, S], so that
// the heads of a group at one chunk form one matrix (the backward's GEMMs).
#include "tc_common.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 256;
constexpr int kDepth = 8;  // chunks per prefetch group

__global__ void __launch_bounds__(kThreads)
state_passing_kernel(const float4 *__restrict__ dstates,
                     const float *__restrict__ G, const float4 *__restrict__ h0,
                     float4 *__restrict__ states, float4 *__restrict__ final_state,
                     int64_t ps4, int64_t nc, int64_t T, int64_t nbh, int tf32_out,
                     int reverse, int64_t cm_nh, int *err) {
  __shared__ float2 gsm[256];  // per chunk: decay, stored-state scale
  // every index below lies in [0, nbh nc ps4) (states, dstates), [0, nbh
  // ps4) (h0, final_state) or [0, nbh nc T) (G) when bh < nbh and e < ps4; a
  // thread past the state (or failing the check) works on element 0 without
  // storing, so that it still takes part in the barriers
  const bool ok = SSD_IN_BOUNDS((int64_t)blockIdx.y < nbh, err, 10);
  const int64_t bh = ok ? blockIdx.y : 0;
  const int64_t ex = (int64_t)blockIdx.x * kThreads + threadIdx.x;  // float4 index in P*S
  const bool live = ok && ex < ps4;
  const int64_t e = live ? ex : 0;
  ptx::griddep_launch_dependents();  // the output pass may be scheduled now
  // dstates and G come from the preceding kernels (and h0 may too, on the
  // step-wise path)
  ptx::griddep_wait();
  float4 h = h0 ? h0[bh * ps4 + e] : make_float4(0.f, 0.f, 0.f, 0.f);
  const float *Gbh = G + bh * nc * T;
  const float4 *dsrc = dstates + bh * nc * ps4 + e;
  // stored state of chunk k: [b, nh, nc, P, S], or chunk-major [b, nc, nh,
  // P, S] when cm_nh (= nh) is set
  auto dst_row = [&](int64_t k) {
    return cm_nh ? ((bh / cm_nh * nc + k) * cm_nh + bh % cm_nh) * ps4 : (bh * nc + k) * ps4;
  };
  float4 *sdst = states + e;
  // the chunk visited at step k: k itself, or nc - 1 - k walking backwards
  auto ck = [&](int64_t k) { return reverse ? nc - 1 - k : k; };
  float4 cur[kDepth], nxt[kDepth];
#pragma unroll
  for (int i = 0; i < kDepth; ++i)
    if (i < nc) cur[i] = dsrc[ck(i) * ps4];
  for (int64_t k0 = 0; k0 < nc; k0 += kDepth) {
    if ((k0 & 255) == 0) {
      // the next 256 chunks' decays and stored-state scales.  With tf32_out
      // the scale is 2^alpha, the factored output pass's anchor (the same
      // rule as fwd_out_tf32; a power of two, so exact), else 1.
      __syncthreads();
      if (k0 + threadIdx.x < nc) {
        const float Glast = Gbh[ck(k0 + threadIdx.x) * T + T - 1];
        float sc = 1.f;
        if (tf32_out) {
          const int alpha = -Glast <= 180.f ? (int)rintf(0.5f * Glast) : 0;
          sc = __int_as_float((127 + alpha) << 23);  // 2^alpha, alpha in [-90, 0]
        }
        gsm[threadIdx.x] = make_float2(exp2f(Glast), sc);
      }
      __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < kDepth; ++i)
      if (k0 + kDepth + i < nc) nxt[i] = dsrc[ck(k0 + kDepth + i) * ps4];
#pragma unroll
    for (int i = 0; i < kDepth; ++i)
      if (k0 + i < nc) {
        const float2 g = gsm[(k0 + i) & 255];
        if (live) {
          sdst[dst_row(ck(k0 + i))] =
              tf32_out ? make_float4(__uint_as_float(to_tf32(g.y * h.x)),
                                     __uint_as_float(to_tf32(g.y * h.y)),
                                     __uint_as_float(to_tf32(g.y * h.z)),
                                     __uint_as_float(to_tf32(g.y * h.w)))
                       : h;
        }
        h.x = fmaf(g.x, h.x, cur[i].x);
        h.y = fmaf(g.x, h.y, cur[i].y);
        h.z = fmaf(g.x, h.z, cur[i].z);
        h.w = fmaf(g.x, h.w, cur[i].w);
      }
#pragma unroll
    for (int i = 0; i < kDepth; ++i) cur[i] = nxt[i];
  }
  if (final_state && live) final_state[bh * ps4 + e] = h;
}

}  // namespace

cudaError_t launch_state_passing(const Dims &d, const float *dstates,
                                 const float *G, const float *h0,
                                 float *states, float *final_state, int *err,
                                 cudaStream_t st, bool tf32_out, bool reverse,
                                 bool chunk_major) {
  const int64_t ps4 = d.P * d.S / 4;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((ps4 + kThreads - 1) / kThreads), (unsigned)(d.b * d.nh));
  cfg.blockDim = dim3(kThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, state_passing_kernel, reinterpret_cast<const float4 *>(dstates),
                            G, reinterpret_cast<const float4 *>(h0),
                            reinterpret_cast<float4 *>(states),
                            reinterpret_cast<float4 *>(final_state), ps4, d.nc, d.T,
                            d.b * d.nh, tf32_out ? 1 : 0, reverse ? 1 : 0,
                            chunk_major ? d.nh : (int64_t)0, err);
}

}  // namespace ssd
