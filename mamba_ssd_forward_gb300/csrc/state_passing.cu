// Step 3: the sequential pass over chunks (the loop of the page's
// fwd_pass_state, "Kernel 2"), given every chunk's jump term:
//
//   h = h0;  for k: states[k] = h;  h = exp2(G_last,k) h + dstates[k]
//   final_state = h
//
// A bandwidth kernel: each thread owns four consecutive elements of one
// (batch, head) state and walks the chunks; one read of dstates, one write
// of states.  The loads of the next chunk's dstates are issued before the
// current chunk's stores so that each thread keeps two loads in flight.
// With tf32_out (the fp32 forward, whose output kernel fwd_out_tf32 reads
// the stored states as tf32 MMA operands with the decay factored about
// alpha_k = rint(G_last,k / 2)) each stored state is the carried state times
// 2^alpha_k (alpha_k = 0 when the chunk decays by more than 2^-180; a power
// of two, so exact), rounded to tf32 (nearest); the carried state and the
// final state stay unscaled fp32.
#include "tc_common.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
state_passing_kernel(const float4 *__restrict__ dstates,
                     const float *__restrict__ G, const float4 *__restrict__ h0,
                     float4 *__restrict__ states, float4 *__restrict__ final_state,
                     int64_t ps4, int64_t nc, int64_t T, int64_t nbh, int tf32_out,
                     int *err) {
  const int64_t bh = blockIdx.y;
  const int64_t e = (int64_t)blockIdx.x * kThreads + threadIdx.x;  // float4 index in P*S
  if (e >= ps4) return;
  // every index below lies in [0, nbh nc ps4) (states, dstates), [0, nbh
  // ps4) (h0, final_state) or [0, nbh nc T) (G)
  if (!SSD_IN_BOUNDS(bh < nbh && e >= 0, err, 10)) return;
  float4 h = h0 ? h0[bh * ps4 + e] : make_float4(0.f, 0.f, 0.f, 0.f);
  const float *Gbh = G + bh * nc * T;
  const float4 *dsrc = dstates + bh * nc * ps4 + e;
  float4 *sdst = states + bh * nc * ps4 + e;
  float4 next = nc > 0 ? dsrc[0] : h;
  for (int64_t k = 0; k < nc; ++k) {
    const float4 cur = next;
    if (k + 1 < nc) next = dsrc[(k + 1) * ps4];
    const float Glast = Gbh[k * T + T - 1];
    const float decay = exp2f(Glast);
    if (tf32_out) {
      // the factored output pass's anchor (the same rule as fwd_out_tf32)
      const int alpha = -Glast <= 180.f ? (int)rintf(0.5f * Glast) : 0;
      const float sc = __int_as_float((127 + alpha) << 23);  // 2^alpha, alpha in [-90, 0]
      sdst[k * ps4] = make_float4(__uint_as_float(to_tf32(sc * h.x)),
                                  __uint_as_float(to_tf32(sc * h.y)),
                                  __uint_as_float(to_tf32(sc * h.z)),
                                  __uint_as_float(to_tf32(sc * h.w)));
    } else {
      sdst[k * ps4] = h;
    }
    h.x = fmaf(decay, h.x, cur.x);
    h.y = fmaf(decay, h.y, cur.y);
    h.z = fmaf(decay, h.z, cur.z);
    h.w = fmaf(decay, h.w, cur.w);
  }
  if (final_state) final_state[bh * ps4 + e] = h;
}

}  // namespace

cudaError_t launch_state_passing(const Dims &d, const float *dstates,
                                 const float *G, const float *h0,
                                 float *states, float *final_state, int *err,
                                 cudaStream_t st, bool tf32_out) {
  const int64_t ps4 = d.P * d.S / 4;
  dim3 grid((unsigned)((ps4 + kThreads - 1) / kThreads), (unsigned)(d.b * d.nh));
  state_passing_kernel<<<grid, kThreads, 0, st>>>(
      reinterpret_cast<const float4 *>(dstates), G,
      reinterpret_cast<const float4 *>(h0), reinterpret_cast<float4 *>(states),
      reinterpret_cast<float4 *>(final_state), ps4, d.nc, d.T, d.b * d.nh, tf32_out ? 1 : 0,
      err);
  return cudaGetLastError();
}

}  // namespace ssd
