// Single-token decode step: one token of the recurrence of "Accelerating
// Mamba-2 with High-Performance Forward Pass Kernels in NVIDIA CUDA Tile",
// section "Mamba-2 architecture", applied to every (batch, head) state:
//
//   h = exp(A dt) h + (dt x) (outer) B          (P x S, fp32, in place)
//   y = h c + D x                                (output from the new state)
//
// A bandwidth kernel: the state is read and written once (8 P S bytes per
// head); x, dt, B and C are a few hundred bytes.  One CTA per (batch, head)
// and, when there are few of those (kSliced), per 32-row slice of P too, so
// that enough CTAs keep the memory system busy; each warp takes rows
// p = p_lo + warp, + 8, ..., four at a time with every load issued first;
// each lane four consecutive state columns of every 128-wide slice of S,
// with B and C in registers.  The row's dot product with C is a warp
// reduction.
#include <type_traits>

#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr int kWarps = 8;
constexpr int kMaxSlices = 8;  // S <= 1024
constexpr int kRows = 4;       // rows per warp in flight
constexpr int kSliceRows = kWarps * kRows;  // rows of P per CTA when sliced

template <typename T>
struct type_tag {
  using type = T;
};

__device__ __forceinline__ void load4(const float *p, float (&v)[4]) {
  const float4 f = *reinterpret_cast<const float4 *>(p);
  v[0] = f.x;
  v[1] = f.y;
  v[2] = f.z;
  v[3] = f.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16 *p, float (&v)[4]) {
  const uint2 u = *reinterpret_cast<const uint2 *>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
  const float2 c = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
  v[0] = a.x;
  v[1] = a.y;
  v[2] = c.x;
  v[3] = c.y;
}

// kNsl: 128-wide slices of S the kernel handles (1, 2, or up to kMaxSlices),
// a compile-time bound so that B and C of small dstates take few registers
// and four CTAs fit on an SM
template <typename IO, bool kSliced, int kNsl>
__global__ void __launch_bounds__(kWarps * 32, kNsl <= 2 ? 4 : 2)
decode_step_kernel(const IO *__restrict__ x, const IO *__restrict__ dt,
                   const float *__restrict__ A, const IO *__restrict__ B,
                   const IO *__restrict__ C, const float *__restrict__ D,
                   float *__restrict__ state, IO *__restrict__ y, int nh, int P, int S, int hpg,
                   int ng, int64_t nbh, int *err) {
  const int64_t bh = blockIdx.x;
  const int64_t bi = bh / nh;
  const int h = (int)(bh % nh);
  const int g = h / hpg;
  // x, dt, y and the state are indexed by bh < nbh, B and C by bi ng + g
  if (!SSD_IN_BOUNDS(bh < nbh && g < ng, err, 20)) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nsl = (S + 127) / 128;
  const float dtv = ld_io(dt + bh);
  const float decay = expf(A[h] * dtv);
  const float Dh = D ? D[h] : 0.f;
  const IO *Brow = B + (bi * ng + g) * S;
  const IO *Crow = C + (bi * ng + g) * S;
  float Bv[kNsl][4], Cv[kNsl][4];
#pragma unroll
  for (int k = 0; k < kNsl; ++k) {
    const int s0 = k * 128 + lane * 4;
    if (k < nsl && s0 < S && SSD_IN_BOUNDS(s0 + 4 <= S, err, 21)) {
      load4(Brow + s0, Bv[k]);
      load4(Crow + s0, Cv[k]);
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) Bv[k][e] = Cv[k][e] = 0.f;
    }
  }
  float *hb = state + bh * (int64_t)P * S;
  // this CTA's rows [p_lo, p_hi), four per warp at a time, every state load
  // issued before the math
  const int p_lo = kSliced ? (int)blockIdx.y * kSliceRows : 0;
  const int p_hi = kSliced ? min(P, p_lo + kSliceRows) : P;
  for (int p0 = p_lo + warp; p0 < p_hi; p0 += kWarps * kRows) {
    float u[kRows], xp[kRows], acc[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      const int p = p0 + r * kWarps;
      xp[r] = p < p_hi ? ld_io(x + bh * P + p) : 0.f;
      u[r] = dtv * xp[r];
      acc[r] = 0.f;
    }
#pragma unroll
    for (int k = 0; k < kNsl; ++k) {
      const int s0 = k * 128 + lane * 4;
      if (k >= nsl || s0 >= S || !SSD_IN_BOUNDS(s0 + 4 <= S, err, 22)) continue;
      float4 hv[kRows];
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        const int p = p0 + r * kWarps;
        if (p < p_hi) hv[r] = *reinterpret_cast<const float4 *>(hb + (int64_t)p * S + s0);
      }
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        const int p = p0 + r * kWarps;
        if (p >= p_hi) continue;
        hv[r].x = fmaf(decay, hv[r].x, u[r] * Bv[k][0]);
        hv[r].y = fmaf(decay, hv[r].y, u[r] * Bv[k][1]);
        hv[r].z = fmaf(decay, hv[r].z, u[r] * Bv[k][2]);
        hv[r].w = fmaf(decay, hv[r].w, u[r] * Bv[k][3]);
        *reinterpret_cast<float4 *>(hb + (int64_t)p * S + s0) = hv[r];
        acc[r] = fmaf(hv[r].x, Cv[k][0], acc[r]);
        acc[r] = fmaf(hv[r].y, Cv[k][1], acc[r]);
        acc[r] = fmaf(hv[r].z, Cv[k][2], acc[r]);
        acc[r] = fmaf(hv[r].w, Cv[k][3], acc[r]);
      }
    }
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], off);
      const int p = p0 + r * kWarps;
      if (lane == 0 && p < p_hi) st_io(y + bh * P + p, fmaf(Dh, xp[r], acc[r]));
    }
  }
}

}  // namespace

cudaError_t launch_decode_step(int64_t b, int64_t nh, int64_t P, int64_t S, int64_t ng,
                               ssd_dtype io, const void *x, const void *dt, const float *A,
                               const void *B, const void *C, const float *D, float *state,
                               void *y, int *err, cudaStream_t st) {
  // slice P when the (batch, head) pairs alone would leave SMs idle
  // (measured: 96 pairs 10.1 -> 9.4 us; 5120 pairs are faster unsliced)
  const bool sliced = b * nh < 4 * (int64_t)sm_count();
  const dim3 grid((unsigned)(b * nh), sliced ? (unsigned)((P + kSliceRows - 1) / kSliceRows) : 1u);
  const int hpg = (int)(nh / ng);
  const int nsl = (int)((S + 127) / 128);
  auto launch = [&](auto io_c, auto sliced_c, auto nsl_c) {
    using IO = typename decltype(io_c)::type;
    decode_step_kernel<IO, decltype(sliced_c)::value, decltype(nsl_c)::value>
        <<<grid, kWarps * 32, 0, st>>>(
            static_cast<const IO *>(x), static_cast<const IO *>(dt), A,
            static_cast<const IO *>(B), static_cast<const IO *>(C), D, state,
            static_cast<IO *>(y), (int)nh, (int)P, (int)S, hpg, (int)ng, b * nh, err);
  };
  auto by_slices = [&](auto io_c, auto sliced_c) {
    if (nsl == 1)
      launch(io_c, sliced_c, std::integral_constant<int, 1>{});
    else if (nsl == 2)
      launch(io_c, sliced_c, std::integral_constant<int, 2>{});
    else
      launch(io_c, sliced_c, std::integral_constant<int, kMaxSlices>{});
  };
  auto by_sliced = [&](auto io_c) {
    if (sliced)
      by_slices(io_c, std::true_type{});
    else
      by_slices(io_c, std::false_type{});
  };
  if (io == SSD_BF16)
    by_sliced(type_tag<__nv_bfloat16>{});
  else
    by_sliced(type_tag<float>{});
  return cudaGetLastError();
}

}  // namespace ssd
