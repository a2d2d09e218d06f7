// Step 1: chunk-local cumulative sum of a_t = A[h] dt_t, scaled by log2(e).
//
// "Accelerating Mamba-2 with High-Performance Forward Pass Kernels in NVIDIA
// CUDA Tile", section "Kernel 1: Computing cumulative sums": the sum restarts
// at every chunk, is inclusive, and is stored times log2(e) so that later
// steps take exp2.  The partial last chunk reads dt = 0 past the end.
//
// Layout change: dt is [b, L, nh] (heads fastest) while G is [b, nh, nc*T]
// (tokens fastest), so each block stages a T x 32-head tile in shared memory
// (coalesced along heads), scans each head's column with one warp, and
// writes it back coalesced along tokens.  One read of dt, one write of G.
#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr int kHeadsPerBlock = 32;
constexpr int kThreads = 256;

template <typename IO, int T>
__global__ void __launch_bounds__(kThreads)
chunk_cumsum_kernel(const IO *__restrict__ dt, const float *__restrict__ A,
                    float *__restrict__ G, int64_t L, int64_t nh, int64_t nc, int64_t nb,
                    int *err) {
  constexpr int kPerLane = T / 32;
  __shared__ float tile[T][kHeadsPerBlock + 1];
  const int64_t k = blockIdx.x;
  const int64_t h_base = (int64_t)blockIdx.y * kHeadsPerBlock;
  const int64_t b = blockIdx.z;
  const int tid = threadIdx.x;

  // a = A * dt, zero past the end of the sequence and past the last head.
  for (int idx = tid; idx < T * kHeadsPerBlock; idx += kThreads) {
    const int t = idx / kHeadsPerBlock, hh = idx % kHeadsPerBlock;
    const int64_t tok = k * T + t, h = h_base + hh;
    float a = 0.f;
    if (tok < L && h < nh) {
      const int64_t i = (b * L + tok) * nh + h;
      if (SSD_IN_BOUNDS(i >= 0 && i < nb * L * nh, err, 1)) a = A[h] * ld_io(dt + i);
    }
    tile[t][hh] = a;
  }
  __syncthreads();

  const int warp = tid / 32, lane = tid % 32;
  for (int hh = warp; hh < kHeadsPerBlock; hh += kThreads / 32) {
    const int64_t h = h_base + hh;
    if (h >= nh) break;
    // Each lane owns kPerLane consecutive tokens: serial scan, then a warp
    // scan of the lane totals.
    float v[kPerLane];
    float run = 0.f;
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
      run += tile[lane * kPerLane + i][hh];
      v[i] = run;
    }
    float incl = run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    const float excl = incl - run;
    const int64_t o = ((b * nh + h) * nc + k) * T + lane * kPerLane;
    if (!SSD_IN_BOUNDS(o >= 0 && o + kPerLane <= nb * nh * nc * T, err, 2)) continue;
    float *out = G + o;
#pragma unroll
    for (int i = 0; i < kPerLane; i += 2) {
      float2 w;
      w.x = (v[i] + excl) * kLog2e;
      w.y = (v[i + 1] + excl) * kLog2e;
      *reinterpret_cast<float2 *>(out + i) = w;
    }
  }
}

template <typename IO>
cudaError_t launch_t(const Dims &d, const void *dt, const float *A, float *G, int *err,
                     cudaStream_t st) {
  dim3 grid((unsigned)d.nc, (unsigned)((d.nh + kHeadsPerBlock - 1) / kHeadsPerBlock),
            (unsigned)d.b);
  const IO *p = static_cast<const IO *>(dt);
  switch (d.T) {
    case 64: chunk_cumsum_kernel<IO, 64><<<grid, kThreads, 0, st>>>(p, A, G, d.L, d.nh, d.nc, d.b, err); break;
    case 128: chunk_cumsum_kernel<IO, 128><<<grid, kThreads, 0, st>>>(p, A, G, d.L, d.nh, d.nc, d.b, err); break;
    default: chunk_cumsum_kernel<IO, 256><<<grid, kThreads, 0, st>>>(p, A, G, d.L, d.nh, d.nc, d.b, err); break;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chunk_cumsum(const Dims &d, ssd_dtype io, const void *dt,
                                const float *A, float *G, int *err, cudaStream_t st) {
  return io == SSD_BF16 ? launch_t<__nv_bfloat16>(d, dt, A, G, err, st)
                        : launch_t<float>(d, dt, A, G, err, st);
}

}  // namespace ssd
