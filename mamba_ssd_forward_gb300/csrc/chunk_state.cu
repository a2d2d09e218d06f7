// Step 2: the jump term of the chunk state update
//
//   dstates[b,h,k][p][s] = sum_{j in chunk k} w_j x[b,j,h,p] B[b,j,g,s],
//   w_j = exp2(G_last,k - G_j) dt_j
//
// ("Accelerating Mamba-2 with High-Performance Forward Pass Kernels in NVIDIA
// CUDA Tile", section "Mamba-2 architecture", the log-space jump formula
// h_{t+T} = exp(G_last) h_t + (exp(G_last - G) B)^T X, second term.)
//
// First-cut SIMT kernel: one block per (chunk, 64x64 state tile, head,
// batch); 256 threads, each accumulating a 4x4 patch over the chunk's tokens
// staged 32 at a time in shared memory.
#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = 64;
constexpr int kTok = 32;

template <typename IO>
__global__ void __launch_bounds__(kThreads)
chunk_state_simt(const IO *__restrict__ x, const IO *__restrict__ Bm,
                 const IO *__restrict__ dt, const float *__restrict__ G,
                 float *__restrict__ dstates, int64_t L, int64_t nh, int64_t P,
                 int64_t S, int64_t ng, int64_t T, int64_t nc) {
  __shared__ float xs[kTok][kTile];
  __shared__ float bs[kTok][kTile];
  const int64_t ptiles = (P + kTile - 1) / kTile, stiles = (S + kTile - 1) / kTile;
  int64_t r = blockIdx.x;
  const int64_t st = r % stiles;
  r /= stiles;
  const int64_t pt = r % ptiles;
  const int64_t k = r / ptiles;
  const int64_t h = blockIdx.y, b = blockIdx.z, g = h / (nh / ng);
  const float *Gc = G + ((b * nh + h) * nc + k) * T;
  const float Glast = Gc[T - 1];
  const int tid = threadIdx.x, tp = tid / 16, ts = tid % 16;

  float acc[4][4] = {};
  for (int64_t j0 = 0; j0 < T; j0 += kTok) {
    for (int idx = tid; idx < kTok * kTile; idx += kThreads) {
      const int jj = idx / kTile, c = idx % kTile;
      const int64_t tok = k * T + j0 + jj;
      const int64_t p = pt * kTile + c, s = st * kTile + c;
      float xv = 0.f, bv = 0.f;
      if (tok < L) {
        const float w = exp2f(Glast - Gc[j0 + jj]) * ld_io(dt + (b * L + tok) * nh + h);
        if (p < P) xv = w * ld_io(x + ((b * L + tok) * nh + h) * P + p);
        if (s < S) bv = ld_io(Bm + ((b * L + tok) * ng + g) * S + s);
      }
      xs[jj][c] = xv;
      bs[jj][c] = bv;
    }
    __syncthreads();
#pragma unroll 4
    for (int jj = 0; jj < kTok; ++jj) {
      float xv[4], bv[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        xv[q] = xs[jj][tp * 4 + q];
        bv[q] = bs[jj][ts * 4 + q];
      }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[a][c] = fmaf(xv[a], bv[c], acc[a][c]);
    }
    __syncthreads();
  }
  float *out = dstates + ((b * nh + h) * nc + k) * P * S;
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int64_t p = pt * kTile + tp * 4 + a;
    if (p >= P) continue;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int64_t s = st * kTile + ts * 4 + c;
      if (s < S) out[p * S + s] = acc[a][c];
    }
  }
}

}  // namespace

cudaError_t launch_chunk_state(const Dims &d, ssd_dtype io, const void *x,
                               const void *B, const void *dt, const float *G,
                               float *dstates, cudaStream_t st) {
  const int64_t tiles = ((d.P + kTile - 1) / kTile) * ((d.S + kTile - 1) / kTile);
  dim3 grid((unsigned)(d.nc * tiles), (unsigned)d.nh, (unsigned)d.b);
  if (io == SSD_BF16)
    chunk_state_simt<__nv_bfloat16><<<grid, kThreads, 0, st>>>(
        (const __nv_bfloat16 *)x, (const __nv_bfloat16 *)B, (const __nv_bfloat16 *)dt, G,
        dstates, d.L, d.nh, d.P, d.S, d.ng, d.T, d.nc);
  else
    chunk_state_simt<float><<<grid, kThreads, 0, st>>>(
        (const float *)x, (const float *)B, (const float *)dt, G, dstates, d.L, d.nh, d.P,
        d.S, d.ng, d.T, d.nc);
  return cudaGetLastError();
}

}  // namespace ssd
