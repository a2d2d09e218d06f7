// Step 4: per-chunk outputs (the page's compute_out), chunked output equation
// of "Accelerating Mamba-2 with High-Performance Forward Pass Kernels in
// NVIDIA CUDA Tile", section "Mamba-2 architecture":
//
//   y_i = exp2(G_i) (states[k] c_i)
//       + sum_{j <= i, j in chunk k} (c_i . B_j) exp2(G_i - G_j) dt_j x_j
//       + D[h] x_i
//
// The causal mask keeps the diagonal (post-update convention), and the
// retained exponents G_i - G_j are <= 0 because every a_t <= 0.
//
// First-cut SIMT kernel: one block per (64-row tile of a chunk, 64-wide
// headdim tile, head, batch).  The 64 x 32 interaction blocks are formed in
// shared memory, decayed and masked there, and never written to memory.
#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 256;
constexpr int kRows = 64;   // rows i per block
constexpr int kCols = 64;   // headdim p per block
constexpr int kJ = 32;      // tokens j per interaction block
constexpr int kSc = 32;     // state entries s per staging step

template <typename IO>
__global__ void __launch_bounds__(kThreads)
chunk_scan_simt(const IO *__restrict__ x, const IO *__restrict__ Bm,
                const IO *__restrict__ Cm, const IO *__restrict__ dt,
                const float *__restrict__ G, const float *__restrict__ states,
                const float *__restrict__ Dv, IO *__restrict__ y, int64_t L,
                int64_t nh, int64_t P, int64_t S, int64_t ng, int64_t T,
                int64_t nc) {
  __shared__ float cs[kRows][kSc + 1];
  __shared__ float hs[kCols][kSc + 1];
  __shared__ float bs[kJ][kSc + 1];
  __shared__ float sb[kRows][kJ + 1];
  __shared__ float xs[kJ][kCols];
  __shared__ float gi[kRows];

  const int64_t ptiles = (P + kCols - 1) / kCols, itiles = T / kRows;
  int64_t r = blockIdx.x;
  const int64_t pt = r % ptiles;
  r /= ptiles;
  const int64_t it = r % itiles;
  const int64_t k = r / itiles;
  const int64_t h = blockIdx.y, b = blockIdx.z, g = h / (nh / ng);
  const int64_t row0 = k * T + it * kRows;  // first token of this tile
  if (row0 >= L) return;
  const float *Gc = G + ((b * nh + h) * nc + k) * T;
  const float *hst = states + ((b * nh + h) * nc + k) * P * S;
  const int tid = threadIdx.x, ti = tid / 16, tp = tid % 16;

  if (tid < kRows) gi[tid] = Gc[it * kRows + tid];

  // Carried-state term: sum_s C_i[s] h[p][s].
  float acc_off[4][4] = {};
  for (int64_t s0 = 0; s0 < S; s0 += kSc) {
    for (int idx = tid; idx < kRows * kSc; idx += kThreads) {
      const int rr = idx / kSc, c = idx % kSc;
      const int64_t tok = row0 + rr, s = s0 + c;
      cs[rr][c] = (tok < L && s < S) ? ld_io(Cm + ((b * L + tok) * ng + g) * S + s) : 0.f;
    }
    for (int idx = tid; idx < kCols * kSc; idx += kThreads) {
      const int pp = idx / kSc, c = idx % kSc;
      const int64_t p = pt * kCols + pp, s = s0 + c;
      hs[pp][c] = (p < P && s < S) ? hst[p * S + s] : 0.f;
    }
    __syncthreads();
    for (int c = 0; c < kSc; ++c) {
      float cv[4], hv[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        cv[q] = cs[ti * 4 + q][c];
        hv[q] = hs[tp * 4 + q][c];
      }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc_off[a][e] = fmaf(cv[a], hv[e], acc_off[a][e]);
    }
    __syncthreads();
  }

  // Intra-chunk term over j-blocks up to the tile's last row.
  float acc[4][4] = {};
  const int64_t jend = (it + 1) * kRows;  // chunk-relative
  for (int64_t j0 = 0; j0 < jend; j0 += kJ) {
    // sb[i][j] = c_i . B_j, accumulated over s in steps of kSc.
    float sacc[8] = {};
    const int si = tid / 4, sj = (tid % 4) * 8;
    for (int64_t s0 = 0; s0 < S; s0 += kSc) {
      for (int idx = tid; idx < kRows * kSc; idx += kThreads) {
        const int rr = idx / kSc, c = idx % kSc;
        const int64_t tok = row0 + rr, s = s0 + c;
        cs[rr][c] = (tok < L && s < S) ? ld_io(Cm + ((b * L + tok) * ng + g) * S + s) : 0.f;
      }
      for (int idx = tid; idx < kJ * kSc; idx += kThreads) {
        const int jj = idx / kSc, c = idx % kSc;
        const int64_t tok = k * T + j0 + jj, s = s0 + c;
        bs[jj][c] = (tok < L && s < S) ? ld_io(Bm + ((b * L + tok) * ng + g) * S + s) : 0.f;
      }
      __syncthreads();
      for (int c = 0; c < kSc; ++c) {
        const float cv = cs[si][c];
#pragma unroll
        for (int q = 0; q < 8; ++q) sacc[q] = fmaf(cv, bs[sj + q][c], sacc[q]);
      }
      __syncthreads();
    }
    // Decay, dt and causal mask (diagonal kept); padded tokens have dt = 0.
    {
      const int64_t i_rel = it * kRows + si;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int64_t j_rel = j0 + sj + q, tok = k * T + j_rel;
        float v = 0.f;
        if (j_rel <= i_rel && tok < L)
          v = sacc[q] * exp2f(gi[si] - Gc[j_rel]) * ld_io(dt + (b * L + tok) * nh + h);
        sb[si][sj + q] = v;
      }
    }
    for (int idx = tid; idx < kJ * kCols; idx += kThreads) {
      const int jj = idx / kCols, pp = idx % kCols;
      const int64_t tok = k * T + j0 + jj, p = pt * kCols + pp;
      xs[jj][pp] = (tok < L && p < P) ? ld_io(x + ((b * L + tok) * nh + h) * P + p) : 0.f;
    }
    __syncthreads();
    for (int jj = 0; jj < kJ; ++jj) {
      float sv[4], xv[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        sv[q] = sb[ti * 4 + q][jj];
        xv[q] = xs[jj][tp * 4 + q];
      }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[a][e] = fmaf(sv[a], xv[e], acc[a][e]);
    }
    __syncthreads();
  }

  const float Dh = Dv ? Dv[h] : 0.f;
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int64_t tok = row0 + ti * 4 + a;
    if (tok >= L) continue;
    const float eg = exp2f(gi[ti * 4 + a]);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int64_t p = pt * kCols + tp * 4 + e;
      if (p >= P) continue;
      const int64_t off = ((b * L + tok) * nh + h) * P + p;
      st_io(y + off, eg * acc_off[a][e] + acc[a][e] + Dh * ld_io(x + off));
    }
  }
}

}  // namespace

cudaError_t launch_chunk_scan(const Dims &d, ssd_dtype io, const void *x,
                              const void *B, const void *C, const void *dt,
                              const float *G, const float *states,
                              const float *D, void *y, cudaStream_t st) {
  const int64_t tiles = ((d.P + kCols - 1) / kCols) * (d.T / kRows);
  dim3 grid((unsigned)(d.nc * tiles), (unsigned)d.nh, (unsigned)d.b);
  if (io == SSD_BF16)
    chunk_scan_simt<__nv_bfloat16><<<grid, kThreads, 0, st>>>(
        (const __nv_bfloat16 *)x, (const __nv_bfloat16 *)B, (const __nv_bfloat16 *)C,
        (const __nv_bfloat16 *)dt, G, states, D, (__nv_bfloat16 *)y, d.L, d.nh, d.P, d.S,
        d.ng, d.T, d.nc);
  else
    chunk_scan_simt<float><<<grid, kThreads, 0, st>>>(
        (const float *)x, (const float *)B, (const float *)C, (const float *)dt, G, states, D,
        (float *)y, d.L, d.nh, d.P, d.S, d.ng, d.T, d.nc);
  return cudaGetLastError();
}

}  // namespace ssd
