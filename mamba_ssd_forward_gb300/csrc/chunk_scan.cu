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
// Tensor-core kernel (tcgen05).  One CTA per (128-row tile i of a chunk,
// chunk, head, batch), 128 threads (thread = row = TMEM lane):
//   phase 1, over 128-byte blocks of S:  TMA stages C (rows i) and B (rows
//     j <= the tile's last row); the threads stage the carried state h
//     (fp32 -> operand type); one thread issues
//       Yoff += C h^T      (M = 128, N = P)
//       S    += C B^T      (M = 128, N = tokens j)
//     into tensor memory;
//   phase 2, over 128-byte blocks of tokens j:  each thread reads its row of
//     S from TMEM, applies exp2(G_i - G_j) dt_j and the causal mask, and
//     writes the row into a K-major swizzled tile; TMA stages x_j; one thread
//     issues Ydiag += S' X  (M = 128, N = P, X as an MN-major operand);
//   epilogue: y_i = exp2(G_i) Yoff_i + Ydiag_i + D x_i, stored in the I/O
//     type.  The T x T interaction tile lives only in TMEM and shared memory.
// With fp32 I/O (kind::tf32, K-major operands only) the threads stage x
// transposed in phase 2 instead of TMA.
#include "tc_common.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 128;
constexpr int kRows = 128;  // rows i per CTA (MMA M)

template <typename IO>
__global__ void __launch_bounds__(kThreads)
chunk_scan_tc(const __grid_constant__ CUtensorMap tm_C, const __grid_constant__ CUtensorMap tm_B,
              const __grid_constant__ CUtensorMap tm_x, const IO *__restrict__ x,
              const IO *__restrict__ dt, const float *__restrict__ G,
              const float *__restrict__ states, const float *__restrict__ Dv,
              IO *__restrict__ y, int *__restrict__ err, int L, int nh, int P, int S, int hpg,
              int T, int nc, int nb) {
  using Tr = IoT<IO>;
  constexpr int kAE = Tr::kAE;
  constexpr int kE = Tr::kE;
  constexpr int kC = kRows * 128;  // bytes of the C block (128 rows)
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ __align__(8) uint64_t full[2], mmad[2];
  __shared__ uint32_t tmem_slot;
  __shared__ float Gs[256], dts[256];

  const int n_it = (T + kRows - 1) / kRows;
  const int k = blockIdx.x / n_it, it = blockIdx.x % n_it;
  const int h = blockIdx.y, b = blockIdx.z, g = h / hpg;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int tok0 = k * T;
  const int valid = min(T, L - tok0);            // real tokens in this chunk
  const int i0 = it * kRows;                     // first row (chunk-relative)
  if (i0 >= valid) return;                       // whole tile past the end
  const int jext = min(min(T, i0 + kRows), (valid + 15) & ~15);  // tokens j used
  const int nBr = (jext + 127) / 128;            // 128-row B boxes
  const int nsb = (S + kAE - 1) / kAE;           // phase-1 blocks along S
  const int njb = (jext + kAE - 1) / kAE;        // phase-2 blocks along j
  const int nPb = (P + kAE - 1) / kAE;
  // phase-1 stage: C (128 rows) | B (nBr*128 rows) | h (P rows), 128 B each
  const int st1 = kC + nBr * 128 * 128 + ((P * 128 + 1023) & ~1023);
  // phase-2 stage: S' (128 rows x 128 B) | X (nPb blocks of kAE rows)
  const int st2 = kC + nPb * kAE * 128;
  const uint32_t col_S = 0, col_off = 256, col_diag = 256 + P;
  const uint32_t ncols = 512;

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&full[i], 1);
      ptx::mbar_init(&mmad[i], 1);
    }
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(&tmem_slot, ncols);
    ptx::tmem_relinquish();
  }
  // extents of the buffers read and written below (debug-bounds builds)
  const int64_t nG = (int64_t)nb * nh * nc * T, ndt = (int64_t)nb * L * nh;
  const int64_t nst = (int64_t)nb * nh * nc * P * S, nx = (int64_t)nb * L * nh * P;
  const int64_t g0 = ((int64_t)(b * nh + h) * nc + k) * T;
  const float *Gc = G + g0;
  for (int j = tid; j < T; j += kThreads) {
    const int64_t idt = ((int64_t)b * L + tok0 + j) * nh + h;
    Gs[j] = SSD_IN_BOUNDS(g0 + j < nG, err, 100) ? Gc[j] : 0.f;
    dts[j] = j < valid && SSD_IN_BOUNDS(idt < ndt, err, 101) ? ld_io(dt + idt) : 0.f;
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const int64_t h0i = ((int64_t)(b * nh + h) * nc + k) * P * S;
  const float *hst = states + h0i;

  // ---------------- phase 1: Yoff = C h^T, S = C B^T over blocks of S
  auto load1 = [&](int sb) {
    const int s = sb & 1;
    uint8_t *Cb = smem + s * st1;
    uint8_t *Bb = Cb + kC;
    ptx::mbar_arrive_expect_tx(&full[s], kC + nBr * 128 * 128);
    ptx::tma_load_4d(Cb, &tm_C, sb * kAE, g, tok0 + i0, b, &full[s]);
    for (int r = 0; r < nBr; ++r)
      ptx::tma_load_4d(Bb + r * 128 * 128, &tm_B, sb * kAE, g, tok0 + r * 128, b, &full[s]);
  };
  if (tid == 0)
    for (int sb = 0; sb < min(nsb, 2); ++sb) load1(sb);

  const uint32_t id_off = mma_idesc<IO>(128, P, false, false);
  const uint32_t id_S = mma_idesc<IO>(128, jext, false, false);
  for (int sb = 0; sb < nsb; ++sb) {
    const int s = sb & 1;
    const uint32_t ph = (sb >> 1) & 1;
    uint8_t *Cb = smem + s * st1;
    uint8_t *Bb = Cb + kC;
    uint8_t *Hb = Bb + nBr * 128 * 128;
    // stage h[:, sb*kAE .. +kAE) as a K-major operand (rows p, 128 B each)
    for (int c = tid; c < P * 8; c += kThreads) {
      const int p = c >> 3, ch = c & 7;
      const int s_first = sb * kAE + ch * (16 / kE);
      float v[8];
      if (s_first < S &&
          SSD_IN_BOUNDS(h0i + (int64_t)p * S + s_first + 16 / kE <= nst, err, 102)) {
        const float4 *src = reinterpret_cast<const float4 *>(hst + (int64_t)p * S + s_first);
        const float4 a = src[0];
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        if (kE == 2) {
          const float4 bq = src[1];
          v[4] = bq.x; v[5] = bq.y; v[6] = bq.z; v[7] = bq.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = 0.f;
      }
      *reinterpret_cast<uint4 *>(Hb + sw128(p, ch * 16)) = pack_op16(v, (IO *)nullptr);
    }
    ptx::mbar_wait(&full[s], ph, err, 41);
    ptx::fence_async_smem();
    __syncthreads();
    if (tid == 0) {
      ptx::tc_fence_after();
      const uint32_t c0 = ptx::smem_u32(Cb), b0 = ptx::smem_u32(Bb), h0 = ptx::smem_u32(Hb);
#pragma unroll
      for (int kk = 0; kk < kAE / Tr::kKmma; ++kk) {
        const uint32_t adv = kk * 32;  // K step inside the 128-byte row
        const uint64_t ad = ptx::smem_desc(c0 + adv, 16, 1024, ptx::kSw128);
        const uint64_t hd = ptx::smem_desc(h0 + adv, 16, 1024, ptx::kSw128);
        const uint64_t bd = ptx::smem_desc(b0 + adv, 16, 1024, ptx::kSw128);
        const uint32_t acc = (sb | kk) ? 1u : 0u;
        ptx::mma_ss<Tr::kTf32>(tmem + col_off, ad, hd, id_off, acc);
        ptx::mma_ss<Tr::kTf32>(tmem + col_S, ad, bd, id_S, acc);
      }
      ptx::mma_commit(&mmad[s]);
      if (sb + 2 < nsb) {
        ptx::mbar_wait(&mmad[s], ph, err, 42);
        load1(sb + 2);
      }
    }
  }
  ptx::mbar_wait(&mmad[(nsb - 1) & 1], ((nsb - 1) >> 1) & 1, err, 43);
  ptx::tc_fence_after();
  __syncthreads();  // every thread is past phase 1 before its buffers are reused

  // ---------------- phase 2: Ydiag = (S * decay * mask) X over blocks of j
  const int row = warp * 32 + lane;  // this thread's row of the tile
  const int i_rel = i0 + row;        // chunk-relative row index
  const float Gi = Gs[min(i_rel, T - 1)];
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  // the phase-1 pipeline left its barriers at a known phase count: continue
  // the parity sequence from there.
  const int base1 = nsb;
  auto load2 = [&](int jb) {
    const int u = base1 + jb, s = u & 1;
    uint8_t *Xb = smem + s * st2 + kC;
    ptx::mbar_arrive_expect_tx(&full[s], nPb * kAE * 128);
    for (int pb = 0; pb < nPb; ++pb)
      ptx::tma_load_4d(Xb + pb * kAE * 128, &tm_x, pb * kAE, h, tok0 + jb * kAE, b, &full[s]);
  };
  if (!Tr::kTf32 && tid == 0)
    for (int jb = 0; jb < min(njb, 2); ++jb) load2(jb);

  const uint32_t id_diag = mma_idesc<IO>(128, P, false, !Tr::kTf32);
  for (int jb = 0; jb < njb; ++jb) {
    const int u = base1 + jb, s = u & 1;
    const uint32_t ph = (u >> 1) & 1;
    uint8_t *Pb = smem + s * st2;
    uint8_t *Xb = Pb + kC;
    // this thread's row of S for tokens jb*kAE .. +kAE -> decayed, masked
#pragma unroll
    for (int q = 0; q < kAE / 16; ++q) {
      float v[16];
      ptx::tmem_ld16_sync(tmem + lane_base + col_S + jb * kAE + q * 16, v);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int j = jb * kAE + q * 16 + e;
        v[e] = (j <= i_rel && j < valid) ? v[e] * exp2f(Gi - Gs[j]) * dts[j] : 0.f;
      }
      constexpr int per16 = 16 / kE;  // values per 16-byte chunk
#pragma unroll
      for (int c = 0; c < 16 / per16; ++c) {
        const int chunk = (q * 16) / per16 + c;
        *reinterpret_cast<uint4 *>(Pb + sw128(row, chunk * 16)) =
            pack_op16(v + c * per16, (IO *)nullptr);
      }
    }
    if constexpr (Tr::kTf32) {
      // X^T (rows p, tokens along the 128-byte row), rounded to tf32: lane =
      // token j, each lane loads four consecutive p (16 bytes) and writes
      // them down four rows at its column (a warp writes 32 consecutive
      // words of a row); every load is issued before the first store
      constexpr int kXqMax = (128 / 4) * kAE / kThreads;  // quads per thread, P <= 128
      const int nXq = (P / 4) * kAE;
      float4 xq[kXqMax];
#pragma unroll
      for (int r = 0; r < kXqMax; ++r) {
        const int idx = tid + r * kThreads, j = idx % kAE, q = idx / kAE;
        const int jt = jb * kAE + j;
        const int64_t ix = (((int64_t)b * L + tok0 + jt) * nh + h) * P + 4 * q;
        xq[r] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (idx < nXq && jt < valid && SSD_IN_BOUNDS(ix + 4 <= nx, err, 103))
          xq[r] = *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(x) + ix);
      }
#pragma unroll
      for (int r = 0; r < kXqMax; ++r) {
        const int idx = tid + r * kThreads, j = idx % kAE, q = idx / kAE;
        if (idx >= nXq) break;
        *reinterpret_cast<uint32_t *>(Xb + sw128(4 * q + 0, j * 4)) = to_tf32(xq[r].x);
        *reinterpret_cast<uint32_t *>(Xb + sw128(4 * q + 1, j * 4)) = to_tf32(xq[r].y);
        *reinterpret_cast<uint32_t *>(Xb + sw128(4 * q + 2, j * 4)) = to_tf32(xq[r].z);
        *reinterpret_cast<uint32_t *>(Xb + sw128(4 * q + 3, j * 4)) = to_tf32(xq[r].w);
      }
    } else {
      ptx::mbar_wait(&full[s], ph, err, 44);
    }
    ptx::fence_async_smem();
    ptx::tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      ptx::tc_fence_after();
      const uint32_t p0 = ptx::smem_u32(Pb), x0 = ptx::smem_u32(Xb);
#pragma unroll
      for (int kk = 0; kk < kAE / Tr::kKmma; ++kk) {
        const uint64_t ad = ptx::smem_desc(p0 + kk * 32, 16, 1024, ptx::kSw128);
        const uint64_t xd =
            Tr::kTf32 ? ptx::smem_desc(x0 + kk * 32, 16, 1024, ptx::kSw128)
                      : ptx::smem_desc(x0 + kk * Tr::kKmma * 128, kAE * 128, 1024, ptx::kSw128);
        ptx::mma_ss<Tr::kTf32>(tmem + col_diag, ad, xd, id_diag, (jb | kk) ? 1u : 0u);
      }
      ptx::mma_commit(&mmad[s]);
      if (jb + 2 < njb) {
        ptx::mbar_wait(&mmad[s], ph, err, 45);
        if (!Tr::kTf32) load2(jb + 2);
      }
    }
  }
  {
    const int u = base1 + njb - 1;
    ptx::mbar_wait(&mmad[u & 1], (u >> 1) & 1, err, 46);
  }
  ptx::tc_fence_after();

  // ---------------- epilogue: y = exp2(G_i) Yoff + Ydiag + D x
  const bool row_ok = i_rel < valid;
  const float eg = exp2f(Gi);
  const float Dh = Dv ? Dv[h] : 0.f;
  const int64_t yoff = (((int64_t)b * L + tok0 + i_rel) * nh + h) * P;
  for (int c0 = 0; c0 < P; c0 += 16) {
    float a[16], d[16];
    ptx::tmem_ld16_sync(tmem + lane_base + col_off + c0, a);
    ptx::tmem_ld16_sync(tmem + lane_base + col_diag + c0, d);
    if (row_ok && SSD_IN_BOUNDS(yoff + P <= nx, err, 104)) {
      constexpr int per16 = 16 / kE;
#pragma unroll
      for (int c = 0; c < 16 / per16; ++c) {
        float xv[8], o[8];
        unpack16(*reinterpret_cast<const uint4 *>(x + yoff + c0 + c * per16), xv, (IO *)nullptr);
#pragma unroll
        for (int e = 0; e < per16; ++e)
          o[e] = fmaf(eg, a[c * per16 + e], d[c * per16 + e]) + Dh * xv[e];
        *reinterpret_cast<uint4 *>(y + yoff + c0 + c * per16) = pack_io16(o, (IO *)nullptr);
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) ptx::tmem_dealloc(tmem, ncols);
}

template <typename IO>
cudaError_t launch_t(const Dims &d, const void *x, const void *B, const void *C, const void *dt,
                     const float *G, const float *states, const float *D, void *y,
                     int *err, cudaStream_t st) {
  constexpr int kAE = IoT<IO>::kAE;
  constexpr bool bf = !IoT<IO>::kTf32;
  CUtensorMap tC, tB, tx;
  if (!make_tmap_bl(&tC, C, bf, d.b, d.L, d.ng, d.S, kRows) ||
      !make_tmap_bl(&tB, B, bf, d.b, d.L, d.ng, d.S, 128) ||
      !make_tmap_bl(&tx, x, bf, d.b, d.L, d.nh, d.P, kAE))
    return cudaErrorInvalidValue;
  const int nBr = (int)((std::min<int64_t>(d.T, 256) + 127) / 128);
  const int nPb = (int)((d.P + kAE - 1) / kAE);
  const int st1 = kRows * 128 + nBr * 128 * 128 + (int)((d.P * 128 + 1023) & ~1023);
  const int st2 = kRows * 128 + nPb * kAE * 128;
  const int smem = 2 * std::max(st1, st2) + 1024;
  auto kern = chunk_scan_tc<IO>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int n_it = (int)((d.T + kRows - 1) / kRows);
  dim3 grid((unsigned)(d.nc * n_it), (unsigned)d.nh, (unsigned)d.b);
  kern<<<grid, kThreads, smem, st>>>(tC, tB, tx, static_cast<const IO *>(x),
                                     static_cast<const IO *>(dt), G, states, D,
                                     static_cast<IO *>(y), err, (int)d.L,
                                     (int)d.nh, (int)d.P, (int)d.S, (int)d.hpg, (int)d.T,
                                     (int)d.nc, (int)d.b);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chunk_scan(const Dims &d, ssd_dtype io, const void *x, const void *B,
                              const void *C, const void *dt, const float *G,
                              const float *states, const float *D, void *y, int *err,
                              cudaStream_t st) {
  return io == SSD_BF16 ? launch_t<__nv_bfloat16>(d, x, B, C, dt, G, states, D, y, err, st)
                        : launch_t<float>(d, x, B, C, dt, G, states, D, y, err, st);
}

}  // namespace ssd
