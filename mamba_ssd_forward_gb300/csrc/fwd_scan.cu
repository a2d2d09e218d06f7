// Forward path, output pass (bf16 I/O): the page's compute_out, chunked
// output equation of "Accelerating Mamba-2 with High-Performance Forward
// Pass Kernels in NVIDIA CUDA Tile", section "Mamba-2 architecture":
//
//   y_i = exp2(G_i) (h_k c_i) + sum_{j<=i in chunk} (c_i . B_j) exp2(G_i - G_j) dt_j x_j
//         + D x_i
//
// One CTA per (128-row tile of a chunk, chunk, group of H heads that share
// B and C, batch), warp-specialised:
//   warp 4 (TMA):  C and B blocks of 64 state entries, the H heads' start
//                  states (bf16 [s][p] tiles), then 64-token blocks of x;
//   warp 5 (MMA):  phase 1, per block of S:  Sc += C B^T (once for all H
//                  heads: they share B and C) and Y_q += C h_q^T;
//                  phase 2, per head q and 64-token block: Y_q += S'_q X_q;
//   warps 0-3 (one thread per row i):  the in-chunk cumsums of the H heads;
//                  Y_q *= exp2(G_i) once phase 1 is done; the decayed, masked
//                  interaction tile S'_q = Sc * exp2(G_i - G_j) dt_j [j <= i]
//                  written to shared memory as a K-major operand, one block
//                  of 64 tokens at a time; and the epilogue y = Y_q + D x.
// Sc lives in tensor-memory columns [0, 256), Y_q in 256 + q P.  The
// interaction tile is never written to global memory.
#include "fwd.cuh"

namespace ssd {
namespace {

constexpr int kRowThreads = 128;
constexpr int kThreads = 192;
constexpr int kMaxH = 4;
constexpr int kBlk = 64 * 128;  // one 64-row, 128-byte-wide block

struct ScanArgs {
  const __nv_bfloat16 *x, *dt;
  const float *A, *D;
  __nv_bfloat16 *y;
  int *err;
  int L, nh, P, S, hpg, T, nc, H;
};

__global__ void __launch_bounds__(kThreads)
fwd_scan_bf16(const __grid_constant__ CUtensorMap tm_C, const __grid_constant__ CUtensorMap tm_B,
              const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_st,
              const ScanArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ __align__(8) uint64_t full1[2], empty1[2], s1_done, pm_full[2], pm_empty[2],
      x_full[2], x_empty[2], ysc[kMaxH], ydone[kMaxH];
  __shared__ uint32_t tmem_slot;
  __shared__ float Gs[kMaxH][256], dts[kMaxH][256];
  __shared__ float warp_tot[4];

  const int L = a.L, nh = a.nh, P = a.P, S = a.S, T = a.T, nc = a.nc, H = a.H;
  const int n_it = (T + 127) / 128;
  const int k = blockIdx.x / n_it, it = blockIdx.x % n_it;
  const int hbase = blockIdx.y * H, b = blockIdx.z, g = hbase / a.hpg;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int tok0 = k * T;
  const int valid = min(T, L - tok0);
  const int i0 = it * 128;
  if (i0 >= valid) return;
  const int jext = min(min(T, i0 + 128), (valid + 15) & ~15);
  const int nBr = (jext + 127) / 128;
  const int nsb = (S + 63) / 64;
  const int njb = (jext + 63) / 64;
  const int nPb = (P + 63) / 64;
  const int st1 = kBlk * 2 + nBr * kBlk * 2 + H * nPb * kBlk;  // C | B | states
  const int st2p = kBlk * 2;                                 // S' (128 rows)
  const int st2x = nPb * kBlk;                               // X (64 rows)
  const uint32_t ncols = 512;

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&full1[i], 1);
      ptx::mbar_init(&empty1[i], 1);
      ptx::mbar_init(&pm_full[i], kRowThreads);
      ptx::mbar_init(&pm_empty[i], 1);
      ptx::mbar_init(&x_full[i], 1);
      ptx::mbar_init(&x_empty[i], 1);
    }
    ptx::mbar_init(&s1_done, 1);
    for (int q = 0; q < kMaxH; ++q) {
      ptx::mbar_init(&ysc[q], kRowThreads);
      ptx::mbar_init(&ydone[q], 1);
    }
    ptx::fence_mbar_init();
  }
  if (warp == 5) {
    ptx::tmem_alloc(&tmem_slot, ncols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if ((tid & 31) == 0) {
      for (int sb = 0; sb < nsb; ++sb) {
        const int s = sb & 1;
        uint8_t *Cb = smem + s * st1;
        uint8_t *Bb = Cb + 2 * kBlk;
        uint8_t *Hb = Bb + nBr * 2 * kBlk;
        ptx::mbar_wait(&empty1[s], ((sb >> 1) & 1) ^ 1, a.err, 81);
        ptx::mbar_arrive_expect_tx(&full1[s], st1);
        ptx::tma_load_4d(Cb, &tm_C, sb * 64, g, tok0 + i0, b, &full1[s]);
        for (int r = 0; r < nBr; ++r)
          ptx::tma_load_4d(Bb + r * 2 * kBlk, &tm_B, sb * 64, g, tok0 + r * 128, b, &full1[s]);
        for (int q = 0; q < H; ++q) {
          const int row = (b * nh + hbase + q) * nc + k;
          for (int pb = 0; pb < nPb; ++pb)
            ptx::tma_load_3d(Hb + (q * nPb + pb) * kBlk, &tm_st, pb * 64, sb * 64, row,
                             &full1[s]);
        }
      }
      // phase-2 buffers overlay phase 1: wait until phase 1 is consumed
      ptx::mbar_wait(&s1_done, 0, a.err, 82);
      for (int q = 0; q < H; ++q)
        for (int jb = 0; jb < njb; ++jb) {
          const int u = q * njb + jb, s = u & 1;
          uint8_t *Xb = smem + 2 * st2p + s * st2x;
          ptx::mbar_wait(&x_empty[s], ((u >> 1) & 1) ^ 1, a.err, 83);
          ptx::mbar_arrive_expect_tx(&x_full[s], st2x);
          for (int pb = 0; pb < nPb; ++pb)
            ptx::tma_load_4d(Xb + pb * kBlk, &tm_x, pb * 64, hbase + q, tok0 + jb * 64, b,
                             &x_full[s]);
        }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if ((tid & 31) == 0) {
      const uint32_t id_S = ptx::idesc_bf16(128, jext, false, false);
      const uint32_t id_Y = ptx::idesc_bf16(128, P, false, true);
      for (int sb = 0; sb < nsb; ++sb) {
        const int s = sb & 1;
        uint8_t *Cb = smem + s * st1;
        uint8_t *Bb = Cb + 2 * kBlk;
        uint8_t *Hb = Bb + nBr * 2 * kBlk;
        ptx::mbar_wait(&full1[s], (sb >> 1) & 1, a.err, 84);
        ptx::tc_fence_after();
        const uint32_t c0 = ptx::smem_u32(Cb), b0 = ptx::smem_u32(Bb), h0 = ptx::smem_u32(Hb);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t cd = ptx::smem_desc(c0 + kk * 32, 16, 1024, ptx::kSw128);
          const uint64_t bd = ptx::smem_desc(b0 + kk * 32, 16, 1024, ptx::kSw128);
          const uint32_t acc = (sb | kk) ? 1u : 0u;
          ptx::mma_ss<false>(tmem, cd, bd, id_S, acc);
          for (int q = 0; q < H; ++q) {
            const uint64_t hd = ptx::smem_desc(h0 + q * nPb * kBlk + kk * 2048, kBlk, 1024,
                                               ptx::kSw128);
            ptx::mma_ss<false>(tmem + 256 + q * P, cd, hd, id_Y, acc);
          }
        }
        ptx::mma_commit(&empty1[s]);
      }
      ptx::mma_commit(&s1_done);
      for (int q = 0; q < H; ++q) {
        ptx::mbar_wait(&ysc[q], 0, a.err, 85);
        ptx::tc_fence_after();
        for (int jb = 0; jb < njb; ++jb) {
          const int u = q * njb + jb, s = u & 1;
          const uint32_t ph = (u >> 1) & 1;
          ptx::mbar_wait(&pm_full[s], ph, a.err, 86);
          ptx::mbar_wait(&x_full[s], ph, a.err, 87);
          ptx::tc_fence_after();
          const uint32_t p0 = ptx::smem_u32(smem + s * st2p);
          const uint32_t x0 = ptx::smem_u32(smem + 2 * st2p + s * st2x);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t pd = ptx::smem_desc(p0 + kk * 32, 16, 1024, ptx::kSw128);
            const uint64_t xd = ptx::smem_desc(x0 + kk * 2048, kBlk, 1024, ptx::kSw128);
            ptx::mma_ss<false>(tmem + 256 + q * P, pd, xd, id_Y, 1u);
          }
          ptx::mma_commit(&pm_empty[s]);
          ptx::mma_commit(&x_empty[s]);
        }
        ptx::mma_commit(&ydone[q]);
      }
    }
  } else {
    // ------------------------------------------------------------ row warps
    const int row = tid;  // 0..127 = TMEM lane
    const int i_rel = i0 + row;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    // in-chunk cumsums (log2 units) of the H heads
    const int per = T > 128 ? 2 : 1;
    for (int q = 0; q < H; ++q) {
      const int h = hbase + q;
      const float Ah = a.A[h] * kLog2e;
      float d[2] = {0.f, 0.f}, c[2] = {0.f, 0.f}, run = 0.f;
      for (int e = 0; e < per; ++e) {
        const int j = row * per + e;
        if (j < valid) d[e] = __bfloat162float(a.dt[((int64_t)b * L + tok0 + j) * nh + h]);
        run += Ah * d[e];
        c[e] = run;
      }
      float incl = run;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_up_sync(0xffffffffu, incl, off);
        if ((row & 31) >= off) incl += o;
      }
      if ((row & 31) == 31) warp_tot[warp] = incl;
      ptx::named_bar_sync(1, kRowThreads);
      float base = incl - run;
      for (int w2 = 0; w2 < warp; ++w2) base += warp_tot[w2];
      for (int e = 0; e < per; ++e) {
        const int j = row * per + e;
        if (j < T) {
          Gs[q][j] = base + c[e];
          dts[q][j] = d[e];
        }
      }
      ptx::named_bar_sync(1, kRowThreads);
    }
    ptx::mbar_wait(&s1_done, 0, a.err, 88);
    ptx::tc_fence_after();

    auto epilogue = [&](int q) {
      ptx::mbar_wait(&ydone[q], 0, a.err, 89);
      ptx::tc_fence_after();
      const int h = hbase + q;
      const float Dh = a.D ? a.D[h] : 0.f;
      const bool ok = i_rel < valid;
      const int64_t off = (((int64_t)b * L + tok0 + i_rel) * nh + h) * P;
      for (int c0 = 0; c0 < P; c0 += 16) {
        float v[16];
        ptx::tmem_ld16_sync(tmem + lane_base + 256 + q * P + c0, v);
        if (ok) {
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            float xv[8];
            unpack16(*reinterpret_cast<const uint4 *>(a.x + off + c0 + half * 8), xv,
                     (__nv_bfloat16 *)nullptr);
#pragma unroll
            for (int e = 0; e < 8; ++e) xv[e] = fmaf(Dh, xv[e], v[half * 8 + e]);
            *reinterpret_cast<uint4 *>(a.y + off + c0 + half * 8) =
                pack_io16(xv, (__nv_bfloat16 *)nullptr);
          }
        }
      }
    };

    for (int q = 0; q < H; ++q) {
      const float Gi = Gs[q][min(i_rel, T - 1)];
      // carried-state term: Y_q *= exp2(G_i), then release Y_q to phase 2
      const float eg = exp2f(Gi);
      for (int c0 = 0; c0 < P; c0 += 16) {
        float v[16];
        ptx::tmem_ld16_sync(tmem + lane_base + 256 + q * P + c0, v);
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] *= eg;
        ptx::tmem_st16(tmem + lane_base + 256 + q * P + c0, v);
      }
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(&ysc[q]);
      // decayed, masked interaction rows, 64 tokens at a time
      for (int jb = 0; jb < njb; ++jb) {
        const int u = q * njb + jb, s = u & 1;
        ptx::mbar_wait(&pm_empty[s], ((u >> 1) & 1) ^ 1, a.err, 90);
        uint8_t *Pb = smem + s * st2p;
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          const int jc = jb * 64 + c4 * 16;
          float v[16];
          ptx::tmem_ld16_sync(tmem + lane_base + jc, v);
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int j = jc + e;
            v[e] = (j <= i_rel && j < valid) ? v[e] * exp2f(Gi - Gs[q][j]) * dts[q][j] : 0.f;
          }
          *reinterpret_cast<uint4 *>(Pb + sw128(row, c4 * 32)) =
              pack_op16(v, (__nv_bfloat16 *)nullptr);
          *reinterpret_cast<uint4 *>(Pb + sw128(row, c4 * 32 + 16)) =
              pack_op16(v + 8, (__nv_bfloat16 *)nullptr);
        }
        ptx::fence_async_smem();
        ptx::tc_fence_before();
        ptx::mbar_arrive(&pm_full[s]);
      }
      if (q > 0) epilogue(q - 1);
    }
    epilogue(H - 1);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 5) ptx::tmem_dealloc(tmem, ncols);
}

}  // namespace

cudaError_t launch_fwd_scan(const Dims &d, const void *x, const void *B, const void *C,
                            const void *dt, const float *A, const void *states, const float *D,
                            void *y, cudaStream_t st) {
  const int H = fwd_scan_heads(d);
  CUtensorMap tC, tB, tx, tS;
  if (!make_tmap_bl(&tC, C, true, d.b, d.L, d.ng, d.S, 128) ||
      !make_tmap_bl(&tB, B, true, d.b, d.L, d.ng, d.S, 128) ||
      !make_tmap_bl(&tx, x, true, d.b, d.L, d.nh, d.P, 64))
    return cudaErrorInvalidValue;
  {
    const uint64_t dims[3] = {(uint64_t)d.P, (uint64_t)d.S, (uint64_t)(d.b * d.nh * d.nc)};
    const uint64_t strides[2] = {(uint64_t)d.P * 2, (uint64_t)(d.S * d.P * 2)};
    const uint32_t box[3] = {64u, 64u, 1u};
    if (!make_tmap_sw128(&tS, states, true, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  const int nBr = (int)((std::min<int64_t>(d.T, 256) + 127) / 128);
  const int nPb = (int)((d.P + 63) / 64);
  const int st1 = kBlk * 2 + nBr * kBlk * 2 + H * nPb * kBlk;
  const int st2 = 2 * (kBlk * 2) + 2 * nPb * kBlk;
  const int smem = std::max(2 * st1, st2) + 1024;
  cudaError_t e =
      cudaFuncSetAttribute(fwd_scan_bf16, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  ScanArgs a;
  a.x = static_cast<const __nv_bfloat16 *>(x);
  a.dt = static_cast<const __nv_bfloat16 *>(dt);
  a.A = A;
  a.D = D;
  a.y = static_cast<__nv_bfloat16 *>(y);
  a.err = device_error_word();
  a.L = (int)d.L;
  a.nh = (int)d.nh;
  a.P = (int)d.P;
  a.S = (int)d.S;
  a.hpg = (int)d.hpg;
  a.T = (int)d.T;
  a.nc = (int)d.nc;
  a.H = H;
  const int n_it = (int)((d.T + 127) / 128);
  dim3 grid((unsigned)(d.nc * n_it), (unsigned)(d.nh / H), (unsigned)d.b);
  fwd_scan_bf16<<<grid, kThreads, smem, st>>>(tC, tB, tx, tS, a);
  return cudaGetLastError();
}

}  // namespace ssd
