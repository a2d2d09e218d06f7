// Forward path, output pass (bf16 I/O): the page's compute_out, chunked
// output equation of "Accelerating Mamba-2 with High-Performance Forward
// Pass Kernels in NVIDIA CUDA Tile", section "Mamba-2 architecture":
//
//   y_i = exp2(G_i) (h_k c_i) + sum_{j<=i in chunk} (c_i . B_j) exp2(G_i - G_j) dt_j x_j
//         + D x_i
//
// One CTA per (128-row tile of a chunk, chunk, group of H heads that share
// B and C, batch), warp-specialised:
//   warp 16 (TMA): C and B blocks of 64 state entries and the H heads' start
//                  states (bf16 [s][p] tiles), then 64-token blocks of x;
//   warp 17 (MMA): phase 1, per block of S:  Sc += C B^T (once for all H
//                  heads: they share B and C) and Y_q += C h_q^T;
//                  phase 2, per head q and 64-token block: Y_q += S'_q X_q;
//   warps 0-15 (four warps per 32-row quadrant of the tile, each taking a
//                  quarter of the columns):  the in-chunk cumsums of the H heads;
//                  Y_q *= exp2(G_i) once phase 1 is done; the decayed, masked
//                  interaction tile S'_q written to shared memory as a
//                  K-major operand, one block of 64 tokens at a time; and the
//                  epilogue y = Y_q + D x.
// Sc lives in tensor-memory columns [0, 256), Y_q in 256 + q P.  The
// interaction tile is never written to global memory.
//
// Decay factors.  For row i and a 64-token column block that ends at r
// strictly before row i's own block, exp2(G_i - G_j) = exp2(G_i - G_r) *
// exp2(G_r - G_j) with both exponents <= 0 (G falls along the chunk): one
// exp per (row, block) and one per column replace one per element.  The
// block holding the diagonal takes exp2(G_i - G_j) directly, and the causal
// mask (j <= i, diagonal kept) zeroes the rest.  No exponent above zero is
// ever evaluated.
#include "fwd.cuh"

namespace ssd {
namespace {

constexpr int kRowWarps = 16;
constexpr int kRowThreads = kRowWarps * 32;
constexpr int kThreads = kRowThreads + 64;
constexpr int kProducerWarp = kRowWarps, kMmaWarp = kRowWarps + 1;
constexpr int kMaxH = 4;
constexpr int kMaxX = 8;        // x pipeline stages (at most)
constexpr int kNP = 4;          // stages of the decayed interaction tile S'

constexpr int kBlk = 64 * 128;  // one 64-row, 128-byte-wide block

struct ScanArgs {
  const __nv_bfloat16 *x, *dt;
  const float *A, *D;
  __nv_bfloat16 *y;
  int *err;
  int L, nh, P, S, hpg, T, nc, H, nX;
  int nb;  // batch count (the extents the debug-bounds checks use)
};

__global__ void __launch_bounds__(kThreads, 1)
fwd_scan_bf16(const __grid_constant__ CUtensorMap tm_C, const __grid_constant__ CUtensorMap tm_B,
              const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_st,
              const ScanArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ __align__(8) uint64_t full1[2], empty1[2], s1_done, pm_full[kNP], pm_empty[kNP],
      x_full[kMaxX], x_empty[kMaxX], ysc[kMaxH], ydone[kMaxH];
  __shared__ uint32_t tmem_slot;
  // per head: G (log2 units), dt, and the column factors v_j of the
  // factored decay (exp2(G_r - G_j) dt_j, r = end of j's 64-token block)
  // read with 16-byte vector loads: each array 16-byte aligned
  __shared__ __align__(16) float Gs[kMaxH][256];
  __shared__ __align__(16) float dts[kMaxH][256];
  __shared__ __align__(16) float vs[kMaxH][256];
  __shared__ float warp_tot[kRowWarps];

  const int L = a.L, nh = a.nh, P = a.P, S = a.S, T = a.T, nc = a.nc, H = a.H, nX = a.nX;
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
  // x stages live after the two phase-1 stages, so their loads overlap
  // phase 1; the kNP S' stages reuse the phase-1 space once it is consumed.
  uint8_t *xbase = smem + 2 * st1;
  const uint32_t ncols = 512;

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&full1[i], 1);
      ptx::mbar_init(&empty1[i], 1);
    }
    for (int i = 0; i < kNP; ++i) {
      ptx::mbar_init(&pm_full[i], kRowThreads);
      ptx::mbar_init(&pm_empty[i], 1);
    }
    for (int i = 0; i < kMaxX; ++i) {
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
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(&tmem_slot, ncols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_slot;

  const bool leader = (tid & 31) == 0;
  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    for (int sb = 0; sb < nsb; ++sb) {
      const int s = sb & 1;
      uint8_t *Cb = smem + s * st1;
      uint8_t *Bb = Cb + 2 * kBlk;
      uint8_t *Hb = Bb + nBr * 2 * kBlk;
      ptx::mbar_wait(&empty1[s], ((sb >> 1) & 1) ^ 1, a.err, 81);
      if (leader) {
        ptx::mbar_arrive_expect_tx(&full1[s], st1);
        ptx::tma_load_4d(Cb, &tm_C, sb * 64, g, tok0 + i0, b, &full1[s]);
        for (int r = 0; r < nBr; ++r)
          ptx::tma_load_4d(Bb + r * 2 * kBlk, &tm_B, sb * 64, g, tok0 + r * 128, b, &full1[s]);
        // the start states are written by the preceding kernel (the state
        // pass), which may still be running when this CTA starts
        if (sb == 0) ptx::griddep_wait();
        for (int q = 0; q < H; ++q) {
          const int row = (b * nh + hbase + q) * nc + k;
          for (int pb = 0; pb < nPb; ++pb)
            ptx::tma_load_3d(Hb + (q * nPb + pb) * kBlk, &tm_st, pb * 64, sb * 64, row,
                             &full1[s]);
        }
      }
      __syncwarp();
    }
    for (int q = 0; q < H; ++q)
      for (int jb = 0; jb < njb; ++jb) {
        const int u = q * njb + jb, s = u % nX;
        uint8_t *Xb = xbase + s * st2x;
        ptx::mbar_wait(&x_empty[s], ((u / nX) & 1) ^ 1, a.err, 83);
        if (leader) {
          ptx::mbar_arrive_expect_tx(&x_full[s], st2x);
          for (int pb = 0; pb < nPb; ++pb)
            ptx::tma_load_4d(Xb + pb * kBlk, &tm_x, pb * 64, hbase + q, tok0 + jb * 64, b,
                             &x_full[s]);
        }
        __syncwarp();
      }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t id_S = ptx::idesc_bf16(128, jext, false, false);
    const uint32_t id_Y = ptx::idesc_bf16(128, P, false, true);
    // with P a multiple of 64 the heads' state tiles abut in shared memory:
    // Y_q += C h_q^T for every head in one N = H P MMA
    const bool merged = (P % 64) == 0;
    const uint32_t id_Yall = ptx::idesc_bf16(128, merged ? H * P : P, false, true);
    const int n_ymma = merged ? 1 : H;
    for (int sb = 0; sb < nsb; ++sb) {
      const int s = sb & 1;
      uint8_t *Cb = smem + s * st1;
      uint8_t *Bb = Cb + 2 * kBlk;
      uint8_t *Hb = Bb + nBr * 2 * kBlk;
      ptx::mbar_wait(&full1[s], (sb >> 1) & 1, a.err, 84);
      ptx::tc_fence_after();
      if (leader) {
        const uint32_t c0 = ptx::smem_u32(Cb), b0 = ptx::smem_u32(Bb), h0 = ptx::smem_u32(Hb);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t cd = ptx::smem_desc(c0 + kk * 32, 16, 1024, ptx::kSw128);
          const uint64_t bd = ptx::smem_desc(b0 + kk * 32, 16, 1024, ptx::kSw128);
          const uint32_t acc = (sb | kk) ? 1u : 0u;
          ptx::mma_ss<false>(tmem, cd, bd, id_S, acc);
          for (int q = 0; q < n_ymma; ++q) {
            const uint64_t hd = ptx::smem_desc(h0 + q * nPb * kBlk + kk * 2048, kBlk, 1024,
                                               ptx::kSw128);
            ptx::mma_ss<false>(tmem + 256 + q * P, cd, hd, id_Yall, acc);
          }
        }
        ptx::mma_commit(&empty1[s]);
      }
      __syncwarp();
    }
    if (leader) ptx::mma_commit(&s1_done);
    __syncwarp();
    for (int q = 0; q < H; ++q) {
      ptx::mbar_wait(&ysc[q], 0, a.err, 85);
      ptx::tc_fence_after();
      for (int jb = 0; jb < njb; ++jb) {
        const int u = q * njb + jb, s = u % kNP, sx = u % nX;
        ptx::mbar_wait(&pm_full[s], (u / kNP) & 1, a.err, 86);
        ptx::mbar_wait(&x_full[sx], (u / nX) & 1, a.err, 87);
        ptx::tc_fence_after();
        if (leader) {
          const uint32_t p0 = ptx::smem_u32(smem + s * st2p);
          const uint32_t x0 = ptx::smem_u32(xbase + sx * st2x);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t pd = ptx::smem_desc(p0 + kk * 32, 16, 1024, ptx::kSw128);
            const uint64_t xd = ptx::smem_desc(x0 + kk * 2048, kBlk, 1024, ptx::kSw128);
            ptx::mma_ss<false>(tmem + 256 + q * P, pd, xd, id_Y, 1u);
          }
          ptx::mma_commit(&pm_empty[s]);
          ptx::mma_commit(&x_empty[sx]);
        }
        __syncwarp();
      }
      if (leader) ptx::mma_commit(&ydone[q]);
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ row warps
    const int quad = warp & 3, qtr = warp >> 2;  // TMEM lane quadrant, column quarter
    const int row = quad * 32 + (tid & 31);       // 0..127 = TMEM lane
    const int i_rel = i0 + row;
    const int rb = i_rel >> 6;                    // row's 64-token block
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;

    // in-chunk cumsums (log2 units) of the H heads, one token per thread;
    // every dt load is issued before the first scan
    float dh[kMaxH];
#pragma unroll
    for (int q = 0; q < kMaxH; ++q)
      dh[q] = (q < H && tid < valid && SSD_IN_BOUNDS(hbase + q < nh && b < a.nb, a.err, 120))
                  ? __bfloat162float(a.dt[((int64_t)b * L + tok0 + tid) * nh + hbase + q])
                  : 0.f;
#pragma unroll
    for (int q = 0; q < kMaxH; ++q) {
      if (q >= H) break;
      const float run = (hbase + q < nh ? a.A[hbase + q] : 0.f) * kLog2e * dh[q];
      float incl = run;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_up_sync(0xffffffffu, incl, off);
        if ((tid & 31) >= off) incl += o;
      }
      if ((tid & 31) == 31) warp_tot[warp] = incl;
      ptx::named_bar_sync(1, kRowThreads);
      float Gj = incl;
      for (int w2 = 0; w2 < warp; ++w2) Gj += warp_tot[w2];
      if (tid < T) {
        Gs[q][tid] = Gj;
        dts[q][tid] = dh[q];
      }
      ptx::named_bar_sync(1, kRowThreads);
      if (tid < T) vs[q][tid] = ptx::ex2_approx(Gs[q][tid | 63] - Gj) * dh[q];
    }
    ptx::named_bar_sync(1, kRowThreads);
    ptx::mbar_wait(&s1_done, 0, a.err, 88);
    ptx::tc_fence_after();

    // x of this thread's row and column groups (16-column group g belongs to
    // the warp with g % 4 == qtr), fetched before the wait on the head's
    // MMAs so the load latency overlaps other work
    uint4 xr[4];
    auto fetch_x = [&](int q) {
      const int64_t off = (((int64_t)b * L + tok0 + i_rel) * nh + hbase + q) * P;
      const bool ok = i_rel < valid;
#pragma unroll
      for (int gi = 0; gi < 2; ++gi) {
        const int c0 = (qtr + 4 * gi) * 16;
        if (c0 < P && ok) {
          xr[2 * gi] = *reinterpret_cast<const uint4 *>(a.x + off + c0);
          xr[2 * gi + 1] = *reinterpret_cast<const uint4 *>(a.x + off + c0 + 8);
        }
      }
    };
    auto epilogue = [&](int q) {
      ptx::mbar_wait(&ydone[q], 0, a.err, 89);
      ptx::tc_fence_after();
      const int h = hbase + q;
      const float Dh = a.D ? a.D[h] : 0.f;
      const int64_t off = (((int64_t)b * L + tok0 + i_rel) * nh + h) * P;
      const bool ok = i_rel < valid &&
                      SSD_IN_BOUNDS(h < nh && off + P <= (int64_t)a.nb * L * nh * P, a.err, 121);
#pragma unroll
      for (int gi = 0; gi < 2; ++gi) {
        const int c0 = (qtr + 4 * gi) * 16;
        if (c0 >= P) break;
        float v[16];
        ptx::tmem_ld16_sync(tmem + lane_base + 256 + q * P + c0, v);
        if (ok) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            float xv[8];
            unpack16(xr[2 * gi + hh], xv, (__nv_bfloat16 *)nullptr);
#pragma unroll
            for (int e = 0; e < 8; ++e) xv[e] = fmaf(Dh, xv[e], v[hh * 8 + e]);
            *reinterpret_cast<uint4 *>(a.y + off + c0 + hh * 8) =
                pack_io16(xv, (__nv_bfloat16 *)nullptr);
          }
        }
      }
    };

    fetch_x(0);
    for (int q = 0; q < H; ++q) {
      const float Gi = Gs[q][min(i_rel, T - 1)];
      // carried-state term: Y_q *= exp2(G_i), then release Y_q to phase 2
      const float eg = ptx::ex2_approx(Gi);
#pragma unroll
      for (int gi = 0; gi < 2; ++gi) {
        const int c0 = (qtr + 4 * gi) * 16;
        if (c0 >= P) break;
        float v[16];
        ptx::tmem_ld16_sync(tmem + lane_base + 256 + q * P + c0, v);
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] *= eg;
        ptx::tmem_st16(tmem + lane_base + 256 + q * P + c0, v);
      }
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(&ysc[q]);
      // decayed, masked interaction rows: this thread takes 16 of each
      // block's 64 tokens
      for (int jb = 0; jb < njb; ++jb) {
        const int u = q * njb + jb, s = u % kNP;
        ptx::mbar_wait(&pm_empty[s], ((u / kNP) & 1) ^ 1, a.err, 90);
        uint8_t *Pb = smem + s * st2p;
        const int jc0 = jb * 64 + qtr * 16;
        float v[16];
        ptx::tmem_ld16_sync(tmem + lane_base + jc0, v);  // every lane of the warp
        if (jb < rb) {
          // whole block before the row's block: factored decay
          const float ui = ptx::ex2_approx(Gi - Gs[q][jb * 64 + 63]);
          const float4 *vp = reinterpret_cast<const float4 *>(&vs[q][jc0]);
#pragma unroll
          for (int e4 = 0; e4 < 4; ++e4) {
            const float4 f = vp[e4];
            v[4 * e4 + 0] *= ui * f.x;
            v[4 * e4 + 1] *= ui * f.y;
            v[4 * e4 + 2] *= ui * f.z;
            v[4 * e4 + 3] *= ui * f.w;
          }
        } else if (jb == rb) {
          const float4 *gp = reinterpret_cast<const float4 *>(&Gs[q][jc0]);
          const float4 *dp = reinterpret_cast<const float4 *>(&dts[q][jc0]);
#pragma unroll
          for (int e4 = 0; e4 < 4; ++e4) {
            const float4 gj = gp[e4], dj = dp[e4];
            const float ga[4] = {gj.x, gj.y, gj.z, gj.w}, da[4] = {dj.x, dj.y, dj.z, dj.w};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int j = jc0 + 4 * e4 + c;
              v[4 * e4 + c] =
                  (j <= i_rel && j < valid) ? v[4 * e4 + c] * ptx::ex2_approx(Gi - ga[c]) * da[c] : 0.f;
            }
          }
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = 0.f;
        }
#pragma unroll
        for (int c = 0; c < 2; ++c)
          *reinterpret_cast<uint4 *>(Pb + sw128(row, (qtr * 2 + c) * 16)) =
              pack_op16(v + c * 8, (__nv_bfloat16 *)nullptr);
        ptx::fence_async_smem();
        ptx::tc_fence_before();
        ptx::mbar_arrive(&pm_full[s]);
      }
      if (q > 0) {
        epilogue(q - 1);  // uses the x rows of head q-1 fetched earlier
        fetch_x(q);       // in flight during the next head's decay pass
      }
    }
    epilogue(H - 1);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) ptx::tmem_dealloc(tmem, ncols);
}

}  // namespace

namespace {

// Shared memory of a launch with H heads per CTA: two phase-1 stages and nX
// x stages, within the 227 KB per CTA less the static arrays.
struct ScanSmem {
  int nX, smem;
};
ScanSmem scan_smem(const Dims &d, int H) {
  const int nBr = (int)((std::min<int64_t>(d.T, 256) + 127) / 128);
  const int nPb = (int)((d.P + 63) / 64);
  const int st1 = kBlk * 2 + nBr * kBlk * 2 + H * nPb * kBlk;
  const int st2x = nPb * kBlk;
  const int budget = 212 * 1024 - 2 * st1;
  ScanSmem m;
  m.nX = std::max(2, std::min(kMaxX, budget / st2x));
  m.smem = 2 * st1 + m.nX * st2x + 1024;
  return m;
}

}  // namespace

bool fwd_scan_heads_ok(const Dims &d, int H) {
  if (H < 1 || H > kMaxH || d.hpg % H || H * d.P > 256) return false;
  return scan_smem(d, H).smem <= 213 * 1024;
}

cudaError_t launch_fwd_scan(const Dims &d, const void *x, const void *B, const void *C,
                            const void *dt, const float *A, const void *states, const float *D,
                            void *y, int H, int *err, cudaStream_t st) {
  if (!fwd_scan_heads_ok(d, H)) return cudaErrorInvalidValue;
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
  const ScanSmem m = scan_smem(d, H);
  const int nX = m.nX, smem = m.smem;
  cudaError_t e =
      cudaFuncSetAttribute(fwd_scan_bf16, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  ScanArgs a;
  a.x = static_cast<const __nv_bfloat16 *>(x);
  a.dt = static_cast<const __nv_bfloat16 *>(dt);
  a.A = A;
  a.D = D;
  a.y = static_cast<__nv_bfloat16 *>(y);
  a.err = err;
  a.L = (int)d.L;
  a.nh = (int)d.nh;
  a.P = (int)d.P;
  a.S = (int)d.S;
  a.hpg = (int)d.hpg;
  a.T = (int)d.T;
  a.nc = (int)d.nc;
  a.nb = (int)d.b;
  a.H = H;
  a.nX = nX;
  const int n_it = (int)((d.T + 127) / 128);
  dim3 grid((unsigned)(d.nc * n_it), (unsigned)(d.nh / H), (unsigned)d.b);
  // programmatic stream serialisation: CTAs may start (barriers, tensor
  // memory, cumsums, C and B loads) while the state pass finishes; the
  // producer waits on the device before loading the start states
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fwd_scan_bf16, tC, tB, tx, tS, a);
}

}  // namespace ssd
