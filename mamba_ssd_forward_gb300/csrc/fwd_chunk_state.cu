// Forward path, chunk jump terms (bf16 I/O): for every chunk k and head h,
//
//   dH[k] = sum_{j in chunk} (exp2(G_last - G_j) dt_j) B_j (outer) x_j      (S x P)
//   gamma[k] = exp2(G_last)
//
// ("Accelerating Mamba-2 with High-Performance Forward Pass Kernels in NVIDIA
// CUDA Tile", section "Mamba-2 architecture": the second term of the
// log-space jump h_{t+T} = exp(G_last) h_t + (exp(G_last - G) B)^T X, with the
// in-chunk cumsum G of "Kernel 1" computed here.)  All chunks are
// independent, so this runs fully in parallel; the sequential part is the
// bandwidth kernel in fwd_state_pass.cu.
//
// One CTA per (chunk, 128-wide slice of S, group of H heads that share B,
// batch).  Warp roles:
//   warp 4 (TMA):  64-token blocks of B (MN-major, s contiguous; loaded once
//                  for the H heads) and of x for each head (MN-major);
//   warp 5 (MMA):  per block and head, M = 128 (s) x N = P MMAs into the
//                  head's tensor-memory accumulator (lane = s, column = p);
//   warps 0-3:     the heads' in-chunk cumsums and jump weights, the scaling
//                  of each x row by its weight (in shared memory), and the
//                  epilogue: dH as bf16 [b, nh, nc, S, P] (p contiguous, the
//                  layout the output kernel reads), gamma as fp32.
#include "fwd.cuh"

namespace ssd {
namespace {

constexpr int kStateThreads = 128;
constexpr int kThreads = kStateThreads + 64;
constexpr int kProducerWarp = 4, kMmaWarp = 5;
constexpr int kKB = 64;  // tokens per pipeline stage
constexpr int kNST = 2;  // pipeline stages
constexpr int kMaxH = 4;
constexpr int kBlk = kKB * 128;

__global__ void __launch_bounds__(kThreads, 2)
fwd_chunk_state_bf16(const __grid_constant__ CUtensorMap tm_B,
                     const __grid_constant__ CUtensorMap tm_x, const __nv_bfloat16 *__restrict__ dt,
                     const float *__restrict__ A, __nv_bfloat16 *__restrict__ dH,
                     float *__restrict__ gamma, int *__restrict__ err, int L, int nh, int P, int S,
                     int hpg, int T, int nc, int H) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ __align__(8) uint64_t full[kNST], scaled[kNST], empty[kNST], done;
  __shared__ uint32_t tmem_slot;
  __shared__ float w_s[kMaxH][256];
  __shared__ float warp_tot[4];

  const int n_st = (S + 127) / 128;
  const int k = blockIdx.x / n_st, st_idx = blockIdx.x % n_st;
  const int hbase = blockIdx.y * H, b = blockIdx.z, g = hbase / hpg;
  const int s0 = st_idx * 128;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int nPb = (P + 63) / 64;
  const int xbytes = nPb * kBlk;                       // one head's x block
  const int stage_bytes = 2 * kBlk + H * xbytes;       // B block | x blocks
  const int tok0 = k * T;
  const int valid = min(T, L - tok0);
  const int nkb = (valid + kKB - 1) / kKB;
  const uint32_t ncols = H * P <= 32 ? 32 : (H * P <= 64 ? 64 : (H * P <= 128 ? 128 : 256));

  if (tid == 0) {
    for (int i = 0; i < kNST; ++i) {
      ptx::mbar_init(&full[i], 1);
      ptx::mbar_init(&scaled[i], kStateThreads);
      ptx::mbar_init(&empty[i], 1);
    }
    ptx::mbar_init(&done, 1);
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
    for (int kb = 0; kb < nkb; ++kb) {
      const int st = kb % kNST;
      ptx::mbar_wait(&empty[st], ((kb / kNST) & 1) ^ 1, err, 101);
      if (leader) {
        uint8_t *Bb = smem + st * stage_bytes;
        uint8_t *Xb = Bb + 2 * kBlk;
        const int tok = tok0 + kb * kKB;
        ptx::mbar_arrive_expect_tx(&full[st], stage_bytes);
        for (int mb = 0; mb < 2; ++mb)
          ptx::tma_load_4d(Bb + mb * kBlk, &tm_B, s0 + mb * 64, g, tok, b, &full[st]);
        for (int q = 0; q < H; ++q)
          for (int pb = 0; pb < nPb; ++pb)
            ptx::tma_load_4d(Xb + q * xbytes + pb * kBlk, &tm_x, pb * 64, hbase + q, tok, b,
                             &full[st]);
      }
      __syncwarp();
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idesc = ptx::idesc_bf16(128, P, true, true);
    for (int kb = 0; kb < nkb; ++kb) {
      const int st = kb % kNST;
      ptx::mbar_wait(&scaled[st], (kb / kNST) & 1, err, 102);
      ptx::tc_fence_after();
      if (leader) {
        const uint32_t b0 = ptx::smem_u32(smem + st * stage_bytes);
        const uint32_t x0 = b0 + 2 * kBlk;
        for (int q = 0; q < H; ++q) {
#pragma unroll
          for (int kk = 0; kk < kKB / 16; ++kk) {
            const uint64_t ad = ptx::smem_desc(b0 + kk * 2048, kBlk, 1024, ptx::kSw128);
            const uint64_t bd =
                ptx::smem_desc(x0 + q * xbytes + kk * 2048, kBlk, 1024, ptx::kSw128);
            ptx::mma_ss<false>(tmem + q * P, ad, bd, idesc, (kb | kk) ? 1u : 0u);
          }
        }
        ptx::mma_commit(&empty[st]);
      }
      __syncwarp();
    }
    if (leader) ptx::mma_commit(&done);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ row warps
    // in-chunk cumsums of the H heads (two tokens per thread), jump weights
    const int per = T > 128 ? 2 : 1;
    float d[kMaxH][2];
#pragma unroll
    for (int q = 0; q < kMaxH; ++q)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int j = tid * per + e;
        d[q][e] = (q < H && e < per && j < valid)
                      ? __bfloat162float(dt[((int64_t)b * L + tok0 + j) * nh + hbase + q])
                      : 0.f;
      }
#pragma unroll
    for (int q = 0; q < kMaxH; ++q) {
      if (q >= H) break;
      const float Ah = A[hbase + q] * kLog2e;
      float c[2], run = 0.f;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        run += Ah * d[q][e];
        c[e] = run;
      }
      float incl = run;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_up_sync(0xffffffffu, incl, off);
        if ((tid & 31) >= off) incl += o;
      }
      if ((tid & 31) == 31) warp_tot[warp] = incl;
      ptx::named_bar_sync(1, kStateThreads);
      float base = incl - run;
      for (int w2 = 0; w2 < warp; ++w2) base += warp_tot[w2];
      // the chunk's last real token is the last nonzero contribution, so the
      // block total equals G at position valid - 1
      float tot = 0.f;
      for (int w2 = 0; w2 < 4; ++w2) tot += warp_tot[w2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int j = tid * per + e;
        if (e < per && j < T) w_s[q][j] = j < valid ? exp2f(tot - (base + c[e])) * d[q][e] : 0.f;
      }
      if (tid == 0 && st_idx == 0) gamma[((int64_t)b * nh + hbase + q) * nc + k] = exp2f(tot);
      ptx::named_bar_sync(1, kStateThreads);
    }
    // scale each head's x rows by its weights
    for (int kb = 0; kb < nkb; ++kb) {
      const int st = kb % kNST;
      uint8_t *Xb = smem + st * stage_bytes + 2 * kBlk;
      ptx::mbar_wait(&full[st], (kb / kNST) & 1, err, 103);
      const int nchunks = nPb * kKB * 8;  // 16-byte chunks of one head's block
      for (int c = tid; c < H * nchunks; c += kStateThreads) {
        const int q = c / nchunks, cc = c % nchunks;
        const float ws = w_s[q][kb * kKB + ((cc >> 3) & (kKB - 1))];
        uint4 *p4 = reinterpret_cast<uint4 *>(Xb + q * xbytes + cc * 16);
        float v[8];
        unpack16(*p4, v, (__nv_bfloat16 *)nullptr);
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] *= ws;
        *p4 = pack_op16(v, (__nv_bfloat16 *)nullptr);
      }
      ptx::fence_async_smem();
      ptx::mbar_arrive(&scaled[st]);
    }
    // epilogue: this thread's row s of every head's dH
    ptx::mbar_wait(&done, 0, err, 104);
    ptx::tc_fence_after();
    const int srow = s0 + tid;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    for (int q = 0; q < H; ++q) {
      __nv_bfloat16 *o = dH + ((((int64_t)b * nh + hbase + q) * nc + k) * S + srow) * P;
      for (int c0 = 0; c0 < P; c0 += 16) {
        float v[16];
        ptx::tmem_ld16_sync(tmem + lane_base + q * P + c0, v);
        if (srow < S) {
          uint4 *o4 = reinterpret_cast<uint4 *>(o + c0);
          o4[0] = pack_io16(v, (__nv_bfloat16 *)nullptr);
          o4[1] = pack_io16(v + 8, (__nv_bfloat16 *)nullptr);
        }
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) ptx::tmem_dealloc(tmem, ncols);
}

}  // namespace

int fwd_state_heads(const Dims &d) {
  const int hmax = (int)std::min<int64_t>(kMaxH, 256 / d.P);
  for (int h = hmax; h > 1; --h)
    if (d.hpg % h == 0) return h;
  return 1;
}

cudaError_t launch_fwd_chunk_state(const Dims &d, const void *x, const void *B, const void *dt,
                                   const float *A, void *dH, float *gamma, cudaStream_t st) {
  const int H = fwd_state_heads(d);
  CUtensorMap tB, tx;
  if (!make_tmap_bl(&tB, B, true, d.b, d.L, d.ng, d.S, kKB) ||
      !make_tmap_bl(&tx, x, true, d.b, d.L, d.nh, d.P, kKB))
    return cudaErrorInvalidValue;
  const int nPb = (int)((d.P + 63) / 64);
  const int smem = kNST * (2 * kBlk + H * nPb * kBlk) + 1024;
  cudaError_t e = cudaFuncSetAttribute(fwd_chunk_state_bf16,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int n_st = (int)((d.S + 127) / 128);
  dim3 grid((unsigned)(d.nc * n_st), (unsigned)(d.nh / H), (unsigned)d.b);
  fwd_chunk_state_bf16<<<grid, kThreads, smem, st>>>(
      tB, tx, static_cast<const __nv_bfloat16 *>(dt), A, static_cast<__nv_bfloat16 *>(dH), gamma,
      device_error_word(), (int)d.L, (int)d.nh, (int)d.P, (int)d.S, (int)d.hpg, (int)d.T,
      (int)d.nc, H);
  return cudaGetLastError();
}

}  // namespace ssd
